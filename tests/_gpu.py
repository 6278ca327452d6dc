"""Helpers for the GPU parity tests: move seeded numpy cases to the device,
run the library step through the C ABI, and compare with the fp64 oracle.

Tolerances (bf16 inputs and output, fp32 accumulation on the GPU):
  * out: max |gpu - oracle| <= 2e-2 (gpu out is bf16, oracle out is fp64);
  * scores: |gpu - oracle| <= 1e-3 * oracle where oracle >= 1e-30
    (below that the fp32 value must itself be < 1e-29);
  * next_slot: equal whenever the oracle's best-to-second-best eligible gap
    exceeds 1e-3 relative; otherwise the GPU's slot must be eligible and its
    oracle score within 1e-3 of the oracle's minimum;
  * caches and mask after the step: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import decode_kv_cache_step_gb300 as lf
import oracle

OUT_ATOL = 2e-2
SCORE_RTOL = 1e-3
GAP_RTOL = 1e-3


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class DevState:
    """Device copies of the resident state plus per-step buffers."""

    def __init__(self, k_cache, v_cache, mask, Hq):
        self.k = to_dev(k_cache)
        self.v = to_dev(v_cache)
        self.mask = to_dev(mask)
        B, Hkv, S, d = k_cache.shape
        self.shape = (B, Hq, Hkv, d, S)
        self.out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
        self.next = torch.empty((B, Hkv), dtype=torch.int32, device="cuda")
        self.scores = torch.empty((B, Hkv, S), dtype=torch.float32, device="cuda")

    def step(self, q, new_k, new_v, write_slot, W, scale, scores=True):
        qd, nk, nv, ws = to_dev(q), to_dev(new_k), to_dev(new_v), to_dev(write_slot)
        if scores:
            lf.decode_step_scores(qd, self.k, self.v, self.mask, nk, nv, ws, self.out, self.next,
                                  self.scores, W, scale)
        else:
            lf.decode_step(qd, self.k, self.v, self.mask, nk, nv, ws, self.out, self.next, W, scale)
        torch.cuda.synchronize()
        res = {
            "out": self.out.float().cpu().numpy().astype(np.float64),
            "next_slot": self.next.cpu().numpy(),
        }
        if scores:
            res["scores"] = self.scores.cpu().numpy().astype(np.float64)
        return res


def oracle_step(state, q, new_k, new_v, write_slot, W, scale, units=None, scores=True):
    """Runs the oracle in place on the host state dict (k_cache, v_cache, mask)."""
    return oracle.decode_step(q, state["k_cache"], state["v_cache"], state["mask"], new_k, new_v,
                              write_slot, W, scale, want_scores=scores, units=units)


def compare_unit(gpu, ora, b, kvh, g, mask_after, W, check_scores=True, where=""):
    """Element-wise comparison of one (b, kvh) unit; returns a dict of stats."""
    o_g = gpu["out"][b, kvh * g:(kvh + 1) * g]
    o_o = ora["out"][b, kvh * g:(kvh + 1) * g]
    err = float(np.max(np.abs(o_g - o_o))) if o_g.size else 0.0
    assert err <= OUT_ATOL, f"{where} unit ({b},{kvh}): out max-abs error {err}"
    stats = {"out_err": err}
    ages = mask_after[b, kvh]
    live = ages >= 0
    if check_scores:
        sg = gpu["scores"][b, kvh]
        so = ora["scores"][b, kvh]
        assert np.all(np.isinf(sg[~live])), f"{where} unit ({b},{kvh}): masked slot has a finite score"
        big = live & (so >= 1e-30)
        rel = np.abs(sg[big] - so[big]) / so[big] if big.any() else np.zeros(1)
        assert np.all(rel <= SCORE_RTOL), \
            f"{where} unit ({b},{kvh}): score rel error {rel.max()} at slot {np.flatnonzero(big)[np.argmax(rel)]}"
        small = live & (so < 1e-30)
        assert np.all(sg[small] < 1e-29), f"{where} unit ({b},{kvh}): tiny score mismatch"
        stats["score_rel"] = float(rel.max())
    n_g = int(gpu["next_slot"][b, kvh])
    n_o = int(ora["next_slot"][b, kvh])
    elig = np.flatnonzero(ages >= W)
    if elig.size == 0:
        assert n_g == -1 and n_o == -1, f"{where} unit ({b},{kvh}): expected -1, gpu {n_g} oracle {n_o}"
        return stats
    so = ora["scores"][b, kvh]
    vals = np.sort(so[elig])
    best = vals[0]
    if elig.size == 1:
        gap = np.inf
    elif best > 0:
        gap = (vals[1] - best) / best
    else:
        gap = np.inf if vals[1] > 0 else 0.0
    assert n_g in set(elig.tolist()), f"{where} unit ({b},{kvh}): gpu slot {n_g} is not eligible"
    if gap > GAP_RTOL:
        assert n_g == n_o, f"{where} unit ({b},{kvh}): next_slot gpu {n_g} oracle {n_o} (gap {gap})"
    else:
        assert so[n_g] <= best * (1 + GAP_RTOL), \
            f"{where} unit ({b},{kvh}): near-tie pick {n_g} scores {so[n_g]} vs min {best}"
    stats["exact_next"] = n_g == n_o
    return stats

