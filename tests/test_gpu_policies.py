"""Multi-step decode policies built from the entry points, against the fp64
oracle step by step.

* Fill then evict: decoding starts from an empty cache; while empty slots
  remain the step returns the lowest one (LF_STEP_FILL_EMPTY_FIRST), so the
  budget fills token by token, and from then on every step evicts the
  LongFlowScore argmin.
* Periodic compression (the baselines' policy of the Fig. 3 caption): every k
  steps the k lowest-score slots are returned at once and masked
  (LF_STEP_MASK_EVICTED); the following steps refill them one per step.

Both sides always write the oracle's chosen slot, so their states stay
identical; the GPU's choices are checked with the same tolerance rule as
next_slot elsewhere.
"""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
import oracle
from decode_kv_cache_step_gb300.workloads import f32_to_bf16_bits

from _gpu import OUT_ATOL, to_dev, to_host_bits
from test_gpu_next import _ranked, compare_topk

pytestmark = pytest.mark.gpu


def _rand(rng, *shape):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32))


def _step_inputs(rng, B, Hq, Hkv, d):
    return {"q": _rand(rng, B, Hq, d), "new_k": _rand(rng, B, Hkv, d), "new_v": _rand(rng, B, Hkv, d)}


def test_fill_then_evict():
    rng = np.random.default_rng(2024)
    B, Hq, Hkv, d, S, W = 2, 8, 2, 64, 192, 8
    scale = 0.125
    k = _rand(rng, B, Hkv, S, d)
    v = _rand(rng, B, Hkv, S, d)
    mask = np.full((B, Hkv, S), -1, dtype=np.int32)          # empty cache
    host = {"k_cache": k.copy(), "v_cache": v.copy(), "mask": mask.copy()}
    dk, dv, dm = to_dev(k), to_dev(v), to_dev(mask)
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty((B, Hkv, 1), dtype=torch.int32, device="cuda")
    ws = np.full((B, Hkv), -1, dtype=np.int32)
    for t in range(S + 40):
        inp = _step_inputs(rng, B, Hq, Hkv, d)
        dinp = {kk: to_dev(vv) for kk, vv in inp.items()}
        lf.decode_step_ex(dinp["q"], dk, dv, dm, dinp["new_k"], dinp["new_v"], to_dev(ws), out,
                          nxt, W, scale, k=1, flags=lf.LF_STEP_FILL_EMPTY_FIRST)
        ora = oracle.decode_step(inp["q"], host["k_cache"], host["v_cache"], host["mask"],
                                 inp["new_k"], inp["new_v"], ws, W, scale, want_scores=True,
                                 fill_first=True)
        torch.cuda.synchronize()
        assert np.array_equal(dm.cpu().numpy(), host["mask"]), f"step {t}: mask"
        err = np.max(np.abs(out.float().cpu().numpy() - ora["out"]))
        assert err <= OUT_ATOL, f"step {t}: out error {err}"
        got = nxt.cpu().numpy()
        live = host["mask"] >= 0
        for b in range(B):
            for h in range(Hkv):
                if not live[b, h].all():
                    # still filling: the lowest empty slot, exactly
                    assert got[b, h, 0] == np.flatnonzero(~live[b, h])[0], f"step {t}"
                ranked = _ranked(ora["scores"][b, h], host["mask"][b, h], W, True)
                compare_topk(got[b, h], ranked, 1, f"step {t} unit ({b},{h})")
        ws = ora["next_slot"].astype(np.int32).copy()
    assert (host["mask"] >= 0).all()                          # the budget filled
    assert np.array_equal(to_host_bits(dk), host["k_cache"])
    assert lf.device_errors() == 0


@pytest.mark.parametrize("period", [8, 32])
def test_periodic_compression(period):
    rng = np.random.default_rng(period)
    B, Hq, Hkv, d, S, W = 2, 8, 2, 128, 256, 16
    scale = 0.088
    k = _rand(rng, B, Hkv, S, d)
    v = _rand(rng, B, Hkv, S, d)
    mask = np.broadcast_to((S - 1 - np.arange(S, dtype=np.int32)), (B, Hkv, S)).copy()
    host = {"k_cache": k.copy(), "v_cache": v.copy(), "mask": mask.copy()}
    dk, dv, dm = to_dev(k), to_dev(v), to_dev(mask)
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    freed = None     # [B][Hkv][period] slots to refill, in order
    for t in range(3 * period):
        inp = _step_inputs(rng, B, Hq, Hkv, d)
        dinp = {kk: to_dev(vv) for kk, vv in inp.items()}
        pos = t % period
        ws = np.full((B, Hkv), -1, dtype=np.int32) if freed is None else freed[:, :, pos].copy()
        if pos == period - 1:
            # compression step: return `period` slots at once and mask them
            nxt = torch.empty((B, Hkv, period), dtype=torch.int32, device="cuda")
            lf.decode_step_ex(dinp["q"], dk, dv, dm, dinp["new_k"], dinp["new_v"], to_dev(ws), out,
                              nxt, W, scale, k=period, flags=lf.LF_STEP_MASK_EVICTED)
            ora = oracle.decode_step(inp["q"], host["k_cache"], host["v_cache"], host["mask"],
                                     inp["new_k"], inp["new_v"], ws, W, scale, want_scores=True,
                                     topk=period)
            torch.cuda.synchronize()
            got = nxt.cpu().numpy()
            for b in range(B):
                for h in range(Hkv):
                    ranked = _ranked(ora["scores"][b, h], host["mask"][b, h], W, False)
                    compare_topk(got[b, h], ranked, period, f"step {t} unit ({b},{h})")
            freed = ora["next_slot"].astype(np.int32).copy()
            for b in range(B):
                for h in range(Hkv):
                    host["mask"][b, h, freed[b, h]] = -1       # the oracle's picks, masked
            # both sides continue from the oracle's choice
            dm.copy_(to_dev(host["mask"]))
        else:
            lf.decode_attention(dinp["q"], dk, dv, dm, dinp["new_k"], dinp["new_v"], to_dev(ws), out,
                                scale)
            ora = oracle.decode_step(inp["q"], host["k_cache"], host["v_cache"], host["mask"],
                                     inp["new_k"], inp["new_v"], ws, W, scale, attention_only=True)
            torch.cuda.synchronize()
            assert np.array_equal(dm.cpu().numpy(), host["mask"]), f"step {t}: mask"
        err = np.max(np.abs(out.float().cpu().numpy() - ora["out"]))
        assert err <= OUT_ATOL, f"step {t}: out error {err}"
        assert np.array_equal(to_host_bits(dk), host["k_cache"]), f"step {t}: k cache"
    assert lf.device_errors() == 0
