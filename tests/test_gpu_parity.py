"""GPU parity: the CUDA decode step against the fp64 oracle on the seeded
workloads, step after step.

Small workloads are compared element by element on every unit. The three
large workloads run at full size in the launch configuration the benchmark
times; the oracle checks a sample of (b, kvh) units one by one, and every unit
is checked for the properties that hold at any size (eligible, never
protected, never masked). Both sides write the oracle's chosen slot at the
next step, so their states stay identical.
"""
import os

import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
from decode_kv_cache_step_gb300.workloads import WORKLOADS, initial_state, step_inputs

from _gpu import DevState, compare_unit, oracle_step, to_host_bits

pytestmark = pytest.mark.gpu


def _sample_units(wl, n, seed=0):
    rng = np.random.default_rng(seed)
    units = {0, wl.units - 1}
    units.update(int(x) for x in rng.choice(wl.units, size=min(n, wl.units), replace=False))
    return sorted(units)


def run_parity(wl, steps, sample=None, check_scores=True, scores_every=1):
    """Steps the GPU and the oracle side by side. With scores_every = n only
    every n-th step exports the GPU's scores (and compares them); the others
    call lf_decode_step itself, the entry point the benchmark times."""
    st = initial_state(wl)
    dev = DevState(st["k_cache"], st["v_cache"], st["mask"], wl.Hq)
    host = {k: st[k] for k in ("k_cache", "v_cache", "mask")}
    ws = np.full((wl.B, wl.Hkv), -1, dtype=np.int32)
    units = list(range(wl.units)) if sample is None else sample
    worst = {"out_err": 0.0, "score_rel": 0.0, "exact_next": 0, "checked": 0}
    for t in range(steps + 1):
        inp = step_inputs(wl, t)
        with_scores = check_scores and t % scores_every == 0
        gpu = dev.step(inp["q"], inp["new_k"], inp["new_v"], ws, wl.W, wl.scale, scores=with_scores)
        ora = oracle_step(host, inp["q"], inp["new_k"], inp["new_v"], ws, wl.W, wl.scale,
                          units=None if sample is None else units)
        mask_gpu = dev.mask.cpu().numpy()
        for u in units:
            b, kvh = divmod(u, wl.Hkv)
            # state after the write: bit-exact
            assert np.array_equal(mask_gpu[b, kvh], host["mask"][b, kvh]), f"step {t}: mask ({b},{kvh})"
            if ws[b, kvh] >= 0:
                s = int(ws[b, kvh])
                assert np.array_equal(to_host_bits(dev.k[b, kvh, s]), host["k_cache"][b, kvh, s])
                assert np.array_equal(to_host_bits(dev.v[b, kvh, s]), host["v_cache"][b, kvh, s])
            stt = compare_unit(gpu, ora, b, kvh, wl.g, host["mask"], wl.W, check_scores=with_scores,
                               where=f"{wl.name} step {t}")
            worst["out_err"] = max(worst["out_err"], stt["out_err"])
            worst["score_rel"] = max(worst["score_rel"], stt.get("score_rel", 0.0))
            worst["exact_next"] += int(stt.get("exact_next", True))
            worst["checked"] += 1
        # properties on every unit
        nxt = gpu["next_slot"]
        live_elig = mask_gpu >= wl.W
        for u in range(wl.units):
            b, kvh = divmod(u, wl.Hkv)
            n = int(nxt[b, kvh])
            if n == -1:
                assert not live_elig[b, kvh].any(), f"step {t}: unit ({b},{kvh}) returned -1"
            else:
                assert 0 <= n < wl.S and live_elig[b, kvh, n], f"step {t}: unit ({b},{kvh}) slot {n}"
        ws = nxt.astype(np.int32).copy()
        for u in units:
            b, kvh = divmod(u, wl.Hkv)
            ws[b, kvh] = ora["next_slot"][b, kvh]
    assert lf.device_errors() == 0
    return worst


def test_parity_tiny_every_step():
    wl = WORKLOADS["tiny_b2_s256"]
    worst = run_parity(wl, wl.steps)
    assert worst["checked"] == (wl.steps + 1) * wl.units


def test_parity_qwen3_b1_s2400_every_step():
    wl = WORKLOADS["qwen3_8b_b1_s2400"]
    worst = run_parity(wl, wl.steps)
    assert worst["checked"] == (wl.steps + 1) * wl.units


@pytest.mark.slow
@pytest.mark.parametrize("name", ["qwen3_8b_b128_s3200", "llama8b_b256_s2400_ragged",
                                  "long_b32_s16384_ragged"])
def test_parity_full_size_sampled(name):
    """Every prescribed decode step of the three large workloads (64, 128
    and 64 after the priming call) at full size, in the benchmark's launch
    plan: 16 sampled units against the oracle at every step (out, scores on
    even steps, next_slot, cache and mask bits), every unit checked for a
    valid choice. The 16K-slot workload runs its split finish throughout."""
    wl = WORKLOADS[name]
    worst = run_parity(wl, steps=wl.steps, sample=_sample_units(wl, 14, seed=len(name)),
                       scores_every=2)
    assert worst["checked"] == (wl.steps + 1) * len(_sample_units(wl, 14, seed=len(name)))


def test_scoreless_entry_point_matches_scores_variant():
    """lf_decode_step (what the benchmark times) and lf_decode_step_scores give
    the same output and slot, bit for bit."""
    wl = WORKLOADS["qwen3_8b_b128_s3200"].with_batch(16)
    st = initial_state(wl)
    inp = step_inputs(wl, 1)
    ws = np.random.default_rng(0).integers(0, wl.S, size=(wl.B, wl.Hkv)).astype(np.int32)
    a = DevState(st["k_cache"], st["v_cache"], st["mask"], wl.Hq)
    b = DevState(st["k_cache"], st["v_cache"], st["mask"], wl.Hq)
    ra = a.step(inp["q"], inp["new_k"], inp["new_v"], ws, wl.W, wl.scale, scores=True)
    rb = b.step(inp["q"], inp["new_k"], inp["new_v"], ws, wl.W, wl.scale, scores=False)
    assert np.array_equal(ra["out"], rb["out"])
    assert np.array_equal(ra["next_slot"], rb["next_slot"])
    assert torch.equal(a.mask, b.mask) and torch.equal(a.k, b.k) and torch.equal(a.v, b.v)


@pytest.mark.parametrize("io", ["pinned", "pageable", "mixed", "pinned_staged"])
def test_host_io_entry_point_matches_device_entry_point(monkeypatch, io):
    """lf_decode_step_host: pinned buffers are used in place by the kernel,
    pageable ones go through device staging (mixed: some of each); both give
    the device entry point's bits."""
    if io == "pinned_staged":
        monkeypatch.setenv("LF_HOST_ZEROCOPY", "0")
    wl = WORKLOADS["llama8b_b256_s2400_ragged"].with_batch(8)
    st = initial_state(wl)
    inp = step_inputs(wl, 2)
    ws = np.full((wl.B, wl.Hkv), 5, dtype=np.int32)
    a = DevState(st["k_cache"], st["v_cache"], st["mask"], wl.Hq)
    b = DevState(st["k_cache"], st["v_cache"], st["mask"], wl.Hq)
    ra = a.step(inp["q"], inp["new_k"], inp["new_v"], ws, wl.W, wl.scale, scores=False)
    def host(x, pinned):
        t = torch.from_numpy((x.view(np.int16) if x.dtype == np.uint16 else x).copy())
        return t.pin_memory() if pinned else t
    pins = {"pinned": [True] * 6, "pinned_staged": [True] * 6, "pageable": [False] * 6,
            "mixed": [True, False, True, False, False, True]}[io]
    q, nk, nv, w = (host(inp["q"], pins[0]), host(inp["new_k"], pins[1]),
                    host(inp["new_v"], pins[2]), host(ws, pins[3]))
    q, nk, nv = q.view(torch.bfloat16), nk.view(torch.bfloat16), nv.view(torch.bfloat16)
    out = torch.full((wl.B, wl.Hq, wl.d), 7.0, dtype=torch.bfloat16)
    nxt = torch.full((wl.B, wl.Hkv), -5, dtype=torch.int32)
    out = out.pin_memory() if pins[4] else out
    nxt = nxt.pin_memory() if pins[5] else nxt
    lf.decode_step_host(q, b.k, b.v, b.mask, nk, nv, w, out, nxt, wl.W, wl.scale)
    torch.cuda.synchronize()
    assert np.array_equal(out.float().numpy().astype(np.float64), ra["out"])
    assert np.array_equal(nxt.numpy(), ra["next_slot"])
    assert torch.equal(a.mask, b.mask) and torch.equal(a.k, b.k)


@pytest.mark.parametrize("cluster,split,deep", [("1", "0", "1"), ("1", "0", "0"), ("0", "0", "1"),
                                                ("0", "1", "1")])
@pytest.mark.parametrize("chunk_tiles", ["1", "3", "32"])
def test_split_shapes_do_not_change_results(monkeypatch, chunk_tiles, cluster, split, deep):
    """Different slot-axis splits, merged inside a thread-block cluster (deep
    or 2-stage TMA ring) or by the unit's last CTA (scoring there or in the
    split-finish kernel), give results within tolerance of the oracle."""
    monkeypatch.setenv("LF_CHUNK_TILES", chunk_tiles)
    monkeypatch.setenv("LF_CLUSTER", cluster)
    monkeypatch.setenv("LF_SPLIT", split)
    monkeypatch.setenv("LF_DEEP", deep)
    wl = WORKLOADS["long_b32_s16384_ragged"].with_batch(2)
    run_parity(wl, steps=2)


@pytest.mark.parametrize("name", ["qwen3_8b_b1_s2400", "tiny_b2_s256"])
def test_two_stage_cluster_path_every_step(monkeypatch, name):
    """The cluster merge with the 2-stage TMA ring (grids of more than one CTA
    per SM, or chunks of fewer than 5 tiles), with the deep ring off."""
    monkeypatch.setenv("LF_DEEP", "0")
    wl = WORKLOADS[name]
    run_parity(wl, min(wl.steps, 32))


@pytest.mark.parametrize("deep", ["0", "1"])
@pytest.mark.parametrize("cmax", ["5", "8", "16"])
def test_cluster_sizes_every_step(monkeypatch, cmax, deep):
    """Clusters capped at 5 CTAs (an odd split of the output row among the
    CTAs), 8 (the portable size; chunks of 5 tiles) and 16 (the default, a
    non-portable size; chunks of 3 tiles), in the deep and the 2-stage TMA
    ring."""
    monkeypatch.setenv("LF_CLUSTER_MAX", cmax)
    monkeypatch.setenv("LF_DEEP", deep)
    wl = WORKLOADS["qwen3_8b_b1_s2400"]
    run_parity(wl, min(wl.steps, 32))


@pytest.mark.parametrize("cmax", ["12", "16"])
def test_cluster_sizes_long_units(monkeypatch, cmax):
    """16K-slot units forced into clusters of 12 or 16 CTAs (chunks of 22 or
    16 tiles)."""
    monkeypatch.setenv("LF_CLUSTER", "1")
    monkeypatch.setenv("LF_CLUSTER_MAX", cmax)
    wl = WORKLOADS["long_b32_s16384_ragged"].with_batch(2)
    run_parity(wl, steps=2)


@pytest.mark.parametrize("name,batch", [("qwen3_8b_b128_s3200", 8), ("qwen3_8b_b128_s3200", 16),
                                        ("long_b32_s16384_ragged", 4)])
def test_mid_batch_cluster_plans(name, batch):
    """Mid-size batches whose default plan takes longer chunks so that every
    unit's cluster is resident at once (6 chunks of 9 tiles, 3 of 17, 12 of
    22 on GB300)."""
    wl = WORKLOADS[name].with_batch(batch)
    p = lf.step_plan(wl.B, wl.Hq, wl.Hkv, wl.d, wl.S)
    assert p["cluster"] and wl.units <= p["cluster_fit"], p
    run_parity(wl, steps=3, sample=_sample_units(wl, 14, seed=batch))


@pytest.mark.parametrize("split", ["0", "1"])
@pytest.mark.parametrize("name", ["qwen3_8b_b1_s2400", "tiny_b2_s256"])
def test_last_cta_merge_path_every_step(monkeypatch, name, split):
    """The merge by the unit's last CTA (used when clusters are off, a unit
    has more chunks than a cluster holds or the clusters would not all be
    resident at once) on every step of the small workloads, scoring in the
    same kernel or in the split-finish kernel."""
    monkeypatch.setenv("LF_CLUSTER", "0")
    monkeypatch.setenv("LF_SPLIT", split)
    wl = WORKLOADS[name]
    run_parity(wl, min(wl.steps, 32))
