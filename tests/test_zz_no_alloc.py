"""The allocation-free entry point, lf_decode_step_noalloc, against lf_decode_step.

Some callers cannot call cudaMalloc once they are running: a serving engine
that hands all free GPU memory to its own pools at start-up has none left,
and a real-time decode loop may not accept the device-wide synchronisation
that cudaMalloc and cudaFree can cause. lf_decode_step_noalloc serves them by
keeping its scratch in a fixed array compiled into the library. These tests
call it through the C ABI and check that two calls in a row give the same
result as the allocating entry point, within the tolerances the other GPU
tests use, that several steps in a row match the fp64 oracle directly, that
its device error bits (an ignored write slot, a pipeline wait that gave up)
reach the caller through lf_device_errors, and that a shape whose scratch
does not fit is refused.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
from decode_kv_cache_step_gb300.workloads import WORKLOADS, initial_state, step_inputs

import _pins
from _gpu import OUT_ATOL, compare_unit, oracle_step, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def _state(st):
    return {"k": to_dev(st["k_cache"]), "v": to_dev(st["v_cache"]), "mask": to_dev(st["mask"])}


def test_noalloc_matches_lf_decode_step_on_two_calls_in_a_row():
    wl = WORKLOADS["qwen3_8b_b128_s3200"].with_batch(8)
    st = initial_state(wl)
    lib = lf.load_library()
    ref, got = _state(st), _state(st)
    shape = (wl.B, wl.Hq, wl.d)
    out_ref = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    out_got = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    ws_ref = torch.full((wl.B, wl.Hkv), -1, dtype=torch.int32, device="cuda")
    ws_got = ws_ref.clone()
    nxt_ref = torch.empty_like(ws_ref)
    nxt_got = torch.empty_like(ws_ref)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        inp = step_inputs(wl, call)
        q, nk, nv = to_dev(inp["q"]), to_dev(inp["new_k"]), to_dev(inp["new_v"])
        lf.decode_step(q, ref["k"], ref["v"], ref["mask"], nk, nv, ws_ref, out_ref, nxt_ref,
                       wl.W, wl.scale)
        rc = lib.lf_decode_step_noalloc(
            q.data_ptr(), got["k"].data_ptr(), got["v"].data_ptr(), got["mask"].data_ptr(),
            nk.data_ptr(), nv.data_ptr(), ws_got.data_ptr(), out_got.data_ptr(),
            nxt_got.data_ptr(), wl.B, wl.Hq, wl.Hkv, wl.d, wl.S, wl.W, ctypes.c_float(wl.scale),
            stream)
        assert rc == lf.LF_OK, lib.lf_last_error().decode()
        torch.cuda.synchronize()
        err = (out_got.float() - out_ref.float()).abs().max().item()
        assert err <= OUT_ATOL, f"call {call}: output differs by {err}"
        assert torch.equal(nxt_got, nxt_ref), f"call {call}: next_slot differs"
        assert torch.equal(got["mask"], ref["mask"]), f"call {call}: mask differs"
        assert torch.equal(got["k"], ref["k"]) and torch.equal(got["v"], ref["v"])
        if call == 1:
            assert (ws_got >= 0).all()  # the second call really wrote new tokens
        ws_ref.copy_(nxt_ref)
        ws_got.copy_(nxt_got)


@pytest.mark.parametrize("cluster", ["0", "1"])
def test_noalloc_long_units(monkeypatch, cluster):
    """9000-slot units: clusters of 16, or (clusters off) the last-CTA merge
    with the split finish's scoring kernel, from the static scratch."""
    monkeypatch.setenv("LF_CLUSTER", cluster)
    rng = np.random.default_rng(12)
    case = _pins.rand_case(rng, 2, 8, 2, 128, 9000, p_masked=0.2, max_age=20000)
    W, scale = 8, 0.088
    p = lf.step_plan(2, 8, 2, 128, 9000)
    assert p["split"] == (cluster == "0")
    dc = {kk: to_dev(vv) for kk, vv in case.items()}
    ref_mask = dc["mask"].clone()
    ref_k, ref_v = dc["k_cache"].clone(), dc["v_cache"].clone()
    out_ref = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    out_got = torch.empty_like(out_ref)
    nxt_ref = torch.empty((2, 2), dtype=torch.int32, device="cuda")
    nxt_got = torch.empty_like(nxt_ref)
    lf.decode_step(dc["q"], ref_k, ref_v, ref_mask, dc["new_k"], dc["new_v"], dc["write_slot"],
                   out_ref, nxt_ref, W, scale)
    lf.decode_step_noalloc(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                           dc["new_v"], dc["write_slot"], out_got, nxt_got, W, scale)
    torch.cuda.synchronize()
    assert torch.equal(out_got, out_ref) and torch.equal(nxt_got, nxt_ref)
    assert torch.equal(dc["mask"], ref_mask)
    assert torch.equal(dc["k_cache"], ref_k) and torch.equal(dc["v_cache"], ref_v)


def test_noalloc_refuses_a_shape_whose_scratch_does_not_fit():
    # One sequence, 8 KV heads x 4 query heads, 2^17 slots: the per-slot score
    # terms alone need 16 MiB. The buffers are real, so nothing could fault
    # even if the size check were missing.
    B, Hq, Hkv, d, S = 1, 32, 8, 128, 1 << 17
    lib = lf.load_library()
    q = torch.zeros(B, Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, Hkv, S, d, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    mask = torch.zeros(B, Hkv, S, dtype=torch.int32, device="cuda")
    nk = torch.zeros(B, Hkv, d, dtype=torch.bfloat16, device="cuda")
    nv = torch.zeros_like(nk)
    ws = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    nxt = torch.empty_like(ws)
    rc = lib.lf_decode_step_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), mask.data_ptr(), nk.data_ptr(), nv.data_ptr(),
        ws.data_ptr(), out.data_ptr(), nxt.data_ptr(), B, Hq, Hkv, d, S, 0,
        ctypes.c_float(0.088), torch.cuda.current_stream().cuda_stream)
    assert rc == lf.LF_ERR_UNSUPPORTED
    assert "static scratch" in lib.lf_last_error().decode()


def test_noalloc_matches_the_oracle_step_after_step():
    """Six steps of four 3200-slot Qwen3 sequences through the static scratch,
    each compared with the oracle on every unit: output, next_slot, and the
    cache and mask bits. Both sides write the oracle's chosen slot."""
    wl = WORKLOADS["qwen3_8b_b128_s3200"].with_batch(4)
    st = initial_state(wl)
    host = {kk: st[kk] for kk in ("k_cache", "v_cache", "mask")}
    dev = _state(st)
    out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty((wl.B, wl.Hkv), dtype=torch.int32, device="cuda")
    ws = np.full((wl.B, wl.Hkv), -1, dtype=np.int32)
    lf.device_errors(clear=True)
    for t in range(6):
        inp = step_inputs(wl, t)
        lf.decode_step_noalloc(to_dev(inp["q"]), dev["k"], dev["v"], dev["mask"],
                               to_dev(inp["new_k"]), to_dev(inp["new_v"]), to_dev(ws), out, nxt,
                               wl.W, wl.scale)
        torch.cuda.synchronize()
        ora = oracle_step(host, inp["q"], inp["new_k"], inp["new_v"], ws, wl.W, wl.scale)
        gpu = {"out": out.float().cpu().numpy().astype(np.float64),
               "next_slot": nxt.cpu().numpy()}
        assert np.array_equal(dev["mask"].cpu().numpy(), host["mask"]), f"step {t}: mask"
        assert np.array_equal(to_host_bits(dev["k"]), host["k_cache"]), f"step {t}: k_cache"
        assert np.array_equal(to_host_bits(dev["v"]), host["v_cache"]), f"step {t}: v_cache"
        for u in range(wl.units):
            b, kvh = divmod(u, wl.Hkv)
            compare_unit(gpu, ora, b, kvh, wl.g, host["mask"], wl.W, check_scores=False,
                         where=f"noalloc step {t}")
        ws = ora["next_slot"].astype(np.int32).copy()
    assert lf.device_errors(clear=True) == 0


def test_noalloc_reports_an_ignored_write_slot():
    """An out-of-range write slot is ignored (the rest of the step is
    correct) and its bit reaches lf_device_errors; clearing it leaves the word
    at zero for the next call."""
    rng = np.random.default_rng(41)
    case = _pins.rand_case(rng, 2, 8, 2, 128, 500, p_masked=0.1, max_age=2000)
    case["write_slot"][1, 0] = 500 + 7
    lf.device_errors(clear=True)
    dc = {kk: to_dev(vv) for kk, vv in case.items()}
    out = torch.empty((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty((2, 2), dtype=torch.int32, device="cuda")
    lf.decode_step_noalloc(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                           dc["new_v"], dc["write_slot"], out, nxt, 8, 0.088)
    flags = lf.device_errors(clear=True)
    assert flags == lf.LF_DEVERR_BAD_WRITE_SLOT
    host = {kk: np.array(case[kk], copy=True) for kk in ("k_cache", "v_cache", "mask")}
    ws = case["write_slot"].copy()
    ws[1, 0] = -1  # what the kernel does with it: no write, nothing ages
    ora = oracle_step(host, case["q"], case["new_k"], case["new_v"], ws, 8, 0.088)
    assert np.array_equal(dc["mask"].cpu().numpy(), host["mask"])
    gpu = {"out": out.float().cpu().numpy().astype(np.float64), "next_slot": nxt.cpu().numpy()}
    for b in range(2):
        for h in range(2):
            compare_unit(gpu, ora, b, h, 4, host["mask"], 8, check_scores=False, where="bad slot")
    assert lf.device_errors(clear=True) == 0


def test_noalloc_reports_a_wait_timeout(monkeypatch):
    """With the pipeline waits cut to 1 ns (LF_WAIT_LIMIT_NS, a diagnostic),
    the waits give up before the copies land: the bit must reach
    lf_device_errors, and the next call with the normal limit must be right."""
    rng = np.random.default_rng(43)
    case = _pins.rand_case(rng, 4, 32, 8, 128, 2000, p_masked=0.1, max_age=5000)
    lf.device_errors(clear=True)
    monkeypatch.setenv("LF_WAIT_LIMIT_NS", "1")
    dc = {kk: to_dev(vv) for kk, vv in case.items()}
    out = torch.empty((4, 32, 128), dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty((4, 8), dtype=torch.int32, device="cuda")
    lf.decode_step_noalloc(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                           dc["new_v"], dc["write_slot"], out, nxt, 16, 0.088)
    flags = lf.device_errors(clear=True)
    assert flags & lf.LF_DEVERR_WAIT_TIMEOUT
    monkeypatch.delenv("LF_WAIT_LIMIT_NS")
    dc = {kk: to_dev(vv) for kk, vv in case.items()}
    lf.decode_step_noalloc(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                           dc["new_v"], dc["write_slot"], out, nxt, 16, 0.088)
    torch.cuda.synchronize()
    host = {kk: np.array(case[kk], copy=True) for kk in ("k_cache", "v_cache", "mask")}
    ora = oracle_step(host, case["q"], case["new_k"], case["new_v"], case["write_slot"], 16,
                      0.088)
    assert np.array_equal(dc["mask"].cpu().numpy(), host["mask"])
    gpu = {"out": out.float().cpu().numpy().astype(np.float64), "next_slot": nxt.cpu().numpy()}
    for b in range(4):
        for h in range(8):
            compare_unit(gpu, ora, b, h, 4, host["mask"], 16, check_scores=False,
                         where="after a timed-out call")
    assert lf.device_errors(clear=True) == 0
