"""Prepared steps (lf_step_prepare / lf_step_run): a token loop through two
handles per layer (write and next slot buffers swapped) gives, step after
step, the same bits as the plain entry point, whether the per-step buffers
are device memory, pinned host memory (used in place), pageable host memory
(staged) or a mix; on the split-finish and cluster plans; captured in a CUDA
graph; with the handle's own error word."""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
from decode_kv_cache_step_gb300.workloads import WORKLOADS, initial_state, step_inputs

import _pins
import oracle
from _gpu import OUT_ATOL, to_dev

pytestmark = pytest.mark.gpu


def _buf(x, where):
    t = torch.from_numpy((x.view(np.int16) if x.dtype == np.uint16 else x).copy())
    if where == "device":
        t = t.cuda()
    elif where == "pinned":
        t = t.pin_memory()
    return t.view(torch.bfloat16) if x.dtype == np.uint16 else t


def _loop(wl, places, steps):
    st = initial_state(wl)
    # Reference: the plain device entry point on its own copy of the state.
    k, v, m = to_dev(st["k_cache"]), to_dev(st["v_cache"]), to_dev(st["mask"])
    k2, v2, m2 = k.clone(), v.clone(), m.clone()
    out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    slots = [torch.full((wl.B, wl.Hkv), -1, dtype=torch.int32, device="cuda"),
             torch.empty((wl.B, wl.Hkv), dtype=torch.int32, device="cuda")]
    # Prepared: fixed input buffers that each step overwrites, two handles.
    inp0 = step_inputs(wl, 0)
    q_b = _buf(inp0["q"], places[0])
    nk_b = _buf(inp0["new_k"], places[1])
    nv_b = _buf(inp0["new_v"], places[2])
    s_b = [_buf(np.full((wl.B, wl.Hkv), -1, dtype=np.int32), places[3]),
           _buf(np.zeros((wl.B, wl.Hkv), dtype=np.int32), places[3])]
    o_b = _buf(np.zeros((wl.B, wl.Hq, wl.d), dtype=np.uint16), places[4])
    hs = [lf.PreparedStep(q_b, k2, v2, m2, nk_b, nv_b, s_b[p], o_b, s_b[1 - p], wl.W, wl.scale)
          for p in range(2)]
    try:
        for t in range(steps):
            inp = step_inputs(wl, t)
            dq, dnk, dnv = to_dev(inp["q"]), to_dev(inp["new_k"]), to_dev(inp["new_v"])
            lf.decode_step(dq, k, v, m, dnk, dnv, slots[t % 2], out, slots[(t + 1) % 2], wl.W,
                           wl.scale)
            torch.cuda.synchronize()
            q_b.copy_(_buf(inp["q"], "cpu")), nk_b.copy_(_buf(inp["new_k"], "cpu"))
            nv_b.copy_(_buf(inp["new_v"], "cpu"))
            hs[t % 2].run()
            torch.cuda.synchronize()
            assert torch.equal(o_b.cpu(), out.cpu()), f"step {t}: out"
            assert torch.equal(s_b[(t + 1) % 2].cpu(), slots[(t + 1) % 2].cpu()), f"step {t}: next"
            assert torch.equal(m2, m) and torch.equal(k2, k) and torch.equal(v2, v), f"step {t}"
        assert all(h.errors() == 0 for h in hs)
    finally:
        for h in hs:
            h.close()
    return hs


PLACES = {"device": ["device"] * 5, "pinned": ["pinned"] * 5, "pageable": ["cpu"] * 5,
          "mixed": ["pinned", "cpu", "device", "pinned", "cpu"]}


@pytest.mark.parametrize("io", list(PLACES))
@pytest.mark.parametrize("name", ["tiny_b2_s256", "qwen3_8b_b1_s2400"])
def test_prepared_loop_matches_plain_entry(name, io):
    wl = WORKLOADS[name]
    _loop(wl, PLACES[io], steps=12)


@pytest.mark.parametrize("name,batch", [("long_b32_s16384_ragged", 2),      # clusters of 16
                                        ("long_b32_s16384_ragged", 8),      # split finish
                                        ("long_b32_s16384_ragged", 32),     # split finish, first 3/8 of the units in-kernel
                                        ("llama8b_b256_s2400_ragged", 8),   # clusters
                                        ("qwen3_8b_b128_s3200", 64)])       # last-CTA merge
def test_prepared_plans(name, batch):
    wl = WORKLOADS[name].with_batch(batch)
    _loop(wl, PLACES["pinned"], steps=3)


def test_prepared_against_oracle():
    """One prepared step on a random case against the fp64 oracle."""
    rng = np.random.default_rng(31)
    case = _pins.rand_case(rng, 2, 8, 2, 128, 700, p_masked=0.3, max_age=2000)
    W, scale = 16, 0.088
    dc = {kk: to_dev(vv) for kk, vv in case.items()}
    B, Hq, d = case["q"].shape
    Hkv = case["k_cache"].shape[1]
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16).pin_memory()
    nxt = torch.full((B, Hkv), -9, dtype=torch.int32).pin_memory()
    with lf.PreparedStep(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                         dc["new_v"], dc["write_slot"], out, nxt, W, scale) as h:
        h.run()
        torch.cuda.synchronize()
        assert h.errors() == 0
    ora = _pins.run(oracle.decode_step, case, W, scale, want_scores=True)
    assert np.max(np.abs(out.float().numpy() - ora["out"])) <= OUT_ATOL
    assert np.array_equal(dc["mask"].cpu().numpy(), ora["state"]["mask"])
    for b in range(B):
        for h in range(Hkv):
            s = ora["scores"][b, h]
            elig = (ora["state"]["mask"][b, h] >= W) & np.isfinite(s)
            j = int(nxt[b, h])
            assert elig[j] and s[j] <= s[elig].min() * (1 + 1e-3), (b, h, j)


def test_prepared_graph_replay_and_errors():
    wl = WORKLOADS["tiny_b2_s256"]
    st = initial_state(wl)
    inp = step_inputs(wl, 0)
    k, v, m = to_dev(st["k_cache"]), to_dev(st["v_cache"]), to_dev(st["mask"])
    q, nk, nv = to_dev(inp["q"]), to_dev(inp["new_k"]), to_dev(inp["new_v"])
    ws = torch.full((wl.B, wl.Hkv), wl.S + 5, dtype=torch.int32, device="cuda")  # out of range
    out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty((wl.B, wl.Hkv), dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        h = lf.PreparedStep(q, k, v, m, nk, nv, ws, out, nxt, wl.W, wl.scale, stream=s)
    h.run()
    s.synchronize()
    assert h.errors(clear=True) == lf.LF_DEVERR_BAD_WRITE_SLOT
    assert h.errors() == 0
    # The step is idempotent here (the write is ignored; ages grow), so
    # compare a graph replay with an eager run from the same state.
    m0 = m.clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        h.run()
    torch.cuda.synchronize()
    m.copy_(m0)
    torch.cuda.synchronize()
    h.run()
    s.synchronize()
    e_out, e_next, e_mask = out.clone(), nxt.clone(), m.clone()
    m.copy_(m0)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, e_out) and torch.equal(nxt, e_next) and torch.equal(m, e_mask)
    h.close()
    h.close()  # idempotent


def test_prepared_argument_errors():
    wl = WORKLOADS["tiny_b2_s256"]
    st = initial_state(wl)
    inp = step_inputs(wl, 0)
    k, v, m = to_dev(st["k_cache"]), to_dev(st["v_cache"]), to_dev(st["mask"])
    q, nk, nv = to_dev(inp["q"]), to_dev(inp["new_k"]), to_dev(inp["new_v"])
    ws = torch.full((wl.B, wl.Hkv), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty((wl.B, wl.Hkv), dtype=torch.int32, device="cuda")
    with pytest.raises(lf.LFError):
        lf.PreparedStep(q, k, v, m, nk, nv, ws, out, nxt, -1, wl.scale)      # W < 0
    with pytest.raises(lf.LFError):
        lf.PreparedStep(q, k, v, m, nk, nv, ws, out, nxt, wl.W, float("nan"))
    with pytest.raises((TypeError, ValueError)):
        lf.PreparedStep(q, k, v, m, nk, nv, ws.float(), out, nxt, wl.W, wl.scale)
