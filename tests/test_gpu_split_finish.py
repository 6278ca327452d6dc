"""The split finish: for top-1 steps over long units the decode-step kernel
stops after the chunk merge and a second kernel scores every chunk in
parallel (LF_SPLIT=1 forces it on every top-1 step without clusters, =0
keeps the scan in the last CTA). On grids of many waves the scoring kernel
takes only the later units, and the first ones still scan in their last CTA
(LF_SPLIT_TAIL sets how many units the scoring kernel takes).

Both finishes do the same arithmetic in the same order, so they must agree
bit for bit: output, chosen slot, every score, caches and mask, for every
entry point that takes the top-1 path and every selection flag. Parity of
the split finish against the oracle runs in the shared parity suites (the
full-size 16K-slot workload takes it by default) and here on the small
shapes and degenerate units, element by element.
"""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
from decode_kv_cache_step_gb300.workloads import WORKLOADS, initial_state, step_inputs

import _pins
from _gpu import compare_unit, to_dev

pytestmark = pytest.mark.gpu


def _step(case, W, scale, entry, flags, monkeypatch, split):
    monkeypatch.setenv("LF_CLUSTER", "0")
    monkeypatch.setenv("LF_SPLIT", split)
    dc = {k: to_dev(v) for k, v in case.items()}
    B, Hq, d = case["q"].shape
    Hkv, S = case["k_cache"].shape[1], case["k_cache"].shape[2]
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.full((B, Hkv), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((B, Hkv, S), -5.0, dtype=torch.float32, device="cuda")
    args = (dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"], dc["new_v"],
            dc["write_slot"], out)
    if entry == "step":
        lf.decode_step(*args, nxt, W, scale)
    elif entry == "scores":
        lf.decode_step_scores(*args, nxt, scores, W, scale)
    else:
        nx3 = nxt.view(B, Hkv, 1)
        lf.decode_step_ex(*args, nx3, W, scale, k=1, flags=flags,
                          scores=scores if entry == "ex_scores" else None)
    torch.cuda.synchronize()
    assert lf.device_errors() == 0
    return {"out": out, "next": nxt, "scores": scores, "mask": dc["mask"], "k": dc["k_cache"],
            "v": dc["v_cache"]}


@pytest.mark.parametrize("entry,flags", [("step", 0), ("scores", 0), ("ex", 1), ("ex", 2),
                                         ("ex", 3), ("ex_scores", 3)])
@pytest.mark.parametrize("d,g,S,p_masked", [(64, 1, 77, 0.2), (128, 4, 1000, 0.3),
                                            (128, 8, 4100, 0.1), (64, 2, 5000, 0.6),
                                            (128, 4, 16384, 0.05)])
def test_split_finish_is_bit_identical(monkeypatch, entry, flags, d, g, S, p_masked):
    rng = np.random.default_rng(7 * S + g + d)
    Hkv = 2
    case = _pins.rand_case(rng, 2, Hkv * g, Hkv, d, S, p_masked=p_masked, max_age=3 * S,
                           ws_mode="any")
    W = min(16, S // 4)
    a = _step(case, W, 0.088, entry, flags, monkeypatch, "0")
    b = _step(case, W, 0.088, entry, flags, monkeypatch, "1")
    for key in ("out", "next", "mask", "k", "v"):
        assert torch.equal(a[key], b[key]), key
    if entry in ("scores", "ex_scores"):
        assert torch.equal(a["scores"], b["scores"])


@pytest.mark.parametrize("parts", ["1", "2", "3", "64"])
@pytest.mark.parametrize("entry,flags", [("scores", 0), ("ex", 3), ("step", 0)])
def test_score_parts_do_not_change_results(monkeypatch, parts, entry, flags):
    """The scoring kernel splits each unit's chunks among `parts` CTAs (one
    CTA: no atomics; several: atomic maximum and the last CTA's read). Ragged
    liveness leaves whole chunks without a live slot."""
    monkeypatch.setenv("LF_CHUNK_TILES", "2")
    rng = np.random.default_rng(int(parts) + len(entry))
    Hkv, g, d, S = 2, 4, 128, 3000
    case = _pins.rand_case(rng, 3, Hkv * g, Hkv, d, S, p_masked=0.1, max_age=3 * S,
                           ws_mode="any")
    case["mask"][0, 0, 700:] = -1       # ragged: chunks past slot 768 hold no live slot
    case["mask"][1, 1, :2000] = -1
    a = _step(case, 16, 0.088, entry, flags, monkeypatch, "0")
    monkeypatch.setenv("LF_SCORE_PARTS", parts)
    b = _step(case, 16, 0.088, entry, flags, monkeypatch, "1")
    for key in ("out", "next", "mask", "k", "v"):
        assert torch.equal(a[key], b[key]), key
    if entry == "scores":
        assert torch.equal(a["scores"], b["scores"])


def test_split_finish_many_units(monkeypatch):
    """More units than resident CTAs: one scoring CTA per unit."""
    monkeypatch.setenv("LF_CHUNK_TILES", "2")
    rng = np.random.default_rng(99)
    case = _pins.rand_case(rng, 160, 16, 8, 64, 1000, p_masked=0.2, max_age=3000, ws_mode="any")
    a = _step(case, 8, 0.125, "scores", 0, monkeypatch, "0")
    b = _step(case, 8, 0.125, "scores", 0, monkeypatch, "1")
    for key in ("out", "next", "mask", "scores"):
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("S", [1, 63, 65, 1000, 4500])
def test_split_finish_matches_oracle(monkeypatch, d, g, S):
    monkeypatch.setenv("LF_CLUSTER", "0")
    monkeypatch.setenv("LF_SPLIT", "1")
    rng = np.random.default_rng(3000 + 100 * d + 10 * g + S)
    Hkv = 2
    case = _pins.rand_case(rng, 2, Hkv * g, Hkv, d, S, p_masked=0.2, max_age=3 * S + 5,
                           ws_mode="any")
    W = min(4, S // 3)
    scale = float(np.float32(1 / np.sqrt(d)))
    gpu = _step(case, W, scale, "scores", 0, monkeypatch, "1")
    ora = _pins.run(__import__("oracle").decode_step, case, W, scale, want_scores=True)
    res = {"out": gpu["out"].float().cpu().numpy().astype(np.float64),
           "next_slot": gpu["next"].cpu().numpy(), "scores": gpu["scores"].cpu().numpy()}
    assert np.array_equal(gpu["mask"].cpu().numpy(), ora["state"]["mask"])
    for b in range(2):
        for h in range(Hkv):
            compare_unit(res, ora, b, h, g, ora["state"]["mask"], W, where=f"d={d} g={g} S={S}")


def test_split_finish_degenerate_units(monkeypatch):
    """Empty units, units with nothing old enough, all-equal scores (ties go
    to the lowest slot) and a unit whose only live slot is the written one."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, d, S = 4, 8, 2, 128, 4160
    case = _pins.rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.1, max_age=1000)
    case["mask"][0, 0] = -1                 # empty, no write: next -1
    case["write_slot"][0, 0] = -1
    case["mask"][0, 1] = 0                  # nothing reaches W after ageing: next -1
    case["mask"][1, 0] = -1                 # only the written slot is live
    case["write_slot"][1, 0] = 4100
    case["v_cache"][2, 1] = 0               # every score 0: lowest eligible slot
    case["mask"][2, 1] = 500
    case["write_slot"][2, 1] = 3
    W = 8
    a = _step(case, W, 0.088, "scores", 0, monkeypatch, "0")
    b = _step(case, W, 0.088, "scores", 0, monkeypatch, "1")
    for key in ("out", "next", "mask", "scores"):
        assert torch.equal(a[key], b[key]), key
    nxt = b["next"].cpu().numpy()
    assert nxt[0, 0] == -1 and nxt[0, 1] == -1 and nxt[1, 0] == -1
    assert nxt[2, 1] == 0


def test_split_finish_full_workload_steps(monkeypatch):
    """Several chained steps of the 16K-slot workload (which takes the split
    finish by default) against the same steps with the scan in the last CTA."""
    wl = WORKLOADS["long_b32_s16384_ragged"].with_batch(4)
    st = initial_state(wl)
    res = {}
    for split in ("0", "1"):
        monkeypatch.setenv("LF_SPLIT", split)
        k, v, mask = to_dev(st["k_cache"]), to_dev(st["v_cache"]), to_dev(st["mask"])
        out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
        ws = torch.full((wl.B, wl.Hkv), -1, dtype=torch.int32, device="cuda")
        outs, slots = [], []
        for t in range(4):
            p = {kk: to_dev(vv) for kk, vv in step_inputs(wl, t).items()}
            nxt = torch.empty((wl.B, wl.Hkv), dtype=torch.int32, device="cuda")
            lf.decode_step(p["q"], k, v, mask, p["new_k"], p["new_v"], ws, out, nxt, wl.W, wl.scale)
            outs.append(out.clone())
            slots.append(nxt)
            ws = nxt
        torch.cuda.synchronize()
        res[split] = (outs, slots, mask, k)
    a, b = res["0"], res["1"]
    assert all(torch.equal(x, y) for x, y in zip(a[0], b[0]))
    assert all(torch.equal(x, y) for x, y in zip(a[1], b[1]))
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])
    assert lf.device_errors() == 0


@pytest.mark.parametrize("tail", ["1", "37", "80", "159", "160"])
@pytest.mark.parametrize("entry,flags", [("scores", 0), ("ex", 3), ("step", 0)])
def test_hybrid_finish_is_bit_identical(monkeypatch, tail, entry, flags):
    """A split finish whose scoring kernel takes only the last `tail` units
    (LF_SPLIT_TAIL; the others scan in their last CTA) gives the same bits as
    the scan in the last CTA for every unit."""
    monkeypatch.setenv("LF_CHUNK_TILES", "2")
    rng = np.random.default_rng(500 + int(tail) + len(entry))
    case = _pins.rand_case(rng, 20, 32, 8, 64, 1000, p_masked=0.2, max_age=3000, ws_mode="any")
    case["mask"][3, 2, 300:] = -1      # ragged: chunks without a live slot
    a = _step(case, 8, 0.125, entry, flags, monkeypatch, "0")
    monkeypatch.setenv("LF_SPLIT_TAIL", tail)
    b = _step(case, 8, 0.125, entry, flags, monkeypatch, "1")
    for key in ("out", "next", "mask", "k", "v"):
        assert torch.equal(a[key], b[key]), key
    if entry == "scores":
        assert torch.equal(a["scores"], b["scores"])


def test_default_hybrid_finish_at_full_size(monkeypatch):
    """The full 16K-slot workload (about nine waves) takes the split finish
    with its first 3/8 units scanning in their last CTA: the same bits as
    every unit split and as every unit scanning in its last CTA."""
    wl = WORKLOADS["long_b32_s16384_ragged"]
    st = initial_state(wl)
    inp = {k: to_dev(v) for k, v in step_inputs(wl, 2).items()}
    ws = to_dev(np.random.default_rng(2).integers(0, wl.S, size=(wl.B, wl.Hkv)).astype(np.int32))
    units = wl.B * wl.Hkv
    for k in ("LF_SPLIT_TAIL", "LF_SPLIT"):
        monkeypatch.delenv(k, raising=False)
    assert lf.step_plan(wl.B, wl.Hq, wl.Hkv, wl.d, wl.S)["split"]
    res = {}
    for name, env in (("default", {}), ("all_split", {"LF_SPLIT_TAIL": str(units)}),
                      ("no_split", {"LF_SPLIT": "0"})):
        for k in ("LF_SPLIT_TAIL", "LF_SPLIT"):
            monkeypatch.delenv(k, raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        mask = to_dev(st["mask"])
        k_c, v_c = to_dev(st["k_cache"]), to_dev(st["v_cache"])
        out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
        nxt = torch.empty((wl.B, wl.Hkv), dtype=torch.int32, device="cuda")
        lf.decode_step(inp["q"], k_c, v_c, mask, inp["new_k"], inp["new_v"], ws, out, nxt,
                       wl.W, wl.scale)
        torch.cuda.synchronize()
        res[name] = (out, nxt, mask)
        del k_c, v_c
    for name in ("all_split", "no_split"):
        for x, y in zip(res["default"], res[name]):
            assert torch.equal(x, y), name
    assert lf.device_errors() == 0
