"""The last CTA's top-1 score scan over live tiles only.

Each chunk CTA publishes which of its 64-slot tiles hold a live slot; when a
unit has a dead tile, the unit's last CTA scans only the slots of the live
tiles (top-1, no score output, no fill-empty-first). These cases put the
live region's end on and around tile boundaries, punch holes of whole
masked tiles into units, write into a dead tile (which makes it live), and
vary the chunking, against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
import oracle

import _pins
from _gpu import OUT_ATOL, to_dev
from test_gpu_next import _ranked, compare_topk

pytestmark = pytest.mark.gpu


def _case(seed, S, patterns, writes):
    B, Hkv, g, d = len(patterns) // 2, 2, 4, 128
    rng = np.random.default_rng(seed)
    case = _pins.rand_case(rng, B, Hkv * g, Hkv, d, S, p_masked=0.0, max_age=4 * S)
    for u, pat in enumerate(patterns):
        b, h = divmod(u, Hkv)
        live = np.zeros(S, dtype=bool)
        if pat[0] == "prefix":
            live[:pat[1]] = True
        else:  # "holes": the listed tiles are entirely masked
            live[:] = True
            for t in pat[1]:
                live[t * 64:(t + 1) * 64] = False
        ages = case["mask"][b, h]
        ages[~live] = -1
        case["mask"][b, h] = ages
        case["write_slot"][b, h] = writes[u]
    return case


PATTERNS = [("prefix", 1), ("prefix", 63), ("prefix", 64), ("prefix", 65), ("prefix", 700),
            ("holes", (1, 2, 5, 6, 7, 8, 9)), ("holes", (0,)), ("holes", (14, 15)),
            ("prefix", 1000), ("holes", tuple(range(1, 15)))]
WRITES = [-1, 62, 64, 200, 10, 100, 5, 999, 500, 70]   # 64, 200, 100, 999, 70: into dead tiles


@pytest.mark.parametrize("entry", ["step", "ex_evict"])
@pytest.mark.parametrize("chunk_tiles", [None, "1", "3", "5", "32"])
def test_live_tile_scan_matches_oracle(monkeypatch, chunk_tiles, entry):
    monkeypatch.setenv("LF_CLUSTER", "0")
    monkeypatch.setenv("LF_SPLIT", "0")
    if chunk_tiles:
        monkeypatch.setenv("LF_CHUNK_TILES", chunk_tiles)
    S, W, scale = 1000, 8, 0.088
    case = _case(17, S, PATTERNS, WRITES)
    dc = {k: to_dev(v) for k, v in case.items()}
    B, Hq, d = case["q"].shape
    Hkv = case["k_cache"].shape[1]
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.full((B, Hkv), -7, dtype=torch.int32, device="cuda")
    args = (dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"], dc["new_v"],
            dc["write_slot"], out)
    if entry == "step":
        lf.decode_step(*args, nxt, W, scale)
    else:
        lf.decode_step_ex(*args, nxt.view(B, Hkv, 1), W, scale, k=1,
                          flags=lf.LF_STEP_MASK_EVICTED)
    torch.cuda.synchronize()
    assert lf.device_errors() == 0
    ora = _pins.run(oracle.decode_step, case, W, scale, want_scores=True)
    assert np.max(np.abs(out.float().cpu().numpy() - ora["out"])) <= OUT_ATOL
    ages = ora["state"]["mask"]
    got = nxt.cpu().numpy()
    mask_gpu = dc["mask"].cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            ranked = _ranked(ora["scores"][b, h], ages[b, h], W, False)
            compare_topk(got[b, h:h + 1], ranked, 1, f"unit ({b},{h}) chunk_tiles={chunk_tiles}")
            want = ages[b, h].copy()
            if entry == "ex_evict" and got[b, h] >= 0:
                want[got[b, h]] = -1
            assert np.array_equal(mask_gpu[b, h], want), f"unit ({b},{h}) mask"


def _run_bits(case, W, scale, scores=False):
    dc = {k: to_dev(v) for k, v in case.items()}
    B, Hq, d = case["q"].shape
    Hkv, S = case["k_cache"].shape[1], case["k_cache"].shape[2]
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.full((B, Hkv), -7, dtype=torch.int32, device="cuda")
    sc = torch.empty((B, Hkv, S), dtype=torch.float32, device="cuda") if scores else None
    args = (dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"], dc["new_v"],
            dc["write_slot"], out, nxt)
    if scores:
        lf.decode_step_scores(*args, sc, W, scale)
    else:
        lf.decode_step(*args, W, scale)
    torch.cuda.synchronize()
    assert lf.device_errors() == 0
    res = [out.view(torch.int16).cpu(), nxt.cpu(), dc["mask"].cpu(),
           dc["k_cache"].view(torch.int16).cpu(), dc["v_cache"].view(torch.int16).cpu()]
    if scores:
        res.append(sc.cpu())
    return res


@pytest.mark.parametrize("plan", ["last_cta", "cluster", "split", "deep"])
@pytest.mark.parametrize("scores", [False, True])
def test_speculative_first_tiles_change_no_bit(monkeypatch, plan, scores):
    """The first wave's CTAs issue their chunk's first tiles before the mask
    says which are live; a dead one is processed as fully masked. Ragged
    units with dead chunks, holes and writes into dead tiles give the same
    bits with speculation off (LF_SPEC=0), on every merge path."""
    env = {"last_cta": {"LF_CLUSTER": "0", "LF_SPLIT": "0"},
           "cluster": {"LF_CLUSTER": "1", "LF_DEEP": "0"},
           "split": {"LF_CLUSTER": "0", "LF_SPLIT": "1"},
           "deep": {"LF_CLUSTER": "1", "LF_DEEP": "1"}}[plan]
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    S, W, scale = 1000, 8, 0.088
    case = _case(23, S, PATTERNS, WRITES)
    on = _run_bits(case, W, scale, scores)
    monkeypatch.setenv("LF_SPEC", "0")
    off = _run_bits(case, W, scale, scores)
    for a, b in zip(on, off):
        assert torch.equal(a, b)
    ora = _pins.run(oracle.decode_step, case, W, scale, want_scores=True)
    assert np.max(np.abs(on[0].view(torch.bfloat16).float().numpy() - ora["out"])) <= OUT_ATOL
