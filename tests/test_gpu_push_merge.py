"""The cluster merge by pushes on every shape it takes: each head dim and
group size, both TMA rings, clusters of 1 to 16 CTAs (including splits in
which some CTAs own no part of the output row), a ragged last tile, the
fused step (two steps, the second writing the slot the first chose) and
attention alone, each against the fp64 oracle. The plan each case runs is
checked first, so that a change of plan cannot silently skip a case."""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf

import _pins
from _gpu import DevState, compare_unit, oracle_step, to_dev, to_host_bits, OUT_ATOL

pytestmark = pytest.mark.gpu

CHUNKS = [1, 2, 3, 5, 7, 12, 16]


def _case(d, g, nchunk, seed):
    # 2 tiles per chunk, the last one ragged (17 slots): S = (2 nchunk - 1) * 64 + 17
    S = (2 * nchunk - 1) * 64 + 17
    rng = np.random.default_rng(seed)
    case = _pins.rand_case(rng, 1, 2 * g, 2, d, S, p_masked=0.2, max_age=3 * S, ws_mode="any")
    return case, S


def _force(monkeypatch, deep):
    monkeypatch.setenv("LF_CLUSTER", "1")
    monkeypatch.setenv("LF_CHUNK_TILES", "2")
    monkeypatch.setenv("LF_DEEP", "1" if deep else "0")


@pytest.mark.parametrize("deep", [False, True])
@pytest.mark.parametrize("nchunk", CHUNKS)
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_push_merge_step(monkeypatch, d, g, nchunk, deep):
    _force(monkeypatch, deep)
    case, S = _case(d, g, nchunk, 1000 * d + 100 * g + 2 * nchunk + deep)
    B, Hkv = 1, 2
    Hq = Hkv * g
    p = lf.step_plan(B, Hq, Hkv, d, S)
    assert p["cluster"] and p["nchunk"] == nchunk and p["chunk_tiles"] == 2, p
    assert p["stages"] == (6 if deep else 2), p
    W = 5
    scale = float(np.float32(1 / np.sqrt(d)))
    where = f"d={d} g={g} nchunk={nchunk} deep={deep}"
    dev = DevState(case["k_cache"], case["v_cache"], case["mask"], Hq)
    host = {kk: np.array(case[kk], copy=True) for kk in ("k_cache", "v_cache", "mask")}
    ws = case["write_slot"]
    for step in range(2):
        gpu = dev.step(case["q"], case["new_k"], case["new_v"], ws, W, scale, scores=True)
        ora = oracle_step(host, case["q"], case["new_k"], case["new_v"], ws, W, scale)
        assert np.array_equal(dev.mask.cpu().numpy(), host["mask"]), where
        assert np.array_equal(to_host_bits(dev.k), host["k_cache"]), where
        assert np.array_equal(to_host_bits(dev.v), host["v_cache"]), where
        for h in range(Hkv):
            compare_unit(gpu, ora, 0, h, g, host["mask"], W, check_scores=True,
                         where=f"{where} step {step}")
        ws = gpu["next_slot"].astype(np.int32)
    assert lf.device_errors() == 0


@pytest.mark.parametrize("deep", [False, True])
@pytest.mark.parametrize("nchunk", [1, 3, 12, 16])
@pytest.mark.parametrize("g", [1, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_push_merge_attention_only(monkeypatch, d, g, nchunk, deep):
    _force(monkeypatch, deep)
    case, S = _case(d, g, nchunk, 7 + 1000 * d + 100 * g + 2 * nchunk + deep)
    scale = float(np.float32(1 / np.sqrt(d)))
    dc = {k: to_dev(v) for k, v in case.items()}
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device="cuda")
    lf.decode_attention(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                        dc["new_v"], dc["write_slot"], out, scale)
    torch.cuda.synchronize()
    ora = _pins.run(__import__("oracle").decode_step, case, 0, scale, attention_only=True)
    assert np.max(np.abs(out.float().cpu().numpy() - ora["out"])) <= OUT_ATOL
    assert np.array_equal(dc["mask"].cpu().numpy(), ora["state"]["mask"])
    assert np.array_equal(to_host_bits(dc["k_cache"]), ora["state"]["k_cache"])
    assert lf.device_errors() == 0
