"""GPU parity of the widened entry points against the fp64 oracle:
lf_decode_attention (attention alone, the overhead baseline), and
lf_decode_step_ex with k-at-once selection, fill-empty-first and
mask-evicted.

Top-k lists are compared the way next_slot is: every returned slot must be a
candidate, the i-th returned slot's oracle score must match the oracle's i-th
smallest within 1e-3 relative, and where the oracle's k-th and (k+1)-th
candidates are more than 1e-3 apart the two sets must be equal.
"""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
from decode_kv_cache_step_gb300.workloads import WORKLOADS, initial_state, step_inputs

import _pins
from _gpu import OUT_ATOL, SCORE_RTOL, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def _dev_case(case):
    return {k: to_dev(v) for k, v in case.items()}


def _ranked(ora_scores, ages, W, fill_first):
    """Oracle candidates of one unit in ascending (class, score, slot) order."""
    c = [(1, float(ora_scores[j]), j) for j in range(len(ages)) if ages[j] >= W]
    if fill_first:
        c += [(0, 0.0, j) for j in range(len(ages)) if ages[j] < 0]
    return sorted(c)


def compare_topk(got, ranked, k, where):
    g = [int(x) for x in got if x >= 0]
    assert all(x == -1 for x in got[len(g):]), f"{where}: -1 before the end of the list"
    want = ranked[:k]
    assert len(g) == len(want), f"{where}: {len(g)} slots returned, oracle {len(want)}"
    assert len(set(g)) == len(g), f"{where}: duplicate slots"
    key = {j: (cls, sc) for cls, sc, j in ranked}
    for i, x in enumerate(g):
        assert x in key, f"{where}: slot {x} is not a candidate"
        cls, sc = key[x]
        wcls, wsc, _ = want[i]
        assert cls == wcls, f"{where}: position {i} class {cls} vs {wcls}"
        assert abs(sc - wsc) <= SCORE_RTOL * abs(wsc) + 1e-30, f"{where}: position {i} score {sc} vs {wsc}"
    if len(ranked) > k:
        a, b = ranked[k - 1], ranked[k]
        clear = a[0] != b[0] or (b[1] - a[1]) > SCORE_RTOL * abs(a[1])
        if clear:
            assert set(g) == {j for _, _, j in want}, f"{where}: selected set differs"


def run_ex(case, W, scale, k, flags):
    B, Hkv, S, d = case["k_cache"].shape
    Hq = case["q"].shape[1]
    dc = _dev_case(case)
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty((B, Hkv, k), dtype=torch.int32, device="cuda")
    scores = torch.empty((B, Hkv, S), dtype=torch.float32, device="cuda")
    lf.decode_step_ex(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"], dc["new_v"],
                      dc["write_slot"], out, nxt, W, scale, k=k, flags=flags, scores=scores)
    torch.cuda.synchronize()
    return {"out": out.float().cpu().numpy().astype(np.float64), "next": nxt.cpu().numpy(),
            "scores": scores.cpu().numpy().astype(np.float64), "mask": dc["mask"].cpu().numpy(),
            "k": to_host_bits(dc["k_cache"]), "v": to_host_bits(dc["v_cache"])}


def check_ex(case, W, scale, k, flags, where):
    fill = bool(flags & lf.LF_STEP_FILL_EMPTY_FIRST)
    evict = bool(flags & lf.LF_STEP_MASK_EVICTED)
    gpu = run_ex(case, W, scale, k, flags)
    # The oracle without eviction gives the pre-eviction ages and the scores.
    ora = _pins.run(__import__("oracle").decode_step, case, W, scale, want_scores=True, topk=k,
                    fill_first=fill)
    ages = ora["state"]["mask"]
    B, Hkv = ages.shape[:2]
    assert np.max(np.abs(gpu["out"] - ora["out"])) <= OUT_ATOL, where
    assert np.array_equal(gpu["k"], ora["state"]["k_cache"]), where
    lst = ora["next_slot"] if k > 1 else ora["next_slot"][:, :, None]
    for b in range(B):
        for h in range(Hkv):
            ranked = _ranked(ora["scores"][b, h], ages[b, h], W, fill)
            compare_topk(gpu["next"][b, h], ranked, k, f"{where} unit ({b},{h})")
            want_mask = ages[b, h].copy()
            if evict:
                chosen = [int(x) for x in gpu["next"][b, h] if x >= 0]
                want_mask[chosen] = -1
            assert np.array_equal(gpu["mask"][b, h], want_mask), f"{where} unit ({b},{h}) mask"
    assert lf.device_errors() == 0
    return gpu, ora


@pytest.mark.parametrize("cluster,deep", [("1", "1"), ("1", "0"), ("0", "1")])
@pytest.mark.parametrize("d,g,S", [(64, 1, 100), (128, 4, 300), (128, 8, 1000), (64, 2, 65)])
def test_attention_only_matches_oracle(monkeypatch, d, g, S, cluster, deep):
    monkeypatch.setenv("LF_CLUSTER", cluster)
    monkeypatch.setenv("LF_DEEP", deep)
    rng = np.random.default_rng(d + g + S)
    case = _pins.rand_case(rng, 2, 2 * g, 2, d, S, p_masked=0.3, max_age=3 * S, ws_mode="any")
    dc = _dev_case(case)
    out = torch.empty(case["q"].shape, dtype=torch.bfloat16, device="cuda")
    scale = float(np.float32(1 / np.sqrt(d)))
    lf.decode_attention(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                        dc["new_v"], dc["write_slot"], out, scale)
    torch.cuda.synchronize()
    ora = _pins.run(__import__("oracle").decode_step, case, 0, scale, attention_only=True)
    err = np.max(np.abs(out.float().cpu().numpy() - ora["out"]))
    assert err <= OUT_ATOL
    assert np.array_equal(dc["mask"].cpu().numpy(), ora["state"]["mask"])
    assert np.array_equal(to_host_bits(dc["k_cache"]), ora["state"]["k_cache"])
    assert np.array_equal(to_host_bits(dc["v_cache"]), ora["state"]["v_cache"])


def test_attention_only_full_size_output_equals_fused_step_output():
    """Same kernel pipeline: the fused step and attention alone give the same
    output bits on the benchmark shape."""
    wl = WORKLOADS["qwen3_8b_b128_s3200"]
    st = initial_state(wl)
    inp = step_inputs(wl, 3)
    ws = np.random.default_rng(1).integers(0, wl.S, size=(wl.B, wl.Hkv)).astype(np.int32)
    case = {**{k: st[k] for k in ("k_cache", "v_cache", "mask")}, **inp, "write_slot": ws}
    a, b = _dev_case(case), _dev_case(case)
    out_a = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out_a)
    nxt = torch.empty((wl.B, wl.Hkv), dtype=torch.int32, device="cuda")
    lf.decode_step(a["q"], a["k_cache"], a["v_cache"], a["mask"], a["new_k"], a["new_v"],
                   a["write_slot"], out_a, nxt, wl.W, wl.scale)
    lf.decode_attention(b["q"], b["k_cache"], b["v_cache"], b["mask"], b["new_k"], b["new_v"],
                        b["write_slot"], out_b, wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(a["k_cache"], b["k_cache"])


@pytest.mark.parametrize("k", [2, 5, 16, 128, 1024])
def test_topk_matches_oracle(k):
    rng = np.random.default_rng(500 + k)
    case = _pins.rand_case(rng, 2, 8, 2, 128, 1500, p_masked=0.2, max_age=5000)
    check_ex(case, 16, 0.088, k, 0, f"k={k}")


@pytest.mark.parametrize("cluster,split,deep", [("1", "0", "1"), ("1", "0", "0"), ("0", "0", "1"),
                                                ("0", "1", "1")])
@pytest.mark.parametrize("k,flags", [(1, 1), (8, 1), (1, 2), (32, 2), (64, 3), (1, 3)])
def test_fill_first_and_mask_evicted(monkeypatch, k, flags, cluster, split, deep):
    monkeypatch.setenv("LF_CLUSTER", cluster)
    monkeypatch.setenv("LF_SPLIT", split)
    monkeypatch.setenv("LF_DEEP", deep)
    rng = np.random.default_rng(600 + 10 * k + flags)
    case = _pins.rand_case(rng, 3, 4, 2, 64, 700, p_masked=0.05, max_age=3000)
    check_ex(case, 8, 0.125, k, flags, f"k={k} flags={flags}")


@pytest.mark.parametrize("chunk_tiles", ["1", "7"])
def test_topk_with_many_chunks(monkeypatch, chunk_tiles):
    monkeypatch.setenv("LF_CHUNK_TILES", chunk_tiles)
    rng = np.random.default_rng(int(chunk_tiles))
    case = _pins.rand_case(rng, 1, 8, 2, 128, 2000, p_masked=0.3, max_age=9000)
    check_ex(case, 32, 0.088, 100, 1, f"chunk_tiles={chunk_tiles}")


def test_periodic_compression_on_benchmark_shape():
    """k = 128 at once with the evicted slots masked, on 8 sequences of the
    Fig. 1 workload."""
    wl = WORKLOADS["qwen3_8b_b128_s3200"].with_batch(8)
    st = initial_state(wl)
    inp = step_inputs(wl, 0)
    case = {**{k: st[k] for k in ("k_cache", "v_cache", "mask")}, **inp,
            "write_slot": np.full((wl.B, wl.Hkv), -1, dtype=np.int32)}
    gpu, _ = check_ex(case, wl.W, wl.scale, 128, lf.LF_STEP_MASK_EVICTED, "periodic k=128")
    assert np.all(gpu["next"] >= 0)
    assert np.all((gpu["mask"] < 0).sum(-1) == 128)


def test_selection_argument_errors():
    dev = "cuda"
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 2, 10, 64, dtype=torch.bfloat16, device=dev)
    mask = torch.zeros(1, 2, 10, dtype=torch.int32, device=dev)
    nk = torch.zeros(1, 2, 64, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(1, 2, dtype=torch.int32, device=dev)
    out = torch.zeros_like(q)
    for kk, flags in ((0, 0), (lf.LF_MAX_TOPK + 1, 0), (1, 8)):  # 8: no such flag bit
        nxt = torch.zeros(1, 2, max(kk, 1), dtype=torch.int32, device=dev)
        lib = lf.load_library()
        rc = lib.lf_decode_step_ex(q.data_ptr(), k.data_ptr(), k.clone().data_ptr(),
                                   mask.data_ptr(), nk.data_ptr(), nk.data_ptr(), ws.data_ptr(),
                                   out.data_ptr(), nxt.data_ptr(), kk, flags, None, 1, 4, 2, 64,
                                   10, 0, __import__("ctypes").c_float(0.1),
                                   torch.cuda.current_stream().cuda_stream)
        assert rc == lf.LF_ERR_INVALID_ARG
