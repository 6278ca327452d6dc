"""GPU edge cases against the fp64 oracle: every supported head dim and
group size, ragged slot counts that leave partial tiles, masked and empty
units, writes into masked slots, garbage in masked slots, invalid write
slots, protected windows, ties, the largest supported cache (also at the
widest group), the most units a launch takes, argument errors, and
concurrent streams."""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
from decode_kv_cache_step_gb300.workloads import f32_to_bf16_bits

import _pins
from _gpu import DevState, compare_unit, oracle_step, to_dev, to_host_bits

pytestmark = pytest.mark.gpu


def check_case(case, W, scale, where=""):
    B, Hkv, S, d = case["k_cache"].shape
    Hq = case["q"].shape[1]
    g = Hq // Hkv
    dev = DevState(case["k_cache"], case["v_cache"], case["mask"], Hq)
    host = {k: np.array(case[k], copy=True) for k in ("k_cache", "v_cache", "mask")}
    gpu = dev.step(case["q"], case["new_k"], case["new_v"], case["write_slot"], W, scale)
    ora = oracle_step(host, case["q"], case["new_k"], case["new_v"], case["write_slot"], W, scale)
    assert np.array_equal(dev.mask.cpu().numpy(), host["mask"]), where
    assert np.array_equal(to_host_bits(dev.k), host["k_cache"]), where
    assert np.array_equal(to_host_bits(dev.v), host["v_cache"]), where
    for b in range(B):
        for h in range(Hkv):
            compare_unit(gpu, ora, b, h, g, host["mask"], W, where=where)
    return gpu, ora, dev


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
@pytest.mark.parametrize("S", [1, 5, 63, 64, 65, 130, 1000])
def test_shapes(d, g, S):
    rng = np.random.default_rng(1000 * d + 10 * g + S)
    Hkv = 2
    case = _pins.rand_case(rng, 2, Hkv * g, Hkv, d, S, p_masked=0.2, max_age=3 * S + 5,
                           ws_mode="any")
    check_case(case, W=min(4, S // 3), scale=float(np.float32(1 / np.sqrt(d))),
               where=f"d={d} g={g} S={S}")


@pytest.mark.parametrize("chunk_tiles", ["1", "2", "7", "32"])
def test_chunking(monkeypatch, chunk_tiles):
    monkeypatch.setenv("LF_CHUNK_TILES", chunk_tiles)
    rng = np.random.default_rng(int(chunk_tiles))
    case = _pins.rand_case(rng, 3, 8, 2, 128, 777, p_masked=0.3, max_age=3000)
    check_case(case, W=8, scale=0.088, where=f"chunk_tiles={chunk_tiles}")


def test_empty_and_degenerate_units():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, d, S = 4, 8, 2, 128, 300
    case = _pins.rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.1, max_age=1000)
    case["mask"][0, 0] = -1          # empty unit, no write: out 0, next -1
    case["write_slot"][0, 0] = -1
    case["mask"][0, 1] = -1          # empty unit with a write: the token is the only slot
    case["write_slot"][0, 1] = 299
    case["mask"][1, 0, :] = -1       # one live slot
    case["mask"][1, 0, 150] = 77
    case["write_slot"][1, 0] = -1
    case["write_slot"][1, 1] = -1    # priming unit: nothing ages
    gpu, ora, dev = check_case(case, W=2, scale=0.1, where="degenerate")
    assert np.all(gpu["out"][0, 0:4] == 0.0) and gpu["next_slot"][0, 0] == -1
    assert gpu["next_slot"][0, 1] == -1           # W = 2 protects the fresh token
    assert gpu["next_slot"][1, 0] == 150
    np.testing.assert_array_equal(dev.mask[1, 1].cpu().numpy(), case["mask"][1, 1])


def test_protected_window_extremes():
    rng = np.random.default_rng(6)
    case = _pins.rand_case(rng, 2, 4, 1, 64, 200, p_masked=0.0, max_age=200)
    for W in (0, 1, 199, 200, 10**6):
        gpu, _, _ = check_case(case, W=W, scale=0.125, where=f"W={W}")
        if W > 200:
            assert np.all(gpu["next_slot"] == -1)


def test_write_into_masked_slot_makes_it_live():
    rng = np.random.default_rng(7)
    case = _pins.rand_case(rng, 1, 4, 1, 128, 100, p_masked=0.0, max_age=100, ws_mode="none")
    case["mask"][0, 0, 90:] = -1
    case["write_slot"][0, 0] = 95
    _, _, dev = check_case(case, W=1, scale=0.08, where="masked write")
    assert int(dev.mask[0, 0, 95]) == 0


def test_garbage_in_masked_slots_is_inert():
    rng = np.random.default_rng(8)
    case = _pins.rand_case(rng, 2, 8, 2, 128, 500, p_masked=0.3, max_age=2000)
    clean, _, _ = check_case(case, W=4, scale=0.088, where="clean")
    dirty = _pins.copy_case(case)
    m = case["mask"] < 0
    dirty["k_cache"][m] = 0x7FC1          # NaN
    dirty["v_cache"][m] = 0x7F80          # +inf
    dirty["v_cache"][m, ::3] = 0xFF80     # -inf
    got, _, _ = check_case(dirty, W=4, scale=0.088, where="dirty")
    assert np.array_equal(got["out"], clean["out"])
    assert np.array_equal(got["next_slot"], clean["next_slot"])
    assert np.array_equal(got["scores"], clean["scores"])


def test_zero_v_ties_pick_lowest_index():
    rng = np.random.default_rng(9)
    case = _pins.rand_case(rng, 1, 8, 2, 128, 400, p_masked=0.0, max_age=400, ws_mode="none")
    case["mask"][0, :] = np.arange(400, dtype=np.int32)[::-1]   # slot j has age 399 - j
    zero = [17, 130, 131, 390]
    case["v_cache"][0, :, zero] = 0
    gpu, _, _ = check_case(case, W=16, scale=0.088, where="ties")
    assert np.all(gpu["scores"][0, :, zero] == 0.0)
    assert list(gpu["next_slot"][0]) == [17, 17]


def test_invalid_write_slot_is_ignored_and_reported():
    rng = np.random.default_rng(10)
    case = _pins.rand_case(rng, 1, 4, 2, 64, 50, p_masked=0.0, max_age=50)
    case["write_slot"][0, 0] = 50
    case["write_slot"][0, 1] = -3
    lf.device_errors(clear=True)
    check_case(case, W=2, scale=0.125, where="invalid write")
    assert lf.device_errors(clear=True) == lf.LF_DEVERR_BAD_WRITE_SLOT
    assert lf.device_errors(clear=True) == 0


def test_largest_supported_cache():
    rng = np.random.default_rng(11)
    S = 1 << 20
    d = 64
    g = lambda *s: f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
    case = {"q": g(1, 1, d), "k_cache": g(1, 1, S, d), "v_cache": g(1, 1, S, d),
            "new_k": g(1, 1, d), "new_v": g(1, 1, d),
            "mask": (S - 1 - np.arange(S, dtype=np.int32)).reshape(1, 1, S),
            "write_slot": np.array([[12345]], dtype=np.int32)}
    check_case(case, W=128, scale=0.125, where="S=2^20")


def test_largest_cache_widest_group():
    """S = 2^20 at d = 128 and g = 8: the split finish over 16384 tiles, with
    the largest score-term scratch a unit takes."""
    rng = np.random.default_rng(12)
    S = 1 << 20
    case = _pins.rand_case(rng, 1, 8, 1, 128, S, p_masked=0.3, max_age=3 * S, ws_mode="any")
    p = lf.step_plan(1, 8, 1, 128, S)
    assert p["split"] and not p["cluster"], p
    check_case(case, W=128, scale=float(np.float32(1 / np.sqrt(128))), where="S=2^20 d=128 g=8")


def test_most_units():
    """B * Hkv = 65535, the most units one launch takes (the grid's y extent),
    with a ragged last tile."""
    rng = np.random.default_rng(13)
    B, Hq, Hkv, d, S = 65535, 2, 1, 64, 70
    case = _pins.rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.2, max_age=200, ws_mode="any")
    check_case(case, W=4, scale=0.125, where="65535 units")


def test_argument_errors():
    dev = torch.device("cuda")
    bf = torch.bfloat16
    q = torch.zeros(1, 4, 128, dtype=bf, device=dev)
    k = torch.zeros(1, 2, 10, 128, dtype=bf, device=dev)
    v = torch.zeros_like(k)
    mask = torch.zeros(1, 2, 10, dtype=torch.int32, device=dev)
    nk = torch.zeros(1, 2, 128, dtype=bf, device=dev)
    nv = torch.zeros_like(nk)
    ws = torch.zeros(1, 2, dtype=torch.int32, device=dev)
    out = torch.zeros_like(q)
    nxt = torch.zeros_like(ws)
    with pytest.raises(lf.LFError) as e:
        lf.decode_step(q, k, v, mask, nk, nv, ws, out, nxt, -1, 0.1)
    assert e.value.status == lf.LF_ERR_INVALID_ARG
    with pytest.raises(lf.LFError) as e:
        lf.decode_step(q, k, v, mask, nk, nv, ws, out, nxt, 0, float("nan"))
    assert e.value.status == lf.LF_ERR_INVALID_ARG
    q3 = torch.zeros(1, 6, 128, dtype=bf, device=dev)   # g = 3
    with pytest.raises(lf.LFError) as e:
        lf.decode_step(q3, k, v, mask, nk, nv, ws, torch.zeros_like(q3), nxt, 0, 0.1)
    assert e.value.status == lf.LF_ERR_UNSUPPORTED
    k96 = torch.zeros(1, 2, 10, 96, dtype=bf, device=dev)
    q96 = torch.zeros(1, 4, 96, dtype=bf, device=dev)
    nk96 = torch.zeros(1, 2, 96, dtype=bf, device=dev)
    with pytest.raises(lf.LFError) as e:
        lf.decode_step(q96, k96, k96.clone(), mask, nk96, nk96.clone(), ws, q96.clone(), nxt, 0, 0.1)
    assert e.value.status == lf.LF_ERR_UNSUPPORTED
    # a valid call still works after the errors
    lf.decode_step(q, k, v, mask, nk, nv, ws, out, nxt, 0, 0.1)
    torch.cuda.synchronize()
    assert lf.device_errors() == 0


def test_two_streams_run_independently():
    rng = np.random.default_rng(12)
    cases = [_pins.rand_case(rng, 4, 8, 2, 128, 900, p_masked=0.2, max_age=2000) for _ in range(2)]
    want = []
    for c in cases:
        g, _, _ = check_case(c, W=8, scale=0.088, where="serial")
        want.append(g)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    states = [DevState(c["k_cache"], c["v_cache"], c["mask"], 8) for c in cases]
    for _ in range(3):
        for c, st, s in zip(cases, states, streams):
            st.k.copy_(to_dev(c["k_cache"]))
            st.v.copy_(to_dev(c["v_cache"]))
            st.mask.copy_(to_dev(c["mask"]))
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                lf.decode_step(to_dev(c["q"]), st.k, st.v, st.mask, to_dev(c["new_k"]),
                               to_dev(c["new_v"]), to_dev(c["write_slot"]), st.out, st.next, 8, 0.088,
                               stream=s)
        torch.cuda.synchronize()
        for st, w in zip(states, want):
            assert np.array_equal(st.out.float().cpu().numpy().astype(np.float64), w["out"])
            assert np.array_equal(st.next.cpu().numpy(), w["next_slot"])
