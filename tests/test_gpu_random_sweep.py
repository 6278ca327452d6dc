"""Seeded random sweep against the fp64 oracle: shapes (d, g, heads, batch,
S from 1 to 9000), masks (random or ragged prefixes), windows, write modes,
entry points and selection options, each under a random launch plan
(clusters on or off and of up to 16 CTAs, split finish on or off, forced
chunk sizes, deep or 2-stage cluster ring). The comparison rules are the parity suite's."""
import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf

import _pins
from _gpu import DevState, compare_unit, oracle_step, to_host_bits
from test_gpu_next import check_ex

pytestmark = pytest.mark.gpu

CASES = 120


def _draw(i):
    rng = np.random.default_rng(7000 + i)
    d = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.integers(1, 4))
    B = int(rng.integers(1, 4))
    S = int(rng.choice([rng.integers(1, 200), rng.integers(200, 3000), rng.integers(4000, 9000)]))
    p_masked = float(rng.choice([0.0, 0.1, 0.5, 0.95]))
    ws_mode = str(rng.choice(["live", "any", "none"]))
    case = _pins.rand_case(rng, B, Hkv * g, Hkv, d, S, p_masked=p_masked, max_age=3 * S + 7,
                           ws_mode=ws_mode)
    if rng.random() < 0.4:  # ragged prefixes
        for b in range(B):
            for h in range(Hkv):
                case["mask"][b, h, int(rng.integers(0, S + 1)):] = -1
    W = int(rng.integers(0, min(S, 64) + 1))
    scale = float(np.float32(1 / np.sqrt(d)))
    env = {}
    for name, choices in (("LF_SPLIT", [None, "0", "1"]), ("LF_CLUSTER", [None, "0", "1"]),
                          ("LF_DEEP", [None, "0", "1"])):
        c = choices[int(rng.integers(0, len(choices)))]
        if c is not None:
            env[name] = c
    if rng.random() < 0.4:
        env["LF_CHUNK_TILES"] = str(int(rng.integers(1, 33)))
    crng = np.random.default_rng(9000 + i)  # a stream of its own: the draws above stay
    if crng.random() < 0.3:
        env["LF_CLUSTER_MAX"] = str(int(crng.integers(2, 17)))
    entry = str(rng.choice(["step", "scores", "ex"]))
    k = int(rng.choice([1, 2, 17]))
    flags = int(rng.integers(0, 4))
    return case, W, scale, env, entry, k, flags


@pytest.mark.parametrize("i", range(CASES))
def test_random_case(monkeypatch, i):
    case, W, scale, env, entry, k, flags = _draw(i)
    for name, val in env.items():
        monkeypatch.setenv(name, val)
    B, Hkv, S, d = case["k_cache"].shape
    Hq = case["q"].shape[1]
    where = f"case {i}: B={B} Hq={Hq} Hkv={Hkv} d={d} S={S} W={W} env={env} entry={entry}"
    if entry == "ex":
        check_ex(case, W, scale, k, flags, where + f" k={k} flags={flags}")
        return
    dev = DevState(case["k_cache"], case["v_cache"], case["mask"], Hq)
    host = {kk: np.array(case[kk], copy=True) for kk in ("k_cache", "v_cache", "mask")}
    gpu = dev.step(case["q"], case["new_k"], case["new_v"], case["write_slot"], W, scale,
                   scores=(entry == "scores"))
    ora = oracle_step(host, case["q"], case["new_k"], case["new_v"], case["write_slot"], W, scale)
    assert np.array_equal(dev.mask.cpu().numpy(), host["mask"]), where
    assert np.array_equal(to_host_bits(dev.k), host["k_cache"]), where
    assert np.array_equal(to_host_bits(dev.v), host["v_cache"]), where
    for b in range(B):
        for h in range(Hkv):
            compare_unit(gpu, ora, b, h, Hq // Hkv, host["mask"], W,
                         check_scores=(entry == "scores"), where=where)
    assert lf.device_errors() == 0
