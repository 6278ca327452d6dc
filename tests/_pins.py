"""Pins of the fp64 oracle: checks that do not re-run the oracle's own formula.

Each ``check_*`` takes ``step``, a callable with the signature of
``oracle.decode_step``, and raises AssertionError when the oracle disagrees
with something the paper or the mathematics fixes:

* brute force on tiny inputs (softmax without max-shift, score via the
  identity I_j = (sum_h p_hj) * ||v_j||_1, argmin by sorting);
* a library routine (torch's fp64 scaled_dot_product_attention and softmax);
* closed forms (zero query or identical keys give uniform weights);
* hand-worked fixtures under tests/golden/;
* invariants (weights sum to one, masked slots weigh nothing and are never
  evicted, a zero-V slot scores 0, the protected window is never evicted,
  permutation equivariance, ages stay distinct across steps).

The same checks run against deliberately broken builds of the oracle in
``test_oracle_mutants.py``; every planted mistake must trip at least one.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

from decode_kv_cache_step_gb300.workloads import (
    WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits, initial_state, step_inputs)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# input helpers
# ---------------------------------------------------------------------------

def rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.2, max_age=50, ws_mode="live"):
    """Random bf16 case with random ages, some masked slots and a write slot per unit."""
    g = lambda *s: f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
    case = {
        "q": g(B, Hq, d), "k_cache": g(B, Hkv, S, d), "v_cache": g(B, Hkv, S, d),
        "new_k": g(B, Hkv, d), "new_v": g(B, Hkv, d),
    }
    mask = np.empty((B, Hkv, S), dtype=np.int32)
    ws = np.empty((B, Hkv), dtype=np.int32)
    for b in range(B):
        for h in range(Hkv):
            ages = rng.permutation(max(max_age, S))[:S].astype(np.int32)
            masked = rng.random(S) < p_masked
            ages[masked] = -1
            mask[b, h] = ages
            live = np.flatnonzero(~masked)
            if ws_mode == "none" or (ws_mode == "live" and live.size == 0):
                ws[b, h] = -1
            elif ws_mode == "live":
                ws[b, h] = int(rng.choice(live))
            else:
                ws[b, h] = int(rng.integers(0, S))
    case["mask"] = mask
    case["write_slot"] = ws
    return case


def copy_case(case):
    return {k: np.array(v, copy=True) for k, v in case.items()}


def run(step, case, W, scale, **kw):
    c = copy_case(case)
    res = step(c["q"], c["k_cache"], c["v_cache"], c["mask"], c["new_k"], c["new_v"],
               c["write_slot"], W, scale, **kw)
    res["state"] = c
    return res


def f(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------
# brute force (pure Python, tiny sizes only)
# ---------------------------------------------------------------------------

def brute_force(case, W, scale, topk=1, fill_first=False, mask_evicted=False):
    """Pure-Python restatement, structured differently from the oracle.

    Softmax without max-shift, score through (sum_h p) * ||v||_1, selection by
    sorting (class, score, index) triples, state kept in dicts.
    """
    q, K, V = f(case["q"]), f(case["k_cache"]), f(case["v_cache"])
    nk, nv = f(case["new_k"]), f(case["new_v"])
    B, Hq, d = q.shape
    Hkv, S = K.shape[1], K.shape[2]
    g = Hq // Hkv
    out = np.zeros((B, Hq, d))
    nxt = np.zeros((B, Hkv, topk), dtype=np.int32)
    scores = np.full((B, Hkv, S), np.inf)
    ages_after = np.array(case["mask"], copy=True)
    for b in range(B):
        for kv in range(Hkv):
            ws = int(case["write_slot"][b, kv])
            ages = {j: int(case["mask"][b, kv, j]) for j in range(S)}
            rows_k = {j: list(K[b, kv, j]) for j in range(S)}
            rows_v = {j: list(V[b, kv, j]) for j in range(S)}
            if 0 <= ws < S:
                rows_k[ws], rows_v[ws] = list(nk[b, kv]), list(nv[b, kv])
                ages = {j: (0 if j == ws else (a + 1 if a >= 0 else a)) for j, a in ages.items()}
            live = [j for j in range(S) if ages[j] >= 0]
            psum = {j: 0.0 for j in live}
            for h in range(g):
                hq = kv * g + h
                e = {j: math.exp(scale * sum(q[b, hq, c] * rows_k[j][c] for c in range(d)))
                     for j in live}
                tot = sum(e.values())
                for c in range(d):
                    out[b, hq, c] = sum(e[j] / tot * rows_v[j][c] for j in live) if live else 0.0
                for j in live:
                    psum[j] += e[j] / tot
            for j in live:
                scores[b, kv, j] = psum[j] * sum(abs(x) for x in rows_v[j])
            elig = [(1, scores[b, kv, j], j) for j in live if ages[j] >= W]
            if fill_first:
                elig += [(0, 0.0, j) for j in range(S) if ages[j] < 0]
            elig.sort()
            for i in range(topk):
                nxt[b, kv, i] = elig[i][2] if i < len(elig) else -1
                if mask_evicted and i < len(elig):
                    ages[elig[i][2]] = -1
            for j in range(S):
                ages_after[b, kv, j] = ages[j]
    if topk == 1:
        nxt = nxt[:, :, 0]
    return {"out": out, "next_slot": nxt, "scores": scores, "mask": ages_after}


# ---------------------------------------------------------------------------
# checks
# ---------------------------------------------------------------------------

def check_brute_force(step, seeds=range(6)):
    shapes = [(1, 1, 1, 3, 5), (1, 2, 1, 4, 6), (2, 4, 2, 2, 7), (1, 3, 1, 4, 8),
              (2, 2, 2, 3, 4), (1, 6, 2, 2, 8)]
    for seed, shp in zip(seeds, shapes):
        rng = np.random.default_rng(100 + seed)
        case = rand_case(rng, *shp, p_masked=0.25, max_age=12)
        W = int(rng.integers(0, 4))
        scale = float(np.float32(0.7))
        res = run(step, case, W, scale, want_scores=True)
        ref = brute_force(case, W, scale)
        np.testing.assert_allclose(res["out"], ref["out"], rtol=0, atol=1e-12)
        live = np.isfinite(ref["scores"])
        assert np.array_equal(np.isfinite(res["scores"]), live)
        np.testing.assert_allclose(res["scores"][live], ref["scores"][live], rtol=1e-12, atol=1e-14)
        assert np.array_equal(res["next_slot"], ref["next_slot"]), (res["next_slot"], ref["next_slot"])
        assert np.array_equal(res["state"]["mask"], ref["mask"])


def check_sdpa(step):
    """torch fp64 scaled_dot_product_attention with a boolean mask and GQA repeat."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, d, S = 2, 8, 2, 32, 96
    case = rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.3, max_age=200)
    scale = float(np.float32(1 / math.sqrt(d)))
    res = run(step, case, 4, scale, want_p=True)
    st = res["state"]
    g = Hq // Hkv
    qt = torch.from_numpy(f(case["q"]))[:, :, None, :]                 # B,Hq,1,d
    kt = torch.from_numpy(f(st["k_cache"])).repeat_interleave(g, dim=1)  # B,Hq,S,d
    vt = torch.from_numpy(f(st["v_cache"])).repeat_interleave(g, dim=1)
    live = torch.from_numpy(st["mask"] >= 0).repeat_interleave(g, dim=1)[:, :, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=live, scale=scale)
    np.testing.assert_allclose(res["out"], ref[:, :, 0, :].numpy(), rtol=0, atol=1e-12)
    logits = (qt @ kt.transpose(-1, -2))[:, :, 0, :] * scale
    logits = logits.masked_fill(~live[:, :, 0, :], float("-inf"))
    p_ref = torch.softmax(logits, dim=-1).numpy()
    np.testing.assert_allclose(res["p"], p_ref, rtol=0, atol=1e-13)


def check_weights_sum_to_one_and_masked_zero(step):
    wl = WORKLOADS["tiny_b2_s256"]
    st = initial_state(wl)
    rng = np.random.default_rng(3)
    for t in range(3):
        inp = step_inputs(wl, t)
        case = {**{k: st[k] for k in ("k_cache", "v_cache", "mask")}, **inp,
                "write_slot": rng.integers(0, 240, size=(wl.B, wl.Hkv)).astype(np.int32)}
        res = run(step, case, wl.W, wl.scale, want_p=True)
        p = res["p"]
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
        masked = np.repeat(res["state"]["mask"] < 0, wl.g, axis=1)
        assert np.all(p[masked] == 0.0)
        assert np.all(p[~masked] > 0.0)


def check_masked_garbage_is_inert(step):
    """NaN / huge values in masked slots change nothing and are never evicted."""
    rng = np.random.default_rng(11)
    case = rand_case(rng, 2, 4, 2, 16, 40, p_masked=0.4, max_age=80)
    clean = run(step, case, 2, 0.25, want_scores=True)
    dirty_case = copy_case(case)
    m = case["mask"] < 0
    ws = case["write_slot"]
    for b in range(2):
        for h in range(2):
            if 0 <= ws[b, h]:
                m[b, h, ws[b, h]] = False  # the write slot becomes live
    nan_bits, inf_bits, big_bits = 0x7FC1, 0x7F80, 0x7F00  # NaN, +inf, 1.7e38
    for name, bits in (("k_cache", nan_bits), ("v_cache", inf_bits)):
        arr = dirty_case[name]
        arr[m] = bits
    dirty_case["k_cache"][m, :3] = big_bits
    dirty = run(step, dirty_case, 2, 0.25, want_scores=True)
    np.testing.assert_array_equal(clean["out"], dirty["out"])
    np.testing.assert_array_equal(clean["next_slot"], dirty["next_slot"])
    np.testing.assert_array_equal(clean["scores"], dirty["scores"])
    mask_after = dirty["state"]["mask"]
    for b in range(2):
        for h in range(2):
            n = dirty["next_slot"][b, h]
            assert n == -1 or mask_after[b, h, n] >= 2


def check_zero_v_scores_zero_and_ties_lowest(step):
    rng = np.random.default_rng(5)
    case = rand_case(rng, 1, 4, 1, 8, 12, p_masked=0.0, max_age=12, ws_mode="none")
    case["mask"][0, 0] = np.arange(12, dtype=np.int32)[::-1]  # slot j has age 11 - j
    zero = [2, 5, 9]
    case["v_cache"][0, 0, zero] = 0
    res = run(step, case, 3, 0.3, want_scores=True)
    sc = res["scores"][0, 0]
    assert np.all(sc[zero] == 0.0)
    assert np.all(sc[[j for j in range(12) if j not in zero]] > 0.0)
    assert res["next_slot"][0, 0] == 2          # tie at 0: lowest index
    res = run(step, case, 3, 0.3)
    # -0.0 rows (sign bit only) are zero vectors too
    case2 = copy_case(case)
    case2["v_cache"][0, 0, 2] = 0x8000
    assert run(step, case2, 3, 0.3)["next_slot"][0, 0] == 2
    # protect slots 5.. (age < W = 7 means slots 5..11): only slot 2 of the zeros is eligible
    res = run(step, case, 7, 0.3)
    assert res["next_slot"][0, 0] == 2
    # W = 10 leaves slots 0 and 1 only
    res = run(step, case, 10, 0.3, want_scores=True)
    sc = res["scores"][0, 0]
    assert res["next_slot"][0, 0] == (0 if sc[0] <= sc[1] else 1)


def check_protected_window(step):
    rng = np.random.default_rng(9)
    for W in (0, 1, 5, 30):
        case = rand_case(rng, 2, 6, 3, 8, 30, p_masked=0.2, max_age=40)
        res = run(step, case, W, 0.5, want_scores=True)
        ages = res["state"]["mask"]
        for b in range(2):
            for h in range(3):
                n = res["next_slot"][b, h]
                elig = [j for j in range(30) if ages[b, h, j] >= W]
                if not elig:
                    assert n == -1
                    continue
                assert ages[b, h, n] >= W
                best = min(res["scores"][b, h, j] for j in elig)
                assert res["scores"][b, h, n] == best
                assert n == min(j for j in elig if res["scores"][b, h, j] == best)


def check_uniform_closed_form(step):
    """q = 0 (and, separately, identical keys) gives p = 1/L: out = mean of live V,
    I_j = g * ||v_j||_1 / L."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, d, S = 2, 6, 2, 8, 20
    for mode in ("zero_q", "same_k"):
        case = rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.3, max_age=30)
        if mode == "zero_q":
            case["q"][:] = 0
        else:
            row = f32_to_bf16_bits(rng.standard_normal(d).astype(np.float32))
            case["k_cache"][:] = row
            case["new_k"][:] = row
        res = run(step, case, 0, 0.4, want_scores=True)
        st = res["state"]
        V = f(st["v_cache"])
        g = Hq // Hkv
        for b in range(B):
            for h in range(Hkv):
                live = st["mask"][b, h] >= 0
                L = int(live.sum())
                mean = V[b, h, live].mean(axis=0)
                for hh in range(g):
                    np.testing.assert_allclose(res["out"][b, h * g + hh], mean, rtol=0, atol=1e-12)
                l1 = np.abs(V[b, h, live]).sum(axis=1)
                np.testing.assert_allclose(res["scores"][b, h, live], g * l1 / L, rtol=1e-12)


def check_score_sum_when_l1_constant(step):
    """All live rows with ||v||_1 = c give sum_j I_j = g * c (each head's weights sum to 1)."""
    rng = np.random.default_rng(4)
    B, Hq, Hkv, d, S = 1, 8, 2, 16, 30
    case = rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.2, max_age=60)
    signs = rng.choice([-1.0, 1.0], size=(B, Hkv, S, d)).astype(np.float32) * 0.5
    case["v_cache"] = f32_to_bf16_bits(signs)
    case["new_v"] = f32_to_bf16_bits(rng.choice([-0.5, 0.5], size=(B, Hkv, d)).astype(np.float32))
    res = run(step, case, 0, 0.3, want_scores=True)
    sc = res["scores"]
    for h in range(Hkv):
        live = np.isfinite(sc[0, h])
        np.testing.assert_allclose(sc[0, h, live].sum(), (Hq // Hkv) * 0.5 * d, rtol=1e-12)


def check_permutation_equivariance(step):
    rng = np.random.default_rng(13)
    B, Hq, Hkv, d, S = 1, 4, 1, 8, 25
    case = rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.2, max_age=40)
    base = run(step, case, 3, 0.35, want_scores=True)
    perm = rng.permutation(S)
    inv = np.argsort(perm)
    pc = copy_case(case)
    for k in ("k_cache", "v_cache"):
        pc[k] = np.ascontiguousarray(case[k][:, :, perm])
    pc["mask"] = np.ascontiguousarray(case["mask"][:, :, perm])
    ws = case["write_slot"][0, 0]
    pc["write_slot"][0, 0] = inv[ws] if ws >= 0 else -1
    res = run(step, pc, 3, 0.35, want_scores=True)
    np.testing.assert_allclose(res["scores"][0, 0], base["scores"][0, 0][perm], rtol=1e-12)
    np.testing.assert_allclose(res["out"], base["out"], rtol=0, atol=1e-12)
    sc = base["scores"][0, 0]
    elig = np.flatnonzero(base["state"]["mask"][0, 0] >= 3)
    vals = np.sort(sc[elig])
    if len(vals) > 1 and vals[1] > vals[0] * (1 + 1e-9):
        assert perm[res["next_slot"][0, 0]] == base["next_slot"][0, 0]


def check_state_transition(step):
    rng = np.random.default_rng(17)
    B, Hq, Hkv, d, S = 2, 2, 2, 4, 10
    case = rand_case(rng, B, Hq, Hkv, d, S, p_masked=0.3, max_age=20, ws_mode="any")
    case["mask"][0, 0, 3] = 2**31 - 1     # saturating age
    case["write_slot"][1, 1] = -1         # priming unit: nothing changes
    m_in = case["mask"]
    res = run(step, case, 1, 0.5)
    st = res["state"]
    assert res["invalid_writes"] == 0
    for b in range(B):
        for h in range(Hkv):
            ws = case["write_slot"][b, h]
            for j in range(S):
                a0, a1 = int(m_in[b, h, j]), int(st["mask"][b, h, j])
                if ws < 0:
                    assert a1 == a0
                elif j == ws:
                    assert a1 == 0
                elif a0 < 0:
                    assert a1 == a0
                else:
                    assert a1 == min(a0 + 1, 2**31 - 1)
            if ws >= 0:
                assert np.array_equal(st["k_cache"][b, h, ws], case["new_k"][b, h])
                assert np.array_equal(st["v_cache"][b, h, ws], case["new_v"][b, h])
                other = [j for j in range(S) if j != ws]
                assert np.array_equal(st["k_cache"][b, h, other], case["k_cache"][b, h, other])
            else:
                assert np.array_equal(st["k_cache"][b, h], case["k_cache"][b, h])
    # invalid write slots are counted and ignored
    bad = copy_case(case)
    bad["write_slot"][0, 0] = S
    bad["write_slot"][1, 0] = -7
    res = run(step, bad, 1, 0.5)
    assert res["invalid_writes"] == 2
    assert np.array_equal(res["state"]["mask"][0, 0], case["mask"][0, 0])
    assert np.array_equal(res["state"]["k_cache"][1, 0], case["k_cache"][1, 0])


def check_degenerate(step):
    rng = np.random.default_rng(23)
    # no live slot, no write: zero output, no eviction
    case = rand_case(rng, 1, 2, 1, 4, 6, p_masked=1.0, ws_mode="none")
    res = run(step, case, 0, 1.0)
    assert np.all(res["out"] == 0.0) and res["next_slot"][0, 0] == -1
    # writing into an empty cache: the written token is the only live slot
    case["write_slot"][0, 0] = 4
    res = run(step, case, 0, 1.0)
    np.testing.assert_allclose(res["out"][0, 0], f(case["new_v"][0, 0]), atol=0)
    assert res["next_slot"][0, 0] == 4       # W = 0: the fresh token may be evicted
    res = run(step, case, 1, 1.0)
    assert res["next_slot"][0, 0] == -1      # W = 1 protects it
    # S = 1
    case = rand_case(rng, 1, 1, 1, 3, 1, p_masked=0.0, max_age=1)
    res = run(step, case, 0, 1.0)
    assert res["next_slot"][0, 0] == 0
    np.testing.assert_allclose(res["out"][0, 0], f(res["state"]["v_cache"][0, 0, 0]), atol=0)


def check_multi_step_invariants(step):
    """Sixteen steps of the small workload: ages of live slots stay distinct,
    the evicted slot receives the next token, the live set never changes."""
    wl = WORKLOADS["tiny_b2_s256"]
    st = initial_state(wl)
    live0 = st["mask"] >= 0
    ws = np.full((wl.B, wl.Hkv), -1, dtype=np.int32)
    for t in range(wl.steps + 1):
        inp = step_inputs(wl, t)
        k, v, m = st["k_cache"], st["v_cache"], st["mask"]
        res = step(inp["q"], k, v, m, inp["new_k"], inp["new_v"], ws, wl.W, wl.scale)
        assert np.array_equal(m >= 0, live0)
        for b in range(wl.B):
            for h in range(wl.Hkv):
                ages = m[b, h][m[b, h] >= 0]
                assert len(np.unique(ages)) == len(ages)
                if ws[b, h] >= 0:
                    assert np.array_equal(k[b, h, ws[b, h]], inp["new_k"][b, h])
                n = res["next_slot"][b, h]
                assert 0 <= n < 240 and m[b, h, n] >= wl.W
        ws = res["next_slot"].copy()


def check_brute_force_selection_options(step):
    """Top-k, fill-empty-first and mask-evicted against the brute force."""
    shapes = [(1, 2, 1, 3, 9), (2, 4, 2, 2, 7), (1, 6, 2, 2, 8), (2, 2, 1, 4, 12)]
    opts = [dict(topk=3), dict(topk=2, fill_first=True), dict(topk=1, fill_first=True),
            dict(topk=4, mask_evicted=True), dict(topk=20, fill_first=True, mask_evicted=True)]
    for i, (shp, opt) in enumerate(zip(shapes * 2, opts)):
        rng = np.random.default_rng(300 + i)
        case = rand_case(rng, *shp, p_masked=0.3, max_age=12)
        W = int(rng.integers(0, 3))
        scale = float(np.float32(0.6))
        res = run(step, case, W, scale, **opt)
        ref = brute_force(case, W, scale, **opt)
        assert np.array_equal(res["next_slot"], ref["next_slot"]), (opt, res["next_slot"], ref["next_slot"])
        assert np.array_equal(res["state"]["mask"], ref["mask"]), opt
        np.testing.assert_allclose(res["out"], ref["out"], rtol=0, atol=1e-12)


def check_topk_properties(step):
    rng = np.random.default_rng(31)
    case = rand_case(rng, 2, 8, 2, 16, 60, p_masked=0.25, max_age=200)
    base = run(step, case, 5, 0.3, want_scores=True)
    for k in (1, 7, 64):
        res = run(step, case, 5, 0.3, topk=k)
        lst = res["next_slot"] if k > 1 else res["next_slot"][:, :, None]
        ages = base["state"]["mask"]
        for b in range(2):
            for h in range(2):
                elig = [j for j in range(60) if ages[b, h, j] >= 5]
                want = sorted(elig, key=lambda j: (base["scores"][b, h, j], j))[:k]
                got = [int(x) for x in lst[b, h] if x >= 0]
                assert got == want, (k, got, want)
                assert all(x == -1 for x in lst[b, h, len(want):])
        if k == 1:
            assert np.array_equal(res["next_slot"], base["next_slot"])


def check_fill_first(step):
    rng = np.random.default_rng(37)
    case = rand_case(rng, 2, 4, 2, 8, 40, p_masked=0.0, max_age=100, ws_mode="none")
    case["mask"][0, 0, [7, 3, 30]] = -1
    res = run(step, case, 2, 0.3, fill_first=True)
    plain = run(step, case, 2, 0.3)
    assert res["next_slot"][0, 0] == 3                       # lowest empty slot first
    assert np.array_equal(res["next_slot"][1], plain["next_slot"][1])   # no empty slot
    assert res["next_slot"][0, 1] == plain["next_slot"][0, 1]
    res3 = run(step, case, 2, 0.3, fill_first=True, topk=4)
    assert list(res3["next_slot"][0, 0, :3]) == [3, 7, 30]
    assert res3["next_slot"][0, 0, 3] == plain["next_slot"][0, 0]


def check_mask_evicted(step):
    rng = np.random.default_rng(41)
    case = rand_case(rng, 1, 4, 2, 8, 30, p_masked=0.1, max_age=60)
    plain = run(step, case, 3, 0.3, topk=5)
    ev = run(step, case, 3, 0.3, topk=5, mask_evicted=True)
    assert np.array_equal(plain["next_slot"], ev["next_slot"])
    m_plain, m_ev = plain["state"]["mask"], ev["state"]["mask"]
    for h in range(2):
        chosen = [int(x) for x in ev["next_slot"][0, h] if x >= 0]
        assert np.all(m_ev[0, h, chosen] == -1)
        rest = [j for j in range(30) if j not in chosen]
        assert np.array_equal(m_ev[0, h, rest], m_plain[0, h, rest])


def check_attention_only(step):
    rng = np.random.default_rng(43)
    case = rand_case(rng, 2, 8, 2, 16, 50, p_masked=0.3, max_age=100, ws_mode="any")
    full = run(step, case, 4, 0.25)
    att = run(step, case, 4, 0.25, attention_only=True)
    assert att["next_slot"] is None
    np.testing.assert_array_equal(att["out"], full["out"])
    m0, m1 = case["mask"], att["state"]["mask"]
    for b in range(2):
        for h in range(2):
            ws = case["write_slot"][b, h]
            for j in range(50):
                if j == ws and m0[b, h, j] < 0:
                    assert m1[b, h, j] == 0
                else:
                    assert m1[b, h, j] == m0[b, h, j]
            assert np.array_equal(att["state"]["k_cache"][b, h], full["state"]["k_cache"][b, h])


def _frac(s):
    return Fraction(s)


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def golden_case(g):
    sh = g["shape"]
    B, Hq, Hkv, d, S = sh["B"], sh["Hq"], sh["Hkv"], sh["d"], sh["S"]
    def bits(key, shape):
        return np.array([int(x, 16) for x in g["inputs"][key]], dtype=np.uint16).reshape(shape)
    case = {
        "q": bits("q", (B, Hq, d)), "k_cache": bits("k_cache", (B, Hkv, S, d)),
        "v_cache": bits("v_cache", (B, Hkv, S, d)), "new_k": bits("new_k", (B, Hkv, d)),
        "new_v": bits("new_v", (B, Hkv, d)),
        "mask": np.array(g["inputs"]["mask"], dtype=np.int32).reshape(B, Hkv, S),
        "write_slot": np.array(g["inputs"]["write_slot"], dtype=np.int32).reshape(B, Hkv),
    }
    return case


def check_golden(step, name):
    g = load_golden(name)
    case = golden_case(g)
    scale = float(np.float32(eval(g["scale"], {"math": math})))  # e.g. "1.0", "math.log(2)"
    res = run(step, case, g["W"], scale, want_p=True, want_scores=True)
    exp = g["expected"]
    tol = float(exp.get("tolerance", 0.0))
    shp = res["out"].shape
    want_out = np.array([float(_frac(x)) for x in exp["out"]]).reshape(shp)
    np.testing.assert_allclose(res["out"], want_out, rtol=tol, atol=tol + 1e-15)
    S = case["mask"].shape[-1]
    sc_want = np.array([np.inf if x == "inf" else float(_frac(x)) for x in exp["scores"]])
    np.testing.assert_allclose(res["scores"].reshape(-1), sc_want, rtol=tol + 1e-15, atol=1e-15)
    if "p" in exp:
        p_want = np.array([float(_frac(x)) for x in exp["p"]]).reshape(res["p"].shape)
        np.testing.assert_allclose(res["p"], p_want, rtol=tol, atol=tol + 1e-15)
    assert res["next_slot"].reshape(-1).tolist() == exp["next_slot"]
    assert res["state"]["mask"].reshape(-1).tolist() == exp["mask_after"]
    assert S == g["shape"]["S"]


GOLDEN_FILES = ("uniform_write_tie.json", "powers_of_two.json", "zero_v_masked_nan.json")

ALL_CHECKS = [
    check_brute_force, check_sdpa, check_weights_sum_to_one_and_masked_zero,
    check_masked_garbage_is_inert, check_zero_v_scores_zero_and_ties_lowest,
    check_protected_window, check_uniform_closed_form, check_score_sum_when_l1_constant,
    check_permutation_equivariance, check_state_transition, check_degenerate,
    check_multi_step_invariants, check_brute_force_selection_options, check_topk_properties,
    check_fill_first, check_mask_evicted, check_attention_only,
] + [
    (lambda name: (lambda step: check_golden(step, name)))(n) for n in GOLDEN_FILES
]
