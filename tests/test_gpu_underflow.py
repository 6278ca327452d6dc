"""Eviction when LongFlowScore lies below fp32's normal range, against the
fp64 oracle.

LongFlow picks the slot to cover next from the score read off G (LongFlow
page: abstract; Fig. 2 caption, Right). When one key dominates a unit, the
other slots' weights p_hj sit hundreds of nats under it and their scores
I_j = sum_h p_hj * ||v_j||_1 fall to 1e-40 .. 1e-250: fp64 still orders them
by many orders of magnitude, while fp32 holds nothing below about 1.2e-38.
The rule stays the same at every scale: next_slot must equal the oracle's
whenever the oracle's best-to-second gap exceeds 1e-3 relative.

The cases are built so that the logits carry almost no rounding: every query
has two non-zero coordinates, so q.k is a sum of two bf16 products, and the
scores' error is the kernel's own fp32 arithmetic. Eligible slots get
logits 100..500 nats under the unit's maximum (a protected slot and the
written token hold logit 0). A second family draws q and K from N(0, 1) with
a large scale (3.0) so that attention is peaked as in a real head.

Every selection path is run: the last CTA's scan (register batches, the
live-tile list of a ragged unit, bulk copies of a long unit), the cluster
merge, the split finish's scoring kernel and k-at-once selection (k = 8).
Scores are compared in the log domain, exported with LF_STEP_LOG2_SCORES:
|log2 I_gpu - log2 I_oracle| <= log2(1 + 1e-3), the 1e-3 relative tolerance.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import decode_kv_cache_step_gb300 as lf
from decode_kv_cache_step_gb300.workloads import f32_to_bf16_bits

import oracle
from _gpu import OUT_ATOL, compare_unit, to_dev, to_host_bits
from test_gpu_next import _ranked, compare_topk

pytestmark = pytest.mark.gpu

LOG2_TOL = math.log2(1.0 + 1e-3)
FP32_MIN_NORMAL = 2.0 ** -126


def _bf16(a):
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def peaked_case(rng, B, g, Hkv, d, S, W, dead_tail=0, p_masked=0.05):
    """Logits s_hj = a_h * b_j + k_j[1] / 4 from q[h] = a_h * e_0 + e_1 / 4
    (two products of bf16 values, one fp32 rounding at most). One protected
    slot and the written token hold b = 0 (the unit's maximum); the other
    live slots get b in [-500, -100], a few in [-60, -5]; k_j[1] ~ N(0, 1)
    spreads slots that share a bf16 value of b."""
    Hq = Hkv * g
    q = np.zeros((B, Hq, d), dtype=np.float32)
    q[:, :, 0] = (1.0 + 0.25 * (np.arange(Hq) % g))[None, :]
    q[:, :, 1] = 0.25
    k = rng.standard_normal((B, Hkv, S, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, S, d)).astype(np.float32)
    mask = np.empty((B, Hkv, S), dtype=np.int32)
    ws = np.empty((B, Hkv), dtype=np.int32)
    for b in range(B):
        for h in range(Hkv):
            ages = rng.permutation(3 * S)[:S].astype(np.int32)
            ages[rng.random(S) < p_masked] = -1
            if dead_tail:
                ages[S - dead_tail:] = -1
            mask[b, h] = ages
            logit = -rng.uniform(100.0, 500.0, size=S)
            few = rng.random(S) < 0.02
            logit[few] = -rng.uniform(5.0, 60.0, size=int(few.sum()))
            live = np.flatnonzero(ages >= 0)
            top = live[np.argmin(ages[live])]  # the youngest live slot: protected
            logit[top] = 0.0
            k[b, h, :, 0] = logit
            ws[b, h] = int(rng.choice(live[ages[live] >= W]))
    new_k = rng.standard_normal((B, Hkv, d)).astype(np.float32)
    new_k[:, :, 0] = 0.0
    new_v = rng.standard_normal((B, Hkv, d)).astype(np.float32)
    return {"q": _bf16(q), "k_cache": _bf16(k), "v_cache": _bf16(v), "mask": mask,
            "new_k": _bf16(new_k), "new_v": _bf16(new_v), "write_slot": ws}


def random_peaked_case(rng, B, g, Hkv, d, S):
    """q, K, V ~ N(0, 1) (bf16); used with scale 3.0, logits spread over
    hundreds of nats."""
    n = lambda *s: _bf16(rng.standard_normal(s))
    mask = np.empty((B, Hkv, S), dtype=np.int32)
    ws = np.empty((B, Hkv), dtype=np.int32)
    for b in range(B):
        for h in range(Hkv):
            ages = rng.permutation(3 * S)[:S].astype(np.int32)
            ages[rng.random(S) < 0.05] = -1
            mask[b, h] = ages
            ws[b, h] = int(rng.choice(np.flatnonzero(ages >= 0)))
    return {"q": n(B, Hkv * g, d), "k_cache": n(B, Hkv, S, d), "v_cache": n(B, Hkv, S, d),
            "mask": mask, "new_k": n(B, Hkv, d), "new_v": n(B, Hkv, d), "write_slot": ws}


def run_gpu(case, W, scale, k=1, scores=True):
    B, Hkv, S, d = case["k_cache"].shape
    Hq = case["q"].shape[1]
    dc = {kk: to_dev(vv) for kk, vv in case.items()}
    out = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty((B, Hkv, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((B, Hkv, S), dtype=torch.float32, device="cuda") if scores else None
    flags = lf.LF_STEP_LOG2_SCORES if scores else 0
    if k == 1 and not scores:
        lf.decode_step(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                       dc["new_v"], dc["write_slot"], out, nxt.view(B, Hkv), W, scale)
    else:
        lf.decode_step_ex(dc["q"], dc["k_cache"], dc["v_cache"], dc["mask"], dc["new_k"],
                          dc["new_v"], dc["write_slot"], out, nxt, W, scale, k=k, flags=flags,
                          scores=sc)
    torch.cuda.synchronize()
    res = {"out": out.float().cpu().numpy().astype(np.float64),
           "next": nxt.cpu().numpy(), "mask": dc["mask"].cpu().numpy(),
           "k": to_host_bits(dc["k_cache"]), "v": to_host_bits(dc["v_cache"])}
    if scores:
        res["log2"] = sc.cpu().numpy().astype(np.float64)
    return res


def run_oracle(case, W, scale, k=1):
    c = {kk: np.array(vv, copy=True) for kk, vv in case.items()}
    ora = oracle.decode_step(c["q"], c["k_cache"], c["v_cache"], c["mask"], c["new_k"],
                             c["new_v"], c["write_slot"], W, scale, want_scores=True, topk=k)
    ora["state"] = c
    return ora


def fp32_linear_pick(scores, ages, W):
    """The slot a linear fp32 key would pick: scores below the normal range
    read 0 and tie to the lowest eligible index."""
    elig = np.flatnonzero(ages >= W)
    if elig.size == 0:
        return -1
    v = scores[elig]
    v = np.where(v < FP32_MIN_NORMAL, 0.0, v)
    return int(elig[np.lexsort((elig, v))[0]])


def check(case, W, scale, where, scores=True):
    gpu = run_gpu(case, W, scale, scores=scores)
    ora = run_oracle(case, W, scale)
    st = ora["state"]
    B, Hkv = st["mask"].shape[:2]
    g = case["q"].shape[1] // Hkv
    assert np.array_equal(gpu["mask"], st["mask"]), where
    assert np.array_equal(gpu["k"], st["k_cache"]) and np.array_equal(gpu["v"], st["v_cache"])
    gpu1 = {"out": gpu["out"], "next_slot": gpu["next"][:, :, 0]}
    deep = differs = 0
    for b in range(B):
        for h in range(Hkv):
            compare_unit(gpu1, ora, b, h, g, st["mask"], W, check_scores=False,
                         where=f"{where} unit ({b},{h})")
            ages = st["mask"][b, h]
            so = ora["scores"][b, h]
            n_o = int(ora["next_slot"][b, h])
            deep += int(n_o >= 0 and so[n_o] < 1e-40)
            differs += int(fp32_linear_pick(so, ages, W) != n_o)
            if scores:
                live = ages >= 0
                lg = gpu["log2"][b, h]
                assert np.all(np.isposinf(lg[~live])), f"{where}: masked slot has a score"
                pos = live & (so > 0)
                err = np.abs(lg[pos] - np.log2(so[pos]))
                assert err.size == 0 or err.max() <= LOG2_TOL, \
                    f"{where} unit ({b},{h}): log2 score error {err.max()}"
                assert np.all(np.isneginf(lg[live & (so == 0)])), f"{where}: zero score"
    assert lf.device_errors() == 0
    return deep, differs, B * Hkv


# (path name, environment switches, S, dead tail, scores exported)
PATHS = [
    ("last_cta_registers", {"LF_CLUSTER": "0", "LF_SPLIT": "0"}, 700, 0, False),
    ("last_cta_live_tiles", {"LF_CLUSTER": "0", "LF_SPLIT": "0"}, 2000, 900, False),
    ("last_cta_bulk", {"LF_CLUSTER": "0", "LF_SPLIT": "0"}, 6000, 0, False),
    ("last_cta_bulk_scores", {"LF_CLUSTER": "0", "LF_SPLIT": "0"}, 6000, 0, True),
    ("cluster", {"LF_CLUSTER": "1"}, 3000, 0, False),
    ("cluster_scores", {"LF_CLUSTER": "1"}, 3000, 0, True),
    ("split_finish", {"LF_CLUSTER": "0", "LF_SPLIT": "1"}, 9000, 0, False),
    ("split_finish_scores", {"LF_CLUSTER": "0", "LF_SPLIT": "1"}, 9000, 0, True),
]


@pytest.mark.parametrize("name,env,S,dead,scores", PATHS, ids=[p[0] for p in PATHS])
def test_selection_exact_below_fp32_range(monkeypatch, name, env, S, dead, scores):
    for kk, vv in env.items():
        monkeypatch.setenv(kk, vv)
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    W = 16
    case = peaked_case(rng, 2, 4, 2, 128, S, W, dead_tail=dead)
    deep, differs, units = check(case, W, 1.0, name, scores=scores)
    # The chosen slots score below 1e-40, where a linear fp32 key would pick
    # another slot: the case exercises what it is meant to.
    assert deep == units and differs >= units - 1


@pytest.mark.parametrize("d,g", [(64, 1), (128, 2), (64, 4), (128, 8)])
@pytest.mark.parametrize("cluster", ["0", "1"])
def test_every_group_size(monkeypatch, d, g, cluster):
    monkeypatch.setenv("LF_CLUSTER", cluster)
    rng = np.random.default_rng(100 * d + 10 * g + int(cluster))
    case = peaked_case(rng, 2, g, 2, d, 1500, 8)
    deep, differs, units = check(case, 8, 1.0, f"d={d} g={g} cluster={cluster}")
    assert deep == units and differs >= units - 1


@pytest.mark.parametrize("cluster,split", [("0", "0"), ("1", "0"), ("0", "1")])
def test_random_peaked_attention(monkeypatch, cluster, split):
    """N(0, 1) q and K at scale 3: logits spread over hundreds of nats, the
    minimum of each unit in the 1e-60 .. 1e-120 range."""
    monkeypatch.setenv("LF_CLUSTER", cluster)
    monkeypatch.setenv("LF_SPLIT", split)
    rng = np.random.default_rng(31 + 2 * int(cluster) + int(split))
    case = random_peaked_case(rng, 2, 4, 4, 128, 4000)
    deep, _, units = check(case, 32, 3.0, f"random cluster={cluster} split={split}")
    assert deep == units


def test_topk_below_fp32_range():
    """k = 8 at once: the radix select runs on the same log-domain keys."""
    rng = np.random.default_rng(808)
    W, k = 16, 8
    case = peaked_case(rng, 2, 4, 2, 128, 2500, W)
    gpu = run_gpu(case, W, 1.0, k=k, scores=True)
    ora = run_oracle(case, W, 1.0, k=k)
    ages = ora["state"]["mask"]
    for b in range(2):
        for h in range(2):
            ranked = _ranked(ora["scores"][b, h], ages[b, h], W, False)
            assert ranked[k - 1][1] < 1e-40  # every winner is below fp32's range
            compare_topk(gpu["next"][b, h], ranked, k, f"top-{k} unit ({b},{h})")
    assert np.max(np.abs(gpu["out"] - ora["out"])) <= OUT_ATOL
    assert lf.device_errors() == 0


def test_zero_v_slot_stays_the_minimum(monkeypatch):
    """A zero V row scores exactly 0 (log2: -inf) and stays below every
    underflowing score; two such slots tie to the lower index."""
    monkeypatch.setenv("LF_CLUSTER", "0")
    rng = np.random.default_rng(9)
    W = 8
    case = peaked_case(rng, 1, 4, 2, 128, 1200, W)
    for h, slots in ((0, [900, 301]), (1, [77])):
        for j in slots:
            case["mask"][0, h, j] = 500 + j
            case["v_cache"][0, h, j] = 0
        case["write_slot"][0, h] = 1100  # written, not one of the zero rows
    gpu = run_gpu(case, W, 1.0, scores=True)
    assert [int(x) for x in gpu["next"][0, :, 0]] == [301, 77]
    assert np.isneginf(gpu["log2"][0, 0, 301]) and np.isneginf(gpu["log2"][0, 0, 900])
    check(case, W, 1.0, "zero V")
