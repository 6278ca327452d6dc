"""Planted mistakes: broken copies of the oracle, built on the CPU, must each
fail at least one of the pins. This shows the pins would catch a dropped
term, a wrong sign, a wrong index or a swapped operand in the oracle."""
import os
import subprocess

import pytest

import oracle
import _pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "lf_oracle.c")

# (name, text in lf_oracle.c, replacement)
MUTANTS = [
    ("v_replaced_by_k_in_G", "p[j] * bf16_to_double(V[", "p[j] * bf16_to_double(K["),
    ("dropped_normaliser", "l += p[j];", "l += 0.0 * p[j] + 1.0;"),
    ("wrong_sign_in_exp", "exp(s[j] - smax)", "exp(smax - s[j])"),
    ("strided_gqa_grouping", "const int hq = kvh * g + h;", "const int hq = h * Hkv + kvh;"),
    ("score_without_abs", "acc += fabs(G[", "acc += (G["),
    ("protected_window_off_by_one", "age[j] >= 0 && age[j] >= W) {", "age[j] >= 0 && age[j] > W) {"),
    ("ties_to_highest_index", "return (a->slot > b->slot) - (a->slot < b->slot);",
     "return (a->slot < b->slot) - (a->slot > b->slot);"),
    ("highest_scores_selected", "return a->score < b->score ? -1 : 1;", "return a->score < b->score ? 1 : -1;"),
    ("empty_slots_ranked_last", "cand[nc].cls = 0;", "cand[nc].cls = 2;"),
    ("evicted_slots_not_masked", "if (slot >= 0 && opt->mask_evicted) age[slot] = -1;", "if (0) age[slot] = -1;"),
    ("topk_list_shifted", "const int slot = (i < nc) ? cand[i].slot : -1;",
     "const int slot = (i + 1 < nc) ? cand[i + 1].slot : -1;"),
    ("attention_only_resets_live_age", "if (age[ws] < 0) age[ws] = 0;", "age[ws] = 0;"),
    ("attention_only_still_ages", "if (opt->attention_only) {\n            /* Attention alone",
     "if (0) {\n            /* Attention alone"),
    ("no_ageing", "age[j] += 1;", "age[j] += 0;"),
    ("new_k_not_written", "memcpy(K + (size_t)ws * d, new_k", "if (0) memcpy(K + (size_t)ws * d, new_k"),
    ("new_v_not_written", "memcpy(V + (size_t)ws * d, new_v", "if (0) memcpy(V + (size_t)ws * d, new_v"),
    ("score_from_unnormalised_weights", "I[j] += acc;", "I[j] += acc * l;"),
    ("missing_scale", "s[j] = scale * acc;", "s[j] = acc;"),
    ("masked_slot_attended", "if (age[j] < 0) continue;\n            double acc = 0.0;\n            for (int c = 0; c < d; ++c)\n                acc += bf16",
     "double acc = 0.0;\n            for (int c = 0; c < d; ++c)\n                acc += bf16"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as fh:
        return fh.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) >= 1, f"mutation anchor for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new, 1))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(src), "-lm"], check=True, capture_output=True)
    lib = oracle.bind_library(str(so))
    step = lambda *a, **k: oracle.decode_step(*a, lib=lib, **k)
    failures = 0
    for check in _pins.ALL_CHECKS:
        try:
            check(step)
        except (AssertionError, ValueError, FloatingPointError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake {name}"
