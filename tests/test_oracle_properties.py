"""Property-based sweep of the fp64 oracle against the pure-Python brute force
(CPU only): random tiny shapes over every group size, window, mask density,
write mode and selection option. The brute force computes the score through
(sum_h p) * ||v||_1, a softmax without max-shift, and selects by sorting, so
it shares no step with the oracle's materialised G."""
import numpy as np
import pytest

import oracle
import _pins

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402


def _same_selection(got, want, scores, where):
    """Exact, unless two candidates' brute-force scores tie to 1e-12."""
    if np.array_equal(got, want):
        return
    for a, b in zip(np.atleast_1d(got), np.atleast_1d(want)):
        if a == b:
            continue
        assert a >= 0 and b >= 0, where
        sa, sb = scores[a], scores[b]
        assert abs(sa - sb) <= 1e-12 * max(abs(sa), abs(sb), 1e-300), where


@settings(max_examples=150, deadline=None)
@given(seed=st.integers(0, 2**31 - 1), B=st.integers(1, 2), Hkv=st.integers(1, 2),
       g=st.sampled_from([1, 2, 4]), d=st.integers(1, 5), S=st.integers(1, 10),
       p_masked=st.sampled_from([0.0, 0.2, 0.6, 1.0]),
       ws_mode=st.sampled_from(["live", "any", "none"]),
       W=st.integers(0, 11), topk=st.sampled_from([1, 2, 3]),
       fill_first=st.booleans(), mask_evicted=st.booleans())
def test_oracle_matches_brute_force(seed, B, Hkv, g, d, S, p_masked, ws_mode, W, topk,
                                    fill_first, mask_evicted):
    rng = np.random.default_rng(seed)
    case = _pins.rand_case(rng, B, Hkv * g, Hkv, d, S, p_masked=p_masked, max_age=2 * S + 3,
                           ws_mode=ws_mode)
    scale = float(np.float32(0.5))
    res = _pins.run(oracle.decode_step, case, W, scale, want_scores=True, topk=topk,
                    fill_first=fill_first, mask_evicted=mask_evicted)
    ref = _pins.brute_force(case, W, scale, topk=topk, fill_first=fill_first,
                            mask_evicted=mask_evicted)
    np.testing.assert_allclose(res["out"], ref["out"], rtol=0, atol=1e-12)
    live = np.isfinite(ref["scores"])
    assert np.array_equal(np.isfinite(res["scores"]), live)
    np.testing.assert_allclose(res["scores"][live], ref["scores"][live], rtol=1e-12, atol=1e-14)
    for b in range(B):
        for h in range(Hkv):
            _same_selection(res["next_slot"][b, h], ref["next_slot"][b, h], ref["scores"][b, h],
                            f"unit ({b},{h})")
    if np.array_equal(res["next_slot"], ref["next_slot"]):
        assert np.array_equal(res["state"]["mask"], ref["mask"])
