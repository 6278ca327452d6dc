"""The fp64 oracle against brute force, closed forms, library routines,
hand-worked fixtures and invariants (CPU only)."""
import pytest

import oracle
import _pins


@pytest.mark.parametrize("check", _pins.ALL_CHECKS,
                         ids=[getattr(c, "__name__", f"golden{i}") for i, c in enumerate(_pins.ALL_CHECKS)])
def test_oracle_pin(check):
    check(oracle.decode_step)


def test_oracle_rejects_bad_arguments():
    import numpy as np
    z16 = lambda *s: np.zeros(s, dtype=np.uint16)
    with pytest.raises(ValueError):
        # Hq not a multiple of Hkv
        oracle.decode_step(z16(1, 3, 4), z16(1, 2, 5, 4), z16(1, 2, 5, 4),
                           np.zeros((1, 2, 5), np.int32), z16(1, 2, 4), z16(1, 2, 4),
                           np.zeros((1, 2), np.int32), 0, 1.0)
    with pytest.raises(ValueError):
        oracle.decode_step(z16(1, 2, 4), z16(1, 2, 5, 4), z16(1, 2, 5, 4),
                           np.zeros((1, 2, 5), np.int32), z16(1, 2, 4), z16(1, 2, 4),
                           np.zeros((1, 2), np.int32), -1, 1.0)


def test_oracle_unit_subset_matches_full():
    import numpy as np
    rng = np.random.default_rng(0)
    case = _pins.rand_case(rng, 3, 4, 2, 8, 30)
    full = _pins.run(oracle.decode_step, case, 2, 0.3, want_scores=True)
    sub = _pins.run(oracle.decode_step, case, 2, 0.3, want_scores=True, units=[1, 4])
    for u in (1, 4):
        b, h = divmod(u, 2)
        np.testing.assert_array_equal(sub["out"][b, h * 2:(h + 1) * 2], full["out"][b, h * 2:(h + 1) * 2])
        assert sub["next_slot"][b, h] == full["next_slot"][b, h]
        np.testing.assert_array_equal(sub["state"]["mask"][b, h], full["state"]["mask"][b, h])
    assert sub["next_slot"][0, 0] == -2  # untouched unit
