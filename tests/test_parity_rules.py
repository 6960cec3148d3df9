"""The comparison rules themselves (CPU): the fp32 round-off escape of
tests/parity.py takes only ill-conditioned dx elements, and counts them."""
import numpy as np
import pytest

import parity


def _roundoff(bound, terms):
    def fn(mask):
        return np.full(int(mask.sum()), bound), np.full(int(mask.sum()), terms)
    return fn


def test_well_conditioned_element_cannot_use_the_escape():
    ref = np.array([1.0, 0.5, 0.25])
    got = ref.copy()
    got[1] += 3e-5          # beyond 1e-5 * max|ref| = 1e-5
    # generous round-off bound, but |dx| / terms = 0.5 / 1.0 is well conditioned
    with pytest.raises(AssertionError):
        parity.check_tensor("dx", got, ref, "f32", "dx", roundoff=_roundoff(1e-3, 1.0))


def test_ill_conditioned_element_passes_and_is_counted():
    ref = np.array([1e-9, 2e-9, 3e-9])
    got = ref + np.array([0.0, 5e-10, 0.0])   # far beyond 1e-5 * max|ref|
    # cancellation ratio 2e-9 / 1.0 is far below KAPPA_ILL; error within the bound
    n = parity.check_tensor("dx", got, ref, "f32", "dx", roundoff=_roundoff(1e-8, 1.0))
    assert n == 1


def test_ill_conditioned_element_beyond_the_round_off_bound_fails():
    ref = np.array([1e-9, 2e-9, 3e-9])
    got = ref + np.array([0.0, 5e-8, 0.0])
    with pytest.raises(AssertionError):
        parity.check_tensor("dx", got, ref, "f32", "dx", roundoff=_roundoff(1e-8, 1.0))


def test_bf16_escape_follows_the_same_rule():
    ref = np.array([1.0, 2.0 ** -20, 0.5])
    got = ref.copy()
    got[1] += 2.0 ** -15     # beyond 1 ulp of ref[1] + 1e-5 * max|ref|
    with pytest.raises(AssertionError):       # well conditioned (terms comparable to |ref|)
        parity.check_tensor("dx", got, ref, "bf16", "dx", roundoff=_roundoff(1.0, 2.0 ** -19))
    n = parity.check_tensor("dx", got, ref, "bf16", "dx", roundoff=_roundoff(1.0, 1.0))
    assert n == 1


def test_exact_results_use_no_escape():
    ref = np.linspace(-1, 1, 11)
    assert parity.check_tensor("dx", ref.copy(), ref, "f32", "dx",
                               roundoff=_roundoff(1.0, 1.0)) == 0
