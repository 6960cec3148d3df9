"""The oracle against its pins (CPU only)."""
import pytest

import oracle
import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    if pin.__name__ in ("bwd_symbolic", "fused_bwd_symbolic"):
        pytest.importorskip("sympy")
    pin(oracle.default())


def test_oracle_thread_count_does_not_change_results():
    import numpy as np
    rng = np.random.default_rng(11)
    M, N = 37, 129
    x = rng.standard_normal((M, N))
    g = 1 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    _, rstd = oracle.rmsnorm_fwd(x, g, 1e-6)
    a = oracle.rmsnorm_bwd(x, g, dy, rstd, nthreads=1)
    b = oracle.rmsnorm_bwd(x, g, dy, rstd, nthreads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
