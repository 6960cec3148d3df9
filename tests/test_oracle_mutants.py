"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutant is a textual edit of oracle/rmsnorm_oracle.c compiled into a
temporary library; the pins of oracle_pins.py then run against it. A mutant
that every pin accepts would mean the pins cannot see that kind of mistake.
"""
import os

import pytest

import oracle
from oracle import build as oracle_build
import oracle_pins

SRC = oracle_build.SRC

# (id, text to replace, replacement, which occurrence: None = the only one)
MUTANTS = [
    ("drop_c1_term", "double d = (wdy - x_hat * c1) * r;", "double d = wdy * r;", None),
    ("c1_sign", "double d = (wdy - x_hat * c1) * r;", "double d = (wdy + x_hat * c1) * r;", None),
    ("c1_divisor", "double c1 = acc / (double)N;", "double c1 = acc / (double)(N + 1);", None),
    ("dx_missing_rstd", "double d = (wdy - x_hat * c1) * r;", "double d = (wdy - x_hat * c1);", None),
    ("dweight_missing_rstd", "dweight[j] += dy[m * N + j] * x_hat;",
     "dweight[j] += dy[m * N + j] * x[m * N + j];", None),
    ("dweight_extra_gamma", "dweight[j] += dy[m * N + j] * x_hat;",
     "dweight[j] += dy[m * N + j] * x_hat * gamma[j];", None),
    ("dweight_wrong_row_rstd", "const double r = rstd[m];", "const double r = rstd[0];", 1),
    ("c1_gamma_reversed", "double wdy = dy[m * N + j] * gamma[j];",
     "double wdy = dy[m * N + j] * gamma[N - 1 - j];", 0),
    ("dx_gamma_transposed", "double wdy = dy[m * N + j] * gamma[j];",
     "double wdy = dy[m * N + j] * gamma[m % N];", 1),
    ("dres_dropped", "if (dres) d += dres[m * N + j];", "", None),
    ("dres_sign", "if (dres) d += dres[m * N + j];", "if (dres) d -= dres[m * N + j];", None),
    ("fwd_sum_not_mean", "double ms = ss / (double)N;", "double ms = ss;", None),
    ("fwd_eps_dropped", "double r = 1.0 / sqrt(ms + eps);", "double r = 1.0 / sqrt(ms);", None),
    ("fwd_eps_outside_sqrt", "double r = 1.0 / sqrt(ms + eps);",
     "double r = 1.0 / (sqrt(ms) + eps);", None),
    ("fwd_gamma_dropped", "y[m * N + j] = xr[j] * r * gamma[j];",
     "y[m * N + j] = xr[j] * r;", None),
    ("fused_fwd_no_rounding", "oracle_round1(x[m * N + j] + residual[m * N + j], dtype)",
     "(x[m * N + j] + residual[m * N + j])", None),
    ("round_ties_away", "double r = rint(v / quantum) * quantum;",
     "double r = round(v / quantum) * quantum;", None),
    ("round_f16_subnormal_quantum", "return round_format(v, 11, -14, 65504.0);",
     "return round_format(v, 11, -15, 65504.0);", None),
    ("round_bf16_precision", "return round_format(v, 8, -126,", "return round_format(v, 9, -126,",
     None),
    ("round_no_overflow", "if (fabs(r) > maxf) return v > 0 ? INFINITY : -INFINITY;", "", None),
    # LayerNorm
    ("ln_mean_divisor", "double mu = s / (double)N;", "double mu = s / (double)(N - 1);", None),
    ("ln_var_unbiased", "double var = v / (double)N;", "double var = v / (double)(N - 1);", None),
    ("ln_var_uncentred", "v += (xr[j] - mu) * (xr[j] - mu);", "v += xr[j] * xr[j];", None),
    ("ln_fwd_uncentred", "double yv = (xr[j] - mu) * r * gamma[j];",
     "double yv = xr[j] * r * gamma[j];", None),
    ("ln_fwd_beta_dropped", "if (beta) yv += beta[j];", "", None),
    ("ln_drop_c2", "dx[m * N + j] = (wdy - c2 - x_hat * c1) * r;",
     "dx[m * N + j] = (wdy - x_hat * c1) * r;", None),
    ("ln_c2_sign", "dx[m * N + j] = (wdy - c2 - x_hat * c1) * r;",
     "dx[m * N + j] = (wdy + c2 - x_hat * c1) * r;", None),
    ("ln_drop_c1", "dx[m * N + j] = (wdy - c2 - x_hat * c1) * r;",
     "dx[m * N + j] = (wdy - c2) * r;", None),
    ("ln_c2_divisor", "double c2 = a2 / (double)N;", "double c2 = a2 / (double)(N + 1);", None),
    ("ln_c1_uncentred", "double x_hat = (x[m * N + j] - mu) * r;",
     "double x_hat = x[m * N + j] * r;", 0),
    ("ln_dx_uncentred", "double x_hat = (x[m * N + j] - mu) * r;",
     "double x_hat = x[m * N + j] * r;", 1),
    ("ln_dgamma_uncentred", "double x_hat = (x[m * N + j] - mu) * r;",
     "double x_hat = x[m * N + j] * r;", 2),
    ("ln_dgamma_extra_gamma", "dgamma[j] += dy[m * N + j] * x_hat;",
     "dgamma[j] += dy[m * N + j] * x_hat * gamma[j];", None),
    ("ln_dbeta_times_xhat", "dbeta[j] += dy[m * N + j];", "dbeta[j] += dy[m * N + j] * x_hat;",
     None),
    ("ln_c2_ungamma", "a2 += wdy;", "a2 += dy[m * N + j];", None),
]


def _mutate(src, old, new, occ):
    n = src.count(old)
    if occ is None:
        assert n == 1, "mutation anchor %r occurs %d times" % (old, n)
        return src.replace(old, new)
    assert n > occ, "mutation anchor %r occurs %d times" % (old, n)
    idx = -1
    for _ in range(occ + 1):
        idx = src.index(old, idx + 1)
    return src[:idx] + new + src[idx + len(old):]


@pytest.mark.parametrize("mid,old,new,occ", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, mid, old, new, occ):
    with open(SRC) as f:
        src = f.read()
    mutated = _mutate(src, old, new, occ)
    assert mutated != src
    cpath = os.path.join(tmp_path, "mutant.c")
    with open(cpath, "w") as f:
        f.write(mutated)
    lib = oracle_build.compile_c(cpath, os.path.join(tmp_path, "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
            caught.append(pin.__name__)
        except ImportError:
            pass
    assert caught, "mutant %s passed every pin" % mid
