"""CPU oracle for RMSNorm forward / backward (plain and fused-add) and for
LayerNorm forward / backward, fp64.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs are the only callers.
The CUDA library and its Python binding never import this package, and this
package imports nothing from them.

This module is argument marshalling over ``rmsnorm_oracle.c`` (numpy float64
arrays in, float64 arrays out); all arithmetic lives in the C file, which
cites the FlyDSL pages it follows (issue #769 "Math" section; PR #800
"What's included"; for LayerNorm, issue #769's plan, which mirrors the RMSNorm
backward with mean handling and dbias -- the formulas are the textbook ones).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
(symbolic gradients, finite differences, the closed-form invariant, library
cross-checks, hand-worked fixtures) and ``tests/test_oracle_mutants.py``
(each planted mistake in the C source fails at least one pin).
"""
import ctypes

import numpy as np

from . import build as _build

F32, F16, BF16 = 0, 1, 2
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16}

_dp = ctypes.POINTER(ctypes.c_double)


def _arr(a, shape=None):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if shape is not None and a.shape != shape:
        raise ValueError("expected shape %s, got %s" % (shape, a.shape))
    return a


def _p(a):
    return a.ctypes.data_as(_dp) if a is not None else None


def _code(dtype):
    return DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)


class Oracle:
    """The oracle's functions, bound to one compiled copy of the C source."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        i64, dbl, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_int
        lib.oracle_round1.argtypes = [dbl, ci]
        lib.oracle_round1.restype = dbl
        lib.oracle_round.argtypes = [_dp, _dp, i64, ci]
        lib.oracle_max_threads.restype = ci
        lib.oracle_rmsnorm_fwd.argtypes = [_dp, _dp, dbl, i64, i64, _dp, _dp, ci]
        lib.oracle_fused_add_rmsnorm_fwd.argtypes = [_dp, _dp, _dp, dbl, i64, i64, ci,
                                                     _dp, _dp, _dp, ci]
        lib.oracle_rmsnorm_bwd.argtypes = [_dp, _dp, _dp, _dp, i64, i64, _dp, _dp, ci]
        lib.oracle_fused_add_rmsnorm_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, i64, i64,
                                                     _dp, _dp, ci]
        lib.oracle_layernorm_fwd.argtypes = [_dp, _dp, _dp, dbl, i64, i64, _dp, _dp, _dp, ci]
        lib.oracle_layernorm_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, i64, i64, _dp, _dp, _dp,
                                             ci]
        self._lib = lib
        self.path = libpath

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def round_to(self, a, dtype):
        """Round each fp64 value to the nearest `dtype` value (ties to even), as fp64."""
        a = _arr(a)
        out = np.empty_like(a)
        self._lib.oracle_round(_p(a), _p(out), a.size, _code(dtype))
        return out

    def rmsnorm_fwd(self, x, gamma, eps, nthreads=0):
        """Return (y, rstd) in fp64; rstd unrounded."""
        x = _arr(x)
        M, N = x.shape
        g = _arr(gamma, (N,))
        y = np.empty_like(x)
        rstd = np.empty(M, np.float64)
        self._lib.oracle_rmsnorm_fwd(_p(x), _p(g), float(eps), M, N, _p(y), _p(rstd), nthreads)
        return y, rstd

    def fused_add_rmsnorm_fwd(self, x, residual, gamma, eps, dtype, nthreads=0):
        """Return (out, residual_out, rstd) in fp64; residual_out is dtype-rounded."""
        x = _arr(x)
        M, N = x.shape
        r = _arr(residual, (M, N))
        g = _arr(gamma, (N,))
        out = np.empty_like(x)
        res_out = np.empty_like(x)
        rstd = np.empty(M, np.float64)
        self._lib.oracle_fused_add_rmsnorm_fwd(_p(x), _p(r), _p(g), float(eps), M, N,
                                               _code(dtype), _p(out), _p(res_out), _p(rstd),
                                               nthreads)
        return out, res_out, rstd

    def rmsnorm_bwd(self, x, gamma, dy, rstd, nthreads=0):
        """Return (dx, dweight) in fp64 from the given saved rstd."""
        x = _arr(x)
        M, N = x.shape
        g = _arr(gamma, (N,))
        d = _arr(dy, (M, N))
        r = _arr(rstd, (M,))
        dx = np.empty_like(x)
        dw = np.empty(N, np.float64)
        self._lib.oracle_rmsnorm_bwd(_p(x), _p(g), _p(d), _p(r), M, N, _p(dx), _p(dw), nthreads)
        return dx, dw

    def fused_add_rmsnorm_bwd(self, added, gamma, dy, rstd, dresidual_out=None, nthreads=0):
        """Return (dx, dweight) in fp64; dx is also dresidual. dresidual_out may be None."""
        a = _arr(added)
        M, N = a.shape
        g = _arr(gamma, (N,))
        d = _arr(dy, (M, N))
        r = _arr(rstd, (M,))
        dres = _arr(dresidual_out, (M, N)) if dresidual_out is not None else None
        dx = np.empty_like(a)
        dw = np.empty(N, np.float64)
        self._lib.oracle_fused_add_rmsnorm_bwd(_p(a), _p(g), _p(d), _p(r), _p(dres), M, N,
                                               _p(dx), _p(dw), nthreads)
        return dx, dw

    def layernorm_fwd(self, x, gamma, beta, eps, nthreads=0):
        """Return (y, mean, rstd) in fp64; beta may be None (no bias)."""
        x = _arr(x)
        M, N = x.shape
        g = _arr(gamma, (N,))
        b = _arr(beta, (N,)) if beta is not None else None
        y = np.empty_like(x)
        mean = np.empty(M, np.float64)
        rstd = np.empty(M, np.float64)
        self._lib.oracle_layernorm_fwd(_p(x), _p(g), _p(b), float(eps), M, N, _p(y), _p(mean),
                                       _p(rstd), nthreads)
        return y, mean, rstd

    def layernorm_bwd(self, x, gamma, dy, mean, rstd, nthreads=0):
        """Return (dx, dgamma, dbeta) in fp64 from the given saved mean and rstd."""
        x = _arr(x)
        M, N = x.shape
        g = _arr(gamma, (N,))
        d = _arr(dy, (M, N))
        mu = _arr(mean, (M,))
        r = _arr(rstd, (M,))
        dx = np.empty_like(x)
        dg = np.empty(N, np.float64)
        db = np.empty(N, np.float64)
        self._lib.oracle_layernorm_bwd(_p(x), _p(g), _p(d), _p(mu), _p(r), M, N, _p(dx), _p(dg),
                                       _p(db), nthreads)
        return dx, dg, db


_default = None


def default() -> Oracle:
    """The oracle built from ``rmsnorm_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def max_threads():
    return default().max_threads()


def round_to(a, dtype):
    return default().round_to(a, dtype)


def rmsnorm_fwd(x, gamma, eps, nthreads=0):
    return default().rmsnorm_fwd(x, gamma, eps, nthreads)


def fused_add_rmsnorm_fwd(x, residual, gamma, eps, dtype, nthreads=0):
    return default().fused_add_rmsnorm_fwd(x, residual, gamma, eps, dtype, nthreads)


def rmsnorm_bwd(x, gamma, dy, rstd, nthreads=0):
    return default().rmsnorm_bwd(x, gamma, dy, rstd, nthreads)


def fused_add_rmsnorm_bwd(added, gamma, dy, rstd, dresidual_out=None, nthreads=0):
    return default().fused_add_rmsnorm_bwd(added, gamma, dy, rstd, dresidual_out, nthreads)


def layernorm_fwd(x, gamma, beta, eps, nthreads=0):
    return default().layernorm_fwd(x, gamma, beta, eps, nthreads)


def layernorm_bwd(x, gamma, dy, mean, rstd, nthreads=0):
    return default().layernorm_bwd(x, gamma, dy, mean, rstd, nthreads)
