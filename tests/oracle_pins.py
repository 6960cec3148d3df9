"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each pin is a function of an ``Oracle`` instance and raises AssertionError on
failure, so the same pins run against the real oracle (test_oracle_pins.py)
and against copies with planted mistakes (test_oracle_mutants.py).

What each pin ties the oracle to:
  * round_*          -- torch / numpy dtype casts (library routines) and
                        hand-worked double-rounding cases
  * fwd_*            -- torch.nn.functional.rms_norm in fp64 (library)
  * bwd_symbolic     -- sympy's exact derivative of L = sum(y*dy), with y
                        typed from the forward definition only
  * bwd_fd           -- central finite differences of the same L
  * bwd_invariant    -- closed form sum_j x_j*dx_j = eps*rstd^3*sum_j x_j*g_j*dy_j
  * bwd_torch_autograd -- torch fp64 autograd of rms_norm (the pages' own check)
  * hand_cases       -- tests/golden/rmsnorm_hand_cases.txt (worked on paper)
  * special cases    -- fused with residual = 0, dres = 0 is plain; exact
                        power-of-two scaling; row permutation
  * ln_*             -- LayerNorm: torch fp64 layer_norm and its autograd,
                        numpy mean/var, sympy's exact derivative, finite
                        differences, the per-row invariants sum dx = 0 and
                        sum x_hat*dx = N*eps*c1*rstd^3, zero-mean rows reducing
                        to RMSNorm, shift invariance, and
                        tests/golden/layernorm_hand_cases.txt
"""
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "rmsnorm_hand_cases.txt")


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / scale)


# ----------------------------------------------------------------- rounding
def _tie_patterns_f32(rng, n):
    """fp32 values: random normals, ties for bf16 and f16, subnormal f16 ties, edges."""
    vals = [rng.standard_normal(n).astype(np.float32)]
    bits = rng.integers(0, 2**31, size=n, dtype=np.int64).astype(np.uint32)
    bits = (bits & np.uint32(0x7F7F0000)) | np.uint32(0x8000)  # exact bf16 ties
    vals.append(bits.view(np.float32) * np.float32(1e-30))   # scale keeps it finite
    vals.append(bits.view(np.float32))
    b16 = (rng.integers(0x38000000, 0x47000000, size=n, dtype=np.int64).astype(np.uint32)
           & np.uint32(0xFFFFE000)) | np.uint32(0x1000)       # exact f16 ties (normal range)
    vals.append(b16.view(np.float32))
    k = rng.integers(1, 2000, size=n) * 2 + 1
    vals.append((k * 2.0**-25).astype(np.float32))            # f16 subnormal ties
    vals.append(np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 65536.0, -65520.0,
                          6.1035156e-05, 5.9604645e-08, 2.9802322e-08, 2.9802326e-08,
                          3.3895314e38, 3.3961775e38, 1.0 + 2**-8, 1.0 + 3 * 2**-8,
                          1e-40, -1e-41], np.float32))
    v = np.concatenate(vals)
    return v[np.isfinite(v)]


def round_vs_torch_casts(orc):
    rng = np.random.default_rng(1)
    v32 = _tie_patterns_f32(rng, 4000)
    t = torch.from_numpy(v32)
    for name, dt in (("bf16", torch.bfloat16), ("f16", torch.float16), ("f32", torch.float32)):
        want = t.to(dt).to(torch.float64).numpy()
        got = orc.round_to(v32.astype(np.float64), name)
        assert np.array_equal(got, want), "rounding to %s disagrees with torch" % name


def round_direct_from_double(orc):
    # numpy rounds float64 -> float32 / float16 directly (one rounding)
    rng = np.random.default_rng(2)
    base = rng.standard_normal(3000) * 10.0
    f32 = base.astype(np.float32).astype(np.float64)
    ulp32 = np.spacing(np.abs(base.astype(np.float32))).astype(np.float64)
    near = np.concatenate([base, f32 + 0.5 * ulp32, f32 - 0.5 * ulp32,
                           f32 + 0.5 * ulp32 * (1 + 2**-20)])
    assert np.array_equal(orc.round_to(near, "f32"), near.astype(np.float32).astype(np.float64))
    f16 = base.astype(np.float16).astype(np.float64)
    ulp16 = np.spacing(np.abs(base.astype(np.float16))).astype(np.float64)
    near16 = np.concatenate([base, f16 + 0.5 * ulp16, f16 + 0.5 * ulp16 * (1 + 2**-30),
                             f16 - 0.5 * ulp16 * (1 + 2**-30)])
    assert np.array_equal(orc.round_to(near16, "f16"),
                          near16.astype(np.float16).astype(np.float64))
    # bf16 from double, worked by hand (spacing of bf16 in [1,2) is 2^-7):
    cases = [
        (1 + 2**-8 + 2**-30, 1 + 2**-7),   # just above the tie -> up (via f32 it would tie to 1)
        (1 + 2**-8, 1.0),                  # exact tie, 1.0 has the even significand
        (1 + 3 * 2**-8, 1 + 2**-6),        # exact tie between 1+2^-7 (odd) and 1+2^-6 (even)
        (1 + 2**-8 - 2**-40, 1.0),         # just below the tie
        (-(1 + 2**-8 + 2**-30), -(1 + 2**-7)),
        (2.0**-133, 2.0**-133),            # smallest bf16 subnormal
        (2.0**-134, 0.0),                  # half of it: tie to even (zero)
        (3 * 2.0**-134, 2 * 2.0**-133),    # 1.5 quanta: tie to even (2 quanta)
        (3.39e38, 3.3895313892515355e38),  # below the top midpoint -> largest finite
        (3.3962e38, float("inf")),         # above (2 - 2^-8) * 2^127 -> overflows
    ]
    got = orc.round_to(np.array([c[0] for c in cases]), "bf16")
    want = np.array([c[1] for c in cases])
    assert np.array_equal(got, want), (got, want)


# ------------------------------------------------------------------ forward
def fwd_vs_torch_rms_norm(orc):
    rng = np.random.default_rng(3)
    for (M, N, eps) in ((5, 7, 1e-5), (3, 64, 1e-2), (2, 300, 1e-6)):
        x = rng.standard_normal((M, N))
        g = 1 + 0.1 * rng.standard_normal(N)
        y, rstd = orc.rmsnorm_fwd(x, g, eps)
        yt = torch.nn.functional.rms_norm(torch.from_numpy(x), (N,), torch.from_numpy(g), eps)
        assert _rel(y, yt.numpy()) < 1e-13
        # rstd tied to the library's output: y = x * rstd * g (read at each row's largest |x|)
        yu = torch.nn.functional.rms_norm(torch.from_numpy(x), (N,), None, eps).numpy()
        jmax = np.argmax(np.abs(x), axis=1)
        rows = np.arange(M)
        assert _rel(rstd, yu[rows, jmax] / x[rows, jmax]) < 1e-13


def fused_fwd_vs_torch(orc):
    rng = np.random.default_rng(4)
    M, N, eps = 4, 40, 1e-6
    for name, dt in (("bf16", torch.bfloat16), ("f16", torch.float16), ("f32", torch.float32)):
        xt = torch.from_numpy(rng.standard_normal((M, N))).to(dt)
        rt = torch.from_numpy(rng.standard_normal((M, N))).to(dt)
        gt = torch.from_numpy(1 + 0.1 * rng.standard_normal(N)).to(dt)
        x, r, g = (t.to(torch.float64).numpy() for t in (xt, rt, gt))
        out, res_out, rstd = orc.fused_add_rmsnorm_fwd(x, r, g, eps, name)
        # residual_out: torch adds two dtype tensors with one rounding to dtype
        assert np.array_equal(res_out, (xt + rt).to(torch.float64).numpy()), name
        ya = torch.nn.functional.rms_norm(torch.from_numpy(res_out), (N,),
                                          torch.from_numpy(g), eps).numpy()
        assert _rel(out, ya) < 1e-13, name


# ----------------------------------------------------------------- backward
def _sym_grads(M, N, x, g, dy, eps, r=None, dres=None):
    """Exact gradients of L = sum(y*dy) [+ sum(added*dres)], y from the forward
    definition rstd = (mean x^2 + eps)^(-1/2), y = x*rstd*g (sympy)."""
    import sympy as sp
    X = sp.Matrix(M, N, lambda i, j: sp.Symbol("x_%d_%d" % (i, j)))
    G = [sp.Symbol("g_%d" % j) for j in range(N)]
    R = sp.Matrix(M, N, lambda i, j: sp.Symbol("r_%d_%d" % (i, j))) if r is not None else None
    A = X + R if R is not None else X
    L = 0
    for i in range(M):
        ms = sum(A[i, j] ** 2 for j in range(N)) / N
        rs = (ms + eps) ** sp.Rational(-1, 2)
        for j in range(N):
            L += A[i, j] * rs * G[j] * dy[i][j]
            if dres is not None:
                L += A[i, j] * dres[i][j]
    subs = {X[i, j]: x[i][j] for i in range(M) for j in range(N)}
    subs.update({G[j]: g[j] for j in range(N)})
    if R is not None:
        subs.update({R[i, j]: r[i][j] for i in range(M) for j in range(N)})
    dX = np.array([[float(sp.diff(L, X[i, j]).subs(subs).evalf(30)) for j in range(N)]
                   for i in range(M)])
    dG = np.array([float(sp.diff(L, G[j]).subs(subs).evalf(30)) for j in range(N)])
    dR = None
    if R is not None:
        dR = np.array([[float(sp.diff(L, R[i, j]).subs(subs).evalf(30)) for j in range(N)]
                       for i in range(M)])
    return dX, dG, dR


def bwd_symbolic(orc):
    import sympy as sp
    Q = sp.Rational
    M, N = 2, 3
    x = [[Q(1, 2), Q(-3, 4), Q(2)], [Q(5, 4), Q(1, 8), Q(-1)]]
    g = [Q(9, 10), Q(11, 10), Q(5, 4)]
    dy = [[Q(1), Q(-2), Q(1, 2)], [Q(3, 4), Q(1, 4), Q(-1)]]
    eps = Q(1, 100)
    dX, dG, _ = _sym_grads(M, N, x, g, dy, eps)
    f = lambda a: np.array(a, dtype=np.float64)
    rstd = np.array([float((sum(v ** 2 for v in row) / N + eps) ** Q(-1, 2)) for row in x])
    dx, dw = orc.rmsnorm_bwd(f(x), f(g), f(dy), rstd)
    assert _rel(dx, dX) < 1e-13 and _rel(dw, dG) < 1e-13, (dx, dX, dw, dG)


def fused_bwd_symbolic(orc):
    import sympy as sp
    Q = sp.Rational
    M, N = 2, 3
    x = [[Q(1, 2), Q(-3, 4), Q(2)], [Q(5, 4), Q(1, 8), Q(-1)]]
    r = [[Q(1, 4), Q(1, 2), Q(-1)], [Q(-1, 2), Q(3, 8), Q(3)]]
    g = [Q(9, 10), Q(11, 10), Q(5, 4)]
    dy = [[Q(1), Q(-2), Q(1, 2)], [Q(3, 4), Q(1, 4), Q(-1)]]
    dres = [[Q(1, 3), Q(0), Q(-1, 5)], [Q(2), Q(-1, 7), Q(1, 9)]]
    eps = Q(1, 50)
    dX, dG, dR = _sym_grads(M, N, x, g, dy, eps, r=r, dres=dres)
    f = lambda a: np.array(a, dtype=np.float64)
    added = [[x[i][j] + r[i][j] for j in range(N)] for i in range(M)]
    rstd = np.array([float((sum(v ** 2 for v in row) / N + eps) ** Q(-1, 2)) for row in added])
    dres_f = np.array([[float(v) for v in row] for row in dres])
    dx, dw = orc.fused_add_rmsnorm_bwd(f(added), f(g), f(dy), rstd, dres_f)
    # d/dx and d/dresidual are the same tensor (added = x + residual)
    assert _rel(dx, dX) < 1e-13 and _rel(dx, dR) < 1e-13 and _rel(dw, dG) < 1e-13


def _loss(orc, x, g, dy, eps, dres=None):
    y, _ = orc.rmsnorm_fwd(x, g, eps)
    L = float(np.sum(y * dy))
    if dres is not None:
        L += float(np.sum(x * dres))
    return L


def bwd_fd(orc):
    rng = np.random.default_rng(5)
    for (M, N, eps) in ((3, 16, 1e-5), (2, 5, 1e-2), (4, 9, 0.0)):
        x = rng.standard_normal((M, N))
        g = 1 + 0.1 * rng.standard_normal(N)
        dy = rng.standard_normal((M, N))
        _, rstd = orc.rmsnorm_fwd(x, g, eps)
        dx, dw = orc.rmsnorm_bwd(x, g, dy, rstd)
        h = 1e-6
        fdx = np.zeros_like(x)
        for i in range(M):
            for j in range(N):
                xp, xm = x.copy(), x.copy()
                xp[i, j] += h
                xm[i, j] -= h
                fdx[i, j] = (_loss(orc, xp, g, dy, eps) - _loss(orc, xm, g, dy, eps)) / (2 * h)
        fdg = np.zeros(N)
        for j in range(N):
            gp, gm = g.copy(), g.copy()
            gp[j] += h
            gm[j] -= h
            fdg[j] = (_loss(orc, x, gp, dy, eps) - _loss(orc, x, gm, dy, eps)) / (2 * h)
        assert _rel(dx, fdx) < 1e-6 and _rel(dw, fdg) < 1e-6


def fused_bwd_fd(orc):
    """L(added) = sum(rmsnorm(added)*dy) + sum(added*dres); since added = x + residual,
    dL/dx = dL/dresidual = dL/dadded, which the fused backward returns as dx."""
    rng = np.random.default_rng(6)
    M, N, eps = 3, 12, 1e-5
    a = rng.standard_normal((M, N))
    g = 1 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    dres = rng.standard_normal((M, N))
    _, rstd = orc.rmsnorm_fwd(a, g, eps)
    for dr in (dres, None):
        dx, dw = orc.fused_add_rmsnorm_bwd(a, g, dy, rstd, dr)
        h = 1e-6
        fda = np.zeros_like(a)
        for i in range(M):
            for j in range(N):
                ap, am = a.copy(), a.copy()
                ap[i, j] += h
                am[i, j] -= h
                fda[i, j] = (_loss(orc, ap, g, dy, eps, dr) - _loss(orc, am, g, dy, eps, dr)) / (2 * h)
        fdg = np.zeros(N)
        for j in range(N):
            gp, gm = g.copy(), g.copy()
            gp[j] += h
            gm[j] -= h
            fdg[j] = (_loss(orc, a, gp, dy, eps, dr) - _loss(orc, a, gm, dy, eps, dr)) / (2 * h)
        assert _rel(dx, fda) < 1e-6 and _rel(dw, fdg) < 1e-6


def bwd_invariant(orc):
    """sum_j x_j*dx_j = eps*rstd^3*sum_j x_j*g_j*dy_j when rstd = (ms+eps)^-1/2
    (derivation: sum x*dx = rstd*S - c1*rstd^2*N*ms with S = sum x*g*dy and
    c1 = rstd*S/N, i.e. rstd*S*(1 - ms/(ms+eps)))."""
    rng = np.random.default_rng(7)
    M, N = 6, 50
    x = rng.standard_normal((M, N))
    g = 1 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    for eps in (1e-1, 1e-2, 1e-5, 0.0):
        _, rstd = orc.rmsnorm_fwd(x, g, eps)
        dx, _ = orc.rmsnorm_bwd(x, g, dy, rstd)
        lhs = np.sum(x * dx, axis=1)
        S = np.sum(x * g * dy, axis=1)
        rhs = eps * rstd ** 3 * S
        scale = np.sum(np.abs(x * dx), axis=1)
        assert np.all(np.abs(lhs - rhs) <= 1e-13 * scale + 1e-300), (eps, lhs, rhs)


def bwd_torch_autograd(orc):
    rng = np.random.default_rng(8)
    M, N, eps = 16, 300, 1e-6
    x = rng.standard_normal((M, N))
    g = 1 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    xt = torch.from_numpy(x).requires_grad_(True)
    gt = torch.from_numpy(g).requires_grad_(True)
    y = torch.nn.functional.rms_norm(xt, (N,), gt, eps)
    y.backward(torch.from_numpy(dy))
    _, rstd = orc.rmsnorm_fwd(x, g, eps)
    dx, dw = orc.rmsnorm_bwd(x, g, dy, rstd)
    assert _rel(dx, xt.grad.numpy()) < 1e-12 and _rel(dw, gt.grad.numpy()) < 1e-12


def fused_reduces_to_plain(orc):
    rng = np.random.default_rng(9)
    M, N, eps = 4, 33, 1e-6
    x = rng.standard_normal((M, N)).astype(np.float32).astype(np.float64)
    g = (1 + 0.1 * rng.standard_normal(N)).astype(np.float32).astype(np.float64)
    dy = rng.standard_normal((M, N))
    y, rstd = orc.rmsnorm_fwd(x, g, eps)
    out, res_out, rstd2 = orc.fused_add_rmsnorm_fwd(x, np.zeros_like(x), g, eps, "f32")
    assert np.array_equal(res_out, x) and np.array_equal(out, y) and np.array_equal(rstd, rstd2)
    dx, dw = orc.rmsnorm_bwd(x, g, dy, rstd)
    for dres in (None, np.zeros_like(x)):
        dx2, dw2 = orc.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres)
        assert np.array_equal(dx, dx2) and np.array_equal(dw, dw2)


def scaling_and_permutation(orc):
    rng = np.random.default_rng(10)
    M, N = 5, 24
    x = rng.standard_normal((M, N))
    g = 1 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    _, rstd = orc.rmsnorm_fwd(x, g, 1e-6)
    dx, dw = orc.rmsnorm_bwd(x, g, dy, rstd)
    dx2, dw2 = orc.rmsnorm_bwd(x, g, dy * 8.0, rstd)        # dy * 2^3 scales exactly
    assert np.array_equal(dx2, dx * 8.0) and np.array_equal(dw2, dw * 8.0)
    # eps = 0: scaling x by 2^k leaves x_hat alone and scales dx by 2^-k
    _, r0 = orc.rmsnorm_fwd(x, g, 0.0)
    dxa, dwa = orc.rmsnorm_bwd(x, g, dy, r0)
    _, r4 = orc.rmsnorm_fwd(x * 4.0, g, 0.0)
    dxb, dwb = orc.rmsnorm_bwd(x * 4.0, g, dy, r4)
    assert _rel(dxb * 4.0, dxa) < 1e-14 and _rel(dwb, dwa) < 1e-14
    perm = rng.permutation(M)
    dxp, dwp = orc.rmsnorm_bwd(x[perm], g, dy[perm], rstd[perm])
    assert np.array_equal(dxp, dx[perm]) and _rel(dwp, dw) < 1e-14


def _parse_golden():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key == "kind":
                cur[key] = vals[0]
            else:
                cur[key] = np.array([float(Fraction(v)) for v in vals])
    return cases


def hand_cases(orc):
    for c in _parse_golden():
        M, N = int(c["M"][0]), int(c["N"][0])
        eps = float(c["eps"][0])
        sh = lambda k: c[k].reshape(M, N)
        if c["kind"] == "plain":
            y, rstd = orc.rmsnorm_fwd(sh("x"), c["gamma"], eps)
            dx, dw = orc.rmsnorm_bwd(sh("x"), c["gamma"], sh("dy"), c["rstd"])
        else:
            y, res_out, rstd = orc.fused_add_rmsnorm_fwd(sh("x"), sh("residual"), c["gamma"],
                                                         eps, "f32")
            assert np.array_equal(res_out, sh("residual_out")), c["name"]
            dx, dw = orc.fused_add_rmsnorm_bwd(res_out, c["gamma"], sh("dy"), c["rstd"],
                                               sh("dres"))
        assert np.allclose(rstd, c["rstd"], rtol=1e-15, atol=0), c["name"]
        assert np.allclose(y, sh("y"), rtol=1e-15, atol=1e-15), c["name"]
        assert np.allclose(dx, sh("dx"), rtol=1e-15, atol=1e-15), c["name"]
        assert np.allclose(dw, c["dweight"], rtol=1e-15, atol=1e-15), c["name"]


# ----------------------------------------------------------------- LayerNorm
LN_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                         "layernorm_hand_cases.txt")


def ln_fwd_vs_torch(orc):
    """torch.nn.functional.layer_norm in fp64 (with and without bias); mean and
    rstd against numpy's mean and (biased) variance."""
    rng = np.random.default_rng(21)
    for (M, N, eps) in ((7, 33, 1e-5), (3, 1000, 1e-6), (2, 1, 1e-2)):
        x = rng.standard_normal((M, N)) * 3 + 1.5
        g = 1 + 0.1 * rng.standard_normal(N)
        b = 0.1 * rng.standard_normal(N)
        for beta in (b, None):
            y, mean, rstd = orc.layernorm_fwd(x, g, beta, eps)
            ref = torch.nn.functional.layer_norm(
                torch.from_numpy(x), (N,), torch.from_numpy(g),
                torch.from_numpy(beta) if beta is not None else None, eps).numpy()
            assert _rel(y, ref) < 1e-13, (M, N, beta is None)
        assert _rel(mean, np.mean(x, axis=1)) < 1e-14
        assert _rel(rstd, 1 / np.sqrt(np.var(x, axis=1) + eps)) < 1e-13


def _ln_sym_grads(M, N, x, g, b, dy, eps):
    """Exact gradients of L = sum(y*dy) with y from the LayerNorm definition (sympy)."""
    import sympy as sp
    X = sp.Matrix(M, N, lambda i, j: sp.Symbol("x_%d_%d" % (i, j)))
    G = [sp.Symbol("g_%d" % j) for j in range(N)]
    B = [sp.Symbol("b_%d" % j) for j in range(N)]
    L = 0
    for i in range(M):
        mu = sum(X[i, j] for j in range(N)) / N
        var = sum((X[i, j] - mu) ** 2 for j in range(N)) / N
        rs = (var + eps) ** sp.Rational(-1, 2)
        for j in range(N):
            L += ((X[i, j] - mu) * rs * G[j] + B[j]) * dy[i][j]
    subs = {X[i, j]: x[i][j] for i in range(M) for j in range(N)}
    subs.update({G[j]: g[j] for j in range(N)})
    subs.update({B[j]: b[j] for j in range(N)})
    ev = lambda e: float(e.subs(subs).evalf(30))
    dX = np.array([[ev(sp.diff(L, X[i, j])) for j in range(N)] for i in range(M)])
    dG = np.array([ev(sp.diff(L, G[j])) for j in range(N)])
    dB = np.array([ev(sp.diff(L, B[j])) for j in range(N)])
    return dX, dG, dB


def ln_bwd_symbolic(orc):
    import sympy as sp
    Q = sp.Rational
    M, N = 2, 3
    x = [[Q(1, 2), Q(-3, 4), Q(2)], [Q(5, 4), Q(1, 8), Q(-1)]]
    g = [Q(9, 10), Q(11, 10), Q(5, 4)]
    b = [Q(1, 10), Q(-1, 5), Q(0)]
    dy = [[Q(1), Q(-2), Q(1, 2)], [Q(3, 4), Q(1, 4), Q(-1)]]
    eps = Q(1, 100)
    dX, dG, dB = _ln_sym_grads(M, N, x, g, b, dy, eps)
    f = lambda a: np.array(a, dtype=np.float64)
    mean = np.array([float(sum(row) / N) for row in x])
    rstd = np.array([float((sum((v - sum(row) / N) ** 2 for v in row) / N + eps) ** Q(-1, 2))
                     for row in x])
    dx, dg, db = orc.layernorm_bwd(f(x), f(g), f(dy), mean, rstd)
    assert _rel(dx, dX) < 1e-13 and _rel(dg, dG) < 1e-13 and _rel(db, dB) < 1e-13, (dx, dX)


def _ln_loss(orc, x, g, b, dy, eps):
    y, _, _ = orc.layernorm_fwd(x, g, b, eps)
    return float(np.sum(y * dy))


def ln_bwd_fd(orc):
    rng = np.random.default_rng(22)
    for (M, N, eps) in ((3, 16, 1e-5), (2, 5, 1e-2)):
        x = rng.standard_normal((M, N)) + 0.7
        g = 1 + 0.1 * rng.standard_normal(N)
        b = 0.1 * rng.standard_normal(N)
        dy = rng.standard_normal((M, N))
        _, mean, rstd = orc.layernorm_fwd(x, g, b, eps)
        dx, dg, db = orc.layernorm_bwd(x, g, dy, mean, rstd)
        h = 1e-6

        def fd(arr, setter):
            out = np.zeros(arr.shape)
            for idx in np.ndindex(arr.shape):
                ap, am = arr.copy(), arr.copy()
                ap[idx] += h
                am[idx] -= h
                out[idx] = (setter(ap) - setter(am)) / (2 * h)
            return out
        fdx = fd(x, lambda v: _ln_loss(orc, v, g, b, dy, eps))
        fdg = fd(g, lambda v: _ln_loss(orc, x, v, b, dy, eps))
        fdb = fd(b, lambda v: _ln_loss(orc, x, g, v, dy, eps))
        assert _rel(dx, fdx) < 1e-6 and _rel(dg, fdg) < 1e-6 and _rel(db, fdb) < 1e-6


def ln_bwd_torch_autograd(orc):
    rng = np.random.default_rng(23)
    M, N, eps = 16, 300, 1e-5
    x = rng.standard_normal((M, N)) * 2 - 0.5
    g = 1 + 0.1 * rng.standard_normal(N)
    b = 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    xt = torch.from_numpy(x).requires_grad_(True)
    gt = torch.from_numpy(g).requires_grad_(True)
    bt = torch.from_numpy(b).requires_grad_(True)
    torch.nn.functional.layer_norm(xt, (N,), gt, bt, eps).backward(torch.from_numpy(dy))
    _, mean, rstd = orc.layernorm_fwd(x, g, b, eps)
    dx, dg, db = orc.layernorm_bwd(x, g, dy, mean, rstd)
    assert _rel(dx, xt.grad.numpy()) < 1e-12
    assert _rel(dg, gt.grad.numpy()) < 1e-12 and _rel(db, bt.grad.numpy()) < 1e-12


def ln_bwd_invariants(orc):
    """Per row, with the exact statistics: sum_j dx_j = 0 (sum_j x_hat_j = 0),
    and sum_j x_hat_j*dx_j = N*eps*c1*rstd^3 (derivation: rstd*(N*c1 - c2*0 -
    c1*N*var*rstd^2) with 1 - var*rstd^2 = eps*rstd^2). dbeta is the column
    sum of dy."""
    rng = np.random.default_rng(24)
    M, N = 6, 50
    x = rng.standard_normal((M, N)) + 2.0
    g = 1 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    for eps in (1e-1, 1e-3, 0.0):
        _, mean, rstd = orc.layernorm_fwd(x, g, None, eps)
        dx, _, db = orc.layernorm_bwd(x, g, dy, mean, rstd)
        scale = np.sum(np.abs(dx), axis=1)
        assert np.all(np.abs(np.sum(dx, axis=1)) <= 1e-13 * scale)
        xh = (x - mean[:, None]) * rstd[:, None]
        c1 = np.mean(xh * dy * g, axis=1)
        lhs = np.sum(xh * dx, axis=1)
        rhs = N * eps * c1 * rstd ** 3
        assert np.all(np.abs(lhs - rhs) <= 1e-13 * np.sum(np.abs(xh * dx), axis=1)), (eps,)
        assert _rel(db, np.sum(dy, axis=0)) < 1e-14


def ln_reduces_to_rms(orc):
    """Rows with an exactly zero mean and no bias: LayerNorm is RMSNorm."""
    rng = np.random.default_rng(25)
    M, N, eps = 4, 32, 1e-6
    half = rng.standard_normal((M, N // 2))
    x = np.empty((M, N))
    x[:, 0::2], x[:, 1::2] = half, -half           # a, -a, b, -b, ...: row sums are exactly 0
    g = 1 + 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    y, mean, rstd = orc.layernorm_fwd(x, g, None, eps)
    assert np.all(mean == 0.0)
    y2, rstd2 = orc.rmsnorm_fwd(x, g, eps)
    assert _rel(y, y2) < 1e-15 and _rel(rstd, rstd2) < 1e-15
    dx, dg, _ = orc.layernorm_bwd(x, g, dy, mean, rstd)
    dx2, dg2 = orc.rmsnorm_bwd(x, g, dy, rstd)
    # the LayerNorm dx has the extra -c2*rstd term; on zero-mean rows it is the
    # projection of the RMSNorm dx onto zero-sum vectors
    c2 = np.mean(dy * g, axis=1)
    assert _rel(dx, dx2 - (c2 * rstd)[:, None]) < 1e-13 and _rel(dg, dg2) < 1e-14


def ln_shift_invariance(orc):
    """Adding a constant to a row moves its mean and leaves y and dx unchanged."""
    rng = np.random.default_rng(26)
    M, N, eps = 5, 24, 1e-5
    x = rng.standard_normal((M, N))
    g = 1 + 0.1 * rng.standard_normal(N)
    b = 0.1 * rng.standard_normal(N)
    dy = rng.standard_normal((M, N))
    shift = np.array([0.0, 1.0, -4.0, 8.0, 0.5])[:, None]
    y, mean, rstd = orc.layernorm_fwd(x, g, b, eps)
    y2, mean2, rstd2 = orc.layernorm_fwd(x + shift, g, b, eps)
    assert _rel(y2, y) < 1e-13 and _rel(mean2, mean + shift[:, 0]) < 1e-14
    dx, dg, db = orc.layernorm_bwd(x, g, dy, mean, rstd)
    dxs, dgs, dbs = orc.layernorm_bwd(x + shift, g, dy, mean2, rstd2)
    assert _rel(dxs, dx) < 1e-12 and _rel(dgs, dg) < 1e-12 and np.array_equal(dbs, db)


def _parse_cases(path):
    cases, cur = [], None
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key == "kind":
                cur[key] = vals[0]
            else:
                cur[key] = np.array([float(Fraction(v)) for v in vals])
    return cases


def ln_hand_cases(orc):
    for c in _parse_cases(LN_GOLDEN):
        M, N = int(c["M"][0]), int(c["N"][0])
        eps = float(c["eps"][0])
        sh = lambda k: c[k].reshape(M, N)
        y, mean, rstd = orc.layernorm_fwd(sh("x"), c["gamma"], c["beta"], eps)
        assert np.allclose(mean, c["mean"], rtol=1e-15, atol=0), c["name"]
        assert np.allclose(rstd, c["rstd"], rtol=1e-15, atol=0), c["name"]
        assert np.allclose(y, sh("y"), rtol=1e-15, atol=1e-15), c["name"]
        dx, dg, db = orc.layernorm_bwd(sh("x"), c["gamma"], sh("dy"), c["mean"], c["rstd"])
        assert np.allclose(dx, sh("dx"), rtol=1e-15, atol=1e-15), c["name"]
        assert np.allclose(dg, c["dgamma"], rtol=1e-15, atol=1e-15), c["name"]
        assert np.allclose(db, c["dbeta"], rtol=1e-15, atol=1e-15), c["name"]


PINS = [
    round_vs_torch_casts,
    round_direct_from_double,
    fwd_vs_torch_rms_norm,
    fused_fwd_vs_torch,
    bwd_symbolic,
    fused_bwd_symbolic,
    bwd_fd,
    fused_bwd_fd,
    bwd_invariant,
    bwd_torch_autograd,
    fused_reduces_to_plain,
    scaling_and_permutation,
    hand_cases,
    ln_fwd_vs_torch,
    ln_bwd_symbolic,
    ln_bwd_fd,
    ln_bwd_torch_autograd,
    ln_bwd_invariants,
    ln_reduces_to_rms,
    ln_shift_invariance,
    ln_hand_cases,
]
