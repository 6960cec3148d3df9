"""Parity helpers: oracle expectations for a case and the comparison rules.

Tolerances (written here, used by every GPU parity test):
  * f32 dx / y:  max|gpu - ref| / max|ref| <= 1e-5 over the tensor.
  * f16/bf16 dx / y:  |gpu - ref| <= 1e-2 + 1.6e-2*|ref| elementwise, AND the
    tighter |gpu - ref| <= ulp_dtype(ref) + 1e-5*max|ref| (one unit in the
    last place of the I/O dtype, plus fp32 round-off relative to the tensor's
    scale for elements near zero).
  * dweight_f32: max|gpu - ref| / max|ref| <= 1e-4; the cast dweight within
    ulp_dtype(ref) + 1e-4*max|ref|.
  * rstd (forward): |gpu - ref| <= 4*2^-24*ref.
  * residual_out (fused forward): bit-exact (one correctly rounded add).
ref is the fp64 oracle on the same inputs; inputs and the saved rstd come
from the seeded generator and the oracle, never from the GPU.

Ill-conditioned elements: where dx is a near-total cancellation of its two
terms (wdy - x_hat*c1; e.g. N = 1, where x_hat^2 = ms/(ms+eps) is 1 - O(eps)),
fp32 arithmetic cannot reach a bound relative to |dx| itself. Only such an
element may pass on a second, round-off bound: its cancellation ratio
kappa = |dx| / (rstd * (|wdy| + |x_hat*c1|)) must be below KAPPA_ILL, and its
error within fp32 round-off of the terms it is made of:
2^-24 * rstd * (16*(|wdy| + |x_hat*c1|) + 4*sqrt(N)*|x_hat|*rstd*mean|x*wdy|)
(pointwise roundings plus the c1 reduction), computed in fp64 from the
inputs for the failing elements only. Every comparison returns how many
elements passed that way; check_bwd asserts none unless the caller allows
them (the degenerate widths), and the workload tests assert zero.
"""
import numpy as np
import torch

import oracle
from rmsnorm_backward_bwd_gb300 import synth

P_BITS = {"f32": 24, "f16": 11, "bf16": 8}
# cancellation ratio below which an element counts as ill-conditioned
KAPPA_ILL = 1e-3
E_MIN = {"f32": -126, "f16": -14, "bf16": -126}


def ulp(ref, dtype):
    a = np.abs(np.asarray(ref, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(np.where(a > 0, e, E_MIN[dtype]), E_MIN[dtype])
    return np.ldexp(1.0, (e - (P_BITS[dtype] - 1)).astype(np.int64))


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check_tensor(name, got, ref, dtype, kind="dx", roundoff=None):
    """Compare one GPU output (torch tensor) with the fp64 reference (numpy).
    roundoff(mask) -> (bound, terms): per-element fp32 round-off bound and the
    magnitude of dx's terms (rstd * (|wdy| + |x_hat*c1|), plus |c2| for
    LayerNorm) for the masked elements (dx only; see the module docstring).
    Returns the number of elements that passed only on the round-off bound."""
    g = to64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "%s has non-finite values" % name
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = np.abs(g - ref)
    if ref.size == 0:
        return 0
    if kind == "dweight_f32":
        rel = float(np.max(err)) / max(scale, 1e-30)
        assert rel <= 1e-4, "%s: max rel err %.3g > 1e-4" % (name, rel)
        return 0
    if kind == "dweight":
        bound = ulp(ref, dtype) + 1e-4 * scale
        bad = err > bound
        assert not bad.any(), "%s: %d elements beyond 1 ulp (worst %.3g vs bound %.3g)" % (
            name, int(bad.sum()), float(err[bad].max()), float(bound[bad][np.argmax(err[bad])]))
        return 0

    def escape(bad, base):
        """Elements of `bad` that are ill-conditioned and within the round-off
        bound (added to `base`, the dtype's own allowance) pass."""
        if not bad.any() or roundoff is None:
            return 0
        rb, terms = roundoff(bad)
        kappa = np.abs(ref[bad]) / np.maximum(terms, 1e-300)
        ok = (kappa < KAPPA_ILL) & (err[bad] <= base + rb)
        bad[bad] = ~ok
        return int(ok.sum())

    if dtype == "f32":
        bad = err > 1e-5 * scale
        n_esc = escape(bad, 0.0)
        assert not bad.any(), "%s: %d elements beyond rel err 1e-5 (max rel %.3g)" % (
            name, int(bad.sum()), float(np.max(err)) / max(scale, 1e-30))
        return n_esc
    loose = err <= 1e-2 + 1.6e-2 * np.abs(ref)
    assert loose.all(), "%s: %d elements outside atol 1e-2 / rtol 1.6e-2" % (name, int((~loose).sum()))
    bound = ulp(ref, dtype) + 1e-5 * scale
    bad = err > bound
    n_esc = escape(bad, ulp(ref[bad], dtype) if bad.any() else 0.0)
    assert not bad.any(), "%s: %d elements beyond 1 ulp (worst excess %.3g)" % (
        name, int(bad.sum()), float((err - bound)[bad].max()))
    return n_esc


class Expected:
    """Inputs (CPU tensors in the I/O dtype) and the oracle's outputs."""


def expected_bwd(case, nthreads=0):
    """Draw the case's inputs; compute `added` (fused) and the saved fp32
    rstd with the oracle's forward; then the oracle's backward."""
    inp = synth.make_inputs(case)
    dt = case.dtype
    tdt = synth.TORCH_DTYPES[dt]
    ex = Expected()
    ex.case = case
    g64 = inp["gamma"].to(torch.float64).numpy()
    x64 = inp["x"].to(torch.float64).numpy()
    if case.fused:
        r64 = inp["residual"].to(torch.float64).numpy()
        _, a64, rstd64 = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(case.eps), dt,
                                                      nthreads)
        ex.x = torch.from_numpy(a64).to(tdt)     # exact: a64 is dtype-rounded
        del r64
    else:
        _, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(case.eps), nthreads)
        a64 = x64
        ex.x = inp["x"]
    rstd32 = oracle.round_to(rstd64, "f32")
    ex.rstd = torch.from_numpy(rstd32).to(torch.float32)
    ex.gamma = inp["gamma"]
    ex.dy = inp["dy"]
    dy64 = inp["dy"].to(torch.float64).numpy()
    ex.dres = inp.get("dres")
    if case.fused:
        dres64 = ex.dres.to(torch.float64).numpy() if ex.dres is not None else None
        ex.dx, ex.dw = oracle.fused_add_rmsnorm_bwd(a64, g64, dy64, rstd32, dres64, nthreads)
    else:
        ex.dx, ex.dw = oracle.rmsnorm_bwd(a64, g64, dy64, rstd32, nthreads)
    ex.a64, ex.g64, ex.dy64, ex.rstd64 = a64, g64, dy64, rstd32
    return ex


def roundoff_bound(ex):
    """fp32 round-off bound of dx's terms and their magnitude, for the
    elements of a mask."""
    def fn(mask):
        rows, cols = np.nonzero(mask.reshape(ex.a64.shape))
        urows = np.unique(rows)
        N = ex.a64.shape[1]
        xr = ex.a64[urows]
        r = ex.rstd64[urows][:, None]
        wdy_r = ex.dy64[urows] * ex.g64
        c1 = np.mean(xr * r * wdy_r, axis=1)
        mabs = np.mean(np.abs(xr * wdy_r), axis=1)
        pos = np.searchsorted(urows, rows)
        xh = ex.a64[rows, cols] * ex.rstd64[rows]
        wdy = ex.dy64[rows, cols] * ex.g64[cols]
        rs = ex.rstd64[rows]
        terms = np.abs(wdy) + np.abs(xh * c1[pos])
        bound = 2.0**-24 * rs * (16 * terms + 4 * np.sqrt(N) * np.abs(xh) * rs * mabs[pos])
        return bound, rs * terms
    return fn


def run_gpu_bwd(ex, dev="cuda", dx_out=None):
    import rmsnorm_backward_bwd_gb300 as rn
    x = ex.x.to(dev)
    g = ex.gamma.to(dev)
    dy = ex.dy.to(dev)
    rstd = ex.rstd.to(dev)
    if ex.case.fused:
        dres = ex.dres.to(dev) if ex.dres is not None else None
        dx, dres_out, dw, dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, dx=dx_out)
        assert dres_out.data_ptr() == dx.data_ptr()
    else:
        dx, dw, dw32 = rn.rmsnorm_bwd(x, g, dy, rstd, dx=dx_out)
    torch.cuda.synchronize()
    return dx, dw, dw32


def check_bwd(ex, dx, dw, dw32, tag="", allow_ill_conditioned=False):
    """dx, dweight_f32 and the cast dweight against the oracle. The round-off
    escape for ill-conditioned dx elements is used only when the caller
    allows it (degenerate widths such as N = 1); returns its count."""
    dt = ex.case.dtype
    n_esc = check_tensor("dx" + tag, dx, ex.dx, dt, "dx", roundoff=roundoff_bound(ex))
    assert allow_ill_conditioned or n_esc == 0, (
        "dx%s: %d elements passed only on the round-off bound" % (tag, n_esc))
    check_tensor("dweight_f32" + tag, dw32, ex.dw, dt, "dweight_f32")
    if dw is not None:
        check_tensor("dweight" + tag, dw, ex.dw, dt, "dweight")
    return n_esc
