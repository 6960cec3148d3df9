"""Host logic of the C++ autograd functions (CPU only).

The differentiable ops (``torch.ops.rn_gb300.rmsnorm`` / ``fused_add_rmsnorm``
/ ``layernorm``, C++ in ``csrc/torch_ops.cpp``) do marshalling: flattening to
[M, N], saving tensors, turning absent gradients into the right call,
returning dx for both x and residual. They reach the computation through the
raw operators (``rn_gb300::rmsnorm_fwd`` etc.), which the library registers
for CUDA tensors only. Here a test-only CPU kernel for each raw operator,
built on the fp64 oracle, is registered with the dispatcher for the length of
a test, so that the C++ plumbing runs on the CPU; the gradients that come out
are compared with torch's own autograd in fp64. The public functions refuse
CPU tensors, which is checked too.
"""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_backward_bwd_gb300 as rn
from rmsnorm_backward_bwd_gb300 import autograd as ag
from rmsnorm_backward_bwd_gb300 import native


def _np(t):
    return t.detach().to(torch.float64).numpy()


class OracleKernels:
    """CPU kernels of the raw operators, computed by the oracle (fp32 I/O)."""

    def __init__(self):
        self.calls = []

    def rmsnorm_fwd(self, x, gamma, eps):
        self.calls.append(("fwd", tuple(x.shape)))
        y, rstd = oracle.rmsnorm_fwd(_np(x), _np(gamma), np.float32(eps))
        return (torch.from_numpy(y).to(x.dtype),
                torch.from_numpy(oracle.round_to(rstd, "f32")).to(torch.float32))

    def fused_add_rmsnorm_fwd(self, x, residual, gamma, eps):
        self.calls.append(("fused_fwd", tuple(x.shape)))
        out, added, rstd = oracle.fused_add_rmsnorm_fwd(_np(x), _np(residual), _np(gamma),
                                                        np.float32(eps), "f32")
        return (torch.from_numpy(out).to(x.dtype), torch.from_numpy(added).to(x.dtype),
                torch.from_numpy(oracle.round_to(rstd, "f32")).to(torch.float32))

    def rmsnorm_bwd(self, x, gamma, dy, rstd, want_cast, want_f32=True):
        self.calls.append(("bwd", tuple(x.shape), want_cast, want_f32))
        assert dy.is_contiguous() and dy.shape == x.shape
        dx, dw = oracle.rmsnorm_bwd(_np(x), _np(gamma), _np(dy), _np(rstd))
        dw32 = torch.from_numpy(dw).to(torch.float32)
        return (torch.from_numpy(dx).to(x.dtype), dw32.to(x.dtype) if want_cast else None,
                dw32 if want_f32 else None)

    def fused_add_rmsnorm_bwd(self, added, gamma, dy, rstd, dres, want_cast, want_f32=True):
        self.calls.append(("fused_bwd", tuple(added.shape), dres is not None, want_cast,
                           want_f32))
        dx, dw = oracle.fused_add_rmsnorm_bwd(_np(added), _np(gamma), _np(dy), _np(rstd),
                                              None if dres is None else _np(dres))
        dx = torch.from_numpy(dx).to(added.dtype)
        dw32 = torch.from_numpy(dw).to(torch.float32)
        return dx, dw32.to(added.dtype) if want_cast else None, dw32 if want_f32 else None

    def layernorm_fwd(self, x, gamma, beta, eps):
        self.calls.append(("ln_fwd", tuple(x.shape), beta is not None))
        y, mean, rstd = oracle.layernorm_fwd(_np(x), _np(gamma),
                                             None if beta is None else _np(beta), np.float32(eps))
        f32 = lambda a: torch.from_numpy(oracle.round_to(a, "f32")).to(torch.float32)  # noqa: E731
        return torch.from_numpy(y).to(x.dtype), f32(mean), f32(rstd)

    def layernorm_bwd(self, x, gamma, dy, mean, rstd, want_dbeta, want_cast, want_f32=True):
        self.calls.append(("ln_bwd", tuple(x.shape), want_dbeta, want_cast, want_f32))
        dx, dg, db = oracle.layernorm_bwd(_np(x), _np(gamma), _np(dy), _np(mean), _np(rstd))
        dg32 = torch.from_numpy(dg).to(torch.float32)
        db32 = torch.from_numpy(db).to(torch.float32) if want_dbeta else None
        return (torch.from_numpy(dx).to(x.dtype), dg32.to(x.dtype) if want_cast else None,
                db32.to(x.dtype) if (want_cast and want_dbeta) else None,
                dg32 if want_f32 else None, db32 if want_f32 else None)


_RAW = ("rmsnorm_fwd", "rmsnorm_bwd", "fused_add_rmsnorm_fwd", "fused_add_rmsnorm_bwd",
        "layernorm_fwd", "layernorm_bwd")


@pytest.fixture
def fake(monkeypatch):
    native.torch_ops()   # the operators must exist before kernels are added to them
    k = OracleKernels()
    lib = torch.library.Library("rn_gb300", "IMPL")
    for name in _RAW:
        lib.impl(name, getattr(k, name), "CPU")
    # let the public functions pass CPU tensors through to the operators
    monkeypatch.setattr(ag, "_on_cuda", lambda name, t: None)
    try:
        yield k
    finally:
        lib._destroy()


def _draw(shape, seed=0):
    g = torch.Generator().manual_seed(seed)
    N = shape[-1]
    x = torch.randn(*shape, generator=g)
    r = torch.randn(*shape, generator=g)
    w = 1 + 0.1 * torch.randn(N, generator=g)
    dy = torch.randn(*shape, generator=g)
    dres = torch.randn(*shape, generator=g)
    return x, r, w, dy, dres


def _torch_rms(x64, w64, eps):
    return torch.nn.functional.rms_norm(x64, (x64.shape[-1],), w64, eps)


def _close(a, b, tol=2e-5):
    a, b = a.detach().double(), b.detach().double()
    assert a.shape == b.shape
    scale = float(b.abs().max()) or 1.0
    assert float((a - b).abs().max()) <= tol * scale, float((a - b).abs().max()) / scale


@pytest.mark.parametrize("shape", [(7, 33), (2, 3, 64), (2, 2, 2, 16)])
def test_rmsnorm_grads_any_rank(fake, shape):
    x, _, w, dy, _ = _draw(shape)
    eps = 1e-5
    xa, wa = x.clone().requires_grad_(), w.clone().requires_grad_()
    y = rn.rmsnorm(xa, wa, eps)
    assert y.shape == x.shape
    (y * dy).sum().backward()
    x64, w64 = x.double().requires_grad_(), w.double().requires_grad_()
    y64 = _torch_rms(x64, w64, eps)
    (y64 * dy.double()).sum().backward()
    _close(y, y64)
    _close(xa.grad, x64.grad)
    _close(wa.grad, w64.grad)
    M = int(np.prod(shape[:-1]))
    # fp32 weight: its gradient is the fp32 sum itself (no cast asked for)
    assert fake.calls == [("fwd", (M, shape[-1])), ("bwd", (M, shape[-1]), False, True)]


def test_bf16_weight_gradient_is_the_cast(fake):
    """A 16-bit weight's gradient is the cast alone (no fp32 output is asked
    for, so the library takes its two-launch scratch path); an fp32 weight's
    is the fp32 sum itself."""
    x, r, w, dy, _ = _draw((4, 32), seed=6)
    for dt, cast in ((torch.bfloat16, True), (torch.float32, False)):
        xa = x.to(dt).requires_grad_()
        wa = w.to(dt).requires_grad_()
        (rn.rmsnorm(xa, wa, 1e-6) * dy.to(dt)).sum().backward()
        assert fake.calls[-1] == ("bwd", (4, 32), cast, not cast)
        assert wa.grad.dtype == dt
        out, _ = rn.fused_add_rmsnorm(xa.detach().requires_grad_(), r.to(dt), wa, 1e-6)
        (out * dy.to(dt)).sum().backward()
        assert fake.calls[-1] == ("fused_bwd", (4, 32), False, cast, not cast)


def test_rmsnorm_weight_grad_not_needed(fake):
    x, _, w, dy, _ = _draw((4, 32))
    xa = x.clone().requires_grad_()
    y = rn.rmsnorm(xa, w, 1e-6)
    y.backward(dy)
    # no weight gradient asked for at all
    assert fake.calls[-1] == ("bwd", (4, 32), False, False)
    assert xa.grad is not None


def test_rmsnorm_noncontiguous_grad(fake):
    x, _, w, _, _ = _draw((5, 16))
    xa = x.clone().requires_grad_()
    rn.rmsnorm(xa, w, 1e-6).sum().backward()   # dy is an expanded (stride 0) tensor
    x64 = x.double().requires_grad_()
    _torch_rms(x64, w.double(), 1e-6).sum().backward()
    _close(xa.grad, x64.grad)


def _fused_reference(x, r, w, dy, dres, eps, use_out=True, use_res=True):
    x64, r64 = x.double().requires_grad_(), r.double().requires_grad_()
    w64 = w.double().requires_grad_()
    added = x64 + r64
    out = _torch_rms(added, w64, eps)
    loss = 0
    if use_out:
        loss = loss + (out * dy.double()).sum()
    if use_res:
        loss = loss + (added * dres.double()).sum()
    loss.backward()
    return out, added, x64.grad, r64.grad, w64.grad


@pytest.mark.parametrize("use_out,use_res", [(True, True), (True, False), (False, True)])
def test_fused_grads(fake, use_out, use_res):
    x, r, w, dy, dres = _draw((2, 5, 48), seed=1)
    eps = 1e-6
    xa, ra, wa = (t.clone().requires_grad_() for t in (x, r, w))
    out, res_out = rn.fused_add_rmsnorm(xa, ra, wa, eps)
    assert out.shape == x.shape and res_out.shape == x.shape
    loss = 0
    if use_out:
        loss = loss + (out * dy).sum()
    if use_res:
        loss = loss + (res_out * dres).sum()
    loss.backward()
    o64, a64, gx, gr, gw = _fused_reference(x, r, w, dy, dres, eps, use_out, use_res)
    _close(out, o64)
    assert torch.equal(res_out, x + r)
    _close(xa.grad, gx)
    assert torch.equal(xa.grad, ra.grad)   # dx == dresidual
    if use_out:
        _close(wa.grad, gw)
    else:
        assert wa.grad is None or float(wa.grad.abs().max()) == 0.0
    last = fake.calls[-1]
    assert last[0] == "fused_bwd" and last[2] == use_res


def test_fused_prenorm_false_returns_out_only(fake):
    x, r, w, dy, _ = _draw((3, 16), seed=2)
    xa = x.clone().requires_grad_()
    out = rn.fused_add_rmsnorm(xa, r, w, 1e-6, prenorm=False)
    assert isinstance(out, torch.Tensor)
    (out * dy).sum().backward()
    _, _, gx, _, _ = _fused_reference(x, r, w, dy, dy, 1e-6, True, False)
    _close(xa.grad, gx)
    assert fake.calls[-1] == ("fused_bwd", (3, 16), False, False, False)


def test_real_calls_refuse_cpu_tensors():
    x = torch.randn(4, 8)
    w = torch.ones(8)
    with pytest.raises(ValueError, match="CUDA devices only"):
        rn.rmsnorm(x, w)
    with pytest.raises(ValueError, match="CUDA devices only"):
        rn.fused_add_rmsnorm(x, x, w)
    with pytest.raises(ValueError, match="CUDA devices only"):
        rn.rmsnorm_bwd(x, w, x, torch.ones(4))


def test_scalar_input_rejected():
    with pytest.raises(ValueError, match="at least one dimension"):
        rn.rmsnorm(torch.tensor(1.0), torch.ones(1))


def _torch_ln(x64, w64, b64, eps):
    return torch.nn.functional.layer_norm(x64, (x64.shape[-1],), w64, b64, eps)


@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("shape", [(6, 40), (2, 3, 24)])
def test_layernorm_grads(fake, shape, with_bias):
    x, _, w, dy, b = _draw(shape, seed=3)
    b = b[(0,) * (len(shape) - 1)] if with_bias else None
    eps = 1e-5
    xa, wa = x.clone().requires_grad_(), w.clone().requires_grad_()
    ba = b.clone().requires_grad_() if with_bias else None
    y = rn.layernorm(xa, wa, ba, eps)
    (y * dy).sum().backward()
    x64, w64 = x.double().requires_grad_(), w.double().requires_grad_()
    b64 = b.double().requires_grad_() if with_bias else None
    (_torch_ln(x64, w64, b64, eps) * dy.double()).sum().backward()
    _close(y, _torch_ln(x.double(), w.double(), None if b is None else b.double(), eps))
    _close(xa.grad, x64.grad)
    _close(wa.grad, w64.grad)
    if with_bias:
        _close(ba.grad, b64.grad)
    M = int(np.prod(shape[:-1]))
    assert fake.calls == [("ln_fwd", (M, shape[-1]), with_bias),
                          ("ln_bwd", (M, shape[-1]), with_bias, False, True)]   # fp32: no cast


def test_layernorm_only_x_grad(fake):
    x, _, w, dy, b = _draw((4, 16), seed=4)
    xa = x.clone().requires_grad_()
    rn.layernorm(xa, w, b[0]).backward(dy)
    # neither weight nor bias needs a gradient: no dbeta, no casts
    assert fake.calls[-1] == ("ln_bwd", (4, 16), False, False, False)
    x64 = x.double().requires_grad_()
    (_torch_ln(x64, w.double(), b[0].double(), 1e-5) * dy.double()).sum().backward()
    _close(xa.grad, x64.grad)


def test_no_input_needs_grad_skips_backward(fake):
    x, _, w, _, _ = _draw((3, 8))
    y = rn.rmsnorm(x, w)
    assert not y.requires_grad
    assert fake.calls == [("fwd", (3, 8))]


def test_residual_shape_checked_by_the_autograd_layer(fake):
    x, r, w, _, _ = _draw((3, 8))
    with pytest.raises(ValueError, match="residual has shape"):
        rn.fused_add_rmsnorm(x, r[:, :4], w)


def test_raw_operators_have_no_cpu_kernel():
    ops = native.torch_ops()
    x = torch.randn(2, 8)
    with pytest.raises(NotImplementedError):
        ops.rmsnorm_fwd(x, torch.ones(8), 1e-6)
    with pytest.raises(NotImplementedError):
        ops.rmsnorm(x, torch.ones(8), 1e-6)


def test_public_classes_forward_to_the_operators(fake):
    x, r, w, _, b = _draw((2, 8), seed=5)
    assert torch.equal(rn.RMSNormFunction.apply(x, w, 1e-6), rn.rmsnorm(x, w, 1e-6))
    out, res = rn.FusedAddRMSNormFunction.apply(x, r, w, 1e-6)
    assert torch.equal(res, x + r)
    assert torch.equal(rn.LayerNormFunction.apply(x, w, b[0], 1e-5), rn.layernorm(x, w, b[0]))
