"""Host logic of the autograd wrappers (CPU only).

The wrappers' own work is marshalling: flattening to [M, N], saving tensors,
turning absent gradients into the right call, returning dx for both x and
residual. Here the binding's calls are replaced by stand-ins built on the
fp64 oracle so that this plumbing runs on the CPU, and the gradients that
come out are compared with torch's own autograd of RMSNorm in fp64. The real
calls refuse CPU tensors, which is checked too.
"""
import numpy as np
import pytest
import torch

import oracle
import rmsnorm_backward_bwd_gb300 as rn
from rmsnorm_backward_bwd_gb300 import autograd as ag


def _np(t):
    return t.detach().to(torch.float64).numpy()


class OracleOps:
    """The four calls of the binding, computed by the oracle (fp32 I/O)."""

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

    def rmsnorm_bwd(self, x, gamma, dy, rstd, want_cast=True):
        self.calls.append(("bwd", tuple(x.shape), want_cast))
        assert dy.is_contiguous() and dy.shape == x.shape
        dx, dw = oracle.rmsnorm_bwd(_np(x), _np(gamma), _np(dy), _np(rstd))
        dw32 = torch.from_numpy(dw).to(torch.float32)
        return (torch.from_numpy(dx).to(x.dtype), dw32.to(x.dtype) if want_cast else None, dw32)

    def fused_add_rmsnorm_bwd(self, added, gamma, dy, rstd, dres=None, want_cast=True):
        self.calls.append(("fused_bwd", tuple(added.shape), dres is not None, want_cast))
        dx, dw = oracle.fused_add_rmsnorm_bwd(_np(added), _np(gamma), _np(dy), _np(rstd),
                                              None if dres is None else _np(dres))
        dx = torch.from_numpy(dx).to(added.dtype)
        dw32 = torch.from_numpy(dw).to(torch.float32)
        return dx, dx, dw32.to(added.dtype) if want_cast else None, dw32


@pytest.fixture
def fake(monkeypatch):
    ops = OracleOps()
    monkeypatch.setattr(ag, "ops", ops)
    return ops


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
    y = ag.rmsnorm(xa, wa, eps)
    assert y.shape == x.shape
    (y * dy).sum().backward()
    x64, w64 = x.double().requires_grad_(), w.double().requires_grad_()
    y64 = _torch_rms(x64, w64, eps)
    (y64 * dy.double()).sum().backward()
    _close(y, y64)
    _close(xa.grad, x64.grad)
    _close(wa.grad, w64.grad)
    M = int(np.prod(shape[:-1]))
    assert fake.calls == [("fwd", (M, shape[-1])), ("bwd", (M, shape[-1]), True)]


def test_rmsnorm_weight_grad_not_needed(fake):
    x, _, w, dy, _ = _draw((4, 32))
    xa = x.clone().requires_grad_()
    y = ag.rmsnorm(xa, w, 1e-6)
    y.backward(dy)
    assert fake.calls[-1] == ("bwd", (4, 32), False)
    assert xa.grad is not None


def test_rmsnorm_noncontiguous_grad(fake):
    x, _, w, _, _ = _draw((5, 16))
    xa = x.clone().requires_grad_()
    ag.rmsnorm(xa, w, 1e-6).sum().backward()   # dy is an expanded (stride 0) tensor
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
    out, res_out = ag.fused_add_rmsnorm(xa, ra, wa, eps)
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
    out = ag.fused_add_rmsnorm(xa, r, w, 1e-6, prenorm=False)
    assert isinstance(out, torch.Tensor)
    (out * dy).sum().backward()
    _, _, gx, _, _ = _fused_reference(x, r, w, dy, dy, 1e-6, True, False)
    _close(xa.grad, gx)
    assert fake.calls[-1] == ("fused_bwd", (3, 16), False, False)


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
