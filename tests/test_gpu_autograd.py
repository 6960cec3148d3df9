"""The autograd wrappers on the GPU against the oracle.

Forward outputs and the gradients of x, residual and weight that autograd
delivers are compared with the oracle's forward and backward on the same
seeded inputs (inputs of rank 2 to 4; aligned, unaligned and small widths;
f32, f16, bf16), with the parity tolerances of the backward tests. The GPU's
backward uses the GPU forward's own rstd; the oracle's uses its fp32-rounded
fp64 rstd: the two differ by a few fp32 ulps, well inside the tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import rmsnorm_backward_bwd_gb300 as rn
from rmsnorm_backward_bwd_gb300 import native, synth
from rmsnorm_backward_bwd_gb300.synth import Case

pytestmark = pytest.mark.gpu

SHAPES = [((2, 64, 1024), "f32"), ((4, 32, 4096), "bf16"), ((3, 5, 3000), "f32"),
          ((2, 7, 1001), "bf16"), ((8, 2048), "f16"), ((2, 2, 3, 520), "f16"), ((1, 4096), "bf16")]


def _case(shape, dt, fused, seed=0):
    M = int(np.prod(shape[:-1]))
    return Case("autograd", M, shape[-1], dt, fused=fused, with_dres=fused, seed=seed)


def _oracle_plain(inp, eps, dt):
    x64, g64, dy64 = (parity.to64(inp[k]) for k in ("x", "gamma", "dy"))
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(eps))
    rstd32 = oracle.round_to(rstd64, "f32")
    dx64, dw64 = oracle.rmsnorm_bwd(x64, g64, dy64, rstd32)
    return y64, dx64, dw64, x64, g64, dy64, rstd32


@pytest.mark.parametrize("shape,dt", SHAPES, ids=lambda v: str(v))
def test_rmsnorm_autograd_matches_oracle(shape, dt):
    case = _case(shape, dt, False)
    eps = case.eps
    inp = synth.make_inputs(case)
    y64, dx64, dw64, x64, g64, dy64, rstd32 = _oracle_plain(inp, eps, dt)
    x = inp["x"].cuda().reshape(shape).requires_grad_()
    w = inp["gamma"].cuda().requires_grad_()
    y = rn.rmsnorm(x, w, eps)
    assert y.shape == shape and y.dtype == x.dtype
    y.backward(inp["dy"].cuda().reshape(shape))
    torch.cuda.synchronize()
    ex = parity.Expected()
    ex.a64, ex.g64, ex.dy64, ex.rstd64 = x64, g64, dy64, rstd32
    parity.check_tensor("y", y.reshape(case.M, case.N), y64, dt, "y")
    assert parity.check_tensor("dx", x.grad.reshape(case.M, case.N), dx64, dt, "dx",
                               roundoff=parity.roundoff_bound(ex)) == 0
    assert w.grad.dtype == w.dtype
    parity.check_tensor("dweight", w.grad, dw64, dt, "dweight")


@pytest.mark.parametrize("shape,dt", SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("use", ["both", "out", "residual_out"])
def test_fused_autograd_matches_oracle(shape, dt, use):
    case = _case(shape, dt, True, seed=3)
    eps = case.eps
    inp = synth.make_inputs(case)
    x64, r64, g64 = (parity.to64(inp[k]) for k in ("x", "residual", "gamma"))
    out64, a64, rstd64 = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(eps), dt)
    rstd32 = oracle.round_to(rstd64, "f32")
    dy64 = parity.to64(inp["dy"]) if use != "residual_out" else np.zeros_like(a64)
    dres64 = parity.to64(inp["dres"]) if use != "out" else None
    dx64, dw64 = oracle.fused_add_rmsnorm_bwd(a64, g64, dy64, rstd32, dres64)

    x = inp["x"].cuda().reshape(shape).requires_grad_()
    r = inp["residual"].cuda().reshape(shape).requires_grad_()
    w = inp["gamma"].cuda().requires_grad_()
    out, res_out = rn.fused_add_rmsnorm(x, r, w, eps)
    loss = 0
    if use != "residual_out":
        loss = loss + (out.float() * inp["dy"].cuda().reshape(shape).float()).sum()
    if use != "out":
        loss = loss + (res_out.float() * inp["dres"].cuda().reshape(shape).float()).sum()
    loss.backward()
    torch.cuda.synchronize()
    assert np.array_equal(parity.to64(res_out.reshape(case.M, case.N)), a64)
    parity.check_tensor("out", out.reshape(case.M, case.N), out64, dt, "y")
    ex = parity.Expected()
    ex.a64, ex.g64, ex.dy64, ex.rstd64 = a64, g64, dy64, rstd32
    assert parity.check_tensor("dx", x.grad.reshape(case.M, case.N), dx64, dt, "dx",
                               roundoff=parity.roundoff_bound(ex)) == 0
    assert torch.equal(x.grad, r.grad)
    parity.check_tensor("dweight", w.grad, dw64, dt, "dweight")


def test_prenorm_false_and_partial_requires_grad():
    case = _case((6, 4096), "bf16", True, seed=5)
    inp = synth.make_inputs(case)
    x = inp["x"].cuda().requires_grad_()
    out = rn.fused_add_rmsnorm(x, inp["residual"].cuda(), inp["gamma"].cuda(), 1e-6,
                               prenorm=False)
    assert isinstance(out, torch.Tensor)
    out.backward(inp["dy"].cuda())
    x64, r64, g64 = (parity.to64(inp[k]) for k in ("x", "residual", "gamma"))
    _, a64, rstd64 = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(1e-6), "bf16")
    dx64, _ = oracle.fused_add_rmsnorm_bwd(a64, g64, parity.to64(inp["dy"]),
                                           oracle.round_to(rstd64, "f32"), None)
    parity.check_tensor("dx", x.grad, dx64, "bf16", "dx")


def test_autograd_guards():
    x = torch.randn(2, 3, 256, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    w = torch.ones(256, device="cuda", dtype=torch.float32, requires_grad=True)
    with pytest.raises(ValueError, match="dtype mismatch"):
        rn.rmsnorm(x, w)
    with pytest.raises(ValueError, match="residual has shape"):
        rn.fused_add_rmsnorm(x, x[:1], w.to(torch.bfloat16))


def test_noncontiguous_input_and_expanded_grad():
    case = _case((16, 512), "f16", False, seed=7)
    inp = synth.make_inputs(case)
    base = inp["x"].cuda().t().contiguous().t()        # column-major view of x
    assert not base.is_contiguous()
    x = base.detach().requires_grad_()
    w = inp["gamma"].cuda().requires_grad_()
    rn.rmsnorm(x, w, case.eps).sum().backward()         # dy = ones, stride 0
    torch.cuda.synchronize()
    x64, g64 = parity.to64(inp["x"]), parity.to64(inp["gamma"])
    _, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(case.eps))
    dx64, dw64 = oracle.rmsnorm_bwd(x64, g64, np.ones_like(x64), oracle.round_to(rstd64, "f32"))
    parity.check_tensor("dx", x.grad, dx64, "f16", "dx")
    parity.check_tensor("dweight", w.grad, dw64, "f16", "dweight")


def test_empty_batch_autograd():
    x = torch.empty(0, 3, 1024, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    w = torch.ones(1024, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    y = rn.rmsnorm(x, w)
    y.sum().backward()
    torch.cuda.synchronize()
    assert x.grad.shape == x.shape
    assert torch.count_nonzero(w.grad).item() == 0
