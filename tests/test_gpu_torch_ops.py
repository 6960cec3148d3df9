"""The PyTorch operator layer (C++, ``torch.ops.rn_gb300``) on the GPU.

The raw calls are compared with the oracle on the same seeded inputs (the
parity tolerances of the backward tests) and with the ctypes binding of the
same C ABI (dx bitwise; the weight gradient bitwise in the deterministic
scratch mode). Their argument checks raise before anything is launched. The
differentiable operators are checked where the C++ autograd function has
logic of its own: the LayerNorm bias slot, gradients that autograd does not
produce, and a forward + backward captured into a CUDA graph and replayed.
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

CASES = [Case("ops plain bf16", 512, 4096, "bf16"),
         Case("ops plain f32 unaligned", 37, 1001, "f32"),
         Case("ops fused f16 +dres", 300, 3000, "f16", fused=True, with_dres=True),
         Case("ops fused bf16 dres=None", 64, 2048, "bf16", fused=True),
         Case("ops long rows", 6, 32768, "bf16")]


@pytest.fixture(autouse=True)
def _reset_options():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    yield
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)


def _ops():
    return native.torch_ops()


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_raw_backward_matches_oracle_and_ctypes_binding(case):
    native.set_option(native.OPT_DWEIGHT_MODE, 1)   # scratch: deterministic dweight
    ex = parity.expected_bwd(case)
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    ops = _ops()
    if case.fused:
        dres = ex.dres.cuda() if ex.dres is not None else None
        dx, dw, dw32 = ops.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, True)
        cdx, _, cdw, cdw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres)
    else:
        dx, dw, dw32 = ops.rmsnorm_bwd(x, g, dy, rstd, True)
        cdx, cdw, cdw32 = rn.rmsnorm_bwd(x, g, dy, rstd)
    torch.cuda.synchronize()
    parity.check_bwd(ex, dx, dw, dw32)
    assert torch.equal(dx, cdx)
    assert torch.equal(dw32, cdw32) and torch.equal(dw, cdw)


def test_raw_backward_without_cast():
    ex = parity.expected_bwd(Case("ops no cast", 128, 4096, "bf16"))
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    dx, dw, dw32 = _ops().rmsnorm_bwd(x, g, dy, rstd, False)
    torch.cuda.synchronize()
    assert dw is None
    parity.check_bwd(ex, dx, None, dw32)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_raw_forwards_match_oracle_and_ctypes_binding(dt):
    case = Case("ops fwd", 96, 2048, dt, fused=True, with_dres=False)
    inp = synth.make_inputs(case)
    x64, r64, g64 = (parity.to64(inp[k]) for k in ("x", "residual", "gamma"))
    x, r, g = (inp[k].cuda() for k in ("x", "residual", "gamma"))
    ops = _ops()
    got = (ops.rmsnorm_fwd(x, g, 1e-6), ops.fused_add_rmsnorm_fwd(x, r, g, 1e-6),
           ops.layernorm_fwd(x, g, g, 1e-5))
    via_ctypes = (rn.rmsnorm_fwd(x, g, 1e-6), rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6),
                  rn.layernorm_fwd(x, g, g, 1e-5))
    torch.cuda.synchronize()
    # the same kernels behind both bindings: every output bitwise equal
    for a, b in zip(got, via_ctypes):
        assert all(torch.equal(u, v) for u, v in zip(a, b))
    y64, _ = oracle.rmsnorm_fwd(x64, g64, np.float32(1e-6))
    out64, a64, _ = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(1e-6), dt)
    yl64, _, _ = oracle.layernorm_fwd(x64, g64, g64, np.float32(1e-5))
    parity.check_tensor("y", got[0][0], y64, dt, "y")
    parity.check_tensor("out", got[1][0], out64, dt, "y")
    assert np.array_equal(parity.to64(got[1][1]), a64)
    parity.check_tensor("layernorm y", got[2][0], yl64, dt, "y")
    assert all(t.dtype == torch.float32 for t in (got[0][1], got[1][2], got[2][1], got[2][2]))


def test_raw_layernorm_backward_masks():
    native.set_option(native.OPT_DWEIGHT_MODE, 1)   # scratch: deterministic dgamma / dbeta
    case = Case("ops ln", 200, 1024, "bf16", eps=1e-5)
    inp = synth.make_ln_inputs(case)
    x, g, b, dy = (inp[k].cuda() for k in ("x", "gamma", "beta", "dy"))
    ops = _ops()
    _, mean, rstd = ops.layernorm_fwd(x, g, b, 1e-5)
    full = ops.layernorm_bwd(x, g, dy, mean, rstd, True, True)
    no_db = ops.layernorm_bwd(x, g, dy, mean, rstd, False, True)
    no_cast = ops.layernorm_bwd(x, g, dy, mean, rstd, True, False)
    via_ctypes = rn.layernorm_bwd(x, g, dy, mean, rstd)
    torch.cuda.synchronize()
    assert all(t is not None for t in full)
    assert no_db[2] is None and no_db[4] is None and no_db[1] is not None
    assert no_cast[1] is None and no_cast[2] is None and no_cast[4] is not None
    # the same kernels behind both bindings (dx, dgamma, dbeta, dgamma_f32, dbeta_f32)
    assert all(torch.equal(u, v) for u, v in zip(full, via_ctypes))
    assert torch.equal(full[0], no_db[0]) and torch.equal(full[0], no_cast[0])
    assert torch.equal(full[3], no_db[3]) and torch.equal(full[4], no_cast[4])
    _, dg64, db64 = oracle.layernorm_bwd(parity.to64(x), parity.to64(g), parity.to64(dy),
                                         parity.to64(mean), parity.to64(rstd))
    parity.check_tensor("dgamma_f32", full[3], dg64, "bf16", "dweight_f32")
    parity.check_tensor("dbeta_f32", full[4], db64, "bf16", "dweight_f32")


def test_raw_call_guards():
    ops = _ops()
    x = torch.randn(4, 256, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(256, device="cuda", dtype=torch.bfloat16)
    rstd = torch.ones(4, device="cuda")
    with pytest.raises(ValueError, match="dtype mismatch"):
        ops.rmsnorm_fwd(x, g.float(), 1e-6)
    with pytest.raises(ValueError, match="weight has shape"):
        ops.rmsnorm_fwd(x, g[:128], 1e-6)
    with pytest.raises(ValueError, match="must be contiguous"):
        ops.rmsnorm_bwd(x, g, x.t().contiguous().t(), rstd, True)
    with pytest.raises(ValueError, match="rstd has shape"):
        ops.rmsnorm_bwd(x, g, x, rstd[:3], True)
    with pytest.raises(ValueError, match="CUDA devices only"):
        ops.rmsnorm_bwd(x, g, x, rstd.cpu(), True)
    with pytest.raises(TypeError, match="unsupported dtype"):
        ops.rmsnorm_fwd(x.double(), g.double(), 1e-6)
    with pytest.raises(ValueError, match="dresidual_out has shape"):
        ops.fused_add_rmsnorm_bwd(x, g, x, rstd, x[:2], True)
    with pytest.raises(ValueError, match="bias has shape"):
        ops.layernorm_fwd(x, g, g[:10], 1e-5)


def test_raw_outputs_carry_no_gradient_history():
    x = torch.randn(8, 512, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    g = torch.ones(512, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    y, rstd = _ops().rmsnorm_fwd(x, g, 1e-6)
    assert not y.requires_grad and not rstd.requires_grad


@pytest.mark.parametrize("with_bias", [True, False])
def test_layernorm_autograd_bias_slot(with_bias):
    case = Case("ops ln autograd", 3 * 40, 768, "f32", eps=1e-5)
    inp = synth.make_ln_inputs(case)
    x = inp["x"].cuda().reshape(3, 40, 768).requires_grad_()
    w = inp["gamma"].cuda().requires_grad_()
    b = inp["beta"].cuda().requires_grad_() if with_bias else None
    y = rn.layernorm(x, w, b)
    y.backward(inp["dy"].cuda().reshape(3, 40, 768))
    torch.cuda.synchronize()
    x64, g64, dy64 = (parity.to64(inp[k]) for k in ("x", "gamma", "dy"))
    b64 = parity.to64(inp["beta"]) if with_bias else None
    y64, mean64, rstd64 = oracle.layernorm_fwd(x64, g64, b64, np.float32(1e-5))
    dx64, dg64, db64 = oracle.layernorm_bwd(x64, g64, dy64, oracle.round_to(mean64, "f32"),
                                            oracle.round_to(rstd64, "f32"))
    parity.check_tensor("y", y.reshape(case.M, case.N), y64, "f32", "y")
    parity.check_tensor("dx", x.grad.reshape(case.M, case.N), dx64, "f32", "dx")
    parity.check_tensor("dgamma", w.grad, dg64, "f32", "dweight")
    if with_bias:
        parity.check_tensor("dbeta", b.grad, db64, "f32", "dweight")


def test_fused_autograd_zero_out_grad_and_unused_residual_out():
    x = torch.randn(4, 1024, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    r = torch.randn(4, 1024, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    w = torch.ones(1024, device="cuda", dtype=torch.bfloat16, requires_grad=True)
    out, res_out = rn.fused_add_rmsnorm(x, r, w)
    # out gets a zero gradient, residual_out none at all (it stays undefined)
    other = (x * 2).sum()
    gx, gr, gw = torch.autograd.grad(other + 0 * out.sum(), (x, r, w))
    torch.cuda.synchronize()
    assert torch.equal(gx, torch.full_like(x, 2))
    assert gr is not None and float(gr.abs().max()) == 0.0
    assert gw is not None and float(gw.float().abs().max()) == 0.0


@pytest.mark.parametrize("op", ["rmsnorm", "fused_add_rmsnorm", "layernorm"])
def test_autograd_step_captured_in_a_cuda_graph(op):
    M, N = 256, 2048
    gen = torch.Generator(device="cpu").manual_seed(11)
    x0 = torch.randn(M, N, generator=gen).to(torch.bfloat16).cuda()
    r0 = torch.randn(M, N, generator=gen).to(torch.bfloat16).cuda()
    w0 = (1 + 0.1 * torch.randn(N, generator=gen)).to(torch.bfloat16).cuda()
    dy = (0.01 * torch.randn(M, N, generator=gen)).to(torch.bfloat16).cuda()
    x = x0.clone().requires_grad_()
    w = w0.clone().requires_grad_()

    def step():
        if op == "rmsnorm":
            y = rn.rmsnorm(x, w)
        elif op == "fused_add_rmsnorm":
            y = rn.fused_add_rmsnorm(x, r0, w)[0]
        else:
            y = rn.layernorm(x, w)
        return torch.autograd.grad(y, (x, w), dy)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):   # first calls (device queries, kernel attributes) outside capture
            eager = step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        captured = step()
    x.data.copy_(x0 * 0.5)           # new inputs, same buffers
    g.replay()
    torch.cuda.synchronize()
    with torch.no_grad():
        x_half = x.detach().clone()
    x2 = x_half.requires_grad_()
    w2 = w0.clone().requires_grad_()
    if op == "rmsnorm":
        y2 = rn.rmsnorm(x2, w2)
    elif op == "fused_add_rmsnorm":
        y2 = rn.fused_add_rmsnorm(x2, r0, w2)[0]
    else:
        y2 = rn.layernorm(x2, w2)
    ref = torch.autograd.grad(y2, (x2, w2), dy)
    torch.cuda.synchronize()
    assert torch.equal(captured[0], ref[0])
    assert torch.allclose(captured[1].float(), ref[1].float(), rtol=1e-2, atol=1e-3)
    assert not torch.equal(captured[0], eager[0])
