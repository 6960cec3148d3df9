"""Forward parity (plain and fused-add) and the small fwd+bwd chain."""
import numpy as np
import pytest
import torch

import oracle
import parity
import rmsnorm_backward_bwd_gb300 as rn
from rmsnorm_backward_bwd_gb300 import native, synth
from rmsnorm_backward_bwd_gb300.synth import Case

pytestmark = pytest.mark.gpu

SHAPES = [(128, 1024, "f32"), (4096, 4096, "bf16"), (1, 4096, "bf16"), (512, 2048, "bf16"),
          (512, 3000, "f32"), (128, 4096, "f16"), (7, 1001, "bf16"), (3, 33, "f16"),
          (16, 16384, "bf16"), (2, 40000, "f32"), (8, 32768, "bf16"), (3, 65536, "f16")]


def _check_rstd(got, ref64):
    g = parity.to64(got)
    assert np.all(np.abs(g - ref64) <= 4 * 2.0**-24 * ref64), float(np.max(np.abs(g / ref64 - 1)))


@pytest.mark.parametrize("M,N,dt", SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("eps", [1e-5, 1e-6, 1e-2])
def test_fwd_matches_oracle(M, N, dt, eps):
    inp = synth.make_inputs(Case("fwd", M, N, dt, eps=eps))
    x64 = parity.to64(inp["x"])
    g64 = parity.to64(inp["gamma"])
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(eps))
    y, rstd = rn.rmsnorm_fwd(inp["x"].cuda(), inp["gamma"].cuda(), eps)
    torch.cuda.synchronize()
    _check_rstd(rstd, rstd64)
    parity.check_tensor("y", y, y64, dt, "y")


@pytest.mark.parametrize("M,N,dt", SHAPES, ids=lambda v: str(v))
def test_fused_fwd_matches_oracle(M, N, dt):
    inp = synth.make_inputs(Case("fused fwd", M, N, dt, fused=True))
    x64, r64, g64 = (parity.to64(inp[k]) for k in ("x", "residual", "gamma"))
    out64, add64, rstd64 = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(1e-6), dt)
    out, res_out, rstd = rn.fused_add_rmsnorm_fwd(inp["x"].cuda(), inp["residual"].cuda(),
                                                  inp["gamma"].cuda(), 1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(parity.to64(res_out), add64)   # one correctly rounded add
    _check_rstd(rstd, rstd64)
    parity.check_tensor("out", out, out64, dt, "y")


@pytest.mark.parametrize("M,N,engine", [(256, 4096, "row"), (8, 40000, "long")])
def test_fwd_plan_names_the_engine(M, N, engine):
    inp = synth.make_inputs(Case("fwd plan", M, N, "bf16", fused=True))
    x, r, g = inp["x"].cuda(), inp["residual"].cuda(), inp["gamma"].cuda()
    rn.rmsnorm_fwd(x, g, 1e-6)
    assert native.last_plan().startswith("rmsnorm_fwd engine=%s" % engine), native.last_plan()
    rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6)
    assert native.last_plan().startswith("fused_add_fwd engine=%s" % engine), native.last_plan()
    rn.layernorm_fwd(x, g, None, 1e-5)
    assert native.last_plan().startswith("layernorm_fwd engine=%s" % engine), native.last_plan()
    torch.cuda.synchronize()


def test_eps_is_honoured():
    inp = synth.make_inputs(Case("eps", 64, 256, "f32"))
    x, g = inp["x"].cuda() * 1e-2, inp["gamma"].cuda()
    r = [rn.rmsnorm_fwd(x, g, eps)[1] for eps in (1e-5, 1e-6, 1e-2)]
    assert not torch.equal(r[0], r[1]) and not torch.equal(r[0], r[2])


def test_small_fwd_bwd_chain():
    """128 x 1024 f32, eps 1e-5: GPU forward, then GPU backward on the GPU's
    own rstd, against the oracle's forward and backward."""
    case = synth.SMALL_F32
    inp = synth.make_inputs(case)
    x64, g64, dy64 = (parity.to64(inp[k]) for k in ("x", "gamma", "dy"))
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(case.eps))
    dx64, dw64 = oracle.rmsnorm_bwd(x64, g64, dy64, oracle.round_to(rstd64, "f32"))
    x, g, dy = inp["x"].cuda(), inp["gamma"].cuda(), inp["dy"].cuda()
    y, rstd = rn.rmsnorm_fwd(x, g, case.eps)
    dx, dw, dw32 = rn.rmsnorm_bwd(x, g, dy, rstd)
    torch.cuda.synchronize()
    parity.check_tensor("y", y, y64, "f32", "y")
    _check_rstd(rstd, rstd64)
    parity.check_tensor("dx", dx, dx64, "f32", "dx")
    parity.check_tensor("dweight_f32", dw32, dw64, "f32", "dweight_f32")


def test_fwd_3d_input_and_guards():
    x = torch.randn(2, 3, 512, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(512, device="cuda", dtype=torch.bfloat16)
    y, rstd = rn.rmsnorm_fwd(x, g, 1e-6)
    assert y.shape == x.shape and rstd.shape == (6,)
    with pytest.raises(ValueError, match="dtype mismatch"):
        rn.rmsnorm_fwd(x, g.to(torch.float16), 1e-6)
    with pytest.raises(ValueError, match="weight has shape"):
        rn.rmsnorm_fwd(x, g[:256], 1e-6)
    with pytest.raises(ValueError, match="contiguous"):
        rn.rmsnorm_fwd(x.transpose(0, 1), g, 1e-6)
    with pytest.raises(ValueError, match="dtype mismatch"):
        rn.fused_add_rmsnorm_fwd(x, x.to(torch.float16), g, 1e-6)


UNALIGNED = [(300, 4095, "bf16"), (97, 2999, "f32"), (64, 1001, "f16"), (5, 7, "bf16"),
             (3, 3, "f32"), (40, 8190, "bf16"), (9, 16385, "f16"), (1000, 4100, "bf16"),
             (17, 515, "bf16"), (600, 2050, "f16"), (33, 4095, "f32"), (1, 4095, "bf16")]


def _shifted_like(t, shift):
    """A CUDA copy of t whose storage starts `shift` elements into a buffer
    (rows stay contiguous; the base moves off 16-byte alignment)."""
    buf = torch.empty(t.numel() + shift, dtype=t.dtype, device="cuda")
    v = buf[shift:].view(t.shape)
    v.copy_(t.cuda() if not t.is_cuda else t)
    return v


@pytest.mark.parametrize("M,N,dt", UNALIGNED, ids=lambda v: str(v))
@pytest.mark.parametrize("phase", ["same", "mismatched"])
def test_fwds_on_unaligned_rows(M, N, dt, phase):
    """Rows that are not 16-byte multiples: with all row tensors at one phase
    (16-byte chunks plus element-wise head and tail: the vector kernel, or for
    the 16-bit LayerNorm the phase-class kernel, each CTA on one alignment
    class of rows), and with the output one element off the input's phase
    (element-wise kernel). RMSNorm, fused-add and LayerNorm against the
    oracle."""
    inp = synth.make_inputs(Case("unaligned fwd", M, N, dt, fused=True, seed=31))
    x64, r64, g64 = (parity.to64(inp[k]) for k in ("x", "residual", "gamma"))
    x, r, g = inp["x"].cuda(), inp["residual"].cuda(), inp["gamma"].cuda()

    def out_buf():
        z = torch.empty(M, N, dtype=x.dtype)
        return _shifted_like(z, 1) if phase == "mismatched" else z.cuda()

    # one phase: the vector kernel, except the 16-bit LayerNorm up to 1024 whole 16-byte
    # chunks (the phase-class kernel)
    wide = N * synth.ELEM_BYTES[dt] // 16 > 1024
    ln_phase = phase == "same" and not wide and dt != "f32"
    engine = "engine=generic vec" if phase == "same" else "engine=generic"
    plans = []
    y, rstd = rn.rmsnorm_fwd(x, g, 1e-6, y=out_buf())
    plans.append(native.last_plan())
    o, ro, frstd = rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6, out=out_buf(), residual_out=out_buf())
    plans.append(native.last_plan())
    yl, mean, lrstd = rn.layernorm_fwd(x, g, g, 1e-5, y=out_buf())
    plans.append(native.last_plan())
    torch.cuda.synchronize()
    for op, plan in zip(("rmsnorm_fwd", "fused_add_fwd", "layernorm_fwd"), plans):
        want = "engine=generic phase" if (op == "layernorm_fwd" and ln_phase) else engine
        assert plan == "%s %s" % (op, want) or plan.startswith("%s %s " % (op, want)), plan
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(1e-6))
    o64, a64, frstd64 = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(1e-6), dt)
    yl64, mean64, lrstd64 = oracle.layernorm_fwd(x64, g64, g64, np.float32(1e-5))
    parity.check_tensor("y", y, y64, dt, "y")
    _check_rstd(rstd, rstd64)
    assert np.array_equal(parity.to64(ro), a64)
    parity.check_tensor("out", o, o64, dt, "y")
    _check_rstd(frstd, frstd64)
    parity.check_tensor("layernorm y", yl, yl64, dt, "y")
    tol = 2.0**-24 * (8 + 4 * np.sqrt(N))
    assert np.all(np.abs(parity.to64(mean) - mean64) <= tol * np.mean(np.abs(x64), axis=1))
    assert np.all(np.abs(parity.to64(lrstd) - lrstd64) <= tol * lrstd64)


def test_unaligned_fwd_gamma_off_16_bytes():
    """gamma itself off 16-byte alignment: the phase-class kernel gathers it
    element by element."""
    M, N, dt = 33, 1001, "bf16"
    inp = synth.make_inputs(Case("unaligned gamma", M, N, dt, seed=32))
    x64, g64 = parity.to64(inp["x"]), parity.to64(inp["gamma"])
    g = _shifted_like(inp["gamma"], 3)
    y, rstd = rn.rmsnorm_fwd(inp["x"].cuda(), g, 1e-6)
    torch.cuda.synchronize()
    assert native.last_plan().startswith("rmsnorm_fwd engine=generic phase"), native.last_plan()
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(1e-6))
    parity.check_tensor("y", y, y64, dt, "y")
    _check_rstd(rstd, rstd64)


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_unaligned_layernorm_fwd_params_off_16_bytes(dt):
    """LayerNorm forward on rows that are not 16-byte multiples with gamma and
    beta off 16-byte alignment: the phase-class kernel gathers both."""
    M, N = 77, 2999
    inp = synth.make_inputs(Case("unaligned ln params", M, N, dt, seed=33))
    x64, g64 = parity.to64(inp["x"]), parity.to64(inp["gamma"])
    b = (inp["gamma"].float() * 0.5 - 0.25).to(inp["gamma"].dtype)
    b64 = parity.to64(b)
    g, bb = _shifted_like(inp["gamma"], 1), _shifted_like(b, 3)
    y, mean, rstd = rn.layernorm_fwd(inp["x"].cuda(), g, bb, 1e-5)
    torch.cuda.synchronize()
    assert native.last_plan().startswith("layernorm_fwd engine=generic phase"), native.last_plan()
    y64, mean64, rstd64 = oracle.layernorm_fwd(x64, g64, b64, np.float32(1e-5))
    parity.check_tensor("layernorm y", y, y64, dt, "y")
    tol = 2.0**-24 * (8 + 4 * np.sqrt(N))
    assert np.all(np.abs(parity.to64(mean) - mean64) <= tol * np.mean(np.abs(x64), axis=1))
    assert np.all(np.abs(parity.to64(rstd) - rstd64) <= tol * rstd64)
