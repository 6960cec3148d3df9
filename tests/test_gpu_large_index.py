"""Row tensors of more than 2^31 elements: every byte offset past the 32-bit
range must be formed in 64 bits. The inputs repeat a block of B rows (row r
holds base row r mod B), so each output row equals the oracle's output for its
base row, and the weight gradient is (M / B) times the oracle's over the block.
Sampled rows cover the start, the rows around element 2^31 and the end; the
weight gradient covers every row. Backward (row, staged, cluster and vector
engines, plain and fused with dresidual_out, both weight-gradient modes),
LayerNorm backward (row engine and staged kernel) and forwards (row engine and
staged forward)."""
import numpy as np
import pytest
import torch

import oracle
import parity
import rmsnorm_backward_bwd_gb300 as rn
from rmsnorm_backward_bwd_gb300 import native, synth
from rmsnorm_backward_bwd_gb300.synth import Case

pytestmark = pytest.mark.gpu

B = 64  # rows of the repeated block


@pytest.fixture(autouse=True)
def _reset_options():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    yield
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    torch.cuda.empty_cache()


def _rows_to_check(M, N):
    """The first rows, the rows around element 2^31 and the last rows."""
    r31 = (1 << 31) // N
    rows = set(range(0, 3)) | set(range(max(0, r31 - 2), min(M, r31 + 3))) | set(range(M - 3, M))
    return sorted(rows)


def _tile(t, reps):
    return t.cuda().repeat(reps, *([1] * (t.dim() - 1)))


@pytest.mark.parametrize("N,engine", [(8192, "row"), (8190, "generic staged"), (32768, "cluster"),
                                      (16393, "generic vec")])
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("mode", [1, 2])
def test_backward_past_2_31_elements(N, engine, fused, mode):
    reps = ((1 << 31) // N) // B + 3      # M*N > 2^31
    M = B * reps
    assert M * N > (1 << 31)
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    ex = parity.expected_bwd(Case("large base", B, N, "bf16", fused=fused, with_dres=fused,
                                  seed=71))
    x, dy, rstd = _tile(ex.x, reps), _tile(ex.dy, reps), _tile(ex.rstd, reps)
    g = ex.gamma.cuda()
    if fused:
        dres = _tile(ex.dres, reps)
        dx, _, dw, dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres)
        del dres
    else:
        dx, dw, dw32 = rn.rmsnorm_bwd(x, g, dy, rstd)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert plan.startswith("engine=%s " % engine), plan
    del x, dy, rstd
    rows = _rows_to_check(M, N)
    got = dx[rows].cpu()
    del dx
    ref = ex.dx[[r % B for r in rows]]
    parity.check_tensor("dx rows %s [%s]" % (rows, plan), got, ref, "bf16", "dx")
    dw_ref = ex.dw * reps
    parity.check_tensor("dweight_f32 [%s]" % plan, dw32, dw_ref, "bf16", "dweight_f32")
    parity.check_tensor("dweight [%s]" % plan, dw, dw_ref, "bf16", "dweight")


@pytest.mark.parametrize("N,engine", [(8192, "row"), (8190, "generic staged")])
def test_forwards_past_2_31_elements(N, engine):
    reps = ((1 << 31) // N) // B + 3
    M = B * reps
    inp = synth.make_inputs(Case("large fwd base", B, N, "bf16", fused=True, seed=72))
    x64, r64, g64 = (parity.to64(inp[k]) for k in ("x", "residual", "gamma"))
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(1e-6))
    o64, a64, frstd64 = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(1e-6), "bf16")
    yl64, mean64, lrstd64 = oracle.layernorm_fwd(x64, g64, g64, np.float32(1e-5))
    x, g = _tile(inp["x"], reps), inp["gamma"].cuda()
    rows = _rows_to_check(M, N)
    base = [r % B for r in rows]

    y, rstd = rn.rmsnorm_fwd(x, g, 1e-6)
    torch.cuda.synchronize()
    assert ("engine=%s " % engine) in native.last_plan(), native.last_plan()
    parity.check_tensor("y", y[rows].cpu(), y64[base], "bf16", "y")
    got = parity.to64(rstd[rows])
    assert np.all(np.abs(got - rstd64[base]) <= 4 * 2.0**-24 * rstd64[base])
    del y, rstd

    yl, mean, lrstd = rn.layernorm_fwd(x, g, g, 1e-5)
    torch.cuda.synchronize()
    assert ("engine=%s " % engine) in native.last_plan(), native.last_plan()
    parity.check_tensor("layernorm y", yl[rows].cpu(), yl64[base], "bf16", "y")
    del yl, mean, lrstd

    r = _tile(inp["residual"], reps)
    o, ro, frstd = rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6)
    torch.cuda.synchronize()
    del x, r
    assert np.array_equal(parity.to64(ro[rows]), a64[base])
    parity.check_tensor("out", o[rows].cpu(), o64[base], "bf16", "y")


@pytest.mark.parametrize("N,engine", [(8192, "ln_row"), (8190, "ln_generic staged")])
def test_layernorm_backward_past_2_31_elements(N, engine):
    reps = ((1 << 31) // N) // B + 3
    M = B * reps
    inp = synth.make_ln_inputs(Case("large ln base", B, N, "bf16", eps=1e-5, seed=73))
    x64, g64, dy64 = (parity.to64(inp[k]) for k in ("x", "gamma", "dy"))
    _, mean64, rstd64 = oracle.layernorm_fwd(x64, g64, None, np.float32(1e-5))
    mean32, rstd32 = oracle.round_to(mean64, "f32"), oracle.round_to(rstd64, "f32")
    dx64, dg64, db64 = oracle.layernorm_bwd(x64, g64, dy64, mean32, rstd32)
    x, dy = _tile(inp["x"], reps), _tile(inp["dy"], reps)
    mean = _tile(torch.from_numpy(mean32).float(), reps)
    rstd = _tile(torch.from_numpy(rstd32).float(), reps)
    dx, dg, db, dg32, db32 = rn.layernorm_bwd(x, inp["gamma"].cuda(), dy, mean, rstd)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert plan.startswith("engine=%s " % engine), plan
    del x, dy
    rows = _rows_to_check(M, N)
    parity.check_tensor("dx rows [%s]" % plan, dx[rows].cpu(), dx64[[r % B for r in rows]],
                        "bf16", "dx")
    parity.check_tensor("dgamma_f32 [%s]" % plan, dg32, dg64 * reps, "bf16", "dweight_f32")
    parity.check_tensor("dbeta_f32 [%s]" % plan, db32, db64 * reps, "bf16", "dweight_f32")
