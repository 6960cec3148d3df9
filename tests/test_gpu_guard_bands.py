"""Out-of-bounds writes, without a sanitizer: every output buffer sits inside
a larger allocation whose margins hold a canary byte pattern, and after each
call the margins must be unchanged while the outputs match the oracle. Small
and ragged shapes (one row, a few rows, widths around the vector tile and the
row engine's chunk limit) on every engine and in both weight-gradient modes.
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

CANARY = 0x5A
PAD = 4096  # bytes of margin on each side (keeps the payload 16-byte aligned)


@pytest.fixture(autouse=True)
def _reset_options():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    yield
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)


class Guarded:
    """A tensor of `shape`/`dtype` inside a canary-filled byte buffer."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((PAD + n + PAD,), CANARY, dtype=torch.uint8, device="cuda")
        self.n = n
        self.t = self.raw[PAD:PAD + n].view(dtype).view(shape)

    def margins_intact(self):
        head = self.raw[:PAD]
        tail = self.raw[PAD + self.n:]
        return bool((head == CANARY).all()) and bool((tail == CANARY).all())


SHAPES = [(M, N) for M in (1, 2, 3, 33) for N in (1, 7, 31, 33, 2047, 2049, 3000)]


@pytest.mark.parametrize("M,N", SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("mode", [1, 2])
def test_backward_writes_stay_in_bounds(M, N, dt, fused, mode):
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    case = Case("guard", M, N, dt, fused=fused, with_dres=fused, seed=M * 7 + N)
    ex = parity.expected_bwd(case)
    tdt = synth.TORCH_DTYPES[dt]
    dx = Guarded((M, N), tdt)
    dw32 = Guarded((N,), torch.float32)
    dw = Guarded((N,), tdt)
    x, g, dy, rstd = ex.x.cuda(), ex.gamma.cuda(), ex.dy.cuda(), ex.rstd.cuda()
    if fused:
        dres = ex.dres.cuda() if ex.dres is not None else None
        rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, dx=dx.t, dweight_f32=dw32.t, dweight=dw.t)
    else:
        rn.rmsnorm_bwd(x, g, dy, rstd, dx=dx.t, dweight_f32=dw32.t, dweight=dw.t)
    torch.cuda.synchronize()
    plan = native.last_plan()
    for name, buf in (("dx", dx), ("dweight_f32", dw32), ("dweight", dw)):
        assert buf.margins_intact(), "%s margin overwritten [%s]" % (name, plan)
    parity.check_bwd(ex, dx.t, dw.t, dw32.t, tag=" [%s]" % plan, allow_ill_conditioned=N == 1)


@pytest.mark.parametrize("engine", [1, 3])
@pytest.mark.parametrize("N", [8, 2048, 2056, 4096])
def test_forced_engines_write_stay_in_bounds(engine, N):
    """The row and cluster engines forced onto aligned bf16 widths."""
    native.set_option(native.OPT_BWD_ENGINE, engine)
    if engine == 3:
        native.set_option(native.OPT_CLUSTER_SIZE, 2)
    case = Case("guard", 5, N, "bf16", seed=N)
    ex = parity.expected_bwd(case)
    dx = Guarded((5, N), torch.bfloat16)
    dw32 = Guarded((N,), torch.float32)
    dw = Guarded((N,), torch.bfloat16)
    rn.rmsnorm_bwd(ex.x.cuda(), ex.gamma.cuda(), ex.dy.cuda(), ex.rstd.cuda(), dx=dx.t,
                   dweight_f32=dw32.t, dweight=dw.t)
    torch.cuda.synchronize()
    plan = native.last_plan()
    for name, buf in (("dx", dx), ("dweight_f32", dw32), ("dweight", dw)):
        assert buf.margins_intact(), "%s margin overwritten [%s]" % (name, plan)
    parity.check_bwd(ex, dx.t, dw.t, dw32.t, tag=" [%s]" % plan)


@pytest.mark.parametrize("M,N", [(1, 7), (3, 33), (33, 2047), (2, 2049), (3, 3000), (4, 4096)],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("mode", [1, 2])
def test_layernorm_writes_stay_in_bounds(M, N, mode):
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    case = Case("guard ln", M, N, "bf16", eps=1e-5, seed=M + N)
    inp = synth.make_ln_inputs(case)
    x64, g64, dy64 = (parity.to64(inp[k]) for k in ("x", "gamma", "dy"))
    _, mean64, rstd64 = oracle.layernorm_fwd(x64, g64, None, np.float32(1e-5))
    mean32, rstd32 = oracle.round_to(mean64, "f32"), oracle.round_to(rstd64, "f32")
    dx64, dg64, db64 = oracle.layernorm_bwd(x64, g64, dy64, mean32, rstd32)
    bufs = {"dx": Guarded((M, N), torch.bfloat16), "dg32": Guarded((N,), torch.float32),
            "db32": Guarded((N,), torch.float32), "dg": Guarded((N,), torch.bfloat16),
            "db": Guarded((N,), torch.bfloat16)}
    rn.layernorm_bwd(inp["x"].cuda(), inp["gamma"].cuda(), inp["dy"].cuda(),
                     torch.from_numpy(mean32).float().cuda(),
                     torch.from_numpy(rstd32).float().cuda(), dx=bufs["dx"].t,
                     dgamma_f32=bufs["dg32"].t, dbeta_f32=bufs["db32"].t, dgamma=bufs["dg"].t,
                     dbeta=bufs["db"].t)
    torch.cuda.synchronize()
    for name, buf in bufs.items():
        assert buf.margins_intact(), "%s margin overwritten [%s]" % (name, native.last_plan())
    parity.check_tensor("dx", bufs["dx"].t, dx64, "bf16", "dx")
    parity.check_tensor("dgamma_f32", bufs["dg32"].t, dg64, "bf16", "dweight_f32")
    parity.check_tensor("dbeta_f32", bufs["db32"].t, db64, "bf16", "dweight_f32")


@pytest.mark.parametrize("M,N,dt", [(1, 7, "bf16"), (3, 33, "f32"), (33, 2047, "bf16"),
                                    (2, 2049, "f32"), (5, 4096, "bf16"), (2, 32768, "bf16")],
                         ids=lambda v: str(v))
def test_forward_writes_stay_in_bounds(M, N, dt):
    tdt = synth.TORCH_DTYPES[dt]
    inp = synth.make_inputs(Case("guard fwd", M, N, dt, fused=True, seed=N))
    x, r, g = inp["x"].cuda(), inp["residual"].cuda(), inp["gamma"].cuda()
    y, rstd = Guarded((M, N), tdt), Guarded((M,), torch.float32)
    rn.rmsnorm_fwd(x, g, 1e-6, y=y.t, rstd=rstd.t)
    out, res_out, rstd2 = Guarded((M, N), tdt), Guarded((M, N), tdt), Guarded((M,), torch.float32)
    rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6, out=out.t, residual_out=res_out.t, rstd=rstd2.t)
    yl, mean, rstd3 = Guarded((M, N), tdt), Guarded((M,), torch.float32), Guarded((M,), torch.float32)
    rn.layernorm_fwd(x, g, g, 1e-5, y=yl.t, mean=mean.t, rstd=rstd3.t)
    torch.cuda.synchronize()
    for name, buf in (("y", y), ("rstd", rstd), ("out", out), ("residual_out", res_out),
                      ("fused rstd", rstd2), ("ln y", yl), ("mean", mean), ("ln rstd", rstd3)):
        assert buf.margins_intact(), "%s margin overwritten" % name
    y64, _ = oracle.rmsnorm_fwd(parity.to64(x.cpu()), parity.to64(g.cpu()), np.float32(1e-6))
    parity.check_tensor("y", y.t, y64, dt, "y")


@pytest.mark.parametrize("M,N,dt", [(1, 7, "bf16"), (3, 33, "f32"), (33, 2047, "bf16"),
                                    (2, 2049, "f16"), (3, 3000, "f32"), (17, 4095, "bf16"),
                                    (5, 8191, "f16"), (9, 16383, "bf16")],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("mode", [1, 2])
def test_staged_kernels_write_stay_in_bounds(M, N, dt, mode):
    """The staged phase-class kernels (RMSNorm backward plain and fused with
    dresidual_out, LayerNorm backward, the three forwards), forced onto
    ragged widths: no write lands in a margin."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    tdt = synth.TORCH_DTYPES[dt]
    plans = []
    for fused in (False, True):
        case = Case("guard staged", M, N, dt, fused=fused, with_dres=fused, seed=M * 3 + N)
        ex = parity.expected_bwd(case)
        dx, dw32, dw = Guarded((M, N), tdt), Guarded((N,), torch.float32), Guarded((N,), tdt)
        x, g, dy, rstd = ex.x.cuda(), ex.gamma.cuda(), ex.dy.cuda(), ex.rstd.cuda()
        if fused:
            rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, ex.dres.cuda(), dx=dx.t, dweight_f32=dw32.t,
                                     dweight=dw.t)
        else:
            rn.rmsnorm_bwd(x, g, dy, rstd, dx=dx.t, dweight_f32=dw32.t, dweight=dw.t)
        torch.cuda.synchronize()
        plans.append(native.last_plan())
        for name, buf in (("dx", dx), ("dweight_f32", dw32), ("dweight", dw)):
            assert buf.margins_intact(), "%s margin overwritten [%s]" % (name, plans[-1])
        parity.check_bwd(ex, dx.t, dw.t, dw32.t, tag=" [%s]" % plans[-1],
                         allow_ill_conditioned=N <= 8)

    inp = synth.make_ln_inputs(Case("guard staged ln", M, N, dt, eps=1e-5, seed=M + N))
    x64, g64, dy64 = (parity.to64(inp[k]) for k in ("x", "gamma", "dy"))
    _, mean64, rstd64 = oracle.layernorm_fwd(x64, g64, None, np.float32(1e-5))
    mean32, rstd32 = oracle.round_to(mean64, "f32"), oracle.round_to(rstd64, "f32")
    dx64, dg64, db64 = oracle.layernorm_bwd(x64, g64, dy64, mean32, rstd32)
    bufs = {"dx": Guarded((M, N), tdt), "dg32": Guarded((N,), torch.float32),
            "db32": Guarded((N,), torch.float32), "dg": Guarded((N,), tdt),
            "db": Guarded((N,), tdt)}
    rn.layernorm_bwd(inp["x"].cuda(), inp["gamma"].cuda(), inp["dy"].cuda(),
                     torch.from_numpy(mean32).float().cuda(),
                     torch.from_numpy(rstd32).float().cuda(), dx=bufs["dx"].t,
                     dgamma_f32=bufs["dg32"].t, dbeta_f32=bufs["db32"].t, dgamma=bufs["dg"].t,
                     dbeta=bufs["db"].t)
    torch.cuda.synchronize()
    plans.append(native.last_plan())
    for name, buf in bufs.items():
        assert buf.margins_intact(), "%s margin overwritten [%s]" % (name, plans[-1])
    parity.check_tensor("dgamma_f32", bufs["dg32"].t, dg64, dt, "dweight_f32")
    parity.check_tensor("dbeta_f32", bufs["db32"].t, db64, dt, "dweight_f32")

    finp = synth.make_inputs(Case("guard staged fwd", M, N, dt, fused=True, seed=N + 1))
    x, r, g = finp["x"].cuda(), finp["residual"].cuda(), finp["gamma"].cuda()
    outs = {k: Guarded((M, N), tdt) for k in ("y", "out", "residual_out", "ln y")}
    stats = {k: Guarded((M,), torch.float32) for k in ("rstd", "fused rstd", "mean", "ln rstd")}
    rn.rmsnorm_fwd(x, g, 1e-6, y=outs["y"].t, rstd=stats["rstd"].t)
    plans.append(native.last_plan())
    rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6, out=outs["out"].t, residual_out=outs["residual_out"].t,
                             rstd=stats["fused rstd"].t)
    plans.append(native.last_plan())
    rn.layernorm_fwd(x, g, g, 1e-5, y=outs["ln y"].t, mean=stats["mean"].t, rstd=stats["ln rstd"].t)
    plans.append(native.last_plan())
    torch.cuda.synchronize()
    for name, buf in list(outs.items()) + list(stats.items()):
        assert buf.margins_intact(), "%s margin overwritten %s" % (name, plans[-3:])
    y64, _ = oracle.rmsnorm_fwd(parity.to64(finp["x"]), parity.to64(finp["gamma"]),
                                np.float32(1e-6))
    parity.check_tensor("y", outs["y"].t, y64, dt, "y")
    # rows that are not 16-byte multiples, of at most 2048 whole chunks, took the staged kernels
    row_bytes = N * synth.ELEM_BYTES[dt]
    chunks, ragged = row_bytes // 16, row_bytes % 16 != 0
    want = [ragged and chunks <= 2048] * 6
    assert [("staged" in p) for p in plans] == want, plans
