"""LayerNorm forward and backward on the GPU, through the C ABI, against the
fp64 oracle on the same seeded inputs.

Tolerances: the backward's dx, dgamma/dbeta (fp32 and cast) use the rules of
parity.py (the same ones as the RMSNorm backward). Forward: y as parity.py's
"y"; the saved fp32 mean and rstd within 2^-24*(8 + 4*sqrt(N)) of the oracle
(relative to mean|x| of the row for the mean, to rstd itself for rstd) -- the
growth of an fp32 sum of N terms with a random-walk error, with margin.
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

SHAPES = [(4096, 4096, "bf16"), (1, 4096, "bf16"), (512, 2048, "bf16"), (512, 3000, "f32"),
          (128, 4096, "f16"), (300, 768, "bf16"), (7, 1001, "bf16"), (3, 33, "f16"),
          (16, 16384, "bf16"), (2, 40000, "f32"), (64, 8192, "f32"), (8, 32768, "bf16")]


@pytest.fixture(autouse=True)
def _default_options():
    yield
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)


def _stat_tol(N):
    return 2.0**-24 * (8 + 4 * np.sqrt(N))


class LnExpected:
    pass


def expected(case, with_bias=True):
    inp = synth.make_ln_inputs(case)
    ex = LnExpected()
    ex.case = case
    ex.inp = inp
    x64, g64, dy64 = (parity.to64(inp[k]) for k in ("x", "gamma", "dy"))
    b64 = parity.to64(inp["beta"]) if with_bias else None
    ex.y64, ex.mean64, ex.rstd64 = oracle.layernorm_fwd(x64, g64, b64, np.float32(case.eps))
    ex.mean32 = oracle.round_to(ex.mean64, "f32")
    ex.rstd32 = oracle.round_to(ex.rstd64, "f32")
    ex.dx, ex.dg, ex.db = oracle.layernorm_bwd(x64, g64, dy64, ex.mean32, ex.rstd32)
    ex.x64, ex.g64, ex.dy64 = x64, g64, dy64
    return ex


def roundoff(ex):
    """fp32 round-off bound of dx's terms and their magnitude, for the
    elements of a mask (the LayerNorm counterpart of parity.roundoff_bound)."""
    def fn(mask):
        rows, cols = np.nonzero(mask.reshape(ex.x64.shape))
        N = ex.x64.shape[1]
        xc = ex.x64[rows] - ex.mean32[rows][:, None]
        rs = ex.rstd32[rows]
        w = ex.dy64[rows] * ex.g64
        c1 = np.mean(xc * rs[:, None] * w, axis=1)
        c2 = np.mean(w, axis=1)
        mxw = np.mean(np.abs(xc * w), axis=1)
        mw = np.mean(np.abs(w), axis=1)
        xh = xc[np.arange(len(rows)), cols] * rs
        wj = w[np.arange(len(rows)), cols]
        terms = np.abs(wj) + np.abs(c2) + np.abs(xh * c1)
        bound = 2.0**-24 * rs * (16 * terms + 4 * np.sqrt(N) * (np.abs(xh) * rs * mxw + mw))
        return bound, rs * terms
    return fn


def run_gpu(ex, with_dbeta=True, dev="cuda"):
    x = ex.inp["x"].to(dev)
    g = ex.inp["gamma"].to(dev)
    dy = ex.inp["dy"].to(dev)
    mean = torch.from_numpy(ex.mean32).float().to(dev)
    rstd = torch.from_numpy(ex.rstd32).float().to(dev)
    out = rn.layernorm_bwd(x, g, dy, mean, rstd, want_dbeta=with_dbeta)
    torch.cuda.synchronize()
    return out


def check(ex, out, with_dbeta=True, tag=""):
    dx, dg, db, dg32, db32 = out
    dt = ex.case.dtype
    n_esc = parity.check_tensor("dx" + tag, dx, ex.dx, dt, "dx", roundoff=roundoff(ex))
    # N <= 2 is the degenerate width: span{1, x_hat} is the whole row, so dx cancels to O(eps)
    assert n_esc == 0 or ex.case.N <= 2, (
        "dx%s: %d elements passed only on the round-off bound" % (tag, n_esc))
    parity.check_tensor("dgamma_f32" + tag, dg32, ex.dg, dt, "dweight_f32")
    parity.check_tensor("dgamma" + tag, dg, ex.dg, dt, "dweight")
    if with_dbeta:
        parity.check_tensor("dbeta_f32" + tag, db32, ex.db, dt, "dweight_f32")
        parity.check_tensor("dbeta" + tag, db, ex.db, dt, "dweight")
    else:
        assert db is None and db32 is None


@pytest.mark.parametrize("M,N,dt", SHAPES, ids=lambda v: str(v))
def test_layernorm_bwd_matches_oracle(M, N, dt):
    ex = expected(Case("ln", M, N, dt, eps=1e-5))
    check(ex, run_gpu(ex))


@pytest.mark.parametrize("M,N,dt", [(512, 2048, "bf16"), (7, 1001, "bf16"), (64, 3000, "f32")],
                         ids=lambda v: str(v))
def test_layernorm_bwd_without_dbeta(M, N, dt):
    ex = expected(Case("ln", M, N, dt, eps=1e-5, seed=4))
    check(ex, run_gpu(ex, with_dbeta=False), with_dbeta=False)


@pytest.mark.parametrize("engine", [1, 2])
@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,dt", [(1000, 4096, "bf16"), (333, 1024, "f16"), (129, 2048, "f32")],
                         ids=lambda v: str(v))
def test_layernorm_forced_engines_and_modes(engine, mode, M, N, dt):
    native.set_option(native.OPT_BWD_ENGINE, engine)
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    ex = expected(Case("ln", M, N, dt, eps=1e-5, seed=2))
    out = run_gpu(ex)
    plan = native.last_plan()
    assert ("ln_row" if engine == 1 else "ln_generic") in plan, plan
    assert ("atomic" if mode == 2 else "scratch") in plan, plan
    check(ex, out, tag=" [%s]" % plan)


@pytest.mark.parametrize("cpt,teams,stages", [(1, 1, 2), (2, 2, 2), (2, 1, 4), (4, 1, 2),
                                              (1, 2, 3)])
def test_layernorm_row_tiles(cpt, teams, stages):
    native.set_option(native.OPT_BWD_ENGINE, 1)
    native.set_option(native.OPT_CHUNKS_PER_THREAD, cpt)
    native.set_option(native.OPT_TEAMS_PER_CTA, teams)
    native.set_option(native.OPT_STAGES, stages)
    ex = expected(Case("ln", 777, 2048, "bf16", eps=1e-5, seed=6))
    out = run_gpu(ex)
    plan = native.last_plan()
    assert "cpt=%d" % cpt in plan and "teams=%d" % teams in plan and "stages=%d" % stages in plan
    check(ex, out, tag=" [%s]" % plan)


def test_layernorm_tile_over_thread_cap_is_refused():
    """One chunk per thread and four teams of 256 threads would need 1024
    threads a CTA; the LayerNorm row engine allows 512 and says so."""
    native.set_option(native.OPT_BWD_ENGINE, 1)
    native.set_option(native.OPT_CHUNKS_PER_THREAD, 1)
    native.set_option(native.OPT_TEAMS_PER_CTA, 4)
    ex = expected(Case("ln", 64, 2048, "bf16", eps=1e-5, seed=6))
    with pytest.raises(native.RNError, match="row engine cannot take"):
        run_gpu(ex)


def test_layernorm_scratch_mode_is_repeatable_and_agrees_with_atomics():
    ex = expected(Case("ln", 2048, 4096, "bf16", eps=1e-5, seed=8))
    native.set_option(native.OPT_DWEIGHT_MODE, 1)
    a = run_gpu(ex)
    b = run_gpu(ex)
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    native.set_option(native.OPT_DWEIGHT_MODE, 2)
    c = run_gpu(ex)
    assert torch.equal(a[0], c[0])   # dx does not depend on the mode
    check(ex, c)


def test_layernorm_row_sum_invariant_full_size():
    """sum_j dx_j = -c1*rstd^2*sum_j (x_j - mean32) per row (zero with the exact
    mean); checked against that value from the fp32 statistics the kernel used."""
    ex = expected(Case("ln", 4096, 4096, "bf16", eps=1e-5, seed=9))
    dx = parity.to64(run_gpu(ex)[0])
    xc = ex.x64 - ex.mean32[:, None]
    c1 = np.mean(xc * ex.rstd32[:, None] * ex.dy64 * ex.g64, axis=1)
    expect = -c1 * ex.rstd32 ** 2 * np.sum(xc, axis=1)
    scale = np.sum(np.abs(dx), axis=1)
    assert np.all(np.abs(np.sum(dx, axis=1) - expect) <= 2e-3 * scale)


def test_layernorm_empty_batch():
    x = torch.empty(0, 1024, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(1024, device="cuda", dtype=torch.bfloat16)
    dy = torch.empty_like(x)
    z = torch.empty(0, device="cuda", dtype=torch.float32)
    dx, dg, db, dg32, db32 = rn.layernorm_bwd(x, g, dy, z, z)
    torch.cuda.synchronize()
    for t in (dg, db, dg32, db32):
        assert torch.count_nonzero(t).item() == 0


def test_layernorm_misaligned_pointers_use_generic_engine():
    ex = expected(Case("ln", 64, 2048, "bf16", eps=1e-5, seed=10))
    x = torch.empty(64 * 2048 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(64, 2048)
    x.copy_(ex.inp["x"].cuda())
    mean = torch.from_numpy(ex.mean32).float().cuda()
    rstd = torch.from_numpy(ex.rstd32).float().cuda()
    out = rn.layernorm_bwd(x, ex.inp["gamma"].cuda(), ex.inp["dy"].cuda(), mean, rstd)
    torch.cuda.synchronize()
    assert "ln_generic" in native.last_plan()
    check(ex, out)


@pytest.mark.parametrize("M,N,dt", SHAPES, ids=lambda v: str(v))
@pytest.mark.parametrize("with_bias", [True, False])
def test_layernorm_fwd_matches_oracle(M, N, dt, with_bias):
    ex = expected(Case("ln", M, N, dt, eps=1e-5, seed=11), with_bias)
    beta = ex.inp["beta"].cuda() if with_bias else None
    y, mean, rstd = rn.layernorm_fwd(ex.inp["x"].cuda(), ex.inp["gamma"].cuda(), beta, 1e-5)
    torch.cuda.synchronize()
    parity.check_tensor("y", y, ex.y64, dt, "y")
    tol = _stat_tol(N)
    mabs = np.mean(np.abs(ex.x64), axis=1)
    assert np.all(np.abs(parity.to64(mean) - ex.mean64) <= tol * mabs)
    assert np.all(np.abs(parity.to64(rstd) - ex.rstd64) <= tol * ex.rstd64)


@pytest.mark.parametrize("shift,M,N,dt", [(1000.0, 64, 4096, "f32"), (-300.0, 33, 1000, "f32"),
                                          (48.0, 128, 4096, "bf16"), (12.0, 40, 8192, "f16"),
                                          (1000.0, 17, 16384, "f32")],
                         ids=lambda v: str(v))
def test_layernorm_fwd_large_mean(shift, M, N, dt):
    """Rows whose mean is far larger than their spread (x = shift + N(0, 1)): the
    statistics merged pairwise over the team (count, mean, centred sum of
    squares) keep mean and rstd within the same bound as centred rows."""
    case = Case("ln large mean", M, N, dt, eps=1e-5, seed=13)
    inp = synth.make_ln_inputs(case, x_shift=shift)
    x64, g64, b64 = (parity.to64(inp[k]) for k in ("x", "gamma", "beta"))
    y64, mean64, rstd64 = oracle.layernorm_fwd(x64, g64, b64, np.float32(case.eps))
    y, mean, rstd = rn.layernorm_fwd(inp["x"].cuda(), inp["gamma"].cuda(), inp["beta"].cuda(),
                                     1e-5)
    torch.cuda.synchronize()
    tol = _stat_tol(N)
    assert np.all(np.abs(parity.to64(mean) - mean64) <= tol * np.mean(np.abs(x64), axis=1))
    assert np.all(np.abs(parity.to64(rstd) - rstd64) <= tol * rstd64)
    # y = (x - mean)*rstd*gamma + beta: an fp32 mean of values near `shift` is off by about
    # shift*2^-24*log2(N) absolute, which y carries relative to |x - mean| ~ 1; below the
    # 16-bit dtypes' unit in the last place, far above the f32 bound
    if dt != "f32":
        parity.check_tensor("y", y, y64, dt, "y")


def test_layernorm_fwd_guards():
    x = torch.randn(4, 256, device="cuda", dtype=torch.bfloat16)
    g = torch.ones(256, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="dtype mismatch"):
        rn.layernorm_fwd(x, g, torch.zeros(256, device="cuda"), 1e-5)
    with pytest.raises(ValueError, match="beta has shape"):
        rn.layernorm_fwd(x, g, g[:128], 1e-5)


@pytest.mark.parametrize("shape,dt", [((2, 64, 1024), "f32"), ((4, 32, 4096), "bf16"),
                                      ((3, 5, 1001), "bf16"), ((8, 2048), "f16")],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("with_bias", [True, False])
def test_layernorm_autograd_matches_oracle(shape, dt, with_bias):
    M = int(np.prod(shape[:-1]))
    case = Case("ln autograd", M, shape[-1], dt, eps=1e-5, seed=12)
    inp = synth.make_ln_inputs(case)
    x64, g64, dy64 = (parity.to64(inp[k]) for k in ("x", "gamma", "dy"))
    b64 = parity.to64(inp["beta"]) if with_bias else None
    y64, mean64, rstd64 = oracle.layernorm_fwd(x64, g64, b64, np.float32(case.eps))
    ex = LnExpected()
    ex.x64, ex.g64, ex.dy64 = x64, g64, dy64
    ex.mean32, ex.rstd32 = oracle.round_to(mean64, "f32"), oracle.round_to(rstd64, "f32")
    dx64, dg64, db64 = oracle.layernorm_bwd(x64, g64, dy64, ex.mean32, ex.rstd32)
    x = inp["x"].cuda().reshape(shape).requires_grad_()
    w = inp["gamma"].cuda().requires_grad_()
    b = inp["beta"].cuda().requires_grad_() if with_bias else None
    y = rn.layernorm(x, w, b, case.eps)
    y.backward(inp["dy"].cuda().reshape(shape))
    torch.cuda.synchronize()
    parity.check_tensor("y", y.reshape(M, -1), y64, dt, "y")
    assert parity.check_tensor("dx", x.grad.reshape(M, -1), dx64, dt, "dx",
                               roundoff=roundoff(ex)) == 0
    parity.check_tensor("dgamma", w.grad, dg64, dt, "dweight")
    if with_bias:
        parity.check_tensor("dbeta", b.grad, db64, dt, "dweight")


@pytest.mark.parametrize("M,N", [(48, 12288), (16, 16384)])
def test_layernorm_rows_up_to_the_tile_limit_use_the_row_engine(M, N):
    """Rows that do not fit the default 2-chunks-per-thread tile take 4
    chunks per thread rather than the generic engine."""
    ex = expected(Case("ln", M, N, "bf16", eps=1e-5, seed=13))
    out = run_gpu(ex)
    plan = native.last_plan()
    assert "engine=ln_row" in plan and "cpt=4" in plan, plan
    check(ex, out)


@pytest.mark.parametrize("M,N,dt,tile", [(1024, 8192, "bf16", "cpt=4 team_threads=256 teams=2"),
                                         (700, 6144, "f16", "cpt=4 team_threads=192 teams=2"),
                                         (600, 4096, "f32", "cpt=4 team_threads=256 teams=2"),
                                         (1024, 16384, "bf16", "cpt=4 team_threads=512 teams=1 stages=2")],
                         ids=lambda v: str(v))
def test_layernorm_wide_rows_default_tile(M, N, dt, tile):
    """Where 2 chunks per thread would leave one team per SM, the default
    tile takes 4 chunks per thread and two teams; a team alone on its SM
    gets a 2-slot ring."""
    ex = expected(Case("ln", M, N, dt, eps=1e-5, seed=15))
    out = run_gpu(ex)
    plan = native.last_plan()
    assert "engine=ln_row" in plan and tile in plan, plan
    check(ex, out, tag=" [%s]" % plan)


@pytest.mark.parametrize("M,N,dt,csize", [(24, 32768, "bf16", 2), (6, 65536, "bf16", 4),
                                          (40, 16392, "bf16", 2), (16, 16384, "f32", 2),
                                          (3, 131072, "f16", 8)],
                         ids=lambda v: str(v))
def test_layernorm_long_rows_take_the_cluster_engine(M, N, dt, csize):
    ex = expected(Case("ln", M, N, dt, eps=1e-5, seed=14))
    out = run_gpu(ex)
    plan = native.last_plan()
    assert "engine=ln_cluster" in plan and "csize=%d" % csize in plan, plan
    check(ex, out, tag=" [%s]" % plan)


@pytest.mark.parametrize("csize", [2, 4, 8, 16])
@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("with_dbeta", [True, False])
def test_layernorm_forced_cluster_sizes(csize, mode, with_dbeta):
    native.set_option(native.OPT_BWD_ENGINE, 3)
    native.set_option(native.OPT_CLUSTER_SIZE, csize)
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    ex = expected(Case("ln", 300, 4096, "bf16", eps=1e-5, seed=15 + csize))
    out = run_gpu(ex, with_dbeta=with_dbeta)
    plan = native.last_plan()
    assert "ln_cluster" in plan and "csize=%d" % csize in plan, plan
    check(ex, out, with_dbeta=with_dbeta, tag=" [%s]" % plan)


def test_layernorm_cluster_scratch_mode_is_repeatable():
    native.set_option(native.OPT_DWEIGHT_MODE, 1)
    ex = expected(Case("ln", 100, 32768, "bf16", eps=1e-5, seed=16))
    a = run_gpu(ex)
    b = run_gpu(ex)
    assert "ln_cluster" in native.last_plan()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    check(ex, a)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("with_dbeta", [True, False])
@pytest.mark.parametrize("M,N,dt,rows", [(700, 4095, "bf16", 2), (97, 2999, "f32", 2),
                                         (130, 1001, "f16", 4), (5, 7, "bf16", 4),
                                         (40, 8190, "bf16", 2), (3, 3, "f32", 4)],
                         ids=lambda v: str(v))
def test_layernorm_generic_vector_variant(M, N, dt, rows, with_dbeta, mode):
    """Rows that are not 16-byte multiples with x, dy and dx at one phase:
    16-byte chunks plus element-wise head and tail, several rows per CTA
    iteration, dgamma / dbeta partials in shared memory; both modes, with and
    without the bias gradient. Chosen by option: the phase-class kernel takes
    these widths by default."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    native.set_option(native.OPT_GENERIC_KERNEL, 2)
    ex = expected(Case("ln vec", M, N, dt, eps=1e-5, seed=33))
    out = run_gpu(ex, with_dbeta=with_dbeta)
    plan = native.last_plan()
    assert "engine=ln_generic vec rows=%d" % rows in plan, plan
    check(ex, out, with_dbeta=with_dbeta, tag=" [%s]" % plan)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("with_dbeta", [True, False])
@pytest.mark.parametrize("M,N,dt,cpt", [(700, 4095, "bf16", 2), (97, 2999, "f32", 2),
                                        (130, 1001, "f16", 1), (5, 7, "bf16", 1),
                                        (40, 8190, "bf16", 2), (3, 3, "f32", 1),
                                        (333, 4100, "bf16", 2), (64, 1022, "f32", 1)],
                         ids=lambda v: str(v))
def test_layernorm_generic_phase_kernel(M, N, dt, cpt, with_dbeta, mode):
    """Rows that are not 16-byte multiples with x, dy and dx at one phase:
    each CTA takes the rows of one residue class modulo the phase period, with
    fixed columns per thread and both partials in registers; both modes, with
    and without the bias gradient."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    ex = expected(Case("ln phase", M, N, dt, eps=1e-5, seed=35))
    out = run_gpu(ex, with_dbeta=with_dbeta)
    plan = native.last_plan()
    assert "engine=ln_generic phase cpt=%d" % cpt in plan, plan
    assert ("atomic" if mode == 2 else "scratch") in plan, plan
    check(ex, out, with_dbeta=with_dbeta, tag=" [%s]" % plan)


def test_layernorm_generic_phase_kernel_small_grid():
    """The grid option below the phase period (bf16 N = 4095: period 8) still
    leaves one CTA per residue class."""
    native.set_option(native.OPT_GRID, 3)
    ex = expected(Case("ln phase grid", 301, 4095, "bf16", eps=1e-5, seed=36))
    out = run_gpu(ex)
    plan = native.last_plan()
    assert "phase" in plan and "grid=8" in plan, plan
    check(ex, out, tag=" [%s]" % plan)


def test_layernorm_mismatched_phases_take_the_scalar_generic_kernel():
    """dx one element off x's alignment phase: element-wise kernel."""
    M, N, dt = 48, 1000, "bf16"
    ex = expected(Case("ln scalar", M, N, dt, eps=1e-5, seed=34))
    x, g, dy = (ex.inp[k].cuda() for k in ("x", "gamma", "dy"))
    mean = torch.from_numpy(ex.mean32).float().cuda()
    rstd = torch.from_numpy(ex.rstd32).float().cuda()
    dx = torch.empty(M * N + 1, dtype=x.dtype, device="cuda")[1:].view(M, N)
    out = rn.layernorm_bwd(x, g, dy, mean, rstd, dx=dx)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert plan.startswith("engine=ln_generic") and "vec" not in plan, plan
    check(ex, out)


@pytest.mark.parametrize("M,N,dt", [(4096, 4096, "bf16"), (33, 4095, "f16"), (7, 40000, "bf16"),
                                    (64, 3000, "f32")], ids=lambda v: str(v))
def test_layernorm_casts_without_fp32_outputs(M, N, dt):
    """dgamma and dbeta asked for without their fp32 buffers: the scratch mode
    runs (even with atomics forced) and the casts match the oracle and the
    scratch mode's own casts bit for bit."""
    ex = expected(Case("ln cast only", M, N, dt, eps=1e-5, seed=44))
    native.set_option(native.OPT_DWEIGHT_MODE, 2)
    x, g, dy = (ex.inp[k].cuda() for k in ("x", "gamma", "dy"))
    mean = torch.from_numpy(ex.mean32).float().cuda()
    rstd = torch.from_numpy(ex.rstd32).float().cuda()
    dx, dg, db, dg32, db32 = rn.layernorm_bwd(x, g, dy, mean, rstd, want_f32=False)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert dg32 is None and db32 is None and "dw=scratch" in plan, plan
    parity.check_tensor("dgamma", dg, ex.dg, dt, "dweight")
    parity.check_tensor("dbeta", db, ex.db, dt, "dweight")
    native.set_option(native.OPT_DWEIGHT_MODE, 1)
    out = rn.layernorm_bwd(x, g, dy, mean, rstd)
    torch.cuda.synchronize()
    check(ex, out)
    assert torch.equal(dx, out[0]) and torch.equal(dg, out[1]) and torch.equal(db, out[2])



@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("with_dbeta", [True, False])
@pytest.mark.parametrize("M,N,dt", [(1000, 4095, "bf16"), (333, 4100, "bf16"), (97, 2999, "f32"),
                                    (130, 1001, "f16"), (5, 7, "bf16"), (3, 3, "f32"),
                                    (64, 515, "bf16"), (17, 8183, "bf16"), (33, 4095, "f32"),
                                    (300, 2050, "f16"), (9, 6, "f16"), (1, 4095, "bf16"),
                                    (2, 1, "f32"), (611, 8190, "bf16"), (40, 4099, "f32"),
                                    (97, 12290, "bf16"), (33, 16383, "bf16"), (17, 8191, "f32"),
                                    (50, 6001, "f32"), (9, 16390, "f16")],
                         ids=lambda v: str(v))
def test_layernorm_staged_kernel(M, N, dt, with_dbeta, mode):
    """The LayerNorm staged phase-class kernel (RN_OPT_GENERIC_KERNEL = 5): each CTA
    on one residue class of rows, every warp staging its own span of the rows (with
    the head and tail blocks for 16-bit types), one to fifteen teams a CTA; both
    weight-gradient modes, with and without the bias gradient. No wait runs out."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    ex = expected(Case("ln staged", M, N, dt, eps=1e-5, seed=37))
    out = run_gpu(ex, with_dbeta=with_dbeta)
    plan = native.last_plan()
    assert plan.startswith("engine=ln_generic staged "), plan
    assert ("atomic" if mode == 2 else "scratch") in plan, plan
    chunks = N * (4 if dt == "f32" else 2) // 16
    assert (" cpt=4 " in plan) == (chunks > 512), plan   # 2 chunks a thread up to 512 a row
    check(ex, out, with_dbeta=with_dbeta, tag=" [%s]" % plan)
    assert native.take_device_status() == 0


@pytest.mark.parametrize("cpt,teams,slots", [(1, 0, 0), (0, 1, 0), (0, 0, 3), (0, 0, 4),
                                             (1, 3, 3), (4, 0, 0), (2, 0, 0), (4, 3, 3)])
@pytest.mark.parametrize("M,N,dt", [(1000, 4095, "bf16"), (130, 1001, "f16"), (97, 2050, "f32"),
                                    (77, 8190, "bf16")],
                         ids=lambda v: str(v))
def test_layernorm_staged_kernel_forced_tiles(M, N, dt, cpt, teams, slots):
    """Chunks per thread, teams per CTA and slots per team forced through the options."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    native.set_option(native.OPT_CHUNKS_PER_THREAD, cpt)
    native.set_option(native.OPT_TEAMS_PER_CTA, teams)
    native.set_option(native.OPT_STAGES, slots)
    ex = expected(Case("ln staged tile", M, N, dt, eps=1e-5, seed=38))
    out = run_gpu(ex)
    plan = native.last_plan()
    chunks = N * (4 if dt == "f32" else 2) // 16
    if (cpt or (2 if chunks <= 512 else 4)) * 512 < chunks:
        # a team of more than 512 threads: the phase-class kernel takes the rows instead
        assert plan.startswith("engine=ln_generic phase "), plan
    else:
        assert plan.startswith("engine=ln_generic staged "), plan
        if cpt:
            assert " cpt=%d " % cpt in plan, plan
    check(ex, out, tag=" [%s]" % plan)
    assert native.take_device_status() == 0


@pytest.mark.parametrize("shift", [1, 3])
@pytest.mark.parametrize("N,dt", [(4096, "bf16"), (1024, "f32"), (4095, "f16")])
def test_layernorm_staged_kernel_offset_base(N, dt, shift):
    """x, dy and dx all starting off a 16-byte boundary (one phase)."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    ex = expected(Case("ln staged base", 77, N, dt, eps=1e-5, seed=39))

    def placed(t):
        buf = torch.empty(t.numel() + shift, dtype=t.dtype, device="cuda")
        v = buf[shift:].view(t.shape)
        v.copy_(t.cuda())
        return v
    x, dy = placed(ex.inp["x"]), placed(ex.inp["dy"])
    dx = placed(torch.zeros_like(ex.inp["x"]))
    mean = torch.from_numpy(ex.mean32).float().cuda()
    rstd = torch.from_numpy(ex.rstd32).float().cuda()
    out = rn.layernorm_bwd(x, ex.inp["gamma"].cuda(), dy, mean, rstd, dx=dx)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert plan.startswith("engine=ln_generic staged "), plan
    check(ex, out, tag=" [%s]" % plan)


@pytest.mark.parametrize("skip", [1, 3])
def test_layernorm_staged_kernel_wait_runs_out(skip):
    """The test hook leaves one row of the first team uncopied: the bounded wait
    runs out, rn_take_device_status() reports bit 0, and the next call is correct."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    # bf16 N = 4095: period 8, 152 CTAs, 2 teams: CTA 0's first team has 7 rows of 2000
    ex = expected(Case("ln staged timeout", 2000, 4095, "bf16", eps=1e-5, seed=40))
    native.set_option(native.OPT_TEST_WAIT_TIMEOUT, skip)
    run_gpu(ex)
    assert native.take_device_status() == 1
    assert native.take_device_status() == 0
    native.set_option(native.OPT_TEST_WAIT_TIMEOUT, 0)
    check(ex, run_gpu(ex))
    assert native.take_device_status() == 0


@pytest.mark.parametrize("M,N,dt,engine", [(2048, 2047, "bf16", "staged"),
                                           (2047, 2047, "bf16", "phase"),
                                           (4096, 1001, "f16", "staged"),
                                           (2048, 4095, "f32", "staged"),
                                           (2048, 4095, "bf16", "staged"),   # two teams: split
                                           (12160, 4095, "bf16", "phase"),   # 40 rows a CTA
                                           (4096, 8190, "bf16", "staged"),   # 4 chunks, split
                                           (2048, 12290, "bf16", "staged"),  # 4 chunks a thread
                                           (300, 12290, "bf16", "staged"),   # past 1024 chunks
                                           (300, 4095, "bf16", "phase"),
                                           (2048, 16393, "bf16", "vec")],    # 2049 chunks
                         ids=lambda v: str(v))
def test_layernorm_staged_kernel_default_choice(M, N, dt, engine):
    """The automatic choice: the staged kernel from 2048 rows, the phase-class kernel
    below (rows past its 1024 chunks: the staged kernel at any row count); a tile of
    two 256-thread teams (bf16 N = 4095) runs as one team a CTA, up to 40 rows a CTA
    of two CTAs an SM (the phase-class kernel, which prefetches, beyond)."""
    ex = expected(Case("ln default", M, N, dt, eps=1e-5, seed=41))
    out = run_gpu(ex)
    plan = native.last_plan()
    assert plan.startswith("engine=ln_generic %s " % engine), plan
    if N == 4095 and dt == "bf16" and engine == "staged":
        assert " teams=1 " in plan and " grid=304 " in plan, plan
    check(ex, out, tag=" [%s]" % plan)


@pytest.mark.parametrize("N,dt", [(6144, "f16"), (6120, "bf16"), (6140, "bf16")])
def test_layernorm_phase_kernel_near_48k_of_shared_memory(N, dt):
    """The phase-class kernel's atomic-mode partials take 8N bytes of dynamic shared
    memory: at N = 6120..6144 that and the kernel's static shared memory together pass
    the 48 KB a launch may use without the opt-in, which the launch must then set."""
    native.set_option(native.OPT_DWEIGHT_MODE, 2)
    ex = expected(Case("ln 48k", 275, N, dt, eps=1e-5, seed=42))
    x = torch.empty(275 * N + 1, dtype=ex.inp["x"].dtype, device="cuda")[1:].view(275, N)
    x.copy_(ex.inp["x"].cuda())
    dy = torch.empty(275 * N + 1, dtype=ex.inp["dy"].dtype, device="cuda")[1:].view(275, N)
    dy.copy_(ex.inp["dy"].cuda())
    dx = torch.empty(275 * N + 1, dtype=ex.inp["x"].dtype, device="cuda")[1:].view(275, N)
    mean = torch.from_numpy(ex.mean32).float().cuda()
    rstd = torch.from_numpy(ex.rstd32).float().cuda()
    out = rn.layernorm_bwd(x, ex.inp["gamma"].cuda(), dy, mean, rstd, dx=dx)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert "ln_generic phase" in plan and "atomic" in plan, plan
    check(ex, out, tag=" [%s]" % plan)
