"""Backward parity: the CUDA library (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from rmsnorm_backward_bwd_gb300 import native, synth
from rmsnorm_backward_bwd_gb300.synth import Case

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    yield
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)


WORKLOADS = [synth.SMALL_F32, synth.PLAIN_4096, synth.FUSED_4096, synth.FUSED_4096_NODRES,
             *synth.edge_cases()]


@pytest.mark.parametrize("case", WORKLOADS, ids=lambda c: c.name)
def test_bwd_matches_oracle(case):
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    assert parity.check_bwd(ex, dx, dw, dw32) == 0   # no element on the round-off escape
    assert "engine=" in native.last_plan()


@pytest.mark.parametrize("eps", [1e-5, 1e-6, 1e-2])
@pytest.mark.parametrize("shape", [(128, 1024, "f32"), (512, 4096, "bf16"), (512, 3000, "f32"),
                                   (128, 4096, "f16")], ids=lambda v: "%dx%d %s" % v)
@pytest.mark.parametrize("fused", [False, True])
def test_bwd_eps_sweep(eps, shape, fused):
    """The workloads' shapes with the forward's eps varied (the saved rstd
    changes with it): no dx element may need the round-off escape."""
    M, N, dt = shape
    case = Case("eps %g %s M=%d N=%d" % (eps, dt, M, N), M, N, dt, fused=fused, with_dres=fused,
                eps=eps, dy_scale=1.0 if dt == "f32" and N == 1024 else 0.01)
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    assert parity.check_bwd(ex, dx, dw, dw32) == 0


@pytest.mark.parametrize("case", [synth.LARGE_PLAIN, synth.LARGE_FUSED], ids=lambda c: c.name)
def test_bwd_large_training_shape(case):
    """16384 x 8192 bf16: the whole tensor against the oracle (all rows)."""
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    assert parity.check_bwd(ex, dx, dw, dw32) == 0
    assert native.last_plan().startswith("engine=row")


SWEEP = [
    Case("bf16 M=33 N=4096", 33, 4096, "bf16"),
    Case("bf16 M=300 N=2048 fused", 300, 2048, "bf16", fused=True, with_dres=True),
    Case("f32 M=7 N=3000", 7, 3000, "f32"),
    Case("f16 M=65 N=1024 fused nodres", 65, 1024, "f16", fused=True),
    Case("bf16 M=5 N=64", 5, 64, "bf16"),
    Case("f32 M=200 N=8", 200, 8, "f32"),
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: c.name)
@pytest.mark.parametrize("engine,mode", [(1, 1), (1, 2), (2, 1), (2, 2)],
                         ids=["row-scratch", "row-atomic", "generic-scratch", "generic-atomic"])
def test_forced_engines(case, engine, mode):
    native.set_option(native.OPT_BWD_ENGINE, engine)
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    parity.check_bwd(ex, dx, dw, dw32)
    plan = native.last_plan()
    assert ("engine=row" if engine == 1 else "engine=generic") in plan, plan
    assert ("dw=atomic" if mode == 2 else "dw=scratch") in plan, plan


@pytest.mark.parametrize("cpt", [1, 2, 4])
@pytest.mark.parametrize("teams,stages", [(1, 1), (1, 8), (2, 3), (3, 4)])
def test_row_engine_tile_shapes(cpt, teams, stages):
    case = Case("bf16 M=97 N=2048 fused", 97, 2048, "bf16", fused=True, with_dres=True)
    native.set_option(native.OPT_BWD_ENGINE, 1)
    native.set_option(native.OPT_CHUNKS_PER_THREAD, cpt)
    native.set_option(native.OPT_TEAMS_PER_CTA, teams)
    native.set_option(native.OPT_STAGES, stages)
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    parity.check_bwd(ex, dx, dw, dw32)
    plan = native.last_plan()
    assert "cpt=%d" % cpt in plan and "teams=%d" % teams in plan and "stages=%d" % stages in plan


@pytest.mark.parametrize("M", [7, 513, 4096])
def test_row_engine_warp_per_row(M):
    """One warp per row: bf16 N = 1024 is 128 chunks, 4 chunks per thread of a
    32-thread team (measured against the default team shapes: not faster)."""
    native.set_option(native.OPT_BWD_ENGINE, 1)
    native.set_option(native.OPT_CHUNKS_PER_THREAD, 4)
    native.set_option(native.OPT_TEAMS_PER_CTA, 12)
    ex = parity.expected_bwd(Case("bf16 M=%d N=1024 fused" % M, M, 1024, "bf16", fused=True,
                                  with_dres=True))
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert "team_threads=32 " in plan and "cpt=4" in plan, plan
    assert parity.check_bwd(ex, dx, dw, dw32) == 0


def test_auto_weight_gradient_mode_by_size():
    """Automatic mode: scratch partials for small problems, atomics for large."""
    ex = parity.expected_bwd(Case("f16 M=128 N=4096", 128, 4096, "f16"))
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    assert "dw=scratch" in native.last_plan()
    parity.check_bwd(ex, dx, dw, dw32)
    ex = parity.expected_bwd(Case("bf16 M=1024 N=4096", 1024, 4096, "bf16"))
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    assert "dw=atomic" in native.last_plan()
    parity.check_bwd(ex, dx, dw, dw32)


@pytest.mark.parametrize("grid", [1, 3, 152])
def test_row_engine_grid_caps(grid):
    native.set_option(native.OPT_GRID, grid)
    case = Case("bf16 M=1000 N=4096", 1000, 4096, "bf16")
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    parity.check_bwd(ex, dx, dw, dw32)


def test_scratch_mode_is_bitwise_repeatable():
    native.set_option(native.OPT_DWEIGHT_MODE, 1)
    ex = parity.expected_bwd(Case("bf16 M=2048 N=4096", 2048, 4096, "bf16"))
    a = parity.run_gpu_bwd(ex)
    b = parity.run_gpu_bwd(ex)
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2]) and torch.equal(a[1], b[1])


def test_fused_dx_may_alias_dresidual_out():
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_DWEIGHT_MODE, 1)  # bitwise comparison: deterministic dweight
    case = Case("bf16 M=257 N=4096 fused", 257, 4096, "bf16", fused=True, with_dres=True)
    ex = parity.expected_bwd(case)
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    dres = ex.dres.cuda()
    ref_dx, _, ref_dw, ref_dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres.clone())
    buf = dres.clone()
    dx, dres_grad, dw, dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, buf, dx=buf)
    torch.cuda.synchronize()
    assert dx.data_ptr() == buf.data_ptr() == dres_grad.data_ptr()
    assert torch.equal(dx, ref_dx) and torch.equal(dw32, ref_dw32)
    parity.check_bwd(ex, dx, dw, dw32)


def test_fused_with_zero_residual_grad_equals_plain():
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_DWEIGHT_MODE, 1)  # bitwise comparison: deterministic dweight
    ex = parity.expected_bwd(Case("bf16 M=128 N=4096", 128, 4096, "bf16"))
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    dx, dw, dw32 = rn.rmsnorm_bwd(x, g, dy, rstd)
    for dres in (None, torch.zeros_like(x)):
        fdx, _, fdw, fdw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres)
        assert torch.equal(fdx, dx) and torch.equal(fdw32, dw32) and torch.equal(fdw, dw)


def test_empty_batch_zeroes_dweight():
    import rmsnorm_backward_bwd_gb300 as rn
    g = torch.ones(4096, dtype=torch.bfloat16, device="cuda")
    x = torch.empty(0, 4096, dtype=torch.bfloat16, device="cuda")
    rstd = torch.empty(0, dtype=torch.float32, device="cuda")
    dw32 = torch.full((4096,), 7.0, device="cuda")
    dw = torch.full((4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    rn.rmsnorm_bwd(x, g, x, rstd, dweight_f32=dw32, dweight=dw)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw32).item() == 0 and torch.count_nonzero(dw).item() == 0


@pytest.mark.parametrize("M,N,dt", [(1, 1, "f32"), (3, 7, "bf16"), (9, 33, "f16"),
                                    (17, 1001, "bf16"), (2, 4099, "f32"), (40, 16384, "bf16"),
                                    (3, 16392, "bf16"), (2, 60000, "f32"), (5, 131072, "bf16")])
@pytest.mark.parametrize("fused", [False, True])
def test_odd_and_extreme_widths(M, N, dt, fused):
    case = Case("%s M=%d N=%d" % (dt, M, N), M, N, dt, fused=fused, with_dres=fused)
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    # N = 1 is the degenerate width: x_hat^2 = ms/(ms+eps), so dx cancels to O(eps)
    parity.check_bwd(ex, dx, dw, dw32, allow_ill_conditioned=N == 1)


def test_misaligned_pointers_take_generic_path():
    import rmsnorm_backward_bwd_gb300 as rn
    case = Case("bf16 M=64 N=4096", 64, 4096, "bf16")
    ex = parity.expected_bwd(case)
    M, N = case.M, case.N
    # storage shifted by one element: rows stay contiguous, bases are 2 mod 16
    def shifted(t):
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        v = buf[1:].view(t.shape)
        v.copy_(t.cuda())
        return v
    x, dy = shifted(ex.x), shifted(ex.dy)
    g, rstd = ex.gamma.cuda(), ex.rstd.cuda()
    dx = torch.empty(M * N + 1, dtype=x.dtype, device="cuda")[1:].view(M, N)
    dx, dw, dw32 = rn.rmsnorm_bwd(x, g, dy, rstd, dx=dx)
    torch.cuda.synchronize()
    assert native.last_plan().startswith("engine=generic")
    parity.check_bwd(ex, dx, dw, dw32)


def test_workspace_contents_do_not_matter():
    """The workspace is scratch: garbage left in it changes nothing."""
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_DWEIGHT_MODE, 1)  # the mode that uses the workspace
    ex = parity.expected_bwd(Case("bf16 M=512 N=4096", 512, 4096, "bf16"))
    a = parity.run_gpu_bwd(ex)
    ws = rn.bwd_workspace(512, 4096, torch.bfloat16, "cuda")
    ws.fill_(0x7F)
    b = parity.run_gpu_bwd(ex)
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])


def test_invariant_holds_at_full_size():
    """sum_j x_j*dx_j = eps*rstd^3*sum_j x_j*gamma_j*dy_j per row (any size),
    here with rstd computed by the oracle for 4096 x 4096 bf16."""
    case = synth.PLAIN_4096
    ex = parity.expected_bwd(case)
    dx, _, _ = parity.run_gpu_bwd(ex)
    x = parity.to64(ex.x)
    d = parity.to64(dx)
    g = parity.to64(ex.gamma)
    dy = parity.to64(ex.dy)
    r = parity.to64(ex.rstd)
    lhs = np.sum(x * d, axis=1)
    rhs = np.float32(case.eps) * r ** 3 * np.sum(x * g * dy, axis=1)
    # dx is bf16-rounded: each term carries up to half an ulp of error
    bound = np.sum(np.abs(x) * parity.ulp(d, "bf16"), axis=1) + 1e-6 * np.sum(np.abs(x * d), axis=1)
    # rstd is fp32 (not exactly (ms+eps)^-1/2): the identity then holds up to that rounding
    bound += 4 * 2.0**-24 * np.abs(np.sum(x * g * dy, axis=1)) * r
    assert np.all(np.abs(lhs - rhs) <= bound)


@pytest.mark.parametrize("case", [synth.PLAIN_4096, synth.FUSED_4096], ids=lambda c: c.name)
def test_atomic_and_scratch_dweight_modes_agree(case):
    ex = parity.expected_bwd(case)
    out = {}
    for mode in (1, 2):
        native.set_option(native.OPT_DWEIGHT_MODE, mode)
        dx, dw, dw32 = parity.run_gpu_bwd(ex)
        parity.check_bwd(ex, dx, dw, dw32)
        assert ("dw=atomic" if mode == 2 else "dw=scratch") in native.last_plan()
        out[mode] = (dx, dw32)
    assert torch.equal(out[1][0], out[2][0])  # dx does not depend on the mode
    parity.check_tensor("dweight_f32 atomic vs scratch", out[2][1], parity.to64(out[1][1]),
                        case.dtype, "dweight_f32")


def test_generic_engine_falls_back_to_scratch_partials_for_wide_rows():
    """Rows too wide for the generic engine's shared-memory partial use the
    scratch mode by default; forcing atomics there is refused."""
    case = Case("f32 M=2 N=60001", 2, 60001, "f32")
    ex = parity.expected_bwd(case)
    dx, dw, dw32 = parity.run_gpu_bwd(ex)
    parity.check_bwd(ex, dx, dw, dw32)
    assert "engine=generic" in native.last_plan() and "dw=scratch" in native.last_plan()
    native.set_option(native.OPT_DWEIGHT_MODE, 2)
    with pytest.raises(native.RNError, match="atomic mode"):
        parity.run_gpu_bwd(ex)


def test_mismatched_alignment_phases_take_the_scalar_generic_kernel():
    """x one element off 16-byte alignment while dy and dx are not: no common
    phase for 16-byte chunks, so the element-wise generic kernel runs."""
    import rmsnorm_backward_bwd_gb300 as rn
    case = Case("bf16 M=48 N=1000", 48, 1000, "bf16")
    ex = parity.expected_bwd(case)
    buf = torch.empty(ex.x.numel() + 1, dtype=ex.x.dtype, device="cuda")
    x = buf[1:].view(ex.x.shape)
    x.copy_(ex.x.cuda())
    dx, dw, dw32 = rn.rmsnorm_bwd(x, ex.gamma.cuda(), ex.dy.cuda(), ex.rstd.cuda())
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert plan.startswith("engine=generic") and "vec" not in plan, plan
    parity.check_bwd(ex, dx, dw, dw32)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,dt,fused,cpb", [
    (777, 8190, "f16", False, 2), (300, 8190, "bf16", False, 2), (17, 8191, "bf16", True, 2),
    (33, 4095, "f32", True, 2), (50, 12289, "bf16", True, 4), (40, 16383, "bf16", False, 4),
    (9, 4097, "f32", False, 4)],
    ids=lambda v: str(v))
def test_generic_realigning_engine(M, N, dt, fused, cpb, mode):
    """Rows of 16 to 32 KB that are not 16-byte multiples, all tensors at one
    phase: aligned chunks through a shared row buffer, fixed column blocks
    read back by the row's phase, dx out as aligned chunks (2 and 4 blocks per
    thread; both weight-gradient modes). The kernel is chosen by option where
    the phase-class kernel would take the width."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    native.set_option(native.OPT_GENERIC_KERNEL, 3)
    ex = parity.expected_bwd(Case("realign %s" % dt, M, N, dt, fused=fused, with_dres=fused,
                                  seed=21))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert "engine=generic realign cpb=%d" % cpb in plan, plan
    assert ("atomic" if mode == 2 else "scratch") in plan, plan
    parity.check_bwd(ex, *out, tag=" [%s]" % plan)


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,dt,fused,rows", [
    (1000, 4095, "bf16", False, 2), (333, 4100, "bf16", True, 2), (97, 2999, "f32", False, 2),
    (130, 1001, "f16", True, 4), (5, 7, "bf16", False, 4), (3, 3, "f32", True, 4),
    (64, 515, "bf16", True, 4), (24, 20001, "bf16", False, 2), (16, 18001, "f16", True, 2)],
    ids=lambda v: str(v))
def test_generic_vector_variant(M, N, dt, fused, rows, mode):
    """Rows that are not 16-byte multiples, all tensors at one phase (past
    2048 whole chunks it is the default; below, forced): 16-byte chunks plus
    element-wise head and tail, several rows per CTA iteration (M not a
    multiple of them), shared partial with atomic adds; both weight-gradient
    modes. The kernel is chosen by option where another generic kernel would
    take the width."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    native.set_option(native.OPT_GENERIC_KERNEL, 2)
    ex = parity.expected_bwd(Case("vec %s" % dt, M, N, dt, fused=fused, with_dres=fused, seed=23))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert "engine=generic vec rows=%d" % rows in plan, plan
    assert ("atomic" if mode == 2 else "scratch") in plan, plan
    parity.check_bwd(ex, *out, tag=" [%s]" % plan)


def test_generic_realigning_small_grid_and_dres_as_dx():
    """Few CTAs for many rows (the grid option), and dx written over
    dresidual_out in place."""
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_GRID, 3)
    native.set_option(native.OPT_GENERIC_KERNEL, 3)
    ex = parity.expected_bwd(Case("realign grid", 501, 8190, "bf16", fused=True, with_dres=True,
                                  seed=22))
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    dres = ex.dres.cuda()
    dx, dres_out, dw, dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, dx=dres)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert "realign" in plan and "grid=3" in plan, plan
    assert dx.data_ptr() == dres.data_ptr()
    parity.check_bwd(ex, dx, dw, dw32)


def _offset(t, shift):
    """A copy of t on the GPU whose data starts `shift` elements past a
    16-byte boundary."""
    buf = torch.empty(t.numel() + shift, dtype=t.dtype, device="cuda")
    v = buf[shift:].view(t.shape)
    v.copy_(t.cuda())
    return v


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,dt,fused,cpt,period", [
    (1000, 4095, "bf16", False, 2, 8), (333, 4100, "bf16", True, 2, 2),
    (97, 2999, "f32", False, 2, 4), (130, 1001, "f16", True, 1, 8), (5, 7, "bf16", False, 1, 8),
    (3, 3, "f32", True, 1, 4), (64, 515, "bf16", True, 1, 8), (17, 8183, "bf16", False, 2, 8),
    (33, 4095, "f32", True, 2, 4), (300, 2050, "f16", False, 1, 4), (9, 6, "f16", True, 1, 4)],
    ids=lambda v: str(v))
def test_generic_phase_kernel(M, N, dt, fused, cpt, period, mode):
    """Rows that are not 16-byte multiples, all tensors at one phase: each CTA
    takes the rows of one residue class modulo the phase period (M below,
    above and not a multiple of it), with fixed columns per thread (1 and 2
    chunks per thread); both weight-gradient modes."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    ex = parity.expected_bwd(Case("phase %s" % dt, M, N, dt, fused=fused, with_dres=fused,
                                  seed=25))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert "engine=generic phase cpt=%d" % cpt in plan, plan
    assert ("atomic" if mode == 2 else "scratch") in plan, plan
    grid = int(plan.split("grid=")[1].split()[0])
    assert grid >= min(M, period) and (grid >= M or grid % period == 0), plan
    parity.check_bwd(ex, *out, tag=" [%s]" % plan)


@pytest.mark.parametrize("rows", [1, 2])
@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,dt,fused", [
    (1000, 4095, "bf16", False), (333, 4100, "bf16", True), (97, 2999, "f32", True),
    (130, 1001, "f16", True), (5, 7, "bf16", False), (17, 8183, "f16", True), (9, 6, "f16", False),
    (611, 8190, "bf16", False)],
    ids=lambda v: str(v))
def test_generic_phase_kernel_rows_per_iteration(M, N, dt, fused, mode, rows):
    """One or two rows of the class per CTA iteration (RN_OPT_TEAMS_PER_CTA),
    with M leaving the last iteration of some CTAs a single row; both
    weight-gradient modes."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    native.set_option(native.OPT_TEAMS_PER_CTA, rows)
    ex = parity.expected_bwd(Case("phase rows %s" % dt, M, N, dt, fused=fused, with_dres=fused,
                                  seed=29))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert "engine=generic phase" in plan and " rows=%d " % rows in plan, plan
    assert parity.check_bwd(ex, *out, tag=" [%s]" % plan) == 0


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,dt,fused", [
    (333, 12290, "bf16", False), (97, 16391, "bf16", True), (50, 8201, "f16", True),
    (17, 6001, "f32", True), (5, 10001, "bf16", False), (300, 4101, "f32", False),
    (9, 16390, "f16", False)],
    ids=lambda v: str(v))
def test_generic_phase_kernel_four_chunks(M, N, dt, fused, mode):
    """Rows of 1025 to 2048 whole 16-byte chunks through the phase-class kernel
    (RN_OPT_GENERIC_KERNEL = 1): four chunks a thread, one row per iteration,
    gamma chunks in shared memory for 16-bit types; both weight-gradient modes."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    native.set_option(native.OPT_GENERIC_KERNEL, 1)
    ex = parity.expected_bwd(Case("phase4 %s" % dt, M, N, dt, fused=fused, with_dres=fused,
                                  seed=30))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert "engine=generic phase cpt=4 rows=1 " in plan, plan
    assert parity.check_bwd(ex, *out, tag=" [%s]" % plan) == 0


@pytest.mark.parametrize("shift", [1, 3])
@pytest.mark.parametrize("N,dt", [(4096, "bf16"), (1024, "f32"), (8192, "f16")])
def test_generic_phase_kernel_aligned_rows_offset_base(N, dt, shift):
    """Rows of whole 16-byte chunks whose tensors all start off a 16-byte
    boundary: period 1, every row split the same way."""
    import rmsnorm_backward_bwd_gb300 as rn
    ex = parity.expected_bwd(Case("phase base %s" % dt, 77, N, dt, seed=26))
    x, dy = _offset(ex.x, shift), _offset(ex.dy, shift)
    dx = _offset(torch.zeros_like(ex.x), shift)
    dx, dw, dw32 = rn.rmsnorm_bwd(x, ex.gamma.cuda(), dy, ex.rstd.cuda(), dx=dx)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert "engine=generic phase" in plan, plan
    parity.check_bwd(ex, dx, dw, dw32, tag=" [%s]" % plan)


@pytest.mark.parametrize("grid", [1, 3, 9])
def test_generic_phase_kernel_small_grid_and_dres_as_dx(grid):
    """The grid option below the phase period still leaves one CTA per residue
    class (bf16 N = 8190: period 4); above it, a multiple of it. dx is written
    over dresidual_out in place."""
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_GRID, grid)
    ex = parity.expected_bwd(Case("phase grid", 501, 8190, "bf16", fused=True, with_dres=True,
                                  seed=27))
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    dres = ex.dres.cuda()
    dx, dres_out, dw, dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, dx=dres)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert "phase" in plan and "grid=%d" % max(4, grid // 4 * 4) in plan, plan
    assert dx.data_ptr() == dres.data_ptr()
    parity.check_bwd(ex, dx, dw, dw32)


@pytest.mark.parametrize("kernel,name", [(1, "phase"), (2, "vec"), (3, "realign"), (4, "")])
def test_generic_kernel_option(kernel, name):
    """RN_OPT_GENERIC_KERNEL picks each generic kernel on one problem (f32
    N = 4095: in every kernel's range)."""
    native.set_option(native.OPT_GENERIC_KERNEL, kernel)
    ex = parity.expected_bwd(Case("pick", 40, 4095, "f32", fused=True, with_dres=True, seed=28))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    head = plan.split()
    assert head[0] == "engine=generic" and (head[1] == name if name else "=" in head[1]), plan
    parity.check_bwd(ex, *out, tag=" [%s]" % plan)


@pytest.mark.parametrize("N,dt,engine", [
    (2055, "bf16", "engine=generic phase cpt=1"),   # 256 whole 16-byte chunks
    (2057, "bf16", "engine=generic phase cpt=2"),   # 257
    (8199, "bf16", "engine=generic phase cpt=2"),   # 1024
    (8201, "bf16", "engine=generic phase cpt=4"),   # 1025 whole chunks
    (16385, "bf16", "engine=generic phase cpt=4"),  # 2048: the phase-class kernel's widest rows
    (16393, "bf16", "engine=generic vec"),          # 2049 whole chunks
    (4099, "f32", "engine=generic phase cpt=2"),    # 1024 chunks of f32
    (4101, "f32", "engine=generic phase cpt=4")],   # 1025
    ids=lambda v: str(v))
@pytest.mark.parametrize("M", [1, 3, 64])
def test_generic_engine_thresholds(N, dt, engine, M):
    """The width thresholds between the generic kernels (phase-class with 1,
    2 or 4 chunks a thread, vector), on both sides, with few and several
    rows."""
    ex = parity.expected_bwd(Case("threshold", M, N, dt, fused=True, with_dres=True, seed=41))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert plan.startswith(engine), plan
    parity.check_bwd(ex, *out, tag=" [%s]" % plan)


def test_generic_engines_empty_batch():
    """M = 0 on unaligned rows: nothing to read, a zero weight gradient."""
    import rmsnorm_backward_bwd_gb300 as rn
    for N in (4095, 8185):
        x = torch.empty(0, N, dtype=torch.bfloat16, device="cuda")
        g = torch.ones(N, dtype=torch.bfloat16, device="cuda")
        dx, dw, dw32 = rn.rmsnorm_bwd(x, g, x, torch.empty(0, device="cuda"))
        torch.cuda.synchronize()
        assert dx.shape == (0, N) and torch.count_nonzero(dw32).item() == 0


def _run_kw(ex, **kw):
    import rmsnorm_backward_bwd_gb300 as rn
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    if ex.case.fused:
        dres = ex.dres.cuda() if ex.dres is not None else None
        dx, _, dw, dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, **kw)
    else:
        dx, dw, dw32 = rn.rmsnorm_bwd(x, g, dy, rstd, **kw)
    torch.cuda.synchronize()
    return dx, dw, dw32


@pytest.mark.parametrize("case", [
    synth.PLAIN_4096, synth.FUSED_4096, Case("bf16 M=33 N=4095", 33, 4095, "bf16"),
    Case("f16 M=9 N=40000 fused", 9, 40000, "f16", fused=True, with_dres=True),
    Case("bf16 M=300 N=12290", 300, 12290, "bf16"), Case("bf16 M=5 N=70001", 5, 70001, "bf16")],
    ids=lambda c: c.name)
def test_cast_only_weight_gradient_takes_the_scratch_mode(case):
    """dweight_f32 = NULL with dweight given: the fp32 sum is not stored and
    the scratch mode runs even with atomics forced; dweight matches the oracle
    and equals, bit for bit, the cast of the scratch mode's fp32 sum (the same
    fixed summation order)."""
    ex = parity.expected_bwd(case)
    native.set_option(native.OPT_DWEIGHT_MODE, 2)
    dx, dw, dw32 = _run_kw(ex, want_f32=False)
    plan = native.last_plan()
    assert dw32 is None and "dw=scratch" in plan, plan
    n_esc = parity.check_tensor("dx", dx, ex.dx, case.dtype, "dx",
                                roundoff=parity.roundoff_bound(ex))
    assert n_esc == 0
    parity.check_tensor("dweight", dw, ex.dw, case.dtype, "dweight")
    native.set_option(native.OPT_DWEIGHT_MODE, 1)
    dx1, dw1, _ = _run_kw(ex)
    assert torch.equal(dx, dx1) and torch.equal(dw, dw1)


def test_no_weight_gradient_asked():
    """Neither dweight_f32 nor dweight: dx alone, no weight gradient."""
    ex = parity.expected_bwd(Case("bf16 M=777 N=4096 fused", 777, 4096, "bf16", fused=True,
                                  with_dres=True))
    dx, dw, dw32 = _run_kw(ex, want_f32=False, want_cast=False)
    assert dw is None and dw32 is None
    assert parity.check_tensor("dx", dx, ex.dx, "bf16", "dx",
                               roundoff=parity.roundoff_bound(ex)) == 0


def test_cast_only_empty_batch():
    import rmsnorm_backward_bwd_gb300 as rn
    x = torch.empty(0, 4095, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(4095, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((4095,), 7.0, dtype=torch.bfloat16, device="cuda")
    dx, dw, dw32 = rn.rmsnorm_bwd(x, g, x, torch.empty(0, device="cuda"), dweight=dw,
                                  want_f32=False)
    torch.cuda.synchronize()
    assert dw32 is None and torch.count_nonzero(dw).item() == 0


@pytest.mark.parametrize("M,N,dt,fused,want", [
    (4096, 1024, "bf16", False, "cpt=1 team_threads=128 teams=6 "),   # >= 4 rows a team
    (4096, 4096, "bf16", True, "cpt=4 team_threads=128 teams=3 "),    # ring under 160 KB
    (4096, 2048, "bf16", True, "cpt=2 team_threads=128 teams=5 "),    # ring under 125 KB
    (4096, 4096, "bf16", False, "cpt=4 team_threads=128 teams=4 "),   # 131 KB ring kept
    (16384, 8192, "bf16", True, "cpt=4 team_threads=256 teams=2 "),   # too few teams to cap
    (512, 2048, "bf16", False, "cpt=2 team_threads=128 teams=4 ")],   # too few rows per SM
    ids=lambda v: str(v))
def test_row_engine_default_tiles(M, N, dt, fused, want):
    """The planner's measured tile rules pick these shapes by default, and
    the results match the oracle."""
    ex = parity.expected_bwd(Case("tile %s" % dt, M, N, dt, fused=fused, with_dres=fused,
                                  seed=45))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert plan.startswith("engine=row ") and want in plan, plan
    assert parity.check_bwd(ex, *out) == 0


@pytest.mark.parametrize("M,N,dt,fused,want", [
    (600, 8183, "f16", True, "cpt=2 rows=2 "),      # wide rows of three tensors: prefetch
    (12288, 2999, "bf16", False, "cpt=2 rows=2 "),  # >= 40 rows per CTA: prefetch
    (1000, 1001, "f16", False, "cpt=1 rows=2 "),    # one chunk a thread: prefetch
    (500, 4095, "bf16", False, "cpt=2 rows=2 ")],   # neither: no prefetch
    ids=lambda v: str(v))
def test_generic_phase_kernel_prefetch(M, N, dt, fused, want):
    """The planner's L2-prefetch choice for the phase-class kernel (forced:
    from 2048 rows the staged kernel is the default), and the results with
    and without it."""
    native.set_option(native.OPT_GENERIC_KERNEL, 1)
    ex = parity.expected_bwd(Case("phase prefetch %s" % dt, M, N, dt, fused=fused,
                                  with_dres=fused, seed=46))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert want in plan, plan
    expect = 0 if (N == 4095 and M == 500) else 1
    assert " prefetch=%d " % expect in plan, plan
    assert parity.check_bwd(ex, *out, tag=" [%s]" % plan) == 0


@pytest.mark.parametrize("N", [12288, 12280])
def test_phase_kernel_near_48k_of_shared_memory(N):
    """bf16 rows off a 16-byte boundary through the phase-class kernel in atomic mode: its
    staged partial is 4N bytes of dynamic shared memory, which with the kernel's static
    shared memory passes the 48 KB a launch may use without the opt-in."""
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_DWEIGHT_MODE, 2)
    native.set_option(native.OPT_GENERIC_KERNEL, 1)
    ex = parity.expected_bwd(Case("phase 48k", 97, N, "bf16", seed=57))
    x, dy = _offset(ex.x, 1), _offset(ex.dy, 1)
    dx = _offset(torch.zeros_like(ex.x), 1)
    dx, dw, dw32 = rn.rmsnorm_bwd(x, ex.gamma.cuda(), dy, ex.rstd.cuda(), dx=dx)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert "engine=generic phase" in plan and "atomic" in plan, plan
    assert parity.check_bwd(ex, dx, dw, dw32, tag=" [%s]" % plan) == 0
