"""The staged phase-class kernel (rows that are not 16-byte multiples, staged in
shared memory by bulk copies) against the fp64 oracle, through the C ABI; and
its bounded wait: a wait made to run out sets the device status word and
leaves the context usable."""
import pytest
import torch

from rmsnorm_backward_bwd_gb300 import native
from rmsnorm_backward_bwd_gb300.synth import Case

import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    native.take_device_status()
    yield
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)


def _plan_field(plan, key):
    return int(plan.split(key + "=")[1].split()[0])


def _period(N, dt):
    """Rows until the alignment phase of a row repeats: 16 / gcd(16, N*s mod 16)."""
    import math
    d = (N * (4 if dt == "f32" else 2)) % 16
    return 1 if d == 0 else 16 // math.gcd(16, d)


SHAPES = [
    (1000, 4095, "bf16", False), (333, 4100, "bf16", True), (97, 2999, "f32", False),
    (130, 1001, "f16", True), (5, 7, "bf16", False), (3, 3, "f32", True), (64, 515, "bf16", True),
    (17, 8183, "bf16", False), (33, 4095, "f32", True), (300, 2050, "f16", False),
    (9, 6, "f16", True), (333, 12290, "bf16", False), (97, 16391, "bf16", True),
    (50, 8201, "f16", True), (17, 6001, "f32", True), (9, 16390, "f16", False),
    (1, 4095, "bf16", True), (2, 1, "f32", False), (611, 8190, "bf16", False)]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("M,N,dt,fused", SHAPES, ids=lambda v: str(v))
def test_staged_kernel(M, N, dt, fused, mode):
    """Each CTA on one residue class of rows modulo the phase period (M below,
    above and not a multiple of it), every warp staging its own span of the
    rows; rows of 1 to 2048 whole chunks (one to fifteen teams a CTA); both
    weight-gradient modes. No wait runs out."""
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    ex = parity.expected_bwd(Case("staged %s" % dt, M, N, dt, fused=fused, with_dres=fused,
                                  seed=51))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert plan.startswith("engine=generic staged "), plan
    assert ("atomic" if mode == 2 else "scratch") in plan, plan
    period = _period(N, dt)
    grid = _plan_field(plan, "grid")
    assert grid >= min(M, period) and (grid >= M or grid % period == 0), plan
    # the degenerate widths (N of a few elements) may need the round-off escape
    n_esc = parity.check_bwd(ex, *out, tag=" [%s]" % plan, allow_ill_conditioned=N <= 8)
    assert N <= 8 or n_esc == 0
    assert native.take_device_status() == 0


@pytest.mark.parametrize("cpt,teams,slots", [(1, 0, 0), (2, 0, 0), (0, 1, 0), (0, 3, 0),
                                             (0, 0, 3), (0, 0, 4), (2, 3, 3)])
@pytest.mark.parametrize("M,N,dt,fused", [(1000, 4095, "bf16", True), (97, 2999, "f32", False),
                                          (130, 1001, "f16", True), (300, 2050, "bf16", False)],
                         ids=lambda v: str(v))
def test_staged_kernel_forced_tiles(M, N, dt, fused, cpt, teams, slots):
    """Chunks per thread, teams per CTA and slots per team forced through the
    options: the rows still map onto the warps' spans and the ring."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    native.set_option(native.OPT_CHUNKS_PER_THREAD, cpt)
    native.set_option(native.OPT_TEAMS_PER_CTA, teams)
    native.set_option(native.OPT_STAGES, slots)
    ex = parity.expected_bwd(Case("staged tile %s" % dt, M, N, dt, fused=fused, with_dres=fused,
                                  seed=52))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    chunks = N * (4 if dt == "f32" else 2) // 16
    if cpt and (chunks + cpt - 1) // cpt > 512:
        # a team of more than 512 threads: the phase-class kernel takes the rows instead
        assert plan.startswith("engine=generic phase "), plan
        assert parity.check_bwd(ex, *out, tag=" [%s]" % plan) == 0
        return
    assert plan.startswith("engine=generic staged "), plan
    if cpt:
        assert _plan_field(plan, "cpt") == cpt, plan
    if teams and teams * _plan_field(plan, "team_threads") <= 512:   # else the planner's count
        assert _plan_field(plan, "teams") == teams, plan
    if slots:
        assert _plan_field(plan, "slots") == slots, plan
    assert parity.check_bwd(ex, *out, tag=" [%s]" % plan) == 0
    assert native.take_device_status() == 0


def _offset(t, shift):
    buf = torch.empty(t.numel() + shift, dtype=t.dtype, device="cuda")
    v = buf[shift:].view(t.shape)
    v.copy_(t.cuda())
    return v


@pytest.mark.parametrize("shift", [1, 3])
@pytest.mark.parametrize("N,dt", [(4096, "bf16"), (1024, "f32"), (8192, "f16"), (4095, "bf16")])
def test_staged_kernel_offset_base(N, dt, shift):
    """Row tensors that all start off a 16-byte boundary (one phase): every
    class has head elements, the bulk copies start inside the rows."""
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    ex = parity.expected_bwd(Case("staged base %s" % dt, 77, N, dt, seed=53))
    x, dy = _offset(ex.x, shift), _offset(ex.dy, shift)
    dx = _offset(torch.zeros_like(ex.x), shift)
    dx, dw, dw32 = rn.rmsnorm_bwd(x, ex.gamma.cuda(), dy, ex.rstd.cuda(), dx=dx)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert plan.startswith("engine=generic staged "), plan
    assert parity.check_bwd(ex, dx, dw, dw32, tag=" [%s]" % plan) == 0


@pytest.mark.parametrize("grid", [1, 3, 9])
def test_staged_kernel_small_grid_and_dres_as_dx(grid):
    """The grid option below the phase period still leaves one CTA per residue
    class (bf16 N = 8190: period 4); dx is written over dresidual_out in place
    (each row's dresidual_out is staged before its dx is stored)."""
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    native.set_option(native.OPT_GRID, grid)
    ex = parity.expected_bwd(Case("staged grid", 501, 8190, "bf16", fused=True, with_dres=True,
                                  seed=54))
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    dres = ex.dres.cuda()
    dx, _, dw, dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, dx=dres)
    torch.cuda.synchronize()
    plan = native.last_plan()
    assert "staged" in plan and "grid=%d " % max(4, grid // 4 * 4) in plan, plan
    assert dx.data_ptr() == dres.data_ptr()
    assert parity.check_bwd(ex, dx, dw, dw32) == 0


@pytest.mark.parametrize("skip", [1, 3])
@pytest.mark.parametrize("mode", [1, 2])
def test_staged_kernel_wait_runs_out(skip, mode):
    """The test hook leaves one row of the first team uncopied: that team's
    bounded wait runs out, the call sets bit 0 of the device status word, and
    the context stays usable: the next call, without the hook, matches the
    oracle and leaves the status clear."""
    import rmsnorm_backward_bwd_gb300 as rn
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    # bf16 N = 4095: period 8, 152 CTAs, 4 teams: CTA 0's first team has 4 rows of 2000
    ex = parity.expected_bwd(Case("staged timeout", 2000, 4095, "bf16", seed=55))
    native.set_option(native.OPT_TEST_WAIT_TIMEOUT, skip)
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    rn.rmsnorm_bwd(x, g, dy, rstd)
    assert native.take_device_status() == 1
    assert native.take_device_status() == 0   # read and cleared
    native.set_option(native.OPT_TEST_WAIT_TIMEOUT, 0)
    out = parity.run_gpu_bwd(ex)
    assert parity.check_bwd(ex, *out) == 0
    assert native.take_device_status() == 0


@pytest.mark.parametrize("M,N,dt,fused,engine", [
    (2048, 4095, "bf16", False, "staged"), (2047, 4095, "bf16", False, "phase"),
    (4096, 1001, "f16", True, "staged"), (1024, 1001, "f16", True, "phase"),
    (2048, 8197, "f32", False, "vec")],   # 2049 whole f32 chunks: past both phase kernels
    ids=lambda v: str(v))
def test_staged_kernel_default_choice(M, N, dt, fused, engine):
    """The automatic choice: the staged kernel from 2048 rows (within 2048
    whole chunks a row), the phase-class kernel below."""
    ex = parity.expected_bwd(Case("default %s" % dt, M, N, dt, fused=fused, with_dres=fused,
                                  seed=56))
    out = parity.run_gpu_bwd(ex)
    plan = native.last_plan()
    assert plan.startswith("engine=generic %s " % engine), plan
    assert parity.check_bwd(ex, *out, tag=" [%s]" % plan) == 0
