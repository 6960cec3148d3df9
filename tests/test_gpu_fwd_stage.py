"""The forward staged phase-class kernel (RMSNorm, fused-add and LayerNorm
forwards on rows that are not 16-byte multiples, staged in shared memory by
bulk copies) against the fp64 oracle, through the C ABI; and its bounded
wait: a wait made to run out sets the device status word and leaves the
context usable."""
import numpy as np
import pytest
import torch

import oracle
import parity
import rmsnorm_backward_bwd_gb300 as rn
from rmsnorm_backward_bwd_gb300 import native, synth
from rmsnorm_backward_bwd_gb300.synth import Case

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


def _check_rstd(got, ref64):
    g = parity.to64(got)
    assert np.all(np.abs(g - ref64) <= 4 * 2.0**-24 * ref64), float(np.max(np.abs(g / ref64 - 1)))


def _shifted_like(t, shift):
    """A CUDA copy of t whose storage starts `shift` elements into a buffer."""
    buf = torch.empty(t.numel() + shift, dtype=t.dtype, device="cuda")
    v = buf[shift:].view(t.shape)
    v.copy_(t.cuda() if not t.is_cuda else t)
    return v


def _run_all(inp, dt, shift=0, ln_beta=True):
    """The three forwards on the same inputs (row tensors `shift` elements off
    the allocation's start), checked against the oracle; returns their plans."""
    M, N = inp["x"].shape
    x64, r64, g64 = (parity.to64(inp[k]) for k in ("x", "residual", "gamma"))
    b = (inp["gamma"].float() * 0.5 - 0.25).to(inp["gamma"].dtype)
    b64 = parity.to64(b)

    def dev(t):
        return _shifted_like(t, shift) if shift else t.cuda()

    def out():
        return dev(torch.zeros(M, N, dtype=inp["x"].dtype))

    x, r = dev(inp["x"]), dev(inp["residual"])
    g, bb = inp["gamma"].cuda(), b.cuda()
    plans = []
    y, rstd = rn.rmsnorm_fwd(x, g, 1e-6, y=out())
    plans.append(native.last_plan())
    o, ro, frstd = rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6, out=out(), residual_out=out())
    plans.append(native.last_plan())
    yl, mean, lrstd = rn.layernorm_fwd(x, g, bb if ln_beta else None, 1e-5, y=out())
    plans.append(native.last_plan())
    torch.cuda.synchronize()
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(1e-6))
    o64, a64, frstd64 = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(1e-6), dt)
    yl64, mean64, lrstd64 = oracle.layernorm_fwd(x64, g64, b64 if ln_beta else None, np.float32(1e-5))
    parity.check_tensor("y", y, y64, dt, "y")
    _check_rstd(rstd, rstd64)
    assert np.array_equal(parity.to64(ro), a64)   # one correctly rounded add
    parity.check_tensor("out", o, o64, dt, "y")
    _check_rstd(frstd, frstd64)
    parity.check_tensor("layernorm y", yl, yl64, dt, "y")
    tol = 2.0**-24 * (8 + 4 * np.sqrt(N))
    assert np.all(np.abs(parity.to64(mean) - mean64) <= tol * np.mean(np.abs(x64), axis=1))
    assert np.all(np.abs(parity.to64(lrstd) - lrstd64) <= tol * lrstd64)
    return plans


SHAPES = [(1000, 4095, "bf16"), (333, 4100, "bf16"), (97, 2999, "f32"), (130, 1001, "f16"),
          (5, 7, "bf16"), (3, 3, "f32"), (64, 515, "bf16"), (17, 8183, "bf16"), (33, 4095, "f32"),
          (300, 2050, "f16"), (9, 6, "f16"), (333, 12290, "bf16"), (97, 16391, "bf16"),
          (50, 8201, "f16"), (17, 6001, "f32"), (9, 16390, "f16"), (1, 4095, "bf16"), (2, 1, "f32"),
          (611, 8190, "bf16"), (40, 8183, "f32")]


@pytest.mark.parametrize("M,N,dt", SHAPES, ids=lambda v: str(v))
def test_staged_forwards(M, N, dt):
    """Each CTA on one residue class of rows modulo the phase period (M below,
    above and not a multiple of it), every warp staging its own span of the
    rows; rows of 1 to 2048 whole chunks; all three forwards."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    inp = synth.make_inputs(Case("fwd staged %s" % dt, M, N, dt, fused=True, seed=61))
    for plan in _run_all(inp, dt):
        assert "engine=generic staged " in plan, plan
    assert native.take_device_status() == 0


@pytest.mark.parametrize("cpt,teams,slots", [(1, 0, 0), (2, 0, 0), (0, 1, 0), (0, 3, 0),
                                             (0, 0, 3), (0, 0, 4), (2, 3, 3)])
@pytest.mark.parametrize("M,N,dt", [(1000, 4095, "bf16"), (97, 2999, "f32"), (130, 1001, "f16"),
                                    (300, 2050, "bf16")], ids=lambda v: str(v))
def test_staged_forwards_forced_tiles(M, N, dt, cpt, teams, slots):
    """Chunks per thread, teams per CTA and slots per team forced through the
    options: the rows still map onto the warps' spans and the ring."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    native.set_option(native.OPT_CHUNKS_PER_THREAD, cpt)
    native.set_option(native.OPT_TEAMS_PER_CTA, teams)
    native.set_option(native.OPT_STAGES, slots)
    inp = synth.make_inputs(Case("fwd staged tile %s" % dt, M, N, dt, fused=True, seed=62))
    chunks = N * synth.ELEM_BYTES[dt] // 16
    staged = not (cpt and (chunks + cpt - 1) // cpt > 512)
    for plan in _run_all(inp, dt):
        if not staged:
            # a team of more than 512 threads: the vector or phase-class forward instead
            assert "staged" not in plan, plan
            continue
        assert "engine=generic staged " in plan, plan
        if cpt:
            assert _plan_field(plan, "cpt") == cpt, plan
        if teams and teams * _plan_field(plan, "team_threads") <= 512:
            assert _plan_field(plan, "teams") == teams, plan
        if slots:
            assert _plan_field(plan, "slots") == slots, plan
    assert native.take_device_status() == 0


@pytest.mark.parametrize("shift", [1, 3])
@pytest.mark.parametrize("N,dt", [(4096, "bf16"), (1024, "f32"), (8192, "f16"), (4095, "bf16"),
                                  (2999, "f32")])
def test_staged_forwards_offset_base(N, dt, shift):
    """Row tensors that all start off a 16-byte boundary (one phase): every
    class has head elements, the bulk copies start inside the rows; LayerNorm
    with and without beta."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    inp = synth.make_inputs(Case("fwd staged base %s" % dt, 77, N, dt, fused=True, seed=63))
    for beta in (True, False):
        for plan in _run_all(inp, dt, shift=shift, ln_beta=beta):
            assert "engine=generic staged " in plan, plan


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_staged_forwards_params_off_16_bytes(dt):
    """gamma and beta off 16-byte alignment: gathered element by element once."""
    M, N = 2100, 2999
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    inp = synth.make_inputs(Case("fwd staged params", M, N, dt, seed=64))
    x64, g64 = parity.to64(inp["x"]), parity.to64(inp["gamma"])
    b = (inp["gamma"].float() * 0.5 - 0.25).to(inp["gamma"].dtype)
    b64 = parity.to64(b)
    g, bb = _shifted_like(inp["gamma"], 1), _shifted_like(b, 3)
    x = inp["x"].cuda()
    y, rstd = rn.rmsnorm_fwd(x, g, 1e-6)
    assert native.last_plan().startswith("rmsnorm_fwd engine=generic staged"), native.last_plan()
    yl, mean, lrstd = rn.layernorm_fwd(x, g, bb, 1e-5)
    assert native.last_plan().startswith("layernorm_fwd engine=generic staged"), native.last_plan()
    torch.cuda.synchronize()
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(1e-6))
    parity.check_tensor("y", y, y64, dt, "y")
    _check_rstd(rstd, rstd64)
    yl64, mean64, lrstd64 = oracle.layernorm_fwd(x64, g64, b64, np.float32(1e-5))
    parity.check_tensor("layernorm y", yl, yl64, dt, "y")
    tol = 2.0**-24 * (8 + 4 * np.sqrt(N))
    assert np.all(np.abs(parity.to64(lrstd) - lrstd64) <= tol * lrstd64)


@pytest.mark.parametrize("skip", [1, 3])
def test_staged_forward_wait_runs_out(skip):
    """The test hook leaves one row of the first team uncopied: that team's
    bounded wait runs out, the call sets bit 0 of the device status word, and
    the context stays usable: the next call, without the hook, matches the
    oracle and leaves the status clear."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5)
    inp = synth.make_inputs(Case("fwd staged timeout", 2000, 4095, "bf16", seed=65))
    x, g = inp["x"].cuda(), inp["gamma"].cuda()
    native.set_option(native.OPT_TEST_WAIT_TIMEOUT, skip)
    rn.rmsnorm_fwd(x, g, 1e-6)
    assert native.take_device_status() == 1
    assert native.take_device_status() == 0   # read and cleared
    native.set_option(native.OPT_TEST_WAIT_TIMEOUT, 0)
    y, rstd = rn.rmsnorm_fwd(x, g, 1e-6)
    torch.cuda.synchronize()
    y64, rstd64 = oracle.rmsnorm_fwd(parity.to64(inp["x"]), parity.to64(inp["gamma"]),
                                     np.float32(1e-6))
    parity.check_tensor("y", y, y64, "bf16", "y")
    _check_rstd(rstd, rstd64)
    assert native.take_device_status() == 0


@pytest.mark.parametrize("M,N,dt,staged", [
    (2048, 4095, "bf16", (False, False, True)), (2047, 4095, "bf16", (False, False, False)),
    (4096, 4095, "bf16", (True, False, True)), (4096, 1001, "f16", (True, True, True)),
    (4096, 2999, "f32", (True, False, True)), (2048, 12290, "bf16", (True, True, True)),
    (2048, 16393, "bf16", (False, False, False)),   # 2049 whole chunks
    (300, 2999, "f32", (False, False, True)), (300, 4095, "bf16", (False, False, False)),
    (255, 2999, "f32", (False, False, False)), (300, 12290, "bf16", (False, False, True))],
    ids=lambda v: str(v))
def test_staged_forward_default_choice(M, N, dt, staged):
    """The automatic choice (RMSNorm, fused-add, LayerNorm): the staged forward
    from 2048 rows within 2048 whole chunks a row; RMSNorm with at least 6 rows
    a team or rows of at most 256 chunks, fused-add with one team a CTA or rows
    of at most 256 chunks; the vector or phase-class forward otherwise. Below
    2048 rows the LayerNorm forward takes it from 256 rows where the vector
    kernel would run (fp32, rows past 1024 chunks)."""
    inp = synth.make_inputs(Case("fwd default %s" % dt, M, N, dt, fused=True, seed=66))
    for plan, want in zip(_run_all(inp, dt), staged):
        assert ("engine=generic staged " in plan) == want, plan
