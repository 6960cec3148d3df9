"""Seeded random problems across every backward and forward engine.

Each case draws M, N, dtype, the variant (plain / fused-add with or without
dresidual_out) and the alignment phase of each row buffer (0 or a few
elements off a 16-byte boundary) from a fixed seed, runs the public calls on
the GPU and compares them with the oracle under the parity tolerances. The
widths cover aligned rows (row and cluster engines), rows that are not
16-byte multiples (phase-class, vector and scalar generic kernels) and
mixed phases. The engine each case took is part of the failure message.
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

WIDTHS = [1, 2, 7, 31, 64, 129, 1000, 1001, 2048, 2999, 4095, 4096, 4100, 6144, 8190, 8192,
          8191, 12289, 16384, 16385, 20001, 24576]


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    dt = ["f32", "f16", "bf16"][rng.integers(3)]
    N = int(rng.choice(WIDTHS))
    M = int(rng.integers(1, 96 if N > 8000 else 400))
    variant = ["plain", "fused", "fused_nodres"][rng.integers(3)]
    # phase of each row buffer in elements: mostly shared, sometimes mixed
    shared = int(rng.choice([0, 0, 1, 3]))
    phases = {k: shared for k in ("x", "dy", "dx", "dres")}
    if rng.random() < 0.25:
        phases[str(rng.choice(["dy", "dx"]))] = int(rng.integers(0, 4))
    return M, N, dt, variant, phases


@pytest.fixture(autouse=True)
def _reset_options():
    yield
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)


_ENGINES = set()   # the backward engines the random cases took (checked by the last test)


def _engine(plan):
    head = plan.split()
    if not head:
        return ""
    if head[0] == "engine=generic" and len(head) > 1 and head[1] in ("phase", "realign", "vec",
                                                                      "staged"):
        return "generic " + head[1]
    return head[0].split("=", 1)[1]


def _placed(t, shift):
    buf = torch.empty(t.numel() + shift, dtype=t.dtype, device="cuda")
    v = buf[shift:].view(t.shape)
    v.copy_(t.cuda())
    return v


@pytest.mark.parametrize("seed", range(48))
def test_random_backward(seed):
    """Odd seeds ask for the staged phase-class kernel (below 2048 rows the
    automatic choice is the phase-class kernel): it takes the one-phase
    unaligned ones; the rest fall back as the automatic choice would."""
    native.set_option(native.OPT_GENERIC_KERNEL, 5 if seed % 2 else 0)
    M, N, dt, variant, ph = _draw(seed)
    fused = variant != "plain"
    case = Case("random %d" % seed, M, N, dt, fused=fused, with_dres=variant == "fused",
                seed=seed)
    ex = parity.expected_bwd(case)
    x, dy = _placed(ex.x, ph["x"]), _placed(ex.dy, ph["dy"])
    g, rstd = ex.gamma.cuda(), ex.rstd.cuda()
    dx = _placed(torch.zeros_like(ex.x), ph["dx"])
    if fused:
        dres = _placed(ex.dres, ph["dres"]) if ex.dres is not None else None
        dx, _, dw, dw32 = rn.fused_add_rmsnorm_bwd(x, g, dy, rstd, dres, dx=dx)
    else:
        dx, dw, dw32 = rn.rmsnorm_bwd(x, g, dy, rstd, dx=dx)
    torch.cuda.synchronize()
    plan = native.last_plan()
    _ENGINES.add(_engine(plan))
    parity.check_bwd(ex, dx, dw, dw32, tag=" [M=%d N=%d %s %s phases=%s: %s]" % (
        M, N, dt, variant, ph, plan), allow_ill_conditioned=N == 1)


def test_random_backward_cases_reached_every_engine():
    """The sweep above is only worth its seeds if it reaches every engine."""
    # (the realigning engine is taken only when asked for: its own tests cover it)
    want = {"row", "cluster", "generic staged", "generic phase", "generic vec", "generic"}
    assert want <= _ENGINES, "engines not reached: %s (reached %s)" % (want - _ENGINES, _ENGINES)


@pytest.mark.parametrize("seed", range(24))
def test_random_forwards(seed):
    """The three forwards on random shapes and phases; odd seeds ask for the
    staged forward (taken wherever the row tensors share one phase)."""
    M, N, dt, _, ph = _draw(100 + seed)
    if seed % 2:
        native.set_option(native.OPT_GENERIC_KERNEL, 5)
    inp = synth.make_inputs(Case("random fwd %d" % seed, M, N, dt, fused=True, seed=seed))
    x64, r64, g64 = (parity.to64(inp[k]) for k in ("x", "residual", "gamma"))
    x, r = _placed(inp["x"], ph["x"]), _placed(inp["residual"], ph["dy"])
    g = inp["gamma"].cuda()
    out = _placed(torch.zeros_like(inp["x"]), ph["dx"])
    ro = _placed(torch.zeros_like(inp["x"]), ph["x"])
    y, rstd = rn.rmsnorm_fwd(x, g, 1e-6, y=out)
    y = y.clone()
    o, ro, frstd = rn.fused_add_rmsnorm_fwd(x, r, g, 1e-6, out=out, residual_out=ro)
    yl, mean, lrstd = rn.layernorm_fwd(x, g, g, 1e-5)
    torch.cuda.synchronize()
    tag = " [M=%d N=%d %s phases=%s]" % (M, N, dt, ph)
    y64, rstd64 = oracle.rmsnorm_fwd(x64, g64, np.float32(1e-6))
    o64, a64, frstd64 = oracle.fused_add_rmsnorm_fwd(x64, r64, g64, np.float32(1e-6), dt)
    yl64, mean64, lrstd64 = oracle.layernorm_fwd(x64, g64, g64, np.float32(1e-5))
    parity.check_tensor("y" + tag, y, y64, dt, "y")
    parity.check_tensor("out" + tag, o, o64, dt, "y")
    assert np.array_equal(parity.to64(ro), a64), "residual_out" + tag
    parity.check_tensor("layernorm y" + tag, yl, yl64, dt, "y")
    for got, ref in ((rstd, rstd64), (frstd, frstd64)):
        assert np.all(np.abs(parity.to64(got) - ref) <= 4 * 2.0**-24 * ref), "rstd" + tag
    tol = 2.0**-24 * (8 + 4 * np.sqrt(N))
    assert np.all(np.abs(parity.to64(mean) - mean64) <= tol * np.mean(np.abs(x64), axis=1))
    assert np.all(np.abs(parity.to64(lrstd) - lrstd64) <= tol * lrstd64)


LN_WIDTHS = [1, 2, 7, 31, 64, 129, 1000, 1001, 2048, 2999, 4095, 4096, 4100, 6144, 8190, 8191,
             8192, 12289, 16384]


@pytest.mark.parametrize("seed", range(24))
def test_random_layernorm_backward(seed):
    """Seeded random LayerNorm backward problems (dtype, width, rows, a base off 16 bytes,
    with or without the bias gradient) against the oracle; odd seeds ask for the staged
    phase-class kernel, the rest take the automatic choice."""
    import test_gpu_layernorm as lnt
    rng = np.random.default_rng(3000 + seed)
    dt = ["f32", "f16", "bf16"][rng.integers(3)]
    N = int(rng.choice(LN_WIDTHS))
    M = int(rng.integers(1, 64 if N > 8000 else 300))
    shift = int(rng.choice([0, 0, 1, 3]))
    with_dbeta = bool(rng.integers(2))
    native.set_option(native.OPT_GENERIC_KERNEL, 5 if seed % 2 else 0)
    ex = lnt.expected(Case("random ln %d" % seed, M, N, dt, eps=1e-5, seed=seed), with_dbeta)
    x, dy = _placed(ex.inp["x"], shift), _placed(ex.inp["dy"], shift)
    dx = _placed(torch.zeros_like(ex.inp["x"]), shift)
    mean = torch.from_numpy(ex.mean32).float().cuda()
    rstd = torch.from_numpy(ex.rstd32).float().cuda()
    out = rn.layernorm_bwd(x, ex.inp["gamma"].cuda(), dy, mean, rstd, dx=dx,
                           want_dbeta=with_dbeta)
    torch.cuda.synchronize()
    lnt.check(ex, out, with_dbeta=with_dbeta,
              tag=" [M=%d N=%d %s shift=%d: %s]" % (M, N, dt, shift, native.last_plan()))
    assert native.take_device_status() == 0
