"""rn_rmsnorm_bwd_noalloc: the backward for callers that cannot allocate.

Such callers (code running while an allocator or memory pool is locked or
being torn down, or an embedder that fixes all device memory up front) get
the scratch from a fixed array inside the library instead of a workspace.
These tests call the new entry point through the C ABI and check that two
calls in a row give what the ordinary workspace entry point gives, within the
tolerances the other parity tests use, and that a problem too large for the
fixed scratch is refused cleanly. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import parity
import rmsnorm_backward_bwd_gb300 as rn
from rmsnorm_backward_bwd_gb300 import native
from rmsnorm_backward_bwd_gb300.synth import Case

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(x, g, dy, rstd, dx, dw32, dw):
    M, N = x.shape
    code = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[x.dtype]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return native.lib().rn_rmsnorm_bwd_noalloc(_p(x), _p(g), _p(dy), _p(rstd), _p(dx), _p(dw32),
                                               _p(dw), M, N, code, stream)


@pytest.fixture(autouse=True)
def _default_options():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 0)
    yield


@pytest.mark.parametrize("mode", [1, 2], ids=["scratch-partials", "atomics"])
@pytest.mark.parametrize("case", [Case("bf16 M=4096 N=4096", 4096, 4096, "bf16"),
                                  Case("f32 M=300 N=1000", 300, 1000, "f32"),
                                  Case("f16 M=7 N=1003", 7, 1003, "f16"),
                                  # rows that are not 16-byte multiples: the staged kernel
                                  Case("bf16 M=2048 N=4095", 2048, 4095, "bf16")],
                         ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point_twice(case, mode):
    # weight-gradient mode 1 keeps the per-CTA partials in the fixed scratch array
    native.set_option(native.OPT_DWEIGHT_MODE, mode)
    ex = parity.expected_bwd(case)
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    ref_dx, ref_dw, ref_dw32 = rn.rmsnorm_bwd(x, g, dy, rstd)
    torch.cuda.synchronize()
    for _ in range(2):
        dx = torch.full_like(x, float("nan"))
        dw32 = torch.full_like(ref_dw32, float("nan"))
        dw = torch.full_like(ref_dw, float("nan"))
        st = _noalloc(x, g, dy, rstd, dx, dw32, dw)
        assert st == native.RN_OK, native.lib().rn_last_error()
        torch.cuda.synchronize()
        if case.N == 4095:
            assert "staged" in native.last_plan(), native.last_plan()
        # against the workspace entry point, with the parity tolerances
        parity.check_tensor("dx", dx, parity.to64(ref_dx), case.dtype, "dx")
        parity.check_tensor("dweight_f32", dw32, parity.to64(ref_dw32), case.dtype, "dweight_f32")
        parity.check_tensor("dweight", dw, parity.to64(ref_dw), case.dtype, "dweight")
        # and against the fp64 oracle
        parity.check_bwd(ex, dx, dw, dw32)


def test_noalloc_refuses_problems_beyond_its_scratch():
    N = 1 << 16  # needs 2 rows of N fp32 per SM: far above the fixed scratch
    x = torch.zeros(4, N, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(N, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(4, device="cuda")
    dw32 = torch.zeros(N, device="cuda")
    st = _noalloc(x, g, x, rstd, torch.empty_like(x), dw32, None)
    assert st == native.RN_ERR_UNSUPPORTED
    assert b"scratch" in native.lib().rn_last_error()


def test_noalloc_cast_only_weight_gradient():
    """dweight_f32 = NULL: the fp32 sum stays in the fixed scratch (scratch
    mode) and only the cast is written; equal, bit for bit, to the workspace
    entry point's scratch-mode cast."""
    native.set_option(native.OPT_DWEIGHT_MODE, 1)
    ex = parity.expected_bwd(Case("bf16 M=2048 N=4096", 2048, 4096, "bf16"))
    x, g, dy, rstd = (t.cuda() for t in (ex.x, ex.gamma, ex.dy, ex.rstd))
    ref_dx, ref_dw, _ = rn.rmsnorm_bwd(x, g, dy, rstd)
    native.set_option(native.OPT_DWEIGHT_MODE, 0)
    dx = torch.full_like(x, float("nan"))
    dw = torch.full_like(ref_dw, float("nan"))
    st = _noalloc(x, g, dy, rstd, dx, None, dw)
    assert st == native.RN_OK, native.lib().rn_last_error()
    torch.cuda.synchronize()
    assert "dw=scratch" in native.last_plan()
    assert torch.equal(dx, ref_dx) and torch.equal(dw, ref_dw)
    parity.check_tensor("dweight", dw, ex.dw, "bf16", "dweight")
