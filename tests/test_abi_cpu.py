"""The C ABI on the host: the library loads, exports what the header
declares, and rejects bad arguments before touching the GPU (CPU only)."""
import ctypes
import os

import pytest
import torch

from rmsnorm_backward_bwd_gb300 import native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_function():
    lib = native.lib()
    names = native.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), "%s declared in the header but not exported" % n


def test_abi_version_and_status_strings():
    lib = native.lib()
    assert lib.rn_abi_version() == 1
    for st in range(5):
        assert native.status_string(st)


def _bwd(lib, **kw):
    a = dict(x=None, g=None, dy=None, rstd=None, dx=None, dw32=None, dw=None, ws=None,
             wsb=0, M=4, N=8, dt=2)
    a.update(kw)
    return lib.rn_rmsnorm_bwd(a["x"], a["g"], a["dy"], a["rstd"], a["dx"], a["dw32"], a["dw"],
                              a["ws"], a["wsb"], a["M"], a["N"], a["dt"], None)


def test_argument_checks_fail_before_any_launch():
    lib = native.lib()
    fake = ctypes.c_void_p(0x1000)
    assert _bwd(lib) == native.RN_ERR_INVALID_ARG                       # gamma missing
    assert b"required" in lib.rn_last_error()
    assert _bwd(lib, dt=7, g=fake, dw32=fake) == native.RN_ERR_INVALID_ARG
    assert _bwd(lib, N=0, g=fake, dw32=fake) == native.RN_ERR_INVALID_ARG
    assert _bwd(lib, M=-1, g=fake, dw32=fake) == native.RN_ERR_INVALID_ARG
    assert _bwd(lib, g=fake, dw32=fake) == native.RN_ERR_INVALID_ARG     # x/dy/rstd/dx missing
    assert _bwd(lib, x=fake, g=fake, dy=fake, rstd=fake, dx=fake, dw32=fake) == \
        native.RN_ERR_INVALID_ARG                                          # dx aliases x
    assert _bwd(lib, N=1 << 40, g=fake, dw32=fake) == native.RN_ERR_UNSUPPORTED
    # buffers off their element size fail before any launch (bf16: 2 bytes; fp32: 4)
    odd = ctypes.c_void_p(0x1001)
    assert _bwd(lib, g=odd, dw32=fake, M=0) == native.RN_ERR_INVALID_ARG
    assert b"gamma is not aligned" in lib.rn_last_error()
    assert _bwd(lib, g=fake, dw32=ctypes.c_void_p(0x1002), M=0) == native.RN_ERR_INVALID_ARG
    assert b"dweight_f32" in lib.rn_last_error()
    assert lib.rn_rmsnorm_fwd(odd, fake, 1e-6, fake, None, 4, 8, 2, None) == \
        native.RN_ERR_INVALID_ARG
    assert lib.rn_layernorm_fwd(fake, fake, None, 1e-5, fake, None, ctypes.c_void_p(0x1006), 4, 8,
                                2, None) == native.RN_ERR_INVALID_ARG
    assert lib.rn_rmsnorm_fwd(None, None, 1e-6, None, None, 4, 8, 2, None) == native.RN_ERR_INVALID_ARG
    assert lib.rn_rmsnorm_fwd(fake, fake, -1.0, fake, None, 4, 8, 2, None) == native.RN_ERR_INVALID_ARG
    assert lib.rn_fused_add_rmsnorm_fwd(fake, None, fake, 1e-6, fake, fake, None, 4, 8, 2,
                                        None) == native.RN_ERR_INVALID_ARG


def test_options_round_trip():
    for opt in range(native.OPT_COUNT):
        native.set_option(opt, 3)
        assert native.get_option(opt) == 3
        native.set_option(opt, 0)
    assert native.lib().rn_set_option(99, 1) == native.RN_ERR_INVALID_ARG
    assert native.lib().rn_set_option(0, -1) == native.RN_ERR_INVALID_ARG
    assert native.get_option(99) == -1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_device_queries_report_cuda_error_without_gpu():
    n = ctypes.c_size_t(0)
    st = native.lib().rn_bwd_workspace_bytes(4, 8, 2, ctypes.byref(n))
    assert st == native.RN_ERR_CUDA


def test_python_guards_refuse_host_tensors():
    """Host pointers never reach the library: CPU tensors are refused before
    any call (there is no CPU path)."""
    import rmsnorm_backward_bwd_gb300 as rn
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    for call in (lambda: rn.rmsnorm_bwd(x, torch.zeros(8, dtype=torch.float16), x, torch.zeros(4)),
                 lambda: rn.rmsnorm_fwd(x, torch.zeros(8, dtype=torch.bfloat16), 1e-6),
                 lambda: rn.fused_add_rmsnorm_fwd(x, x, torch.zeros(8, dtype=torch.bfloat16), 1e-6),
                 lambda: rn.fused_add_rmsnorm_bwd(x, torch.zeros(8, dtype=torch.bfloat16), x,
                                                  torch.zeros(4))):
        with pytest.raises(ValueError, match="CUDA devices only"):
            call()


@pytest.mark.parametrize("env,opt,want", [({"RN_BWD_ENGINE": "cluster"}, 0, 3),
                                          ({"RN_BWD_ENGINE": "generic"}, 0, 2),
                                          ({"RN_DWEIGHT_MODE": "scratch"}, 1, 1),
                                          ({"RN_DWEIGHT_MODE": "ATOMIC"}, 1, 2),
                                          ({"RN_GENERIC_KERNEL": "realign"}, 7, 3),
                                          ({"RN_GENERIC_KERNEL": "staged"}, 7, 5)])
def test_environment_overrides_options(env, opt, want):
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r); from rmsnorm_backward_bwd_gb300 import native; "
            "print(native.get_option(%d))" % (ROOT, opt))
    out = subprocess.run([sys.executable, "-c", code], env={**os.environ, **env},
                         capture_output=True, text=True, check=True).stdout.strip()
    assert int(out) == want


def test_environment_override_rejects_unknown_values():
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r); from rmsnorm_backward_bwd_gb300 import native; "
            "native.lib()" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], env={**os.environ, "RN_BWD_ENGINE": "warp"},
                       capture_output=True, text=True)
    assert r.returncode != 0 and "RN_BWD_ENGINE" in r.stderr
