"""ctypes view of the C ABI declared in ``include/rmsnorm_gb300.h``, and the
loader of the PyTorch operator library over it.

Loads ``_build/librn_gb300.so`` and ``_build/librn_torch.so`` (built in-tree
by ``build.py``). There is no fallback: if a library is missing or fails to
load, every call that needs it raises.
"""
import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "librn_gb300.so")
TORCH_LIB_PATH = os.path.join(HERE, "_build", "librn_torch.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "rmsnorm_gb300.h")

RN_OK, RN_ERR_INVALID_ARG, RN_ERR_UNSUPPORTED, RN_ERR_CUDA, RN_ERR_WORKSPACE = range(5)
RN_F32, RN_F16, RN_BF16 = 0, 1, 2
(OPT_BWD_ENGINE, OPT_DWEIGHT_MODE, OPT_CHUNKS_PER_THREAD, OPT_TEAMS_PER_CTA, OPT_STAGES, OPT_GRID,
 OPT_CLUSTER_SIZE, OPT_GENERIC_KERNEL, OPT_TEST_WAIT_TIMEOUT) = range(9)
OPT_COUNT = 9

_lib = None


class RNError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s (status %d): %s" % (status_string(status), status, msg))
        self.status = status


def _bind(lib):
    vp, i64, ci, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.rn_abi_version.restype = ci
    lib.rn_abi_version.argtypes = []
    lib.rn_status_string.restype = ctypes.c_char_p
    lib.rn_status_string.argtypes = [ci]
    lib.rn_last_error.restype = ctypes.c_char_p
    lib.rn_last_error.argtypes = []
    lib.rn_last_plan.restype = ctypes.c_char_p
    lib.rn_last_plan.argtypes = []
    lib.rn_rmsnorm_fwd.restype = ci
    lib.rn_rmsnorm_fwd.argtypes = [vp, vp, f32, vp, vp, i64, i64, ci, vp]
    lib.rn_fused_add_rmsnorm_fwd.restype = ci
    lib.rn_fused_add_rmsnorm_fwd.argtypes = [vp, vp, vp, f32, vp, vp, vp, i64, i64, ci, vp]
    lib.rn_bwd_workspace_bytes.restype = ci
    lib.rn_bwd_workspace_bytes.argtypes = [i64, i64, ci, ctypes.POINTER(sz)]
    lib.rn_rmsnorm_bwd.restype = ci
    lib.rn_rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, sz, i64, i64, ci, vp]
    lib.rn_fused_add_rmsnorm_bwd.restype = ci
    lib.rn_fused_add_rmsnorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i64, i64, ci, vp]
    lib.rn_layernorm_fwd.restype = ci
    lib.rn_layernorm_fwd.argtypes = [vp, vp, vp, f32, vp, vp, vp, i64, i64, ci, vp]
    lib.rn_layernorm_bwd_workspace_bytes.restype = ci
    lib.rn_layernorm_bwd_workspace_bytes.argtypes = [i64, i64, ci, ctypes.POINTER(sz)]
    lib.rn_layernorm_bwd.restype = ci
    lib.rn_layernorm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i64, i64,
                                     ci, vp]
    lib.rn_rmsnorm_bwd_noalloc.restype = ci
    lib.rn_rmsnorm_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, vp]
    lib.rn_set_option.restype = ci
    lib.rn_set_option.argtypes = [ci, ci]
    lib.rn_get_option.restype = ci
    lib.rn_get_option.argtypes = [ci]
    lib.rn_set_profile_events.restype = ci
    lib.rn_set_profile_events.argtypes = [vp, vp]
    lib.rn_take_device_status.restype = ci
    lib.rn_take_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    return lib


# Process-wide overrides read from the environment when the library loads:
#   RN_BWD_ENGINE   = auto | row | generic | cluster
#   RN_DWEIGHT_MODE = auto | scratch (deterministic) | atomic
#   RN_GENERIC_KERNEL = auto | phase | vec | realign | scalar | staged (unaligned rows)
ENV_OPTIONS = {
    "RN_BWD_ENGINE": (0, {"auto": 0, "row": 1, "generic": 2, "cluster": 3}),
    "RN_DWEIGHT_MODE": (1, {"auto": 0, "scratch": 1, "atomic": 2}),
    "RN_GENERIC_KERNEL": (7, {"auto": 0, "phase": 1, "vec": 2, "realign": 3, "scalar": 4,
                              "staged": 5}),
}


def _apply_env(lib_):
    for var, (opt, values) in ENV_OPTIONS.items():
        v = os.environ.get(var)
        if v is None:
            continue
        if v.lower() not in values:
            raise ValueError("%s=%r: expected one of %s" % (var, v, ", ".join(values)))
        lib_.rn_set_option(opt, values[v.lower()])


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("CUDA library %s is not built; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        loaded = _bind(ctypes.CDLL(LIB_PATH))
        _apply_env(loaded)
        _lib = loaded
    return _lib


_torch_ops = None


def torch_ops():
    """The operator namespace ``torch.ops.rn_gb300`` (the differentiable ops
    and the raw calls as C++ PyTorch operators). The CUDA library is loaded
    first, so that both views share one copy of it (one set of options)."""
    global _torch_ops
    if _torch_ops is None:
        import torch
        lib()
        if not os.path.exists(TORCH_LIB_PATH):
            raise RuntimeError("operator library %s is not built; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`"
                               % TORCH_LIB_PATH)
        torch.ops.load_library(TORCH_LIB_PATH)
        _torch_ops = torch.ops.rn_gb300
    return _torch_ops


def status_string(st):
    return lib().rn_status_string(int(st)).decode()


def check(st):
    if st != RN_OK:
        raise RNError(st, lib().rn_last_error().decode())


def header_functions():
    """Names of the functions include/rmsnorm_gb300.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rn_[a-z0-9_]+)\s*\(", text)))


def last_plan():
    return lib().rn_last_plan().decode()


def take_device_status():
    """Read and clear the current device's status word (bit 0: a bounded wait
    in a kernel ran out). Synchronizes the device."""
    v = ctypes.c_uint(0)
    check(lib().rn_take_device_status(ctypes.byref(v)))
    return int(v.value)


def set_option(opt, value):
    check(lib().rn_set_option(int(opt), int(value)))


def get_option(opt):
    return int(lib().rn_get_option(int(opt)))
