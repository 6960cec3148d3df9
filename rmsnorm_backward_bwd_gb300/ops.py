"""PyTorch-facing calls with the C ABI's names (argument marshalling only).

Every step of the computation runs in the CUDA library; these functions
check dtypes, devices, shapes and contiguity (the FlyDSL pages' guards:
matching I/O dtypes, contiguous rows, ``x.shape[-1] == len(weight)``, and
launching on the tensor's own device -- PR #800 review fixes), allocate
outputs with torch when the caller does not pass them, and forward pointers
and the current CUDA stream to the library.
"""
import ctypes

import torch

from . import native

_CODES = {torch.float32: native.RN_F32, torch.float16: native.RN_F16,
          torch.bfloat16: native.RN_BF16}


def _code(t):
    try:
        return _CODES[t.dtype]
    except KeyError:
        raise TypeError("unsupported dtype %s (f32, f16, bf16 only)" % t.dtype) from None


def _need(name, t, ref, shape=None, dtype=None):
    if t is None:
        raise ValueError("%s is required" % name)
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cuda":
        # the library takes device pointers only; there is no CPU path
        raise ValueError("%s is on %s: these ops run on CUDA devices only" % (name, t.device))
    if t.device != ref.device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, ref.device))
    want = ref.dtype if dtype is None else dtype
    if t.dtype != want:
        raise ValueError("dtype mismatch: %s is %s, expected %s" % (name, t.dtype, want))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _rows(x, gamma):
    if x.dim() < 1:
        raise ValueError("input must have at least one dimension")
    N = x.shape[-1]
    if gamma.dim() != 1 or gamma.shape[0] != N:
        raise ValueError("weight has shape %s, expected (%d,)" % (tuple(gamma.shape), N))
    M = x.numel() // N if N else 0
    return M, N


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


_WS = {}


def bwd_workspace(M, N, dtype, device):
    """A workspace for the backward on `device`, cached per (device, stream)
    so that calls sharing it are ordered on the GPU."""
    device = torch.device(device)
    with torch.cuda.device(device):
        nbytes = ctypes.c_size_t(0)
        native.check(native.lib().rn_bwd_workspace_bytes(
            int(M), int(N), _CODES[dtype], ctypes.byref(nbytes)))
        key = (device.index, torch.cuda.current_stream().cuda_stream)
        ws = _WS.get(key)
        if ws is None or ws.numel() < nbytes.value:
            ws = torch.empty(nbytes.value, dtype=torch.uint8, device=device)
            _WS[key] = ws
        return ws


def rmsnorm_fwd(x, gamma, eps, *, y=None, rstd=None, store_rstd=True):
    """y = x * rstd * gamma with rstd = 1/sqrt(mean(x^2) + eps) per row.
    Returns (y, rstd); rstd is fp32 [M] (None when store_rstd is False)."""
    _need("x", x, x)
    _need("gamma", gamma, x)
    M, N = _rows(x, gamma)
    with torch.cuda.device(x.device):
        y = torch.empty_like(x) if y is None else _need("y", y, x, x.shape)
        if store_rstd:
            rstd = (torch.empty(M, dtype=torch.float32, device=x.device) if rstd is None
                    else _need("rstd", rstd, x, (M,), torch.float32))
        else:
            rstd = None
        native.check(native.lib().rn_rmsnorm_fwd(_ptr(x), _ptr(gamma), float(eps), _ptr(y),
                                                 _ptr(rstd), M, N, _code(x), _stream()))
    return y, rstd


def fused_add_rmsnorm_fwd(x, residual, gamma, eps, *, out=None, residual_out=None, rstd=None,
                          store_rstd=True):
    """added = x + residual (rounded to the dtype) -> residual_out;
    out = added * rstd * gamma. Returns (out, residual_out, rstd)."""
    _need("x", x, x)
    _need("residual", residual, x, x.shape)
    _need("gamma", gamma, x)
    M, N = _rows(x, gamma)
    with torch.cuda.device(x.device):
        out = torch.empty_like(x) if out is None else _need("out", out, x, x.shape)
        residual_out = (torch.empty_like(x) if residual_out is None
                        else _need("residual_out", residual_out, x, x.shape))
        if store_rstd:
            rstd = (torch.empty(M, dtype=torch.float32, device=x.device) if rstd is None
                    else _need("rstd", rstd, x, (M,), torch.float32))
        else:
            rstd = None
        native.check(native.lib().rn_fused_add_rmsnorm_fwd(
            _ptr(x), _ptr(residual), _ptr(gamma), float(eps), _ptr(out), _ptr(residual_out),
            _ptr(rstd), M, N, _code(x), _stream()))
    return out, residual_out, rstd


def _bwd_outputs(x, M, N, dx, dweight_f32, dweight, want_cast):
    dx = torch.empty_like(x) if dx is None else _need("dx", dx, x, x.shape)
    dweight_f32 = (torch.empty(N, dtype=torch.float32, device=x.device) if dweight_f32 is None
                   else _need("dweight_f32", dweight_f32, x, (N,), torch.float32))
    if dweight is None and want_cast:
        dweight = torch.empty(N, dtype=x.dtype, device=x.device)
    elif dweight is not None:
        _need("dweight", dweight, x, (N,))
    return dx, dweight_f32, dweight


def rmsnorm_bwd(x, gamma, dy, rstd, *, dx=None, dweight_f32=None, dweight=None,
                want_cast=True, workspace=None):
    """Gradients of y = rmsnorm(x) * gamma given dy and the saved fp32 rstd.
    Returns (dx, dweight, dweight_f32); dweight is dweight_f32 cast to the
    I/O dtype (None when want_cast is False and no buffer was passed)."""
    _need("x", x, x)
    _need("gamma", gamma, x)
    _need("dy", dy, x, x.shape)
    M, N = _rows(x, gamma)
    _need("rstd", rstd, x, (M,), torch.float32)
    with torch.cuda.device(x.device):
        dx, dweight_f32, dweight = _bwd_outputs(x, M, N, dx, dweight_f32, dweight, want_cast)
        ws = bwd_workspace(M, N, x.dtype, x.device) if workspace is None else workspace
        native.check(native.lib().rn_rmsnorm_bwd(
            _ptr(x), _ptr(gamma), _ptr(dy), _ptr(rstd), _ptr(dx), _ptr(dweight_f32),
            _ptr(dweight), _ptr(ws), ws.numel(), M, N, _code(x), _stream()))
    return dx, dweight, dweight_f32


def fused_add_rmsnorm_bwd(added, gamma, dy, rstd, dresidual_out=None, *, dx=None,
                          dweight_f32=None, dweight=None, want_cast=True, workspace=None):
    """Backward of the fused-add (prenorm) RMSNorm. `added` is the saved
    residual_out; dresidual_out (may be None) is the gradient flowing into
    residual_out. Returns (dx, dresidual, dweight, dweight_f32) where
    dresidual is the same tensor as dx. dx may be dresidual_out itself."""
    _need("added", added, added)
    _need("gamma", gamma, added)
    _need("dy", dy, added, added.shape)
    M, N = _rows(added, gamma)
    _need("rstd", rstd, added, (M,), torch.float32)
    if dresidual_out is not None:
        _need("dresidual_out", dresidual_out, added, added.shape)
    with torch.cuda.device(added.device):
        dx, dweight_f32, dweight = _bwd_outputs(added, M, N, dx, dweight_f32, dweight, want_cast)
        ws = bwd_workspace(M, N, added.dtype, added.device) if workspace is None else workspace
        native.check(native.lib().rn_fused_add_rmsnorm_bwd(
            _ptr(added), _ptr(gamma), _ptr(dy), _ptr(rstd), _ptr(dresidual_out), _ptr(dx),
            _ptr(dweight_f32), _ptr(dweight), _ptr(ws), ws.numel(), M, N, _code(added),
            _stream()))
    return dx, dx, dweight, dweight_f32
