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
    if not isinstance(t, torch.Tensor):
        if t is None:
            raise ValueError("%s is required" % name)
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        # the library takes device pointers only; there is no CPU path
        raise ValueError("%s is on %s: these ops run on CUDA devices only" % (name, t.device))
    if t is not ref and t.get_device() != ref.get_device():
        raise ValueError("%s is on %s, expected %s" % (name, t.device, ref.device))
    want = ref.dtype if dtype is None else dtype
    if t.dtype != want:
        raise ValueError("dtype mismatch: %s is %s, expected %s" % (name, t.dtype, want))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and t.shape != shape:
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t


def _ptr(t):
    # plain ints: the bound argtypes (c_void_p) convert them
    return t.data_ptr() if t is not None else None


def _rows(x, gamma):
    if x.dim() < 1:
        raise ValueError("input must have at least one dimension")
    N = x.shape[-1]
    if gamma.dim() != 1 or gamma.shape[0] != N:
        raise ValueError("weight has shape %s, expected (%d,)" % (tuple(gamma.shape), N))
    M = x.numel() // N if N else 0
    return M, N


# The raw handle of the current stream without building a Stream object (a
# few microseconds per call saved); the public query is the fallback.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(index):
    if _raw_stream is not None:
        return _raw_stream(index)
    return torch.cuda.current_stream(index).cuda_stream


class _on_device:
    """Make `index` the current device for the block (no-op when it is)."""

    __slots__ = ("index", "prev")

    def __init__(self, index):
        self.index = index
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.index:
            self.prev = cur
            torch.cuda.set_device(self.index)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


_WS = {}
_WS_BYTES = {}
# Workspaces replaced by a larger one stay allocated: a CUDA graph captured
# on that stream may still use the smaller buffer, and freeing it would let
# the allocator hand the memory to someone else under the graph.
_WS_RETIRED = []


def _ws_bytes(M, N, code, index):
    """Workspace size the library asks for (it depends on the shape, dtype and
    the device's SM count only), cached."""
    key = (M, N, code, index)
    n = _WS_BYTES.get(key)
    if n is None:
        nbytes = ctypes.c_size_t(0)
        native.check(native.lib().rn_bwd_workspace_bytes(int(M), int(N), code,
                                                         ctypes.byref(nbytes)))
        n = _WS_BYTES[key] = nbytes.value
    return n


def _ln_ws_bytes(M, N, code, index):
    key = ("ln", M, N, code, index)
    n = _WS_BYTES.get(key)
    if n is None:
        nbytes = ctypes.c_size_t(0)
        native.check(native.lib().rn_layernorm_bwd_workspace_bytes(int(M), int(N), code,
                                                                   ctypes.byref(nbytes)))
        n = _WS_BYTES[key] = nbytes.value
    return n


def _workspace(M, N, code, index, layernorm=False):
    # index is the current device here
    n = _ln_ws_bytes(M, N, code, index) if layernorm else _ws_bytes(M, N, code, index)
    key = (index, _stream_handle(index))
    ws = _WS.get(key)
    if ws is None or ws.numel() < n:
        if ws is not None:
            _WS_RETIRED.append(ws)
        ws = torch.empty(n, dtype=torch.uint8, device=torch.device("cuda", index))
        _WS[key] = ws
    return ws


def bwd_workspace(M, N, dtype, device):
    """A workspace for the backward on `device`, cached per (device, stream)
    so that calls sharing it are ordered on the GPU."""
    device = torch.device(device)
    index = device.index if device.index is not None else torch.cuda.current_device()
    with _on_device(index):
        return _workspace(M, N, _CODES[dtype], index)


def rmsnorm_fwd(x, gamma, eps, *, y=None, rstd=None, store_rstd=True):
    """y = x * rstd * gamma with rstd = 1/sqrt(mean(x^2) + eps) per row.
    Returns (y, rstd); rstd is fp32 [M] (None when store_rstd is False)."""
    _need("x", x, x)
    _need("gamma", gamma, x)
    M, N = _rows(x, gamma)
    with _on_device(x.get_device()):
        y = torch.empty_like(x) if y is None else _need("y", y, x, x.shape)
        if store_rstd:
            rstd = (torch.empty(M, dtype=torch.float32, device=x.device) if rstd is None
                    else _need("rstd", rstd, x, (M,), torch.float32))
        else:
            rstd = None
        native.check(native.lib().rn_rmsnorm_fwd(_ptr(x), _ptr(gamma), float(eps), _ptr(y),
                                                 _ptr(rstd), M, N, _code(x), _stream_handle(x.get_device())))
    return y, rstd


def fused_add_rmsnorm_fwd(x, residual, gamma, eps, *, out=None, residual_out=None, rstd=None,
                          store_rstd=True):
    """added = x + residual (rounded to the dtype) -> residual_out;
    out = added * rstd * gamma. Returns (out, residual_out, rstd)."""
    _need("x", x, x)
    _need("residual", residual, x, x.shape)
    _need("gamma", gamma, x)
    M, N = _rows(x, gamma)
    with _on_device(x.get_device()):
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
            _ptr(rstd), M, N, _code(x), _stream_handle(x.get_device())))
    return out, residual_out, rstd


def _bwd_outputs(x, M, N, dx, dweight_f32, dweight, want_cast, want_f32):
    dx = torch.empty_like(x) if dx is None else _need("dx", dx, x, x.shape)
    if dweight_f32 is not None:
        _need("dweight_f32", dweight_f32, x, (N,), torch.float32)
    elif want_f32:
        dweight_f32 = torch.empty(N, dtype=torch.float32, device=x.device)
    if dweight is None and want_cast:
        dweight = torch.empty(N, dtype=x.dtype, device=x.device)
    elif dweight is not None:
        _need("dweight", dweight, x, (N,))
    return dx, dweight_f32, dweight


def rmsnorm_bwd(x, gamma, dy, rstd, *, dx=None, dweight_f32=None, dweight=None,
                want_cast=True, want_f32=True, workspace=None):
    """Gradients of y = rmsnorm(x) * gamma given dy and the saved fp32 rstd.
    Returns (dx, dweight, dweight_f32); dweight is the weight gradient cast
    to the I/O dtype (None when want_cast is False and no buffer was passed),
    dweight_f32 its fp32 sum (None when want_f32 is False and no buffer was
    passed: the library then sums in its deterministic scratch mode)."""
    _need("x", x, x)
    _need("gamma", gamma, x)
    _need("dy", dy, x, x.shape)
    M, N = _rows(x, gamma)
    _need("rstd", rstd, x, (M,), torch.float32)
    with _on_device(x.get_device()):
        dx, dweight_f32, dweight = _bwd_outputs(x, M, N, dx, dweight_f32, dweight, want_cast,
                                                want_f32)
        ws = _workspace(M, N, _code(x), x.get_device()) if workspace is None else workspace
        native.check(native.lib().rn_rmsnorm_bwd(
            _ptr(x), _ptr(gamma), _ptr(dy), _ptr(rstd), _ptr(dx), _ptr(dweight_f32),
            _ptr(dweight), _ptr(ws), ws.numel(), M, N, _code(x), _stream_handle(x.get_device())))
    return dx, dweight, dweight_f32


def fused_add_rmsnorm_bwd(added, gamma, dy, rstd, dresidual_out=None, *, dx=None,
                          dweight_f32=None, dweight=None, want_cast=True, want_f32=True,
                          workspace=None):
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
    with _on_device(added.get_device()):
        dx, dweight_f32, dweight = _bwd_outputs(added, M, N, dx, dweight_f32, dweight, want_cast,
                                                want_f32)
        ws = (_workspace(M, N, _code(added), added.get_device()) if workspace is None
              else workspace)
        native.check(native.lib().rn_fused_add_rmsnorm_bwd(
            _ptr(added), _ptr(gamma), _ptr(dy), _ptr(rstd), _ptr(dresidual_out), _ptr(dx),
            _ptr(dweight_f32), _ptr(dweight), _ptr(ws), ws.numel(), M, N, _code(added),
            _stream_handle(added.get_device())))
    return dx, dx, dweight, dweight_f32


def layernorm_fwd(x, gamma, beta, eps, *, y=None, mean=None, rstd=None, store_stats=True):
    """y = (x - mean) * rstd * gamma + beta per row, with mean and
    rstd = 1/sqrt(var + eps) over the last dimension (biased variance).
    beta may be None. Returns (y, mean, rstd); mean and rstd are fp32 [M]
    (None when store_stats is False)."""
    _need("x", x, x)
    _need("gamma", gamma, x)
    M, N = _rows(x, gamma)
    if beta is not None:
        _need("beta", beta, x, (N,))
    with _on_device(x.get_device()):
        y = torch.empty_like(x) if y is None else _need("y", y, x, x.shape)
        if store_stats:
            mean = (torch.empty(M, dtype=torch.float32, device=x.device) if mean is None
                    else _need("mean", mean, x, (M,), torch.float32))
            rstd = (torch.empty(M, dtype=torch.float32, device=x.device) if rstd is None
                    else _need("rstd", rstd, x, (M,), torch.float32))
        else:
            mean = rstd = None
        native.check(native.lib().rn_layernorm_fwd(
            _ptr(x), _ptr(gamma), _ptr(beta), float(eps), _ptr(y), _ptr(mean), _ptr(rstd), M, N,
            _code(x), _stream_handle(x.get_device())))
    return y, mean, rstd


def layernorm_bwd(x, gamma, dy, mean, rstd, *, dx=None, dgamma_f32=None, dbeta_f32=None,
                  dgamma=None, dbeta=None, want_dbeta=True, want_cast=True, want_f32=True,
                  workspace=None):
    """Gradients of y = layernorm(x) * gamma (+ beta) given dy and the saved
    fp32 mean and rstd. Returns (dx, dgamma, dbeta, dgamma_f32, dbeta_f32):
    the casts to the I/O dtype are None when want_cast is False, the fp32
    sums when want_f32 is False (and no buffer was passed); the dbeta pair is
    None when want_dbeta is False."""
    _need("x", x, x)
    _need("gamma", gamma, x)
    _need("dy", dy, x, x.shape)
    M, N = _rows(x, gamma)
    _need("mean", mean, x, (M,), torch.float32)
    _need("rstd", rstd, x, (M,), torch.float32)
    with _on_device(x.get_device()):
        dx = torch.empty_like(x) if dx is None else _need("dx", dx, x, x.shape)
        f32 = dict(dtype=torch.float32, device=x.device)
        if dgamma_f32 is not None:
            _need("dgamma_f32", dgamma_f32, x, (N,), torch.float32)
        elif want_f32:
            dgamma_f32 = torch.empty(N, **f32)
        if want_dbeta:
            if dbeta_f32 is not None:
                _need("dbeta_f32", dbeta_f32, x, (N,), torch.float32)
            elif want_f32:
                dbeta_f32 = torch.empty(N, **f32)
        else:
            dbeta_f32 = dbeta = None
        if dgamma is None and want_cast:
            dgamma = torch.empty(N, dtype=x.dtype, device=x.device)
        elif dgamma is not None:
            _need("dgamma", dgamma, x, (N,))
        if want_dbeta:
            if dbeta is None and want_cast:
                dbeta = torch.empty(N, dtype=x.dtype, device=x.device)
            elif dbeta is not None:
                _need("dbeta", dbeta, x, (N,))
        ws = (_workspace(M, N, _code(x), x.get_device(), layernorm=True) if workspace is None
              else workspace)
        native.check(native.lib().rn_layernorm_bwd(
            _ptr(x), _ptr(gamma), _ptr(dy), _ptr(mean), _ptr(rstd), _ptr(dx), _ptr(dgamma_f32),
            _ptr(dbeta_f32), _ptr(dgamma), _ptr(dbeta), _ptr(ws), ws.numel(), M, N, _code(x),
            _stream_handle(x.get_device())))
    return dx, dgamma, dbeta, dgamma_f32, dbeta_f32


def layernorm_bwd_workspace(M, N, dtype, device):
    """A workspace for layernorm_bwd on `device` (shared with the RMSNorm
    backward's cache: one buffer per (device, stream), grown as needed)."""
    device = torch.device(device)
    index = device.index if device.index is not None else torch.cuda.current_device()
    with _on_device(index):
        return _workspace(M, N, _CODES[dtype], index, layernorm=True)
