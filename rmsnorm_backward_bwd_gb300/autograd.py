"""Autograd wrappers over the backward calls: ``rmsnorm`` and
``fused_add_rmsnorm`` as differentiable functions of (x, [residual], weight),
and ``layernorm`` of (x, weight, [bias]).

FlyDSL PR #800 ("Add fused-add / residual backward"), section "Summary" and
its PR 1 notes: the forward saves the per-row fp32 rstd; ``RMSNormFunction``
saves x, weight and rstd and its backward calls the RMSNorm backward; the
public ``rmsnorm(x, weight, eps)`` accepts inputs of any rank >= 1 (rows =
all leading dimensions). ``FusedAddRMSNormFunction`` is the prenorm variant:
it returns (out, residual_out), saves residual_out (= x + residual, the
tensor the statistic is taken of) and its backward consumes the gradients of
both outputs; the gradient of x and of residual is one and the same tensor
(dx == dresidual, since added = x + residual). Issue #769, "Proposed
approach" item 3: gradients flow through these wrappers transparently.

Marshalling only: inputs are flattened to [M, N] (a view when the input is
contiguous), gradients are made contiguous, and everything is computed by
the CUDA library. CUDA tensors only; weight (and bias) have the input's
dtype. ``LayerNormFunction`` follows the same pattern with the forward's mean
and rstd saved (issue #769 plan, "PR 5 -- LayerNorm backward"); its default
eps is torch's LayerNorm default, 1e-5 (the pages give none for it).
"""
import torch

from . import ops


def _rows2d(t, N):
    return t.reshape(-1, N).contiguous()


def _width(x):
    if x.dim() < 1:
        raise ValueError("input must have at least one dimension")
    return x.shape[-1]


class RMSNormFunction(torch.autograd.Function):
    """y = x * rstd * weight, rstd = 1/sqrt(mean(x^2) + eps) over the last dim."""

    @staticmethod
    def forward(ctx, x, weight, eps):
        shape = x.shape
        x2 = _rows2d(x, _width(x))
        y, rstd = ops.rmsnorm_fwd(x2, weight.contiguous(), eps)
        ctx.save_for_backward(x2, weight, rstd)
        ctx.shape = shape
        return y.view(shape)

    @staticmethod
    def backward(ctx, dy):
        x2, weight, rstd = ctx.saved_tensors
        need_x, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if not (need_x or need_w):
            return None, None, None
        dy2 = _rows2d(dy, x2.shape[1])
        dx, dweight, _ = ops.rmsnorm_bwd(x2, weight.contiguous(), dy2, rstd, want_cast=need_w)
        return (dx.view(ctx.shape) if need_x else None, dweight if need_w else None, None)


class FusedAddRMSNormFunction(torch.autograd.Function):
    """residual_out = x + residual (rounded to the dtype);
    out = residual_out * rstd * weight. Returns (out, residual_out)."""

    @staticmethod
    def forward(ctx, x, residual, weight, eps):
        shape = x.shape
        if residual.shape != shape:
            raise ValueError("residual has shape %s, expected %s" % (tuple(residual.shape),
                                                                    tuple(shape)))
        N = _width(x)
        out, residual_out, rstd = ops.fused_add_rmsnorm_fwd(
            _rows2d(x, N), _rows2d(residual, N), weight.contiguous(), eps)
        ctx.save_for_backward(residual_out, weight, rstd)
        ctx.shape = shape
        # a gradient that autograd does not produce stays None: no zero
        # tensor is made for residual_out when only `out` is used
        ctx.set_materialize_grads(False)
        return out.view(shape), residual_out.view(shape)

    @staticmethod
    def backward(ctx, d_out, d_residual_out):
        added, weight, rstd = ctx.saved_tensors
        need_x, need_r, need_w = ctx.needs_input_grad[:3]
        if not (need_x or need_r or need_w):
            return None, None, None, None
        N = added.shape[1]
        if d_out is None:
            if d_residual_out is None:
                return None, None, None, None
            # only residual_out was used: out's gradient is zero
            d_out = torch.zeros_like(added)
        dres = _rows2d(d_residual_out, N) if d_residual_out is not None else None
        dx, dresidual, dweight, _ = ops.fused_add_rmsnorm_bwd(
            added, weight.contiguous(), _rows2d(d_out, N), rstd, dres, want_cast=need_w)
        g = dx.view(ctx.shape)
        return (g if need_x else None, dresidual.view(ctx.shape) if need_r else None,
                dweight if need_w else None, None)


class LayerNormFunction(torch.autograd.Function):
    """y = (x - mean) * rstd * weight + bias over the last dim (bias may be None)."""

    @staticmethod
    def forward(ctx, x, weight, bias, eps):
        shape = x.shape
        x2 = _rows2d(x, _width(x))
        y, mean, rstd = ops.layernorm_fwd(x2, weight.contiguous(),
                                          bias.contiguous() if bias is not None else None, eps)
        ctx.save_for_backward(x2, weight, mean, rstd)
        ctx.shape = shape
        ctx.has_bias = bias is not None
        return y.view(shape)

    @staticmethod
    def backward(ctx, dy):
        x2, weight, mean, rstd = ctx.saved_tensors
        need_x, need_w, need_b = ctx.needs_input_grad[:3]
        need_b = need_b and ctx.has_bias
        if not (need_x or need_w or need_b):
            return None, None, None, None
        dy2 = _rows2d(dy, x2.shape[1])
        dx, dgamma, dbeta, _, _ = ops.layernorm_bwd(
            x2, weight.contiguous(), dy2, mean, rstd, want_dbeta=need_b,
            want_cast=need_w or need_b)
        return (dx.view(ctx.shape) if need_x else None, dgamma if need_w else None,
                dbeta if need_b else None, None)


def rmsnorm(x, weight, eps=1e-6):
    """Differentiable RMSNorm over the last dimension of x (any rank >= 1)."""
    return RMSNormFunction.apply(x, weight, eps)


def fused_add_rmsnorm(x, residual, weight, eps=1e-6, prenorm=True):
    """Differentiable fused residual add + RMSNorm. With prenorm (default)
    returns (out, residual_out); otherwise out alone."""
    out, residual_out = FusedAddRMSNormFunction.apply(x, residual, weight, eps)
    return (out, residual_out) if prenorm else out


def layernorm(x, weight, bias=None, eps=1e-5):
    """Differentiable LayerNorm over the last dimension of x (any rank >= 1);
    bias may be None."""
    return LayerNormFunction.apply(x, weight, bias, eps)
