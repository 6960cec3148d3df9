"""Differentiable ``rmsnorm``, ``fused_add_rmsnorm`` and ``layernorm``.

FlyDSL PR #800 ("Add fused-add / residual backward"), section "Summary" and
its PR 1 notes: the forward saves the per-row fp32 rstd; ``RMSNormFunction``
saves x, weight and rstd and its backward calls the RMSNorm backward; the
public ``rmsnorm(x, weight, eps)`` accepts inputs of any rank >= 1 (rows =
all leading dimensions). ``FusedAddRMSNormFunction`` is the prenorm variant:
it returns (out, residual_out), saves residual_out (= x + residual, the
tensor the statistic is taken of) and its backward consumes the gradients of
both outputs; the gradient of x and of residual is one and the same tensor
(dx == dresidual, since added = x + residual). Issue #769, "Proposed
approach" item 3: gradients flow through these functions transparently.
``LayerNormFunction`` follows the same pattern with the forward's mean and
rstd saved (issue #769 plan, "PR 5 -- LayerNorm backward"); its default eps
is torch's LayerNorm default, 1e-5 (the pages give none for it).

The autograd functions themselves are C++ (``csrc/torch_ops.cpp``, the
operators ``torch.ops.rn_gb300.rmsnorm`` / ``fused_add_rmsnorm`` /
``layernorm``): their backward runs on the autograd engine's device thread
without entering Python, and every step of the computation runs in the CUDA
library. This module checks the device and forwards the call. CUDA tensors
only; weight (and bias) have the input's dtype.
"""
import torch

from . import native


def _ops():
    return native.torch_ops()


def _on_cuda(name, t):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dim() < 1:
        raise ValueError("input must have at least one dimension")
    if not t.is_cuda:
        # the library takes device pointers only; there is no CPU path
        raise ValueError("%s is on %s: these ops run on CUDA devices only" % (name, t.device))


class RMSNormFunction:
    """y = x * rstd * weight, rstd = 1/sqrt(mean(x^2) + eps) over the last
    dim; the C++ autograd function behind ``rmsnorm``."""

    @staticmethod
    def apply(x, weight, eps):
        _on_cuda("x", x)
        return _ops().rmsnorm(x, weight, float(eps))


class FusedAddRMSNormFunction:
    """residual_out = x + residual (rounded to the dtype);
    out = residual_out * rstd * weight. ``apply`` returns (out, residual_out)."""

    @staticmethod
    def apply(x, residual, weight, eps):
        _on_cuda("x", x)
        return _ops().fused_add_rmsnorm(x, residual, weight, float(eps))


class LayerNormFunction:
    """y = (x - mean) * rstd * weight + bias over the last dim (bias may be None)."""

    @staticmethod
    def apply(x, weight, bias, eps):
        _on_cuda("x", x)
        return _ops().layernorm(x, weight, bias, float(eps))


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
