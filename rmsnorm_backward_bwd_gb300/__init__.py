"""GB300-native RMSNorm forward/backward (plain and fused-add), with LayerNorm
forward/backward alongside.

The compute runs in a CUDA library for sm_103a (``csrc/``, C ABI in
``include/rmsnorm_gb300.h``); this package is its thin PyTorch binding.
"""
from .ops import (bwd_workspace, fused_add_rmsnorm_bwd, fused_add_rmsnorm_fwd, layernorm_bwd,
                  layernorm_bwd_workspace, layernorm_fwd, rmsnorm_bwd, rmsnorm_fwd)
from .autograd import (FusedAddRMSNormFunction, LayerNormFunction, RMSNormFunction,
                       fused_add_rmsnorm, layernorm, rmsnorm)

__all__ = ["rmsnorm_fwd", "rmsnorm_bwd", "fused_add_rmsnorm_fwd", "fused_add_rmsnorm_bwd",
           "bwd_workspace", "rmsnorm", "fused_add_rmsnorm", "RMSNormFunction",
           "FusedAddRMSNormFunction", "layernorm_fwd", "layernorm_bwd",
           "layernorm_bwd_workspace", "layernorm", "LayerNormFunction"]
