"""GB300-native RMSNorm forward/backward (plain and fused-add).

The compute runs in a CUDA library for sm_103a (``csrc/``, C ABI in
``include/rmsnorm_gb300.h``); this package is its thin PyTorch binding.
"""
from .ops import (bwd_workspace, fused_add_rmsnorm_bwd, fused_add_rmsnorm_fwd, rmsnorm_bwd,
                  rmsnorm_fwd)
from .autograd import FusedAddRMSNormFunction, RMSNormFunction, fused_add_rmsnorm, rmsnorm

__all__ = ["rmsnorm_fwd", "rmsnorm_bwd", "fused_add_rmsnorm_fwd", "fused_add_rmsnorm_bwd",
           "bwd_workspace", "rmsnorm", "fused_add_rmsnorm", "RMSNormFunction",
           "FusedAddRMSNormFunction"]
