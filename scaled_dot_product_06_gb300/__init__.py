"""GB300-native fused scaled-dot-product attention (forward and backward).

The compute path is libsdpa.so (hand-written sm_103a CUDA behind the C ABI in
include/sdpa.h); this package is its PyTorch binding.
"""
from ._native import (SDPA_BWD_ALL, SDPA_BWD_DETERMINISTIC, SDPA_BWD_DKDV, SDPA_BWD_DQ,
                      SDPA_BWD_PREPROCESS)
from .api import (sdpa_bwd, sdpa_bwd_phases, sdpa_bwd_phases_varlen, sdpa_bwd_varlen,
                  sdpa_bwd_varlen_workspace_size, sdpa_bwd_workspace_size, sdpa_debug_fault,
                  sdpa_device_error, sdpa_dropout_mask, sdpa_fwd, sdpa_fwd_varlen,
                  sdpa_status_string)

__all__ = ["sdpa_fwd", "sdpa_bwd", "sdpa_bwd_phases", "SDPA_BWD_PREPROCESS", "SDPA_BWD_DKDV",
           "SDPA_BWD_DQ", "SDPA_BWD_ALL", "SDPA_BWD_DETERMINISTIC", "sdpa_bwd_workspace_size", "sdpa_dropout_mask",
           "sdpa_device_error", "sdpa_debug_fault", "sdpa_status_string", "sdpa_fwd_varlen",
           "sdpa_bwd_varlen", "sdpa_bwd_phases_varlen", "sdpa_bwd_varlen_workspace_size"]
