"""GB300-native fused GEMM-epilogue and back-to-back GEMM library.

The compute path is ``libcf_gb300.so`` (hand-written sm_103a CUDA behind the
C ABI in ``include/cf.h``); this package only builds it and marshals torch
tensors into its calls.  See ``binding`` for the wrappers.
"""
from .binding import (CFError, cf_b2bgemm, cf_cost_b2bgemm, cf_cost_gemm_epilogue, cf_gemm_epilogue,  # noqa: F401
                      cf_gemm_epilogue_noalloc, cf_last_device_status, cf_status_string, cf_unfused_b2bgemm,
                      cf_unfused_gemm_epilogue, cf_workspace_size, load_library)

__all__ = ["CFError", "cf_b2bgemm", "cf_cost_b2bgemm", "cf_cost_gemm_epilogue", "cf_gemm_epilogue",
           "cf_gemm_epilogue_noalloc", "cf_last_device_status", "cf_status_string", "cf_unfused_b2bgemm",
           "cf_unfused_gemm_epilogue", "cf_workspace_size", "load_library"]
