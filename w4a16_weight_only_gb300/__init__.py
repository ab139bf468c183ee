"""AWQ W4A16 weight-only linear for GB300 (sm_103a).

The computation lives in ``libawq_gb300.so`` (C ABI in ``include/awq.h``, CUDA sources
in ``csrc/``).  This package only builds it (``build.py``) and marshals arguments
(``_binding.py``); PyTorch supplies device memory and streams.
"""
from ._binding import (AwqError, AwqLinear, PATHS, awq_dequant, awq_dequant_w8, awq_gemm, awq_gemm_grouped,
                       awq_gemm_packed, awq_gemm_packed_grouped, awq_gemm_packed_noalloc,
                       awq_gemm_packed_workspace_size, awq_repack, awq_repack_experts, awq_repack_size,
                       awq_gemm_w8, awq_quantize_rtn,
                       device_status,
                       last_error, load_library, runtime_available, select_path,
                       selftest_wait_timeout)

__all__ = ["AwqError", "AwqLinear", "PATHS", "awq_dequant", "awq_dequant_w8", "awq_gemm", "awq_gemm_grouped",
           "awq_gemm_packed", "awq_gemm_packed_grouped", "awq_gemm_packed_noalloc",
           "awq_gemm_packed_workspace_size", "awq_repack", "awq_repack_experts", "awq_repack_size",
           "awq_gemm_w8", "awq_quantize_rtn",
           "device_status",
           "last_error",
           "load_library", "runtime_available", "select_path", "selftest_wait_timeout"]
