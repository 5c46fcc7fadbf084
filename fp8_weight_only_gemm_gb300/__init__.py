"""GB300-native (sm_103a) W8A16 block-scaled GEMM.

C[M, N] (BF16) = A[M, K] (BF16, any row pitch) x dequant(W[N, K] FP8 E4M3, one FP32
scale per 128x128 block)^T, computed by hand-written tcgen05/TMA kernels in
``libw8a16.so`` behind a C ABI (include/w8a16.h). This package is the thin
Python binding: torch provides device memory and streams only. The library also
holds the weight block quantiser that produces W and the block scales.
"""
from .binding import (FLAG_PDL, Plan, VARIANT_AUTO, VARIANT_SIMT, VARIANT_TC, VARIANT_TC8, VARIANT_W8A8,
                      VARIANT_PRESPLIT, WEIGHTS_BF16, WEIGHTS_F32, W8A16Error,
                      check_args, cluster_capacity, device_status, gemm, gemm_host, gemm_noalloc, gemm_ptr,
                      gemm_split_terms, gemm_w8a8, gemm_w8a8_ptr, gemm_ws, gemm_ws_ptr, quantize_activations,
                      split_activations, workspace_bytes, workspace_bytes_for, VARIANT_GEMV, VARIANT_STREAM,
                      header_functions, last_error, load, plan_current, plan_for, plan_variant, plan_ws,
                      quantize_weights, quantize_weights_ptr, selftest_wait_timeout, strerror,
                      version)

__all__ = ["FLAG_PDL", "Plan", "VARIANT_AUTO", "VARIANT_SIMT", "VARIANT_TC", "VARIANT_TC8", "VARIANT_W8A8",
           "VARIANT_PRESPLIT", "WEIGHTS_BF16", "WEIGHTS_F32", "W8A16Error",
           "check_args", "cluster_capacity", "device_status", "gemm", "gemm_host", "gemm_noalloc", "gemm_ptr",
           "gemm_split_terms", "gemm_w8a8", "gemm_w8a8_ptr", "gemm_ws", "gemm_ws_ptr", "quantize_activations",
           "split_activations", "workspace_bytes", "workspace_bytes_for", "VARIANT_GEMV", "VARIANT_STREAM",
           "header_functions", "last_error", "load", "plan_current", "plan_for", "plan_variant", "plan_ws",
           "quantize_weights", "quantize_weights_ptr", "selftest_wait_timeout", "strerror",
           "version"]
