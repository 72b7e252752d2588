"""2:4 semi-structured sparse training of transformer FFN layers on NVIDIA GB300.

The work is done by libprune24 (C ABI, include/prune24.h; CUDA kernels for
sm_103a under csrc/). This package is its thin Python binding: the functions
below carry the C names and only marshal torch tensors into pointers, sizes
and strides. There is no CPU fallback.
"""
from ._native import (P24_ECAPACITY, Hybrid, hyb_compress, hyb_sddmm, hyb_spmm, P24_EPI_ACT24, P24_EPI_BIAS, P24_EPI_RELU, P24_STEP_ACT24, P24_STEP_ADAPTERS,
                      P24_STEP_KEEP_MASKS, P24_STEP_VNM, STEP_PHASE_NAMES,
                      STEP_PHASES, STEP_WEIGHTS, P24Error, Sparse24, ffn24_step, ffn24_workspace_size,
                      ffn24_workspace_size_lowrank, ld_meta, ld_vals,
                      lib, masked_dw_gemm, p24_colsum, p24_colsum_noalloc, p24_gemm_nt, p24_gemm_tn,
                      p24_launch_count, p24_query_status, p24_query_timeout, p24_selftest_timeout, p24_transpose, prune24_compress,
                      prune24_compress_both, prune24_transpose_repack, spmm24_bwd_dx, spmm24_bwd_dx_lowrank,
                      spmm24_fwd, spmm24_fwd_lowrank, spmm24_fwd_sparse_act, vnm24_compress, vnm24_spmm)

__all__ = [
    "P24Error", "P24_ECAPACITY", "Sparse24", "Hybrid", "lib", "ld_meta", "ld_vals", "hyb_compress", "hyb_spmm", "hyb_sddmm",
    "prune24_compress", "prune24_compress_both", "prune24_transpose_repack", "vnm24_compress", "vnm24_spmm",
    "spmm24_fwd", "spmm24_fwd_sparse_act", "spmm24_bwd_dx", "masked_dw_gemm",
    "spmm24_fwd_lowrank", "spmm24_bwd_dx_lowrank", "p24_gemm_nt", "p24_gemm_tn", "p24_transpose",
    "p24_colsum", "p24_colsum_noalloc", "ffn24_step", "ffn24_workspace_size", "ffn24_workspace_size_lowrank",
    "p24_launch_count", "p24_query_status", "p24_query_timeout", "p24_selftest_timeout",
    "STEP_PHASES", "STEP_PHASE_NAMES", "STEP_WEIGHTS",
    "P24_EPI_ACT24", "P24_EPI_BIAS", "P24_EPI_RELU", "P24_STEP_ACT24", "P24_STEP_KEEP_MASKS", "P24_STEP_ADAPTERS", "P24_STEP_VNM",
]
