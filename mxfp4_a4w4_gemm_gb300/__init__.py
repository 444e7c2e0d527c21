"""GB300-native (sm_103a) MXFP4 A4W4 GEMM library.

The computation lives in liba4w4.so (hand-written CUDA: tcgen05 block-scaled
MMA, TMA bulk copies, TMEM accumulators); this package is its Python binding,
with the same names as the C ABI in include/a4w4.h.  PyTorch is used only for
device memory and streams.  Build the library with
``python -m mxfp4_a4w4_gemm_gb300.build``.
"""

from ._native import (  # noqa: F401
    A4W4_GEMM_WEIGHT_PREFETCH,
    A4W4_MOE_ACT_SILU,
    A4W4_MOE_ACT_SWIGLU,
    A4W4_MOE_OUT_ROWS,
    A4W4_MOE_OUT_TILES,
    A4W4Error,
    DEBUG_SIGNATURES,
    LIB_PATH,
    SIGNATURES,
    a4w4_debug_gemm_activation_layout,
    a4w4_debug_gemm_export,
    a4w4_debug_moe_gemm1_export,
    a4w4_gemm,
    a4w4_gemm_a16w4,
    a4w4_gemm_ex,
    a4w4_gemm_kernel_name,
    a4w4_gemm_noalloc,
    a4w4_gemm_workspace_bytes,
    a4w4_get_device_status,
    a4w4_moe_gemm1,
    a4w4_moe_gemm1_ex,
    a4w4_moe_gemm1_workspace_bytes,
    a4w4_moe_gemm2,
    a4w4_moe_gemm2_workspace_bytes,
    a4w4_moe_max_blocks,
    a4w4_moe_prepare_w1,
    a4w4_moe_sort,
    a4w4_moe_sort_aux,
    a4w4_moe_sort_aux_workspace_bytes,
    a4w4_moe_sort_workspace_bytes,
    a4w4_moe_tiles_codes_bytes,
    a4w4_moe_tiles_scales_bytes,
    a4w4_moe_w1_codes_bytes,
    a4w4_moe_w1_scales_bytes,
    a4w4_mxfp4_quant,
    a4w4_prepare_gemm_weight,
    a4w4_set_wait_limit_ns,
    a4w4_strerror,
    a4w4_weight_codes_bytes,
    a4w4_weight_scales_bytes,
    a4w4_workspace_init,
    lib,
)

A4W4_OK, A4W4_ERR_ARG, A4W4_ERR_DEVICE, A4W4_ERR_WORKSPACE, A4W4_ERR_LAUNCH, A4W4_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
