"""GB300-native (sm_103a) W8A8 INT8 quantized linear layer.

The compute lives in libw8a8.so (hand-written CUDA behind the C ABI declared in
include/w8a8.h); this package is its thin ctypes binding plus seeded workload
generators.  Importing the package does not load the library; the first call does,
and raises if the library is missing.
"""

from ._binding import (  # noqa: F401
    ACT_DYN_TOKEN_ASYM,
    ACT_DYN_TOKEN_SYM,
    ACT_STATIC_TENSOR_ASYM,
    ACT_STATIC_TENSOR_SYM,
    LIB_PATH,
    PackedActivations,
    SIGNATURES,
    act_packed_size,
    grouped_mm_packed,
    moe_quantize_gather_packed,
    moe_quantize_scatter_packed,
    quantize_act_packed,
    scaled_mm_packed,
    silu_mul_quant_packed,
    W8A8Error,
    W_CHANNEL,
    W_TENSOR,
    azp_adj,
    fp8block_to_int8_rowwise,
    fp8block_to_int8_rowwise_batched,
    grouped_mm,
    lib,
    linear,
    linear_workspace_size,
    moe_combine,
    moe_forward,
    moe_quantize_gather,
    moe_route,
    quantize_act,
    quantize_weight,
    requantize_max_scale,
    scaled_mm,
    set_gemm_engine,
    splitk_workspace_size,
    weight_sumsq,
    silu_mul_quant,
)
