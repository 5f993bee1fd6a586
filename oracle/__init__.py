"""CPU oracle for the W8A8 INT8 quantized linear layer -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously correct restatement of what the GPU
library computes.  It exists so that tests, the package's smoke check and the
benchmark's CPU-baseline leg can compare the CUDA kernels against something
written directly from the method's published description.  The product path
never imports it and it imports nothing from the product package.

Sources (cited throughout by these short names):

  [vLLM-W8A8]  "vLLM INT8 W8A8 量化实战：用 llm-compressor 制作 8 位权重与 8 位激活的推理模型"
               (blog.gitcode.com); sections 4.1 方案判定, 4.2 权重布局与 kernel 选择.
  [SGLang-CT]  "[SGLang] W4A8, W8A8, W4A4: 혼합 정밀도 양자화 스킴"
               (blog.secrett2633.cloud); items 3 (W8A8 INT8: 정수 양자화),
               4 (W8A8 INT8 비대칭 양자화: AZP 보정), 7 (텐서별 스케일 후처리:
               requantize_with_max_scale), 설계 근거 3 (Fused 모듈 호환).
  [Kunlun-INT8] "MiniMax-M2.7 FP8 转昆仑芯 INT8" (README on dev.modelhub.org.cn);
               sections 转换关系 (conversion relation) and 验证 (validation).

Pin status of each function (what ties it to something other than itself; the
pins live in tests/test_oracle_*.py and tests/golden/):

  quantize_act_dynamic_symmetric   pinned: hand-worked golden example, half-step
                                   bound, absmax -> +-127, zero rows, zero padding.
  quantize_act_dynamic_asymmetric  pinned by invariants only (reconstruction bound,
                                   endpoint mapping, integer zero point); the pages
                                   name the mode but print no formula -- the affine
                                   min/max reading is ours.
  quantize_act_static_*            pinned: hand-worked golden example, half-step bound.
  int8_gemm                        pinned: brute-force integer triple loop.
  azp_adj                          pinned: brute-force sum, and the identity
                                   sum_k (q-zp)*w == acc - zp*azp_adj.
  scaled_mm_epilogue               pinned: hand-worked golden example; closed-form
                                   error bound against the unquantized fp64 product.
  quantize_weight_per_channel      pinned as quantize_act_dynamic_symmetric (same rule).
  e4m3_to_f32                      pinned: all 256 codes against hand-derived table
                                   values and a library cast.
  fp8_block_to_int8_rowwise        pinned: half-step bound, zero rows, ragged == padded,
                                   illegal scales, hand-worked golden example.
  moe_forward                      pinned: segment == dense per-expert call, combine
                                   == per-token loop, empty experts.
  moe_combine                      pinned: through moe_forward (above); one slot of
                                   weight 1 gathers the rows exactly, power-of-two
                                   weights scale exactly.
  requantize_with_max_scale        pinned: the max-scale partition is unchanged for
                                   every code, power-of-two ratios reduce to
                                   rint(q / 2^j) (ties to even), the half-step bound
                                   of the requantized value against q * s_p.
  moe_route                        pinned: brute-force top-k by pairwise comparison
                                   (ties to the lower index), weights summing to 1
                                   over all experts, hand-worked example.
"""

from .w8a8_oracle import (  # noqa: F401
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    quantize_act_dynamic_symmetric,
    quantize_act_dynamic_asymmetric,
    quantize_act_static_symmetric,
    quantize_act_static_asymmetric,
    static_scale_from_tensor,
    int8_gemm,
    azp_adj,
    scaled_mm_epilogue,
    w8a8_linear,
    quantize_weight_per_channel,
    e4m3_to_f32,
    fp8_block_to_int8_rowwise,
    silu_mul_bf16,
    moe_sort,
    moe_forward,
    moe_combine,
    moe_route,
    requantize_with_max_scale,
)
