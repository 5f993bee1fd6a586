// Shared device helpers for the W8A8 INT8 library (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "w8a8.h"

namespace w8a8 {

// ---------------------------------------------------------------------------
// Rounding helpers.  Every quotient is the IEEE float32 round-to-nearest division
// and every integer conversion rounds half to even, so that the int8 codes agree
// bit for bit with a plain float32 evaluation of the same formulas.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// rint(x / s) clamped to [-127, 127]
__device__ __forceinline__ int quant_sym(float x, float s) {
  int v = __float2int_rn(__fdiv_rn(x, s));
  return min(127, max(-127, v));
}

// rint(x / s) + zp clamped to [-128, 127]; the sum is formed in 64 bits so that a
// saturated conversion plus a zero point cannot wrap.
__device__ __forceinline__ int quant_asym(float x, float s, int zp) {
  long long v = (long long)__float2int_rn(__fdiv_rn(x, s)) + (long long)zp;
  return (int)min(127ll, max(-128ll, v));
}

__device__ __forceinline__ uint32_t pack4_i8(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xFF) | ((uint32_t)(b & 0xFF) << 8) | ((uint32_t)(c & 0xFF) << 16) |
         ((uint32_t)(d & 0xFF) << 24);
}

// two small integers (|v| <= 2048, exact in fp16) packed as fp16x2
__device__ __forceinline__ uint32_t pack_f16x2(int lo, int hi) {
  __half2 v = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// Epilogue: y = bf16( (s_x*s_w) * f32(acc - zp*azp_adj) (+ bias) ), one rounding per
// operation, no contraction into fused multiply-add.
// ---------------------------------------------------------------------------
struct EpiParams {
  int act_mode;          // w8a8_act_mode
  int w_mode;            // w8a8_w_mode
  const float* s_x;      // [M] (dynamic) or [1] (static)
  const int32_t* zp;     // [M] (dynamic asym) or unused
  const int32_t* azp;    // [N] (asym) or unused
  const float* s_w;      // [N] (channel) or [1] (tensor)
  const __nv_bfloat16* bias;  // [N] or nullptr
};

__device__ __forceinline__ float epi_row_scale(const EpiParams& p, int64_t m) {
  return (p.act_mode == W8A8_ACT_DYN_TOKEN_SYM || p.act_mode == W8A8_ACT_DYN_TOKEN_ASYM) ? p.s_x[m]
                                                                                        : p.s_x[0];
}
__device__ __forceinline__ int epi_row_zp(const EpiParams& p, int64_t m) {
  return p.act_mode == W8A8_ACT_DYN_TOKEN_ASYM ? p.zp[m] : 0;
}
__device__ __forceinline__ float epi_apply(const EpiParams& p, int32_t acc, float sx, int zp_m,
                                           int64_t n) {
  long long c = acc;
  if (p.act_mode == W8A8_ACT_DYN_TOKEN_ASYM) c -= (long long)zp_m * (long long)p.azp[n];
  else if (p.act_mode == W8A8_ACT_STATIC_TENSOR_ASYM) c -= (long long)p.azp[n];
  const float cf = __ll2float_rn(c);
  const float sw = (p.w_mode == W8A8_W_CHANNEL) ? p.s_w[n] : p.s_w[0];
  const float t = __fmul_rn(sx, sw);
  float y = __fmul_rn(t, cf);
  if (p.bias) y = __fadd_rn(y, __bfloat162float(p.bias[n]));
  return y;
}

// Record a device-side condition: the first non-zero code wins.
__device__ __forceinline__ void report_status(int32_t* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

}  // namespace w8a8
