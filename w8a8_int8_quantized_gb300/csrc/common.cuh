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

// The same integer as rint_div, returned as an int and computed without conversion-pipe
// instructions on the fast path: for |t| < 2^22, t + 1.5*2^23 lands in [2^23, 2^24) where
// float32 spacing is exactly 1, so the addition itself rounds t to the nearest integer
// (ties to even), subtracting 1.5*2^23 back is exact, and the integer is the low mantissa
// bits of the sum minus 2^22.  The fast path is only taken for |t| < 2^19.  The slow path
// clamps to +-2^30 so that adding a zero point cannot overflow.
__device__ __forceinline__ int rint_div_i(float x, float s, float r) {
  const float t = __fmul_rn(x, r);
  const float m = __fadd_rn(t, 12582912.0f);
  const float n = __fsub_rn(m, 12582912.0f);
  const float d = fabsf(__fsub_rn(fabsf(__fsub_rn(t, n)), 0.5f));
  if (d > __fmul_rn(fabsf(t), 0x1p-20f)) return __float_as_int(m) - 0x4B400000;
  const float e = rintf(__fdiv_rn(x, s));
  return __float2int_rn(fminf(fmaxf(e, -1073741824.0f), 1073741824.0f));
}

// rint_div_i for quotients known to satisfy |x/s| <= 256 (a row divided by its own
// absmax/127, or anything clamped to int8 range afterwards when it is that small): the
// margin |t|*2^-20 is then at most 2^-12, used as a constant, and the slow path needs no
// clamp.
__device__ __forceinline__ int rint_div_small(float x, float s, float r) {
  const float t = __fmul_rn(x, r);
  const float m = __fadd_rn(t, 12582912.0f);
  const float e = __fsub_rn(t, __fsub_rn(m, 12582912.0f));
  if (fabsf(e) < 0.499755859375f) return __float_as_int(m) - 0x4B400000;  // 0.5 - 2^-12, exact
  return __float2int_rn(rintf(__fdiv_rn(x, s)));
}

// ---- packed float32 pairs (sm_100+ f32x2 arithmetic): element 0 in the low 32 bits
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// The symmetric row rule's codes rint(RN(x / s)) for N values (N even), without a division:
// q0 = RN(x * r) with r = RN(1 / s), the remainder x - q0 * s (exact by fma), and one
// correction q = RN(q0 + (x - q0 * s) * r) (Markstein's correction step, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34, 1990).
// q is RN(x / s) or an adjacent float; rint(q) equals rint(RN(x / s)) for every bf16 x with
// |x| <= a and s = RN(a / 127), a any finite positive bf16 with s in [2^-100, 2^100]: checked
// exhaustively against the IEEE division (quotient_check.cu, run by the GPU tests).  An exact
// tie x / s = k + 1/2 gives q = k + 1/2 exactly, which rint breaks to even, so no tie needs
// detecting.  rint is the addition of 1.5 * 2^23 (|q| <= 128): the integer is the low
// mantissa bits of the sum, returned here as the sum's bit pattern.  Scales outside that
// range divide.
template <int N>
__device__ __forceinline__ void quant_row_group_x2(const float* x, float s, float r, uint32_t* b) {
  const uint64_t kMagic = 0x4B4000004B400000ull;  // 1.5*2^23 in both lanes
  if (s >= 0x1p-100f && s <= 0x1p100f) {
    const uint64_t r2 = f2pack(r, r), ns2 = f2pack(-s, -s);
#pragma unroll
    for (int j = 0; j < N; j += 2) {
      const uint64_t x2 = f2pack(x[j], x[j + 1]);
      const uint64_t q0 = f2mul(x2, r2);
      const uint64_t q = f2fma(f2fma(q0, ns2, x2), r2, q0);
      float m0, m1;
      f2unpack(f2add(q, kMagic), m0, m1);
      b[j] = __float_as_uint(m0);
      b[j + 1] = __float_as_uint(m1);
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) b[j] = 0x4B400000u + (uint32_t)__float2int_rn(rintf(__fdiv_rn(x[j], s)));
  }
}

// The per-token row rule: scale (and zero point) of one row from its statistics.  Symmetric:
// s = absmax / 127 (a zero row gets s = 1).  Affine: s = (hi - lo) / 255, zp = rint(-128 - lo / s)
// (int32, unclamped); a constant row (hi == lo) falls back to the symmetric rule with zp = 0.
// Shared by the stand-alone quantizers and the quantizer fused into the decode GEMM, so both
// produce the same codes.
struct RowQuant {
  float s;
  int zp;
  int affine;
};

__device__ __forceinline__ RowQuant row_quant_sym(float absmax) {
  RowQuant r;
  r.s = (absmax == 0.f) ? 1.f : __fdiv_rn(absmax, 127.f);
  r.zp = 0;
  r.affine = 0;
  return r;
}

__device__ __forceinline__ RowQuant row_quant_asym(float lo, float hi) {
  RowQuant r;
  if (hi == lo) {
    r.s = (hi == 0.f) ? 1.f : __fdiv_rn(fabsf(hi), 127.f);
    r.zp = 0;
    r.affine = 0;
  } else {
    r.s = __fdiv_rn(__fsub_rn(hi, lo), 255.f);
    r.zp = __float2int_rn(__fsub_rn(-128.f, __fdiv_rn(lo, r.s)));
    r.affine = 1;
  }
  return r;
}

__device__ __forceinline__ int apply_rq(const RowQuant& r, float x) {
  return r.affine ? quant_asym(x, r.s, r.zp) : quant_sym(x, r.s);
}

// four int32 values saturated to [-128, 127] and packed into one word, byte 0 = a
__device__ __forceinline__ uint32_t pack4_i8_sat(int a, int b, int c, int d) {
  uint32_t hi, w;
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi) : "r"(d), "r"(c));
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(w) : "r"(b), "r"(a), "r"(hi));
  return w;
}

// Per-byte +1 / -1 for the signs of four int8 values (prmt with sign replication gives
// 0xFF for a negative byte, 0x00 otherwise; or-ing 0x01 makes those -1 and +1).
__device__ __forceinline__ int sign_bytes(uint32_t w) {
  uint32_t s;
  asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(s) : "r"(w));
  return (int)(s | 0x01010101u);
}
// sum and sum of absolute values of the four int8 values of w, added to acc
__device__ __forceinline__ int sum4_i8(uint32_t w, int acc) { return __dp4a((int)w, 0x01010101, acc); }
__device__ __forceinline__ int abssum4_i8(uint32_t w, int acc) { return __dp4a((int)w, sign_bytes(w), acc); }

// ---- affine row rule q = clamp(rint(RN(x / s)) + zp, -128, 127) without dividing.
//
// Fast path: m = RN(x * r + (1.5*2^23 + zp)) by one fma (r = RN(1/s)); the low mantissa bits
// of m are rint(P) + zp with P = x * r the exact product (1.5*2^23 + zp is exact for |zp| <
// 2^22 and the sum lands where float spacing is 1).  P is within |x / s| * 2^-24 < ulp(x / s)
// of x / s, so within 1.5 ulps of RN(x / s).  With thr = 0.5 - tmax * 2^-21 (tmax the row's
// largest |x / s|, the callers' margin of at least four such ulps), every value whose
// e = RN(P - rint(P)) satisfies |e| < thr has rint(RN(x / s)) = rint(P).  The others lie near
// a half-integer (rows of bf16 values put a few tenths of a percent of their values there:
// quotients of short mantissas cluster near half-integers) and are flagged for
// affine_code_exact.  The packed operations are written as fma so that the compiler has no
// multiply-add left to fuse: the fast path's code is then reproducible one value at a time
// (affine_code_fast_one).
__device__ __forceinline__ bool affine_fast_ok(float s, float thr) {
  return s >= 0x1p-100f && s <= 0x1p100f && thr > 0.25f;
}

// N values (N even): codes (unclamped; 0 where the fast path does not apply) and the mask of
// values that need affine_code_exact
template <int N>
__device__ __forceinline__ uint32_t affine_codes_fast(const float* x, float s, float r, int zp, float thr, int* qv) {
  if (!affine_fast_ok(s, thr)) {
#pragma unroll
    for (int j = 0; j < N; ++j) qv[j] = 0;
    return (N >= 32) ? 0xFFFFFFFFu : ((1u << N) - 1u);
  }
  const float mg = __fadd_rn(12582912.0f, (float)zp);
  const uint64_t mg2 = f2pack(mg, mg);
  const uint64_t r2 = f2pack(r, r);
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    const uint64_t x2 = f2pack(x[j], x[j + 1]);
    const uint64_t mm = f2fma(x2, r2, mg2);
    const uint64_t e2 = f2fma(x2, r2, f2sub(mg2, mm));  // RN(P - rint(P)); mg - m is exact
    float e0, e1, m0, m1;
    f2unpack(e2, e0, e1);
    f2unpack(mm, m0, m1);
    m |= ((fabsf(e0) < thr) ? 0u : (1u << j)) | ((fabsf(e1) < thr) ? 0u : (2u << j));
    qv[j] = __float_as_int(m0) - 0x4B400000;
    qv[j + 1] = __float_as_int(m1) - 0x4B400000;
  }
  return m;
}

// the code affine_codes_fast gives one value, clamped as the packing does
__device__ __forceinline__ int affine_code_fast_one(float x, float s, float r, int zp, float thr) {
  if (!affine_fast_ok(s, thr)) return 0;
  const float m = __fmaf_rn(x, r, __fadd_rn(12582912.0f, (float)zp));
  return min(127, max(-128, __float_as_int(m) - 0x4B400000));
}

// rint(RN(x / s)) + zp exactly (clamped), for any value; the common case without dividing.
// With t = RN(x * r) and h the half-integer nearest t: RN(x / s) equals h when |x / s - h| <
// ulp(h) / 2, is above h when x / s is above h + ulp(h) / 2 and below it symmetrically.  Scaled
// by s > 0 the test compares D = x - h * s with tau = s * ulp(h) / 2 = s * 2^(exponent of h) *
// 2^-24, which is exact for s in [2^-100, 2^100].  For |h| >= 1.5 both neighbours of h are
// ulp(h) away (h is not a power of two); for h = +-1/2 the neighbour toward zero is only
// ulp(h) / 2 away, but there the even code and the code toward zero are both 0, so the same
// test decides.  fma(-h, s, x) rounds D once, so |fma| < tau proves |D| < tau (code: h rounded
// half to even) and |fma| > tau proves |D| > tau (code: h + 1/2 or h - 1/2 by its sign).
// The same decision is right for a value far from every half-integer (x / s is then within
// 1/2 of h with the sign of D, as t is).  |fma| == tau (or NaN) and scales or quotients
// outside the fast path's range divide.
__device__ __forceinline__ int affine_code_exact(float x, float s, float r, int zp, float thr) {
  int code;
  bool divide = !affine_fast_ok(s, thr);
  if (!divide) {
    const float mg = __fadd_rn(12582912.0f, (float)zp);
    const float t = __fmul_rn(x, r);
    const float k = __fsub_rn(__fadd_rn(t, mg), mg);
    const float e = __fsub_rn(t, k);
    const float h = __fadd_rn(k, __uint_as_float((__float_as_uint(e) & 0x80000000u) | 0x3F000000u));
    const float dd = __fmaf_rn(-h, s, x);
    const float d = fabsf(dd);
    const float tau = __fmul_rn(__uint_as_float(__float_as_uint(h) & 0x7F800000u), __fmul_rn(s, 0x1p-24f));
    const int kd = __float_as_int(__fadd_rn(__fsub_rn(h, 0.5f), mg)) - 0x4B400000;  // h - 1/2 + zp
    code = kd + ((d < tau) ? ((kd - zp) & 1) : (dd > 0.f ? 1 : 0));
    divide = !(d < tau || d > tau);
  }
  if (divide) {
    const long long v = (long long)__float2int_rn(rintf(__fdiv_rn(x, s))) + (long long)zp;
    code = (int)min(127ll, max(-128ll, v));
  }
  return min(127, max(-128, code));
}

// N values (N % 4 == 0) of a row under the affine rule, written as N/4 packed words: the fast
// path, then each flagged value decided by affine_code_exact.
template <int N>
__device__ __forceinline__ void quant_row_group_affine_x2(const float* x, float s, float r, int zp, float thr,
                                                          uint32_t* out) {
  int qv[N];
  uint32_t m = affine_codes_fast<N>(x, s, r, zp, thr, qv);
  while (m) {  // rare: one value per iteration
    const int j = __ffs(m) - 1;
    m &= m - 1;
    float xj = x[0];
#pragma unroll
    for (int i = 1; i < N; ++i) xj = (j == i) ? x[i] : xj;
    const int v = affine_code_exact(xj, s, r, zp, thr);
#pragma unroll
    for (int i = 0; i < N; ++i) qv[i] = (j == i) ? v : qv[i];
  }
#pragma unroll
  for (int g = 0; g < N / 4; ++g) out[g] = pack4_i8_sat(qv[4 * g], qv[4 * g + 1], qv[4 * g + 2], qv[4 * g + 3]);
}

// four int8 values (low bytes of a, b, c, d) packed into one word, byte 0 = a
__device__ __forceinline__ uint32_t pack4_i8_prmt(int a, int b, int c, int d) {
  const uint32_t lo = __byte_perm((uint32_t)a, (uint32_t)b, 0x0040);
  const uint32_t hi = __byte_perm((uint32_t)c, (uint32_t)d, 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

// int8 x 4 -> fp16 x 4, exact: (v ^ 0x80) is v + 128 as an unsigned byte; placing it in the
// mantissa of 1024.0 (0x6400) gives 1024 + 128 + v, and subtracting 1152 leaves v.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(x, 0x64646464u, 0x4140);
  const uint32_t b = __byte_perm(x, 0x64646464u, 0x4342);
  const uint32_t bias = 0x64806480u;  // 1152.0 in both halves
  asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(lo) : "r"(a), "r"(bias));
  asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(hi) : "r"(b), "r"(bias));
}

// a value of a row quantized with that row's own absmax scale: |x / s| <= 127 (+ rounding)
__device__ __forceinline__ int quant_row_sym(float x, float s, float r) { return rint_div_small(x, s, r); }

__device__ __forceinline__ uint32_t pack4_i8(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xFF) | ((uint32_t)(b & 0xFF) << 8) | ((uint32_t)(c & 0xFF) << 16) |
         ((uint32_t)(d & 0xFF) << 24);
}

// two small integers (|v| <= 2048, exact in fp16) packed as fp16x2
__device__ __forceinline__ uint32_t pack_f16x2(int lo, int hi) {
  __half2 v = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
  return *reinterpret_cast<uint32_t*>(&v);
}

// two small integral floats (exact in fp16) packed as fp16x2

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

// ---------------------------------------------------------------------------
// Bounds-checked build (-DW8A8_DEBUG, libw8a8_debug.so): W8A8_DOK(cond, site) guards a
// global-memory access whose index the kernel itself computed.  When the invariant fails it
// records `site` in the error word registered with w8a8_debug_set_error_word (first code
// wins) and the access is skipped, so a broken index never reaches memory and never traps.
// In the release build it is the constant true and compiles away.
// ---------------------------------------------------------------------------
#ifdef W8A8_DEBUG
static __device__ int32_t* g_w8a8_debug_word = nullptr;
__device__ __forceinline__ bool w8a8_dok(bool ok, int site) {
  if (!ok) {
    int32_t* w = g_w8a8_debug_word;
    if (w) atomicCAS(w, 0, site);
  }
  return ok;
}
#define W8A8_DOK(cond, site) ::w8a8::w8a8_dok((cond), (site))
// this translation unit's copy of the error-word pointer (called from its register function)
static inline cudaError_t w8a8_debug_register_here(int32_t* word) {
  return cudaMemcpyToSymbol(g_w8a8_debug_word, &word, sizeof(word));
}
#else
#define W8A8_DOK(cond, site) true
#endif

// Record a device-side condition: the first non-zero code wins.
__device__ __forceinline__ void report_status(int32_t* st, int code) {
  if (st) atomicCAS(st, 0, code);
}

}  // namespace w8a8
