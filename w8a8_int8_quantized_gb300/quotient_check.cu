// Checks of the division-free rounding of the row rules (a standalone program, not part of
// libw8a8.so; built and run by quotient_check.py and the GPU tests).
//
// Symmetric rule, exhaustively: the quantizers compute the codes rint(RN(x / s)) of a bf16 row
// with s = RN(absmax / 127) without dividing (quant_row_group_x2 in common.cuh).  This program
// runs that very function on every case the rule can meet: every finite positive bf16 absmax
// a, and every bf16 x with |x| <= a, in groups of 8 as the kernels call it, and compares each
// code with rint of the IEEE float32 quotient (__fdiv_rn), ties to even.
//
// Affine rule, on 65536 row ranges: (lo, hi) pairs of bf16 values drawn by a counter-based
// hash (SplitMix64), three in four with random signs and exponents and one in four with an
// exact power-of-two scale s = 2^j and lo = -k s (exact ties, odd and even zero points); for
// each, every bf16 x in [lo, hi] goes through quant_row_group_affine_x2 with the scale, zero
// point and window the activation quantizer computes, against clamp(rint(IEEE x / s) + zp);
// affine_code_exact, the decision the flagged values get, is also run on every one of them.
//
// Prints the numbers of values tested and of mismatching codes as JSON.  Device work only;
// no waits.
#include <cstdio>
#include <cstdint>

#include "common.cuh"

using namespace w8a8;

__global__ void __launch_bounds__(256) sym_codes_kernel(unsigned long long* cnt) {
  const uint32_t ab = blockIdx.x + 1;  // positive bf16 patterns 0x0001 .. 0x7F7F
  const float a = __uint_as_float(ab << 16);
  const RowQuant rq = row_quant_sym(a);
  const float r = __frcp_rn(rq.s);
  unsigned long long tested = 0, bad = 0;
  // 8192 groups of 8 consecutive bf16 patterns cover all 65536
  for (uint32_t gidx = threadIdx.x; gidx < 8192u; gidx += blockDim.x) {
    float f[8];
    bool use[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = __uint_as_float((gidx * 8u + (uint32_t)j) << 16);
      use[j] = fabsf(x) <= a;  // excludes NaN and values beyond the row's absmax
      f[j] = use[j] ? x : 0.f;
    }
    uint32_t b[8];
    quant_row_group_x2<8>(f, rq.s, r, b);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!use[j]) continue;
      const int code = (int)(b[j] - 0x4B400000u);
      const int ref = __float2int_rn(rintf(__fdiv_rn(f[j], rq.s)));
      ++tested;
      bad += (code != ref);
    }
  }
  atomicAdd(&cnt[0], tested);
  atomicAdd(&cnt[1], bad);
}

__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// one (lo, hi) range per block
__global__ void __launch_bounds__(256) affine_codes_kernel(unsigned long long* cnt) {
  const uint64_t h = splitmix64(blockIdx.x);
  float lo, hi;
  if ((blockIdx.x & 3) == 3) {
    const int j = (int)(h % 16) - 10;  // s = 2^j, j in [-10, 5]
    const float s = ldexpf(1.f, j);
    const int k = (int)((h >> 8) % 256);
    lo = -(float)k * s;
    hi = lo + 255.f * s;
  } else {
    // bf16 values with biased exponents 110 .. 141 and random signs and mantissas
    const uint32_t a = ((uint32_t)(h & 0x807F) | ((110u + (uint32_t)((h >> 16) & 31)) << 7)) << 16;
    const uint32_t b = ((uint32_t)((h >> 24) & 0x807F) | ((110u + (uint32_t)((h >> 40) & 31)) << 7)) << 16;
    lo = fminf(__uint_as_float(a), __uint_as_float(b));
    hi = fmaxf(__uint_as_float(a), __uint_as_float(b));
  }
  if (!(lo < hi)) return;
  const RowQuant rq = row_quant_asym(lo, hi);
  const float r = __frcp_rn(rq.s);
  const float tmax = __fmul_rn(fmaxf(fabsf(lo), fabsf(hi)), r);
  const float thr = __fsub_rd(0.5f, __fmul_rn(tmax, 0x1p-21f));
  unsigned long long tested = 0, bad = 0, bad_exact = 0;
  for (uint32_t gidx = threadIdx.x; gidx < 8192u; gidx += blockDim.x) {
    float f[8];
    bool use[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = __uint_as_float((gidx * 8u + (uint32_t)j) << 16);
      use[j] = x >= lo && x <= hi;  // excludes NaN and values outside the row's range
      f[j] = use[j] ? x : lo;
    }
    uint32_t w[2];
    quant_row_group_affine_x2<8>(f, rq.s, r, rq.zp, thr, w);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (!use[j]) continue;
      const int code = (int)(int8_t)((w[j >> 2] >> (8 * (j & 3))) & 0xFFu);
      const long long v = (long long)__float2int_rn(rintf(__fdiv_rn(f[j], rq.s))) + rq.zp;
      const int ref = (int)min(127ll, max(-128ll, v));
      ++tested;
      bad += (code != ref);
      bad_exact += (affine_code_exact(f[j], rq.s, r, rq.zp, thr) != ref);
    }
  }
  atomicAdd(&cnt[2], tested);
  atomicAdd(&cnt[3], bad);
  atomicAdd(&cnt[4], bad_exact);
}

int main() {
  unsigned long long* d = nullptr;
  if (cudaMalloc(&d, 5 * sizeof(unsigned long long)) != cudaSuccess) return 1;
  cudaMemset(d, 0, 5 * sizeof(unsigned long long));
  sym_codes_kernel<<<0x7F7F, 256>>>(d);
  affine_codes_kernel<<<65536, 256>>>(d);
  const cudaError_t e = cudaDeviceSynchronize();
  unsigned long long h[5] = {0, 0, 0, 0, 0};
  cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  printf("{\"symmetric_rule\": {\"values\": %llu, \"code_mismatches\": %llu}, "
         "\"affine_rule\": {\"values\": %llu, \"code_mismatches\": %llu, \"exact_resolver_mismatches\": %llu}, "
         "\"cuda_error\": %d}\n",
         h[0], h[1], h[2], h[3], h[4], (int)e);
  return e == cudaSuccess ? 0 : 1;
}
