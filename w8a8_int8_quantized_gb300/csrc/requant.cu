// FP8 E4M3 block-scaled weight -> INT8 weight with one float32 scale per row.
//
// "MiniMax-M2.7 FP8 转昆仑芯 INT8" README, section 转换关系:
//   W[i,j] = W_fp8[i,j] * weight_scale_inv[i//128, j//128]   (the _inv scale multiplies)
//   s[i]   = max_j |W[i,j]| / 127 ;  q = clamp(round(W / s), -127, 127) ;  zero row -> q=0, s=1.
// Rows are independent (the README's tool also works matrix by matrix, row chunk by row
// chunk), so one warp owns one row: it reads the row's codes once with 16-byte loads,
// keeps them in registers, reduces the absmax with shuffles and writes q from the cached
// codes.  One launch covers a whole batch of matrices through a by-value descriptor table.
#include "common.cuh"
#include "internal.h"

namespace w8a8 {

// E4M3 ("fn": bias 7, no infinities) -> float32, from the format definition: the 7
// exponent+mantissa bits are placed at the top of a float32's exponent/mantissa fields,
// which reads them with bias 127 instead of 7, and the 2^120 factor restores the value.
// Exponent field 0 lands on float32 subnormals, which the exact power-of-two multiply
// turns into m * 2^-9.  NaN codes (S.1111.111) are screened by the caller.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t b = ((c & 0x80u) << 24) | ((c & 0x7Fu) << 20);
  return __fmul_rn(__uint_as_float(b), 0x1p120f);
}
__device__ __forceinline__ bool e4m3_is_nan(uint32_t c) { return (c & 0x7Fu) == 0x7Fu; }
__device__ __forceinline__ bool scale_ok(float s) { return (s > 0.f) && (s <= 3.402823466e38f); }

constexpr int kReqMaxVec = 8;   // 16-byte vectors cached per lane -> rows up to 4096 codes

__device__ __forceinline__ void req_row_vec(const ReqMat& mt, int64_t i, int lane, int32_t* st) {
  const int64_t K = mt.K;
  const int nv = (int)(K / 16);
  const int nbc = (int)((K + 127) / 128);
  const uint4* wr = reinterpret_cast<const uint4*>(mt.w + i * K);
  const float* srow = mt.sinv + (i / 128) * nbc;
  uint4 c[kReqMaxVec];
  float amax = 0.f;
  bool bad = false;
#pragma unroll
  for (int v = 0; v < kReqMaxVec; ++v) {
    const int idx = lane + v * 32;
    if (idx < nv) {
      c[v] = wr[idx];
      const float sc = srow[idx >> 3];  // 16 codes per vector, 8 vectors per 128-column block
      bad |= !scale_ok(sc);
      const uint32_t wd[4] = {c[v].x, c[v].y, c[v].z, c[v].w};
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t code = (wd[j >> 2] >> (8 * (j & 3))) & 0xFFu;
        bad |= e4m3_is_nan(code);
        const float f = __fmul_rn(e4m3_value(code), sc);
        bad |= !(fabsf(f) <= 3.402823466e38f);
        amax = fmaxf(amax, fabsf(f));
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  bad = __any_sync(0xffffffffu, bad);
  float s = 1.f;
  if (!bad && amax != 0.f) s = __fdiv_rn(amax, 127.f);
  uint4* qr = reinterpret_cast<uint4*>(mt.q + i * K);
#pragma unroll
  for (int v = 0; v < kReqMaxVec; ++v) {
    const int idx = lane + v * 32;
    if (idx < nv) {
      uint4 o = make_uint4(0, 0, 0, 0);
      if (!bad) {
        const float sc = srow[idx >> 3];
        const uint32_t wd[4] = {c[v].x, c[v].y, c[v].z, c[v].w};
        uint32_t ow[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          int qq[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t code = (wd[g] >> (8 * j)) & 0xFFu;
            qq[j] = quant_sym(__fmul_rn(e4m3_value(code), sc), s);
          }
          ow[g] = pack4_i8(qq[0], qq[1], qq[2], qq[3]);
        }
        o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
      qr[idx] = o;
    }
  }
  if (lane == 0) {
    mt.s[i] = s;
    if (bad) report_status(st, W8A8_ERR_BAD_SCALE);
  }
}

// Any K and alignment: byte loads, two passes over the row.
__device__ __forceinline__ void req_row_generic(const ReqMat& mt, int64_t i, int lane, int32_t* st) {
  const int64_t K = mt.K;
  const int nbc = (int)((K + 127) / 128);
  const uint8_t* wr = mt.w + i * K;
  const float* srow = mt.sinv + (i / 128) * nbc;
  float amax = 0.f;
  bool bad = false;
  for (int64_t j = lane; j < K; j += 32) {
    const uint32_t code = wr[j];
    const float sc = srow[j >> 7];
    bad |= !scale_ok(sc) || e4m3_is_nan(code);
    const float f = __fmul_rn(e4m3_value(code), sc);
    bad |= !(fabsf(f) <= 3.402823466e38f);
    amax = fmaxf(amax, fabsf(f));
  }
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  bad = __any_sync(0xffffffffu, bad);
  float s = 1.f;
  if (!bad && amax != 0.f) s = __fdiv_rn(amax, 127.f);
  int8_t* qr = mt.q + i * K;
  for (int64_t j = lane; j < K; j += 32) {
    int v = 0;
    if (!bad) v = quant_sym(__fmul_rn(e4m3_value(wr[j]), srow[j >> 7]), s);
    qr[j] = (int8_t)v;
  }
  if (lane == 0) {
    mt.s[i] = s;
    if (bad) report_status(st, W8A8_ERR_BAD_SCALE);
  }
}

constexpr int kReqWarps = 8;

__global__ void __launch_bounds__(kReqWarps * 32)
requant_batch_kernel(const __grid_constant__ ReqBatch b, int32_t* st) {
  const int lane = threadIdx.x & 31;
  const int64_t grow = (int64_t)blockIdx.x * kReqWarps + (threadIdx.x >> 5);
  if (grow >= b.total_rows) return;
  // locate the matrix holding this global row (row0 is increasing)
  int lo = 0, hi = b.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (b.m[mid].row0 <= grow) lo = mid; else hi = mid - 1;
  }
  const ReqMat& mt = b.m[lo];
  const int64_t i = grow - mt.row0;
  if (mt.vec) req_row_vec(mt, i, lane, st);
  else req_row_generic(mt, i, lane, st);
}

cudaError_t requant_batch(const ReqBatch& b, int32_t* st, cudaStream_t stream) {
  if (b.total_rows == 0) return cudaSuccess;
  const int64_t blocks = (b.total_rows + kReqWarps - 1) / kReqWarps;
  requant_batch_kernel<<<(unsigned)blocks, kReqWarps * 32, 0, stream>>>(b, st);
  return cudaGetLastError();
}

bool requant_vec_ok(const uint8_t* w, const int8_t* q, int64_t K) {
  return (K % 16 == 0) && (K / 16 <= (int64_t)kReqMaxVec * 32) &&
         ((reinterpret_cast<uintptr_t>(w) & 15) == 0) && ((reinterpret_cast<uintptr_t>(q) & 15) == 0);
}

}  // namespace w8a8
