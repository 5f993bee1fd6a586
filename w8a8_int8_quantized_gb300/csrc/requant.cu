// FP8 E4M3 block-scaled weight -> INT8 weight with one float32 scale per row.
//
// "MiniMax-M2.7 FP8 转昆仑芯 INT8" README, section 转换关系:
//   W[i,j] = W_fp8[i,j] * weight_scale_inv[i//128, j//128]   (the _inv scale multiplies)
//   s[i]   = max_j |W[i,j]| / 127 ;  q = clamp(round(W / s), -127, 127) ;  zero row -> q=0, s=1.
// Rows are independent (the README's tool also works matrix by matrix, row chunk by row
// chunk), so one CTA owns one row: it reads the row's codes once with 16-byte loads,
// decodes them once into registers, reduces the absmax across the CTA and writes q from
// the cached values.  One launch covers a whole batch of matrices through a by-value
// descriptor table; ragged or unaligned matrices take a warp-per-row byte-load path.
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

// Vector path (K % 16 == 0, 16-byte aligned rows, any length): one warp per row, many
// warps per SM.  Pass 1 reads the row (16-byte groups) and finds its absmax; pass 2 reads it
// again, from L1/L2, and quantizes it.
//
// Row absmax without decoding every code: the codes of one 16-byte group share one block
// scale sc > 0, E4M3 magnitude grows with the 7-bit code (exponent bits above mantissa
// bits), and rounding is monotone, so max_j RN(|v_j| * sc) = RN(v(max_j code_j) * sc).
// The largest 7-bit code of a group is a byte-wise max; 0x7F, the largest, is the NaN
// code, so a group holds a NaN exactly when that max is 0x7F.
constexpr int kReqWarpsPerCta = 8;

// value of a non-negative 7-bit E4M3 code times 2^-120, exactly (as a float32 bit pattern)
__device__ __forceinline__ float e4m3_mag_scaled(uint32_t code7) { return __uint_as_float(code7 << 20); }

// any byte of w equal to 0x7F or 0xFF (the E4M3 NaN codes)
__device__ __forceinline__ bool has_nan_code(uint32_t w) {
  return (((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u) != 0u;
}

// The largest 7-bit code among 16 codes.
__device__ __forceinline__ uint32_t max_code7(const uint4& c) {
  uint32_t m = __vmaxu4(__vmaxu4(c.x & 0x7F7F7F7Fu, c.y & 0x7F7F7F7Fu), __vmaxu4(c.z & 0x7F7F7F7Fu, c.w & 0x7F7F7F7Fu));
  m = __vmaxu4(m, m >> 16);
  m = __vmaxu4(m, m >> 8);
  return m & 0xFFu;
}

// 16 codes of one group -> 16 int8 codes: Wf = RN(value * sc) (as (value*2^-120)*(sc*2^120),
// one rounding, or decoded exactly first when sc*2^120 would overflow), then q = rint(Wf/s)
// by the rint_div_small rule (|Wf| <= absmax, so |Wf / s| stays within 128).
__device__ __forceinline__ uint4 requant_group(const uint4& c, float sc, float s, float r) {
  const bool fast = fabsf(sc) < 256.f;
  const float sc2 = fast ? __fmul_rn(sc, 0x1p120f) : sc;
  const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
  float wf[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t top = __byte_perm(wd[j >> 2], 0u, 0x0444u | (uint32_t)((j & 3) << 12));  // byte -> bits 31:24
    float a = __uint_as_float((uint32_t)((int32_t)top >> 4) & 0x87F00000u);
    if (!fast) a = __fmul_rn(a, 0x1p120f);
    wf[j] = __fmul_rn(a, sc2);
  }
  uint32_t b[16];
  quant_row_group_x2<16>(wf, s, r, b);
  uint32_t out[4];
#pragma unroll
  for (int g = 0; g < 4; ++g)
    out[g] = __byte_perm(__byte_perm(b[4 * g], b[4 * g + 1], 0x0040), __byte_perm(b[4 * g + 2], b[4 * g + 3], 0x0040),
                         0x5410);
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__global__ void __launch_bounds__(kReqWarpsPerCta * 32)
requant_warp_kernel(const __grid_constant__ ReqBatch b, int32_t* st) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * kReqWarpsPerCta;
  for (int64_t grow = (int64_t)blockIdx.x * kReqWarpsPerCta + (threadIdx.x >> 5); grow < b.total_rows;
       grow += stride) {
    int lo = 0, hi = b.count - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (b.m[mid].row0 <= grow) lo = mid; else hi = mid - 1;
    }
    const ReqMat& mt = b.m[lo];
    const int64_t i = grow - mt.row0;
    const int K = mt.K;
    const int nv = K / 16;
    const int nbc = (K + 127) / 128;
    const uint4* wr = reinterpret_cast<const uint4*>(mt.w + i * (int64_t)K);
    const float* srow = mt.sinv + (i / 128) * nbc;
    // pass 1: absmax from the per-group largest code (reads the row from HBM into L1)
    float amax = 0.f;
    bool bad = false;
#pragma unroll 2
    for (int idx = lane; idx < nv; idx += 32) {
      const uint4 c = wr[idx];
      const float sc = srow[idx >> 3];  // 16 codes per group, 8 groups per 128-column block
      const uint32_t mc = max_code7(c);
      bad |= (mc == 0x7Fu) || !scale_ok(sc);
      amax = fmaxf(amax, __fmul_rn(__fmul_rn(__uint_as_float(mc << 20), 0x1p120f), sc));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    bad = __any_sync(0xffffffffu, bad) || !(amax <= 3.402823466e38f);
    float s = 1.f;
    if (!bad && amax != 0.f) s = __fdiv_rn(amax, 127.f);
    const float r = __frcp_rn(s);
    // pass 2: decode, quantize, store (the row is read again, now from L1/L2)
    uint4* qr = reinterpret_cast<uint4*>(mt.q + i * (int64_t)K);
#pragma unroll 2
    for (int idx = lane; idx < nv; idx += 32)
      qr[idx] = bad ? make_uint4(0u, 0u, 0u, 0u) : requant_group(wr[idx], srow[idx >> 3], s, r);
    if (lane == 0) {
      mt.s[i] = s;
      if (bad) report_status(st, W8A8_ERR_BAD_SCALE);
    }
  }
}

static void launch_requant_warps(const ReqBatch& b, int32_t* st, cudaStream_t stream) {
  static unsigned cached = 0;
  if (cached == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, requant_warp_kernel, kReqWarpsPerCta * 32, 0) !=
            cudaSuccess || per_sm < 1)
      per_sm = 1;
    cached = (unsigned)((sms < 1 ? 1 : sms) * per_sm);
  }
  const int64_t need = (b.total_rows + kReqWarpsPerCta - 1) / kReqWarpsPerCta;
  const unsigned grid = (unsigned)(need < (int64_t)cached ? need : (int64_t)cached);
  requant_warp_kernel<<<grid, kReqWarpsPerCta * 32, 0, stream>>>(b, st);
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

// Non-vector matrices: one warp per row (byte loads).
__global__ void __launch_bounds__(kReqWarps * 32)
requant_generic_kernel(const __grid_constant__ ReqBatch b, int32_t* st) {
  const int lane = threadIdx.x & 31;
  const int64_t grow = (int64_t)blockIdx.x * kReqWarps + (threadIdx.x >> 5);
  if (grow >= b.total_rows) return;
  int lo = 0, hi = b.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (b.m[mid].row0 <= grow) lo = mid; else hi = mid - 1;
  }
  req_row_generic(b.m[lo], grow - b.m[lo].row0, lane, st);
}

cudaError_t requant_batch(const ReqBatch& b, int32_t* st, cudaStream_t stream) {
  if (b.total_rows == 0) return cudaSuccess;
  // one launch per path: rows of vector matrices and rows of the others come in separate
  // row ranges of the two descriptor tables
  ReqBatch vb, gb;
  vb.count = gb.count = 0;
  vb.pad = gb.pad = 0;
  vb.total_rows = gb.total_rows = 0;
  for (int k = 0; k < b.count; ++k) {
    ReqBatch& t = b.m[k].vec ? vb : gb;
    t.m[t.count] = b.m[k];
    t.m[t.count].row0 = t.total_rows;
    t.total_rows += b.m[k].N;
    ++t.count;
  }
  if (vb.total_rows > 0) {
    launch_requant_warps(vb, st, stream);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (gb.total_rows > 0) {
    const int64_t blocks = (gb.total_rows + kReqWarps - 1) / kReqWarps;
    requant_generic_kernel<<<(unsigned)blocks, kReqWarps * 32, 0, stream>>>(gb, st);
  }
  return cudaGetLastError();
}

bool requant_vec_ok(const uint8_t* w, const int8_t* q, int64_t K) {
  return (K % 16 == 0) &&
         ((reinterpret_cast<uintptr_t>(w) & 15) == 0) && ((reinterpret_cast<uintptr_t>(q) & 15) == 0);
}

}  // namespace w8a8
