// Row-wise quantizers: activations (dynamic/static, symmetric/asymmetric), per-channel
// weights (+ azp_adj column sums), the MoE gather-quantizer, the SiLU*up glue quantizer
// and the MoE combine.
//
// Layout: one CTA per row.  A row is read once with 16-byte loads and kept in registers
// (up to 8 x 16 B per thread), reduced (absmax or min/max) with warp shuffles plus one
// shared-memory step, and quantized from registers, so each element crosses HBM once in
// each direction (2 B read + 1 B written).  Rows too long for the register cache, or not
// 16-byte aligned, take a two-pass loop that re-reads the row (from L2).
//
// The rounding rule is the per-row rule of "MiniMax-M2.7 FP8 转昆仑芯 INT8" (转换关系):
// s = absmax/127, q = clamp(round(x/s), -127, 127), zero row -> q = 0, s = 1; with
// IEEE float32 division and ties-to-even rounding.
#include "common.cuh"
#include "internal.h"

namespace w8a8 {


struct RowStats {
  float a, b;  // sym: a = absmax; asym: a = min, b = max
};

template <int THREADS>
__device__ __forceinline__ float block_reduce_max(float v, float* sh) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = sh[0];
#pragma unroll
  for (int i = 1; i < THREADS / 32; ++i) v = fmaxf(v, sh[i]);
  return v;
}

template <int THREADS>
__device__ __forceinline__ float block_reduce_min(float v, float* sh) {
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = sh[0];
#pragma unroll
  for (int i = 1; i < THREADS / 32; ++i) v = fminf(v, sh[i]);
  return v;
}

template <int THREADS>
__device__ __forceinline__ int block_reduce_sum_i(int v, int* sh) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = 0;
#pragma unroll
  for (int i = 0; i < THREADS / 32; ++i) v += sh[i];
  return v;
}

// Scale and zero point of one row from its statistics.  Returns kind: 0 = symmetric
// rule with scale s, 1 = affine rule with (s, zp).
__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// ---------------------------------------------------------------------------
// Vector path: K % 8 == 0, ldx % 8 == 0, 16-byte aligned rows, K <= 8*NV*THREADS.
// MODE: w8a8_act_mode.  row_index: optional gather (MoE), sum_out: optional per-row sum
// of q (weight azp_adj).
// ---------------------------------------------------------------------------
// Scatter of the output rows (MoE): input row t is written to output rows
// row_of[t * topk + j], j < topk, of the out_rows rows of the output.
struct RowScatter {
  const int64_t* row_of;
  int topk;
  int64_t out_rows;
};

template <int MODE, int THREADS, int NV, bool F16, bool SUM, bool SC = false>
__global__ void __launch_bounds__(THREADS, THREADS >= 512 ? 2 : 0)
quant_rows_vec(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t K, int64_t ldx,
               const int64_t* __restrict__ row_index, int8_t* __restrict__ q, __half* __restrict__ q16,
               float* __restrict__ scale, int32_t* __restrict__ zp, int32_t* __restrict__ sum_out,
               int32_t* __restrict__ norm_out, const RowScatter sc) {
  constexpr int W = THREADS / 32;
  constexpr bool DYN = (MODE == W8A8_ACT_DYN_TOKEN_SYM || MODE == W8A8_ACT_DYN_TOKEN_ASYM);
  // row sums of squares of the codes (the GEMM's Cauchy-Schwarz test) with every packed output
  constexpr bool SQ = F16;
  // One CTA barrier per row: per-warp partials go to a double-buffered shared array, so a
  // warp may start writing row k+1's partials while slower warps still read row k's; the
  // row sums of row k (SUM / F16) are completed behind row k+1's barrier.
  __shared__ float sh_lo[2][W], sh_hi[2][W];
  __shared__ int sh_sum[2][W], sh_abs[2][W], sh_sq[2][W];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = (int)(K / 8);
  // Persistent: this CTA quantizes rows blockIdx.x, + gridDim.x, ...; the next row's loads
  // are issued before the current row is processed so that HBM traffic overlaps the math.
  uint4 nxt[NV];
  int64_t row = blockIdx.x, prev = -1;
  int buf = 0;
  auto load_row = [&](int64_t r, uint4 (&dst)[NV]) {
    const int64_t src = row_index ? row_index[r] : r;
    const uint4* xr = reinterpret_cast<const uint4*>(x + src * ldx);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = threadIdx.x + i * THREADS;
      if (idx < nvec && W8A8_DOK(r < rows && src >= 0, 101)) dst[i] = ldg_stream(xr + idx);
    }
  };
  auto finish_sums = [&](int b, int64_t r) {
    int s = 0, a = 0, q2 = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      if (SUM) s += sh_sum[b][i];
      if (F16) a += sh_abs[b][i];
      if (SQ) q2 += sh_sq[b][i];
    }
    if (!W8A8_DOK(r < rows, 104)) return;
    if constexpr (SC) {
      for (int j = 0; j < sc.topk; ++j) {
        const int64_t d = sc.row_of[r * sc.topk + j];
        if (W8A8_DOK(d >= 0 && d < sc.out_rows, 107)) {
          norm_out[d] = a;                  // L1 norm of the codes
          norm_out[sc.out_rows + d] = q2;   // sum of their squares
        }
      }
      return;
    }
    if (SUM) sum_out[r] = s;
    if (F16) norm_out[r] = a;         // L1 norm of the codes
    if (SQ) norm_out[rows + r] = q2;  // sum of their squares, right after the rows' L1 norms
  };
  if (row < rows) load_row(row, nxt);
  for (; row < rows; row += gridDim.x, buf ^= 1) {
    uint4 v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = nxt[i];
    if (row + gridDim.x < rows) load_row(row + gridDim.x, nxt);
    // row statistics on packed bf16 pairs (max/min are exact): |x| max for the symmetric
    // rule, min and max for the affine rule
    if (DYN) {
      __nv_bfloat162 m0 = __floats2bfloat162_rn(MODE == W8A8_ACT_DYN_TOKEN_ASYM ? __int_as_float(0x7f800000) : 0.f,
                                                MODE == W8A8_ACT_DYN_TOKEN_ASYM ? __int_as_float(0x7f800000) : 0.f);
      __nv_bfloat162 m1 = __floats2bfloat162_rn(__int_as_float(0xff800000), __int_as_float(0xff800000));
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int idx = threadIdx.x + i * THREADS;
        if (idx < nvec) {
          const uint32_t wd[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (MODE == W8A8_ACT_DYN_TOKEN_SYM) {
              const uint32_t a = wd[j] & 0x7FFF7FFFu;
              m0 = __hmax2(m0, *reinterpret_cast<const __nv_bfloat162*>(&a));
            } else {
              m0 = __hmin2(m0, *reinterpret_cast<const __nv_bfloat162*>(&wd[j]));
              m1 = __hmax2(m1, *reinterpret_cast<const __nv_bfloat162*>(&wd[j]));
            }
          }
        }
      }
      float lo = MODE == W8A8_ACT_DYN_TOKEN_SYM ? fmaxf(__low2float(m0), __high2float(m0))
                                                : fminf(__low2float(m0), __high2float(m0));
      float hi = fmaxf(__low2float(m1), __high2float(m1));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        if (MODE == W8A8_ACT_DYN_TOKEN_SYM) {
          lo = fmaxf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        } else {
          lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
          hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
      }
      if (lane == 0) {
        sh_lo[buf][warp] = lo;
        sh_hi[buf][warp] = hi;
      }
    }
    __syncthreads();
    if ((SUM || F16) && threadIdx.x == 0 && prev >= 0) finish_sums(buf ^ 1, prev);
    RowQuant rq;
    float rq_lo = 0.f, rq_hi = 0.f;
    if (MODE == W8A8_ACT_DYN_TOKEN_SYM) {
      float a = sh_lo[buf][0];
#pragma unroll
      for (int i = 1; i < W; ++i) a = fmaxf(a, sh_lo[buf][i]);
      rq = row_quant_sym(a);
    } else if (MODE == W8A8_ACT_DYN_TOKEN_ASYM) {
      rq_lo = sh_lo[buf][0];
      rq_hi = sh_hi[buf][0];
#pragma unroll
      for (int i = 1; i < W; ++i) {
        rq_lo = fminf(rq_lo, sh_lo[buf][i]);
        rq_hi = fmaxf(rq_hi, sh_hi[buf][i]);
      }
      rq = row_quant_asym(rq_lo, rq_hi);
    } else {
      rq.s = scale[0];
      rq.zp = (MODE == W8A8_ACT_STATIC_TENSOR_ASYM) ? zp[0] : 0;
      rq.affine = (MODE == W8A8_ACT_STATIC_TENSOR_ASYM);
    }
    const float r = __frcp_rn(rq.s);
    const int qlo = rq.affine ? -128 : -127;
    // dynamic affine rows: the margin of the packed fast path grows with max|x / s| (t = x * r
    // is within 3 * 2^-24 * |x / s| of the IEEE quotient; 2^-21 leaves room for tmax's own
    // rounding).  For bf16 rows |x / s| < 2^17; beyond 2^20 thr <= 0 and every value divides.
    float thr = 0.f;
    if (MODE == W8A8_ACT_DYN_TOKEN_ASYM) {
      const float tmax = __fmul_rn(fmaxf(fabsf(rq_lo), fabsf(rq_hi)), r);
      thr = __fsub_rd(0.5f, __fmul_rn(tmax, 0x1p-21f));
    }
    int qsum = 0, qabs = 0, qsq = 0;
    uint32_t near = 0;  // affine rule: values (bit 8*i + j) left to the exact decision
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = threadIdx.x + i * THREADS;
      if (idx < nvec) {
        float f[8];
        unpack8(v[i], f);
        uint32_t w0, w1;
        if (MODE == W8A8_ACT_DYN_TOKEN_SYM) {
          // |x| <= absmax: codes never exceed +-127
          uint32_t b[8];
          quant_row_group_x2<8>(f, rq.s, r, b);
          w0 = pack4_i8_prmt(b[0], b[1], b[2], b[3]);
          w1 = pack4_i8_prmt(b[4], b[5], b[6], b[7]);
        } else if (MODE == W8A8_ACT_DYN_TOKEN_ASYM) {
          // |x / s| <= 127 in a degenerate (symmetric-rule) row, so the [-128, 127] saturation
          // of the packing never differs from the symmetric clamp there.  Values near a
          // half-integer keep the fast path's code here and are corrected after the loop, which
          // keeps this loop free of branches.
          int c[8];
          near |= affine_codes_fast<8>(f, rq.s, r, rq.zp, thr, c) << (8 * i);
          w0 = pack4_i8_sat(c[0], c[1], c[2], c[3]);
          w1 = pack4_i8_sat(c[4], c[5], c[6], c[7]);
        } else {
          int c[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            int n = rint_div_i(f[j], rq.s, r);
            if (rq.affine) n += rq.zp;
            c[j] = min(127, max(qlo, n));
          }
          w0 = pack4_i8_prmt(c[0], c[1], c[2], c[3]);
          w1 = pack4_i8_prmt(c[4], c[5], c[6], c[7]);
        }
        if (SUM) qsum = sum4_i8(w1, sum4_i8(w0, qsum));
        if (F16) qabs = abssum4_i8(w1, abssum4_i8(w0, qabs));
        if (SQ) qsq = __dp4a((int)w1, (int)w1, __dp4a((int)w0, (int)w0, qsq));
        if (F16) {
          uint4 o;
          i8x4_to_f16x4(w0, o.x, o.y);
          i8x4_to_f16x4(w1, o.z, o.w);
          if constexpr (SC) {
            for (int j = 0; j < sc.topk; ++j) {
              const int64_t d = __ldg(sc.row_of + row * sc.topk + j);
              if (W8A8_DOK(d >= 0 && d < sc.out_rows && (int64_t)(idx + 1) * 8 <= K, 108))
                reinterpret_cast<uint4*>(q16 + d * K)[idx] = o;
            }
          } else {
            if (W8A8_DOK(row < rows && (int64_t)(idx + 1) * 8 <= K, 102)) reinterpret_cast<uint4*>(q16 + row * K)[idx] = o;
          }
        } else {
          if (W8A8_DOK(row < rows && (int64_t)(idx + 1) * 8 <= K, 102)) reinterpret_cast<uint2*>(q + row * K)[idx] = make_uint2(w0, w1);
        }
      }
    }
    if (MODE == W8A8_ACT_DYN_TOKEN_ASYM) {
      // the flagged values (a few per thousand): exact code, stored over the fast path's, and
      // the row sums moved by the difference
      while (near) {
        const int b = __ffs(near) - 1;
        near &= near - 1;
        const int i = b >> 3, j = b & 7;
        uint4 vs = v[0];
#pragma unroll
        for (int ii = 1; ii < NV; ++ii) vs = (i == ii) ? v[ii] : vs;
        const uint32_t wd = (j < 4) ? ((j < 2) ? vs.x : vs.y) : ((j < 6) ? vs.z : vs.w);
        const float xj = (j & 1) ? bf16_hi(wd) : bf16_lo(wd);
        const int c0 = affine_code_fast_one(xj, rq.s, r, rq.zp, thr);
        const int c1 = affine_code_exact(xj, rq.s, r, rq.zp, thr);
        const int64_t col = (int64_t)(threadIdx.x + i * THREADS) * 8 + j;
        if (F16) {
          if (W8A8_DOK(row < rows && col < K, 106)) q16[row * K + col] = __int2half_rn(c1);
        } else {
          if (W8A8_DOK(row < rows && col < K, 106)) q[row * K + col] = (int8_t)c1;
        }
        if (SUM) qsum += c1 - c0;
        if (F16) qabs += abs(c1) - abs(c0);
        if (SQ) qsq += c1 * c1 - c0 * c0;
      }
    }
    if constexpr (SC) {
      if (threadIdx.x < sc.topk) {
        const int64_t d = sc.row_of[row * sc.topk + threadIdx.x];
        if (W8A8_DOK(row < rows && d >= 0 && d < sc.out_rows, 109)) scale[d] = rq.s;
      }
    } else if (threadIdx.x == 0 && W8A8_DOK(row < rows, 103)) {
      if (DYN) scale[row] = rq.s;
      if (MODE == W8A8_ACT_DYN_TOKEN_ASYM) zp[row] = rq.zp;
    }
    if (SUM || F16) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        if (SUM) qsum += __shfl_xor_sync(0xffffffffu, qsum, o);
        if (F16) qabs += __shfl_xor_sync(0xffffffffu, qabs, o);
        if (SQ) qsq += __shfl_xor_sync(0xffffffffu, qsq, o);
      }
      if (lane == 0) {
        sh_sum[buf][warp] = qsum;
        sh_abs[buf][warp] = qabs;
        if (SQ) sh_sq[buf][warp] = qsq;
      }
      prev = row;
    }
  }
  if (SUM || F16) {
    __syncthreads();
    if (threadIdx.x == 0 && prev >= 0) finish_sums(buf ^ 1, prev);
  }
}

// Persistent grid for a row kernel: enough CTAs to fill every SM once, never more than rows.
template <typename Kern>
static unsigned persistent_grid(Kern kern, int threads, int64_t rows) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  if (sms < 1) sms = 1;
  const int64_t g = (int64_t)sms * per_sm;
  return (unsigned)(rows < g ? rows : g);
}

// ---------------------------------------------------------------------------
// Generic path: any K, any alignment.  Two passes over the row.
// ---------------------------------------------------------------------------
template <int MODE, int THREADS>
__global__ void __launch_bounds__(THREADS)
quant_rows_generic(const __nv_bfloat16* __restrict__ x, int64_t K, int64_t ldx,
                   const int64_t* __restrict__ row_index, int8_t* __restrict__ q, __half* __restrict__ q16,
                   float* __restrict__ scale, int32_t* __restrict__ zp,
                   int32_t* __restrict__ sum_out, int32_t* __restrict__ norm_out) {
  __shared__ float sh[THREADS / 32];
  __shared__ int shi[THREADS / 32];
  const int64_t row = blockIdx.x;
  const int64_t src = row_index ? row_index[row] : row;
  const __nv_bfloat16* xr = x + src * ldx;
  RowQuant rq;
  if (MODE == W8A8_ACT_DYN_TOKEN_SYM) {
    float a = 0.f;
    for (int64_t k = threadIdx.x; k < K; k += THREADS) a = fmaxf(a, fabsf(__bfloat162float(xr[k])));
    rq = row_quant_sym(block_reduce_max<THREADS>(a, sh));
  } else if (MODE == W8A8_ACT_DYN_TOKEN_ASYM) {
    float lo = __int_as_float(0x7f800000), hi = __int_as_float(0xff800000);
    for (int64_t k = threadIdx.x; k < K; k += THREADS) {
      const float f = __bfloat162float(xr[k]);
      lo = fminf(lo, f);
      hi = fmaxf(hi, f);
    }
    lo = block_reduce_min<THREADS>(lo, sh);
    hi = block_reduce_max<THREADS>(hi, sh);
    rq = row_quant_asym(lo, hi);
  } else {
    rq.s = scale[0];
    rq.zp = (MODE == W8A8_ACT_STATIC_TENSOR_ASYM) ? zp[0] : 0;
    rq.affine = (MODE == W8A8_ACT_STATIC_TENSOR_ASYM);
  }
  int qsum = 0, qabs = 0, qsq = 0;
  for (int64_t k = threadIdx.x; k < K; k += THREADS) {
    const int c = apply_rq(rq, __bfloat162float(xr[k]));
    if (!W8A8_DOK(src >= 0 && k < K, 105)) continue;
    if (q16) q16[row * K + k] = __int2half_rn(c);
    else q[row * K + k] = (int8_t)c;
    qsum += c;
    qabs += abs(c);
    qsq += c * c;
  }
  if (threadIdx.x == 0) {
    if (MODE == W8A8_ACT_DYN_TOKEN_SYM || MODE == W8A8_ACT_DYN_TOKEN_ASYM) scale[row] = rq.s;
    if (MODE == W8A8_ACT_DYN_TOKEN_ASYM) zp[row] = rq.zp;
  }
  if (sum_out) {
    const int tot = block_reduce_sum_i<THREADS>(qsum, shi);
    if (threadIdx.x == 0) sum_out[row] = tot;
  }
  if (norm_out) {
    const int tot = block_reduce_sum_i<THREADS>(qabs, shi);
    if (threadIdx.x == 0) norm_out[row] = tot;
    const int tot2 = block_reduce_sum_i<THREADS>(qsq, shi);
    if (threadIdx.x == 0) norm_out[gridDim.x + row] = tot2;  // one CTA per row: gridDim.x rows
  }
}

template <int MODE, int THREADS, int NV, bool F16, bool SUM, bool SC = false>
static void launch_vec(const __nv_bfloat16* x, int64_t rows, int64_t K, int64_t ldx, const int64_t* row_index,
                       int8_t* q, __half* q16, float* scale, int32_t* zp, int32_t* sum_out, int32_t* norm_out,
                       cudaStream_t st, const RowScatter& sc = RowScatter{nullptr, 0, 0}) {
  auto kern = quant_rows_vec<MODE, THREADS, NV, F16, SUM, SC>;
  static thread_local unsigned cached = 0;  // per instantiation: CTAs that fill the GPU once
  if (cached == 0) cached = persistent_grid(kern, THREADS, (int64_t)1 << 40);
  const unsigned grid = (unsigned)(rows < (int64_t)cached ? rows : (int64_t)cached);
  kern<<<grid, THREADS, 0, st>>>(x, rows, K, ldx, row_index, q, q16, scale, zp, sum_out, norm_out, sc);
}

template <int MODE, bool F16, bool SUM, bool SC = false>
static void launch_vec_k(const __nv_bfloat16* x, int64_t rows, int64_t K, int64_t ldx, const int64_t* row_index,
                         int8_t* q, __half* q16, float* scale, int32_t* zp, int32_t* sum_out, int32_t* norm_out,
                         cudaStream_t st, const RowScatter& sc = RowScatter{nullptr, 0, 0}) {
  // Rows are latency-bound at these sizes (one CTA-wide reduction per row), so short rows get
  // small CTAs and many rows in flight per SM; about 16-32 values per thread.
  const int64_t nvec = K / 8;
  if (nvec <= 128 * 2)
    launch_vec<MODE, 128, 2, F16, SUM, SC>(x, rows, K, ldx, row_index, q, q16, scale, zp, sum_out, norm_out, st, sc);
  else if (nvec <= 128 * 4)
    launch_vec<MODE, 128, 4, F16, SUM, SC>(x, rows, K, ldx, row_index, q, q16, scale, zp, sum_out, norm_out, st, sc);
  else if (nvec <= 256 * 4)
    launch_vec<MODE, 256, 4, F16, SUM, SC>(x, rows, K, ldx, row_index, q, q16, scale, zp, sum_out, norm_out, st, sc);
  else
    launch_vec<MODE, 512, 4, F16, SUM, SC>(x, rows, K, ldx, row_index, q, q16, scale, zp, sum_out, norm_out, st, sc);
}

template <int MODE>
static cudaError_t launch_quant_rows(const __nv_bfloat16* x, int64_t rows, int64_t K, int64_t ldx,
                                     const int64_t* row_index, int8_t* q, __half* q16, float* scale,
                                     int32_t* zp, int32_t* sum_out, int32_t* norm_out, cudaStream_t st) {
  const bool aligned = (K % 8 == 0) && (ldx % 8 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0) &&
                       (q16 ? ((reinterpret_cast<uintptr_t>(q16) & 15) == 0)
                            : ((reinterpret_cast<uintptr_t>(q) & 7) == 0));
  const int64_t nvec = K / 8;
  if (aligned && nvec <= 512 * 4) {
    if (q16) launch_vec_k<MODE, true, false>(x, rows, K, ldx, row_index, q, q16, scale, zp, sum_out, norm_out, st);
    else if (sum_out) launch_vec_k<MODE, false, true>(x, rows, K, ldx, row_index, q, q16, scale, zp, sum_out, norm_out, st);
    else launch_vec_k<MODE, false, false>(x, rows, K, ldx, row_index, q, q16, scale, zp, sum_out, norm_out, st);
  } else {
    quant_rows_generic<MODE, 256><<<(unsigned)rows, 256, 0, st>>>(x, K, ldx, row_index, q, q16, scale, zp,
                                                                   sum_out, norm_out);
  }
  return cudaGetLastError();
}

cudaError_t quant_rows(int mode, const void* x, int64_t rows, int64_t K, int64_t ldx,
                       const int64_t* row_index, int8_t* q, void* q_f16, float* scale, int32_t* zp,
                       int32_t* sum_out, int32_t* norm_out, cudaStream_t st) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  __half* qh = static_cast<__half*>(q_f16);
  switch (mode) {
    case W8A8_ACT_DYN_TOKEN_SYM:
      return launch_quant_rows<W8A8_ACT_DYN_TOKEN_SYM>(xb, rows, K, ldx, row_index, q, qh, scale, zp, sum_out,
                                                       norm_out, st);
    case W8A8_ACT_DYN_TOKEN_ASYM:
      return launch_quant_rows<W8A8_ACT_DYN_TOKEN_ASYM>(xb, rows, K, ldx, row_index, q, qh, scale, zp, sum_out,
                                                        norm_out, st);
    case W8A8_ACT_STATIC_TENSOR_SYM:
      return launch_quant_rows<W8A8_ACT_STATIC_TENSOR_SYM>(xb, rows, K, ldx, row_index, q, qh, scale, zp,
                                                           sum_out, norm_out, st);
    default:
      return launch_quant_rows<W8A8_ACT_STATIC_TENSOR_ASYM>(xb, rows, K, ldx, row_index, q, qh, scale, zp,
                                                            sum_out, norm_out, st);
  }
}

// MoE: each token row quantized once (dynamic symmetric, packed fp16 codes) and written to
// its topk expert-sorted rows.  K % 8 == 0, 16-byte aligned rows, K <= 16384.
cudaError_t quant_rows_scatter_packed(const void* x, int64_t T, int64_t K, int64_t ldx, const int64_t* row_of,
                                      int topk, int64_t R, void* q_f16, float* scale, int32_t* norm_out,
                                      cudaStream_t st) {
  const RowScatter sc{row_of, topk, R};
  launch_vec_k<W8A8_ACT_DYN_TOKEN_SYM, true, false, true>(static_cast<const __nv_bfloat16*>(x), T, K, ldx, nullptr,
                                                          nullptr, static_cast<__half*>(q_f16), scale, nullptr,
                                                          nullptr, norm_out, st, sc);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// azp_adj[n] = zp * sum_k wq[n, k] for an already-quantized weight.
// ---------------------------------------------------------------------------
// Per-row sums of int8 codes (azp_adj, optionally times a zero point) or of their squares (SQ:
// the weight side of the GEMM's Cauchy-Schwarz exactness bound).
template <int THREADS, bool SQ>
__global__ void __launch_bounds__(THREADS)
row_sum_i8(const int8_t* __restrict__ w, int64_t K, const int32_t* __restrict__ zp,
           int32_t* __restrict__ out) {
  __shared__ int shi[THREADS / 32];
  const int64_t row = blockIdx.x;
  const int8_t* wr = w + row * K;
  int s = 0;
  if ((K % 16 == 0) && ((reinterpret_cast<uintptr_t>(w) & 15) == 0)) {
    const uint4* v = reinterpret_cast<const uint4*>(wr);
    for (int64_t i = threadIdx.x; i < K / 16; i += THREADS) {
      const uint4 u = v[i];
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) s = __dp4a((int)wd[j], SQ ? (int)wd[j] : 0x01010101, s);
    }
  } else {
    for (int64_t k = threadIdx.x; k < K; k += THREADS) s += SQ ? (int)wr[k] * (int)wr[k] : (int)wr[k];
  }
  s = block_reduce_sum_i<THREADS>(s, shi);
  if (threadIdx.x == 0) out[row] = (!SQ && zp) ? s * zp[0] : s;
}

cudaError_t azp_rows(const int8_t* w, int64_t N, int64_t K, const int32_t* zp, int32_t* out,
                     cudaStream_t st) {
  row_sum_i8<256, false><<<(unsigned)N, 256, 0, st>>>(w, K, zp, out);
  return cudaGetLastError();
}

cudaError_t sumsq_rows(const int8_t* w, int64_t N, int64_t K, int32_t* out, cudaStream_t st) {
  row_sum_i8<256, true><<<(unsigned)N, 256, 0, st>>>(w, K, nullptr, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// MoE glue: g = bf16(silu(gate) * up) then per-row symmetric quantization.
// h row = [gate (I) | up (I)], I % 8 == 0.  Persistent like quant_rows_vec: the next row's
// loads are issued before the current row is processed, one CTA barrier per row.  The SiLU
// uses the fast exponential and division (g is compared with the oracle's float64 SiLU within
// the bf16 tolerance); the quantization of g is the exact row rule.
// ---------------------------------------------------------------------------
template <int THREADS, int NV, bool F16>
__global__ void __launch_bounds__(THREADS)
silu_mul_quant_kernel(const __nv_bfloat16* __restrict__ h, int64_t rows, int64_t I, int8_t* __restrict__ gq,
                      __half* __restrict__ g16, int32_t* __restrict__ norm_out, float* __restrict__ sg) {
  constexpr int W = THREADS / 32;
  __shared__ float sh_a[2][W];
  __shared__ int sh_abs[2][W], sh_sq[2][W];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = (int)(I / 8);
  uint4 ng[NV], nu[NV];
  // packed output: row L1 norms [rows] then sums of squares [rows] of the codes
  auto finish = [&](int b, int64_t r) {
    int t = 0, t2 = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      t += sh_abs[b][i];
      t2 += sh_sq[b][i];
    }
    norm_out[r] = t;
    norm_out[rows + r] = t2;
  };
  auto load_row = [&](int64_t r) {
    const uint4* gate = reinterpret_cast<const uint4*>(h + r * 2 * I);
    const uint4* up = reinterpret_cast<const uint4*>(h + r * 2 * I + I);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = threadIdx.x + i * THREADS;
      if (idx < nvec) {
        ng[i] = ldg_stream(gate + idx);
        nu[i] = ldg_stream(up + idx);
      }
    }
  };
  int64_t row = blockIdx.x, prev = -1;
  int buf = 0;
  if (row < rows) load_row(row);
  for (; row < rows; row += gridDim.x, buf ^= 1) {
    float g[NV][8];
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = threadIdx.x + i * THREADS;
      if (idx < nvec) {
        float fa[8], fb[8];
        unpack8(ng[i], fa);
        unpack8(nu[i], fb);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float sl = __fdividef(fa[j], 1.f + __expf(-fa[j]));
          const float v = __bfloat162float(__float2bfloat16_rn(__fmul_rn(sl, fb[j])));
          g[i][j] = v;
          a = fmaxf(a, fabsf(v));
        }
      }
    }
    if (row + gridDim.x < rows) load_row(row + gridDim.x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) sh_a[buf][warp] = a;
    __syncthreads();
    if (F16 && threadIdx.x == 0 && prev >= 0) finish(buf ^ 1, prev);
    a = sh_a[buf][0];
#pragma unroll
    for (int i = 1; i < W; ++i) a = fmaxf(a, sh_a[buf][i]);
    const RowQuant rq = row_quant_sym(a);
    const float rcp = __frcp_rn(rq.s);
    int qabs = 0, qsq = 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int idx = threadIdx.x + i * THREADS;
      if (idx < nvec) {
        uint32_t b[8];
        quant_row_group_x2<8>(g[i], rq.s, rcp, b);  // |g| <= absmax: codes within +-127
        const uint32_t w0 = pack4_i8_prmt(b[0], b[1], b[2], b[3]);
        const uint32_t w1 = pack4_i8_prmt(b[4], b[5], b[6], b[7]);
        if (F16) {
          qabs = abssum4_i8(w1, abssum4_i8(w0, qabs));
          qsq = __dp4a((int)w1, (int)w1, __dp4a((int)w0, (int)w0, qsq));
          uint4 o;
          i8x4_to_f16x4(w0, o.x, o.y);
          i8x4_to_f16x4(w1, o.z, o.w);
          reinterpret_cast<uint4*>(g16 + row * I)[idx] = o;
        } else {
          reinterpret_cast<uint2*>(gq + row * I)[idx] = make_uint2(w0, w1);
        }
      }
    }
    if (threadIdx.x == 0) sg[row] = rq.s;
    if (F16) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        qabs += __shfl_xor_sync(0xffffffffu, qabs, o);
        qsq += __shfl_xor_sync(0xffffffffu, qsq, o);
      }
      if (lane == 0) {
        sh_abs[buf][warp] = qabs;
        sh_sq[buf][warp] = qsq;
      }
      prev = row;
    }
  }
  if (F16) {
    __syncthreads();
    if (threadIdx.x == 0 && prev >= 0) finish(buf ^ 1, prev);
  }
}

template <int THREADS, int NV, bool F16>
static void launch_silu(const __nv_bfloat16* h, int64_t R, int64_t I, int8_t* gq, __half* g16, int32_t* norms,
                        float* sg, cudaStream_t st) {
  auto kern = silu_mul_quant_kernel<THREADS, NV, F16>;
  static thread_local unsigned cached = 0;
  if (cached == 0) cached = persistent_grid(kern, THREADS, (int64_t)1 << 40);
  const unsigned grid = (unsigned)(R < (int64_t)cached ? R : (int64_t)cached);
  kern<<<grid, THREADS, 0, st>>>(h, R, I, gq, g16, norms, sg);
}

template <bool F16>
static cudaError_t launch_silu_k(const __nv_bfloat16* h, int64_t R, int64_t I, int8_t* gq, __half* g16,
                                 int32_t* norms, float* sg, cudaStream_t st) {
  const int64_t nvec = I / 8;
  // rows of up to 192 vectors (I <= 1536) on 64-thread CTAs: more rows in flight per SM
  // (I = 1408: 601.9-603.6 us per MoE layer against 605.6-608.5 with 128 x 2)
  if (nvec <= 64 * 3) launch_silu<64, 3, F16>(h, R, I, gq, g16, norms, sg, st);
  else if (nvec <= 128 * 2) launch_silu<128, 2, F16>(h, R, I, gq, g16, norms, sg, st);
  else if (nvec <= 128 * 4) launch_silu<128, 4, F16>(h, R, I, gq, g16, norms, sg, st);
  else if (nvec <= 256 * 4) launch_silu<256, 4, F16>(h, R, I, gq, g16, norms, sg, st);
  else if (nvec <= 512 * 4) launch_silu<512, 4, F16>(h, R, I, gq, g16, norms, sg, st);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t silu_mul_quant(const void* h, int64_t R, int64_t I, int8_t* gq, void* g16, int32_t* norms, float* sg,
                           cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  const __nv_bfloat16* hb = static_cast<const __nv_bfloat16*>(h);
  __half* gh = static_cast<__half*>(g16);
  return g16 ? launch_silu_k<true>(hb, R, I, gq, gh, norms, sg, st)
             : launch_silu_k<false>(hb, R, I, gq, gh, norms, sg, st);
}

// ---------------------------------------------------------------------------
// MoE combine: y[t] = bf16( sum_j w[t,j] * out[row_of[t,j]] ), slots in order.
// Up to 8 slots: the token's rows and weights are read once and the loads of all its
// routed rows are issued together; more slots take the plain loop.  Both add in slot order.
// ---------------------------------------------------------------------------
constexpr int kCombineSlots = 8;

__global__ void __launch_bounds__(128)
moe_combine_few_kernel(const __nv_bfloat16* __restrict__ out, const int64_t* __restrict__ row_of,
                       const float* __restrict__ tw, int topk, int64_t H, __nv_bfloat16* __restrict__ y) {
  const int64_t t = blockIdx.x;
  const int nvec = (int)(H / 8);
  int64_t rr[kCombineSlots];
  float ww[kCombineSlots];
#pragma unroll
  for (int s = 0; s < kCombineSlots; ++s) {
    rr[s] = s < topk ? row_of[t * topk + s] : 0;
    ww[s] = s < topk ? tw[t * topk + s] : 0.f;
  }
  for (int idx = threadIdx.x; idx < nvec; idx += blockDim.x) {
    uint4 v[kCombineSlots];
#pragma unroll
    for (int s = 0; s < kCombineSlots; ++s)
      if (s < topk) v[s] = reinterpret_cast<const uint4*>(out + rr[s] * H)[idx];
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
    for (int s = 0; s < kCombineSlots; ++s) {
      if (s < topk) {
        float f[8];
        unpack8(v[s], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn(ww[s], f[j]));
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(y + t * H)[idx] = o;
  }
}

__global__ void __launch_bounds__(128)
moe_combine_kernel(const __nv_bfloat16* __restrict__ out, const int64_t* __restrict__ row_of,
                   const float* __restrict__ tw, int topk, int64_t H, __nv_bfloat16* __restrict__ y) {
  const int64_t t = blockIdx.x;
  const int nvec = (int)(H / 8);
  for (int idx = threadIdx.x; idx < nvec; idx += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int s = 0; s < topk; ++s) {
      const int64_t r = row_of[t * topk + s];
      const float w = tw[t * topk + s];
      float f[8];
      unpack8(reinterpret_cast<const uint4*>(out + r * H)[idx], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn(w, f[j]));
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(y + t * H)[idx] = o;
  }
}

cudaError_t moe_combine(const void* out, const int64_t* row_of, const float* tw, int64_t T, int topk,
                        int64_t H, void* y, cudaStream_t st) {
  if (topk <= kCombineSlots)
    moe_combine_few_kernel<<<(unsigned)T, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(out), row_of, tw, topk, H,
                                                        static_cast<__nv_bfloat16*>(y));
  else
    moe_combine_kernel<<<(unsigned)T, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(out), row_of, tw, topk, H,
                                                    static_cast<__nv_bfloat16*>(y));
  return cudaGetLastError();
}

#ifdef W8A8_DEBUG
cudaError_t debug_register_quant(int32_t* word) { return w8a8_debug_register_here(word); }
#endif

}  // namespace w8a8
