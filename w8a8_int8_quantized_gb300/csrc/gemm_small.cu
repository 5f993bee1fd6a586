// Weight-streaming INT8 GEMM for few activation rows (decode-sized M).
//
// With M <= 16 the layer is bound by reading the int8 weight once from HBM (2*M ops per
// weight byte), so the kernels are shaped for bandwidth, not for tensor-core peak.  Blocks
// of 16 output channels; 8 warps split K into interleaved 64-byte chunks so that
// neighbouring warps read neighbouring bytes of a weight row; the integer products run on
// the exact s8 x s8 -> s32 warp MMA (m16n8k32), with the weight as the 16-row operand and
// the tokens as the 8-column operand; the partial sums of the 8 warps are added in shared
// memory and the scale/azp/bias epilogue is applied before one bf16 store.  Three forms:
//   gemm_small_m_kernel     one block of 16 channels x 16 token rows per CTA, four chunks of
//                           16-byte loads in flight per thread (9-16 rows, grouped segments,
//                           rows too long to stage);
//   gemm_small_m_xs_kernel  at most 8 rows staged in shared memory once per persistent CTA,
//                           eight chunks in flight per thread;
//   gemm_small_m_fq_kernel  one dynamic bf16 row quantized inside the CTA (the stand-alone
//                           quantizer's exact rules) before the same streaming;
//   gemv_kernel             one or two token rows (given codes, or one dynamic bf16 row)
//                           on dp4a instead of the warp MMA, which would be mostly padding
//                           (below).
//
// K order inside a 64-byte chunk: each thread loads 16 contiguous bytes of a row and
// feeds them to the MMA as its k-slots; A and B use the same mapping, so the sum over k
// is unchanged.
#include "common.cuh"
#include "internal.h"

namespace w8a8 {

constexpr int kSmWarps = 8;
constexpr int kSmUnroll = 4;

__device__ __forceinline__ void mma_s8_16832(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ld16_or_zero(const int8_t* p, bool ok) {
  uint4 v = make_uint4(0, 0, 0, 0);
  if (ok) v = __ldg(reinterpret_cast<const uint4*>(p));
  return v;
}

__device__ __forceinline__ uint4 ld16_stream_or_zero(const int8_t* p, bool ok) {
  uint4 v = make_uint4(0, 0, 0, 0);
  if (ok)
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kSmWarps * 32)
gemm_small_m_kernel(const int8_t* __restrict__ xq, const int8_t* __restrict__ wq, int64_t rows,
                    int64_t N, int64_t K, int E, const int64_t* __restrict__ seg, EpiParams ep,
                    __nv_bfloat16* __restrict__ y) {
  __shared__ int red[kSmWarps][16][17];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t n0 = (int64_t)blockIdx.x * 16;

  // which segment / row block this CTA owns
  int e = 0;
  int64_t m0 = (int64_t)blockIdx.y * 16, mend = rows;
  if (seg) {
    int64_t tb = blockIdx.y, acc_tiles = 0;
    bool found = false;
    for (int s = 0; s < E; ++s) {
      const int64_t lo = seg[s], hi = seg[s + 1];
      const int64_t nt = (hi - lo + 15) / 16;
      if (tb < acc_tiles + nt) {
        e = s;
        m0 = lo + (tb - acc_tiles) * 16;
        mend = hi;
        found = true;
        break;
      }
      acc_tiles += nt;
    }
    if (!found) return;
  }
  const int8_t* wbase = wq + (int64_t)e * N * K;

  const bool wr0 = (n0 + g) < N, wr1 = (n0 + g + 8) < N;
  const bool xr0 = (m0 + g) < mend, xr1 = (m0 + g + 8) < mend;
  const int8_t* pw0 = wbase + (n0 + g) * K;
  const int8_t* pw1 = wbase + (n0 + g + 8) * K;
  const int8_t* px0 = xq + (m0 + g) * K;
  const int8_t* px1 = xq + (m0 + g + 8) * K;

  int acc0[4] = {0, 0, 0, 0}, acc1[4] = {0, 0, 0, 0};
  const bool two = (m0 + 8) < mend;  // second group of 8 token rows present (CTA-uniform)
  const int64_t nchunks = (K + 63) / 64;
  for (int64_t c0 = warp; c0 < nchunks; c0 += (int64_t)kSmWarps * kSmUnroll) {
    uint4 wa[kSmUnroll][2], xb[kSmUnroll][2];
#pragma unroll
    for (int u = 0; u < kSmUnroll; ++u) {
      const int64_t c = c0 + (int64_t)u * kSmWarps;
      const int64_t kb = c * 64 + tq * 16;
      const bool kin = (c < nchunks) && (kb < K);
      wa[u][0] = ld16_stream_or_zero(pw0 + kb, kin && wr0);
      wa[u][1] = ld16_stream_or_zero(pw1 + kb, kin && wr1);
      xb[u][0] = ld16_or_zero(px0 + kb, kin && xr0);
      xb[u][1] = ld16_or_zero(px1 + kb, kin && xr1 && two);
    }
#pragma unroll
    for (int u = 0; u < kSmUnroll; ++u) {
      const uint32_t A0[4] = {wa[u][0].x, wa[u][0].y, wa[u][0].z, wa[u][0].w};
      const uint32_t A1[4] = {wa[u][1].x, wa[u][1].y, wa[u][1].z, wa[u][1].w};
      const uint32_t B0[4] = {xb[u][0].x, xb[u][0].y, xb[u][0].z, xb[u][0].w};
      const uint32_t B1[4] = {xb[u][1].x, xb[u][1].y, xb[u][1].z, xb[u][1].w};
#pragma unroll
      for (int j = 0; j < 2; ++j)
        mma_s8_16832(acc0, A0[2 * j], A1[2 * j], A0[2 * j + 1], A1[2 * j + 1], B0[2 * j], B0[2 * j + 1]);
      if (two) {  // blocks of at most 8 token rows (decode) skip the all-zero second group
#pragma unroll
        for (int j = 0; j < 2; ++j)
          mma_s8_16832(acc1, A0[2 * j], A1[2 * j], A0[2 * j + 1], A1[2 * j + 1], B1[2 * j], B1[2 * j + 1]);
      }
    }
  }
  // D fragment: (row g / g+8 = channel, col 2tq / 2tq+1 = token)
  red[warp][g][2 * tq] = acc0[0];
  red[warp][g][2 * tq + 1] = acc0[1];
  red[warp][g + 8][2 * tq] = acc0[2];
  red[warp][g + 8][2 * tq + 1] = acc0[3];
  red[warp][g][8 + 2 * tq] = acc1[0];
  red[warp][g][8 + 2 * tq + 1] = acc1[1];
  red[warp][g + 8][8 + 2 * tq] = acc1[2];
  red[warp][g + 8][8 + 2 * tq + 1] = acc1[3];
  __syncthreads();
  const int tok = threadIdx.x >> 4, ch = threadIdx.x & 15;
  const int64_t m = m0 + tok, n = n0 + ch;
  if (m < mend && n < N) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < kSmWarps; ++w) s += red[w][ch][tok];
    EpiParams p = ep;
    if (p.w_mode == W8A8_W_CHANNEL) p.s_w = ep.s_w + (int64_t)e * N;
    const float v = epi_apply(p, s, epi_row_scale(p, m), epi_row_zp(p, m), n);
    if (W8A8_DOK(m < rows && e < E, 401)) y[m * N + n] = __float2bfloat16_rn(v);
  }
}

// Dense launches of at most 8 token rows whose rows fit in shared memory (<= 96 KB): a
// persistent CTA stages the rows once and then walks 16-channel blocks, issuing all its weight
// loads for kXsUnroll chunks per warp before the first MMA, so a K = 4096 block needs one
// dependent round trip to HBM; two CTAs per SM overlap one's loads with the other's reduction
// and epilogue.  Warp w only ever reads the 64-byte K-chunks c = w (mod kSmWarps), so it stages
// exactly those with asynchronous copies, issued before its first weight loads and waited for
// (this warp's copies only, then a warp barrier) just before its first shared-memory read.  The
// staged row stride is 64 mod 128 bytes: the two rows one quarter-warp reads, 64 bytes each,
// cover all 32 banks once.
constexpr int kXsUnroll = 8;
__host__ __device__ inline int64_t xs_stride(int64_t K) { return (K + 127) / 128 * 128 + 64; }

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}

__global__ void __launch_bounds__(kSmWarps * 32)
gemm_small_m_xs_kernel(const int8_t* __restrict__ xq, const int8_t* __restrict__ wq, int64_t rows, int64_t N,
                       int64_t K, EpiParams ep, __nv_bfloat16* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t xs[];
  __shared__ int red[kSmWarps][16][17];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int nr = (int)rows;  // <= 8 (the second token group serves the 9-16 row callers of this form)
  const int64_t ld = xs_stride(K);
  const int64_t nchunks = (K + 63) / 64;
  {
    const int64_t mine = nchunks > warp ? (nchunks - warp + kSmWarps - 1) / kSmWarps : 0;
    const int64_t pieces = (int64_t)nr * mine * 4;
    for (int64_t i = lane; i < pieces; i += 32) {
      const int64_t r = i / (mine * 4), rem = i % (mine * 4);
      const int64_t kb = (warp + (rem >> 2) * kSmWarps) * 64 + (rem & 3) * 16;
      if (kb < K) cp_async16(xs + r * ld + kb, xq + r * K + kb);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  }
  bool staged = false;
  const bool xr0 = g < nr, xr1 = (g + 8) < nr;
  const bool two = nr > 8;
  const uint8_t* sx0 = xs + g * ld;
  const uint8_t* sx1 = xs + (g + 8) * ld;
  const int64_t nbn = (N + 15) / 16;
  for (int64_t nb = blockIdx.x; nb < nbn; nb += gridDim.x) {
    const int64_t n0 = nb * 16;
    const bool wr0 = (n0 + g) < N, wr1 = (n0 + g + 8) < N;
    const int8_t* pw0 = wq + (n0 + g) * K;
    const int8_t* pw1 = wq + (n0 + g + 8) * K;
    int acc0[2][4] = {}, acc1[2][4] = {};  // split by k-half: shorter dependent MMA chains
    for (int64_t c0 = warp; c0 < nchunks; c0 += (int64_t)kSmWarps * kXsUnroll) {
      uint4 wa[kXsUnroll][2];
#pragma unroll
      for (int u = 0; u < kXsUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kSmWarps;
        const int64_t kb = c * 64 + tq * 16;
        const bool kin = (c < nchunks) && (kb < K);
        wa[u][0] = ld16_stream_or_zero(pw0 + kb, kin && wr0);
        wa[u][1] = ld16_stream_or_zero(pw1 + kb, kin && wr1);
      }
      if (!staged) {  // warp-uniform
        asm volatile("cp.async.wait_all;\n" ::: "memory");
        __syncwarp();
        staged = true;
      }
#pragma unroll
      for (int u = 0; u < kXsUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kSmWarps;
        const int64_t kb = c * 64 + tq * 16;
        const bool kin = (c < nchunks) && (kb < K);
        const uint4 x0 = (kin && xr0) ? *reinterpret_cast<const uint4*>(sx0 + kb) : make_uint4(0, 0, 0, 0);
        const uint32_t A0[4] = {wa[u][0].x, wa[u][0].y, wa[u][0].z, wa[u][0].w};
        const uint32_t A1[4] = {wa[u][1].x, wa[u][1].y, wa[u][1].z, wa[u][1].w};
        const uint32_t B0[4] = {x0.x, x0.y, x0.z, x0.w};
#pragma unroll
        for (int j = 0; j < 2; ++j)
          mma_s8_16832(acc0[j], A0[2 * j], A1[2 * j], A0[2 * j + 1], A1[2 * j + 1], B0[2 * j], B0[2 * j + 1]);
        if (two) {
          const uint4 x1 = (kin && xr1) ? *reinterpret_cast<const uint4*>(sx1 + kb) : make_uint4(0, 0, 0, 0);
          const uint32_t B1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int j = 0; j < 2; ++j)
            mma_s8_16832(acc1[j], A0[2 * j], A1[2 * j], A0[2 * j + 1], A1[2 * j + 1], B1[2 * j], B1[2 * j + 1]);
        }
      }
    }
    // D fragment: (row g / g+8 = channel, col 2tq / 2tq+1 = token)
    red[warp][g][2 * tq] = acc0[0][0] + acc0[1][0];
    red[warp][g][2 * tq + 1] = acc0[0][1] + acc0[1][1];
    red[warp][g + 8][2 * tq] = acc0[0][2] + acc0[1][2];
    red[warp][g + 8][2 * tq + 1] = acc0[0][3] + acc0[1][3];
    red[warp][g][8 + 2 * tq] = acc1[0][0] + acc1[1][0];
    red[warp][g][8 + 2 * tq + 1] = acc1[0][1] + acc1[1][1];
    red[warp][g + 8][8 + 2 * tq] = acc1[0][2] + acc1[1][2];
    red[warp][g + 8][8 + 2 * tq + 1] = acc1[0][3] + acc1[1][3];
    __syncthreads();
    const int tok = threadIdx.x >> 4, ch = threadIdx.x & 15;
    const int64_t n = n0 + ch;
    if (tok < nr && n < N) {
      int sum = 0;
#pragma unroll
      for (int w = 0; w < kSmWarps; ++w) sum += red[w][ch][tok];
      if (W8A8_DOK(tok < rows, 402))
        y[tok * N + n] = __float2bfloat16_rn(epi_apply(ep, sum, epi_row_scale(ep, tok), epi_row_zp(ep, tok), n));
    }
    __syncthreads();  // red is rewritten by the next block
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");  // warps that read no chunk still own copies
}

// Decode launches of dynamic per-token symmetric activations with the quantizer fused in
// (at most 8 bf16 token rows whose codes fit the 96 KB shared-memory copy): every CTA
// quantizes the rows itself, straight into its shared-memory copy, with the stand-alone
// quantizer's exact row rule (s = RN(absmax / 127), or 1 for a zero row; codes
// rint(RN(x / s)) from the division-free rounding with exact near-tie resolution).  This
// takes the separate quantizer launch and its int8 round trip through memory off a decode
// step.  The first round of weight loads is issued before the quantization so that it
// overlaps the row reads.
template <int MODE>
__global__ void __launch_bounds__(kSmWarps * 32)
gemm_small_m_fq_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx, const int8_t* __restrict__ wq,
                       int64_t rows, int64_t N, int64_t K, EpiParams ep, __nv_bfloat16* __restrict__ y) {
  constexpr bool ASYM = MODE == W8A8_ACT_DYN_TOKEN_ASYM;
  extern __shared__ __align__(16) uint8_t xs[];
  __shared__ int red[kSmWarps][16][17];
  __shared__ float sh_amax[kSmWarps][8], sh_hi[kSmWarps][8];
  __shared__ float sh_s[8], sh_r[8], sh_thr[8];
  __shared__ int sh_zp[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int nr = (int)rows;  // <= 8
  const int64_t ld = xs_stride(K);
  const int64_t nchunks = (K + 63) / 64;
  const int64_t nbn = (N + 15) / 16;
  const int nvec = (int)(K / 8);
  auto load_round = [&](int64_t nb, int64_t c0, uint4 (&wa)[kXsUnroll][2]) {
    const int64_t n0 = nb * 16;
    const bool wr0 = (n0 + g) < N, wr1 = (n0 + g + 8) < N;
    const int8_t* pw0 = wq + (n0 + g) * K;
    const int8_t* pw1 = wq + (n0 + g + 8) * K;
#pragma unroll
    for (int u = 0; u < kXsUnroll; ++u) {
      const int64_t c = c0 + (int64_t)u * kSmWarps;
      const int64_t kb = c * 64 + tq * 16;
      const bool kin = (c < nchunks) && (kb < K);
      wa[u][0] = ld16_stream_or_zero(pw0 + kb, kin && wr0);
      wa[u][1] = ld16_stream_or_zero(pw1 + kb, kin && wr1);
    }
  };
  uint4 wa[kXsUnroll][2];
  bool preloaded = false;
  if ((int64_t)blockIdx.x < nbn) {
    load_round(blockIdx.x, warp, wa);
    preloaded = true;
  }
  // row statistics (exact: max / min of exact values), one CTA reduction for all rows:
  // absmax for the symmetric rule, min and max for the affine one
  float am[8], ah[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    am[r] = ASYM ? __int_as_float(0x7f800000) : 0.f;
    ah[r] = __int_as_float(0xff800000);
    if (r < nr) {
      const uint4* xr = reinterpret_cast<const uint4*>(x + r * ldx);
      for (int c = threadIdx.x; c < nvec; c += kSmWarps * 32) {
        const uint4 v = __ldg(xr + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (ASYM) {
            am[r] = fminf(am[r], fminf(bf16_lo(w[k]), bf16_hi(w[k])));
            ah[r] = fmaxf(ah[r], fmaxf(bf16_lo(w[k]), bf16_hi(w[k])));
          } else {
            am[r] = fmaxf(am[r], fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      if (ASYM) {
        am[r] = fminf(am[r], __shfl_xor_sync(0xffffffffu, am[r], o));
        ah[r] = fmaxf(ah[r], __shfl_xor_sync(0xffffffffu, ah[r], o));
      } else {
        am[r] = fmaxf(am[r], __shfl_xor_sync(0xffffffffu, am[r], o));
      }
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      sh_amax[warp][r] = am[r];
      if (ASYM) sh_hi[warp][r] = ah[r];
    }
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    RowQuant rq;
    float lo = 0.f, hi = 0.f;
    if (ASYM) {
      lo = sh_amax[0][threadIdx.x];
      hi = sh_hi[0][threadIdx.x];
#pragma unroll
      for (int w = 1; w < kSmWarps; ++w) {
        lo = fminf(lo, sh_amax[w][threadIdx.x]);
        hi = fmaxf(hi, sh_hi[w][threadIdx.x]);
      }
      rq = row_quant_asym(lo, hi);
    } else {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kSmWarps; ++w) a = fmaxf(a, sh_amax[w][threadIdx.x]);
      rq = row_quant_sym(a);
    }
    const float rc = __frcp_rn(rq.s);
    sh_s[threadIdx.x] = rq.s;
    sh_r[threadIdx.x] = rc;
    sh_zp[threadIdx.x] = rq.zp;
    // the stand-alone affine quantizer's margin of its division-free fast path
    sh_thr[threadIdx.x] = ASYM ? __fsub_rd(0.5f, __fmul_rn(__fmul_rn(fmaxf(fabsf(lo), fabsf(hi)), rc), 0x1p-21f)) : 0.f;
  }
  __syncthreads();
  // codes into the shared-memory copy, by the stand-alone quantizer's rules (symmetric:
  // |x| <= absmax, every code within +-127; affine: zero point folded into the rounding,
  // saturated to [-128, 127])
  for (int r = 0; r < nr; ++r) {
    const float sc = sh_s[r], rc = sh_r[r];
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * ldx);
    for (int c = threadIdx.x; c < nvec; c += kSmWarps * 32) {
      const uint4 v = __ldg(xr + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float f[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        f[2 * k] = bf16_lo(w[k]);
        f[2 * k + 1] = bf16_hi(w[k]);
      }
      uint2 packed;
      if (ASYM) {
        uint32_t o2[2];
        quant_row_group_affine_x2<8>(f, sc, rc, sh_zp[r], sh_thr[r], o2);
        packed = make_uint2(o2[0], o2[1]);
      } else {
        uint32_t b[8];
        quant_row_group_x2<8>(f, sc, rc, b);
        packed = make_uint2(pack4_i8_prmt(b[0], b[1], b[2], b[3]), pack4_i8_prmt(b[4], b[5], b[6], b[7]));
      }
      *reinterpret_cast<uint2*>(xs + r * ld + (int64_t)c * 8) = packed;
    }
  }
  __syncthreads();
  const bool xr0 = g < nr;
  const uint8_t* sx0 = xs + g * ld;
  for (int64_t nb = blockIdx.x; nb < nbn; nb += gridDim.x) {
    const int64_t n0 = nb * 16;
    int acc0[2][4] = {};
    for (int64_t c0 = warp; c0 < nchunks; c0 += (int64_t)kSmWarps * kXsUnroll) {
      if (!preloaded) load_round(nb, c0, wa);
      preloaded = false;
#pragma unroll
      for (int u = 0; u < kXsUnroll; ++u) {
        const int64_t c = c0 + (int64_t)u * kSmWarps;
        const int64_t kb = c * 64 + tq * 16;
        const bool kin = (c < nchunks) && (kb < K);
        const uint4 x0 = (kin && xr0) ? *reinterpret_cast<const uint4*>(sx0 + kb) : make_uint4(0, 0, 0, 0);
        const uint32_t A0[4] = {wa[u][0].x, wa[u][0].y, wa[u][0].z, wa[u][0].w};
        const uint32_t A1[4] = {wa[u][1].x, wa[u][1].y, wa[u][1].z, wa[u][1].w};
        const uint32_t B0[4] = {x0.x, x0.y, x0.z, x0.w};
#pragma unroll
        for (int j = 0; j < 2; ++j)
          mma_s8_16832(acc0[j], A0[2 * j], A1[2 * j], A0[2 * j + 1], A1[2 * j + 1], B0[2 * j], B0[2 * j + 1]);
      }
    }
    preloaded = false;  // a warp with no chunk in the first block discards its preload
    red[warp][g][2 * tq] = acc0[0][0] + acc0[1][0];
    red[warp][g][2 * tq + 1] = acc0[0][1] + acc0[1][1];
    red[warp][g + 8][2 * tq] = acc0[0][2] + acc0[1][2];
    red[warp][g + 8][2 * tq + 1] = acc0[0][3] + acc0[1][3];
    __syncthreads();
    const int tok = threadIdx.x >> 4, ch = threadIdx.x & 15;
    const int64_t n = n0 + ch;
    if (tok < nr && n < N) {
      int sum = 0;
#pragma unroll
      for (int w = 0; w < kSmWarps; ++w) sum += red[w][ch][tok];
      if (W8A8_DOK(tok < rows, 403))
        y[tok * N + n] = __float2bfloat16_rn(epi_apply(ep, sum, sh_s[tok], ASYM ? sh_zp[tok] : 0, n));
    }
    __syncthreads();  // red is rewritten by the next block
  }
}

// ---- one or two token rows: a GEMV on dp4a.  The warp MMA above computes 16 x 8 outputs
// per instruction, so with one token 7/8 of its work is padding, and this GPU's int8 warp
// MMA rate is low enough (about 158 TOPS) that the padded products take about 70 % of the
// time the weight takes to stream from HBM.  Here each weight byte costs a quarter of a dp4a
// per token (exact s8 x s8 -> s32 products, int32 sums below 2^31 for K <= 65536).  A warp
// owns whole weight rows (rows gw, gw + warps, ...), read in units of 4096 bytes: lane l
// loads the 16-byte chunks l, l + 32, ... of the unit (each load instruction covers 512
// contiguous bytes), with the next unit's loads in flight while the current one is summed;
// the tokens' codes sit in shared memory (zero past K).  One warp reduction per row and
// token, then the epilogue by lane t for token t.  The codes are either given (XM = 0, up
// to MT = 2 rows) or computed in every CTA from one bf16 row with the stand-alone
// quantizer's exact rules (XM = 1 dynamic symmetric, XM = 2 dynamic asymmetric; the first
// weight unit is in flight meanwhile).
constexpr int kGvWarps = 8;
constexpr int kGvKU = 8;                       // 16-byte chunks per lane per unit
constexpr int kGvUnit = 32 * 16 * kGvKU;       // 4096 weight bytes per unit

__host__ __device__ inline int64_t gemv_xs_bytes(int64_t K) { return (K + kGvUnit - 1) / kGvUnit * kGvUnit; }

template <int XM, int MT>
__global__ void __launch_bounds__(kGvWarps * 32)
gemv_kernel(const __nv_bfloat16* __restrict__ x, const int8_t* __restrict__ xq, int64_t M, const int8_t* __restrict__ wq,
            int64_t N, int64_t K, EpiParams ep, __nv_bfloat16* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t xs[];
  __shared__ float sh_a[kGvWarps], sh_b[kGvWarps];
  __shared__ float sh_s, sh_r, sh_thr;
  __shared__ int sh_zp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tw = (int64_t)gridDim.x * kGvWarps;
  const int64_t gw = (int64_t)blockIdx.x * kGvWarps + warp;
  const int64_t nseg = gemv_xs_bytes(K) / kGvUnit;
  const int64_t units = gw < N ? ((N - gw + tw - 1) / tw) * nseg : 0;
  uint4 w0[kGvKU], w1[kGvKU];
  auto load_unit = [&](int64_t u, uint4 (&d)[kGvKU]) {
    const int64_t n = gw + (u / nseg) * tw, sg = u % nseg;
    const int8_t* wr = wq + n * K;
#pragma unroll
    for (int c = 0; c < kGvKU; ++c) {
      const int64_t k = (sg * kGvKU + c) * 512 + lane * 16;
      d[c] = ld16_stream_or_zero(wr + k, k < K && W8A8_DOK(n < N, 404));
    }
  };
  if (units > 0) load_unit(0, w0);

  // the tokens' codes into shared memory ([MT][xs bytes]), zero past K and for tokens >= M
  const int64_t nx = gemv_xs_bytes(K) / 16;
  if (XM == 0) {
    for (int64_t c = threadIdx.x; c < nx * MT; c += kGvWarps * 32) {
      const int64_t t = c / nx, k = (c - t * nx) * 16;
      reinterpret_cast<uint4*>(xs)[c] = ld16_or_zero(xq + t * K + k, t < M && k < K);
    }
  } else {
    constexpr bool ASYM = XM == 2;
    const int64_t nv = K / 8;
    const uint4* xr = reinterpret_cast<const uint4*>(x);
    float a = ASYM ? __int_as_float(0x7f800000) : 0.f, b = __int_as_float(0xff800000);
    for (int64_t c = threadIdx.x; c < nv; c += kGvWarps * 32) {
      const uint4 v = __ldg(xr + c);
      const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (ASYM) {
          a = fminf(a, fminf(bf16_lo(wd[k]), bf16_hi(wd[k])));
          b = fmaxf(b, fmaxf(bf16_lo(wd[k]), bf16_hi(wd[k])));
        } else {
          a = fmaxf(a, fmaxf(fabsf(bf16_lo(wd[k])), fabsf(bf16_hi(wd[k]))));
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      if (ASYM) {
        a = fminf(a, __shfl_xor_sync(0xffffffffu, a, o));
        b = fmaxf(b, __shfl_xor_sync(0xffffffffu, b, o));
      } else {
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      }
    }
    if (lane == 0) {
      sh_a[warp] = a;
      sh_b[warp] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float lo = sh_a[0], hi = sh_b[0];
#pragma unroll
      for (int w = 1; w < kGvWarps; ++w) {
        lo = ASYM ? fminf(lo, sh_a[w]) : fmaxf(lo, sh_a[w]);
        hi = fmaxf(hi, sh_b[w]);
      }
      const RowQuant rq = ASYM ? row_quant_asym(lo, hi) : row_quant_sym(lo);
      const float rc = __frcp_rn(rq.s);
      sh_s = rq.s;
      sh_r = rc;
      sh_zp = rq.zp;
      // the stand-alone affine quantizer's margin of its division-free fast path
      sh_thr = ASYM ? __fsub_rd(0.5f, __fmul_rn(__fmul_rn(fmaxf(fabsf(lo), fabsf(hi)), rc), 0x1p-21f)) : 0.f;
    }
    __syncthreads();
    const float sc = sh_s, rc = sh_r, thr = sh_thr;
    const int zpv = sh_zp;
    for (int64_t c = threadIdx.x; c < nx * 2; c += kGvWarps * 32) {
      uint2 packed = make_uint2(0, 0);
      if (c < nv) {
        const uint4 v = __ldg(xr + c);
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
        float f[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          f[2 * k] = bf16_lo(wd[k]);
          f[2 * k + 1] = bf16_hi(wd[k]);
        }
        if (ASYM) {
          uint32_t o2[2];
          quant_row_group_affine_x2<8>(f, sc, rc, zpv, thr, o2);
          packed = make_uint2(o2[0], o2[1]);
        } else {
          uint32_t q8[8];
          quant_row_group_x2<8>(f, sc, rc, q8);
          packed = make_uint2(pack4_i8_prmt(q8[0], q8[1], q8[2], q8[3]), pack4_i8_prmt(q8[4], q8[5], q8[6], q8[7]));
        }
      }
      reinterpret_cast<uint2*>(xs)[c] = packed;
    }
  }
  __syncthreads();
  // row scale and zero point of token `lane` (lane t < M writes token t's outputs)
  const int tl = lane < MT ? lane : 0;
  const float sx = XM == 0 ? (tl < M ? epi_row_scale(ep, tl) : 0.f) : sh_s;
  const int zpm = XM == 0 ? (tl < M ? epi_row_zp(ep, tl) : 0) : (XM == 2 ? sh_zp : 0);

  int acc[MT];
#pragma unroll
  for (int t = 0; t < MT; ++t) acc[t] = 0;
  auto sum_unit = [&](int64_t u, const uint4 (&d)[kGvKU]) {
    const int64_t sg = u % nseg;
#pragma unroll
    for (int c = 0; c < kGvKU; ++c) {
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const uint4 xv = reinterpret_cast<const uint4*>(xs)[t * nx + (sg * kGvKU + c) * 32 + lane];
        acc[t] = __dp4a((int)d[c].x, (int)xv.x, acc[t]);
        acc[t] = __dp4a((int)d[c].y, (int)xv.y, acc[t]);
        acc[t] = __dp4a((int)d[c].z, (int)xv.z, acc[t]);
        acc[t] = __dp4a((int)d[c].w, (int)xv.w, acc[t]);
      }
    }
    if (sg == nseg - 1) {
      int mine = 0;
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const int tot = __reduce_add_sync(0xffffffffu, acc[t]);
        mine = (lane == t) ? tot : mine;
        acc[t] = 0;
      }
      const int64_t n = gw + (u / nseg) * tw;
      if (lane < MT && lane < M && W8A8_DOK(n < N, 405))
        y[lane * N + n] = __float2bfloat16_rn(epi_apply(ep, mine, sx, zpm, n));
    }
  };
  for (int64_t u = 0; u < units; u += 2) {
    if (u + 1 < units) load_unit(u + 1, w1);
    sum_unit(u, w0);
    if (u + 2 < units) load_unit(u + 2, w0);
    if (u + 1 < units) sum_unit(u + 1, w1);
  }
}

// up to 2 token rows: the dp4a work grows with the tokens (a quarter instruction per weight
// byte and token) while the padded warp MMA costs the same up to 8; measured against the
// staged MMA kernel, 2 rows gain (28672 x 4096: 29.6 -> 26.9 us) and 3-4 rows lose on long
// rows (4096 x 14336 at 4 rows: 20.2 -> 26.5 us), so those stay there
constexpr int kGvMaxRows = 2;
bool gemv_ok(int64_t rows, int64_t K) {
  return rows >= 1 && rows <= kGvMaxRows && K > 0 && K % 16 == 0 && K <= 65536;
}

// x: the bf16 row (xm 1/2, one row) or null; g.a: the int8 codes (xm 0)
static cudaError_t gemv(int xm, const void* x, const GemmArgs& g, const EpiParams& ep, cudaStream_t st) {
  static thread_local int s_dev = -1, s_sms = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev != s_dev) {
    const int big = 64 * 1024;
    e = cudaFuncSetAttribute(gemv_kernel<0, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_kernel<0, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * big);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_kernel<1, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_kernel<2, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, big);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&s_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    s_dev = dev;
  }
  const int mt = g.rows <= 1 ? 1 : 2;
  const size_t xs_bytes = (size_t)gemv_xs_bytes(g.K) * (size_t)mt;
  // two CTAs per SM at most (registers, and the codes' shared memory); no more CTAs than
  // 8-row groups of the weight
  const int64_t want = (g.N + kGvWarps - 1) / kGvWarps;
  const int64_t cap = (xs_bytes <= 100 * 1024 ? 2 : 1) * (int64_t)s_sms;
  const unsigned grid = (unsigned)(want < cap ? want : cap);
  __nv_bfloat16* y = static_cast<__nv_bfloat16*>(g.y);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (xm == 1)
    gemv_kernel<1, 1><<<grid, kGvWarps * 32, xs_bytes, st>>>(xb, nullptr, 1, g.w, g.N, g.K, ep, y);
  else if (xm == 2)
    gemv_kernel<2, 1><<<grid, kGvWarps * 32, xs_bytes, st>>>(xb, nullptr, 1, g.w, g.N, g.K, ep, y);
  else if (mt == 1)
    gemv_kernel<0, 1><<<grid, kGvWarps * 32, xs_bytes, st>>>(nullptr, g.a, g.rows, g.w, g.N, g.K, ep, y);
  else
    gemv_kernel<0, 2><<<grid, kGvWarps * 32, xs_bytes, st>>>(nullptr, g.a, g.rows, g.w, g.N, g.K, ep, y);
  return cudaGetLastError();
}

bool gemm_small_m_fused_ok(int64_t rows, int64_t K) { return rows == 1 && xs_stride(K) <= 96 * 1024; }

cudaError_t gemm_small_m_fused(const void* x, int64_t ldx, const GemmArgs& g, cudaStream_t st) {
  const bool asym = g.act_mode == W8A8_ACT_DYN_TOKEN_ASYM;
  if (!asym && g.act_mode != W8A8_ACT_DYN_TOKEN_SYM) return cudaErrorInvalidValue;
  if (asym && !g.azp) return cudaErrorInvalidValue;
  EpiParams ep;
  ep.act_mode = g.act_mode;
  ep.w_mode = g.w_mode;
  ep.s_x = nullptr;
  ep.zp = nullptr;
  ep.azp = asym ? g.azp : nullptr;
  ep.s_w = g.s_w;
  ep.bias = static_cast<const __nv_bfloat16*>(g.bias);
  static thread_local int s_dev = -1, s_grid = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev != s_dev) {
    e = cudaFuncSetAttribute(gemm_small_m_fq_kernel<W8A8_ACT_DYN_TOKEN_SYM>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_small_m_fq_kernel<W8A8_ACT_DYN_TOKEN_ASYM>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    s_grid = 2 * sms;
    s_dev = dev;
  }
  if (g.rows == 1 && gemv_ok(1, g.K) && (reinterpret_cast<uintptr_t>(g.w) & 15) == 0)
    return gemv(asym ? 2 : 1, x, g, ep, st);
  const int64_t gx = (g.N + 15) / 16;
  const unsigned grid = (unsigned)(gx < s_grid ? gx : s_grid);
  const size_t xs_bytes = (size_t)(g.rows * xs_stride(g.K));
  if (asym)
    gemm_small_m_fq_kernel<W8A8_ACT_DYN_TOKEN_ASYM><<<grid, kSmWarps * 32, xs_bytes, st>>>(
        static_cast<const __nv_bfloat16*>(x), ldx, g.w, g.rows, g.N, g.K, ep, static_cast<__nv_bfloat16*>(g.y));
  else
    gemm_small_m_fq_kernel<W8A8_ACT_DYN_TOKEN_SYM><<<grid, kSmWarps * 32, xs_bytes, st>>>(
        static_cast<const __nv_bfloat16*>(x), ldx, g.w, g.rows, g.N, g.K, ep, static_cast<__nv_bfloat16*>(g.y));
  return cudaGetLastError();
}

cudaError_t gemm_small_m(const GemmArgs& g, cudaStream_t st) {
  EpiParams ep;
  ep.act_mode = g.act_mode;
  ep.w_mode = g.w_mode;
  ep.s_x = g.s_x;
  ep.zp = g.zp;
  ep.azp = g.azp;
  ep.s_w = g.s_w;
  ep.bias = static_cast<const __nv_bfloat16*>(g.bias);
  if (!g.seg && gemv_ok(g.rows, g.K) && (reinterpret_cast<uintptr_t>(g.w) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(g.a) & 15) == 0)
    return gemv(0, nullptr, g, ep, st);
  const int64_t gx = (g.N + 15) / 16;
  {
    const int64_t xs_bytes = g.rows * xs_stride(g.K);
    if (!g.seg && g.rows > 0 && g.rows <= 8 && xs_bytes <= 96 * 1024) {
      static thread_local int s_dev = -1, s_grid = 0;
      int dev = 0;
      cudaError_t e = cudaGetDevice(&dev);
      if (e != cudaSuccess) return e;
      if (dev != s_dev) {
        e = cudaFuncSetAttribute(gemm_small_m_xs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
        if (e != cudaSuccess) return e;
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        s_grid = 2 * sms;  // two CTAs per SM (registers and up to 2 x 96 KB of staged rows)
        s_dev = dev;
      }
      const unsigned grid = (unsigned)(gx < s_grid ? gx : s_grid);
      gemm_small_m_xs_kernel<<<grid, kSmWarps * 32, (size_t)xs_bytes, st>>>(g.a, g.w, g.rows, g.N, g.K, ep,
                                                                         static_cast<__nv_bfloat16*>(g.y));
      return cudaGetLastError();
    }
  }
  const int64_t gy = g.seg ? (g.rows + 15) / 16 + g.E : (g.rows + 15) / 16;
  if (gx == 0 || gy == 0) return cudaSuccess;
  if (gy > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)gx, (unsigned)gy);
  gemm_small_m_kernel<<<grid, kSmWarps * 32, 0, st>>>(g.a, g.w, g.rows, g.N, g.K, g.E, g.seg, ep,
                                                      static_cast<__nv_bfloat16*>(g.y));
  return cudaGetLastError();
}

#ifdef W8A8_DEBUG
cudaError_t debug_register_gemm_small(int32_t* word) { return w8a8_debug_register_here(word); }
#endif

}  // namespace w8a8
