// Weight-streaming INT8 GEMM for few activation rows (decode-sized M).
//
// With M <= 16 the layer is bound by reading the int8 weight once from HBM (2*M ops per
// weight byte), so the kernel is shaped for bandwidth, not for tensor-core peak: each CTA
// owns 16 output channels and 16 token rows, its 8 warps split K into interleaved
// 64-byte chunks so that neighbouring warps read neighbouring bytes of a weight row, and
// each thread keeps four chunks of 16-byte loads in flight.  The integer products run on
// the exact s8 x s8 -> s32 warp MMA (m16n8k32), with the weight as the 16-row operand
// and the tokens as the 8-column operand.  The partial sums of the 8 warps are added in
// shared memory and the scale/azp/bias epilogue is applied before one bf16 store.
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
    y[m * N + n] = __float2bfloat16_rn(v);
  }
}

// Dense decode blocks (at most 2 token rows): the rows are staged in shared memory once (row
// stride K + 16 bytes so rows read by one quarter-warp fall in different banks), then every
// thread issues its weight loads for kXsUnroll chunks before the first MMA, so a K = 4096
// block needs a single dependent round trip to HBM instead of two.
constexpr int kXsUnroll = 8;
__global__ void __launch_bounds__(kSmWarps * 32)
gemm_small_m_xs_kernel(const int8_t* __restrict__ xq, const int8_t* __restrict__ wq, int64_t rows, int64_t N,
                       int64_t K, EpiParams ep, __nv_bfloat16* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t xs[];
  __shared__ int red[kSmWarps][16][17];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t n0 = (int64_t)blockIdx.x * 16;
  const int64_t m0 = (int64_t)blockIdx.y * 16;
  const int nr = (int)((rows - m0) < 16 ? (rows - m0) : 16);
  const int64_t ld = K + 16;
  // stage the token rows (K % 16 == 0, rows 16-byte aligned)
  for (int64_t i = threadIdx.x; i < (int64_t)nr * (K / 16); i += blockDim.x) {
    const int64_t r = i / (K / 16), c = i % (K / 16);
    *reinterpret_cast<uint4*>(xs + r * ld + c * 16) = __ldg(reinterpret_cast<const uint4*>(xq + (m0 + r) * K) + c);
  }
  __syncthreads();
  const bool wr0 = (n0 + g) < N, wr1 = (n0 + g + 8) < N;
  const bool xr0 = g < nr, xr1 = (g + 8) < nr;
  const bool two = nr > 8;
  const int8_t* pw0 = wq + (n0 + g) * K;
  const int8_t* pw1 = wq + (n0 + g + 8) * K;
  const uint8_t* sx0 = xs + g * ld;
  const uint8_t* sx1 = xs + (g + 8) * ld;
  int acc0[4] = {0, 0, 0, 0}, acc1[4] = {0, 0, 0, 0};
  const int64_t nchunks = (K + 63) / 64;
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
        mma_s8_16832(acc0, A0[2 * j], A1[2 * j], A0[2 * j + 1], A1[2 * j + 1], B0[2 * j], B0[2 * j + 1]);
      if (two) {
        const uint4 x1 = (kin && xr1) ? *reinterpret_cast<const uint4*>(sx1 + kb) : make_uint4(0, 0, 0, 0);
        const uint32_t B1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int j = 0; j < 2; ++j)
          mma_s8_16832(acc1, A0[2 * j], A1[2 * j], A0[2 * j + 1], A1[2 * j + 1], B1[2 * j], B1[2 * j + 1]);
      }
    }
  }
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
  if (tok < nr && n < N) {
    int sum = 0;
#pragma unroll
    for (int w = 0; w < kSmWarps; ++w) sum += red[w][ch][tok];
    y[m * N + n] = __float2bfloat16_rn(epi_apply(ep, sum, epi_row_scale(ep, m), epi_row_zp(ep, m), n));
  }
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
  const int64_t gx = (g.N + 15) / 16;
  {
    // decode (at most 2 token rows): staging the rows once per CTA removes the second
    // dependent load round; with more rows the staging traffic outweighs it
    const int64_t xs_bytes = (g.rows < 16 ? g.rows : 16) * (g.K + 16);
    if (!g.seg && g.rows > 0 && g.rows <= 2 && xs_bytes <= 96 * 1024) {
      static int s_attr = 0;
      if (xs_bytes > 48 * 1024 && !s_attr) {
        cudaError_t e = cudaFuncSetAttribute(gemm_small_m_xs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
        if (e != cudaSuccess) return e;
        s_attr = 1;
      }
      dim3 grid((unsigned)gx, (unsigned)((g.rows + 15) / 16));
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

}  // namespace w8a8
