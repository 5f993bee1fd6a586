// MoE routing on the GPU: per-token top-k expert choice with softmax weights, and the stable
// counting sort of the (token, slot) pairs into per-expert segments that the grouped GEMM,
// the gather-quantizer and the combine consume.
//
// The MoE INT8 scheme ([SGLang-CT] file tree, compressed_tensors_w8a8_int8_moe; [Kunlun-INT8]
// MoE method over experts w1/w2/w3) routes each token to its experts; the pages leave the
// router to the framework, so the rule is the plain one: the topk largest logits (equal
// logits: the lower expert index first), weights = softmax over all E logits at the chosen
// experts (not renormalised), and the routed rows ordered by expert, then token, then slot.

#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace w8a8 {

constexpr int kRouteWarps = 8;      // tokens per CTA in the top-k kernel
constexpr int kSortChunk = 256;     // routed entries per warp in the sort passes

// One warp per token.  Lane l holds experts l, l + 32, ... (EPL of them).  Softmax in fp32
// (max-subtracted exponentials, warp-tree sums); top-k by k rounds of a warp argmax whose
// ties go to the lower expert index.
template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int topk, int32_t* __restrict__ ids,
                  float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  float l[EPL];
  float m = -__int_as_float(0x7f800000);
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = lane + 32 * j;
    l[j] = e < E ? logits[t * E + e] : -__int_as_float(0x7f800000);
    m = fmaxf(m, l[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < EPL; ++j)
    if (lane + 32 * j < E) sum = __fadd_rn(sum, expf(__fsub_rn(l[j], m)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, o));
  uint32_t taken = 0u;  // bit j: expert lane + 32 j already chosen
  for (int r = 0; r < topk; ++r) {
    float bv = 0.f;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = lane + 32 * j;
      if (e < E && !((taken >> j) & 1u) && (be == 0x7FFFFFFF || l[j] > bv)) {
        bv = l[j];  // experts of one lane come in increasing order: '>' keeps the lower on ties
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (oe != 0x7FFFFFFF && (be == 0x7FFFFFFF || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == 0) {
      ids[t * topk + r] = be;
      w[t * topk + r] = __fdiv_rn(expf(__fsub_rn(bv, m)), sum);
    }
  }
}

// The routed entries of one warp's range, kSortChunk / 32 per lane, all loaded before use so
// that the range costs one memory round trip (-1 past the end).
constexpr int kSortPerLane = kSortChunk / 32;
__device__ __forceinline__ void load_range(const int32_t* __restrict__ ids, int64_t R, int64_t r0, int lane,
                                           int (&id)[kSortPerLane]) {
#pragma unroll
  for (int j = 0; j < kSortPerLane; ++j) {
    const int64_t i = r0 + 32 * j + lane;
    id[j] = i < R ? ids[i] : -1;
  }
}

// Pass 1: expert histogram of each warp's range of kSortChunk routed entries.
__global__ void __launch_bounds__(32)
route_hist_kernel(const int32_t* __restrict__ ids, int64_t R, int E, int32_t* __restrict__ counts) {
  __shared__ int hist[256];
  const int lane = threadIdx.x;
  int id[kSortPerLane];
  load_range(ids, R, (int64_t)blockIdx.x * kSortChunk, lane, id);
  for (int e = lane; e < E; e += 32) hist[e] = 0;
  __syncwarp();
#pragma unroll
  for (int j = 0; j < kSortPerLane; ++j)
    if (id[j] >= 0) atomicAdd(&hist[id[j]], 1);
  __syncwarp();
  for (int e = lane; e < E; e += 32) counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

// Pass 2 (one CTA, thread e = expert e): column prefix over the ranges (in place: counts[b][e]
// becomes the number of expert-e entries before range b), then the segment offsets.  The
// [B, E] table is walked in tiles of 32 ranges, loaded and stored coalesced through shared
// memory.
constexpr int kScanTile = 32;
__global__ void __launch_bounds__(256)
route_scan_kernel(int32_t* __restrict__ counts, int64_t B, int E, int64_t* __restrict__ seg) {
  __shared__ int tile[kScanTile * 256];
  __shared__ int64_t tot[256];
  const int e = threadIdx.x;
  int64_t run = 0;
  for (int64_t b0 = 0; b0 < B; b0 += kScanTile) {
    const int nb = (int)(B - b0 < kScanTile ? B - b0 : kScanTile);
    for (int i = threadIdx.x; i < nb * E; i += 256) tile[i] = counts[b0 * E + i];
    __syncthreads();
    if (e < E) {
      for (int j = 0; j < nb; ++j) {
        const int c = tile[j * E + e];
        tile[j * E + e] = (int)run;
        run += c;
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nb * E; i += 256) counts[b0 * E + i] = tile[i];
    __syncthreads();
  }
  tot[e] = e < E ? run : 0;
  __syncthreads();
  if (e == 0) {
    int64_t acc = 0;
    for (int f = 0; f < E; ++f) {
      const int64_t c = tot[f];
      seg[f] = acc;
      acc += c;
    }
    seg[E] = acc;
  }
}

// Pass 3: each warp walks its range again in order, 32 entries at a time; lanes holding the
// same expert are ranked by lane (match_any), so equal experts keep their (token, slot) order.
__global__ void __launch_bounds__(32)
route_scatter_kernel(const int32_t* __restrict__ ids, int64_t R, int E, int topk,
                     const int32_t* __restrict__ counts, const int64_t* __restrict__ seg,
                     int64_t* __restrict__ row_index, int64_t* __restrict__ row_of) {
  __shared__ int64_t next[256];
  const int lane = threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.x * kSortChunk;
  int id[kSortPerLane];
  load_range(ids, R, r0, lane, id);
  for (int e = lane; e < E; e += 32) next[e] = seg[e] + counts[(int64_t)blockIdx.x * E + e];
  __syncwarp();
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kSortPerLane; ++j) {
    const int64_t i = r0 + 32 * j + lane;
    const bool valid = id[j] >= 0;
    const uint32_t peers = __match_any_sync(0xffffffffu, id[j]);
    int64_t pos = 0;
    if (valid) pos = next[id[j]] + __popc(peers & lt);
    __syncwarp();
    if (valid && (peers & lt) == 0u) next[id[j]] += __popc(peers);  // the lowest lane of each group
    __syncwarp();
    if (valid) {
      row_index[pos] = i / topk;
      row_of[i] = pos;
    }
  }
}

size_t moe_route_workspace(int64_t T, int E, int topk) {
  const int64_t R = T * topk;
  const int64_t B = (R + kSortChunk - 1) / kSortChunk;
  return (size_t)((B * E * 4 + 255) / 256 * 256);
}

cudaError_t moe_route(const float* logits, int64_t T, int E, int topk, int32_t* ids, float* w, int64_t* seg,
                      int64_t* row_index, int64_t* row_of, void* ws, cudaStream_t st) {
  const int64_t R = T * topk;
  const int64_t B = (R + kSortChunk - 1) / kSortChunk;
  int32_t* counts = static_cast<int32_t*>(ws);
  if (T > 0) {
    const unsigned g = (unsigned)((T + kRouteWarps - 1) / kRouteWarps);
    const int epl = (E + 31) / 32;
    if (epl <= 1)
      route_topk_kernel<1><<<g, kRouteWarps * 32, 0, st>>>(logits, T, E, topk, ids, w);
    else if (epl <= 2)
      route_topk_kernel<2><<<g, kRouteWarps * 32, 0, st>>>(logits, T, E, topk, ids, w);
    else if (epl <= 4)
      route_topk_kernel<4><<<g, kRouteWarps * 32, 0, st>>>(logits, T, E, topk, ids, w);
    else
      route_topk_kernel<8><<<g, kRouteWarps * 32, 0, st>>>(logits, T, E, topk, ids, w);
    route_hist_kernel<<<(unsigned)B, 32, 0, st>>>(ids, R, E, counts);
  }
  route_scan_kernel<<<1, 256, 0, st>>>(counts, B, E, seg);
  if (T > 0) route_scatter_kernel<<<(unsigned)B, 32, 0, st>>>(ids, R, E, topk, counts, seg, row_index, row_of);
  return cudaGetLastError();
}

#ifdef W8A8_DEBUG
cudaError_t debug_register_moe_route(int32_t* word) { return w8a8_debug_register_here(word); }
#endif

}  // namespace w8a8
