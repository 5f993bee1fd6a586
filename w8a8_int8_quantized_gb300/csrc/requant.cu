// FP8 E4M3 block-scaled weight -> INT8 weight with one float32 scale per row.
//
// "MiniMax-M2.7 FP8 转昆仑芯 INT8" README, section 转换关系:
//   W[i,j] = W_fp8[i,j] * weight_scale_inv[i//128, j//128]   (the _inv scale multiplies)
//   s[i]   = max_j |W[i,j]| / 127 ;  q = clamp(round(W / s), -127, 127) ;  zero row -> q=0, s=1.
// Rows are independent (the README's tool also works matrix by matrix, row chunk by row
// chunk), so one warp owns one row at a time.  Aligned rows (K % 16 == 0) are brought into
// shared memory by one bulk copy each and read twice on chip (absmax, then quantize); rows
// of K % 4 == 0 up to 4096 on 4-byte boundaries are held in registers as words; the others
// take a warp-per-row byte-load path.  One launch per path covers a whole batch of matrices
// through a by-value descriptor table, optionally writing each row's code sum (azp_adj).
// Also here: the requantization of a fused weight's per-tensor partitions to their largest
// scale ("[SGLang] W4A8, W8A8, W4A4", item 7, requantize_with_max_scale).
#include <atomic>

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

// ---------------------------------------------------------------- vector path
// Matrices with K % 16 == 0 and 16-byte aligned rows.  One warp per row; the row is read
// twice on chip (pass 1: absmax, pass 2: quantize) but from HBM once.
//
// Decoding.  The hardware E4M3 -> fp16x2 conversion is exact (every E4M3 value is an fp16
// value) and costs one instruction per two codes; fp16 -> fp32 is exact too.
//
// Pass 1, absmax without the block scale per code: the codes of one 128-column block share
// one scale sc > 0, so max_j RN(|v_j| * sc) = RN(max_j |v_j| * sc) (rounding is monotone).
// max_j |v_j| is taken on the fp16 values with the NaN-propagating absolute maximum, so an
// E4M3 NaN code (S.1111.111) anywhere in the block leaves a NaN there.
//
// Pass 2, q = rint(RN(Wf / s)) with Wf = RN(v * sc), from one multiply per code: with
// r = RN(1/s) and the block factor c = RN(sc * r), t = RN(v * c) differs from Wf / s by at
// most |Wf / s| * 4.0001 * 2^-24 < 2^-15 (|Wf / s| <= 127 * (1 + 2^-24) because |Wf| is at
// most the row absmax), and RN(Wf / s) differs from Wf / s by less than 2^-17.  So when t is
// more than 2^-14 away from every half-integer, rint(t) = rint(RN(Wf / s)).  t + 1.5 * 2^23
// rounds t to an integer (ties to even) and its low byte is the int8 code; the distance to
// that integer is exact.  Groups with a value within 2^-14 of a tie (about 1 code in 8000),
// and blocks whose scale or factor lies outside [2^-100, 2^100] (where the products above
// could leave the normal range), are decided by the IEEE division itself.

// sum over the warp (the row sums of the codes: the weight's azp_adj)
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// largest |value| of n16 groups of 16 codes as fp16 bits (> 0x7C00: a NaN code)
__device__ __forceinline__ uint32_t habsmax_nan(uint32_t acc, uint32_t h) {
  asm("max.NaN.xorsign.abs.f16x2 %0, %0, %1;" : "+r"(acc) : "r"(h));
  return acc;
}
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& h01, uint32_t& h23) {
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.rn.f16x2.e4m3x2 %0, lo; cvt.rn.f16x2.e4m3x2 %1, hi; }"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
}
__device__ __forceinline__ uint32_t group_absmax(uint32_t acc, const uint4& c) {
  uint32_t h0, h1, h2, h3, h4, h5, h6, h7;
  e4m3x4_to_f16x4(c.x, h0, h1);
  e4m3x4_to_f16x4(c.y, h2, h3);
  e4m3x4_to_f16x4(c.z, h4, h5);
  e4m3x4_to_f16x4(c.w, h6, h7);
  return habsmax_nan(habsmax_nan(habsmax_nan(habsmax_nan(acc, h0), h1), habsmax_nan(h2, h3)),
                     habsmax_nan(habsmax_nan(h4, h5), habsmax_nan(h6, h7)));
}
// the block absmax times the block scale, RN(max|v| * sc); NaN codes and illegal scales flag bad
__device__ __forceinline__ float block_amax(uint32_t acc, float sc, bool& bad) {
  const uint32_t hm = max(acc & 0x7FFFu, (acc >> 16) & 0x7FFFu);  // non-negative fp16 bits order like values
  bad |= (hm > 0x7C00u) || !scale_ok(sc);
  return __fmul_rn(__half2float(__ushort_as_half((unsigned short)hm)), sc);
}
// block factor c = RN(sc * r), or -1 when the fast path's range conditions do not hold
__device__ __forceinline__ float block_factor(float sc, float r) {
  const float c = __fmul_rn(sc, r);
  return (sc >= 0x1p-100f && c >= 0x1p-100f && c <= 0x1p100f) ? c : -1.f;
}

// 4*NW codes (NW words) -> 4*NW int8 codes (see the note above); c < 0 takes the exact path
// for all of them.
template <int NW>
__device__ __forceinline__ void requant_words(const uint32_t* wd, float c, const float* sc_ptr, float s,
                                              uint32_t* out) {
  constexpr int NV = 4 * NW;
  float f[NV];
#pragma unroll
  for (int g = 0; g < NW; ++g) {
    uint32_t h01, h23;
    e4m3x4_to_f16x4(wd[g], h01, h23);
    const __half2 a = *reinterpret_cast<const __half2*>(&h01), b = *reinterpret_cast<const __half2*>(&h23);
    f[4 * g] = __low2float(a);
    f[4 * g + 1] = __high2float(a);
    f[4 * g + 2] = __low2float(b);
    f[4 * g + 3] = __high2float(b);
  }
  const uint64_t kMagic = 0x4B4000004B400000ull;  // 1.5*2^23 in both lanes
  const uint64_t c2 = f2pack(c, c);
  uint32_t bq[NV];
  float emax = 0.f;
#pragma unroll
  for (int j = 0; j < NV; j += 2) {
    const uint64_t t = f2mul(f2pack(f[j], f[j + 1]), c2);
    const uint64_t m = f2add(t, kMagic);
    float e0, e1, m0, m1;
    f2unpack(f2sub(t, f2sub(m, kMagic)), e0, e1);
    f2unpack(m, m0, m1);
    emax = fmaxf(emax, fmaxf(fabsf(e0), fabsf(e1)));
    bq[j] = __float_as_uint(m0);
    bq[j + 1] = __float_as_uint(m1);
  }
  if (!(emax < 0.49993896484375f) || c < 0.f) {  // 0.5 - 2^-14
    const float sc = *sc_ptr;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const float t = __fmul_rn(f[j], c);
      const float e = __fsub_rn(t, __fsub_rn(__fadd_rn(t, 12582912.0f), 12582912.0f));
      if (c < 0.f || !(fabsf(e) < 0.49993896484375f))
        bq[j] = 0x4B400000u + (uint32_t)__float2int_rn(rintf(__fdiv_rn(__fmul_rn(f[j], sc), s)));
    }
  }
#pragma unroll
  for (int g = 0; g < NW; ++g) out[g] = pack4_i8_prmt(bq[4 * g], bq[4 * g + 1], bq[4 * g + 2], bq[4 * g + 3]);
}

__device__ __forceinline__ uint4 requant_group(const uint4& cd, float c, const float* sc_ptr, float s) {
  const uint32_t wd[4] = {cd.x, cd.y, cd.z, cd.w};
  uint32_t out[4];
  requant_words<4>(wd, c, sc_ptr, s, out);
  return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ const ReqMat& find_mat(const ReqBatch& b, int64_t grow) {
  int lo = 0, hi = b.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (b.m[mid].row0 <= grow) lo = mid; else hi = mid - 1;
  }
  return b.m[lo];
}

// Pass 1 over a row held in shared memory: lane l owns the 128-column blocks l, l + 32, ...
// A full block is read in a lane-rotated order so that the eight lanes of each quarter-warp
// touch eight different 16-byte bank groups.
__device__ __forceinline__ void row_absmax_smem(const uint4* rowv, const float* srow, int nv, int nbc, int lane,
                                                float& amax, bool& bad) {
  for (int b = lane; b < nbc; b += 32) {
    const int n16 = min(8, nv - 8 * b);
    uint32_t acc = 0u;
    if (n16 == 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j) acc = group_absmax(acc, rowv[8 * b + ((j + lane) & 7)]);
    } else {
      for (int j = 0; j < n16; ++j) acc = group_absmax(acc, rowv[8 * b + j]);
    }
    amax = fmaxf(amax, block_amax(acc, srow[b], bad));
  }
}

__device__ __forceinline__ float row_scale(float amax, bool& bad) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  bad = __any_sync(0xffffffffu, bad) || !(amax <= 3.402823466e38f);
  return (!bad && amax != 0.f) ? __fdiv_rn(amax, 127.f) : 1.f;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Bounded waits of the row ring: the limit (2 s) and, for tests of the timeout path only, a
// number of bytes that the first row's barrier of the launch expects beyond what its bulk
// copy delivers, so that its wait cannot complete (set by w8a8_test_requant_wait_fault; both
// off by default).
struct RingWait {
  uint64_t limit_ns;
  uint32_t extra_tx;
  uint32_t pad;
};

// waits for the phase with the given parity; false once `limit_ns` has passed
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    if (ok) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > limit_ns) return false;
  }
}

// Row-ring kernel: every warp owns one shared-memory slot of `slot` bytes and walks the
// batch's rows gw, gw + warps, ...; a row is brought in by one bulk copy (issued right after
// the warp has finished the previous row), so many rows per SM are in flight while other
// warps compute.  slot >= the largest K of the batch, a multiple of 128.
template <int WARPS, bool ADJ>
__global__ void __launch_bounds__(WARPS * 32, 1024 / (WARPS * 32))
requant_ring_kernel(const __grid_constant__ ReqBatch b, int slot, int32_t* st, const RingWait rw) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + (size_t)warp * slot;
  float* cb = reinterpret_cast<float*>(smem + (size_t)WARPS * slot) + (size_t)warp * (slot / 128);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (size_t)WARPS * slot + (size_t)WARPS * (slot / 128) * 4) + warp;
  const uint32_t sbar = (uint32_t)__cvta_generic_to_shared(bar);
  const uint32_t sring = (uint32_t)__cvta_generic_to_shared(ring);
  const int64_t gw = (int64_t)blockIdx.x * WARPS + warp, tw = (int64_t)gridDim.x * WARPS;
  if (gw >= b.total_rows) return;
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(sbar));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    const ReqMat& m0 = find_mat(b, gw);
    // (the test hook's extra bytes go to the launch's first row only; the copy itself
    // completes as usual)
    if (gw == 0 && rw.extra_tx)
      asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;\n" ::"r"(sbar), "r"(rw.extra_tx) : "memory");
    bulk_load(sring, m0.w + (gw - m0.row0) * (int64_t)m0.K, (uint32_t)m0.K, sbar);
  }
  __syncwarp();
  uint32_t phase = 0;
  for (int64_t grow = gw; grow < b.total_rows; grow += tw, phase ^= 1u) {
    const ReqMat& mt = find_mat(b, grow);
    const int64_t i = grow - mt.row0;
    const int K = mt.K, nv = K / 16, nbc = (K + 127) / 128;
    if (!__all_sync(0xffffffffu, bar_wait(sbar, phase, rw.limit_ns))) {
      if (lane == 0) report_status(st, W8A8_ERR_TIMEOUT);
      return;
    }
    const uint4* rowv = reinterpret_cast<const uint4*>(ring);
    const float* srow = mt.sinv + (i / 128) * nbc;
    float amax = 0.f;
    bool bad = false;
    row_absmax_smem(rowv, srow, nv, nbc, lane, amax, bad);
    const float s = row_scale(amax, bad);
    uint4* qr = reinterpret_cast<uint4*>(mt.q + i * (int64_t)K);
    int qsum = 0;
    if (!bad) {
      const float r = __frcp_rn(s);
      for (int bb = lane; bb < nbc; bb += 32) cb[bb] = block_factor(srow[bb], r);
      __syncwarp();
#pragma unroll 2
      for (int idx = lane; idx < nv; idx += 32) {
        const uint4 o = requant_group(rowv[idx], cb[idx >> 3], srow + (idx >> 3), s);
        if (W8A8_DOK(i < mt.N && (int64_t)(idx + 1) * 16 <= K, 201)) qr[idx] = o;
        if (ADJ && mt.adj) qsum = sum4_i8(o.w, sum4_i8(o.z, sum4_i8(o.y, sum4_i8(o.x, qsum))));
      }
    } else {
      for (int idx = lane; idx < nv; idx += 32) qr[idx] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (ADJ && mt.adj) qsum = warp_sum_i(qsum);
    if (lane == 0 && W8A8_DOK(i >= 0 && i < mt.N, 202)) {
      mt.s[i] = s;
      if (ADJ && mt.adj) mt.adj[i] = qsum;
      if (bad) report_status(st, W8A8_ERR_BAD_SCALE);
    }
    __syncwarp();  // every lane is done with the slot (and with cb)
    if (lane == 0 && grow + tw < b.total_rows) {
      const ReqMat& mn = find_mat(b, grow + tw);
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      bulk_load(sring, mn.w + (grow + tw - mn.row0) * (int64_t)mn.K, (uint32_t)mn.K, sbar);
    }
  }
}

// Rows too long for a shared-memory slot: a warp streams its row from global memory twice
// (the second pass mostly from L1/L2).
constexpr int kReqStreamWarps = 8;
constexpr int kReqWordWarps = 8;
constexpr int kReqWordMaxK = 128 * 32;
template <bool ADJ>
__global__ void __launch_bounds__(kReqStreamWarps * 32)
requant_stream_kernel(const __grid_constant__ ReqBatch b, int32_t* st) {
  const int lane = threadIdx.x & 31;
  const int64_t tw = (int64_t)gridDim.x * kReqStreamWarps;
  for (int64_t grow = (int64_t)blockIdx.x * kReqStreamWarps + (threadIdx.x >> 5); grow < b.total_rows; grow += tw) {
    const ReqMat& mt = find_mat(b, grow);
    const int64_t i = grow - mt.row0;
    const int K = mt.K, nv = K / 16, nbc = (K + 127) / 128;
    const uint4* wr = reinterpret_cast<const uint4*>(mt.w + i * (int64_t)K);
    const float* srow = mt.sinv + (i / 128) * nbc;
    float amax = 0.f;
    bool bad = false;
    for (int bb = lane; bb < nbc; bb += 32) {
      const int n16 = min(8, nv - 8 * bb);
      uint32_t acc = 0u;
      for (int j = 0; j < n16; ++j) acc = group_absmax(acc, wr[8 * bb + j]);
      amax = fmaxf(amax, block_amax(acc, srow[bb], bad));
    }
    const float s = row_scale(amax, bad);
    uint4* qr = reinterpret_cast<uint4*>(mt.q + i * (int64_t)K);
    int qsum = 0;
    if (!bad) {
      const float r = __frcp_rn(s);
#pragma unroll 2
      for (int idx = lane; idx < nv; idx += 32) {
        const uint4 o = requant_group(wr[idx], block_factor(srow[idx >> 3], r), srow + (idx >> 3), s);
        qr[idx] = o;
        if (ADJ && mt.adj) qsum = sum4_i8(o.w, sum4_i8(o.z, sum4_i8(o.y, sum4_i8(o.x, qsum))));
      }
    } else {
      for (int idx = lane; idx < nv; idx += 32) qr[idx] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (ADJ && mt.adj) qsum = warp_sum_i(qsum);
    if (lane == 0) {
      mt.s[i] = s;
      if (ADJ && mt.adj) mt.adj[i] = qsum;
      if (bad) report_status(st, W8A8_ERR_BAD_SCALE);
    }
  }
}

// ring slot bytes for a largest row of kmax bytes; warps per CTA so that two CTAs fit an SM
static int ring_slot(int64_t kmax) { return (int)((kmax + 127) / 128 * 128); }
static size_t ring_smem(int warps, int slot) {
  return (size_t)warps * slot + (size_t)warps * (slot / 128) * 4 + (size_t)warps * 8;
}

static std::atomic<uint64_t> g_ring_limit_ns{2000000000ull};
static std::atomic<uint32_t> g_ring_extra_tx{0u};

static RingWait ring_wait() {
  RingWait w;
  w.limit_ns = g_ring_limit_ns.load(std::memory_order_relaxed);
  w.extra_tx = g_ring_extra_tx.load(std::memory_order_relaxed);
  w.pad = 0;
  return w;
}

template <int WARPS, bool ADJ>
static cudaError_t launch_ring(const ReqBatch& b, int slot, int32_t* st, cudaStream_t stream) {
  static thread_local int s_dev = -1, s_sms = 0;
  static thread_local size_t s_attr = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = ring_smem(WARPS, slot);
  if (s_dev != dev) {
    e = cudaDeviceGetAttribute(&s_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    s_dev = dev;
    s_attr = 0;
  }
  if (smem > s_attr) {
    e = cudaFuncSetAttribute(requant_ring_kernel<WARPS, ADJ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    s_attr = smem;
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, requant_ring_kernel<WARPS, ADJ>, WARPS * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t need = (b.total_rows + WARPS - 1) / WARPS;
  const int64_t cap = (int64_t)s_sms * per_sm;
  requant_ring_kernel<WARPS, ADJ><<<(unsigned)(need < cap ? need : cap), WARPS * 32, smem, stream>>>(b, slot, st,
                                                                                                  ring_wait());
  return cudaGetLastError();
}

template <bool ADJ>
static cudaError_t launch_vec(const ReqBatch& b, int32_t* st, cudaStream_t stream) {
  int64_t kmax = 0;
  for (int k = 0; k < b.count; ++k) kmax = b.m[k].K > kmax ? b.m[k].K : kmax;
  const int slot = ring_slot(kmax);
  // slots of 16 warps up to 112 KB per CTA, so that two CTAs share an SM
  if (ring_smem(16, slot) <= (size_t)112 * 1024) return launch_ring<16, ADJ>(b, slot, st, stream);
  if (ring_smem(8, slot) <= (size_t)112 * 1024) return launch_ring<8, ADJ>(b, slot, st, stream);
  if (ring_smem(4, slot) <= (size_t)200 * 1024) return launch_ring<4, ADJ>(b, slot, st, stream);
  static thread_local unsigned cached = 0;
  if (cached == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, requant_stream_kernel<ADJ>, kReqStreamWarps * 32, 0) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    cached = (unsigned)((sms < 1 ? 1 : sms) * per_sm);
  }
  const int64_t need = (b.total_rows + kReqStreamWarps - 1) / kReqStreamWarps;
  requant_stream_kernel<ADJ><<<(unsigned)(need < (int64_t)cached ? need : (int64_t)cached), kReqStreamWarps * 32, 0,
                          stream>>>(b, st);
  return cudaGetLastError();
}

// Rows of K % 4 == 0 (K <= 128 * WPL) on 4-byte aligned but not 16-byte aligned storage
// (e.g. K = 1500): a warp holds its row in registers as 32-bit words, word 32 j + l in lane l,
// so a lane's j-th word lies in the row's 128-column block j.  The row absmax is then one warp
// reduction of the per-lane maxima of RN(max|v| * sc_j), the codes are rewritten with the same
// one-multiply rule as the vector path (exact fallback included), and each word is stored
// back with one 4-byte store.
template <int WPL, bool ADJ>
__global__ void __launch_bounds__(kReqWordWarps * 32)
requant_word_kernel(const __grid_constant__ ReqBatch b, int32_t* st) {
  const int lane = threadIdx.x & 31;
  const int64_t tw = (int64_t)gridDim.x * kReqWordWarps;
  for (int64_t grow = (int64_t)blockIdx.x * kReqWordWarps + (threadIdx.x >> 5); grow < b.total_rows; grow += tw) {
    const ReqMat& mt = find_mat(b, grow);
    const int64_t i = grow - mt.row0;
    const int K = mt.K, nw = K / 4, nbc = (K + 127) / 128;
    const uint32_t* wr = reinterpret_cast<const uint32_t*>(mt.w + i * (int64_t)K);
    const float* srow = mt.sinv + (i / 128) * nbc;
    uint32_t v[WPL];
#pragma unroll
    for (int j = 0; j < WPL; ++j) {
      const int w = 32 * j + lane;
      v[j] = w < nw ? __ldg(wr + w) : 0u;  // code 0 (+0) past the end: no effect on the max
    }
    float amax = 0.f;
    bool bad = false;
#pragma unroll
    for (int j = 0; j < WPL; ++j) {
      if (j < nbc) {
        uint32_t h01, h23;
        e4m3x4_to_f16x4(v[j], h01, h23);
        amax = fmaxf(amax, block_amax(habsmax_nan(habsmax_nan(0u, h01), h23), srow[j], bad));
      }
    }
    const float s = row_scale(amax, bad);
    uint32_t* qr = reinterpret_cast<uint32_t*>(mt.q + i * (int64_t)K);
    int qsum = 0;
    if (!bad) {
      const float r = __frcp_rn(s);
#pragma unroll
      for (int j = 0; j < WPL; ++j) {
        const int w = 32 * j + lane;
        if (w < nw) {
          uint32_t o;
          requant_words<1>(&v[j], block_factor(srow[j], r), srow + j, s, &o);
          qr[w] = o;
          if (ADJ && mt.adj) qsum = sum4_i8(o, qsum);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < WPL; ++j)
        if (32 * j + lane < nw) qr[32 * j + lane] = 0u;
    }
    if (ADJ && mt.adj) qsum = warp_sum_i(qsum);
    if (lane == 0) {
      mt.s[i] = s;
      if (ADJ && mt.adj) mt.adj[i] = qsum;
      if (bad) report_status(st, W8A8_ERR_BAD_SCALE);
    }
  }
}

template <int WPL, bool ADJ>
static cudaError_t launch_word(const ReqBatch& b, int32_t* st, cudaStream_t stream) {
  static thread_local unsigned cached = 0;
  if (cached == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, requant_word_kernel<WPL, ADJ>, kReqWordWarps * 32,
                                                      0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    cached = (unsigned)((sms < 1 ? 1 : sms) * per_sm);
  }
  const int64_t need = (b.total_rows + kReqWordWarps - 1) / kReqWordWarps;
  requant_word_kernel<WPL, ADJ><<<(unsigned)(need < (int64_t)cached ? need : (int64_t)cached), kReqWordWarps * 32,
                                  0, stream>>>(b, st);
  return cudaGetLastError();
}

template <bool ADJ>
static cudaError_t launch_words(const ReqBatch& b, int32_t* st, cudaStream_t stream) {
  int64_t kmax = 0;
  for (int k = 0; k < b.count; ++k) kmax = b.m[k].K > kmax ? b.m[k].K : kmax;
  if (kmax <= 128 * 4) return launch_word<4, ADJ>(b, st, stream);
  if (kmax <= 128 * 12) return launch_word<12, ADJ>(b, st, stream);
  return launch_word<32, ADJ>(b, st, stream);
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
  int qsum = 0;
  for (int64_t j = lane; j < K; j += 32) {
    int v = 0;
    if (!bad) v = quant_sym(__fmul_rn(e4m3_value(wr[j]), srow[j >> 7]), s);
    qr[j] = (int8_t)v;
    qsum += v;
  }
  if (mt.adj) qsum = warp_sum_i(qsum);
  if (lane == 0) {
    mt.s[i] = s;
    if (mt.adj) mt.adj[i] = qsum;
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
  ReqBatch vb, wb, gb;
  vb.count = wb.count = gb.count = 0;
  vb.pad = wb.pad = gb.pad = 0;
  vb.total_rows = wb.total_rows = gb.total_rows = 0;
  for (int k = 0; k < b.count; ++k) {
    ReqBatch& t = b.m[k].vec == 1 ? vb : (b.m[k].vec == 2 ? wb : gb);
    t.m[t.count] = b.m[k];
    t.m[t.count].row0 = (int32_t)t.total_rows;
    t.total_rows += b.m[k].N;
    ++t.count;
  }
  if (vb.total_rows > 0) {
    bool adj = false;
    for (int k = 0; k < vb.count; ++k) adj |= vb.m[k].adj != nullptr;
    cudaError_t e = adj ? launch_vec<true>(vb, st, stream) : launch_vec<false>(vb, st, stream);
    if (e != cudaSuccess) return e;
  }
  if (wb.total_rows > 0) {
    bool adj = false;
    for (int k = 0; k < wb.count; ++k) adj |= wb.m[k].adj != nullptr;
    cudaError_t e = adj ? launch_words<true>(wb, st, stream) : launch_words<false>(wb, st, stream);
    if (e != cudaSuccess) return e;
  }
  if (gb.total_rows > 0) {
    const int64_t blocks = (gb.total_rows + kReqWarps - 1) / kReqWarps;
    requant_generic_kernel<<<(unsigned)blocks, kReqWarps * 32, 0, stream>>>(gb, st);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Per-tensor scales of a fused weight (Q/K/V partitions) unified to their maximum:
//   w'[n,k] = clamp(rint(RN(RN(q[n,k] * s_p) / s_max)), -127, 127)
// The result depends only on the code and its partition, so every CTA first evaluates that
// rule (one fp32 multiply, the IEEE division, ties-to-even conversion) for the 256 codes of
// each partition into a shared-memory table; the weight is then streamed through the table,
// 16 bytes per load, in place.  A partition scale that is not positive and finite leaves the
// weight and s_out untouched and reports W8A8_ERR_BAD_SCALE.
// ---------------------------------------------------------------------------
constexpr int kMsThreads = 256;
constexpr int kMsUnroll = 4;

__device__ __forceinline__ uint32_t lut_map4(const int8_t* lut, uint32_t w) {
  const uint32_t b0 = (uint8_t)lut[w & 0xFFu], b1 = (uint8_t)lut[(w >> 8) & 0xFFu];
  const uint32_t b2 = (uint8_t)lut[(w >> 16) & 0xFFu], b3 = (uint8_t)lut[w >> 24];
  return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

template <bool VEC>
__global__ void __launch_bounds__(kMsThreads)
max_scale_requant_kernel(int8_t* __restrict__ wq, int64_t units, const float* __restrict__ scales,
                         const __grid_constant__ MaxScaleParts parts, float* __restrict__ s_out, int32_t* st) {
  __shared__ int8_t lut[kMaxScaleParts][256];
  __shared__ float sh_max;
  __shared__ int sh_ok;
  const int P = parts.P;
  if (threadIdx.x < 32) {
    float m = 0.f;
    bool ok = true;
    for (int p = threadIdx.x; p < P; p += 32) {
      const float v = scales[p];
      ok &= (v > 0.f) && (v <= 3.402823466e38f);
      m = fmaxf(m, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    ok = __all_sync(0xffffffffu, ok);
    if (threadIdx.x == 0) {
      sh_max = m;
      sh_ok = ok ? 1 : 0;
    }
  }
  __syncthreads();
  if (!sh_ok) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report_status(st, W8A8_ERR_BAD_SCALE);
    return;
  }
  const float smax = sh_max;
  for (int i = threadIdx.x; i < P * 256; i += kMsThreads) {
    const int p = i >> 8;
    const float c = (float)(int)(int8_t)(uint8_t)(i & 255);  // the code whose byte is i & 255
    const int n = __float2int_rn(__fdiv_rn(__fmul_rn(c, scales[p]), smax));
    lut[p][i & 255] = (int8_t)min(127, max(-127, n));
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *s_out = smax;
  __syncthreads();
  const int64_t stride = (int64_t)gridDim.x * kMsThreads * kMsUnroll;
  for (int64_t u0 = (int64_t)blockIdx.x * kMsThreads * kMsUnroll + threadIdx.x; u0 < units; u0 += stride) {
    if (VEC) {
      uint4 v[kMsUnroll];
#pragma unroll
      for (int j = 0; j < kMsUnroll; ++j) {
        const int64_t u = u0 + (int64_t)j * kMsThreads;
        if (u < units) v[j] = *reinterpret_cast<const uint4*>(wq + u * 16);
      }
#pragma unroll
      for (int j = 0; j < kMsUnroll; ++j) {
        const int64_t u = u0 + (int64_t)j * kMsThreads;
        if (u < units) {
          int p = 0;
          while (p + 1 < P && u >= parts.end[p]) ++p;
          const int8_t* t = lut[p];
          *reinterpret_cast<uint4*>(wq + u * 16) =
              make_uint4(lut_map4(t, v[j].x), lut_map4(t, v[j].y), lut_map4(t, v[j].z), lut_map4(t, v[j].w));
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < kMsUnroll; ++j) {
        const int64_t u = u0 + (int64_t)j * kMsThreads;
        if (u < units) {
          int p = 0;
          while (p + 1 < P && u >= parts.end[p]) ++p;
          wq[u] = lut[p][(uint8_t)wq[u]];
        }
      }
    }
  }
}

cudaError_t requant_max_scale(int8_t* wq, int64_t units, const float* scales, const MaxScaleParts& parts,
                              float* s_out, int32_t* st, cudaStream_t stream) {
  static thread_local int s_dev = -1, s_sms = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev != s_dev) {
    e = cudaDeviceGetAttribute(&s_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    s_dev = dev;
  }
  // enough CTAs for every unit in one sweep, at most 8 per SM (each builds its own table)
  const int64_t need = (units + kMsThreads * kMsUnroll - 1) / (kMsThreads * kMsUnroll);
  const int64_t cap = (int64_t)s_sms * 8;
  const unsigned grid = (unsigned)(need < 1 ? 1 : (need < cap ? need : cap));
  if (parts.vec)
    max_scale_requant_kernel<true><<<grid, kMsThreads, 0, stream>>>(wq, units, scales, parts, s_out, st);
  else
    max_scale_requant_kernel<false><<<grid, kMsThreads, 0, stream>>>(wq, units, scales, parts, s_out, st);
  return cudaGetLastError();
}

int requant_path(const uint8_t* w, const int8_t* q, int64_t K) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(q);
  if (K % 16 == 0 && (a & 15) == 0) return 1;
  if (K % 4 == 0 && K <= kReqWordMaxK && (a & 3) == 0) return 2;
  return 0;
}

#ifdef W8A8_DEBUG
cudaError_t debug_register_requant(int32_t* word) { return w8a8_debug_register_here(word); }
#endif

}  // namespace w8a8

extern "C" w8a8_status w8a8_test_requant_wait_fault(uint32_t extra_tx_bytes, uint64_t wait_limit_ns) {
  if (extra_tx_bytes > 4096 || (wait_limit_ns != 0 && (wait_limit_ns < 100000ull || wait_limit_ns > 2000000000ull)))
    return W8A8_ERR_INVALID_ARG;
  w8a8::g_ring_extra_tx.store(extra_tx_bytes, std::memory_order_relaxed);
  w8a8::g_ring_limit_ns.store(wait_limit_ns ? wait_limit_ns : 2000000000ull, std::memory_order_relaxed);
  return W8A8_OK;
}
