// INT8 x INT8 -> INT32 GEMM on the sm_103a tensor cores, with the scale/azp/bias epilogue
// fused ("[SGLang] W4A8, W8A8, W4A4", item 3: int8_scaled_mm; item 4: azp_adj).
//
// Engine.  GB300 has no integer tcgen05 MMA kind, and its legacy s8 warp MMA runs at a
// small fraction of the fp16 tensor rate.  Every int8 value is exact in fp16, every
// product of two is an integer of magnitude <= 128*128, and an fp32 sum of such integers
// is exact while every partial sum stays within 2^24.  So the products run as
// fp16 x fp16 -> fp32 `tcgen05.mma .kind::f16` into TMEM, and exactness is guaranteed per
// output tile in one of two ways:
//   - single pass: if every activation row r of the tile has sum_k |a[r,k]| < 2^17, then
//     |any partial sum| <= 2^17 * 128 = 2^24 and the fp32 accumulator over the whole K is
//     exact (the activation producer writes these row L1 norms next to the fp16 codes); or,
//     for asymmetric activations with the weight's row sums of squares given, if
//     ||a_r||_2 * ||w_n||_2 < 2^24 over the tile (Cauchy-Schwarz bounds every partial sum);
//   - chunked: otherwise the K loop is cut into chunks of 1024 (1024 * 128 * 128 = 2^24),
//     each chunk goes to TMEM buffer 0, and the epilogue adds the chunk's exact fp32 result
//     into an int32 running sum kept in TMEM buffer 1 (tcgen05.ld / tcgen05.st).
// Either way the result equals the int32 GEMM exactly, for any int8 data.
//
// Shape.  CTA pairs (cluster of 2, `cta_group::2`) compute 256 x 256 output tiles with
// M = 256, N = 256, K = 16 MMAs issued by one thread of the even CTA.  Each CTA holds its
// own 128 activation rows and its 128-row half of the weight tile, so a CTA converts only
// 128 x 64 weight bytes per K step.
//   activations: fp16 integer codes [rows, K] -> TMA, 128-byte swizzle, straight into the
//                MMA operand ring (6 stages x 16 KB)
//   weights:     int8 [E*N, K] -> TMA -> int8 staging ring (5 x 8 KB) -> 5 converter warps,
//                each owning every 5th K step: int8 -> fp16 (exact: 0x6400|(v^0x80) - 1152)
//                into the swizzled operand layout (5 x 16 KB)
//   accumulator: two 256-column TMEM buffers per CTA, alternating per single-pass tile
//   epilogue:    8 warps per CTA read TMEM, apply y = bf16((s_x*s_w) * f32(acc - zp*azp_adj)
//                + bias), store.
// The pair is persistent and walks a static list of (segment, row tile, column tile) work
// items, so grouped (MoE) and dense launches are the same kernel.
//
// Under-filled launches.  A dense launch with fewer tiles than two waves of pairs (a few
// hundred tokens or less) leaves pairs idle for most of its run.  Given scratch, the tiles
// past its first full wave (all of them when there is none) are cut along K at 1024-element
// boundaries into parts that run on the idle pairs (a separate instantiation, so launches
// that do not split run the kernel without this code).  A part is a run of whole chunks, so
// its sums are exact by the argument above; it stores them as an int32 partial tile, and a
// second kernel adds the parts and applies the same epilogue: the integer is the same, so is
// the output.
//
// Every wait is bounded in time: a wait that runs out records W8A8_ERR_TIMEOUT, raises a
// CTA-wide abort flag, and all roles leave their loops; each CTA then waits (bounded) for
// its own outstanding TMA copies and MMAs, both CTAs meet at a cluster barrier, and TMEM is
// released.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace w8a8 {
namespace tc {

constexpr int BM = 256;        // activation rows per pair tile
constexpr int BM_CTA = 128;    // activation rows per CTA
constexpr int BN = 256;        // weight rows (output columns) per pair tile
constexpr int BN_CTA = 128;    // weight rows converted and held per CTA
constexpr int BK = 64;
constexpr int SA = 6;          // activation ring (fp16 tiles straight from TMA)
constexpr int CONV_WARPS = 5;  // converter warp w owns the K steps it with it % 5 == w
constexpr int SB = CONV_WARPS; // converted weight ring: slot w belongs to converter warp w
constexpr int S8 = CONV_WARPS; // int8 weight staging ring: slot w belongs to converter warp w
constexpr int CHUNK_STEPS = 16;   // 16 * 64 = 1024 K per exact fp32 chunk
constexpr int32_t kNormSingle = 131072;  // row L1 norm below 2^17 -> single pass is exact
constexpr int A16 = BM_CTA * BK * 2;     // 16 KB
constexpr int B16 = BN_CTA * BK * 2;     // 16 KB
constexpr int B8 = BN_CTA * BK;          // 8 KB
constexpr int OFF_B16 = SA * A16;
constexpr int OFF_B8 = OFF_B16 + SB * B16;
constexpr int DATA_BYTES = OFF_B8 + S8 * B8;
constexpr int MAX_SEG = 1024;
constexpr int NUM_THREADS = 512;
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;

struct __align__(8) Bars {
  uint64_t full_a[SA];     // activation tile landed (TMA tx)
  uint64_t stepdone[SA];   // the MMAs of step it (it % SA) finished: frees its activation slot and
                           // its converted weight slot (one multicast commit per step)
  uint64_t full16[SB];     // both CTAs' operands of the step ready (leader only; 2 arrivals)
  uint64_t full8[S8];      // int8 weight tile landed (TMA tx)
  uint64_t empty8[S8];     // converter done reading the int8 tile
  uint64_t accfull[2];     // accumulator buffer ready (multicast commit)
  uint64_t accempty[2];    // both CTAs drained the buffer (leader only; 2 x EPI_WARPS arrivals)
  uint64_t mma_done;
  uint64_t qfull[4];       // work-item queue (rank 0): entry written by warp 5
  uint64_t qempty[4];      // entry read by the MMA thread
  uint32_t tmem_base;
  int32_t abort;
  int32_t tiles_total;
  int32_t pad;
  int32_t qsingle[4];
  int32_t qpad[4];
  int64_t qrow0[4], qrow_end[4], qn0[4];
  int32_t qe[4], qkb0[4], qkb1[4], qtail[4], qpart[4];
  int32_t tile_prefix[MAX_SEG + 1];
};

constexpr size_t SMEM_BYTES = 1024 + DATA_BYTES + sizeof(Bars);
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// shared::cluster address of the same shared variable in CTA `rank` of this cluster
__device__ __forceinline__ uint32_t map_to(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_arrive_local(uint64_t* b) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n" ::"r"(su32(b)) : "memory");
}
// Arrive on a barrier given by its shared::cluster address (own CTA or the peer).
// CTA-scope release: everything a CTA publishes to its peer this way lives in the
// publishing CTA's own shared memory (converted weight tiles, landed activation tiles) or
// TMEM, and is handed to the tensor-core (async) proxy by fence.proxy.async /
// tcgen05.fence before the arrive.  A cluster-scope release would add a fence costing
// ~1.6k cycles per arrive on this part without ordering anything more that the MMA needs.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];\n" ::"r"(caddr) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Bounded wait.  Returns false (after recording a timeout and raising the abort flag) if
// the phase did not complete within the limit, or if another role of this CTA aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* b, uint32_t parity, Bars* bars, int32_t* status) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(b, parity)) return true;
    if ((i & 63) == 0) {
      if (*(volatile int32_t*)&bars->abort) return false;
      if (gtimer() - t0 > kWaitLimitNs) {
        *(volatile int32_t*)&bars->abort = 1;
        report_status(status, W8A8_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// bounded wait used on the exit path (no abort short-cut)
__device__ __forceinline__ void drain_wait(uint64_t* b, uint32_t parity, int32_t* status) {
  const uint64_t t0 = gtimer();
  while (!mbar_try(b, parity)) {
    if (gtimer() - t0 > kWaitLimitNs) {
      report_status(status, W8A8_ERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          su32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(su32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset: unused for swizzled K-major
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;            // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}

// kind::f16, A = B = fp16, D = fp32, both K-major, M = 256 (pair), N = 256
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f16_pair(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(kIdesc), "r"(accumulate));
}
// arrive once on the barrier at this offset in both CTAs when all prior MMAs complete
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  const uint16_t mask = 0x3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(
          su32(bar)),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const int32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
      "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
      "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// ------------------------------------------------------------------ work list
struct Tile {
  int e;
  int64_t row0, row_end, n0;
};

__device__ __forceinline__ Tile decode_tile(int t, const Bars* bars, int E, const int64_t* seg, int64_t rows) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bars->tile_prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int local = t - bars->tile_prefix[lo];
  const int64_t s0 = seg ? seg[lo] : 0;
  const int64_t s1 = seg ? seg[lo + 1] : rows;
  const int64_t ntm = (s1 - s0 + BM - 1) / BM;
  Tile r;
  r.e = lo;
  r.row0 = s0 + (int64_t)(local % ntm) * BM;
  r.row_end = s1;
  r.n0 = (int64_t)(local / ntm) * BN;
  (void)W8A8_DOK(lo >= 0 && lo < E && r.row0 < r.row_end && r.row_end <= rows, 301);
  return r;
}

struct KParams {
  int64_t rows, N, K;
  int E;
  const int64_t* seg;
  const int32_t* norms;  // [rows] sum_k |a[r, k]|
  const int32_t* asq;    // [rows] sum_k a[r, k]^2, or null (dense GEMMs with weight squares only)
  const int32_t* wsq;    // [N] sum_k w[n, k]^2, or null
  int az_small;          // 127 * K < 2^22: every azp_adj = sum_k w[n, k] is below 2^22 in magnitude
  int dp_units;          // split launches: work items that are whole tiles (the first)
  int split;             // split launches: parts per remaining tile
  int32_t* partials;     // split launches: [split tiles][split][BM][BN] int32 partial sums
  EpiParams ep;
  __nv_bfloat16* y;
  int32_t* status;
};

// One work item: a whole tile (tail < 0) or part `part` of split tile `tail`, over the K
// steps [kb0, kb1).  Parts start on chunk boundaries and each holds at least one chunk.
struct Work {
  Tile tl;
  int kb0, kb1, tail, part;
};

template <bool SPLIT>
__device__ __forceinline__ Work decode_work(int u, const Bars* bars, const KParams& p, int nkb) {
  Work w;
  int t = u;
  w.tail = -1;
  w.part = 0;
  w.kb0 = 0;
  w.kb1 = nkb;
  if constexpr (SPLIT) {
    if (u >= p.dp_units) {
      const int v = u - p.dp_units;
      w.tail = v / p.split;
      w.part = v - w.tail * p.split;
      t = p.dp_units + w.tail;
      const int nch = (nkb + CHUNK_STEPS - 1) / CHUNK_STEPS;
      w.kb0 = CHUNK_STEPS * (w.part * nch / p.split);
      w.kb1 = min(nkb, CHUNK_STEPS * ((w.part + 1) * nch / p.split));
    }
  }
  w.tl = decode_tile(t, bars, p.E, p.seg, p.rows);
  return w;
}

// Whether the pair tile starting at row0 can run single pass (warp-wide, all lanes agree).
// Every partial sum of the fp32 accumulation is an integer bounded by sum_k |a_k| |w_k|, so
// the pass is exact when that bound stays below 2^24.  Two bounds: 127 * (row L1 norm), i.e.
// a norm below 2^17; or, when the weight's sums of squares are given (the activation format
// always carries the rows'; grouped weights are indexed by expert), Cauchy-Schwarz:
// ||a||_2 ||w||_2 < 2^24,
// tested exactly as max_rows(sum a^2) * max_cols(sum w^2) < 2^48 in 64-bit integers.  The
// second is only evaluated when the first fails.
__device__ __forceinline__ bool tile_single_pass(const KParams& p, const Tile& tl, int lane) {
  int32_t mx = 0;
#pragma unroll
  for (int j = 0; j < BM / 32; ++j) {
    const int64_t r = tl.row0 + lane + 32 * j;
    if (r < tl.row_end) mx = max(mx, p.norms[r]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (mx < kNormSingle || !p.asq) return mx < kNormSingle;
  int32_t mq = 0, mw = 0;
#pragma unroll
  for (int j = 0; j < BM / 32; ++j) {
    const int64_t r = tl.row0 + lane + 32 * j;
    if (r < tl.row_end) mq = max(mq, p.asq[r]);
  }
#pragma unroll
  for (int j = 0; j < BN / 32; ++j) {
    const int64_t n = tl.n0 + lane + 32 * j;
    if (n < p.N) mw = max(mw, p.wsq[(int64_t)tl.e * p.N + n]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mq = max(mq, __shfl_xor_sync(0xffffffffu, mq, o));
    mw = max(mw, __shfl_xor_sync(0xffffffffu, mw, o));
  }
  return (uint64_t)(uint32_t)mq * (uint64_t)(uint32_t)mw < (1ull << 48);
}

template <bool SPLIT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const KParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ringA = smem;
  uint8_t* ringB16 = smem + OFF_B16;
  uint8_t* ring8 = smem + OFF_B8;
  Bars* bars = reinterpret_cast<Bars*>(smem + DATA_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = (int)cluster_id();
  const int npairs = (int)cluster_count();
  const int nt_n = (int)((p.N + BN - 1) / BN);
  const int nkb = (int)((p.K + BK - 1) / BK);

  if (threadIdx.x == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(&bars->full_a[i], 1);
      mbar_init(&bars->stepdone[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&bars->full16[i], 2);
    }
    for (int i = 0; i < S8; ++i) {
      mbar_init(&bars->full8[i], 1);
      mbar_init(&bars->empty8[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->accfull[i], 1);
      mbar_init(&bars->accempty[i], 2 * EPI_WARPS);
    }
    mbar_init(&bars->mma_done, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars->qfull[i], 1);
      mbar_init(&bars->qempty[i], 1);
    }
    bars->abort = 0;
    int acc = 0;
    for (int e = 0; e < p.E; ++e) {
      bars->tile_prefix[e] = acc;
      const int64_t s0 = p.seg ? p.seg[e] : 0;
      const int64_t s1 = p.seg ? p.seg[e + 1] : p.rows;
      const int64_t len = s1 > s0 ? s1 - s0 : 0;
      acc += (int)((len + BM - 1) / BM) * nt_n;
    }
    bars->tile_prefix[p.E] = acc;
    bars->tiles_total = acc;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(&bars->tmem_base)),
                 "r"(TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive or multicast commit
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const int tiles = bars->tiles_total;
  const int units = SPLIT ? p.dp_units + (tiles - p.dp_units) * p.split : tiles;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (each CTA)
    if (lane == 0) {
      uint32_t nb = 0, na = 0;  // weight / activation copies issued
      bool ok = true;
      for (int t = pair; t < units && ok; t += npairs) {
        const Work wk = decode_work<SPLIT>(t, bars, p, nkb);
        const Tile& tl = wk.tl;
        const int32_t arow = (int32_t)(tl.row0 + BM_CTA * rank);
        const int32_t brow = (int32_t)((int64_t)tl.e * p.N + tl.n0 + BN_CTA * rank);
        for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
          const uint32_t sa = na % SA, pha = (na / SA) & 1;
          if (!wait_bar(&bars->stepdone[sa], pha ^ 1, bars, p.status)) { ok = false; break; }
          mbar_expect_tx(&bars->full_a[sa], A16);
          tma_load_2d(ringA + sa * A16, &tmA, kb * BK, arow, &bars->full_a[sa]);
          ++na;
          const uint32_t s8 = nb % S8, ph8 = (nb / S8) & 1;
          if (!wait_bar(&bars->empty8[s8], ph8 ^ 1, bars, p.status)) { ok = false; break; }
          mbar_expect_tx(&bars->full8[s8], B8);
          tma_load_2d(ring8 + s8 * B8, &tmB, kb * BK, brow, &bars->full8[s8]);
          ++nb;
        }
      }
      // every issued copy must land before the CTA may exit
      for (uint32_t j = (nb > (uint32_t)S8 ? nb - S8 : 0); j < nb; ++j)
        drain_wait(&bars->full8[j % S8], (j / S8) & 1, p.status);
      for (uint32_t j = (na > (uint32_t)SA ? na - SA : 0); j < na; ++j)
        drain_wait(&bars->full_a[j % SA], (j / SA) & 1, p.status);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    // Accumulator buffers: a single-pass tile takes the next buffer (alternating, so its
    // epilogue overlaps the following tile's MMAs).  A chunked tile takes both: buffer 0
    // receives each 1024-K chunk, buffer 1 is the epilogue's int32 running sum.  Every
    // acquisition of a buffer waits for the epilogue's release of the previous one.
    // The issuing thread is on the critical path (a cta_group::2 MMA costs ~45 cycles to issue
    // and a commit ~44): the loop keeps its ring positions as counters, builds descriptors by
    // adding offsets to precomputed bases, and commits once per step.
    if (rank == 0) {
      uint32_t nbuf = 0;
      uint32_t acq0 = 0u, acq1 = 0u;  // acquisitions of buffer 0 / 1 so far
      uint32_t sa = 0, sb = 0, phb = 0;  // next step: activation slot, weight slot and its phase
      const uint64_t adesc0 = desc_sw128(su32(ringA)), bdesc0 = desc_sw128(su32(ringB16));
      bool ok = true;
      uint32_t nq = 0;
      for (int t = pair; t < units && ok; t += npairs) {
        if (lane == 0) {
          const uint32_t qs = nq & 3;
          if (!wait_bar(&bars->qfull[qs], (nq >> 2) & 1, bars, p.status)) { ok = false; }
          Work wk;
          wk.tl.e = bars->qe[qs];
          wk.tl.row0 = bars->qrow0[qs];
          wk.tl.row_end = bars->qrow_end[qs];
          wk.tl.n0 = bars->qn0[qs];
          wk.kb0 = bars->qkb0[qs];
          wk.kb1 = bars->qkb1[qs];
          wk.tail = bars->qtail[qs];
          wk.part = bars->qpart[qs];
          const bool single = bars->qsingle[qs] != 0;
          mbar_arrive_local(&bars->qempty[qs]);
          ++nq;
          const int nsteps = ok ? wk.kb1 - wk.kb0 : 0;
          const int spc = single ? nsteps : CHUNK_STEPS;
          uint32_t b = 0;
          if (single) {
            b = nbuf;
            nbuf ^= 1u;
          } else {
            if (!wait_bar(&bars->accempty[1], (acq1 & 1) ^ 1, bars, p.status)) ok = false;
            ++acq1;
          }
          const uint32_t dcol = tmem + b * BN;
          int kc = 0;  // step within the current chunk (the whole item when single)
          for (int kr = 0; kr < nsteps && ok; ++kr) {
            if (kc == 0) {
              const uint32_t a = b ? acq1 : acq0;
              if (!wait_bar(&bars->accempty[b], (a & 1) ^ 1, bars, p.status)) { ok = false; break; }
              if (b) ++acq1; else ++acq0;
              tc_fence_after();
            }
            if (!wait_bar(&bars->full16[sb], phb, bars, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t ad = adesc0 + (uint64_t)(sa * (A16 >> 4));
            const uint64_t bd = bdesc0 + (uint64_t)(sb * (B16 >> 4));
            mma_f16_pair(dcol, ad, bd, kc != 0 ? 1u : 0u);
            mma_f16_pair(dcol, ad + 2, bd + 2, 1u);
            mma_f16_pair(dcol, ad + 4, bd + 4, 1u);
            mma_f16_pair(dcol, ad + 6, bd + 6, 1u);
            mma_commit_pair(&bars->stepdone[sa]);
            if (++kc == spc || kr == nsteps - 1) {
              mma_commit_pair(&bars->accfull[b]);
              kc = 0;
            }
            if (++sa == SA) sa = 0;
            if (++sb == SB) { sb = 0; phb ^= 1u; }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (lane == 0) {
        // all MMAs issued by this thread complete before TMEM is released
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                         su32(&bars->mma_done))
                     : "memory");
        drain_wait(&bars->mma_done, 0, p.status);
      }
    }
  } else if (warp == 5) {
    // Planner (rank 0; warp 5 shares the MMA thread's scheduler but does little): decodes the
    // work items (segment bounds from global memory) and takes their single-pass decisions
    // (the rows' norms) ahead of the MMA thread, which reads them from a 4-entry queue, so
    // those global-memory round trips leave the issue path at tile boundaries (MoE layer
    // 602 -> 590 us, o projection 111 -> 108 us).
    if (rank == 0) {
      uint32_t nq = 0;
      bool ok = true;
      for (int t = pair; t < units && ok; t += npairs) {
        const Work wk = decode_work<SPLIT>(t, bars, p, nkb);
        const bool single = tile_single_pass(p, wk.tl, lane);
        if (lane == 0) {
          const uint32_t qs = nq & 3;
          if (!wait_bar(&bars->qempty[qs], ((nq >> 2) & 1) ^ 1, bars, p.status)) ok = false;
          else {
            bars->qe[qs] = wk.tl.e;
            bars->qrow0[qs] = wk.tl.row0;
            bars->qrow_end[qs] = wk.tl.row_end;
            bars->qn0[qs] = wk.tl.n0;
            bars->qkb0[qs] = wk.kb0;
            bars->qkb1[qs] = wk.kb1;
            bars->qtail[qs] = wk.tail;
            bars->qpart[qs] = wk.part;
            bars->qsingle[qs] = single ? 1 : 0;
            mbar_arrive_local(&bars->qfull[qs]);
          }
        }
        ++nq;
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
  } else if (warp < 8) {
    // ---------------------------------------------------------------- converters (each CTA)
    // Converter w (warps 2, 3, 4, 6, 7) converts whole K steps it = w, w + 5, ...: the
    // 128 x 64 int8 weight tile of the step (int8 slot w) into the fp16 operand layout (fp16
    // slot w), so five steps are in flight at once and the per-step synchronisation latency
    // overlaps.  The K loop is bound by the hand-off between these warps and the one
    // MMA-issuing thread (warp 1), not by the conversion itself: keeping the converters off
    // warp 1's scheduler partition and a fifth step in flight shortened it (gate_up at
    // M = 4096: 643 -> 589 us).
    const int cw = warp == 2 ? 0 : warp == 3 ? 1 : warp == 4 ? 2 : warp == 6 ? 3 : 4;
    const uint32_t full16_leader = map_to(su32(&bars->full16[cw]), 0);
    const uint8_t* src = ring8 + cw * B8;
    uint8_t* dst = ringB16 + cw * B16;
    uint32_t it = 0;  // global step counter (same sequence as the producer and the MMA)
    uint32_t use = 0; // how many steps this warp has converted
    bool ok = true;
    for (int t = pair; t < units && ok; t += npairs) {
      const Work wk = decode_work<SPLIT>(t, bars, p, nkb);
      for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it) {
        if ((int)(it % CONV_WARPS) != cw) continue;
        const uint32_t ph = use & 1;
        ++use;
        // every lane waits; the outcome is made warp-uniform so the warp stays converged
        if (!__all_sync(0xffffffffu, wait_bar(&bars->full8[cw], ph, bars, p.status))) { ok = false; break; }
        // 512 units of 16 int8 (128 rows x 4): 16 per lane, in two batches of 8 loads each.
        // The compiler cannot move loads of the int8 slot above stores into the fp16 slot,
        // so every batch costs a shared-memory latency: few, large batches, and the first
        // issued before the wait for the fp16 slot, whose latency then hides it.
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int u = lane + 32 * i;
          v[i] = *reinterpret_cast<const uint4*>(src + (u >> 2) * 64 + (u & 3) * 16);
        }
        // the slot's previous use, step it - SB, must be finished
        if (it >= (uint32_t)SB) {
          const uint32_t j = it - SB;
          if (!__all_sync(0xffffffffu, wait_bar(&bars->stepdone[j % SA], (j / SA) & 1, bars, p.status))) {
            ok = false;
            break;
          }
        }
#pragma unroll
        for (int bt = 0; bt < 2; ++bt) {
          if (bt == 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int u = lane + 32 * (8 + i);
              v[i] = *reinterpret_cast<const uint4*>(src + (u >> 2) * 64 + (u & 3) * 16);
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int u = lane + 32 * (8 * bt + i);
            const int r = u >> 2, sgm = u & 3;
            uint32_t o[8];
            i8x4_to_f16x4(v[i].x, o[0], o[1]);
            i8x4_to_f16x4(v[i].y, o[2], o[3]);
            i8x4_to_f16x4(v[i].z, o[4], o[5]);
            i8x4_to_f16x4(v[i].w, o[6], o[7]);
            uint8_t* rowp = dst + r * 128;
            *reinterpret_cast<uint4*>(rowp + (((2 * sgm) ^ (r & 7)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(rowp + (((2 * sgm + 1) ^ (r & 7)) * 16)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_local(&bars->empty8[cw]);
          // the activation tile of this step must have landed before the pair's MMA reads it
          if (!wait_bar(&bars->full_a[it % SA], (it / SA) & 1, bars, p.status)) ok = false;
          else mbar_arrive_cluster(full16_leader);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (8 warps, each CTA)
    // Warp (q, h) owns TMEM lanes 32q..32q+31 (its CTA's rows) and columns 128h..128h+127,
    // processed in groups of 32 columns.
    const int q = warp & 3;
    const int h = (warp - 8) >> 2;
    const uint32_t accempty0 = map_to(su32(&bars->accempty[0]), 0);
    const uint32_t accempty1 = map_to(su32(&bars->accempty[1]), 0);
    const uint32_t lanebase = tmem + ((uint32_t)(q * 32) << 16) + h * 128;
    uint32_t nbuf = 0;
    uint32_t filled0 = 0u, filled1 = 0u;  // fills of buffer 0 / 1 consumed so far
    bool ok = true;
    for (int t = pair; t < units && ok; t += npairs) {
      const Work wk = decode_work<SPLIT>(t, bars, p, nkb);
      const Tile& tl = wk.tl;
      const bool single = tile_single_pass(p, tl, lane);
      const int rloc = BM_CTA * (int)rank + q * 32 + lane;  // row within the pair tile
      const int64_t m = tl.row0 + rloc;
      const bool row_ok = m < tl.row_end;
      EpiParams ep = p.ep;
      if (ep.w_mode == W8A8_W_CHANNEL) ep.s_w = p.ep.s_w + (int64_t)tl.e * p.N;
      const float sx = row_ok ? epi_row_scale(ep, m) : 0.f;
      const int zpm = row_ok ? epi_row_zp(ep, m) : 0;
      const int64_t nb = tl.n0 + h * 128;
      __nv_bfloat16* yrow = p.y + (row_ok ? m : 0) * p.N;
      const int nch = single ? 1 : (wk.kb1 - wk.kb0 + CHUNK_STEPS - 1) / CHUNK_STEPS;
      const uint32_t b = single ? nbuf : 0u;
      if (single) nbuf ^= 1u;
      // Single-pass tiles: every fp32 accumulator is the exact integer (|acc| <= 2^24), which is
      // also f32(acc), so y follows from it without the int32/int64 round trip; per-channel
      // scales and bias are read 16 bytes at a time.  Dynamic asymmetric rows need
      // f32(acc - zp*azp_adj): acc, zp and azp_adj (|azp_adj| <= 127*K < 2^24) are exact floats,
      // so one fma rounds the exact difference once, as the integer path does (rows with
      // |zp| >= 2^24, which bf16 inputs never produce, take the integer form).
      const bool dyn_asym = ep.act_mode == W8A8_ACT_DYN_TOKEN_ASYM;
      const bool direct = single && wk.tail < 0 && (ep.act_mode == W8A8_ACT_DYN_TOKEN_SYM ||
                                     ep.act_mode == W8A8_ACT_STATIC_TENSOR_SYM || dyn_asym);
      const bool zp_exact = zpm > -16777216 && zpm < 16777216;
      const float zpf = (float)zpm;
      const bool azp_vec = dyn_asym && (reinterpret_cast<uintptr_t>(ep.azp) & 15) == 0;
      const bool sw_vec = ep.w_mode == W8A8_W_CHANNEL && (reinterpret_cast<uintptr_t>(ep.s_w) & 15) == 0;
      const bool bias_vec = ep.bias && (reinterpret_cast<uintptr_t>(ep.bias) & 15) == 0;
      for (int c = 0; c < nch; ++c) {
        const uint32_t fcount = b ? filled1 : filled0;
        if (!__all_sync(0xffffffffu, wait_bar(&bars->accfull[b], fcount & 1, bars, p.status))) {
          ok = false;
          break;
        }
        if (b) ++filled1; else ++filled0;
        tc_fence_after();
        const bool last = (c == nch - 1);
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          uint32_t r[32];
          tmem_ld32(lanebase + b * BN + g * 32, r);
          if (direct) {
            tmem_ld_wait();
            if (!row_ok) continue;
            const int64_t n0 = nb + g * 32;
            if (((p.N & 7) == 0) && n0 + 32 <= p.N && (sw_vec || ep.w_mode != W8A8_W_CHANNEL) &&
                (!ep.bias || bias_vec) && (!dyn_asym || azp_vec)) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float sw[8], bb[8];
                if (ep.w_mode == W8A8_W_CHANNEL) {
                  const float4 a0 = __ldg(reinterpret_cast<const float4*>(ep.s_w + n0 + 8 * j));
                  const float4 a1 = __ldg(reinterpret_cast<const float4*>(ep.s_w + n0 + 8 * j + 4));
                  sw[0] = a0.x; sw[1] = a0.y; sw[2] = a0.z; sw[3] = a0.w;
                  sw[4] = a1.x; sw[5] = a1.y; sw[6] = a1.z; sw[7] = a1.w;
                } else {
#pragma unroll
                  for (int i = 0; i < 8; ++i) sw[i] = ep.s_w[0];
                }
                if (ep.bias) {
                  const uint4 bv = __ldg(reinterpret_cast<const uint4*>(ep.bias + n0 + 8 * j));
                  const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    bb[2 * i] = bf16_lo(bw[i]);
                    bb[2 * i + 1] = bf16_hi(bw[i]);
                  }
                }
                float cf[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) cf[i] = __uint_as_float(r[8 * j + i]);
                if (dyn_asym) {
                  const int4 z0 = __ldg(reinterpret_cast<const int4*>(ep.azp + n0 + 8 * j));
                  const int4 z1 = __ldg(reinterpret_cast<const int4*>(ep.azp + n0 + 8 * j + 4));
                  const int az[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
                  // acc, zp and azp_adj are exact floats here: one fma forms f32(acc - zp * azp)
                  // with a single rounding.  azp_adj below 2^22 converts exactly by adding it
                  // into the mantissa of 1.5 * 2^23 (integer add, float subtract) instead of a
                  // conversion instruction per output.
                  if (zp_exact && p.az_small) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                      cf[i] = __fmaf_rn(-zpf, __fsub_rn(__int_as_float(az[i] + 0x4B400000), 12582912.0f), cf[i]);
                  } else if (zp_exact) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) cf[i] = __fmaf_rn(-zpf, __int2float_rn(az[i]), cf[i]);
                  } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                      cf[i] = __ll2float_rn((long long)cf[i] - (long long)zpm * (long long)az[i]);
                  }
                }
                float f[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  f[i] = __fmul_rn(__fmul_rn(sx, sw[i]), cf[i]);
                  if (ep.bias) f[i] = __fadd_rn(f[i], bb[i]);
                }
                uint4 o;
                o.x = pack_bf16x2(f[0], f[1]);
                o.y = pack_bf16x2(f[2], f[3]);
                o.z = pack_bf16x2(f[4], f[5]);
                o.w = pack_bf16x2(f[6], f[7]);
                if (W8A8_DOK(m < p.rows && n0 + 8 * j + 8 <= p.N, 302)) *reinterpret_cast<uint4*>(yrow + n0 + 8 * j) = o;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (n0 + i < p.N && W8A8_DOK(m < p.rows, 303))
                  yrow[n0 + i] = __float2bfloat16_rn(epi_apply(ep, (int32_t)__uint_as_float(r[i]), sx, zpm, n0 + i));
            }
            continue;
          }
          int32_t v[32];
          if (c > 0) {
            uint32_t pr[32];
            tmem_ld32(lanebase + BN + g * 32, pr);  // running int32 sum (buffer 1)
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = (int32_t)pr[i] + __float2int_rn(__uint_as_float(r[i]));
          } else {
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float2int_rn(__uint_as_float(r[i]));
          }
          if (!last) {
            tmem_st32(lanebase + BN + g * 32, v);
          } else if (SPLIT && wk.tail >= 0) {
            if (row_ok && W8A8_DOK(wk.part < p.split && rloc < BM && wk.tail >= 0, 304)) {  // this part's int32 sums; the reduce kernel applies the epilogue
              int4* dst = reinterpret_cast<int4*>(
                  p.partials + ((size_t)(wk.tail * p.split + wk.part) * BM + rloc) * BN + h * 128 + g * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j) __stcg(dst + j, make_int4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            }
          } else if (row_ok) {
            const int64_t n0 = nb + g * 32;
            if (((p.N & 7) == 0) && n0 + 32 <= p.N) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float f[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = epi_apply(ep, v[8 * j + i], sx, zpm, n0 + 8 * j + i);
                uint4 o;
                o.x = pack_bf16x2(f[0], f[1]);
                o.y = pack_bf16x2(f[2], f[3]);
                o.z = pack_bf16x2(f[4], f[5]);
                o.w = pack_bf16x2(f[6], f[7]);
                if (W8A8_DOK(m < p.rows && n0 + 8 * j + 8 <= p.N, 305)) *reinterpret_cast<uint4*>(yrow + n0 + 8 * j) = o;
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (n0 + i < p.N && W8A8_DOK(m < p.rows, 306))
                  yrow[n0 + i] = __float2bfloat16_rn(epi_apply(ep, v[i], sx, zpm, n0 + i));
            }
          }
        }
        if (!last) tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(b ? accempty1 : accempty0);
      }
      if (!ok) break;
      if (!single) {
        // the running-sum buffer is free again
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(accempty1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrive or MMA can target a CTA that has left
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(TMEM_COLS));
  }
}

// int8 -> fp16 integer codes, row L1 norms and row sums of squares (the GEMM-ready
// activation format: norms[row], then norms[gridDim.x + row] for the squares)
__global__ void __launch_bounds__(256)
to_gemm_ready_kernel(const int8_t* __restrict__ a, int64_t K, __half* __restrict__ a16, int32_t* __restrict__ norms) {
  __shared__ int sh[8], sh2[8];
  const int64_t row = blockIdx.x;
  int s = 0, s2 = 0;
  const int8_t* ar = a + row * K;
  __half* hr = a16 + row * K;
  for (int64_t i = threadIdx.x; i < K / 16; i += 256) {
    const uint4 v = reinterpret_cast<const uint4*>(ar)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      i8x4_to_f16x4(w[j], o[2 * j], o[2 * j + 1]);
#pragma unroll
      for (int b = 0; b < 4; ++b) s += abs((int)(int8_t)(w[j] >> (8 * b)));
      s2 = __dp4a((int)w[j], (int)w[j], s2);
    }
    reinterpret_cast<uint4*>(hr)[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<uint4*>(hr)[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    s2 += __shfl_xor_sync(0xffffffffu, s2, o);
  }
  if ((threadIdx.x & 31) == 0) {
    sh[threadIdx.x >> 5] = s;
    sh2[threadIdx.x >> 5] = s2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0, t2 = 0;
    for (int i = 0; i < 8; ++i) {
      t += sh[i];
      t2 += sh2[i];
    }
    norms[row] = t;
    norms[gridDim.x + row] = t2;
  }
}

// The split tiles of a split launch: add each output's K parts and apply the epilogue.
// Block b covers 8 rows of split tile b / (BM / 8); thread (row, 8-column group).
__global__ void __launch_bounds__(256)
split_reduce_kernel(const int32_t* __restrict__ partials, int dp_units, int split, int64_t rows, int64_t N,
                    const EpiParams ep, __nv_bfloat16* __restrict__ y) {
  const int tt = blockIdx.x / (BM / 8);
  const int r = (blockIdx.x % (BM / 8)) * 8 + (threadIdx.x >> 5);
  const int c = (threadIdx.x & 31) * 8;
  const int64_t t = dp_units + tt;
  const int64_t ntm = (rows + BM - 1) / BM;
  const int64_t m = (t % ntm) * BM + r;
  const int64_t n0 = (t / ntm) * BN + c;
  if (m >= rows || n0 >= N) return;
  if (!W8A8_DOK(r < BM && c + 8 <= BN, 307)) return;
  const int32_t* src = partials + ((size_t)tt * split * BM + r) * BN + c;
  int32_t v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = 0;
  for (int s = 0; s < split; ++s) {
    const int4 a = __ldcg(reinterpret_cast<const int4*>(src + (size_t)s * BM * BN));
    const int4 b = __ldcg(reinterpret_cast<const int4*>(src + (size_t)s * BM * BN + 4));
    v[0] += a.x;
    v[1] += a.y;
    v[2] += a.z;
    v[3] += a.w;
    v[4] += b.x;
    v[5] += b.y;
    v[6] += b.z;
    v[7] += b.w;
  }
  const float sx = epi_row_scale(ep, m);
  const int zpm = epi_row_zp(ep, m);
  __nv_bfloat16* yrow = y + m * N;
  if (((N & 7) == 0) && n0 + 8 <= N) {
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = epi_apply(ep, v[i], sx, zpm, n0 + i);
    uint4 o;
    o.x = pack_bf16x2(f[0], f[1]);
    o.y = pack_bf16x2(f[2], f[3]);
    o.z = pack_bf16x2(f[4], f[5]);
    o.w = pack_bf16x2(f[6], f[7]);
    *reinterpret_cast<uint4*>(yrow + n0) = o;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (n0 + i < N) yrow[n0 + i] = __float2bfloat16_rn(epi_apply(ep, v[i], sx, zpm, n0 + i));
  }
}

}  // namespace tc

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

static bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int64_t rows, int64_t K,
                     uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * (cuuint64_t)esize};
  cuuint32_t box[2] = {(cuuint32_t)tc::BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int gemm_tc_max_segments() { return tc::MAX_SEG; }

namespace {

// Work decomposition of a dense launch on `pairs_max` CTA pairs: the tiles past the last
// full wave (all of them when there is none) are cut into `split` parts, as many as fill the
// pairs that wave would leave idle, at most one per chunk.  The 6144-column layer at
// M = 4096, for instance, has 384 tiles on 76 pairs: five full waves and 4 tiles, which now
// run as 16 quarter-K parts instead of a sixth wave with 72 idle pairs.
struct SplitPlan {
  int64_t units;     // work items
  int dp_units;      // whole tiles (first)
  int split;         // parts per remaining tile (1: no split)
  int64_t tail;      // split tiles
  size_t partial_bytes;
};

SplitPlan plan_dense(int64_t rows, int64_t N, int64_t K, int64_t pairs_max) {
  SplitPlan s{};
  const int64_t tiles = ((rows + tc::BM - 1) / tc::BM) * ((N + tc::BN - 1) / tc::BN);
  s.units = tiles;
  s.split = 1;
  if (pairs_max < 1) return s;
  const int64_t nch = ((K + tc::BK - 1) / tc::BK + tc::CHUNK_STEPS - 1) / tc::CHUNK_STEPS;
  const int64_t full = (tiles / pairs_max) * pairs_max;
  const int64_t tail = tiles - full;
  if (tail == 0) return s;
  int64_t f = pairs_max / tail;
  if (f > nch) f = nch;
  if (f < 2) return s;
  s.split = (int)f;
  s.dp_units = (int)full;
  s.tail = tail;
  s.units = full + tail * f;
  s.partial_bytes = (size_t)tail * (size_t)f * tc::BM * tc::BN * sizeof(int32_t);
  return s;
}

int sm_count(int dev) {
  static thread_local int s_dev = -1, s_sms = 0;
  if (s_dev != dev) {
    if (cudaDeviceGetAttribute(&s_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    s_dev = dev;
  }
  return s_sms;
}

}  // namespace

size_t gemm_split_bytes(int64_t rows, int64_t N, int64_t K) {
  int dev = 0;
  if (rows <= 0 || N <= 0 || K <= 0 || cudaGetDevice(&dev) != cudaSuccess) return 0;
  const SplitPlan s = plan_dense(rows, N, K, sm_count(dev) / 2);
  return s.split > 1 ? s.partial_bytes : 0;
}

cudaError_t to_gemm_ready(const int8_t* a, int64_t rows, int64_t K, void* a16, int32_t* norms, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  tc::to_gemm_ready_kernel<<<(unsigned)rows, 256, 0, st>>>(a, K, static_cast<__half*>(a16), norms);
  return cudaGetLastError();
}

cudaError_t gemm_tcgen05(const GemmArgs& g, cudaStream_t st) {
  if (g.E > tc::MAX_SEG) return cudaErrorNotSupported;
  if (g.rows == 0 || g.N == 0) return cudaSuccess;
  if (!g.a16 || !g.norms) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static thread_local int s_attr_dev = -1;
  if (s_attr_dev != dev) {
    e = cudaFuncSetAttribute(tc::gemm_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc::gemm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    s_attr_dev = dev;
  }
  const int64_t max_pairs = sm_count(dev) / 2;
  if (max_pairs < 1) return cudaErrorNotSupported;
  CUtensorMap ma, mb;
  if (!make_map(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.a16, g.rows, g.K, tc::BM_CTA,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!make_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.w, (int64_t)g.E * g.N, g.K, tc::BN_CTA,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  tc::KParams p;
  p.rows = g.rows;
  p.N = g.N;
  p.K = g.K;
  p.E = g.E;
  p.seg = g.seg;
  p.norms = g.norms;
  // the squares follow the L1 norms in the activation format (every producer writes them);
  // with the weight's squares given, tiles that fail the L1 test try Cauchy-Schwarz
  p.asq = g.wsq ? g.norms + g.rows : nullptr;
  p.wsq = g.wsq;
  p.az_small = 127 * g.K < (int64_t(1) << 22) ? 1 : 0;
  p.ep.act_mode = g.act_mode;
  p.ep.w_mode = g.w_mode;
  p.ep.s_x = g.s_x;
  p.ep.zp = g.zp;
  p.ep.azp = g.azp;
  p.ep.s_w = g.s_w;
  p.ep.bias = static_cast<const __nv_bfloat16*>(g.bias);
  p.y = static_cast<__nv_bfloat16*>(g.y);
  p.status = g.status;
  p.dp_units = 0;
  p.split = 1;
  p.partials = nullptr;
  const int64_t nt_n = (g.N + tc::BN - 1) / tc::BN;
  if (!g.seg && g.split_ws) {
    const SplitPlan s = plan_dense(g.rows, g.N, g.K, max_pairs);
    if (s.split > 1 && g.split_bytes >= s.partial_bytes) {
      p.dp_units = s.dp_units;
      p.split = s.split;
      p.partials = static_cast<int32_t*>(g.split_ws);
      const int pairs = (int)(s.units < max_pairs ? s.units : max_pairs);
      tc::gemm_tc_kernel<true><<<2 * pairs, tc::NUM_THREADS, tc::SMEM_BYTES, st>>>(ma, mb, p);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      tc::split_reduce_kernel<<<(unsigned)(s.tail * (tc::BM / 8)), 256, 0, st>>>(p.partials, s.dp_units, s.split,
                                                                                 g.rows, g.N, p.ep, p.y);
      return cudaGetLastError();
    }
  }
  const int64_t tiles_ub = g.seg ? ((g.rows + tc::BM - 1) / tc::BM + g.E) * nt_n : ((g.rows + tc::BM - 1) / tc::BM) * nt_n;
  const int pairs = (int)(tiles_ub < max_pairs ? tiles_ub : max_pairs);
  tc::gemm_tc_kernel<false><<<2 * pairs, tc::NUM_THREADS, tc::SMEM_BYTES, st>>>(ma, mb, p);
  return cudaGetLastError();
}

#ifdef W8A8_DEBUG
cudaError_t debug_register_gemm_tc(int32_t* word) { return w8a8_debug_register_here(word); }
#endif

}  // namespace w8a8
