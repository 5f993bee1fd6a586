// Tensor-engine probe for sm_103a: the numbers behind the GEMM's engine choice and the
// denominator of "% of INT8 tensor peak".  A standalone program (not part of libw8a8.so);
// built and run by engine_rates.py, which prints its JSON.
//
//   1. mma.sync.m16n8k32 s8 x s8 -> s32 (the only integer tensor-core instruction that
//      assembles for sm_103a): dense TOPS over all SMs.
//   2. tcgen05.mma.cta_group::2.kind::f16 (fp16 x fp16 -> fp32 in TMEM), M = 256: clocks per
//      MMA on one CTA pair and TFLOP/s over all SM pairs, with A from shared memory (N = 256,
//      192) and from TMEM (N = 192).
//   3. Issue costs of the single issuing thread: N = 16 MMAs (8 cycles of tensor work each),
//      alone, with two commits per four MMAs, and with a barrier poll.
//   4. Exactness of the fp32 TMEM accumulation for integer operands: K = 1024 sums of int8-
//      valued fp16 products (all partial sums below 2^24) compared with int64 host sums,
//      including all-127 rows (1024 * 127 * 127 = 16 516 096) and a +-16129 term followed
//      by +-1 terms.
// Every device wait is bounded (2 s) and only reports if it runs out.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#define CK(x)                                                                                     \
  do {                                                                                            \
    cudaError_t e_ = (x);                                                                         \
    if (e_ != cudaSuccess) {                                                                      \
      fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__);   \
      exit(1);                                                                                    \
    }                                                                                             \
  } while (0)

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ uint64_t gtime() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// returns false if the phase did not complete within 2 s
__device__ __forceinline__ bool wait_phase(uint64_t* b, uint32_t parity) {
  const uint64_t t0 = gtime();
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (gtime() - t0 > 2000000000ull) return false;
  }
}

// ------------------------------------------------------------------ 1. mma.sync s8
__global__ void __launch_bounds__(256) mma_sync_s8_kernel(int iters, int* sink) {
  int a0 = threadIdx.x * 0x01010101, a1 = a0 + 1, a2 = a0 + 2, a3 = a0 + 3, b0 = a0 ^ 0x5A5A5A5A, b1 = b0 + 7;
  int c[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) c[j][i] = 0;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      asm volatile(
          "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
          : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  int s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
  if (s == 0x7FFFFFFF) sink[0] = s;
}

// ------------------------------------------------------------------ 2/3. tcgen05 rates
// MODE bits: 1 = A from TMEM, 2 = two multicast commits per four MMAs, 4 = a barrier poll per
// four MMAs.  One thread of the even CTA issues; both CTAs wait for the final commit.
template <int N, int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1) tc_rate_kernel(int iters, unsigned long long* out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* s = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar, sbar[3];
  __shared__ uint32_t tbase;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  for (int i = threadIdx.x; i < 32768 / 4; i += 128) {
    uint32_t h = (uint32_t)i * 2654435761u + rank * 40503u;
    h ^= h >> 13;
    const __half2 v = __halves2half2(__int2half_rn((int)(h & 0xFF) - 128), __int2half_rn((int)((h >> 8) & 0xFF) - 128));
    reinterpret_cast<uint32_t*>(s)[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&bar)));
    for (int i = 0; i < 3; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&sbar[i])));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 512;\n" ::"r"(su32(&tbase)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n");
  }
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  const uint32_t tm = tbase;
  const uint32_t idesc = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
  bool ok = true;
  if (rank == 0 && threadIdx.x == 0) {
    const uint64_t da = desc_sw128(su32(s)), db = desc_sw128(su32(s + 16384));
    const uint64_t c0 = clock64(), g0 = gtime();
    for (int i = 0; i < iters; ++i) {
      if (MODE & 4) {
        uint32_t r;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 1;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(r)
            : "r"(su32(&sbar[2]))
            : "memory");
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t acc = (i | kk) ? 1u : 0u;
        if (MODE & 1)
          asm volatile(
              "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(tm),
              "r"(tm + 384 + 8 * kk), "l"(db + 2 * kk), "r"(idesc), "r"(acc));
        else
          asm volatile(
              "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tm),
              "l"(da + 2 * kk), "l"(db + 2 * kk), "r"(idesc), "r"(acc));
      }
      if (MODE & 2) {
        const uint16_t m2 = 3;
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(
                su32(&sbar[i & 1])),
            "h"(m2)
            : "memory");
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(
                su32(&sbar[2])),
            "h"(m2)
            : "memory");
      }
    }
    const uint16_t mask = 3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n" ::"r"(
            su32(&bar)),
        "h"(mask)
        : "memory");
    ok = wait_phase(&bar, 0);
    const uint64_t c1 = clock64(), g1 = gtime();
    unsigned cid;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(cid));
    out[3 * cid] = c1 - c0;
    out[3 * cid + 1] = g1 - g0;
    out[3 * cid + 2] = ok ? 0 : 1;
  } else if (rank == 1 && threadIdx.x == 0) {
    ok = wait_phase(&bar, 0);
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 512;\n" ::"r"(tm));
  }
}

// ------------------------------------------------------------------ 4. accumulation exactness
// One CTA, cta_group::1, M = 128 rows of A, N = 16 rows of B, K = 1024 in 16 slices of 64.
// A and B are int8-valued fp16 in global memory ([rows, 1024] row-major); each slice is
// written into the 128-byte-swizzled K-major layout (16-byte chunk c of row r at c ^ (r & 7)),
// then 4 MMAs of K = 16 accumulate into TMEM.  D is read back as fp32.
constexpr int EX_M = 128, EX_N = 16, EX_K = 1024;
__global__ void __launch_bounds__(128, 1) tc_exact_kernel(const __half* A, const __half* B, float* D, int* status) {
  __shared__ __align__(1024) uint8_t sa[EX_M * 128];
  __shared__ __align__(1024) uint8_t sb[EX_N * 128];
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(su32(&bar)));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;\n" ::"r"(su32(&tbase)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  const uint32_t tm = tbase;
  const uint32_t idesc = (1u << 4) | ((uint32_t)(EX_N >> 3) << 17) | ((uint32_t)(EX_M >> 4) << 24);
  bool ok = true;
  for (int sl = 0; sl < EX_K / 64; ++sl) {
    // 16-byte chunks: A has 128 rows x 8 chunks, B 16 x 8
    for (int u = threadIdx.x; u < EX_M * 8; u += 128) {
      const int r = u >> 3, c = u & 7;
      *reinterpret_cast<uint4*>(sa + r * 128 + ((c ^ (r & 7)) * 16)) =
          *reinterpret_cast<const uint4*>(A + (size_t)r * EX_K + sl * 64 + c * 8);
    }
    for (int u = threadIdx.x; u < EX_N * 8; u += 128) {
      const int r = u >> 3, c = u & 7;
      *reinterpret_cast<uint4*>(sb + r * 128 + ((c ^ (r & 7)) * 16)) =
          *reinterpret_cast<const uint4*>(B + (size_t)r * EX_K + sl * 64 + c * 8);
    }
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
      asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
      const uint64_t da = desc_sw128(su32(sa)), db = desc_sw128(su32(sb));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tm),
            "l"(da + 2 * kk), "l"(db + 2 * kk), "r"(idesc), "r"((sl | kk) ? 1u : 0u));
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(su32(&bar))
                   : "memory");
      ok = wait_phase(&bar, sl & 1) && ok;
    }
    __syncthreads();  // the operands may be overwritten once the slice's MMAs are done
  }
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(tm + ((uint32_t)(warp * 32) << 16)));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
  for (int j = 0; j < EX_N; ++j) D[(warp * 32 + lane) * EX_N + j] = __uint_as_float(r[j]);
  if (threadIdx.x == 0 && !ok) *status = 1;
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;\n" ::"r"(tm));
  }
}

// ------------------------------------------------------------------ host
template <int N, int MODE>
static void tc_rate(const char* name, int pairs, int iters, int sms, bool last) {
  unsigned long long* d;
  CK(cudaMalloc(&d, (size_t)3 * pairs * sizeof(unsigned long long)));
  auto f = tc_rate_kernel<N, MODE>;
  const int smem = 120000;  // also keeps one CTA per SM
  CK(cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  f<<<2 * pairs, 128, smem>>>(iters, d);
  CK(cudaDeviceSynchronize());
  f<<<2 * pairs, 128, smem>>>(iters, d);
  CK(cudaDeviceSynchronize());
  std::vector<unsigned long long> h(3 * pairs);
  CK(cudaMemcpy(h.data(), d, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost));
  CK(cudaFree(d));
  double clk = 0, ns = 0;
  int bad = 0;
  for (int i = 0; i < pairs; ++i) {
    clk += (double)h[3 * i];
    ns = ns > (double)h[3 * i + 1] ? ns : (double)h[3 * i + 1];
    bad += (int)h[3 * i + 2];
  }
  clk /= pairs;
  const double mmas = 4.0 * iters;
  const double tflops = 2.0 * 256 * N * 16 * mmas * pairs / ns / 1e3;
  printf("    \"%s\": {\"pairs\": %d, \"clk_per_mma\": %.1f, \"clk_per_4mma_step\": %.1f, \"ideal_clk_per_mma\": %.1f, "
         "\"tflops\": %.1f, \"sms\": %d, \"timeouts\": %d}%s\n",
         name, pairs, clk / mmas, 4 * clk / mmas, 2.0 * 256 * N * 16 / 2 / 8192.0, tflops, 2 * pairs, bad,
         last ? "" : ",");
}

int main() {
  int dev = 0, sms = 0, clock_khz = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, dev));
  cudaDeviceGetAttribute(&clock_khz, cudaDevAttrClockRate, dev);
  printf("{\n  \"gpu\": \"%s\", \"sms\": %d, \"cc\": \"%d.%d\",\n", prop.name, sms, prop.major, prop.minor);

  // 1. mma.sync s8
  {
    int* sink;
    CK(cudaMalloc(&sink, 4));
    const int iters = 20000, blocks = sms * 4;
    mma_sync_s8_kernel<<<blocks, 256>>>(100, sink);
    CK(cudaDeviceSynchronize());
    cudaEvent_t a, b;
    CK(cudaEventCreate(&a));
    CK(cudaEventCreate(&b));
    CK(cudaEventRecord(a));
    mma_sync_s8_kernel<<<blocks, 256>>>(iters, sink);
    CK(cudaEventRecord(b));
    CK(cudaEventSynchronize(b));
    float ms = 0;
    CK(cudaEventElapsedTime(&ms, a, b));
    const double ops = 2.0 * 16 * 8 * 32 * 8.0 * iters * (blocks * 8.0);
    printf("  \"mma_sync_s8_m16n8k32\": {\"tops\": %.1f, \"ms\": %.3f, \"warps\": %d},\n", ops / (ms * 1e-3) / 1e12, ms,
           blocks * 8);
    CK(cudaFree(sink));
  }

  // 2/3. tcgen05 kind::f16
  printf("  \"tcgen05_f16_cta_pair\": {\n");
  const int P = sms / 2;
  tc_rate<256, 0>("ss_n256_one_pair", 1, 4096, sms, false);
  tc_rate<256, 0>("ss_n256_all_pairs", P, 4096, sms, false);
  tc_rate<192, 0>("ss_n192_all_pairs", P, 4096, sms, false);
  tc_rate<192, 1>("ts_n192_all_pairs", P, 4096, sms, false);
  tc_rate<16, 0>("issue_n16_4mma", 1, 2048, sms, false);
  tc_rate<16, 2>("issue_n16_4mma_2commits", 1, 2048, sms, false);
  tc_rate<16, 6>("issue_n16_4mma_2commits_poll", 1, 2048, sms, true);
  printf("  },\n");

  // 4. exactness
  {
    std::vector<__half> hA((size_t)EX_M * EX_K), hB((size_t)EX_N * EX_K);
    std::vector<int> iA((size_t)EX_M * EX_K), iB((size_t)EX_N * EX_K);
    uint32_t s = 12345u;
    auto rnd = [&]() { s = s * 1664525u + 1013904223u; return (int)((s >> 8) % 255u) - 127; };
    for (int r = 0; r < EX_M; ++r)
      for (int k = 0; k < EX_K; ++k) {
        int v;
        if (r == 0) v = 127;                                  // all-127 row
        else if (r == 1) v = (k == 0) ? 127 : 1;              // one 16129 term, then +-1 terms
        else if (r == 2) v = (k == 0) ? -127 : ((k & 1) ? 1 : -1);
        else if (r == 3) v = (k < 512) ? 127 : -127;          // rises to 2^23 and back
        else v = rnd();
        iA[(size_t)r * EX_K + k] = v;
      }
    for (int n = 0; n < EX_N; ++n)
      for (int k = 0; k < EX_K; ++k) {
        int v;
        if (n == 0) v = 127;
        else if (n == 1) v = (k == 0) ? 127 : ((k & 1) ? -1 : 1);
        else if (n == 2) v = -127;
        else v = rnd();
        iB[(size_t)n * EX_K + k] = v;
      }
    for (size_t i = 0; i < iA.size(); ++i) hA[i] = __int2half_rn(iA[i]);
    for (size_t i = 0; i < iB.size(); ++i) hB[i] = __int2half_rn(iB[i]);
    __half *dA, *dB;
    float* dD;
    int* dst;
    CK(cudaMalloc(&dA, hA.size() * 2));
    CK(cudaMalloc(&dB, hB.size() * 2));
    CK(cudaMalloc(&dD, (size_t)EX_M * EX_N * 4));
    CK(cudaMalloc(&dst, 4));
    CK(cudaMemset(dst, 0, 4));
    CK(cudaMemcpy(dA, hA.data(), hA.size() * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dB, hB.data(), hB.size() * 2, cudaMemcpyHostToDevice));
    tc_exact_kernel<<<1, 128>>>(dA, dB, dD, dst);
    CK(cudaDeviceSynchronize());
    std::vector<float> hD((size_t)EX_M * EX_N);
    int st = 0;
    CK(cudaMemcpy(hD.data(), dD, hD.size() * 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&st, dst, 4, cudaMemcpyDeviceToHost));
    int mism = 0;
    long long maxabs = 0;
    for (int m = 0; m < EX_M; ++m)
      for (int n = 0; n < EX_N; ++n) {
        long long ref = 0;
        for (int k = 0; k < EX_K; ++k) ref += (long long)iA[(size_t)m * EX_K + k] * iB[(size_t)n * EX_K + k];
        maxabs = llabs(ref) > maxabs ? llabs(ref) : maxabs;
        if ((double)hD[(size_t)m * EX_N + n] != (double)ref) ++mism;
      }
    printf("  \"tmem_fp32_accumulation_exactness\": {\"sums\": %d, \"mismatches\": %d, \"max_abs_sum\": %lld, "
           "\"all127_sum\": %.1f, \"timeouts\": %d}\n",
           EX_M * EX_N, mism, maxabs, (double)hD[0], st);
    CK(cudaFree(dA));
    CK(cudaFree(dB));
    CK(cudaFree(dD));
    CK(cudaFree(dst));
  }
  printf("}\n");
  return 0;
}
