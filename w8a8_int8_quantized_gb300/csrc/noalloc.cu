// w8a8_scaled_mm_noalloc: the INT8 GEMM + epilogue of w8a8_scaled_mm for callers that
// cannot allocate device memory.
//
// w8a8_scaled_mm stages the int8 activations as fp16 codes plus row L1 norms in a
// caller-supplied workspace before its tensor-core kernel reads them.  Some callers have no
// way to provide one: a host runtime that owns only the tensors it hands over and has no
// device allocator of its own to lend, or a latency-critical loop where cudaMalloc (which
// can synchronize the whole device) is not allowed.  This entry point takes the same inputs
// and output but stages into a fixed buffer that belongs to the library itself: a
// file-scope __device__ array that the CUDA driver places in device memory when this
// module is loaded on a GPU and that stays allocated until the process exits.  Nothing here
// calls cudaMalloc, cudaFree or any allocating routine.
//
// The buffer is shared by every call on a device and keeps whatever the last call wrote.
// Each call writes every byte it later reads (the fp16 codes of all M rows and their norms)
// before the GEMM kernel reads them, so nothing needs clearing between calls.  Calls whose
// work overlaps on the same GPU (for example on two streams at once) race on the buffer.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)36 << 20;  // 36 MiB: M*K up to 4096 x 4096
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

// Device address of the scratch array on the current device.  In host code the array's
// name is only a host-side handle, so the address is asked from the runtime once per
// device (with that device current) and cached.
w8a8_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return W8A8_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return W8A8_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return W8A8_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return W8A8_OK;
}

}  // namespace

extern "C" w8a8_status w8a8_scaled_mm_noalloc(const int8_t* xq, const int8_t* wq, int64_t M, int64_t N, int64_t K,
                                              int act_mode, const float* s_x, const int32_t* zp,
                                              const int32_t* azp_adj, int w_mode, const float* s_w,
                                              const void* bias, void* y, int32_t* dev_status, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 1 || K > 131072) return W8A8_ERR_INVALID_ARG;
  if (act_mode < W8A8_ACT_DYN_TOKEN_SYM || act_mode > W8A8_ACT_STATIC_TENSOR_ASYM) return W8A8_ERR_INVALID_ARG;
  if (w_mode != W8A8_W_CHANNEL && w_mode != W8A8_W_TENSOR) return W8A8_ERR_INVALID_ARG;
  if (K % 16 != 0) return W8A8_ERR_MISALIGNED;
  if (M == 0 || N == 0) return W8A8_OK;
  if (!xq || !wq || !s_x || !s_w || !y) return W8A8_ERR_INVALID_ARG;
  if (act_mode == W8A8_ACT_DYN_TOKEN_ASYM && (!zp || !azp_adj)) return W8A8_ERR_INVALID_ARG;
  if (act_mode == W8A8_ACT_STATIC_TENSOR_ASYM && !azp_adj) return W8A8_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(xq) | reinterpret_cast<uintptr_t>(wq) | reinterpret_cast<uintptr_t>(y)) & 15) != 0)
    return W8A8_ERR_MISALIGNED;
  const size_t codes_bytes = round256((size_t)M * (size_t)K * 2);
  // codes, then the row L1 norms and sums of squares (2 * M int32) that the conversion writes
  if (codes_bytes + round256((size_t)M * 8) > kNoallocScratchBytes) return W8A8_ERR_WORKSPACE;
  int dev = -1, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return W8A8_ERR_CUDA;
  if (major != 10 || minor != 3) return W8A8_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  w8a8_status s = scratch_on_current_device(&scratch);
  if (s != W8A8_OK) return s;
  uint8_t* base = static_cast<uint8_t*>(scratch);
  int32_t* norms = reinterpret_cast<int32_t*>(base + codes_bytes);
  if (w8a8::to_gemm_ready(xq, M, K, base, norms, stream) != cudaSuccess) return W8A8_ERR_CUDA;
  w8a8::GemmArgs g{};
  g.a16 = base;
  g.norms = norms;
  g.w = wq;
  g.rows = M;
  g.N = N;
  g.K = K;
  g.E = 1;
  g.act_mode = act_mode;
  g.w_mode = w_mode;
  g.s_x = s_x;
  g.zp = zp;
  g.azp = azp_adj;
  g.s_w = s_w;
  g.bias = bias;
  g.y = y;
  g.status = dev_status;
  return w8a8::gemm_tcgen05(g, stream) == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA;
}
