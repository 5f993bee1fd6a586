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
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = (size_t)36 << 20;  // 36 MiB: M*K up to 4096 x 4096
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
// Per device: the context the address was looked up in, and the address.
CUcontext g_noalloc_ctx[kMaxDevices] = {};
void* g_noalloc_addr[kMaxDevices] = {};

size_t round256(size_t v) { return (v + 255) & ~(size_t)255; }

PFN_cuCtxGetCurrent_v4000 ctx_getter() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  });
  return fn;
}

CUcontext current_ctx() {
  CUcontext c = nullptr;
  auto fn = ctx_getter();
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// Device address of the scratch array on the current device.  In host code the array's
// name is only a host-side handle, so the address is asked from the runtime (with the
// device current) and cached per device.  The cache remembers the CUDA context it was
// looked up in and asks again when the current context differs (another context on the
// device, or a new primary context after cudaDeviceReset), so a stale address of an
// unloaded module is never handed to a kernel.
w8a8_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return W8A8_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return W8A8_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const CUcontext before = current_ctx();
  if (g_noalloc_addr[dev] && before && before == g_noalloc_ctx[dev]) {
    *out = g_noalloc_addr[dev];
    return W8A8_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return W8A8_ERR_CUDA;
  g_noalloc_ctx[dev] = current_ctx();  // the lookup made the device's context current
  g_noalloc_addr[dev] = p;
  *out = p;
  return W8A8_OK;
}

}  // namespace

extern "C" w8a8_status w8a8_scaled_mm_noalloc(const int8_t* xq, const int8_t* wq, int64_t M, int64_t N, int64_t K,
                                              int act_mode, const float* s_x, const int32_t* zp,
                                              const int32_t* azp_adj, int w_mode, const float* s_w,
                                              const void* bias, void* y, int32_t* dev_status, cudaStream_t stream) {
  // the same checks as w8a8_scaled_mm (shapes, modes, null pointers, 16-byte operands,
  // 2-byte bias), then the one limit of this entry point: the staged codes must fit
  w8a8_status s = w8a8::check_scaled_mm_args(xq, wq, M, N, K, act_mode, s_x, zp, azp_adj, w_mode, s_w, bias, y);
  if (s != W8A8_OK || M == 0 || N == 0) return s;
  const size_t codes_bytes = round256((size_t)M * (size_t)K * 2);
  // codes, then the row L1 norms and sums of squares (2 * M int32) that the conversion writes
  if (codes_bytes + round256((size_t)M * 8) > kNoallocScratchBytes) return W8A8_ERR_WORKSPACE;
  s = w8a8::check_device();
  if (s != W8A8_OK) return s;
  void* scratch = nullptr;
  s = scratch_on_current_device(&scratch);
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
