// C-ABI entry points: argument validation on the host, then launches on the caller's
// stream.  Nothing here allocates device memory.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "internal.h"

using namespace w8a8;

namespace {

constexpr int64_t kMaxK = 131072;  // 128 * 127 * K < 2^31

thread_local int g_engine = 0;  // 0 auto, 1 tcgen05, 2 warp mma

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

w8a8_status cuda_status(cudaError_t e) { return e == cudaSuccess ? W8A8_OK : W8A8_ERR_CUDA; }

bool valid_act_mode(int m) { return m >= W8A8_ACT_DYN_TOKEN_SYM && m <= W8A8_ACT_STATIC_TENSOR_ASYM; }
bool valid_w_mode(int m) { return m == W8A8_W_CHANNEL || m == W8A8_W_TENSOR; }

bool use_small_engine(int64_t rows, bool dense) { return g_engine == 2 || (g_engine == 0 && dense && rows <= 16); }

size_t a256(size_t v) { return (v + 255) & ~(size_t)255; }

// Workspace of the tcgen05 engine: fp16 activation codes, then their row L1 norms [rows] and
// row sums of squares [rows] (one region of 2 * rows int32).
size_t ready_bytes(int64_t rows, int64_t K) { return a256((size_t)rows * (size_t)K * 2) + a256((size_t)rows * 8); }

w8a8_status run_gemm(GemmArgs g, cudaStream_t st, void* ws, bool small, bool a_is_ready) {
  cudaError_t e;
  if (small) {
    e = gemm_small_m(g, st);
  } else {
    uint8_t* w8 = static_cast<uint8_t*>(ws);
    g.a16 = w8;
    g.norms = reinterpret_cast<const int32_t*>(w8 + a256((size_t)g.rows * (size_t)g.K * 2));
    if (!a_is_ready) {
      e = to_gemm_ready(g.a, g.rows, g.K, w8, const_cast<int32_t*>(g.norms), st);
      if (e != cudaSuccess) return W8A8_ERR_CUDA;
    }
    e = gemm_tcgen05(g, st);
  }
  return cuda_status(e);
}

}  // namespace

namespace w8a8 {

// Only compute capability 10.3 (GB300, sm_103a) runs the kernels built here.
w8a8_status check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return W8A8_ERR_CUDA;
  static thread_local int cached_dev = -2;
  static thread_local w8a8_status cached = W8A8_OK;
  if (dev == cached_dev) return cached;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return W8A8_ERR_CUDA;
  cached = (major == 10 && minor == 3) ? W8A8_OK : W8A8_ERR_UNSUPPORTED;
  cached_dev = dev;
  return cached;
}

// Argument checks of the dense GEMM entry points (every one of them applies the same rules).
w8a8_status check_scaled_mm_args(const int8_t* xq, const int8_t* wq, int64_t M, int64_t N, int64_t K,
                                 int act_mode, const float* s_x, const int32_t* zp, const int32_t* azp_adj,
                                 int w_mode, const float* s_w, const void* bias, const void* y) {
  if (M < 0 || N < 0 || K < 1 || K > kMaxK) return W8A8_ERR_INVALID_ARG;
  if (!valid_act_mode(act_mode) || !valid_w_mode(w_mode)) return W8A8_ERR_INVALID_ARG;
  if (K % 16 != 0) return W8A8_ERR_MISALIGNED;
  if (M == 0 || N == 0) return W8A8_OK;
  if (!xq || !wq || !s_x || !s_w || !y) return W8A8_ERR_INVALID_ARG;
  if (act_mode == W8A8_ACT_DYN_TOKEN_ASYM && (!zp || !azp_adj)) return W8A8_ERR_INVALID_ARG;
  if (act_mode == W8A8_ACT_STATIC_TENSOR_ASYM && !azp_adj) return W8A8_ERR_INVALID_ARG;
  if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(y, 16)) return W8A8_ERR_MISALIGNED;
  if (bias && !aligned(bias, 2)) return W8A8_ERR_MISALIGNED;
  return W8A8_OK;
}

}  // namespace w8a8

extern "C" {

const char* w8a8_status_string(int s) {
  switch (s) {
    case W8A8_OK: return "ok";
    case W8A8_ERR_INVALID_ARG: return "invalid argument";
    case W8A8_ERR_UNSUPPORTED: return "unsupported mode or device";
    case W8A8_ERR_MISALIGNED: return "misaligned pointer or size";
    case W8A8_ERR_BAD_SCALE: return "illegal block scale or NaN code";
    case W8A8_ERR_TIMEOUT: return "device wait timed out";
    case W8A8_ERR_CUDA: return "CUDA error";
    case W8A8_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int w8a8_version(void) { return 100; }

w8a8_status w8a8_debug_set_error_word(int32_t* word) {
#ifdef W8A8_DEBUG
  if (debug_register_quant(word) != cudaSuccess || debug_register_requant(word) != cudaSuccess ||
      debug_register_gemm_tc(word) != cudaSuccess || debug_register_gemm_small(word) != cudaSuccess ||
      debug_register_moe_route(word) != cudaSuccess)
    return W8A8_ERR_CUDA;
  return W8A8_OK;
#else
  (void)word;
  return W8A8_ERR_UNSUPPORTED;
#endif
}

int w8a8_debug_build(void) {
#ifdef W8A8_DEBUG
  return 1;
#else
  return 0;
#endif
}

w8a8_status w8a8_set_gemm_engine(int engine) {
  if (engine < 0 || engine > 2) return W8A8_ERR_INVALID_ARG;
  g_engine = engine;
  return W8A8_OK;
}

w8a8_status w8a8_quantize_act(const void* x, int64_t M, int64_t K, int64_t ldx, int mode, int8_t* q,
                              float* scale, int32_t* zp, cudaStream_t stream) {
  if (M < 0 || K < 0 || !valid_act_mode(mode)) return W8A8_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return W8A8_OK;
  if (ldx < K || !x || !q || !scale) return W8A8_ERR_INVALID_ARG;
  if ((mode == W8A8_ACT_DYN_TOKEN_ASYM || mode == W8A8_ACT_STATIC_TENSOR_ASYM) && !zp) return W8A8_ERR_INVALID_ARG;
  if (M > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (!aligned(x, 2)) return W8A8_ERR_MISALIGNED;
  w8a8_status s = check_device();
  if (s != W8A8_OK) return s;
  return cuda_status(quant_rows(mode, x, M, K, ldx, nullptr, q, nullptr, scale, zp, nullptr, nullptr, stream));
}

size_t w8a8_scaled_mm_workspace_size(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0) return 0;
  return ready_bytes(M, K);
}

w8a8_status w8a8_scaled_mm(const int8_t* xq, const int8_t* wq, int64_t M, int64_t N, int64_t K, int act_mode,
                           const float* s_x, const int32_t* zp, const int32_t* azp_adj, int w_mode,
                           const float* s_w, const int32_t* w_sumsq, const void* bias, void* y, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream) {
  w8a8_status s = check_scaled_mm_args(xq, wq, M, N, K, act_mode, s_x, zp, azp_adj, w_mode, s_w, bias, y);
  if (s != W8A8_OK || M == 0 || N == 0) return s;
  const bool small = use_small_engine(M, true);
  if (!small && (!workspace || workspace_bytes < ready_bytes(M, K))) return W8A8_ERR_WORKSPACE;
  if (!small && !aligned(workspace, 256)) return W8A8_ERR_MISALIGNED;
  s = check_device();
  if (s != W8A8_OK) return s;
  GemmArgs g{};
  g.a = xq;
  g.w = wq;
  g.rows = M;
  g.N = N;
  g.K = K;
  g.E = 1;
  g.seg = nullptr;
  g.act_mode = act_mode;
  g.w_mode = w_mode;
  g.s_x = s_x;
  g.zp = zp;
  g.azp = azp_adj;
  g.s_w = s_w;
  g.wsq = w_sumsq;
  g.bias = bias;
  g.y = y;
  g.status = dev_status;
  if (!small && workspace_bytes > ready_bytes(M, K)) {
    g.split_ws = static_cast<uint8_t*>(workspace) + ready_bytes(M, K);
    g.split_bytes = workspace_bytes - ready_bytes(M, K);
  }
  return run_gemm(g, stream, workspace, small, false);
}

size_t w8a8_splitk_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || K > kMaxK) return 0;
  if (check_device() != W8A8_OK) return 0;
  if (use_small_engine(M, true)) return 0;
  return gemm_split_bytes(M, N, K);
}

size_t w8a8_linear_workspace_size(int64_t M, int64_t K, int act_mode) {
  if (M <= 0 || K <= 0 || !valid_act_mode(act_mode)) return 0;
  // quantized activations (fp16 codes + norms for tcgen05, or int8 codes) + scales + zero points
  return ready_bytes(M, K) + 2 * a256((size_t)M * 4);
}

w8a8_status w8a8_linear(const void* x, int64_t M, int64_t K, int64_t ldx, int act_mode, const float* input_scale,
                        const int32_t* input_zero_point, const int8_t* wq, int64_t N, int w_mode,
                        const float* s_w, const int32_t* azp_adj, const int32_t* w_sumsq, const void* bias,
                        void* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 1 || K > kMaxK || !valid_act_mode(act_mode) || !valid_w_mode(w_mode))
    return W8A8_ERR_INVALID_ARG;
  if (K % 16 != 0) return W8A8_ERR_MISALIGNED;
  if (M == 0 || N == 0) return W8A8_OK;
  if (!x || ldx < K || !wq || !s_w || !y) return W8A8_ERR_INVALID_ARG;
  const bool is_static = act_mode == W8A8_ACT_STATIC_TENSOR_SYM || act_mode == W8A8_ACT_STATIC_TENSOR_ASYM;
  if (is_static && !input_scale) return W8A8_ERR_INVALID_ARG;
  if (act_mode == W8A8_ACT_STATIC_TENSOR_ASYM && !input_zero_point) return W8A8_ERR_INVALID_ARG;
  if (act_mode == W8A8_ACT_DYN_TOKEN_ASYM || act_mode == W8A8_ACT_STATIC_TENSOR_ASYM) {
    if (!azp_adj) return W8A8_ERR_INVALID_ARG;
  }
  const size_t need = w8a8_linear_workspace_size(M, K, act_mode);
  if (!workspace || workspace_bytes < need) return W8A8_ERR_WORKSPACE;
  if (!aligned(workspace, 256) || !aligned(wq, 16) || !aligned(y, 16) || !aligned(x, 2)) return W8A8_ERR_MISALIGNED;
  w8a8_status s = check_device();
  if (s != W8A8_OK) return s;
  const bool small = use_small_engine(M, true);
  if (small && (act_mode == W8A8_ACT_DYN_TOKEN_SYM || act_mode == W8A8_ACT_DYN_TOKEN_ASYM) &&
      gemm_small_m_fused_ok(M, K) && aligned(x, 16) && ldx % 8 == 0) {
    // decode: the per-token quantizer (symmetric, or affine with zp * azp_adj in the
    // epilogue) runs inside the small-M GEMM (no separate launch)
    GemmArgs g{};
    g.w = wq;
    g.rows = M;
    g.N = N;
    g.K = K;
    g.E = 1;
    g.act_mode = act_mode;
    g.w_mode = w_mode;
    g.azp = azp_adj;
    g.s_w = s_w;
    g.bias = bias;
    g.y = y;
    g.status = dev_status;
    return cuda_status(gemm_small_m_fused(x, ldx, g, stream));
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  size_t off = ready_bytes(M, K);
  float* sx = const_cast<float*>(input_scale);
  int32_t* zp = const_cast<int32_t*>(input_zero_point);
  if (!is_static) {
    sx = reinterpret_cast<float*>(ws + off);
    if (act_mode == W8A8_ACT_DYN_TOKEN_ASYM) zp = reinterpret_cast<int32_t*>(ws + off + a256((size_t)M * 4));
  }
  // the quantizer writes the GEMM engine's own activation format directly
  int8_t* q = small ? reinterpret_cast<int8_t*>(ws) : nullptr;
  void* q16 = small ? nullptr : ws;
  int32_t* norms = small ? nullptr : reinterpret_cast<int32_t*>(ws + a256((size_t)M * (size_t)K * 2));
  cudaError_t e = quant_rows(act_mode, x, M, K, ldx, nullptr, q, q16, sx, zp, nullptr, norms, stream);
  if (e != cudaSuccess) return W8A8_ERR_CUDA;
  GemmArgs g{};
  g.a = q;
  g.w = wq;
  g.rows = M;
  g.N = N;
  g.K = K;
  g.E = 1;
  g.seg = nullptr;
  g.act_mode = act_mode;
  g.w_mode = w_mode;
  g.s_x = sx;
  g.zp = zp;
  g.azp = azp_adj;
  g.s_w = s_w;
  g.wsq = w_sumsq;
  g.bias = bias;
  g.y = y;
  g.status = dev_status;
  if (!small && workspace_bytes > need) {
    g.split_ws = ws + need;
    g.split_bytes = workspace_bytes - need;
  }
  return run_gemm(g, stream, workspace, small, true);
}

w8a8_status w8a8_quantize_weight(const void* w, int64_t N, int64_t K, int8_t* wq, float* s_w, int32_t* azp_adj,
                                 int32_t* w_sumsq, cudaStream_t stream) {
  if (N < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return W8A8_OK;
  if (!w || !wq || !s_w || K > kMaxK || N > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (!aligned(w, 2)) return W8A8_ERR_MISALIGNED;
  w8a8_status s = check_device();
  if (s != W8A8_OK) return s;
  cudaError_t e =
      quant_rows(W8A8_ACT_DYN_TOKEN_SYM, w, N, K, K, nullptr, wq, nullptr, s_w, nullptr, azp_adj, nullptr, stream);
  if (e == cudaSuccess && w_sumsq) e = sumsq_rows(wq, N, K, w_sumsq, stream);
  return cuda_status(e);
}

w8a8_status w8a8_weight_sumsq(const int8_t* wq, int64_t N, int64_t K, int32_t* w_sumsq, cudaStream_t stream) {
  if (N < 0 || K < 0 || K > kMaxK || N > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (N == 0) return W8A8_OK;
  if (!w_sumsq || (K > 0 && !wq)) return W8A8_ERR_INVALID_ARG;
  if (!aligned(w_sumsq, 4)) return W8A8_ERR_MISALIGNED;
  w8a8_status s = check_device();
  if (s != W8A8_OK) return s;
  return cuda_status(sumsq_rows(wq, N, K, w_sumsq, stream));
}

w8a8_status w8a8_azp_adj(const int8_t* wq, int64_t N, int64_t K, const int32_t* input_zero_point, int32_t* azp_adj,
                         cudaStream_t stream) {
  if (N < 0 || K < 0 || K > kMaxK || N > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (N == 0) return W8A8_OK;
  if (!azp_adj || (K > 0 && !wq)) return W8A8_ERR_INVALID_ARG;
  w8a8_status s = check_device();
  if (s != W8A8_OK) return s;
  return cuda_status(azp_rows(wq, N, K, input_zero_point, azp_adj, stream));
}

w8a8_status fp8block_to_int8_rowwise_batched(int count, const uint8_t* const* w, const float* const* scale_inv,
                                             const int64_t* N, const int64_t* K, int8_t* const* q, float* const* s,
                                             int32_t* dev_status, cudaStream_t stream) {
  return fp8block_to_int8_rowwise_batched_adj(count, w, scale_inv, N, K, q, s, nullptr, dev_status, stream);
}

w8a8_status fp8block_to_int8_rowwise_batched_adj(int count, const uint8_t* const* w, const float* const* scale_inv,
                                                 const int64_t* N, const int64_t* K, int8_t* const* q,
                                                 float* const* s, int32_t* const* azp_adj, int32_t* dev_status,
                                                 cudaStream_t stream) {
  if (count < 0) return W8A8_ERR_INVALID_ARG;
  if (count == 0) return W8A8_OK;
  if (!w || !scale_inv || !N || !K || !q || !s) return W8A8_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    if (N[i] < 0 || K[i] < 0 || N[i] > 0x7FFFFFFF || K[i] > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
    if (N[i] > 0 && K[i] > 0 && (!w[i] || !scale_inv[i] || !q[i] || !s[i])) return W8A8_ERR_INVALID_ARG;
    if (N[i] > 0 && K[i] > 0 && !aligned(s[i], 4)) return W8A8_ERR_MISALIGNED;
    if (N[i] > 0 && K[i] > 0 && azp_adj && azp_adj[i] && !aligned(azp_adj[i], 4)) return W8A8_ERR_MISALIGNED;
  }
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  int i = 0;
  while (i < count) {
    ReqBatch b;
    memset(&b, 0, sizeof(b));
    int64_t rows = 0;
    while (i < count && b.count < kReqMaxBatch && rows + N[i] <= 0x7FFFFFFF) {
      if (N[i] > 0 && K[i] > 0) {
        ReqMat& m = b.m[b.count++];
        m.w = w[i];
        m.sinv = scale_inv[i];
        m.q = q[i];
        m.s = s[i];
        m.adj = azp_adj ? azp_adj[i] : nullptr;
        m.row0 = (int32_t)rows;
        m.N = (int32_t)N[i];
        m.K = (int32_t)K[i];
        m.vec = requant_path(w[i], q[i], K[i]);
        rows += N[i];
      } else if (N[i] > 0 && K[i] == 0) {
        // no columns: every row is an all-zero row (q empty, s = 1)
        return W8A8_ERR_INVALID_ARG;
      }
      ++i;
    }
    b.total_rows = rows;
    if (b.count > 0) {
      cudaError_t e = requant_batch(b, dev_status, stream);
      if (e != cudaSuccess) return W8A8_ERR_CUDA;
    }
  }
  return W8A8_OK;
}

static bool route_args_ok(int64_t T, int E, int topk) {
  return T >= 0 && T <= 0x7FFFFFFF && E >= 1 && E <= 256 && topk >= 1 && topk <= 8 && topk <= E;
}

size_t w8a8_moe_route_workspace_size(int64_t T, int E, int topk) {
  return route_args_ok(T, E, topk) ? moe_route_workspace(T, E, topk) : 0;
}

w8a8_status w8a8_moe_route(const float* logits, int64_t T, int E, int topk, int32_t* topk_ids, float* topk_w,
                           int64_t* seg_offsets, int64_t* row_index, int64_t* row_of, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (!route_args_ok(T, E, topk) || !seg_offsets) return W8A8_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_ids || !topk_w || !row_index || !row_of)) return W8A8_ERR_INVALID_ARG;
  if (T > 0 && (!workspace || workspace_bytes < moe_route_workspace(T, E, topk))) return W8A8_ERR_WORKSPACE;
  if (!aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(seg_offsets, 8) ||
      !aligned(row_index, 8) || !aligned(row_of, 8) || !aligned(workspace, 4))
    return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  return cuda_status(moe_route(logits, T, E, topk, topk_ids, topk_w, seg_offsets, row_index, row_of, workspace,
                               stream));
}

w8a8_status w8a8_requantize_max_scale(int8_t* wq, int64_t N, int64_t K, const float* scales,
                                      const int64_t* logical_widths, int P, float* s_max, int32_t* dev_status,
                                      cudaStream_t stream) {
  if (N < 0 || K < 0 || P < 1 || P > kMaxScaleParts) return W8A8_ERR_INVALID_ARG;
  if (!scales || !logical_widths || !s_max || (N > 0 && K > 0 && !wq)) return W8A8_ERR_INVALID_ARG;
  if (!aligned(scales, 4) || !aligned(s_max, 4)) return W8A8_ERR_MISALIGNED;
  int64_t rows = 0;
  for (int p = 0; p < P; ++p) {
    if (logical_widths[p] < 0) return W8A8_ERR_INVALID_ARG;
    rows += logical_widths[p];
  }
  if (rows != N) return W8A8_ERR_INVALID_ARG;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  MaxScaleParts parts;
  memset(&parts, 0, sizeof(parts));
  parts.P = P;
  parts.vec = (K % 16 == 0 && aligned(wq, 16)) ? 1 : 0;
  const int64_t per_row = parts.vec ? K / 16 : K;  // units of the flattened weight per row
  int64_t end = 0;
  for (int p = 0; p < P; ++p) {
    end += logical_widths[p] * per_row;
    parts.end[p] = end;
  }
  return cuda_status(requant_max_scale(wq, N * per_row, scales, parts, s_max, dev_status, stream));
}

w8a8_status fp8block_to_int8_rowwise(const uint8_t* w, const float* scale_inv, int64_t N, int64_t K, int8_t* q,
                                     float* s, int32_t* dev_status, cudaStream_t stream) {
  if (N < 0 || K < 0) return W8A8_ERR_INVALID_ARG;
  if (N == 0) return W8A8_OK;
  if (K == 0) return W8A8_ERR_INVALID_ARG;
  return fp8block_to_int8_rowwise_batched(1, &w, &scale_inv, &N, &K, &q, &s, dev_status, stream);
}

size_t w8a8_grouped_mm_workspace_size(int64_t R, int64_t K) {
  if (R <= 0 || K <= 0) return 0;
  return ready_bytes(R, K);
}

w8a8_status w8a8_grouped_mm(const int8_t* xq_sorted, const float* s_x, const int8_t* w, const float* s_w,
                            const int32_t* w_sumsq, const int64_t* seg_offsets, int E, int64_t max_rows, int64_t N,
                            int64_t K, void* y, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            cudaStream_t stream) {
  if (E < 1 || E > gemm_tc_max_segments() || max_rows < 0 || N < 0 || K < 1 || K > kMaxK)
    return W8A8_ERR_INVALID_ARG;
  if (K % 16 != 0) return W8A8_ERR_MISALIGNED;
  if (max_rows == 0 || N == 0) return W8A8_OK;
  if (!xq_sorted || !s_x || !w || !s_w || !seg_offsets || !y) return W8A8_ERR_INVALID_ARG;
  if (!aligned(xq_sorted, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(seg_offsets, 8) ||
      !aligned(w_sumsq, 4))
    return W8A8_ERR_MISALIGNED;
  const bool small = use_small_engine(max_rows, false);
  if (!small && (!workspace || workspace_bytes < ready_bytes(max_rows, K))) return W8A8_ERR_WORKSPACE;
  if (!small && !aligned(workspace, 256)) return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  GemmArgs g{};
  g.a = xq_sorted;
  g.w = w;
  g.rows = max_rows;
  g.N = N;
  g.K = K;
  g.E = E;
  g.seg = seg_offsets;
  g.act_mode = W8A8_ACT_DYN_TOKEN_SYM;
  g.w_mode = W8A8_W_CHANNEL;
  g.s_x = s_x;
  g.zp = nullptr;
  g.azp = nullptr;
  g.s_w = s_w;
  g.wsq = w_sumsq;
  g.bias = nullptr;
  g.y = y;
  g.status = dev_status;
  return run_gemm(g, stream, workspace, small, false);
}

w8a8_status w8a8_moe_quantize_gather(const void* x, int64_t T, int64_t K, int64_t ldx, const int64_t* row_index,
                                     int64_t R, int8_t* xq_sorted, float* s_x, cudaStream_t stream) {
  if (T < 0 || K < 0 || R < 0 || R > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (R == 0 || K == 0) return W8A8_OK;
  if (!x || !row_index || !xq_sorted || !s_x || ldx < K || T == 0) return W8A8_ERR_INVALID_ARG;
  if (!aligned(x, 2) || !aligned(row_index, 8)) return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  return cuda_status(
      quant_rows(W8A8_ACT_DYN_TOKEN_SYM, x, R, K, ldx, row_index, xq_sorted, nullptr, s_x, nullptr, nullptr, nullptr,
                 stream));
}

w8a8_status w8a8_silu_mul_quant(const void* h, int64_t R, int64_t I, int8_t* gq, float* s_g, cudaStream_t stream) {
  if (R < 0 || I < 0 || R > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (R == 0 || I == 0) return W8A8_OK;
  if (!h || !gq || !s_g || I > 16384) return W8A8_ERR_INVALID_ARG;
  if (I % 8 != 0 || !aligned(h, 16) || !aligned(gq, 8)) return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  return cuda_status(silu_mul_quant(h, R, I, gq, nullptr, nullptr, s_g, stream));
}

w8a8_status w8a8_moe_combine(const void* out, const int64_t* row_of, const float* topk_w, int64_t T, int topk,
                             int64_t H, void* y, cudaStream_t stream) {
  if (T < 0 || topk < 1 || H < 0 || T > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (T == 0 || H == 0) return W8A8_OK;
  if (!out || !row_of || !topk_w || !y) return W8A8_ERR_INVALID_ARG;
  if (H % 8 != 0 || !aligned(out, 16) || !aligned(y, 16)) return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  return cuda_status(moe_combine(out, row_of, topk_w, T, topk, H, y, stream));
}

// ---------------------------------------------------------------- packed activations
size_t w8a8_act_packed_size(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0) return 0;
  return ready_bytes(M, K);
}

w8a8_status w8a8_quantize_act_packed(const void* x, int64_t M, int64_t K, int64_t ldx, int mode, void* packed,
                                     float* scale, int32_t* zp, cudaStream_t stream) {
  if (M < 0 || K < 0 || !valid_act_mode(mode)) return W8A8_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return W8A8_OK;
  if (ldx < K || !x || !packed || !scale || M > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if ((mode == W8A8_ACT_DYN_TOKEN_ASYM || mode == W8A8_ACT_STATIC_TENSOR_ASYM) && !zp) return W8A8_ERR_INVALID_ARG;
  if (K % 16 != 0 || !aligned(packed, 256) || !aligned(x, 2)) return W8A8_ERR_MISALIGNED;
  w8a8_status s = check_device();
  if (s != W8A8_OK) return s;
  uint8_t* pk = static_cast<uint8_t*>(packed);
  int32_t* norms = reinterpret_cast<int32_t*>(pk + a256((size_t)M * (size_t)K * 2));
  return cuda_status(quant_rows(mode, x, M, K, ldx, nullptr, nullptr, pk, scale, zp, nullptr, norms, stream));
}

w8a8_status w8a8_scaled_mm_packed(const void* packed, const int8_t* wq, int64_t M, int64_t N, int64_t K, int act_mode,
                                  const float* s_x, const int32_t* zp, const int32_t* azp_adj, int w_mode,
                                  const float* s_w, const int32_t* w_sumsq, const void* bias, void* y,
                                  void* split_ws, size_t split_bytes, int32_t* dev_status, cudaStream_t stream) {
  const int8_t* dummy = static_cast<const int8_t*>(packed);
  w8a8_status s = check_scaled_mm_args(dummy, wq, M, N, K, act_mode, s_x, zp, azp_adj, w_mode, s_w, bias, y);
  if (s != W8A8_OK || M == 0 || N == 0) return s;
  if (!aligned(packed, 256) || !aligned(split_ws, 256)) return W8A8_ERR_MISALIGNED;
  s = check_device();
  if (s != W8A8_OK) return s;
  GemmArgs g{};
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
  g.wsq = w_sumsq;
  g.bias = bias;
  g.y = y;
  g.status = dev_status;
  g.split_ws = split_ws;
  g.split_bytes = split_ws ? split_bytes : 0;
  return run_gemm(g, stream, const_cast<void*>(packed), false, true);
}

w8a8_status w8a8_grouped_mm_packed(const void* packed, const float* s_x, const int8_t* w, const float* s_w,
                                   const int32_t* w_sumsq, const int64_t* seg_offsets, int E, int64_t max_rows,
                                   int64_t N, int64_t K, void* y, int32_t* dev_status, cudaStream_t stream) {
  if (E < 1 || E > gemm_tc_max_segments() || max_rows < 0 || N < 0 || K < 1 || K > kMaxK)
    return W8A8_ERR_INVALID_ARG;
  if (K % 16 != 0) return W8A8_ERR_MISALIGNED;
  if (max_rows == 0 || N == 0) return W8A8_OK;
  if (!packed || !s_x || !w || !s_w || !seg_offsets || !y) return W8A8_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(w, 16) || !aligned(y, 16) || !aligned(seg_offsets, 8) ||
      !aligned(w_sumsq, 4))
    return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  GemmArgs g{};
  g.w = w;
  g.rows = max_rows;
  g.N = N;
  g.K = K;
  g.E = E;
  g.seg = seg_offsets;
  g.act_mode = W8A8_ACT_DYN_TOKEN_SYM;
  g.w_mode = W8A8_W_CHANNEL;
  g.s_x = s_x;
  g.s_w = s_w;
  g.wsq = w_sumsq;
  g.y = y;
  g.status = dev_status;
  return run_gemm(g, stream, const_cast<void*>(packed), false, true);
}

w8a8_status w8a8_moe_quantize_gather_packed(const void* x, int64_t T, int64_t K, int64_t ldx,
                                            const int64_t* row_index, int64_t R, void* packed, float* s_x,
                                            cudaStream_t stream) {
  if (T < 0 || K < 0 || R < 0 || R > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (R == 0 || K == 0) return W8A8_OK;
  if (!x || !row_index || !packed || !s_x || ldx < K || T == 0) return W8A8_ERR_INVALID_ARG;
  if (K % 16 != 0 || !aligned(x, 2) || !aligned(row_index, 8) || !aligned(packed, 256)) return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  uint8_t* pk = static_cast<uint8_t*>(packed);
  int32_t* norms = reinterpret_cast<int32_t*>(pk + a256((size_t)R * (size_t)K * 2));
  return cuda_status(quant_rows(W8A8_ACT_DYN_TOKEN_SYM, x, R, K, ldx, row_index, nullptr, pk, s_x, nullptr, nullptr,
                                norms, stream));
}

w8a8_status w8a8_moe_quantize_scatter_packed(const void* x, int64_t T, int64_t K, int64_t ldx,
                                             const int64_t* row_of, int topk, int64_t R, void* packed, float* s_x,
                                             cudaStream_t stream) {
  if (T < 0 || K < 0 || R < 0 || R > 0x7FFFFFFF || T > 0x7FFFFFFF || topk < 1 || topk > 32 || K > 16384)
    return W8A8_ERR_INVALID_ARG;
  if (T == 0 || K == 0 || R == 0) return W8A8_OK;
  if (!x || !row_of || !packed || !s_x || ldx < K) return W8A8_ERR_INVALID_ARG;
  if (K % 16 != 0 || ldx % 8 != 0 || !aligned(x, 16) || !aligned(row_of, 8) || !aligned(packed, 256))
    return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  uint8_t* pk = static_cast<uint8_t*>(packed);
  int32_t* norms = reinterpret_cast<int32_t*>(pk + a256((size_t)R * (size_t)K * 2));
  return cuda_status(quant_rows_scatter_packed(x, T, K, ldx, row_of, topk, R, pk, s_x, norms, stream));
}

w8a8_status w8a8_silu_mul_quant_packed(const void* h, int64_t R, int64_t I, void* packed, float* s_g,
                                       cudaStream_t stream) {
  if (R < 0 || I < 0 || R > 0x7FFFFFFF) return W8A8_ERR_INVALID_ARG;
  if (R == 0 || I == 0) return W8A8_OK;
  if (!h || !packed || !s_g || I > 16384) return W8A8_ERR_INVALID_ARG;
  if (I % 16 != 0 || !aligned(h, 16) || !aligned(packed, 256)) return W8A8_ERR_MISALIGNED;
  w8a8_status st = check_device();
  if (st != W8A8_OK) return st;
  uint8_t* pk = static_cast<uint8_t*>(packed);
  int32_t* norms = reinterpret_cast<int32_t*>(pk + a256((size_t)R * (size_t)I * 2));
  return cuda_status(silu_mul_quant(h, R, I, nullptr, pk, norms, s_g, stream));
}

}  // extern "C"
