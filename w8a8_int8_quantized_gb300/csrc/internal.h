// Internal launcher declarations shared between the C-ABI layer and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "w8a8.h"

namespace w8a8 {

struct EpiParams;

// quant.cu
// q_i8: int8 codes [rows, K] or nullptr; q_f16: the same codes as fp16 [rows, K] (the GEMM-ready
// activation format) or nullptr; norm_out: sum_k |q| per row (with q_f16); sum_out: sum_k q.
cudaError_t quant_rows_scatter_packed(const void* x, int64_t T, int64_t K, int64_t ldx, const int64_t* row_of,
                                      int topk, int64_t R, void* q_f16, float* scale, int32_t* norm_out,
                                      cudaStream_t st);
cudaError_t quant_rows(int mode, const void* x, int64_t rows, int64_t K, int64_t ldx,
                       const int64_t* row_index, int8_t* q_i8, void* q_f16, float* scale, int32_t* zp,
                       int32_t* sum_out, int32_t* norm_out, cudaStream_t st);
cudaError_t azp_rows(const int8_t* w, int64_t N, int64_t K, const int32_t* zp, int32_t* out,
                     cudaStream_t st);
cudaError_t sumsq_rows(const int8_t* w, int64_t N, int64_t K, int32_t* out, cudaStream_t st);
// gq: int8 codes, or g16 + norms: the packed (fp16 codes + row L1 norms) format
cudaError_t silu_mul_quant(const void* h, int64_t R, int64_t I, int8_t* gq, void* g16, int32_t* norms, float* sg,
                           cudaStream_t st);
cudaError_t moe_combine(const void* out, const int64_t* row_of, const float* tw, int64_t T, int topk,
                        int64_t H, void* y, cudaStream_t st);

// requant.cu
struct ReqMat {
  const uint8_t* w;
  const float* sinv;
  int8_t* q;
  float* s;
  int32_t* adj;  // optional [N]: row sums of q (the weight's azp_adj), or null
  int32_t row0;  // first row of this matrix in the batch (a batch holds fewer than 2^31 rows)
  int32_t N;
  int32_t K;
  int32_t vec;   // requant_path(): 1 vector rows, 2 word rows, 0 byte rows
};
constexpr int kReqMaxBatch = 64;
struct ReqBatch {
  int32_t count;
  int32_t pad;
  int64_t total_rows;
  ReqMat m[kReqMaxBatch];
};
static_assert(sizeof(ReqBatch) <= 4096, "kernel parameter block must stay within 4 KB");
cudaError_t requant_batch(const ReqBatch& b, int32_t* st, cudaStream_t stream);
// 1: 16-byte vector path, 2: 4-byte word path (K % 4 == 0, K <= 4096), 0: byte path
int requant_path(const uint8_t* w, const int8_t* q, int64_t K);
// MoE routing: top-k + softmax weights per token, stable counting sort into expert segments.
size_t moe_route_workspace(int64_t T, int E, int topk);
cudaError_t moe_route(const float* logits, int64_t T, int E, int topk, int32_t* ids, float* w, int64_t* seg,
                      int64_t* row_index, int64_t* row_of, void* ws, cudaStream_t st);
// Fused weight with per-tensor scales -> one scale (the largest): partition p covers the
// units [end[p-1], end[p]) of the flattened weight, in 16-byte chunks (vec) or bytes.
constexpr int kMaxScaleParts = 16;
struct MaxScaleParts {
  int32_t P;
  int32_t vec;
  int64_t end[kMaxScaleParts];
};
cudaError_t requant_max_scale(int8_t* wq, int64_t units, const float* scales, const MaxScaleParts& parts,
                              float* s_out, int32_t* st, cudaStream_t stream);

// GEMM problem description shared by both GEMM engines.  Rows of A are grouped into
// segments; segment e multiplies weight rows [e*N, (e+1)*N).  A dense GEMM is one segment.
struct GemmArgs {
  const int8_t* a;      // [rows, K] int8 codes (warp-MMA engine)
  const void* a16;      // [rows, K] the same codes as fp16 (tcgen05 engine)
  const int32_t* norms; // [rows] sum_k |a[r, k]| (tcgen05 engine)
  const int8_t* w;      // [E*N, K]
  int64_t rows;         // rows of A (dense M, or an upper bound for grouped)
  int64_t N, K;
  int E;                // number of segments
  const int64_t* seg;   // device [E+1] or nullptr (dense: one segment [0, rows))
  int act_mode, w_mode;
  const float* s_x;
  const int32_t* zp;
  const int32_t* azp;
  const float* s_w;     // [E*N] (channel) or [1] (tensor)
  const int32_t* wsq;   // [N] sum_k w[n, k]^2 (dense only, optional): admits single-pass tiles
                        // by the Cauchy-Schwarz bound
  const void* bias;     // [N] or nullptr
  void* y;              // [rows, N] bf16
  int32_t* status;
  void* split_ws;       // optional scratch that lets an under-filled dense launch split along K
  size_t split_bytes;
};

// api.cu: the device check every entry point runs, and the argument checks of the dense GEMM
// entry points (w8a8_scaled_mm, w8a8_scaled_mm_packed, w8a8_scaled_mm_noalloc)
w8a8_status check_device();
w8a8_status check_scaled_mm_args(const int8_t* xq, const int8_t* wq, int64_t M, int64_t N, int64_t K,
                                 int act_mode, const float* s_x, const int32_t* zp, const int32_t* azp_adj,
                                 int w_mode, const float* s_w, const void* bias, const void* y);

#ifdef W8A8_DEBUG
// bounds-checked build: each translation unit's copy of the error-word pointer
cudaError_t debug_register_quant(int32_t* word);
cudaError_t debug_register_requant(int32_t* word);
cudaError_t debug_register_gemm_tc(int32_t* word);
cudaError_t debug_register_gemm_small(int32_t* word);
cudaError_t debug_register_moe_route(int32_t* word);
#endif

// gemm_small.cu: mma.sync s8 weight-streaming kernel (small M)
cudaError_t gemm_small_m(const GemmArgs& g, cudaStream_t st);
// Dynamic per-token decode (at most 8 bf16 rows x; symmetric, or affine with g.azp the
// weight's azp_adj) with the quantizer fused into the small-M GEMM; g carries the weight side,
// the mode and the output (g.a, g.s_x, g.zp unused).
bool gemm_small_m_fused_ok(int64_t rows, int64_t K);
cudaError_t gemm_small_m_fused(const void* x, int64_t ldx, const GemmArgs& g, cudaStream_t st);
// gemm_tc.cu: tcgen05 kernel; returns cudaErrorNotSupported when it cannot run
cudaError_t gemm_tcgen05(const GemmArgs& g, cudaStream_t st);
// int8 codes -> fp16 codes + row L1 norms (K % 16 == 0, 16-byte aligned rows)
cudaError_t to_gemm_ready(const int8_t* a, int64_t rows, int64_t K, void* a16, int32_t* norms, cudaStream_t st);
int gemm_tc_max_segments();
// scratch a dense tcgen05 launch of this shape uses to split along K on the current device
// (0: the launch does not split)
size_t gemm_split_bytes(int64_t rows, int64_t N, int64_t K);

}  // namespace w8a8
