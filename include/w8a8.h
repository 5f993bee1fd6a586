/*
 * w8a8.h -- C ABI of the GB300 (sm_103a) W8A8 INT8 quantized linear library.
 *
 * Sources cited below by short name:
 *   [vLLM-W8A8]   "vLLM INT8 W8A8 量化实战：用 llm-compressor 制作 8 位权重与 8 位激活的推理模型"
 *                 (blog.gitcode.com), sections 4.1 方案判定, 4.2 权重布局与 kernel 选择, 4.3 未匹配时的行为.
 *   [SGLang-CT]   "[SGLang] W4A8, W8A8, W4A4: 혼합 정밀도 양자화 스킴", items 3 (W8A8 INT8) and
 *                 4 (비대칭 양자화: AZP 보정), and the scheme file tree (MoE INT8).
 *   [Kunlun-INT8] "MiniMax-M2.7 FP8 转昆仑芯 INT8" README, sections 转换关系 and 验证.
 *
 * Conventions shared by every entry point:
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller owns every
 *     buffer.  No entry point allocates device memory: scratch, where needed, is a
 *     caller-provided workspace whose size a *_workspace_size() query returns.
 *   - Matrices are row-major.  bf16 tensors are passed as void* (2 bytes per element).
 *   - Work is enqueued on `stream` and is asynchronous; nothing synchronizes.
 *     Argument errors are detected on the host and returned before any launch.
 *   - Device-side conditions (illegal FP8 block scales, a bounded wait that ran out) are
 *     reported through an optional `int32_t* dev_status` word (device memory).  The
 *     library only ever writes a non-zero w8a8_status code into it (never clears it);
 *     the caller zeroes it and reads it after synchronizing.  NULL means "not reported".
 *   - Only GPUs of compute capability 10.3 (GB300) are supported; others get
 *     W8A8_ERR_UNSUPPORTED.  There is no CPU fallback.
 *   - int32 accumulation is exact for K <= 131072 (|acc| <= 128*127*K < 2^31); larger K is
 *     rejected with W8A8_ERR_INVALID_ARG.
 */
#ifndef W8A8_H
#define W8A8_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  W8A8_ERR_UNSUPPORTED is the counterpart of the NotImplementedError a
 * scheme lookup raises for an unsupported parameter combination ([vLLM-W8A8] 4.3). */
typedef enum {
  W8A8_OK = 0,
  W8A8_ERR_INVALID_ARG = 1,   /* bad size, null pointer, bad mode */
  W8A8_ERR_UNSUPPORTED = 2,   /* mode combination or device not supported */
  W8A8_ERR_MISALIGNED = 3,    /* pointer or leading dimension breaks an alignment rule */
  W8A8_ERR_BAD_SCALE = 4,     /* device side: illegal FP8 block scale / NaN code */
  W8A8_ERR_TIMEOUT = 5,       /* device side: a bounded wait inside a kernel ran out */
  W8A8_ERR_CUDA = 6,          /* a CUDA runtime/driver call failed */
  W8A8_ERR_WORKSPACE = 7      /* workspace missing or too small */
} w8a8_status;

/* Activation quantization schemes ([vLLM-W8A8] 4.1: static per-tensor or dynamic
 * per-token, symmetric or asymmetric activations). */
typedef enum {
  W8A8_ACT_DYN_TOKEN_SYM = 0,
  W8A8_ACT_DYN_TOKEN_ASYM = 1,
  W8A8_ACT_STATIC_TENSOR_SYM = 2,
  W8A8_ACT_STATIC_TENSOR_ASYM = 3
} w8a8_act_mode;

/* Weight scale strategy ([vLLM-W8A8] 4.2: weight_scale [out_features, 1] for CHANNEL,
 * one value per layer for TENSOR).  Weights are always symmetric ([vLLM-W8A8] 4.1). */
typedef enum { W8A8_W_CHANNEL = 0, W8A8_W_TENSOR = 1 } w8a8_w_mode;

/* Human-readable name of a status code (static storage, never NULL). */
const char* w8a8_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int w8a8_version(void);

/* GEMM engine selection for w8a8_scaled_mm / w8a8_linear / w8a8_grouped_mm, a tuning and
 * testing control that applies to the calling host thread:
 *   0 = automatic (the warp-MMA weight-streaming kernel for dense calls with M <= 16, the
 *       tcgen05 kernel otherwise), 1 = always tcgen05, 2 = always the warp-MMA kernel.
 * Both engines compute the same exact int32 sums and the same epilogue. */
w8a8_status w8a8_set_gemm_engine(int engine);

/*
 * Bounds-checked build.  Built with -DW8A8_DEBUG (libw8a8_debug.so, `build.py --debug`),
 * every kernel checks the index invariants of its global-memory accesses (row within the
 * rows, column block within K or N, segment within E, partial tile within the split
 * scratch); a violated one records a site code in a caller-provided device int32 (the
 * first code wins, 0 = none) and skips that access instead of trapping.  No counterpart on
 * the pages: it is a test instrument.
 *   w8a8_debug_set_error_word: registers the device word (device pointer, or NULL to stop
 *   recording); W8A8_ERR_UNSUPPORTED in the release build.  w8a8_debug_build: 1 in the
 *   bounds-checked build, 0 otherwise.
 */
w8a8_status w8a8_debug_set_error_word(int32_t* word);
int w8a8_debug_build(void);

/*
 * w8a8_test_requant_wait_fault -- test hook for the device-side timeout path
 * ([Kunlun-INT8] 验证: the converter's tests include illegal inputs; this one makes a wait
 * run out on purpose).  Not for production use; process-wide; off by default.
 *   wait_limit_ns: limit of the requantizer row ring's bounded waits (100 us .. 2 s; 0
 *   restores the default 2 s).  extra_tx_bytes (0 .. 4096): bytes that the barrier of the
 *   first row of the next ring launches expects beyond what the row's bulk copy delivers,
 *   so that wait cannot complete: the copy itself lands as usual, the wait runs out after
 *   wait_limit_ns, the kernel records W8A8_ERR_TIMEOUT in dev_status and returns; nothing
 *   faults or hangs, and the context stays usable.  Call with (0, 0) to switch it off.
 *   Returns W8A8_ERR_INVALID_ARG for values out of range.
 */
w8a8_status w8a8_test_requant_wait_fault(uint32_t extra_tx_bytes, uint64_t wait_limit_ns);

/*
 * w8a8_quantize_act -- activation quantization ([SGLang-CT] item 3, per_token_quant_int8;
 * per-row rule of [Kunlun-INT8] 转换关系; modes of [vLLM-W8A8] 4.1/4.2).
 *   x      bf16 [M, K] with row stride ldx (elements, ldx >= K).
 *   q      int8 [M, K] contiguous (output).
 *   scale  DYN modes: float [M] output, s[m] = rowabsmax/127 (sym) or (max-min)/255 (asym);
 *          STATIC modes: float [1] input (the calibrated input_scale).
 *   zp     DYN_ASYM: int32 [M] output zero points; STATIC_ASYM: int32 [1] input
 *          (input_zero_point, an int8 value); symmetric modes: ignored (may be NULL).
 * Rounding: q = clamp(rint(x / s) (+ zp), lo, hi), IEEE float32 division, ties to even;
 * [lo, hi] = [-127, 127] symmetric, [-128, 127] asymmetric.  All-zero rows give q = 0, s = 1.
 * The static scale must be finite and positive (results are unspecified otherwise).
 * Activations are expected finite: a row holding NaN or an infinity gets unspecified codes
 * (saturated to the code range; nothing faults).
 * M == 0 or K == 0 is a no-op returning W8A8_OK.
 */
w8a8_status w8a8_quantize_act(const void* x, int64_t M, int64_t K, int64_t ldx, int mode,
                              int8_t* q, float* scale, int32_t* zp, cudaStream_t stream);

/*
 * w8a8_scaled_mm -- INT8 x INT8 -> INT32 GEMM with the fused scale/azp/bias epilogue
 * ([SGLang-CT] item 3: int8_scaled_mm(x_q, W, x_scale, w_scale, out_dtype, bias);
 * item 4: azp_adj correction).
 *   xq      int8 [M, K] contiguous (quantized activations).
 *   wq      int8 [N, K] contiguous ([vLLM-W8A8] 4.2 layout [out_features, in_features]).
 *   act_mode  which activation scheme produced xq (w8a8_act_mode):
 *             DYN_TOKEN_SYM    s_x float [M]; zp, azp_adj unused.
 *             DYN_TOKEN_ASYM   s_x float [M]; zp int32 [M]; azp_adj int32 [N] = sum_k wq[n,k].
 *             STATIC_SYM       s_x float [1].
 *             STATIC_ASYM      s_x float [1]; azp_adj int32 [N] premultiplied by the
 *                              input zero point; zp unused.
 *   w_mode  W8A8_W_CHANNEL: s_w float [N];  W8A8_W_TENSOR: s_w float [1].
 *   w_sumsq int32 [N] = sum_k wq[n,k]^2 (w8a8_weight_sumsq / w8a8_quantize_weight), or NULL.
 *           Optional, results do not depend on it: with an asymmetric act_mode, the
 *           tensor-core engine may then finish more tiles in one exact fp32 pass.  Each
 *           partial sum is at most ||x_m||_2 * ||w_n||_2, and a tile is exact in fp32 when
 *           that stays below 2^24.  Without it, the test is 127 * L1(x_m) < 2^24 alone;
 *           affine codes, and symmetric codes of rows without outliers, often fail that test
 *           and their tiles then accumulate in 1024-K chunks.  Used in every mode.
 *   bias    bf16 [N] or NULL.
 *   y       bf16 [M, N] contiguous (output).
 *   workspace  device scratch of at least w8a8_scaled_mm_workspace_size(M, K) bytes,
 *              256-byte aligned (the tensor-core engine stages the activations there as
 *              fp16 integer codes with their row L1 norms and sums of squares).  May be
 *              NULL only when the warp-MMA engine runs (M <= 16 under automatic selection).
 *              Bytes past that size are split scratch (see w8a8_splitk_workspace_size).
 * Epilogue, float32 with one rounding per step and no fused multiply-add:
 *   c = acc - zp[m]*azp_adj[n] (exact integer, rounded to float32);
 *   y = bf16_rne( (s_x[m]*s_w[n]) * c (+ bias[n]) ).
 * The int32 accumulation is exact for all int8 inputs.
 * Requirements: K % 16 == 0; xq, wq and y 16-byte aligned; 1 <= K <= 131072.
 * dev_status: optional (see conventions); a kernel whose internal wait ran out writes
 * W8A8_ERR_TIMEOUT there and leaves y unspecified.
 */
size_t w8a8_scaled_mm_workspace_size(int64_t M, int64_t K);
w8a8_status w8a8_scaled_mm(const int8_t* xq, const int8_t* wq, int64_t M, int64_t N, int64_t K,
                           int act_mode, const float* s_x, const int32_t* zp,
                           const int32_t* azp_adj, int w_mode, const float* s_w,
                           const int32_t* w_sumsq, const void* bias, void* y, void* workspace,
                           size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/*
 * w8a8_splitk_workspace_size -- scratch for K-split GEMMs.
 *   The tensor-core engine runs persistent CTA pairs over 256 x 256 output tiles.  A launch
 *   whose tiles do not fill its last wave of pairs (and one of a few hundred rows, which fills
 *   no wave) leaves pairs idle; with this much scratch it cuts the tiles past its last full
 *   wave (all of them when there is none) along K at 1024-element boundaries, into as many
 *   parts as fill the idle pairs, runs the parts there, and a second kernel adds their int32
 *   partial sums and applies the epilogue: the result is the same integer, so y is unchanged.
 *   Returns the extra bytes a w8a8_scaled_mm or w8a8_linear call of this shape uses for it on
 *   the current device, placed right after the call's own workspace size (so a workspace of
 *   w8a8_linear_workspace_size(M, K, mode) + w8a8_splitk_workspace_size(M, N, K) bytes).  0
 *   when the shape does not split, or for invalid sizes or devices.  The scratch needs no
 *   initialization; calls that share a workspace must not overlap.  At most
 *   (SMs / 2) * 256 KiB.
 */
size_t w8a8_splitk_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * w8a8_linear -- the whole layer forward: quantize x (any act_mode) then w8a8_scaled_mm
 * ([SGLang-CT] item 3 apply_weights; [vLLM-W8A8] 4.2 apply_weights(layer, x, bias)).
 *   x bf16 [M, K] (row stride ldx); wq/s_w/azp_adj/w_sumsq/bias as for w8a8_scaled_mm.
 *   input_scale / input_zero_point: float [1] / int32 [1] for the static modes, else NULL.
 *   workspace: device buffer of at least w8a8_linear_workspace_size(M, K, act_mode) bytes,
 *   256-byte aligned; it holds the quantized activations (in the format the selected GEMM
 *   engine reads), their scales and zero points between the two kernels.  Bytes past that
 *   size are split scratch (see w8a8_splitk_workspace_size).
 */
size_t w8a8_linear_workspace_size(int64_t M, int64_t K, int act_mode);
w8a8_status w8a8_linear(const void* x, int64_t M, int64_t K, int64_t ldx, int act_mode,
                        const float* input_scale, const int32_t* input_zero_point,
                        const int8_t* wq, int64_t N, int w_mode, const float* s_w,
                        const int32_t* azp_adj, const int32_t* w_sumsq, const void* bias, void* y,
                        void* workspace, size_t workspace_bytes,
                        int32_t* dev_status, cudaStream_t stream);

/*
 * w8a8_quantize_weight -- per-output-channel symmetric weight quantization
 * ([vLLM-W8A8] 4.2: int8 weight [out_features, in_features], float32 weight_scale
 * [out_features, 1]; rule of [Kunlun-INT8] 转换关系: s = rowabsmax/127,
 * q = clamp(round(W/s), -127, 127), all-zero row -> q = 0, s = 1).
 *   w bf16 [N, K] contiguous;  wq int8 [N, K] (output);  s_w float [N] (output);
 *   azp_adj int32 [N] (optional output, NULL to skip): sum_k wq[n, k] ([SGLang-CT] item 4).
 *   w_sumsq int32 [N] (optional output, NULL to skip): sum_k wq[n, k]^2 (see
 *   w8a8_weight_sumsq).
 */
w8a8_status w8a8_quantize_weight(const void* w, int64_t N, int64_t K, int8_t* wq, float* s_w,
                                 int32_t* azp_adj, int32_t* w_sumsq, cudaStream_t stream);

/*
 * w8a8_weight_sumsq -- w_sumsq[n] = sum_k wq[n, k]^2 (int32, exact for K <= 131072) of an
 * already-quantized weight, the optional operand of the GEMM entry points that lets them
 * prove more tiles exact in one fp32 pass (Cauchy-Schwarz; see w8a8_scaled_mm).  The pages
 * have no counterpart: it is this engine's exactness bookkeeping, computed once per weight
 * like azp_adj.  wq int8 [N, K] (device); w_sumsq int32 [N] (device, 4-byte aligned).
 */
w8a8_status w8a8_weight_sumsq(const int8_t* wq, int64_t N, int64_t K, int32_t* w_sumsq,
                              cudaStream_t stream);

/*
 * w8a8_azp_adj -- azp_adj[n] = input_zero_point * sum_k wq[n, k] for an int8 weight that
 * is already quantized ([SGLang-CT] item 4: computed once after loading; premultiplied by
 * the zero point for the static scheme).  input_zero_point: int32 [1] device value, or
 * NULL for the plain column sum used by the dynamic asymmetric scheme.
 */
w8a8_status w8a8_azp_adj(const int8_t* wq, int64_t N, int64_t K, const int32_t* input_zero_point,
                         int32_t* azp_adj, cudaStream_t stream);

/*
 * fp8block_to_int8_rowwise -- FP8 E4M3 block-scaled weight -> INT8 weight with one float32
 * scale per output row ([Kunlun-INT8] 转换关系):
 *   Wf[i,j] = e4m3(w[i,j]) * scale_inv[i/128, j/128]   (the "_inv" scale multiplies)
 *   s[i] = max_j |Wf[i,j]| / 127;  q = clamp(rint(Wf / s), -127, 127);
 *   all-zero row -> q = 0, s = 1.
 *   w         uint8 [N, K] E4M3 codes (the "fn" encoding: no infinities, 0x7F/0xFF NaN).
 *   scale_inv float [ceil(N/128), ceil(K/128)] row-major.
 *   q int8 [N, K], s float [N] (outputs).  Any K >= 1 is accepted, aligned or not.
 * A row touching a non-finite or <= 0 block scale, holding a NaN code, or whose dequantized
 * values overflow, gets q = 0, s = 1 and W8A8_ERR_BAD_SCALE is written to dev_status
 * ([Kunlun-INT8] 验证 tests illegal scales).
 */
w8a8_status fp8block_to_int8_rowwise(const uint8_t* w, const float* scale_inv, int64_t N, int64_t K,
                                     int8_t* q, float* s, int32_t* dev_status, cudaStream_t stream);

/*
 * fp8block_to_int8_rowwise_batched -- the same for `count` matrices in one launch per up to
 * 64 matrices.  The four pointer arrays and the N/K arrays are HOST arrays of length count
 * holding device pointers / sizes; they are read before the call returns.
 */
w8a8_status fp8block_to_int8_rowwise_batched(int count, const uint8_t* const* w,
                                             const float* const* scale_inv, const int64_t* N,
                                             const int64_t* K, int8_t* const* q, float* const* s,
                                             int32_t* dev_status, cudaStream_t stream);

/*
 * fp8block_to_int8_rowwise_batched_adj -- the batched requantization that also writes, for
 * each matrix whose azp_adj[i] is non-null, the row sums of its int8 codes:
 *   azp_adj[i][n] = sum_k q_i[n, k]   (int32, exact; 0 for a row zeroed as illegal)
 * i.e. the weight-side correction term of asymmetric activations ([SGLang-CT] item 4,
 * AZP 보정: azp_adj is the column sum of the int8 weight along K), produced in the same pass
 * that converts an FP8-block checkpoint ([Kunlun-INT8] FP8 -> INT8 conversion), so the
 * converted weight is never read again to form it.  azp_adj is a HOST array of length count
 * (or null for none) of device int32 [N_i] pointers (4-byte aligned, or null).  Everything
 * else is as in fp8block_to_int8_rowwise_batched.
 */
w8a8_status fp8block_to_int8_rowwise_batched_adj(int count, const uint8_t* const* w,
                                                 const float* const* scale_inv, const int64_t* N,
                                                 const int64_t* K, int8_t* const* q, float* const* s,
                                                 int32_t* const* azp_adj, int32_t* dev_status,
                                                 cudaStream_t stream);

/*
 * w8a8_moe_route -- the routing that feeds the MoE INT8 path ([SGLang-CT] file tree:
 * compressed_tensors_w8a8_int8_moe; [Kunlun-INT8] MoE method over experts w1/w2/w3; the
 * pages leave the router to the framework, so the rule is the plain one):
 *   topk_ids[t, :] = the topk experts with the largest logits, in descending order, equal
 *                    logits broken by the lower expert index;
 *   topk_w[t, j]   = softmax(logits[t, :])[topk_ids[t, j]] over all E experts (fp32,
 *                    max-subtracted; not renormalised over the chosen experts);
 * then the T*topk (token, slot) pairs sorted stably by expert (ties keep token, then slot
 * order) -- a counting sort:
 *   seg_offsets[e] .. seg_offsets[e+1]  the routed rows of expert e (seg_offsets[E] = T*topk);
 *   row_index[r]   = token of routed row r      (what w8a8_moe_quantize_gather reads);
 *   row_of[t, j]   = routed row of (t, slot j)  (what w8a8_moe_combine reads).
 *   logits float [T, E]; topk_ids int32 [T, topk]; topk_w float [T, topk];
 *   seg_offsets int64 [E+1]; row_index int64 [T*topk]; row_of int64 [T, topk] (all device).
 *   1 <= E <= 256, 1 <= topk <= min(8, E).  workspace: at least
 *   w8a8_moe_route_workspace_size(T, E, topk) bytes (4-byte aligned; null allowed for T = 0).
 */
size_t w8a8_moe_route_workspace_size(int64_t T, int E, int topk);
w8a8_status w8a8_moe_route(const float* logits, int64_t T, int E, int topk, int32_t* topk_ids,
                           float* topk_w, int64_t* seg_offsets, int64_t* row_index, int64_t* row_of,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * w8a8_requantize_max_scale -- one per-tensor scale for a fused weight ([SGLang-CT] item 7,
 * 텐서별 스케일 후처리: requantize_with_max_scale; 설계 근거 3, Fused 모듈 호환).  A fused
 * module (e.g. Q/K/V stacked along the output dimension) whose P logical partitions were
 * quantized with their own per-tensor scales gets the largest of them as its single scale,
 * and every code is requantized against it, in place:
 *   s_max = max_p scales[p];
 *   wq[n, k] <- clamp(rint(RN(RN(q[n, k] * scales[p]) / s_max)), -127, 127)
 * for the rows n of partition p (fp32 multiply, IEEE fp32 division, ties to even).
 *   wq int8 [N, K] (device; read and rewritten in place; any K, 16-byte alignment and
 *   K % 16 == 0 take the vector path); scales float [P] (device); logical_widths int64 [P]
 *   (HOST, rows per partition, summing to N); 1 <= P <= 16; s_max float [1] (device, out).
 * A scale that is not positive and finite leaves wq and s_max untouched and writes
 * W8A8_ERR_BAD_SCALE to dev_status (may be null).
 */
w8a8_status w8a8_requantize_max_scale(int8_t* wq, int64_t N, int64_t K, const float* scales,
                                      const int64_t* logical_widths, int P, float* s_max,
                                      int32_t* dev_status, cudaStream_t stream);

/*
 * w8a8_grouped_mm -- MoE expert GEMMs over token-sorted segments ([SGLang-CT] MoE INT8
 * scheme; [Kunlun-INT8] W8A8 MoE method with per-channel symmetric expert weights and
 * per-token dynamic symmetric activations).  Rows [seg[e], seg[e+1]) of xq_sorted belong to
 * expert e and are multiplied by that expert's weight:
 *   y[r, :] = bf16( s_x[r] * s_w[e, n] * sum_k xq_sorted[r, k] * w[e, n, k] ).
 *   xq_sorted int8 [R, K];  s_x float [R];  w int8 [E, N, K];  s_w float [E, N];
 *   seg_offsets int64 [E+1] (DEVICE array, non-decreasing, seg[0] = 0, seg[E] = R);
 *   y bf16 [R, N].  R is seg[E]; max_rows is a host-side upper bound on R used to size the
 *   launch and the workspace (pass R when known).  workspace: at least
 *   w8a8_grouped_mm_workspace_size(max_rows, K) bytes, 256-byte aligned.  E <= 1024.
 *   w_sumsq: int32 [E, N] row sums of squares of the expert weights (w8a8_weight_sumsq over
 *   the E*N rows), or NULL; when given, tiles whose activation rows fail the L1 exactness
 *   test may still run in one pass by the Cauchy-Schwarz test (see w8a8_scaled_mm).
 *   Requirements as for w8a8_scaled_mm.
 */
size_t w8a8_grouped_mm_workspace_size(int64_t max_rows, int64_t K);
w8a8_status w8a8_grouped_mm(const int8_t* xq_sorted, const float* s_x, const int8_t* w,
                            const float* s_w, const int32_t* w_sumsq, const int64_t* seg_offsets,
                            int E, int64_t max_rows, int64_t N, int64_t K, void* y, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);

/*
 * w8a8_moe_quantize_gather -- per-token symmetric quantization of x rows taken in expert-
 * sorted order: for r in [0, R): (xq_sorted[r], s_x[r]) = quantize(x[row_index[r]]).
 *   x bf16 [T, K] (row stride ldx);  row_index int64 [R] (device);  xq_sorted int8 [R, K];
 *   s_x float [R].  Same rounding as w8a8_quantize_act in mode DYN_TOKEN_SYM.
 */
w8a8_status w8a8_moe_quantize_gather(const void* x, int64_t T, int64_t K, int64_t ldx,
                                     const int64_t* row_index, int64_t R, int8_t* xq_sorted,
                                     float* s_x, cudaStream_t stream);

/*
 * w8a8_silu_mul_quant -- glue between the two expert GEMMs: g = bf16(silu(h[:, :I]) * h[:, I:])
 * in float32 (gate columns first), then per-row symmetric quantization of g.
 *   h bf16 [R, 2I];  gq int8 [R, I];  s_g float [R].  I % 8 == 0.
 */
w8a8_status w8a8_silu_mul_quant(const void* h, int64_t R, int64_t I, int8_t* gq, float* s_g,
                                cudaStream_t stream);

/*
 * w8a8_moe_combine -- y[t, :] = bf16( sum_{j < topk} topk_w[t, j] * out[row_of[t, j], :] ),
 * float32, slots in order, one multiply and one add per slot.
 *   out bf16 [R, H];  row_of int64 [T, topk];  topk_w float [T, topk];  y bf16 [T, H].
 */
w8a8_status w8a8_moe_combine(const void* out, const int64_t* row_of, const float* topk_w,
                             int64_t T, int topk, int64_t H, void* y, cudaStream_t stream);

/*
 * Packed activations.  The tensor-core GEMM engine reads activations as fp16 integer codes
 * (every int8 value is exact in fp16) together with each row's L1 norm sum_k |q[r, k]|,
 * which tells the GEMM whether a single fp32 pass over K is provably exact.  The "packed"
 * entry points produce and consume that format in one caller buffer of
 * w8a8_act_packed_size(M, K) bytes (256-byte aligned): fp16 codes [M, K] row-major, then
 * int32 row L1 norms [M] at byte offset roundup(M*K*2, 256), immediately followed by the
 * int32 row sums of squares [M] of the codes (written by the asymmetric modes only).  The codes are the same integers the
 * int8 entry points produce; only their storage differs.  w8a8_linear runs
 * w8a8_quantize_act_packed followed by w8a8_scaled_mm_packed (for M > 16).
 * K % 16 == 0 for every packed entry point.
 */
size_t w8a8_act_packed_size(int64_t M, int64_t K);

/* w8a8_quantize_act with the packed output; scale / zp exactly as for w8a8_quantize_act. */
w8a8_status w8a8_quantize_act_packed(const void* x, int64_t M, int64_t K, int64_t ldx, int mode,
                                     void* packed, float* scale, int32_t* zp, cudaStream_t stream);

/* w8a8_scaled_mm reading packed activations (nothing is staged).  split_ws: optional K-split
 * scratch of w8a8_splitk_workspace_size(M, N, K) bytes, 256-byte aligned (NULL or fewer bytes:
 * no split). */
w8a8_status w8a8_scaled_mm_packed(const void* packed, const int8_t* wq, int64_t M, int64_t N,
                                  int64_t K, int act_mode, const float* s_x, const int32_t* zp,
                                  const int32_t* azp_adj, int w_mode, const float* s_w,
                                  const int32_t* w_sumsq, const void* bias, void* y,
                                  void* split_ws, size_t split_bytes, int32_t* dev_status,
                                  cudaStream_t stream);

/* w8a8_grouped_mm reading packed activations (max_rows: the rows the packed buffer holds). */
w8a8_status w8a8_grouped_mm_packed(const void* packed, const float* s_x, const int8_t* w,
                                   const float* s_w, const int32_t* w_sumsq,
                                   const int64_t* seg_offsets, int E, int64_t max_rows, int64_t N,
                                   int64_t K, void* y, int32_t* dev_status, cudaStream_t stream);

/* w8a8_moe_quantize_gather / w8a8_silu_mul_quant writing packed activations
 * (packed holds R rows; for the SiLU glue K is I). */
w8a8_status w8a8_moe_quantize_gather_packed(const void* x, int64_t T, int64_t K, int64_t ldx,
                                            const int64_t* row_index, int64_t R, void* packed,
                                            float* s_x, cudaStream_t stream);
w8a8_status w8a8_silu_mul_quant_packed(const void* h, int64_t R, int64_t I, void* packed,
                                       float* s_g, cudaStream_t stream);

/*
 * w8a8_moe_quantize_scatter_packed -- the packed result of w8a8_moe_quantize_gather_packed,
 * computed the other way round ([SGLang-CT] MoE INT8 scheme: per-token dynamic symmetric
 * activations of the expert GEMMs): each token row x[t] is quantized once and its codes,
 * L1 norm and scale are written to the routed rows row_of[t, j], j < topk, instead of
 * quantizing every routed row from its token.
 *   x bf16 [T, K] (row stride ldx; 16-byte aligned rows);  row_of int64 [T, topk] (device;
 *   the w8a8_moe_route output: distinct rows in [0, R));  packed: R rows of the packed
 *   activation format;  s_x float [R].  K % 16 == 0, K <= 16384, 1 <= topk <= 32.
 *   Routed rows that no (t, j) names are left untouched.  Returns W8A8_ERR_MISALIGNED for
 *   unaligned x, row_of or packed, W8A8_ERR_INVALID_ARG for sizes out of range.
 */
w8a8_status w8a8_moe_quantize_scatter_packed(const void* x, int64_t T, int64_t K, int64_t ldx,
                                             const int64_t* row_of, int topk, int64_t R, void* packed,
                                             float* s_x, cudaStream_t stream);

/*
 * w8a8_scaled_mm_noalloc -- w8a8_scaled_mm without a workspace, for callers that cannot
 * allocate device memory (a host runtime that owns only the tensors it passes in and has no
 * allocator to lend, or a latency-critical path where cudaMalloc's possible device-wide
 * synchronization is not allowed).  The pages describe no counterpart: it exists only for
 * such callers.
 *   Arguments, results and requirements are those of w8a8_scaled_mm, except that there is
 *   no workspace: the activations are staged in a 36 MiB buffer owned by the library (a
 *   device array placed in GPU memory when the library's module is loaded on a device and
 *   kept until the process exits).  It always runs the tensor-core engine.
 *   Limit: roundup(M*K*2, 256) + roundup(M*8, 256) <= 36 MiB (e.g. M*K up to 4096 x 4096);
 *   larger problems return W8A8_ERR_WORKSPACE before any launch.
 *   The first call on each device looks up the buffer's device address (no allocation) and
 *   caches it with the CUDA context it was found in; make that first call before any stream
 *   capture.  A call under another context (a non-primary context, or the new primary
 *   context after cudaDeviceReset) looks the address up again, and that call too must come
 *   before any capture.
 *   All calls on a device share the one buffer, which keeps the last call's contents; every
 *   call rewrites all of it that it reads, so nothing needs clearing.  Calls whose work
 *   overlaps on the same GPU (e.g. issued to two streams at once) race on the buffer.
 */
w8a8_status w8a8_scaled_mm_noalloc(const int8_t* xq, const int8_t* wq, int64_t M, int64_t N,
                                   int64_t K, int act_mode, const float* s_x, const int32_t* zp,
                                   const int32_t* azp_adj, int w_mode, const float* s_w,
                                   const void* bias, void* y, int32_t* dev_status,
                                   cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W8A8_H */
