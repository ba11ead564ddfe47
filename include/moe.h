/*
 * moe.h -- C ABI of libmoe: the forward pass of a DeepSeekMoE layer with
 * auxiliary-loss-free (bias-steered) top-k routing, on one B300 (sm_103a).
 *
 * The layer, as the pages state it:
 *   - "DeepSeek-V3 详解" (yudonglee.me), section 2.2: fine-grained routed
 *     experts plus one always-on shared expert, top-8 of 256 per token;
 *     section 2.3: a per-expert bias, update speed gamma = 0.001.
 *   - "deepseek-v3-report" (dynmi.github.io), load-balancing paragraph: the
 *     bias b_i is added to the routing score, lowered for an overloaded expert
 *     and raised for an idle one, and stays out of the gradient.
 *   - "DeepSeek-V3 技术报告要点" (deepseek.csdn.net), section 4.2: the bias is
 *     moved from the load observed in each batch; section 3 table: hidden
 *     size 7168, expert intermediate size 2048; section 1: SwiGLU FFN.
 *   - FP8 path: "DeepSeek-V3 详解", section 4.2 (1x128 activation tiles,
 *     128x128 weight blocks) and 4.3 (FP32 accumulation).
 * Where the pages are silent the library takes these readings: affinity
 * s = sigmoid(x . w_i [+ o_i]); selection by the k largest s + b (descending,
 * ties to the lower expert index); gate = s / (sum of s over the chosen k);
 * shared experts ungated; output excludes the residual.
 *
 * Conventions for every call:
 *   - Every pointer is a DEVICE pointer unless stated; the caller owns all
 *     memory, including the workspace.  The library never allocates or frees.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream);
 *     none synchronises the host, except moe_get_device_status.
 *   - A call runs on the calling host thread's current CUDA device, which must
 *     own the buffers and the stream; in a thread that has not used the CUDA
 *     runtime yet, the library makes that device's primary context current.
 *   - Arguments are validated before anything is launched; a non-OK status
 *     means nothing was enqueued.  No C++ exception crosses the ABI.
 *   - Row-major tensors must start on a 16-byte boundary.
 *   - With T = 0 every buffer sized by the tokens (or the routed rows) may be
 *     NULL; the calls then only produce what does not depend on tokens (zero
 *     counts and offsets, an unchanged bias, zero weight gradients).
 *   - bf16 tensors are passed as `const void*` holding IEEE bfloat16 bits;
 *     FP8 tensors hold OCP E4M3 ("e4m3fn") bytes.
 *   - Errors found on the device (a wait that timed out, an index out of
 *     range) are recorded in a status word inside the workspace and read back
 *     with moe_get_device_status.
 *   - Shape limits: T >= 0, d % 128 == 0 (128 <= d <= 65536),
 *     I % 128 == 0 (128 <= I <= 65536), 1 <= E <= 256, 0 <= S <= 8,
 *     1 <= k <= min(E, 16), (T*k + S*T) * max(d, I) < 2^31.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad shape, bad gamma          */
  MOE_ERR_UNSUPPORTED = 2, /* valid layer, outside this library's limits  */
  MOE_ERR_ALIGNMENT = 3,   /* a tensor does not start on 16 bytes         */
  MOE_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required  */
  MOE_ERR_CUDA = 5,        /* a CUDA runtime / driver call failed         */
  MOE_ERR_TIMEOUT = 6,     /* device: a bounded wait gave up              */
  MOE_ERR_DEVICE = 7       /* device: an index or count was inconsistent  */
} moe_status_t;

/* Arithmetic of the expert GEMMs.  FP8 ("DeepSeek-V3 详解" 4.2-4.3): E4M3 codes with one
 * scale per 1x128 activation tile (per token per 128 channels) and per 128x128 weight
 * block, FP32 accumulation, bf16 output.  The pages fix the granularity, not the scale
 * format: MOE_FP8_E4M3 takes scale = amax / 448 in FP32 and promotes each 128-wide K
 * block's partial product through registers; MOE_FP8_E4M3_POW2 takes the smallest power
 * of two with amax <= 448 * scale (codes in (224, 448] at the tile maximum), which the
 * tensor core applies itself as UE8M0 block scales (kind::mxf8f6f4), accumulating in FP32
 * in TMEM.  Both keep the scales as FP32 arrays of the same shapes; POW2 scales must be
 * powers of two (moe_permute and moe_quantize_weights_fp8_pow2 make them so).  POW2
 * layers use the permuted copy (moe_expert_ffn_gather returns MOE_ERR_UNSUPPORTED). */
typedef enum { MOE_BF16 = 0, MOE_FP8_E4M3 = 1, MOE_FP8_E4M3_POW2 = 2 } moe_dtype_t;

/* T tokens, d model width, E routed experts, S shared experts, k experts
 * chosen per token, I expert intermediate size; dtype of the expert GEMMs.
 * n_group, topk_group: group-limited routing ("DeepSeek-V3 技术报告要点" section 9
 * table; "DeepSeek-V3 详解" 2.4, experts of a token on at most M nodes): the E
 * experts form n_group contiguous groups, a group's score is the FP32 sum of its
 * ceil(k/topk_group) largest biased scores (descending), only the topk_group best
 * groups (ties to the lower group) are eligible for the top-k.  0, 0 = no groups.
 * Limits: E % n_group == 0, n_group <= 32, 1 <= topk_group <= n_group,
 * k <= topk_group * E/n_group, ceil(k/topk_group) <= E/n_group. */
typedef struct {
  int T, d, E, S, k, I;
  moe_dtype_t dtype;
  int n_group, topk_group;
} moe_shape_t;

/* A CUDA stream (same type as cudaStream_t). */
typedef struct CUstream_st* moe_stream_t;

/* Bytes of workspace every call below needs for `shape` (the maximum over all
 * calls, so one buffer serves them all); 0 if the shape is invalid.  The
 * workspace must start on 256 bytes and its first 2048 bytes (the control
 * block: the device status word, and the router's load counters, which every
 * moe_route call leaves cleared) must be zero before its first use; the rest
 * needs no initialisation.  Calls that share a workspace run in stream order
 * (not concurrently). */
MOE_API size_t moe_workspace_bytes(const moe_shape_t* shape);

/* Router ("deepseek-v3-report", load-balancing paragraph; "DeepSeek-V3 详解"
 * 2.3).  For every token t and routed expert i:
 *     z = x[t] . w_router[i] (+ logit_offset[i]),  s = sigmoid(z),
 *     chosen = the k largest s + bias[i] (descending, ties -> lower i),
 *     gate   = s[chosen] / sum_j s[chosen_j].
 *   x            bf16 [T, d]          token activations (input)
 *   w_router     bf16 [E, d]          router weight (input)
 *   bias         f32  [E]             selection bias b (input; selection only)
 *   logit_offset f32  [E] or NULL     per-expert logit offset added to z
 *   topk_idx     int32 [T, k]  out    chosen experts
 *   topk_gate    f32  [T, k]   out    gates
 *   counts       int32 [E]     out    tokens routed to each expert (load)
 *   offsets      int32 [E+1]   out    exclusive prefix sum of counts
 * z is accumulated in FP32 on the tensor cores; s, s + b and the gates are
 * FP32.  Deterministic run to run.  One kernel launch (T > 0): the load is
 * summed in the workspace's control block and written out, with its prefix
 * sum, by the last block to finish. */
MOE_API moe_status_t moe_route(const moe_shape_t* shape, const void* x, const void* w_router,
                       const float* bias, const float* logit_offset, int32_t* topk_idx,
                       float* topk_gate, int32_t* counts, int32_t* offsets, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* Dispatch: group the (token, slot) pairs by expert, tokens ascending inside
 * an expert (the single-GPU form of the all-to-all dispatch in "DeepSeek-V3
 * Overview and Key Innovations", Training Infrastructure and Optimization).
 *   x            bf16 [T, d]          (input)
 *   topk_idx     int32 [T, k]         (input, values in [0, E))
 *   offsets      int32 [E+1]          (input, from moe_route)
 *   x_perm       [T*k, d]      out    bf16, or E4M3 bytes when dtype = FP8
 *   x_perm_scale f32 [T*k, d/128] out FP8 only (1x128 tile scales), else NULL
 *   perm_token   int32 [T*k]   out    token of each permuted row
 *   inv_pos      int32 [T, k]  out    permuted row of (t, j)
 * FP8 quantisation (per 1x128 tile, the scale of the layer's dtype, RNE,
 * saturating) is done on the way.  Inconsistent idx/offsets set MOE_ERR_DEVICE.
 * x_perm = NULL (and x_perm_scale = NULL): only perm_token and inv_pos are
 * built, no row is copied -- the input of moe_expert_ffn_gather. */
MOE_API moe_status_t moe_permute(const moe_shape_t* shape, const void* x, const int32_t* topk_idx,
                         const int32_t* offsets, void* x_perm, float* x_perm_scale,
                         int32_t* perm_token, int32_t* inv_pos, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* Experts ("DeepSeek-V3 技术报告要点" section 1 and section 3 table): for every
 * routed expert e its rows of x_perm, and for every shared expert s all T rows
 * of x, go through the SwiGLU FFN
 *     h = silu(X W_gate^T) * (X W_up^T),   Y = h W_down^T.
 *   x_perm      [T*k, d]   bf16 / E4M3 (input, from moe_permute)
 *   x_perm_scale f32 [T*k, d/128] FP8 only, else NULL
 *   x           bf16 [T, d]           input of the shared experts
 *   offsets     int32 [E+1]           routed group boundaries in x_perm
 *   w_gate_up   [E+S, 2I, d]  bf16 / E4M3: rows 0..I-1 gate, I..2I-1 up;
 *               experts E..E+S-1 are the shared experts
 *   w_gu_scale  f32 [E+S, 2I/128, d/128]  FP8 only (128x128 block scales)
 *   w_down      [E+S, d, I]   bf16 / E4M3
 *   w_down_scale f32 [E+S, d/128, I/128]  FP8 only
 *   y           bf16 [T*k + S*T, d] out   rows 0..T*k-1 follow x_perm; row
 *               T*k + s*T + t is shared expert s on token t
 * FP32 accumulation; h is rounded to bf16 (BF16) or quantised per 1x128 to
 * E4M3 (FP8) before the down projection. */
MOE_API moe_status_t moe_expert_ffn(const moe_shape_t* shape, const void* x_perm, const float* x_perm_scale,
                            const void* x, const int32_t* offsets, const void* w_gate_up,
                            const float* w_gu_scale, const void* w_down, const float* w_down_scale,
                            void* y, void* ws, size_t ws_bytes, moe_stream_t stream);

/* The expert FFN with the dispatch copy fused into the gate/up GEMM: routed
 * row r of expert e is read straight from x[perm_token[r]] while the GEMM
 * stages its operand, so no x_perm is written or read (the single-GPU form of
 * the dispatch step in "DeepSeek-V3 Overview and Key Innovations", Training
 * Infrastructure and Optimization, folded into the experts of "DeepSeek-V3
 * 技术报告要点" section 1).  Same arithmetic and bit-identical y as
 * moe_expert_ffn on the rows that moe_permute would have written.
 *   x           bf16 [T, d]           input (routed and shared experts)
 *   perm_token  int32 [T*k]           from moe_permute (values in [0, T); an
 *                                     out-of-range value sets MOE_ERR_DEVICE
 *                                     and row 0 is read instead)
 *   offsets, w_gate_up, w_gu_scale, w_down, w_down_scale, y: as moe_expert_ffn
 * FP8: x is quantised per 1x128 tile to E4M3 inside the call (one copy of the
 * T rows in `ws`), exactly as moe_permute quantises each permuted row. */
MOE_API moe_status_t moe_expert_ffn_gather(const moe_shape_t* shape, const void* x, const int32_t* perm_token,
                                           const int32_t* offsets, const void* w_gate_up,
                                           const float* w_gu_scale, const void* w_down,
                                           const float* w_down_scale, void* y, void* ws, size_t ws_bytes,
                                           moe_stream_t stream);

/* Combine: the layer output of each token is its shared experts' outputs, ungated,
 * plus its k routed experts' outputs weighted by their gates ("deepseek-v3-report",
 * model table: 8 routed + 1 shared experts per token; "拆解DeepSeek V3", section
 * "让256个专家都干活": the shared expert serves every token; the single-GPU form of
 * the all-to-all combine in "DeepSeek-V3 Overview and Key Innovations", Training
 * Infrastructure and Optimization):
 *     out[t] = sum_s y[T*k + s*T + t] + sum_j topk_gate[t, j] * y[inv_pos[t, j]]
 * (shared experts first, then slots j = 0..k-1, FP32 sum, bf16 store).
 *   y bf16 [T*k + S*T, d]; topk_gate f32 [T, k]; inv_pos int32 [T, k];
 *   out bf16 [T, d] (out).  Deterministic run to run. */
MOE_API moe_status_t moe_combine(const moe_shape_t* shape, const void* y, const float* topk_gate,
                         const int32_t* inv_pos, void* out, moe_stream_t stream);

/* Bias update ("DeepSeek-V3 详解" 2.3, "deepseek-v3-report"):
 *     bias[i] += gamma * sign(T*k/E - counts[i]),  sign(0) = 0,
 * the sign decided on integers, the add in FP32.  In place on `bias` [E]. */
MOE_API moe_status_t moe_bias_update(const moe_shape_t* shape, const int32_t* counts, float* bias,
                             float gamma, moe_stream_t stream);

/* The whole layer: moe_route, the dispatch, the expert FFN, moe_combine and,
 * when update_bias != 0, moe_bias_update with this batch's counts (after the
 * routing has used the old bias).  This is the MoE layer of "DeepSeek-V3 详解"
 * 2.2-2.3 (fine-grained routed experts plus a shared expert, selection by the
 * biased score, the bias moved after each step) with the sizes of
 * "DeepSeek-V3 技术报告要点" section 3, and the per-batch bias update of its
 * section 4.2.  topk_idx, topk_gate and counts are optional
 * outputs (NULL keeps them in the workspace).  All intermediates live in `ws`.
 * The dispatch takes one of two forms (moe_forward_gathers tells which; both
 * give bit-identical results): for batches with T*k <= 4096 moe_permute builds
 * only the tables and moe_expert_ffn_gather reads the routed rows from x; for
 * larger batches moe_permute writes the permuted copy and moe_expert_ffn reads
 * it with whole-tile loads, which keeps the tensor cores fed better. */
MOE_API moe_status_t moe_forward(const moe_shape_t* shape, const void* x, const void* w_router,
                         float* bias, const float* logit_offset, const void* w_gate_up,
                         const float* w_gu_scale, const void* w_down, const float* w_down_scale,
                         void* out, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                         float gamma, int update_bias, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* 1 if moe_forward fuses the dispatch into the expert GEMM for this shape
 * (moe_permute tables only + moe_expert_ffn_gather), 0 if it writes the
 * permuted copy (moe_permute + moe_expert_ffn), -1 for an invalid shape. */
MOE_API int moe_forward_gathers(const moe_shape_t* shape);

/* The expert FFN (same arguments and results as moe_expert_ffn) for callers
 * that cannot allocate device memory -- a plugin inside a host framework that
 * owns all device memory and offers no workspace, or a serving loop that
 * forbids cudaMalloc after start-up.  The paper has no counterpart; this is a
 * deployment convenience of the library.
 *   - Scratch (status word, schedule, the E4M3 copy of x on the FP8 path, the
 *     SwiGLU intermediate h) comes from one 64 MiB array compiled into the
 *     library, held on every GPU that loads the library until the process
 *     exits.  Layers needing more scratch are rejected with MOE_ERR_WORKSPACE
 *     before anything is enqueued; at d=7168, 256+1 experts, top-8, I=2048 the
 *     scratch is about 36 KB per token in bf16 (up to about 1800 tokens) and
 *     26 KB per token in FP8 (up to about 2500 tokens).
 *   - The first call on a device looks up the array's address; make that call
 *     before any stream capture.
 *   - All calls share the array; overlapping calls on the GPU race and give
 *     wrong results.  The status word is cleared at the start of each call;
 *     read it with moe_get_static_device_status.
 *   - Allocates nothing (no cudaMalloc / cudaFree). */
MOE_API moe_status_t moe_expert_ffn_static(const moe_shape_t* shape, const void* x_perm,
                                           const float* x_perm_scale, const void* x,
                                           const int32_t* offsets, const void* w_gate_up,
                                           const float* w_gu_scale, const void* w_down,
                                           const float* w_down_scale, void* y, moe_stream_t stream);

/* Reads (synchronising `stream`) and clears the device status word of the array
 * that moe_expert_ffn_static uses on the current device, as moe_get_device_status
 * does for a workspace: MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE (MOE_ERR_CUDA if
 * the read fails).  The paper has no counterpart. */
MOE_API moe_status_t moe_get_static_device_status(moe_stream_t stream);

/* FP8 weight preparation ("DeepSeek-V3 详解" 4.2): quantise `w` bf16
 * [G, N, K] (N % 128 == 0, K % 128 == 0) per 128x128 block to E4M3 `w_q`
 * [G, N, K] with f32 scales `w_scale` [G, N/128, K/128] (scale = amax/448,
 * 1 for an all-zero block).  Used once, before the FP8 layer runs. */
MOE_API moe_status_t moe_quantize_weights_fp8(int G, int N, int K, const void* w, void* w_q,
                                      float* w_scale, moe_stream_t stream);

/* As moe_quantize_weights_fp8, with power-of-two block scales (the smallest power of
 * two with amax <= 448 * scale, 1 for an all-zero block): the weights of a
 * MOE_FP8_E4M3_POW2 layer. */
MOE_API moe_status_t moe_quantize_weights_fp8_pow2(int G, int N, int K, const void* w, void* w_q,
                                                   float* w_scale, moe_stream_t stream);

/* Backward pass of the layer for the routing the forward chose (the gradients
 * that training needs; "DeepSeek-V3 详解" 2.2-2.3 for the layer, and
 * "deepseek-v3-report", load-balancing paragraph: the selection bias only picks
 * the experts and gets no gradient, so the chosen set is an input).  With
 * a = x Wg^T, u = x Wu^T, h = silu(a) u, y = h Wd^T per expert and
 * out[t] = sum_shared y + sum_j g_j y_j, g_j = s_j / sum_i s_i, s = sigmoid(z):
 *   dx         bf16 [T, d]          out  d sum(out * dout) / dx
 *   dw_router  f32  [E, d]          out  ... / d w_router
 *   dw_gate_up bf16 [E+S, 2I, d]    out  ... / d w_gate_up (every expert, 0 if unused)
 *   dw_down    bf16 [E+S, d, I]     out  ... / d w_down
 * Inputs: x bf16 [T, d]; w_router bf16 [E, d]; logit_offset f32 [E] or NULL (as
 * moe_route); w_gate_up bf16 [E+S, 2I, d] and w_down bf16 [E+S, d, I] as the
 * forward takes them (no transposed copies: the input-gradient GEMMs read them
 * MN-major); topk_idx int32 [T, k] (moe_route's; distinct experts per token,
 * values in [0, E)); dout bf16 [T, d] (the gradient of the layer output).
 * The affinities of the chosen experts are recomputed in FP32; every GEMM
 * accumulates in FP32 on the tensor cores; a, u and dh are kept in FP32; h,
 * dy = g dout, [da du] and each row's dx contribution are rounded to bf16.  dtype must be MOE_BF16
 * (MOE_ERR_UNSUPPORTED otherwise).  Deterministic run to run.  `ws`
 * (moe_backward_workspace_bytes; 256-byte aligned, first 256 bytes zero before
 * first use) holds every intermediate; bad topk_idx sets MOE_ERR_DEVICE. */
MOE_API size_t moe_backward_workspace_bytes(const moe_shape_t* shape);
MOE_API moe_status_t moe_backward(const moe_shape_t* shape, const void* x, const void* w_router,
                                  const float* logit_offset, const void* w_gate_up, const void* w_down,
                                  const int32_t* topk_idx, const void* dout, void* dx, float* dw_router,
                                  void* dw_gate_up, void* dw_down, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* Expert parallelism ("DeepSeek-V3 Overview and Key Innovations", Training
 * Infrastructure and Optimization: experts spread over GPUs, all-to-all dispatch
 * and combine; "拆解DeepSeek V3": 8 GPUs per node over NVLink/NVSwitch).  The E
 * routed experts are split into G contiguous ranges of E_loc = E / G, one per
 * rank, so moe_permute's expert-major copy is already ordered by destination rank
 * and the dispatch is one all-to-all of row ranges (done by the caller, e.g. with
 * NCCL).  A rank then holds rows in source-major order: for each source rank s,
 * the rows s sent for each local expert e in turn (tokens ascending).  This call
 * moves rows between that order and the local expert-major order (expert e: the
 * rows of every source s in turn) that moe_expert_ffn takes, and back:
 *   recv_counts   int32 [G, E_loc]  rows source s sent for local expert e (device)
 *   rows          the total of recv_counts (rows of src and dst)
 *   src, dst      [rows, row_bytes] (row_bytes % 16 == 0; bf16 or E4M3 rows)
 *   src_scale, dst_scale  f32 [rows, scale_cols] moved with the rows (FP8 1x128
 *                 scales), or NULL with scale_cols = 0
 *   local_offsets int32 [E_loc + 1] out or NULL: expert-major group offsets
 *   to_local      1: source-major src -> expert-major dst (after the dispatch);
 *                 0: expert-major src -> source-major dst (before the combine)
 *   ws            a workspace as above (its status word only)
 * Counts that are negative or do not add up to `rows` set MOE_ERR_DEVICE, move
 * nothing and set local_offsets to zero.  Limits: G * E_loc <= 256. */
MOE_API moe_status_t moe_ep_regroup(int G, int E_loc, const int32_t* recv_counts, int rows, const void* src,
                                    void* dst, size_t row_bytes, const float* src_scale, float* dst_scale,
                                    int scale_cols, int32_t* local_offsets, int to_local, void* ws,
                                    moe_stream_t stream);

/* Reads (synchronising `stream`) and clears the device status word in `ws`:
 * MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE (or MOE_ERR_CUDA if the read
 * itself fails).  `ws` must be a workspace used by the calls above. */
MOE_API moe_status_t moe_get_device_status(void* ws, moe_stream_t stream);

/* Self-test of the bounded-wait path: launches one block that waits on a
 * barrier nothing will complete, with a limit of `limit_us` microseconds
 * (1..1000000), after which it records MOE_ERR_TIMEOUT in `ws` and exits.
 * Used to check failure detection without hanging the GPU. */
MOE_API moe_status_t moe_debug_wait_timeout(void* ws, unsigned limit_us, moe_stream_t stream);

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(moe_status_t status);

/* Library version, e.g. "libmoe 0.1 sm_103a". */
MOE_API const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
