// Internal declarations shared by the libmoe translation units: limits,
// workspace layout, the expert-GEMM schedule format and host helpers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // bounded waits: 2 s
constexpr int kMaxE = 256;
constexpr int kMaxS = 8;
constexpr int kMaxK = 16;
constexpr int kRouterTileM = 128;  // tokens per router tile
constexpr int kChunkMax = 256;     // tokens per expert-GEMM tile (tcgen05 N)
// tokens per tile of the block-scaled FP8 GEMM: each of its two epilogue groups holds its
// (at most three) 32-token chunks in registers between reading and releasing TMEM
constexpr int kChunkMxMax = 192;
constexpr int kBoxRows = 32;       // token rows per TMA box in the expert GEMM
constexpr size_t kForwardGatherMaxRows = 4096;  // moe_forward gathers routed rows while T*k <= this

// Failure-site ids recorded next to the status word (diagnostics only).
enum Site : int {
  kSiteRouterProducer = 1,
  kSiteRouterMma = 2,
  kSiteRouterEpi = 3,
  kSiteGemmProducer = 11,
  kSiteGemmMma = 12,
  kSiteGemmEpi = 13,
  kSiteGemmTeardown = 14,
  kSitePermute = 21,
  kSiteSchedule = 22,
  kSiteBackward = 31,
  kSiteEp = 41,
  kSiteDebug = 90,
};

// Per-group record of the expert-GEMM schedule (routed experts 0..E-1, then
// shared experts).  Written on the device by the schedule kernel.
struct GroupInfo {
  int n;         // tokens in the group
  int in_row0;   // first row of the group in the gate/up B source (x_perm or x)
  int out_row0;  // first row of the group in h / y
  int csize;     // tokens per chunk (multiple of 16, <= kChunkMax)
  int nchunks;   // chunks
  int expert;    // weight index (0..E+S-1)
  int pad0, pad1;
};

struct Schedule {
  // layout inside the workspace: GroupInfo[G], int tile_start_gu[G+1], int tile_start_dn[G+1]
  static size_t bytes(int G) { return sizeof(GroupInfo) * G + sizeof(int) * 2 * (G + 1); }
};

struct WsLayout {
  size_t status, counts, offsets, idx, gate, perm_token, inv_pos, sched;
  size_t x_perm, x_perm_scale, xq, xq_scale, h, h_scale, y;
  // power-of-two FP8 only: UE8M0 bytes of the token scales, K-block major ([K/128][rows])
  // for the routed rows of x_perm, the shared experts' rows of x and the rows of h
  size_t sb_xp, sb_xq, sb_h;
  size_t total;
};

// Workspace of moe_backward (byte offsets; all 1024-aligned).  R = T*k routed rows;
// kcap = rows of the row buffers (every expert's rows, routed and shared, padded to
// a multiple of 64).
struct BwdLayout {
  size_t status, counts, offsets, perm_token, inv_pos, s, gate, pinv, dz, dgate_prow, dz_prow;
  size_t sched, wsched_a, wsched_b, kb_start;
  size_t xp, dyp, au, h, dh, dgu, dx_rows;
  size_t total;
};
size_t bwd_kcap(const moe_shape_t& s);
BwdLayout bwd_layout(const moe_shape_t& s);

bool shape_valid(const moe_shape_t* s);
// E4M3 activations and weights with 1x128 / 128x128 scales (FP32 scales, or powers of two)
inline bool is_fp8(moe_dtype_t t) { return t == MOE_FP8_E4M3 || t == MOE_FP8_E4M3_POW2; }
bool forward_gathers(const moe_shape_t& s);  // moe_forward's dispatch form (see moe_forward_gathers)
WsLayout ws_layout(const moe_shape_t& s);
// The expert FFN's scratch alone (status word, schedule, FP8 copy of x and its scales,
// h and its scales), packed; the other fields are 0 and unused.  `total` is its size.
WsLayout ffn_ws_layout(const moe_shape_t& s);

// The workspace's control block (its first kWsCtrlBytes, zero before first use): the
// device status word at offset 0, and at offset 256 the router's load counters
// (kMaxE counts and a ticket), which every router launch leaves cleared.
constexpr size_t kWsCtrlBytes = 2048;
inline int* ws_status(void* ws) { return reinterpret_cast<int*>(ws); }
inline int* ws_load_acc(void* ws) { return reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws) + 256); }
static_assert(256 + 4 * (kMaxE + 1) <= kWsCtrlBytes, "router load counters do not fit the control block");

// host helpers
moe_status_t check_ws(const moe_shape_t& s, void* ws, size_t ws_bytes);
bool aligned16(const void* p);
int sm_count();
// clusters of `cluster` CTAs of `kernel` that fit on the GPU at once (0 if the query fails); cached
int max_active_clusters(const void* kernel, int cluster, int threads, size_t smem);
// grid (in CTAs) of a persistent kernel launched in clusters of 2: 2 x the clusters that fit at once
int pair_grid(const void* kernel, int threads, size_t smem);
moe_status_t cuda_status(cudaError_t e);

// TMA descriptors (128-byte swizzle, zero fill out of bounds)
bool make_map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
                 uint64_t outer, uint32_t box_inner, uint32_t box_outer);
// 3-D map with 64-byte swizzle (box rows of 64 bytes; TMA stores of staged tiles)
bool make_map_3d_sw64(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
                      uint64_t mid, uint64_t outer, uint32_t box_inner, uint32_t box_mid);
bool make_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
                 uint64_t mid, uint64_t outer, uint32_t box_inner, uint32_t box_mid);
// the two 128-row A blocks of a tile in one load (see api.cu): 4-D {K, rows, 2, groups} and
// 5-D {K, rows, 2, blocks, groups}
bool make_map_pair_rows(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t K,
                        uint64_t rows, uint64_t gap, uint64_t groups, uint64_t g_stride, uint32_t box_k);
bool make_map_pair_rows5(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t K,
                         uint64_t rows, uint64_t gap, uint64_t blocks, uint64_t b_stride, uint64_t groups,
                         uint64_t g_stride, uint32_t box_k);

// launchers (each returns MOE_OK or MOE_ERR_CUDA); pointers already validated
moe_status_t launch_route(const moe_shape_t& s, const void* x, const void* w_router, const float* bias,
                          const float* logit_offset, int32_t* idx, float* gate, int32_t* counts,
                          int32_t* offsets, void* ws, cudaStream_t st);
// x_perm == nullptr: only the permutation tables (perm_token, inv_pos), no row copies
moe_status_t launch_permute(const moe_shape_t& s, const void* x, const int32_t* idx, const int32_t* offsets,
                            void* x_perm, float* x_perm_scale, int32_t* perm_token, int32_t* inv_pos, void* ws,
                            cudaStream_t st);
// perm_token == nullptr: routed rows from x_perm (+ x_perm_scale); otherwise the
// gate/up GEMM gathers them from x through perm_token and x_perm is unused
// `layout` places the FFN's scratch inside `ws` (nullptr: ws_layout(s), the layout of
// every call that takes a workspace)
moe_status_t launch_expert_ffn(const moe_shape_t& s, const void* x_perm, const float* x_perm_scale,
                               const void* x, const int32_t* perm_token, const int32_t* offsets,
                               const void* w_gate_up, const float* w_gu_scale, const void* w_down,
                               const float* w_down_scale, void* y, void* ws, cudaStream_t st,
                               const WsLayout* layout = nullptr);
moe_status_t launch_expert_ffn_fp8(const moe_shape_t& s, const void* x_perm, const float* x_perm_scale,
                                   const void* x, const int32_t* perm_token, const int32_t* offsets,
                                   const void* w_gate_up, const float* w_gu_scale, const void* w_down,
                                   const float* w_down_scale, void* y, void* ws, cudaStream_t st,
                                   const WsLayout* layout = nullptr);
// block-scaled E4M3 expert FFN (power-of-two scales; csrc/expert_gemm_mx.cu); routed rows from x_perm
moe_status_t launch_expert_ffn_mx(const moe_shape_t& s, const void* x_perm, const float* x_perm_scale, const void* x,
                                  const int32_t* offsets, const void* w_gate_up, const float* w_gu_scale,
                                  const void* w_down, const float* w_down_scale, void* y, void* ws, cudaStream_t st,
                                  const WsLayout* layout = nullptr);
// per-group token counts, chunking (<= chunk_max tokens) and tile prefix sums (one block of 512 threads)
__global__ void schedule_kernel(const int32_t* __restrict__ offsets, int T, int k, int E, int S, int m_gu, int m_dn,
                                int chunk_max, GroupInfo* __restrict__ groups, int* __restrict__ ts_gu,
                                int* __restrict__ ts_dn, int* __restrict__ status);
// Backward-pass launches of the grouped expert GEMM (one persistent launch each);
// every map has 128-byte swizzle:
//   kGateUpRaw  out = FP32 [a | u] rows (width 2I), out2 = bf16 h rows (width I); A = map_w
//               [G][2I][K] (box 64 x 128), B rows map_b0 / map_b1 at in_row0 (box 64 x 32)
//   kDgrad      out = B W[g] (width `width`); map_w [G][K][width] (box 64 x 64, read
//               MN-major), B = map_b0 rows at in_row0 (box 64 x 32)
//   kWgrad      out[g] = A^T B over the group's rows [64 pad0, 64 (pad0 + pad1)):
//               map_w [1][rows][M] and map_b0 [rows][N] (boxes 64 x 64, MN-major);
//               out[g][M index][N index] (M: 512 per tile, `I` per group; N: chunks of
//               256), written by TMA stores through map_out ([G][I][N], 64-byte
//               swizzle, box 32 x 128)
//   kDgrad32    as kDgrad, out = FP32 rows
enum class GemmMode : int { kGateUpRaw, kDgrad, kWgrad, kDgrad32 };
moe_status_t launch_gemm_bwd(GemmMode mode, const CUtensorMap& map_w, const CUtensorMap& map_b0,
                             const CUtensorMap& map_b1, const GroupInfo* groups, const int* tile_start, int G, int E,
                             int K, int I, int width, void* out, void* out2, int* status, cudaStream_t st,
                             const CUtensorMap* map_out = nullptr);
moe_status_t launch_backward(const moe_shape_t& s, const void* x, const void* w_router, const float* logit_offset,
                             const void* w_gate_up, const void* w_down, const int32_t* topk_idx, const void* dout,
                             void* dx, float* dw_router, void* dw_gate_up, void* dw_down, void* ws, cudaStream_t st);
moe_status_t launch_combine(const moe_shape_t& s, const void* y, const float* gate, const int32_t* inv_pos,
                            void* out, cudaStream_t st);
moe_status_t launch_bias_update(const moe_shape_t& s, const int32_t* counts, float* bias, float gamma,
                                cudaStream_t st);
moe_status_t launch_quant_weights(int G, int N, int K, const void* w, void* w_q, float* w_scale, bool pow2,
                                  cudaStream_t st);
moe_status_t launch_debug_wait(void* ws, unsigned limit_us, cudaStream_t st);
// expert parallelism: rows between source-major and local expert-major order (csrc/ep.cu)
moe_status_t launch_ep_regroup(int G, int E_loc, const int32_t* counts, int rows, const void* src, void* dst,
                               size_t row_bytes, const float* src_scale, float* dst_scale, int scale_n,
                               int32_t* local_offsets, int to_local, void* ws, cudaStream_t st);

}  // namespace moe
