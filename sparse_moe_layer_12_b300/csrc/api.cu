// libmoe C ABI: argument validation, workspace layout, TMA descriptors and the
// entry points declared in include/moe.h.  Every entry validates before it
// enqueues anything; compute happens only in the kernels of the other files.
#include <cuda.h>
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool shape_valid(const moe_shape_t* s) {
  if (!s) return false;
  if (s->T < 0 || s->d < 128 || s->I < 128 || s->E < 1 || s->S < 0 || s->k < 1) return false;
  if (s->d % 128 || s->I % 128 || s->d > 65536 || s->I > 65536) return false;
  if (s->k > s->E) return false;
  if (s->dtype != MOE_BF16 && !is_fp8(s->dtype)) return false;
  if (s->n_group == 0) return s->topk_group == 0;
  if (s->n_group < 1 || s->n_group > 32 || s->E % s->n_group) return false;
  if (s->topk_group < 1 || s->topk_group > s->n_group) return false;
  const int gsz = s->E / s->n_group;
  if (s->k > s->topk_group * gsz || (s->k + s->topk_group - 1) / s->topk_group > gsz) return false;
  return true;
}

static bool shape_supported(const moe_shape_t& s) {
  if (s.E > kMaxE || s.S > kMaxS || s.k > kMaxK) return false;
  const long long rows = (long long)s.T * s.k + (long long)s.S * s.T;
  const long long w = s.d > s.I ? s.d : s.I;
  if (rows * w >= (1ll << 31)) return false;
  return true;
}

// Which form of the dispatch moe_forward uses.  Reading the routed rows straight
// from x inside the gate/up GEMM (TMA row gathers, 512 bytes per operation) saves
// the permuted copy but keeps far fewer bytes in flight per SM than 32-row box
// loads of a contiguous copy; measured on B300 it wins only while the batch is
// small (T*k = 512: 0.030 ms against 0.053 ms; T*k = 2048: even; T*k = 24576:
// 0.67 ms against 0.52 ms; T*k = 65536: 8.6 ms against 6.1 ms).
bool forward_gathers(const moe_shape_t& s) {
  // the block-scaled FP8 GEMM reads whole-tile boxes only
  return s.dtype != MOE_FP8_E4M3_POW2 && (size_t)s.T * s.k <= kForwardGatherMaxRows;
}

WsLayout ws_layout(const moe_shape_t& s) {
  WsLayout L{};
  const size_t A = 1024;
  const size_t Tk = (size_t)s.T * s.k;
  const size_t rows = Tk + (size_t)s.S * s.T;
  const bool f8 = is_fp8(s.dtype);
  const size_t es = f8 ? 1 : 2;
  size_t o = 0;
  L.status = o;      o = align_up(o + kWsCtrlBytes, A);
  L.counts = o;      o = align_up(o + 4 * (size_t)s.E, A);
  L.offsets = o;     o = align_up(o + 4 * ((size_t)s.E + 1), A);
  L.idx = o;         o = align_up(o + 4 * Tk, A);
  L.gate = o;        o = align_up(o + 4 * Tk, A);
  L.perm_token = o;  o = align_up(o + 4 * Tk, A);
  L.inv_pos = o;     o = align_up(o + 4 * Tk, A);
  L.sched = o;       o = align_up(o + Schedule::bytes(s.E + s.S), A);
  const size_t xp_rows = forward_gathers(s) ? 0 : Tk;  // moe_forward's permuted copy of x
  L.x_perm = o;      o = align_up(o + xp_rows * s.d * es, A);
  L.x_perm_scale = o; o = align_up(o + (f8 ? xp_rows * (s.d / 128) * 4 : 0), A);
  L.xq = o;          o = align_up(o + (f8 ? (size_t)s.T * s.d : 0), A);
  L.xq_scale = o;    o = align_up(o + (f8 ? (size_t)s.T * (s.d / 128) * 4 : 0), A);
  L.h = o;           o = align_up(o + rows * s.I * es, A);
  L.h_scale = o;     o = align_up(o + (f8 ? rows * (s.I / 128) * 4 : 0), A);
  L.y = o;           o = align_up(o + rows * s.d * 2, A);
  const bool p2 = s.dtype == MOE_FP8_E4M3_POW2;
  L.sb_xp = o;       o = align_up(o + (p2 ? Tk * (s.d / 128) : 0), A);
  L.sb_xq = o;       o = align_up(o + (p2 ? (size_t)s.T * (s.d / 128) : 0), A);
  L.sb_h = o;        o = align_up(o + (p2 ? rows * (s.I / 128) : 0), A);
  L.total = o;
  return L;
}

WsLayout ffn_ws_layout(const moe_shape_t& s) {
  WsLayout L{};
  const size_t A = 1024;
  const size_t rows = (size_t)s.T * s.k + (size_t)s.S * s.T;
  const bool f8 = is_fp8(s.dtype);
  size_t o = 0;
  L.status = o;      o = align_up(o + 256, A);
  L.sched = o;       o = align_up(o + Schedule::bytes(s.E + s.S), A);
  L.xq = o;          o = align_up(o + (f8 ? (size_t)s.T * s.d : 0), A);
  L.xq_scale = o;    o = align_up(o + (f8 ? (size_t)s.T * (s.d / 128) * 4 : 0), A);
  L.h = o;           o = align_up(o + rows * s.I * (f8 ? 1 : 2), A);
  L.h_scale = o;     o = align_up(o + (f8 ? rows * (s.I / 128) * 4 : 0), A);
  const bool p2 = s.dtype == MOE_FP8_E4M3_POW2;
  L.sb_xp = o;       o = align_up(o + (p2 ? (size_t)s.T * s.k * (s.d / 128) : 0), A);
  L.sb_xq = o;       o = align_up(o + (p2 ? (size_t)s.T * (s.d / 128) : 0), A);
  L.sb_h = o;        o = align_up(o + (p2 ? rows * (s.I / 128) : 0), A);
  L.total = o;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// a buffer with one entry per token (or per routed row) may be NULL when there are no tokens
static inline bool tok(const void* p, const moe_shape_t& s) { return p != nullptr || s.T == 0; }

moe_status_t check_ws(const moe_shape_t& s, void* ws, size_t ws_bytes) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < ws_layout(s).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int max_active_clusters(const void* kernel, int cluster, int threads, size_t smem) {
  // the occupancy query costs host time on every call; cache it per device and launch shape
  struct Entry {
    int dev, cluster, threads, value;
    const void* kernel;
    size_t smem;
  };
  static Entry cache[64];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].dev == dev && cache[i].kernel == kernel && cache[i].cluster == cluster &&
          cache[i].threads == threads && cache[i].smem == smem)
        return cache[i].value;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = static_cast<unsigned>(cluster);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();  // clear the failed query
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (used < 64) cache[used++] = Entry{dev, cluster, threads, clusters, kernel, smem};
  return clusters;
}

int pair_grid(const void* kernel, int threads, size_t smem) {
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const int clusters = max_active_clusters(kernel, 2, threads, smem);
  return clusters > 0 ? 2 * clusters : sms & ~1;
}

// ---------------------------------------------------------------- TMA descriptors

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The tensor-map encoder is a driver entry point that needs the calling thread's
// context to be current, which the runtime only makes so on its first call in that
// thread: a host thread whose first library call builds a tensor map gets the
// current device's primary context here, once.
static bool thread_context_ready() {
  thread_local bool ready = false;
  if (!ready) ready = cudaFree(nullptr) == cudaSuccess;
  return ready;
}

static EncodeTiledFn encode_fn() {
  if (!thread_context_ready()) return nullptr;
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_map_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
                 uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn f = encode_fn();
  if (!f || !aligned16(base)) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (uint64_t)esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return f(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d_sw64(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
                      uint64_t mid, uint64_t outer, uint32_t box_inner, uint32_t box_mid) {
  EncodeTiledFn f = encode_fn();
  if (!f || !aligned16(base)) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * (uint64_t)esize, inner * mid * (uint64_t)esize};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return f(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
                 uint64_t mid, uint64_t outer, uint32_t box_inner, uint32_t box_mid) {
  EncodeTiledFn f = encode_fn();
  if (!f || !aligned16(base)) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {inner * (uint64_t)esize, inner * mid * (uint64_t)esize};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return f(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weight view that fetches the two 128-row A blocks of an expert-GEMM tile in one load:
// dims {K, rows, 2, groups} with the "2" dimension `gap` rows apart (gate/up: the up rows
// are I rows after the gate rows; group g = one expert, g_stride rows apart), box
// {box_k, 128, 2, 1}, 128-byte swizzle.  The two blocks land one after the other.
bool make_map_pair_rows(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t K,
                        uint64_t rows, uint64_t gap, uint64_t groups, uint64_t g_stride, uint32_t box_k) {
  EncodeTiledFn f = encode_fn();
  if (!f || !aligned16(base)) return false;
  cuuint64_t dims[4] = {K, rows, 2, groups};
  cuuint64_t strides[3] = {K * (uint64_t)esize, gap * K * (uint64_t)esize, g_stride * K * (uint64_t)esize};
  cuuint32_t box[4] = {box_k, 128, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return f(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// As make_map_pair_rows with a further dimension: {K, rows, 2, blocks, groups}, the "2"
// dimension `gap` rows apart, `blocks` of `b_stride` rows (W_down: channel blocks 0 and 1 of
// a 512-channel tile, 256 rows apart, tiles 512 rows apart).
bool make_map_pair_rows5(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t K,
                         uint64_t rows, uint64_t gap, uint64_t blocks, uint64_t b_stride, uint64_t groups,
                         uint64_t g_stride, uint32_t box_k) {
  EncodeTiledFn f = encode_fn();
  if (!f || !aligned16(base)) return false;
  const uint64_t rb = K * (uint64_t)esize;
  cuuint64_t dims[5] = {K, rows, 2, blocks, groups};
  cuuint64_t strides[4] = {rb, gap * rb, b_stride * rb, g_stride * rb};
  cuuint32_t box[5] = {box_k, 128, 2, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return f(m, dt, 5, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- debug wait kernel

__global__ void debug_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);  // nothing ever arrives on this barrier
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_wait(&bar, 0, &abort_flag, status, status + 1, kSiteDebug, limit_ns);
  }
  __syncthreads();
}

moe_status_t launch_debug_wait(void* ws, unsigned limit_us, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(ws_status(ws), (unsigned long long)limit_us * 1000ull);
  return cuda_status(cudaGetLastError());
}

}  // namespace moe

using namespace moe;

namespace {
// NVTX range around each entry point (no cost unless a profiler is attached)
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
}  // namespace

#define MOE_TRY(expr)                     \
  do {                                    \
    moe_status_t _st = (expr);            \
    if (_st != MOE_OK) return _st;        \
  } while (0)

extern "C" {

size_t moe_workspace_bytes(const moe_shape_t* shape) {
  if (!shape_valid(shape)) return 0;
  return ws_layout(*shape).total;
}

static moe_status_t validate_shape(const moe_shape_t* shape) {
  if (!shape_valid(shape)) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(*shape)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t moe_route(const moe_shape_t* shape, const void* x, const void* w_router, const float* bias,
                       const float* logit_offset, int32_t* topk_idx, float* topk_gate, int32_t* counts,
                       int32_t* offsets, void* ws, size_t ws_bytes, moe_stream_t stream) {
  NvtxRange nvtx_range("moe_route");
  MOE_TRY(validate_shape(shape));
  const moe_shape_t& s = *shape;
  if (!tok(x, s) || !w_router || !bias || !tok(topk_idx, s) || !tok(topk_gate, s) || !counts || !offsets)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_ALIGNMENT;
  MOE_TRY(check_ws(s, ws, ws_bytes));
  return launch_route(s, x, w_router, bias, logit_offset, topk_idx, topk_gate, counts, offsets, ws,
                      (cudaStream_t)stream);
}

moe_status_t moe_permute(const moe_shape_t* shape, const void* x, const int32_t* topk_idx,
                         const int32_t* offsets, void* x_perm, float* x_perm_scale, int32_t* perm_token,
                         int32_t* inv_pos, void* ws, size_t ws_bytes, moe_stream_t stream) {
  NvtxRange nvtx_range("moe_permute");
  MOE_TRY(validate_shape(shape));
  const moe_shape_t& s = *shape;
  if (!tok(x, s) || !tok(topk_idx, s) || !offsets || !tok(perm_token, s) || !tok(inv_pos, s))
    return MOE_ERR_INVALID_ARG;
  if (!x_perm && x_perm_scale) return MOE_ERR_INVALID_ARG;  // tables only: no rows, no scales
  if (x_perm && is_fp8(s.dtype) && !x_perm_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_ALIGNMENT;
  MOE_TRY(check_ws(s, ws, ws_bytes));
  return launch_permute(s, x, topk_idx, offsets, x_perm, x_perm_scale, perm_token, inv_pos, ws,
                        (cudaStream_t)stream);
}

moe_status_t moe_expert_ffn(const moe_shape_t* shape, const void* x_perm, const float* x_perm_scale,
                            const void* x, const int32_t* offsets, const void* w_gate_up,
                            const float* w_gu_scale, const void* w_down, const float* w_down_scale, void* y,
                            void* ws, size_t ws_bytes, moe_stream_t stream) {
  NvtxRange nvtx_range("moe_expert_ffn");
  MOE_TRY(validate_shape(shape));
  const moe_shape_t& s = *shape;
  if (!tok(x_perm, s) || !tok(x, s) || !offsets || !w_gate_up || !w_down || !tok(y, s)) return MOE_ERR_INVALID_ARG;
  if (is_fp8(s.dtype) && (!tok(x_perm_scale, s) || !w_gu_scale || !w_down_scale)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(x) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(y))
    return MOE_ERR_ALIGNMENT;
  MOE_TRY(check_ws(s, ws, ws_bytes));
  return launch_expert_ffn(s, x_perm, x_perm_scale, x, nullptr, offsets, w_gate_up, w_gu_scale, w_down, w_down_scale,
                           y, ws, (cudaStream_t)stream);
}

moe_status_t moe_expert_ffn_gather(const moe_shape_t* shape, const void* x, const int32_t* perm_token,
                                   const int32_t* offsets, const void* w_gate_up, const float* w_gu_scale,
                                   const void* w_down, const float* w_down_scale, void* y, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  NvtxRange nvtx_range("moe_expert_ffn_gather");
  MOE_TRY(validate_shape(shape));
  const moe_shape_t& s = *shape;
  if (!tok(x, s) || !tok(perm_token, s) || !offsets || !w_gate_up || !w_down || !tok(y, s)) return MOE_ERR_INVALID_ARG;
  if (s.dtype == MOE_FP8_E4M3_POW2) return MOE_ERR_UNSUPPORTED;  // block-scaled GEMM: permuted copy only
  if (is_fp8(s.dtype) && (!w_gu_scale || !w_down_scale)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(y)) return MOE_ERR_ALIGNMENT;
  MOE_TRY(check_ws(s, ws, ws_bytes));
  return launch_expert_ffn(s, nullptr, nullptr, x, perm_token, offsets, w_gate_up, w_gu_scale, w_down,
                           w_down_scale, y, ws, (cudaStream_t)stream);
}

moe_status_t moe_combine(const moe_shape_t* shape, const void* y, const float* topk_gate,
                         const int32_t* inv_pos, void* out, moe_stream_t stream) {
  NvtxRange nvtx_range("moe_combine");
  MOE_TRY(validate_shape(shape));
  const moe_shape_t& s = *shape;
  if (!tok(y, s) || !tok(topk_gate, s) || !tok(inv_pos, s) || !tok(out, s)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out)) return MOE_ERR_ALIGNMENT;
  return launch_combine(s, y, topk_gate, inv_pos, out, (cudaStream_t)stream);
}

moe_status_t moe_bias_update(const moe_shape_t* shape, const int32_t* counts, float* bias, float gamma,
                             moe_stream_t stream) {
  NvtxRange nvtx_range("moe_bias_update");
  MOE_TRY(validate_shape(shape));
  if (!counts || !bias) return MOE_ERR_INVALID_ARG;
  if (!(gamma >= 0.0f) || gamma > 1.0f) return MOE_ERR_INVALID_ARG;
  return launch_bias_update(*shape, counts, bias, gamma, (cudaStream_t)stream);
}

moe_status_t moe_forward(const moe_shape_t* shape, const void* x, const void* w_router, float* bias,
                         const float* logit_offset, const void* w_gate_up, const float* w_gu_scale,
                         const void* w_down, const float* w_down_scale, void* out, int32_t* topk_idx,
                         float* topk_gate, int32_t* counts, float gamma, int update_bias, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  NvtxRange nvtx_range("moe_forward");
  MOE_TRY(validate_shape(shape));
  const moe_shape_t& s = *shape;
  if (!tok(x, s) || !w_router || !bias || !w_gate_up || !w_down || !tok(out, s)) return MOE_ERR_INVALID_ARG;
  if (is_fp8(s.dtype) && (!w_gu_scale || !w_down_scale)) return MOE_ERR_INVALID_ARG;
  if (update_bias && (!(gamma >= 0.0f) || gamma > 1.0f)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(out))
    return MOE_ERR_ALIGNMENT;
  MOE_TRY(check_ws(s, ws, ws_bytes));
  const WsLayout L = ws_layout(s);
  char* w = static_cast<char*>(ws);
  int32_t* idx = topk_idx ? topk_idx : reinterpret_cast<int32_t*>(w + L.idx);
  float* gate = topk_gate ? topk_gate : reinterpret_cast<float*>(w + L.gate);
  int32_t* cnt = counts ? counts : reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* off = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* ptok = reinterpret_cast<int32_t*>(w + L.perm_token);
  int32_t* inv = reinterpret_cast<int32_t*>(w + L.inv_pos);
  void* y = w + L.y;
  cudaStream_t st = (cudaStream_t)stream;
  MOE_TRY(launch_route(s, x, w_router, bias, logit_offset, idx, gate, cnt, off, ws, st));
  if (forward_gathers(s)) {
    // dispatch fused into the gate/up GEMM: only the permutation tables are built,
    // the GEMM gathers each routed row from x through perm_token
    MOE_TRY(launch_permute(s, x, idx, off, nullptr, nullptr, ptok, inv, ws, st));
    MOE_TRY(launch_expert_ffn(s, nullptr, nullptr, x, ptok, off, w_gate_up, w_gu_scale, w_down, w_down_scale, y,
                              ws, st));
  } else {
    void* xp = w + L.x_perm;
    float* xps = is_fp8(s.dtype) ? reinterpret_cast<float*>(w + L.x_perm_scale) : nullptr;
    MOE_TRY(launch_permute(s, x, idx, off, xp, xps, ptok, inv, ws, st));
    MOE_TRY(launch_expert_ffn(s, xp, xps, x, nullptr, off, w_gate_up, w_gu_scale, w_down, w_down_scale, y, ws,
                              st));
  }
  MOE_TRY(launch_combine(s, y, gate, inv, out, st));
  if (update_bias) MOE_TRY(launch_bias_update(s, cnt, bias, gamma, st));
  return MOE_OK;
}

int moe_forward_gathers(const moe_shape_t* shape) {
  if (!shape || !shape_valid(shape)) return -1;
  return forward_gathers(*shape) ? 1 : 0;
}

moe_status_t moe_quantize_weights_fp8(int G, int N, int K, const void* w, void* w_q, float* w_scale,
                                      moe_stream_t stream) {
  NvtxRange nvtx_range("moe_quantize_weights_fp8");
  if (G < 0 || N < 0 || K < 0 || N % 128 || K % 128) return MOE_ERR_INVALID_ARG;
  if ((long long)G * N * K >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  if (G == 0 || N == 0 || K == 0) return MOE_OK;
  if (!w || !w_q || !w_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(w_q)) return MOE_ERR_ALIGNMENT;
  return launch_quant_weights(G, N, K, w, w_q, w_scale, false, (cudaStream_t)stream);
}

moe_status_t moe_quantize_weights_fp8_pow2(int G, int N, int K, const void* w, void* w_q, float* w_scale,
                                           moe_stream_t stream) {
  NvtxRange nvtx_range("moe_quantize_weights_fp8_pow2");
  if (G < 0 || N < 0 || K < 0 || N % 128 || K % 128) return MOE_ERR_INVALID_ARG;
  if ((long long)G * N * K >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  if (G == 0 || N == 0 || K == 0) return MOE_OK;
  if (!w || !w_q || !w_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(w_q)) return MOE_ERR_ALIGNMENT;
  return launch_quant_weights(G, N, K, w, w_q, w_scale, true, (cudaStream_t)stream);
}

size_t moe_backward_workspace_bytes(const moe_shape_t* shape) {
  if (!shape_valid(shape)) return 0;
  return bwd_layout(*shape).total;
}

// limits of the backward pass on top of the forward's
static moe_status_t backward_supported(const moe_shape_t& s) {
  if (s.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const long long rows = (long long)s.T * s.k + (long long)s.S * s.T;
  if (rows * 2 * s.I >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (bwd_kcap(s) >= (size_t)(1u << 31)) return MOE_ERR_UNSUPPORTED;  // row indices stay int
  if ((long long)(s.E + s.S) * 2 * s.I >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t moe_backward(const moe_shape_t* shape, const void* x, const void* w_router, const float* logit_offset,
                          const void* w_gate_up, const void* w_down, const int32_t* topk_idx, const void* dout,
                          void* dx, float* dw_router, void* dw_gate_up, void* dw_down, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  NvtxRange nvtx_range("moe_backward");
  MOE_TRY(validate_shape(shape));
  const moe_shape_t& s = *shape;
  MOE_TRY(backward_supported(s));
  if (!tok(x, s) || !w_router || !w_gate_up || !w_down || !tok(topk_idx, s) || !tok(dout, s) || !tok(dx, s) ||
      !dw_router || !dw_gate_up || !dw_down)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(dout) ||
      !aligned16(dx) || !aligned16(dw_router) || !aligned16(dw_gate_up) || !aligned16(dw_down))
    return MOE_ERR_ALIGNMENT;
  if (!ws) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < bwd_layout(s).total) return MOE_ERR_WORKSPACE;
  return launch_backward(s, x, w_router, logit_offset, w_gate_up, w_down, topk_idx, dout, dx, dw_router, dw_gate_up,
                         dw_down, ws, (cudaStream_t)stream);
}

moe_status_t moe_ep_regroup(int G, int E_loc, const int32_t* recv_counts, int rows, const void* src, void* dst,
                            size_t row_bytes, const float* src_scale, float* dst_scale, int scale_cols,
                            int32_t* local_offsets, int to_local, void* ws, moe_stream_t stream) {
  NvtxRange nvtx_range("moe_ep_regroup");
  if (G < 1 || E_loc < 1 || (long long)G * E_loc > kMaxE || rows < 0 || scale_cols < 0) return MOE_ERR_INVALID_ARG;
  if (row_bytes == 0 || row_bytes % 16 || row_bytes > (1u << 20)) return MOE_ERR_INVALID_ARG;
  if (!recv_counts || ((!src || !dst) && rows > 0)) return MOE_ERR_INVALID_ARG;
  if (scale_cols > 0 && rows > 0 && (!src_scale || !dst_scale)) return MOE_ERR_INVALID_ARG;
  if ((long long)rows * (long long)(row_bytes / 16) >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(src) || !aligned16(dst)) return MOE_ERR_ALIGNMENT;
  if (!ws) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_ALIGNMENT;
  return launch_ep_regroup(G, E_loc, recv_counts, rows, src, dst, row_bytes, src_scale, dst_scale, scale_cols,
                           local_offsets, to_local ? 1 : 0, ws, (cudaStream_t)stream);
}

moe_status_t moe_get_device_status(void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  int h[2] = {0, 0};
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (h[0] != 0) {
    if (cudaMemsetAsync(ws, 0, sizeof(h), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  switch (h[0]) {
    case 0: return MOE_OK;
    case MOE_ERR_TIMEOUT: return MOE_ERR_TIMEOUT;
    default: return MOE_ERR_DEVICE;
  }
}

moe_status_t moe_debug_wait_timeout(void* ws, unsigned limit_us, moe_stream_t stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  return launch_debug_wait(ws, limit_us, (cudaStream_t)stream);
}

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_version(void) { return "libmoe 0.1 sm_103a"; }

}  // extern "C"
