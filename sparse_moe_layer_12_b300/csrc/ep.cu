// Expert parallelism: the regroup step between the all-to-all exchanges.
//
// "DeepSeek-V3 Overview and Key Innovations" (Training Infrastructure and
// Optimization) describes the experts spread over GPUs with custom all-to-all
// dispatch and combine kernels over NVLink and InfiniBand; "拆解DeepSeek V3"
// gives the node (8 GPUs, NVLink/NVSwitch inside).  Here the E routed experts
// are split into G contiguous ranges of E_loc = E / G, one per rank, so the
// expert-major permuted copy of a rank's tokens is already ordered by destination
// rank and the dispatch is one all-to-all of contiguous row ranges.  What a rank
// receives is source-major: for source s = 0..G-1, the rows it sent for local
// expert e = 0..E_loc-1 (tokens ascending).  The local expert GEMMs want the rows
// expert-major (all sources' rows of expert 0, then expert 1, ...), and the
// results must go back source-major for the return all-to-all.  This file moves
// rows between the two orders:
//
//   source-major segment (s, e) starts at  sum of counts[s', e'] over (s', e') < (s, e)
//   expert-major segment (s, e) starts at  local_off[e] + sum_{s' < s} counts[s', e],
//   local_off[e] = sum_{e' < e} sum_s counts[s, e']
//
// and keeps the order inside a segment.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRegroupThreads = 256;

// seg_src[j], seg_loc[j] for the nseg = G * E_loc segments (j = s * E_loc + e);
// seg_src[nseg] = total rows.  One block computes them in shared memory.
__device__ void regroup_tables(const int32_t* __restrict__ counts, int G, int E_loc, int* seg_src, int* seg_loc,
                               int* loc_off, int* bad) {
  const int nseg = G * E_loc;
  // serial scans: at most 256 segments, done by one warp-free thread (cheap next to the copy)
  if (threadIdx.x == 0) {
    int acc = 0, neg = 0;
    for (int j = 0; j < nseg; ++j) {
      const int c = counts[j];
      neg |= c < 0;
      seg_src[j] = acc;
      acc += c < 0 ? 0 : c;
    }
    seg_src[nseg] = acc;
    int lo = 0;
    for (int e = 0; e < E_loc; ++e) {
      loc_off[e] = lo;
      for (int s = 0; s < G; ++s) {
        const int c = counts[s * E_loc + e];
        seg_loc[s * E_loc + e] = lo;
        lo += c < 0 ? 0 : c;
      }
    }
    loc_off[E_loc] = lo;
    *bad = neg;
  }
  __syncthreads();
}

// Rows in source-major order j <-> expert-major order; to_local: dst[loc(j)] = src[j],
// else dst[j] = src[loc(j)].  row_vec 16-byte vectors per row; scale_n floats per row.
__global__ void __launch_bounds__(kRegroupThreads)
    ep_regroup_kernel(const int32_t* __restrict__ counts, int G, int E_loc, int rows, const uint4* __restrict__ src,
                      uint4* __restrict__ dst, int row_vec, const float* __restrict__ src_scale,
                      float* __restrict__ dst_scale, int scale_n, int32_t* __restrict__ local_offsets, int to_local,
                      int* __restrict__ status) {
  __shared__ int seg_src[kMaxE + 1], seg_loc[kMaxE], loc_off[kMaxE + 1];
  __shared__ int bad;
  regroup_tables(counts, G, E_loc, seg_src, seg_loc, loc_off, &bad);
  const int nseg = G * E_loc;
  if (bad || seg_src[nseg] != rows) {
    // inconsistent counts: no row moves; the offsets say "no rows", which the expert
    // GEMM's schedule rejects as well unless there are none
    if (blockIdx.x == 0) {
      if (threadIdx.x == 0) set_error(status, status + 1, MOE_ERR_DEVICE, kSiteEp);
      if (local_offsets)
        for (int e = threadIdx.x; e <= E_loc; e += blockDim.x) local_offsets[e] = 0;
    }
    return;
  }
  if (blockIdx.x == 0 && local_offsets)
    for (int e = threadIdx.x; e <= E_loc; e += blockDim.x) local_offsets[e] = loc_off[e];
  for (int j = blockIdx.x; j < rows; j += gridDim.x) {
    // the segment holding row j: the last one starting at or before j (empty ones share
    // their start with the next, so the last is the non-empty one)
    int lo = 0, hi = nseg;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (seg_src[mid] <= j) lo = mid;
      else hi = mid;
    }
    const int l = seg_loc[lo] + (j - seg_src[lo]);
    const int from = to_local ? j : l, to = to_local ? l : j;
    const uint4* s = src + (size_t)from * row_vec;
    uint4* d = dst + (size_t)to * row_vec;
    for (int v = threadIdx.x; v < row_vec; v += blockDim.x) d[v] = s[v];
    if (scale_n > 0)
      for (int v = threadIdx.x; v < scale_n; v += blockDim.x)
        dst_scale[(size_t)to * scale_n + v] = src_scale[(size_t)from * scale_n + v];
  }
}

}  // namespace

moe_status_t launch_ep_regroup(int G, int E_loc, const int32_t* counts, int rows, const void* src, void* dst,
                               size_t row_bytes, const float* src_scale, float* dst_scale, int scale_n,
                               int32_t* local_offsets, int to_local, void* ws, cudaStream_t st) {
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  const int grid = rows > 0 ? (rows < 8 * sms ? rows : 8 * sms) : 1;
  ep_regroup_kernel<<<grid, kRegroupThreads, 0, st>>>(counts, G, E_loc, rows, static_cast<const uint4*>(src),
                                                      static_cast<uint4*>(dst), static_cast<int>(row_bytes / 16),
                                                      src_scale, dst_scale, scale_n, local_offsets, to_local,
                                                      ws_status(ws));
  return cuda_status(cudaGetLastError());
}

}  // namespace moe
