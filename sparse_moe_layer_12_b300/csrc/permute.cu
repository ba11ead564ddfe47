// Dispatch on one GPU: group the (token, slot) pairs by expert, tokens
// ascending inside each expert, and copy each token row to its k places
// (the single-GPU form of the dispatch side of the expert all-to-all in
// "DeepSeek-V3 Overview and Key Innovations", Training Infrastructure and
// Optimization).  On the FP8 path the rows are quantised on the way, one
// scale per 1x128 tile ("DeepSeek-V3 详解" 4.2), scale = amax / 448.
//
// Two kernels:
//   rank    one block per expert scans topk_idx in token order and gives each
//           (t, j) routed to it its row offsets[e] + (#earlier tokens of e)
//           -- deterministic, no atomics;
//   scatter one block per token reads x[t] once (16-byte vectors) and writes
//           it to its k rows.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRankThreads = 512;
constexpr int kScatterThreads = 128;

__global__ void __launch_bounds__(kRankThreads)
    permute_rank_kernel(const int32_t* __restrict__ idx, const int32_t* __restrict__ offsets, int T, int k, int E,
                        int32_t* __restrict__ perm_token, int32_t* __restrict__ inv_pos, int* __restrict__ status) {
  __shared__ int warp_tot[kRankThreads / 32];
  __shared__ int warp_pre[kRankThreads / 32];
  __shared__ int block_tot;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lo = offsets[e], hi = offsets[e + 1];
  const bool bad_offsets = hi < lo || lo < 0 || hi > T * k || (e == E - 1 && hi != T * k) || (e == 0 && lo != 0);
  if (bad_offsets) {
    if (tid == 0) set_error(status, status + 1, MOE_ERR_DEVICE, kSitePermute);
    return;
  }
  int running = 0;
  for (int t0 = 0; t0 < T; t0 += kRankThreads) {
    const int t = t0 + tid;
    int slot = -1;
    if (t < T) {
      for (int j = 0; j < k; ++j) {
        const int v = idx[(size_t)t * k + j];
        if (v == e) slot = j;
        if (e == 0 && (v < 0 || v >= E)) set_error(status, status + 1, MOE_ERR_DEVICE, kSitePermute);
      }
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, slot >= 0);
    if (lane == 0) warp_tot[warp] = __popc(ballot);
    __syncthreads();
    if (warp == 0) {
      const int v = lane < kRankThreads / 32 ? warp_tot[lane] : 0;
      int inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += n;
      }
      if (lane < kRankThreads / 32) warp_pre[lane] = inc - v;
      if (lane == kRankThreads / 32 - 1) block_tot = inc;
    }
    __syncthreads();
    if (slot >= 0) {
      const int pos = lo + running + warp_pre[warp] + __popc(ballot & ((1u << lane) - 1u));
      if (pos < hi) {
        inv_pos[(size_t)t * k + slot] = pos;
        perm_token[pos] = t;
      } else {
        set_error(status, status + 1, MOE_ERR_DEVICE, kSitePermute);
      }
    }
    running += block_tot;
    __syncthreads();
  }
  if (tid == 0 && running != hi - lo) set_error(status, status + 1, MOE_ERR_DEVICE, kSitePermute);
}

template <bool FP8, bool POW2 = false>
__global__ void __launch_bounds__(kScatterThreads)
    permute_scatter_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ inv_pos, int T, int d, int k,
                           uint8_t* __restrict__ x_perm, float* __restrict__ x_perm_scale, int* __restrict__ status) {
  __shared__ int pos[kMaxK];
  const int t = blockIdx.x;
  const int rows = T * k;
  if (threadIdx.x < k) {
    int p = inv_pos[(size_t)t * k + threadIdx.x];
    if (p < 0 || p >= rows) {
      set_error(status, status + 1, MOE_ERR_DEVICE, kSitePermute);
      p = -1;
    }
    pos[threadIdx.x] = p;
  }
  __syncthreads();
  const int nvec = d / 8;  // 16-byte vectors of bf16
  const uint4* xr = x + (size_t)t * nvec;
  if (!FP8) {
    uint4* out = reinterpret_cast<uint4*>(x_perm);
    for (int v = threadIdx.x; v < nvec; v += kScatterThreads) {
      const uint4 val = __ldg(xr + v);
      for (int j = 0; j < k; ++j) {
        const int p = pos[j];
        if (p >= 0) out[(size_t)p * nvec + v] = val;
      }
    }
  } else {
    // 16 lanes cover one 1x128 tile (8 values each); nvec is a multiple of 16
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ntiles = d / 128;
    for (int v0 = warp * 32; v0 < nvec; v0 += kScatterThreads) {
      const int v = v0 + lane;
      const bool valid = v < nvec;
      float f[8];
      uint4 raw = make_uint4(0, 0, 0, 0);
      if (valid) raw = __ldg(xr + v);
      bf16x8_to_f32(raw, f);
      uint2 q;
      const float scale = quant_tile16<POW2>(f, q);
      if (valid) {
        const int tile = v >> 4;
        for (int j = 0; j < k; ++j) {
          const int p = pos[j];
          if (p < 0) continue;
          *reinterpret_cast<uint2*>(x_perm + (size_t)p * d + (size_t)v * 8) = q;
          if ((lane & 15) == 0) x_perm_scale[(size_t)p * ntiles + tile] = scale;
        }
      }
    }
  }
}

}  // namespace

moe_status_t launch_permute(const moe_shape_t& s, const void* x, const int32_t* idx, const int32_t* offsets,
                            void* x_perm, float* x_perm_scale, int32_t* perm_token, int32_t* inv_pos, void* ws,
                            cudaStream_t st) {
  if (s.T == 0) return MOE_OK;
  int* status = ws_status(ws);
  permute_rank_kernel<<<s.E, kRankThreads, 0, st>>>(idx, offsets, s.T, s.k, s.E, perm_token, inv_pos, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (x_perm == nullptr) return MOE_OK;  // tables only (the fused forward gathers rows in the GEMM)
  if (s.dtype == MOE_FP8_E4M3)
    permute_scatter_kernel<true><<<s.T, kScatterThreads, 0, st>>>(
        static_cast<const uint4*>(x), inv_pos, s.T, s.d, s.k, static_cast<uint8_t*>(x_perm), x_perm_scale, status);
  else if (s.dtype == MOE_FP8_E4M3_POW2)
    permute_scatter_kernel<true, true><<<s.T, kScatterThreads, 0, st>>>(
        static_cast<const uint4*>(x), inv_pos, s.T, s.d, s.k, static_cast<uint8_t*>(x_perm), x_perm_scale, status);
  else
    permute_scatter_kernel<false><<<s.T, kScatterThreads, 0, st>>>(
        static_cast<const uint4*>(x), inv_pos, s.T, s.d, s.k, static_cast<uint8_t*>(x_perm), nullptr, status);
  return cuda_status(cudaGetLastError());
}

}  // namespace moe
