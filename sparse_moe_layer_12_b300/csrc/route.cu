// Router: z = x . w_router^T on the tcgen05 tensor cores, fused with the
// sigmoid affinity, the selection bias, the per-token top-k, the gate
// normalisation over the chosen set and the per-expert load histogram.
//
// Pages: "deepseek-v3-report" (dynmi.github.io), load-balancing paragraph (b_i
// added to the routing score for selection, out of the gradient);
// "DeepSeek-V3 详解" (yudonglee.me) 2.2-2.3 (top-8 of 256, bias); readings for
// the silent points (sigmoid, gate normalisation, tie-break) in include/moe.h.
//
// One CTA owns 128 tokens (the M side of the MMA, one token per TMEM lane) and
// all E <= 256 experts (the N side, padded to 16).  Warp roles: warp 0 issues
// TMA loads of x and w_router in 64-wide K blocks through a 4-stage ring, warp 1
// issues tcgen05.mma into a TMEM accumulator, warps 2-5 (one per TMEM lane
// quadrant) turn the logits into affinities in shared memory; then every warp
// takes whole tokens and selects their top-k cooperatively (8 experts a lane).
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;

struct RouterSmem {
  uint32_t a_bytes, b_bytes, stage_bytes, ctrl;
};

__host__ __device__ inline RouterSmem router_smem(int E) {
  RouterSmem r;
  const int np = (E + 15) & ~15;
  r.a_bytes = kRouterTileM * 128;
  r.b_bytes = np * 128;
  r.stage_bytes = r.a_bytes + r.b_bytes;  // multiple of 2048
  r.ctrl = kStages * r.stage_bytes;
  return r;
}

constexpr size_t kCtrlBytes = 4096;  // barriers, flags, bias, offsets, histogram

__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, int T,
                  int d, int E, int k, const float* __restrict__ bias, const float* __restrict__ logit_offset,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate, int32_t* __restrict__ counts,
                  int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const RouterSmem L = router_smem(E);
  uint8_t* ctrl = smem + L.ctrl;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);          // [kStages]
  uint64_t* empty = full + kStages;                             // [kStages]
  uint64_t* tmem_full = empty + kStages;
  uint64_t* drain = tmem_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 80);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 84);
  volatile int* zero_flag = reinterpret_cast<volatile int*>(ctrl + 88);  // stays 0
  int* last_round = reinterpret_cast<int*>(ctrl + 96);                   // [kStages]
  float* s_bias = reinterpret_cast<float*>(ctrl + 256);
  float* s_off = s_bias + kMaxE;
  int* s_hist = reinterpret_cast<int*>(s_off + kMaxE);
  float* s_score = reinterpret_cast<float*>(smem);  // [128][np + 1], reuses the ring after the MMAs

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x;
  const int nk = d / 64;
  const int np = (E + 15) & ~15;
  uint32_t ncols = 32;
  while ((int)ncols < np) ncols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      last_round[s] = -1;
    }
    mbar_init(tmem_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *zero_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_w);
  }
  for (int i = threadIdx.x; i < kMaxE; i += kThreads) {
    s_bias[i] = i < E ? bias[i] : 0.0f;
    s_off[i] = (i < E && logit_offset) ? logit_offset[i] : 0.0f;
    s_hist[i] = 0;
  }
  if (warp == 1) tmem_alloc(tmem_slot, ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages, r = kb / kStages;
      if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, status, status + 1, kSiteRouterProducer)) break;
      uint8_t* st = smem + s * L.stage_bytes;
      mbar_arrive_expect_tx(&full[s], L.stage_bytes);
      tma_load_2d(st, &map_x, &full[s], kb * 64, tile * kRouterTileM);
      tma_load_2d(st + L.a_bytes, &map_w, &full[s], kb * 64, 0);
      last_round[s] = r;
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = idesc_bf16(128, np);
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages, r = kb / kStages;
      if (!mbar_wait(&full[s], r & 1, abort_flag, status, status + 1, kSiteRouterMma)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a = smem_u32(smem + s * L.stage_bytes);
      const uint32_t b = a + L.a_bytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tmem, sdesc_k128(a + kk * 32), sdesc_k128(b + kk * 32), idesc, (kb | kk) != 0);
      mma_commit(&empty[s]);
    }
    if (ok) mma_commit(tmem_full);
    // drain: every MMA of this thread has finished before TMEM is released
    mma_commit(drain);
    mbar_wait(drain, 0, abort_flag, status, status + 1, kSiteRouterMma, 100000000ull);
  } else if (warp >= 2) {
    // ---- phase 1 (warps 2-5, one token per TMEM lane): s = sigmoid(z + o) into
    // shared memory, [token][expert] with a padded row, reusing the drained ring
    const int q = warp & 3;
    const int row = q * 32 + lane;
    if (mbar_wait(tmem_full, 0, abort_flag, status, status + 1, kSiteRouterEpi)) {
      tc_fence_after();
      for (int c0 = 0; c0 < np; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c0 + i;
          if (e < np) {
            const float z = __uint_as_float(r[i]) + s_off[e];
            s_score[row * (np + 1) + e] = __fdividef(1.0f, 1.0f + __expf(-z));
          }
        }
      }
      tc_fence_before();
    }
  }
  __syncthreads();
  if (!*abort_flag) {
    // ---- phase 2 (all warps): top-k of s + b by k rounds of a warp arg-max over 8
    // experts per lane (expert e = lane + 32 i); ties go to the lower expert index;
    // gates = chosen s / sum of chosen s.  Each warp works on kTok tokens at once so
    // that their shuffle chains overlap.
    constexpr int kPer = kMaxE / 32;
    constexpr int kTok = 4;
    for (int row0 = warp * kTok; row0 < kRouterTileM; row0 += (kThreads / 32) * kTok) {
      float v[kTok][kPer], sc[kTok][kPer];
#pragma unroll
      for (int tt = 0; tt < kTok; ++tt) {
        const int row = row0 + tt;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int e = lane + 32 * i;
          if (e < E) {
            sc[tt][i] = s_score[row * (np + 1) + e];
            const float b = sc[tt][i] + s_bias[e];
            v[tt][i] = (b == b) ? fminf(fmaxf(b, -3.0e38f), 3.0e38f) : -3.0e38f;
          } else {
            sc[tt][i] = 0.0f;
            v[tt][i] = -INFINITY;
          }
        }
      }
      int my_idx[kTok];
      float my_s[kTok], sum[kTok];
#pragma unroll
      for (int tt = 0; tt < kTok; ++tt) {
        my_idx[tt] = 0;
        my_s[tt] = 0.0f;
        sum[tt] = 0.0f;
      }
      for (int j = 0; j < k; ++j) {
        float bv[kTok];
        int bi[kTok];
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt) {  // lane-local best (value descending, index ascending)
          bv[tt] = -INFINITY;
          bi[tt] = 0x7fffffff;
#pragma unroll
          for (int i = 0; i < kPer; ++i)
            if (v[tt][i] > bv[tt]) {
              bv[tt] = v[tt][i];
              bi[tt] = lane + 32 * i;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
          for (int tt = 0; tt < kTok; ++tt) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv[tt], o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi[tt], o);
            if (ov > bv[tt] || (ov == bv[tt] && oi < bi[tt])) {
              bv[tt] = ov;
              bi[tt] = oi;
            }
          }
        }
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt) {  // the owner lane retires the winner and shares its affinity
          float ws = 0.0f;
          if ((bi[tt] & 31) == lane) {
#pragma unroll
            for (int i = 0; i < kPer; ++i)
              if (lane + 32 * i == bi[tt]) {
                ws = sc[tt][i];
                v[tt][i] = -INFINITY;
              }
          }
          ws = __shfl_sync(0xffffffffu, ws, bi[tt] & 31);
          sum[tt] += ws;
          if (lane == j) {
            my_idx[tt] = bi[tt];
            my_s[tt] = ws;
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kTok; ++tt) {
        const int t = tile * kRouterTileM + row0 + tt;
        if (lane < k && t < T) {
          topk_idx[(size_t)t * k + lane] = my_idx[tt];
          topk_gate[(size_t)t * k + lane] = __fdiv_rn(my_s[tt], sum[tt]);
          atomicAdd(&s_hist[my_idx[tt]], 1);
        }
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kThreads)
    if (s_hist[e]) atomicAdd(&counts[e], s_hist[e]);
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // do not leave TMA writes in flight into shared memory
    for (int s = 0; s < kStages; ++s)
      if (last_round[s] >= 0)
        mbar_wait(&full[s], last_round[s] & 1, zero_flag, status, status + 1, kSiteRouterProducer,
                  100000000ull);
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// offsets[0] = 0, offsets[i+1] = offsets[i] + counts[i]
__global__ void offsets_kernel(const int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int E) {
  __shared__ int buf[2][kMaxE];
  const int i = threadIdx.x;
  int v = i < E ? counts[i] : 0;
  int cur = 0;
  buf[0][i] = v;
  __syncthreads();
  for (int off = 1; off < kMaxE; off <<= 1) {
    const int nv = buf[cur][i] + (i >= off ? buf[cur][i - off] : 0);
    buf[cur ^ 1][i] = nv;
    cur ^= 1;
    __syncthreads();
  }
  if (i < E) offsets[i + 1] = buf[cur][i];
  if (i == 0) offsets[0] = 0;
}

}  // namespace

moe_status_t launch_route(const moe_shape_t& s, const void* x, const void* w_router, const float* bias,
                          const float* logit_offset, int32_t* idx, float* gate, int32_t* counts, int32_t* offsets,
                          void* ws, cudaStream_t st) {
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.E, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (s.T > 0) {
    CUtensorMap mx, mw;
    const int np = (s.E + 15) & ~15;
    if (!make_map_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.d, s.T, 64, kRouterTileM)) return MOE_ERR_CUDA;
    if (!make_map_2d(&mw, w_router, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.d, s.E, 64, np)) return MOE_ERR_CUDA;
    const RouterSmem L = router_smem(s.E);
    const size_t smem = 1024 + L.ctrl + kCtrlBytes;
    const int grid = (s.T + kRouterTileM - 1) / kRouterTileM;
    int* status = ws_status(ws);
    auto kern = router_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    kern<<<grid, kThreads, smem, st>>>(mx, mw, s.T, s.d, s.E, s.k, bias, logit_offset, idx, gate, counts, status);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  offsets_kernel<<<1, kMaxE, 0, st>>>(counts, offsets, s.E);
  return cuda_status(cudaGetLastError());
}

}  // namespace moe
