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
constexpr int kThreads = 512;  // 16 warps: roles in warps 0-5, all warps in the top-k phase

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

__device__ __forceinline__ uint32_t order_key(float v) {  // monotone float -> uint32
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Group-limited selection for one token held by a warp (expert e = lane + 32 i):
// group score = FP32 sum, in descending order, of the group's ceil(k / topk_group)
// largest biased scores; the topk_group best groups (ties to the lower group) stay
// eligible, every other expert's score becomes -inf.
__device__ __forceinline__ void group_limit(float (&v)[kMaxE / 32], int lane, int E, int k, int n_group,
                                            int topk_group) {
  constexpr int kPer = kMaxE / 32;
  const int gsz = E / n_group;
  const int m = (k + topk_group - 1) / topk_group;
  float gs_lane = -INFINITY;  // lane g holds the score of group g
  for (int g = 0; g < n_group; ++g) {
    uint32_t taken = 0;
    float sum = 0.0f;
    for (int r = 0; r < m; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        const bool ok = e < E && e / gsz == g && !((taken >> i) & 1u) && v[i] > bv;
        bv = ok ? v[i] : bv;
        bi = ok ? e : bi;
      }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(bv));
      const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, order_key(bv) == kmax ? (uint32_t)bi : 0x7fffffffu));
      sum += key_value(kmax);
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (lane + 32 * i == win) taken |= 1u << i;
    }
    gs_lane = lane == g ? sum : gs_lane;
  }
  uint32_t keep = 0;
  float gv = lane < n_group ? gs_lane : -INFINITY;
  for (int r = 0; r < topk_group; ++r) {
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, order_key(gv));
    const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, order_key(gv) == kmax ? (uint32_t)lane : 32u));
    keep |= 1u << win;
    gv = lane == win ? -INFINITY : gv;
  }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    if (e < E && !((keep >> (e / gsz)) & 1u)) v[i] = -INFINITY;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, int T,
                  int d, int E, int k, const float* __restrict__ bias, const float* __restrict__ logit_offset,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate, int32_t* __restrict__ counts,
                  int ksplit, int n_group, int topk_group, int* __restrict__ status) {
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
  float* s_z = reinterpret_cast<float*>(smem);  // [128][np + 1] logits, reuses the ring after the MMAs

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / ksplit;
  const int part = blockIdx.x - tile * ksplit;
  const int nk_all = d / 64;
  const int per = (nk_all + ksplit - 1) / ksplit;
  const int kb0 = part * per;
  const int nk = max(0, min(nk_all, kb0 + per) - kb0);  // K blocks of this CTA: [kb0, kb0 + nk)
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
      tma_load_2d(st, &map_x, &full[s], (kb0 + kb) * 64, tile * kRouterTileM);
      tma_load_2d(st + L.a_bytes, &map_w, &full[s], (kb0 + kb) * 64, 0);
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
  } else if (warp >= 2 && warp < 6) {
    // ---- phase 1 (warps 2-5, one token per TMEM lane): this CTA's partial logits
    // into shared memory, [token][expert] with a padded row, reusing the drained ring
    const int q = warp & 3;
    const int row = q * 32 + lane;
    if (mbar_wait(tmem_full, 0, abort_flag, status, status + 1, kSiteRouterEpi)) {
      tc_fence_after();
      for (int c0 = 0; c0 < np; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < np) s_z[row * (np + 1) + c0 + i] = nk > 0 ? __uint_as_float(r[i]) : 0.0f;
      }
      tc_fence_before();
    }
  }
  __syncthreads();
  // With the K range split over the two CTAs of a cluster, each CTA takes half of
  // the tile's tokens and reads the peer's partial logits for them from the peer's
  // shared memory; the parts are added in part order (part 0 + part 1).
  int row_lo = 0, row_hi = kRouterTileM;
  if (ksplit == 2) {
    cluster_sync_all();
    row_lo = part * (kRouterTileM / 2);
    row_hi = row_lo + kRouterTileM / 2;
    const uint32_t peer = static_cast<uint32_t>(1 - part);
    for (int row = row_lo + warp; row < row_hi; row += kThreads / 32) {
      for (int e = lane; e < E; e += 32) {
        float* zz = s_z + row * (np + 1) + e;
        const float pv = ld_dsmem_f32(map_to_rank(smem_u32(zz), peer));
        *zz = part == 0 ? *zz + pv : pv + *zz;
      }
    }
  }
  __syncthreads();
  if (!*abort_flag) {
    // ---- phase 2 (all warps): top-k of s + b by k rounds of a warp arg-max over 8
    // experts per lane (expert e = lane + 32 i); ties go to the lower expert index;
    // gates = chosen s / sum of chosen s.  Each warp works on kTok tokens at once so
    // that their shuffle chains overlap.
    constexpr int kPer = kMaxE / 32;
    constexpr int kTok = 2;
    for (int row0 = row_lo + warp * kTok; row0 < row_hi; row0 += (kThreads / 32) * kTok) {
      float v[kTok][kPer], sc[kTok][kPer];
#pragma unroll
      for (int tt = 0; tt < kTok; ++tt) {
        const int row = row0 + tt;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int e = lane + 32 * i;
          if (e < E && tile * kRouterTileM + row < T) {
            const float z = s_z[row * (np + 1) + e] + s_off[e];
            sc[tt][i] = __fdividef(1.0f, 1.0f + __expf(-z));
            const float b = sc[tt][i] + s_bias[e];
            v[tt][i] = (b == b) ? fminf(fmaxf(b, -3.0e38f), 3.0e38f) : -3.0e38f;
          } else {
            sc[tt][i] = 0.0f;
            v[tt][i] = -INFINITY;
          }
        }
      }
      if (n_group > 0) {
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt) group_limit(v[tt], lane, E, k, n_group, topk_group);
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
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt) {
          // this lane's best remaining expert (value descending, index ascending)
          float bv = -INFINITY;
          int bi = 0x7fffffff;
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const bool gt = v[tt][i] > bv;
            bv = gt ? v[tt][i] : bv;
            bi = gt ? lane + 32 * i : bi;
          }
          // the warp's best value via an order-preserving integer key, then the lowest
          // expert index among the lanes that hold it
          const uint32_t bits = __float_as_uint(bv);
          const uint32_t key = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
          const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
          const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, key == kmax ? (uint32_t)bi : 0x7fffffffu));
          // the owner lane retires the winner; its affinity is broadcast
          float ws = 0.0f;
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            const bool hit = lane + 32 * i == win;
            ws = hit ? sc[tt][i] : ws;
            v[tt][i] = hit ? -INFINITY : v[tt][i];
          }
          ws = __shfl_sync(0xffffffffu, ws, win & 31);
          sum[tt] += ws;
          my_idx[tt] = lane == j ? win : my_idx[tt];
          my_s[tt] = lane == j ? ws : my_s[tt];
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
  if (ksplit == 2) cluster_sync_all();  // the peer has finished reading this CTA's shared memory
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
    const int ntiles = (s.T + kRouterTileM - 1) / kRouterTileM;
    // split K over the two CTAs of a cluster when that still fits one wave (1 CTA per SM)
    const int ksplit = (2 * ntiles <= sm_count() && s.d >= 256) ? 2 : 1;
    CUtensorMap mx, mw;
    const int np = (s.E + 15) & ~15;
    if (!make_map_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.d, s.T, 64, kRouterTileM)) return MOE_ERR_CUDA;
    if (!make_map_2d(&mw, w_router, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.d, s.E, 64, np)) return MOE_ERR_CUDA;
    const RouterSmem L = router_smem(s.E);
    const size_t smem = 1024 + L.ctrl + kCtrlBytes;
    int* status = ws_status(ws);
    auto kern = router_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ntiles * ksplit), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(ksplit);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mx, mw, s.T, s.d, s.E, s.k, bias, logit_offset, idx, gate, counts, ksplit,
                           s.n_group, s.topk_group, status) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  offsets_kernel<<<1, kMaxE, 0, st>>>(counts, offsets, s.E);
  return cuda_status(cudaGetLastError());
}

}  // namespace moe
