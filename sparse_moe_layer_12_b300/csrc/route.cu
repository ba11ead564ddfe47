// Router: z = x . w_router^T on the tcgen05 tensor cores, fused with the
// sigmoid affinity, the selection bias, the per-token top-k, the gate
// normalisation over the chosen set and the per-expert load histogram.
//
// Pages: "deepseek-v3-report" (dynmi.github.io), load-balancing paragraph (b_i
// added to the routing score for selection, out of the gradient);
// "DeepSeek-V3 详解" (yudonglee.me) 2.2-2.3 (top-8 of 256, bias); readings for
// the silent points (sigmoid, gate normalisation, tie-break) in include/moe.h.
//
// Work split: a cluster of 2 * ksplit CTAs owns 256 tokens.  Its CTAs form
// ksplit pairs (cluster ranks 2p and 2p + 1), pair p covering K range p; each pair
// runs M = 256 tcgen05 MMAs over both CTAs (cta_group::2): CTA q of the pair loads
// its own 128 token rows and half of the expert rows of w_router (so a stage is
// 32 KB and six fit), the even CTA issues the MMAs, and each CTA ends with its
// 128 tokens x E partial logits in TMEM (one token per lane).  With ksplit = 2 the
// two K halves of a token tile sit in CTAs 2 apart; each keeps 64 of the tile's
// tokens and receives the other CTA's partial logits for them in one bulk
// shared-to-shared copy.  Warp roles: warp 0 TMA producer, warp 1 MMA issuer (even
// CTA), warps 2-5 move TMEM to shared memory (one lane quadrant each); then all 16
// warps select the top-k of whole tokens (8 threads a token).  The load histogram
// goes into counters in the workspace; the last CTA to finish writes counts and
// offsets and clears the counters, so one launch does the whole call.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kStages = 6;
constexpr int kThreads = 512;  // 16 warps: roles in warps 0-5, all warps in the top-k phase

struct RouterSmem {
  uint32_t a_bytes, b_bytes, stage_bytes, zrow, z_bytes, recv_bytes, region;
};

// Shared-memory plan: a ring of kStages (token rows + half of the expert rows);
// after the MMAs the same region holds the partial logits [128][np + 1] FP32 and,
// with the K split, the partner's [64][np + 1] partial for this CTA's tokens.
__host__ __device__ inline RouterSmem router_smem(int E, int ksplit) {
  RouterSmem r;
  const int np = (E + 15) & ~15;
  r.a_bytes = kRouterTileM * 128;
  r.b_bytes = (np / 2) * 128;
  r.stage_bytes = (r.a_bytes + r.b_bytes + 1023) & ~1023u;
  r.zrow = (np + 1) * 4;
  r.z_bytes = kRouterTileM * r.zrow;
  r.recv_bytes = ksplit == 2 ? (kRouterTileM / 2) * r.zrow : 0;
  const uint32_t ring = kStages * r.stage_bytes;
  const uint32_t z = (r.z_bytes + r.recv_bytes + 1023) & ~1023u;
  r.region = ring > z ? ring : z;
  return r;
}

constexpr size_t kCtrlBytes = 4096;  // barriers, flags, bias, offsets, histogram

// The candidate filter of the top-k: scores are first estimated as
// v' = (1 + tanh(z' / 2)) / 2 + b with one tanh.approx (relative error below 2^-10.9,
// so |v' - v| < 2.5e-4 plus rounding); kFilterEps bounds |v' - v| with margin.
constexpr float kFilterEps = 2.0e-3f;

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

// (v, e) ranks above (w, f): larger biased score first, lower expert index on ties.
__device__ __forceinline__ bool ranks_above(float v, int e, float w, int f) { return v > w || (v == w && e < f); }

// Top-8 of one token held by 8 consecutive lanes, each with its own descending list
// (lv, le) of 8: three rounds of exchanging lists with the lane 1, 2, 4 apart and
// keeping the better half (bitonic: pair own entry i with the partner's entry 7 - i,
// then sort the bitonic 8 with compare-exchanges at distances 4, 2, 1).  Every lane
// of the group ends with the token's top-8, in ranking order.
__device__ __forceinline__ void merge_top8(float (&lv)[8], int (&le)[8]) {
#pragma unroll
  for (int m = 1; m < 8; m <<= 1) {
    float pv[8];
    int pe[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      pv[i] = __shfl_xor_sync(0xffffffffu, lv[i], m);
      pe[i] = __shfl_xor_sync(0xffffffffu, le[i], m);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool mine = ranks_above(lv[i], le[i], pv[7 - i], pe[7 - i]);
      lv[i] = mine ? lv[i] : pv[7 - i];
      le[i] = mine ? le[i] : pe[7 - i];
    }
#pragma unroll
    for (int dist = 4; dist >= 1; dist >>= 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if ((i & dist) == 0) {
          const int j = i + dist;
          const bool keep = ranks_above(lv[i], le[i], lv[j], le[j]);
          const float a = lv[i], b = lv[j];
          const int ea = le[i], eb = le[j];
          lv[i] = keep ? a : b;
          le[i] = keep ? ea : eb;
          lv[j] = keep ? b : a;
          le[j] = keep ? eb : ea;
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    router_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, int T,
                  int d, int E, int k, const float* __restrict__ bias, const float* __restrict__ logit_offset,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_gate, int32_t* __restrict__ counts,
                  int32_t* __restrict__ offsets, int* __restrict__ load_acc, int ksplit, int n_group, int topk_group,
                  int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const RouterSmem L = router_smem(E, ksplit);
  uint8_t* ctrl = smem + L.region;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);          // [kStages], used in the even CTA
  uint64_t* empty = full + kStages;                             // [kStages]
  uint64_t* tmem_full = empty + kStages;
  uint64_t* drain = tmem_full + 1;
  uint64_t* xchg = drain + 1;                                   // partner's partial logits arrived
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 132);
  volatile int* zero_flag = reinterpret_cast<volatile int*>(ctrl + 136);  // stays 0
  int* last_round = reinterpret_cast<int*>(ctrl + 144);                   // [kStages]
  int* s_last = reinterpret_cast<int*>(ctrl + 200);                       // this CTA finished last
  float* s_bias = reinterpret_cast<float*>(ctrl + 256);
  float* s_off = s_bias + kMaxE;
  int* s_hist = reinterpret_cast<int*>(s_off + kMaxE);
  int* s_wsum = s_hist;  // [kThreads / 32] warp sums of the offsets scan, once s_hist is spent
  float* s_z = reinterpret_cast<float*>(smem);                      // [128][np + 1], after the MMAs
  float* s_recv = reinterpret_cast<float*>(smem + L.z_bytes);       // [64][np + 1], K split only

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank();
  const uint32_t q = crank & 1u;            // token tile of the pair / half of the expert rows
  const int part = static_cast<int>(crank >> 1);  // K range
  const uint32_t leader = crank & ~1u;      // even CTA of this pair
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << leader);
  const int tok0 = static_cast<int>(cluster_id_x()) * (2 * kRouterTileM) + static_cast<int>(q) * kRouterTileM;
  const int nk_all = d / 64;
  const int per = (nk_all + ksplit - 1) / ksplit;
  const int kb0 = part * per;
  const int nk = max(0, min(nk_all, kb0 + per) - kb0);  // K blocks of this pair: [kb0, kb0 + nk)
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
    mbar_init(xchg, 1);
    *abort_flag = 0;
    *zero_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_w);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, ncols);
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in every CTA of the cluster
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t full_leader = map_to_rank(smem_u32(full), leader);

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: this CTA's token rows and its half of the expert rows; every
    // load of a stage completes on the even CTA's barrier
    const uint32_t bytes_pair = 2 * (L.a_bytes + L.b_bytes);
    for (int kb = 0; kb < nk; ++kb) {
      const int s = kb % kStages, r = kb / kStages;
      if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, status, status + 1, kSiteRouterProducer)) break;
      uint8_t* st = smem + s * L.stage_bytes;
      const uint32_t fb = full_leader + s * 8;
      if (q == 0) mbar_arrive_expect_tx(&full[s], bytes_pair);
      tma_load_2d_pair(st, &map_x, fb, (kb0 + kb) * 64, tok0);
      tma_load_2d_pair(st + L.a_bytes, &map_w, fb, (kb0 + kb) * 64, static_cast<int>(q) * (np / 2));
      last_round[s] = r;
    }
  } else if (warp == 1 && lane == 0 && q == 0) {
    // ---- MMA issuer (even CTA): M = 256 tokens of the pair, N = np experts
    const uint32_t idesc = idesc_bf16(256, np);
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
        mma_bf16_pair(tmem, sdesc_k128(a + kk * 32), sdesc_k128(b + kk * 32), idesc, (kb | kk) != 0);
      mma_commit_pair_mc(&empty[s], pair_mask);
    }
    if (ok) mma_commit_pair_mc(tmem_full, pair_mask);
    // drain: every MMA of this thread has finished before TMEM is released
    mma_commit_pair(drain);
    mbar_wait(drain, 0, zero_flag, status, status + 1, kSiteRouterMma, 100000000ull);
  } else if (warp >= 2 && warp < 6) {
    // ---- phase 1 (one token per TMEM lane): this CTA's partial logits into shared
    // memory, [token][expert] with a padded row, reusing the drained ring
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    if (mbar_wait(tmem_full, 0, abort_flag, status, status + 1, kSiteRouterEpi)) {
      tc_fence_after();
      for (int c0 = 0; c0 < np; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(qd * 32) << 16) + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < np) s_z[row * (np + 1) + c0 + i] = nk > 0 ? __uint_as_float(r[i]) : 0.0f;
      }
      tc_fence_before();
    }
  } else if (warp >= 6) {
    // ---- meanwhile: selection bias, logit offsets and the histogram into shared memory
    for (int i = threadIdx.x - 192; i < kMaxE; i += kThreads - 192) {
      s_bias[i] = i < E ? bias[i] : 0.0f;
      s_off[i] = (i < E && logit_offset) ? logit_offset[i] : 0.0f;
      s_hist[i] = 0;
    }
  }
  __syncthreads();
  // With the K range split over the two pairs, each CTA keeps half of its tile's
  // tokens and receives the partner's partial logits for them (one bulk copy per
  // 16 rows into the partner's shared memory); z = own part + partner's part.
  int row_lo = 0, row_hi = kRouterTileM;
  if (ksplit == 2) {
    fence_proxy_async_smem();  // the bulk copy reads what phase 1 stored
    cluster_sync_all();        // every CTA has its partial in place and its ring free
    row_lo = part * (kRouterTileM / 2);
    row_hi = row_lo + kRouterTileM / 2;
    if (threadIdx.x == 0) {
      const uint32_t partner = crank ^ 2u;
      const int give = (1 - part) * (kRouterTileM / 2);  // the rows the partner keeps
      const uint32_t chunk = 16 * L.zrow;
      mbar_arrive_expect_tx(xchg, (kRouterTileM / 2) * L.zrow);
      const uint32_t dst = map_to_rank(smem_u32(s_recv), partner);
      const uint32_t bar = map_to_rank(smem_u32(xchg), partner);
      for (int c = 0; c < kRouterTileM / 2 / 16; ++c)
        bulk_copy_to_peer(dst + c * chunk, s_z + (size_t)(give + 16 * c) * (np + 1), chunk, bar);
    }
    // the partner's partial is added in place here for the warp-per-token path, and as
    // it is read by the 8-threads-per-token path below
    if (mbar_wait(xchg, 0, abort_flag, status, status + 1, kSiteRouterEpi) && (n_group > 0 || k > 8)) {
      for (int row = row_lo + warp; row < row_hi; row += kThreads / 32) {
        float* zz = s_z + row * (np + 1);
        const float* pp = s_recv + (row - row_lo) * (np + 1);
        for (int e = lane; e < E; e += 32) zz[e] = zz[e] + pp[e];
      }
    }
    __syncthreads();
  }
  if (!*abort_flag && n_group == 0 && k <= 8) {
    // ---- phase 2, plain top-k (k <= 8): 8 threads per token.  Thread (token, sub) owns
    // experts e = 32 b + 4 sub + c (b = 0..7, c = 0..3): for a fixed step the 32 lanes
    // of a warp (4 tokens x 8 subs) read 32 different shared-memory banks.
    //  (1) estimates v' of its 32 scores (kFilterEps above) and their maximum; tau' =
    //      the smallest of the token's 8 maxima.  Every thread's best element has
    //      v >= tau' - eps, so at least 8 scores reach tau' - eps, and each that does
    //      has v' >= tau' - 2 eps: those candidates hold the token's top-k;
    //  (2) the exact score v = sigmoid(z) + b of each candidate enters the thread's
    //      descending list of 8, experts in ascending order (a later expert enters only
    //      on a strictly larger score, so ties keep the lower index);
    //  (3) the 8 lists of the token are merged; gates = chosen s / sum of the chosen s,
    //      summed in ranking order.
    const int sub = threadIdx.x & 7;
    for (int tb = row_lo; tb < row_hi; tb += kThreads / 8) {
      const int row = tb + (threadIdx.x >> 3);
      const bool live = row < row_hi && tok0 + row < T;
      float* zr = s_z + row * (np + 1);
      const float* pr = s_recv + (row - row_lo) * (np + 1);  // the partner's partial (K split)
      auto logit = [&](int e) -> float {
        float z = zr[e];
        if (ksplit == 2) z = z + pr[e];
        return z + s_off[e];
      };
      auto score = [&](int e) -> float {
        const float sc = __fdividef(1.0f, 1.0f + __expf(-logit(e)));
        const float b = sc + s_bias[e];
        return (b == b) ? fminf(fmaxf(b, -3.0e38f), 3.0e38f) : -3.0e38f;
      };
      float v[32];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int e = 32 * (j >> 2) + 4 * sub + (j & 3);
        float a = -INFINITY;
        if (live && e < E) {
          float t;
          asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * logit(e)));
          a = fminf(fmaxf(fmaf(0.5f, t, 0.5f) + s_bias[e], -3.0e38f), 3.0e38f);  // NaN -> -3e38
        }
        v[j] = a;
        mx = fmaxf(mx, a);
      }
      float tau = mx;
      tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, 1));
      tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, 2));
      tau = fminf(tau, __shfl_xor_sync(0xffffffffu, tau, 4));
      tau -= 2.0f * kFilterEps;
      uint32_t cand = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) cand |= (v[j] < tau ? 0u : 1u) << j;
      if (!live) cand = 0;
      float lv[8];
      int le[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        lv[i] = -INFINITY;
        le[i] = 0x7fffffff;
      }
      while (cand) {
        const int j = __ffs(cand) - 1;
        cand &= cand - 1;
        const int e = 32 * (j >> 2) + 4 * sub + (j & 3);
        const float w = e < E ? score(e) : -INFINITY;
        bool c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = w > lv[i];
#pragma unroll
        for (int i = 7; i >= 1; --i) {
          lv[i] = c[i - 1] ? lv[i - 1] : (c[i] ? w : lv[i]);
          le[i] = c[i - 1] ? le[i - 1] : (c[i] ? e : le[i]);
        }
        lv[0] = c[0] ? w : lv[0];
        le[0] = c[0] ? e : le[0];
      }
      merge_top8(lv, le);
      // lane `sub` of the token's group takes rank sub; the k affinities are gathered
      // from the group's lanes and summed in ranking order
      int my_e = le[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) my_e = sub == i ? le[i] : my_e;
      float my_s = 0.0f;
      if (live && sub < k && my_e < E) my_s = __fdividef(1.0f, 1.0f + __expf(-logit(my_e)));
      float sum = 0.0f;
      const int grp = lane & ~7;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float si = __shfl_sync(0xffffffffu, my_s, grp | i);
        if (i < k) sum += si;
      }
      if (live && sub < k) {
        const int t = tok0 + row;
        if (my_e >= 0 && my_e < E) {
          topk_idx[(size_t)t * k + sub] = my_e;
          topk_gate[(size_t)t * k + sub] = __fdiv_rn(my_s, sum);
          atomicAdd(&s_hist[my_e], 1);
        } else {  // fewer than k entries: cannot happen for k <= E
          set_error(status, status + 1, MOE_ERR_DEVICE, kSiteRouterEpi);
        }
      }
    }
  } else if (!*abort_flag) {
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
          if (e < E && tok0 + row < T) {
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
        const int t = tok0 + row0 + tt;
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
    if (s_hist[e]) atomicAdd(&load_acc[e], s_hist[e]);
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag && q == 0) {
    // this pair's loads completed on this CTA's barriers: do not leave TMA writes in flight
    for (int s = 0; s < kStages; ++s)
      if (last_round[s] >= 0)
        mbar_wait(&full[s], last_round[s] & 1, zero_flag, status, status + 1, kSiteRouterProducer,
                  100000000ull);
  }
  tc_fence_before();
  cluster_sync_all();  // the partner has read this CTA's partial; the pair is done with TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, ncols);
  }
  // ---- the load: every CTA has added its histogram into load_acc[0, E); a ticket in
  // load_acc[kMaxE] finds the last CTA, which writes counts and their exclusive prefix
  // sum (offsets[0] = 0, offsets[i+1] = offsets[i] + counts[i]) and clears the counters
  // and the ticket for the next call
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *s_last = atomicAdd(&load_acc[kMaxE], 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (*s_last) {
    __threadfence();
    const int c = threadIdx.x < E ? atomicExch(&load_acc[threadIdx.x], 0) : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_wsum[w];
    if (threadIdx.x < E) {
      counts[threadIdx.x] = c;
      offsets[threadIdx.x + 1] = base + incl;
    }
    if (threadIdx.x == 0) {
      offsets[0] = 0;
      atomicExch(&load_acc[kMaxE], 0);
    }
  }
}

}  // namespace

moe_status_t launch_route(const moe_shape_t& s, const void* x, const void* w_router, const float* bias,
                          const float* logit_offset, int32_t* idx, float* gate, int32_t* counts, int32_t* offsets,
                          void* ws, cudaStream_t st) {
  if (s.T == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.E, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (s.E + 1), st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  {
    const int nsuper = (s.T + 2 * kRouterTileM - 1) / (2 * kRouterTileM);  // 256-token tiles
    CUtensorMap mx, mw;
    const int np = (s.E + 15) & ~15;
    if (!make_map_2d(&mx, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.d, s.T, 64, kRouterTileM)) return MOE_ERR_CUDA;
    if (!make_map_2d(&mw, w_router, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.d, s.E, 64, np / 2)) return MOE_ERR_CUDA;
    auto kern = router_kernel;
    int* status = ws_status(ws);
    // split K over two pairs (clusters of 4) when all clusters fit at once
    int ksplit = 1;
    if (s.d >= 256) {
      const size_t smem4 = 1024 + router_smem(s.E, 2).region + kCtrlBytes;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem4) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (max_active_clusters((const void*)kern, 4, kThreads, smem4) >= nsuper) ksplit = 2;
    }
    const size_t smem = 1024 + router_smem(s.E, ksplit).region + kCtrlBytes;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nsuper * 2 * ksplit), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(2 * ksplit);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, mx, mw, s.T, s.d, s.E, s.k, bias, logit_offset, idx, gate, counts, offsets,
                           ws_load_acc(ws), ksplit, s.n_group, s.topk_group, status) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
