// FP8 (E4M3) grouped SwiGLU expert GEMMs with the pages' fine-grained scaling:
// activations carry one FP32 scale per 1x128 tile (per token per 128 channels),
// weights one per 128x128 block, and the products are accumulated in FP32
// ("DeepSeek-V3 详解" 4.2 fine-grained quantization, 4.3 FP32 accumulation;
// "deepseek-v3-report" FP8 paragraph).
//
//   y[f, t] = sum_kb  s_w[f/128, kb] * s_a[t, kb] * P_kb[f, t],
//   P_kb    = sum_{k in block kb} q_w[f, k] * q_a[t, k]        (tcgen05 kind::f8f6f4, FP32)
//
// The scales differ per 128-wide K block, so the tensor core accumulates one K
// block at a time into a TMEM partial (two partials, double-buffered) and the
// epilogue warps promote each partial into FP32 register accumulators with the
// product of the two scales -- the block-wise FP32 promotion the pages describe.
//
// Tile: M = 128 weight rows (two of them per tile, as in the bf16 kernel: gate
// and up rows of the same 128 features, or two 128-channel blocks of W_down),
// N <= 96 tokens of one group, K block = 128 bytes = one 128-byte swizzle row.
// In the gathering variant (the fused forward) the routed token rows are read
// straight from the E4M3 copy of x: lane q of the producer warp gathers rows
// 4q .. 4q + 3 of the chunk with one TMA row gather per K block (token indices
// from the permutation table), and the scales come from the per-token scale
// rows -- the dispatch step fused into the operand load.
// Warps: 0 TMA producer, 1 MMA issuer, 2-13 promotion/epilogue in three groups
// of four (group g owns token columns [32g, 32g + 32), warp w TMEM lanes of
// quadrant w % 4).  The gate/up epilogue computes h = silu(g) * u and
// quantises it per token per 128 features (one tile = the tile's 128
// features) into E4M3 + FP32 scale for the down GEMM; the down epilogue writes
// bf16 rows of y.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kGroups = 3;       // epilogue groups, 32 token columns each
constexpr int kChunk = 32 * kGroups;  // tokens per tile (N)
constexpr int kStages = 4;

constexpr int kThreads = 64 + kGroups * 128;
constexpr uint32_t kATile = 128 * 128;
constexpr uint32_t kBTile = kChunk * 128;
constexpr uint32_t kBox = kBoxRows * 128;
constexpr uint32_t kStage = 2 * kATile + kBTile;  // 48 KB
constexpr int kStgStride = 136;                   // bf16 elements per staging row
constexpr uint32_t kStgBytes = kGroups * 32 * kStgStride * 2;
constexpr uint32_t kCtrl = 4096;
constexpr size_t kSmemBytes = 1024 + kStages * kStage + kStgBytes + kCtrl;

enum Mode : int { kGateUp = 0, kDown = 1 };

struct TileInfo {
  int g, m, tok0, n, expert, brow0, out_row0;
  bool shared_b;
};

__device__ __forceinline__ bool decode_tile(const GroupInfo* __restrict__ groups, const int* __restrict__ ts,
                                            int G, int E, int tile, int mode, TileInfo& ti) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ts + mid) <= tile) lo = mid;
    else hi = mid;
  }
  const GroupInfo gi = groups[lo];
  if (gi.nchunks <= 0) return false;
  const int local = tile - __ldg(ts + lo);
  ti.g = lo;
  ti.m = local / gi.nchunks;
  const int c = local - ti.m * gi.nchunks;
  ti.tok0 = c * gi.csize;
  ti.n = min(gi.csize, gi.n - ti.tok0);
  ti.expert = gi.expert;
  ti.out_row0 = gi.out_row0 + ti.tok0;
  ti.shared_b = (mode == kGateUp) && lo >= E;
  ti.brow0 = (mode == kGateUp ? gi.in_row0 : gi.out_row0) + ti.tok0;
  return ti.n > 0;
}

// GATHER (gate/up only): routed rows are gathered from the E4M3 copy of x (map_xg:
// [x_rows, K] bytes, box 128 x 1 row; scales sa1) through perm_token instead of
// read from map_b0 / sa0.
template <int MODE, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1)
    expert_gemm_fp8_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_b0,
                           const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_xg,
                           const GroupInfo* __restrict__ groups, const int* __restrict__ tile_start, int G, int E,
                           int K, int I, int d, const float* __restrict__ sa0, const float* __restrict__ sa1,
                           const float* __restrict__ sw, int w_rows, const int32_t* __restrict__ perm_token,
                           int x_rows, uint8_t* __restrict__ out, float* __restrict__ out_scale,
                           int* __restrict__ status) {
  static_assert(!GATHER || MODE == kGateUp, "row gather feeds the gate/up GEMM only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint16_t* stg = reinterpret_cast<uint16_t*>(smem + kStages * kStage);
  uint8_t* ctrl = smem + kStages * kStage + kStgBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);  // [kStages]
  uint64_t* empty = full + kStages;                    // [kStages]
  uint64_t* pfull = empty + kStages;                   // [2]
  uint64_t* pempty = pfull + 2;                        // [2]
  uint64_t* drain = pempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 132);
  volatile int* zero_flag = reinterpret_cast<volatile int*>(ctrl + 136);
  int* last_round = reinterpret_cast<int*>(ctrl + 144);           // [kStages]
  float* fac = reinterpret_cast<float*>(ctrl + 256);              // [kGroups][2 buffers][2][32]
  float* colmax = reinterpret_cast<float*>(ctrl + 256 + 2048);    // [kGroups][4 quadrants][32]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = K / 128;
  const int total = __ldg(tile_start + G);
  const int wblk_rows = w_rows / 128;  // 128-row weight blocks per expert

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      last_round[s] = -1;
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(&pfull[p], 1);
      mbar_init(&pempty[p], kGroups * 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *zero_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_b0);
    tma_prefetch_desc(&map_b1);
    if (GATHER) tma_prefetch_desc(&map_xg);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && GATHER) {
    // ---------------- producer with row gather (whole warp): lane 0 issues the weight
    // loads (and the shared experts' contiguous token rows), lane q gathers token rows
    // 4q .. 4q + 3 of a routed chunk
    uint32_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      TileInfo ti;
      if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti)) continue;
      const bool gat = !ti.shared_b;
      const int nm = (ti.n + 15) & ~15;
      const int nbox = gat ? 0 : (ti.n + kBoxRows - 1) / kBoxRows;
      const uint32_t bytes = 2 * kATile + (gat ? nm * 128u : nbox * kBox);
      const int a0 = ti.m * 128, a1 = I + ti.m * 128;
      const bool my_rows = gat && 4 * lane < nm;
      int tk[4] = {0, 0, 0, 0};
      if (my_rows) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int row = 4 * lane + u;  // padding rows repeat the chunk's first token
          int t = __ldg(perm_token + ti.brow0 + (row < ti.n ? row : 0));
          if (t < 0 || t >= x_rows) {
            set_error(status, status + 1, MOE_ERR_DEVICE, kSiteGemmProducer);
            t = 0;
          }
          tk[u] = t;
        }
      }
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = it % kStages, r = it / kStages;
        int waited = 1;
        if (lane == 0)
          waited = mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, status, status + 1, kSiteGemmProducer) ? 1 : 0;
        waited = __shfl_sync(0xffffffffu, waited, 0);
        if (!waited) {
          ok = false;
          break;
        }
        uint8_t* st = smem + s * kStage;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], bytes);
          tma_load_3d(st, &map_w, &full[s], kb * 128, a0, ti.expert);
          tma_load_3d(st + kATile, &map_w, &full[s], kb * 128, a1, ti.expert);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(st + 2 * kATile + b * kBox, &map_b1, &full[s], kb * 128, ti.brow0 + b * kBoxRows);
          last_round[s] = r;
        }
        if (my_rows) tma_gather4(st + 2 * kATile + lane * 512, &map_xg, &full[s], kb * 128, tk[0], tk[1], tk[2], tk[3]);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        TileInfo ti;
        if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti)) continue;
        const int nbox = (ti.n + kBoxRows - 1) / kBoxRows;
        const uint32_t bytes = 2 * kATile + nbox * kBox;
        const int a0 = MODE == kGateUp ? ti.m * 128 : ti.m * 256;
        const int a1 = MODE == kGateUp ? I + ti.m * 128 : ti.m * 256 + 128;
        const CUtensorMap* mb = ti.shared_b ? &map_b1 : &map_b0;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages, r = it / kStages;
          if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, status, status + 1, kSiteGemmProducer)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kStage;
          mbar_arrive_expect_tx(&full[s], bytes);
          tma_load_3d(st, &map_w, &full[s], kb * 128, a0, ti.expert);
          tma_load_3d(st + kATile, &map_w, &full[s], kb * 128, a1, ti.expert);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(st + 2 * kATile + b * kBox, mb, &full[s], kb * 128, ti.brow0 + b * kBoxRows);
          last_round[s] = r;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: one K block per TMEM partial
      uint32_t it = 0, u = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        TileInfo ti;
        if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti)) continue;
        const uint32_t idesc = idesc_e4m3(128, (ti.n + 15) & ~15);
        for (int kb = 0; kb < nk; ++kb, ++it, ++u) {
          const int s = it % kStages, r = it / kStages;
          const int p = u & 1;
          if (!mbar_wait(&pempty[p], ((u >> 1) & 1) ^ 1, abort_flag, status, status + 1, kSiteGemmMma) ||
              !mbar_wait(&full[s], r & 1, abort_flag, status, status + 1, kSiteGemmMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * kStage);
          const uint32_t d0 = tmem + p * 256;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = sdesc_k128(sa + 2 * kATile + kk * 32);
            mma_e4m3(d0, sdesc_k128(sa + kk * 32), bd, idesc, kk != 0);
            mma_e4m3(d0 + 128, sdesc_k128(sa + kATile + kk * 32), bd, idesc, kk != 0);
          }
          mma_commit(&empty[s]);
          mma_commit(&pfull[p]);
        }
      }
      mma_commit(drain);
      mbar_wait(drain, 0, zero_flag, status, status + 1, kSiteGemmTeardown, 100000000ull);
    }
  } else {
    // ---------------- promotion + epilogue
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int etid = (threadIdx.x - 64) & 127;
    const int f = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    float* gfac = fac + grp * 128;  // [2 buffers][2 operands][32]
    uint16_t* sg = stg + grp * (32 * kStgStride);
    uint32_t u = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      TileInfo ti;
      if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti)) continue;
      const int c0 = grp * 32;
      const bool has = c0 < ti.n;  // warp-uniform
      // scale factor computation for this thread (etid < 64): operand etid / 32, column etid % 32
      const int fop = etid >> 5, fcol = etid & 31;
      const float* sa_src = (GATHER || ti.shared_b) ? sa1 : sa0;
      const bool fvalid = etid < 64 && c0 + fcol < ti.n;
      size_t sa_rowi = (size_t)(ti.brow0 + c0 + fcol);  // scale row: permuted row, or token
      if (GATHER && !ti.shared_b && fvalid) {
        const int t = __ldg(perm_token + ti.brow0 + c0 + fcol);
        sa_rowi = (t < 0 || t >= x_rows) ? 0 : (size_t)t;
      }
      const int wrow = MODE == kGateUp ? (fop == 0 ? ti.m : I / 128 + ti.m) : 2 * ti.m + fop;
      const float* sw_row = sw + ((size_t)ti.expert * wblk_rows + (wrow < wblk_rows ? wrow : 0)) * nk;
      const float* sa_row = sa_src + sa_rowi * nk;
      float sa_next = fvalid ? __ldg(sa_row) : 0.0f;
      float sw_next = (etid < 64) ? __ldg(sw_row) : 0.0f;
      float acc_a[32], acc_b[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        acc_a[i] = 0.0f;
        acc_b[i] = 0.0f;
      }
      for (int kb = 0; kb < nk; ++kb, ++u) {
        const int p = u & 1;
        const float sa_cur = sa_next, sw_cur = sw_next;
        if (kb + 1 < nk) {
          sa_next = fvalid ? __ldg(sa_row + kb + 1) : 0.0f;
          sw_next = (etid < 64) ? __ldg(sw_row + kb + 1) : 0.0f;
        }
        float* fb = gfac + (kb & 1) * 64;
        if (etid < 64) fb[etid] = sa_cur * sw_cur;
        named_bar_sync(1 + grp, 128);
        if (!mbar_wait(&pfull[p], (u >> 1) & 1, abort_flag, status, status + 1, kSiteGemmEpi)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (has) {
          // stream 16-column slices of each operand's partial through the registers
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            const int op = sl >> 1, half = sl & 1;
            uint32_t r[16];
            tmem_ld16(tmem + lane_base + p * 256 + op * 128 + c0 + half * 16, r);
            tmem_ld_wait();
            if (sl == 3) {
              tc_fence_before();
              mbar_arrive(&pempty[p]);
            }
            const float* fs = fb + op * 32 + half * 16;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (op == 0) acc_a[half * 16 + i] = fmaf(__uint_as_float(r[i]), fs[i], acc_a[half * 16 + i]);
              else acc_b[half * 16 + i] = fmaf(__uint_as_float(r[i]), fs[i], acc_b[half * 16 + i]);
            }
          }
        } else {
          tc_fence_before();
          mbar_arrive(&pempty[p]);
        }
      }
      if (!ok) break;
      const int rows_here = min(32, ti.n - c0);
      if (MODE == kGateUp) {
        // h = silu(g) * u; one 1x128 tile per token = this tile's 128 features
        float* h = acc_a;  // h overwrites the gate accumulator
#pragma unroll
        for (int i = 0; i < 32; ++i) h[i] = __fdividef(acc_a[i], 1.0f + __expf(-acc_a[i])) * acc_b[i];
        // |h| max over the 32 lanes of this warp, per token column (bit pattern of |h| is monotone)
        uint32_t mine = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h[i])));
          if (lane == i) mine = m;
        }
        float* gmax = colmax + grp * 128;
        gmax[q * 32 + lane] = __uint_as_float(mine);
        named_bar_sync(1 + grp, 128);
        if (q == 0) {
          const float amax = fmaxf(fmaxf(gmax[lane], gmax[32 + lane]), fmaxf(gmax[64 + lane], gmax[96 + lane]));
          const float sc = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
          gmax[lane] = sc;  // reuse row 0 for the scales
          if (has && lane < rows_here) out_scale[(size_t)(ti.out_row0 + c0 + lane) * (I / 128) + ti.m] = sc;
        }
        named_bar_sync(1 + grp, 128);
        // codes, transposed to [token][feature] bytes in the staging tile
        uint8_t* sb = reinterpret_cast<uint8_t*>(sg);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const uint16_t c2 = f32x2_to_e4m3x2(__fdiv_rn(h[i], gmax[i]), __fdiv_rn(h[i + 1], gmax[i + 1]));
          sb[i * 128 + f] = static_cast<uint8_t>(c2 & 0xff);
          sb[(i + 1) * 128 + f] = static_cast<uint8_t>(c2 >> 8);
        }
        named_bar_sync(1 + grp, 128);
        if (has) {
          const int ch = etid & 7;  // 8 x 16 bytes per 128-byte token row
          for (int rr = etid >> 3; rr < rows_here; rr += 16) {
            const uint4 v = *reinterpret_cast<const uint4*>(sb + rr * 128 + ch * 16);
            *reinterpret_cast<uint4*>(out + (size_t)(ti.out_row0 + c0 + rr) * I + ti.m * 128 + ch * 16) = v;
          }
        }
        named_bar_sync(1 + grp, 128);
      } else {
        uint16_t* y = reinterpret_cast<uint16_t*>(out);
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            sg[i * kStgStride + f] = __bfloat16_as_ushort(__float2bfloat16_rn(pass == 0 ? acc_a[i] : acc_b[i]));
          named_bar_sync(1 + grp, 128);
          const int ch = etid & 15;
          const int col = ti.m * 256 + pass * 128 + ch * 8;
          if (has && col < d) {
            for (int rr = etid >> 4; rr < rows_here; rr += 8) {
              const uint4 v = *reinterpret_cast<const uint4*>(sg + rr * kStgStride + ch * 8);
              *reinterpret_cast<uint4*>(y + (size_t)(ti.out_row0 + c0 + rr) * d + col) = v;
            }
          }
          named_bar_sync(1 + grp, 128);
        }
      }
    }
  }
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    for (int s = 0; s < kStages; ++s)
      if (last_round[s] >= 0)
        mbar_wait(&full[s], last_round[s] & 1, zero_flag, status, status + 1, kSiteGemmTeardown, 100000000ull);
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// x [T, d] bf16 -> E4M3 codes + per-1x128 scales (input of the shared experts)
__global__ void __launch_bounds__(128) quant_rows_kernel(const uint4* __restrict__ x, int d, uint8_t* __restrict__ q,
                                                         float* __restrict__ scale) {
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = d / 8;
  for (int v0 = warp * 32; v0 < nvec; v0 += 128) {
    const int v = v0 + lane;
    const bool valid = v < nvec;
    float f[8];
    bf16x8_to_f32(valid ? __ldg(x + (size_t)t * nvec + v) : make_uint4(0, 0, 0, 0), f);
    uint2 c;
    const float sc = quant_tile16(f, c);
    if (valid) {
      *reinterpret_cast<uint2*>(q + (size_t)t * d + (size_t)v * 8) = c;
      if ((lane & 15) == 0) scale[(size_t)t * (d / 128) + (v >> 4)] = sc;
    }
  }
}

}  // namespace

moe_status_t launch_expert_ffn_fp8(const moe_shape_t& s, const void* x_perm, const float* x_perm_scale,
                                   const void* x, const int32_t* perm_token, const int32_t* offsets,
                                   const void* w_gate_up, const float* w_gu_scale, const void* w_down,
                                   const float* w_down_scale, void* y, void* ws, cudaStream_t st,
                                   const WsLayout* layout) {
  const bool gather = perm_token != nullptr;
  const WsLayout L = layout ? *layout : ws_layout(s);
  char* w = static_cast<char*>(ws);
  const int G = s.E + s.S;
  GroupInfo* groups = reinterpret_cast<GroupInfo*>(w + L.sched);
  int* ts_gu = reinterpret_cast<int*>(groups + G);
  int* ts_dn = ts_gu + (G + 1);
  uint8_t* xq = reinterpret_cast<uint8_t*>(w + L.xq);
  float* xq_scale = reinterpret_cast<float*>(w + L.xq_scale);
  uint8_t* hq = reinterpret_cast<uint8_t*>(w + L.h);
  float* h_scale = reinterpret_cast<float*>(w + L.h_scale);
  int* status = ws_status(ws);
  const int Tk = s.T * s.k;
  const int rows = Tk + s.S * s.T;

  schedule_kernel<<<1, 512, 0, st>>>(offsets, s.T, s.k, s.E, s.S, s.I / 128, (s.d + 255) / 256, kChunk, groups,
                                     ts_gu, ts_dn, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (s.S > 0 || gather) {  // E4M3 copy of x: the shared experts' input, and the gather source
    quant_rows_kernel<<<s.T, 128, 0, st>>>(static_cast<const uint4*>(x), s.d, xq, xq_scale);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }

  CUtensorMap m_wgu, m_xp, m_x, m_xg, m_wd, m_h;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (!make_map_3d(&m_wgu, w_gate_up, u8, 1, s.d, 2 * (uint64_t)s.I, G, 128, 128)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_x, xq, u8, 1, s.d, s.T, 128, kBoxRows)) return MOE_ERR_CUDA;
  if (gather) {  // routed rows gathered from the E4M3 copy of x one row at a time
    if (!make_map_2d(&m_xg, xq, u8, 1, s.d, s.T, 128, 1)) return MOE_ERR_CUDA;
    m_xp = m_x;
  } else {
    if (!make_map_2d(&m_xp, x_perm, u8, 1, s.d, Tk, 128, kBoxRows)) return MOE_ERR_CUDA;
    m_xg = m_x;
  }
  if (!make_map_3d(&m_wd, w_down, u8, 1, s.I, s.d, G, 128, 128)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_h, hq, u8, 1, s.I, rows, 128, kBoxRows)) return MOE_ERR_CUDA;

  const int grid = sm_count();
  if (grid <= 0) return MOE_ERR_CUDA;
  auto k_gu = gather ? expert_gemm_fp8_kernel<kGateUp, true> : expert_gemm_fp8_kernel<kGateUp, false>;
  auto k_dn = expert_gemm_fp8_kernel<kDown, false>;
  if (cudaFuncSetAttribute(k_gu, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(k_dn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  k_gu<<<grid, kThreads, kSmemBytes, st>>>(m_wgu, m_xp, m_x, m_xg, groups, ts_gu, G, s.E, s.d, s.I, s.d,
                                           x_perm_scale, xq_scale, w_gu_scale, 2 * s.I, perm_token, s.T, hq, h_scale,
                                           status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  k_dn<<<grid, kThreads, kSmemBytes, st>>>(m_wd, m_h, m_h, m_h, groups, ts_dn, G, s.E, s.I, s.I, s.d, h_scale,
                                           h_scale, w_down_scale, s.d, nullptr, 0, static_cast<uint8_t*>(y), nullptr,
                                           status);
  return cuda_status(cudaGetLastError());
}

}  // namespace moe
