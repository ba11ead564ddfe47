// Grouped SwiGLU expert GEMMs on the tcgen05 tensor cores ("DeepSeek-V3 技术报告要点"
// section 1 (SwiGLU FFN) and section 3 table (expert intermediate 2048);
// "DeepSeek-V3 详解" 2.2 (256 fine-grained routed experts + 1 shared expert)).
//
//   gate/up:  h[r, f] = silu(X[r] . Wg[f]) * (X[r] . Wu[f])   (SiLU*mul fused)
//   down:     y[r, c] = h[r] . Wd[c]
//
// The backward pass reuses the same tiles: "gate/up raw" writes the two
// pre-activations next to h; "input gradient" mode reads the weight operand
// MN-major (the stored W, contracted over its output dimension: dh = dy Wd,
// dx = [da du] [Wg; Wu]), so no transposed weight copy exists; "weight gradient"
// mode reads both operands MN-major from token-row buffers and computes
// dW[g] = B_g^T A_g over the group's own rows (whole 64-row blocks, zero-padded
// by the caller), one output matrix per group.
//
// Every routed expert is a group of rows of x_perm; every shared expert is a
// group over all T rows of x, scheduled in the same persistent launch.
//
// Tile shape ("swap AB"): the MMA's M side carries weight rows (output
// features) and its N side up to 256 tokens of one group, so a group of n
// tokens is padded to a multiple of 16 only.  Two CTAs of a cluster form a pair
// and run M = 256 MMAs (tcgen05 cta_group::2): each CTA stages its own 128
// weight rows and half of the token rows, so a 48 KB stage feeds as much
// tensor work per SM as a 64 KB single-CTA stage would, and four stages fit.
// Each K step issues two MMAs sharing the token operand: gate rows and up rows
// of the same 256 features (the even CTA's TMEM lanes hold features 0-127, the
// odd CTA's 128-255, so one lane holds g and u of one feature), or two
// 256-channel blocks of W_down.  Two FP32 accumulators of 256 columns fill the
// 512 TMEM columns of each CTA.
//
// Warp roles (320 threads per CTA, one CTA per SM, persistent over pair tiles):
//   warp 0      TMA producer of this CTA's operand halves; all loads of a stage
//               complete on the even CTA's barrier.  In the gathering variant
//               (the fused forward) the routed token rows are not read from a
//               permuted copy but straight from x: each lane holds four of the
//               chunk's token indices (from the permutation table) and issues
//               one TMA row gather of those four rows per K block, landing in
//               the same swizzled layout as a box load (the dispatch step of the
//               pages' layer fused into the expert GEMM's operand load);
//   warp 1      TMEM allocation; in the even CTA the single MMA-issuing thread,
//               whose commits are multicast to both CTAs;
//   warps 2-9   epilogue in two groups of four (one TMEM lane quadrant per
//               warp, alternate 32-token chunks per group): tcgen05.ld, SwiGLU,
//               bf16 rounding, transpose through shared memory, coalesced
//               16-byte stores of the token rows.  TMEM is handed back to the
//               MMA thread right after the last TMEM read of a tile.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kStages = 4;
constexpr int kThreads = 320;                  // producer warp, MMA warp, 8 epilogue warps
constexpr int kKStagger = 5;                   // K-block offset between consecutive feature blocks
constexpr uint32_t kATile = 128 * 128;         // 128 weight rows x 128 bytes
constexpr uint32_t kBTile = (kChunkMax / 2) * 128;  // this CTA's half of <= 256 token rows
constexpr uint32_t kBox = kBoxRows * 128;      // one TMA box of token rows
constexpr uint32_t kStage = 2 * kATile + kBTile;  // 48 KB
constexpr int kStgStride = 136;                // staging row stride (bf16), 16-byte multiple
// epilogue staging: one [32][136] tile per group, or (weight gradient) two dense
// [32][128] tiles per group, the sources of its TMA stores
constexpr uint32_t kStgBytes = 2 * 2 * 32 * 128 * 2;
constexpr uint32_t kCtrl = 1024;
constexpr size_t kSmemBytes = 1024 + kStages * kStage + kStgBytes + kCtrl;

// kGateUp     A = [Wg; Wu] of the group's expert, B = token rows (routed: in_row0,
//             shared experts: map_b1), out = h (SwiGLU fused)
// kDown       A = W_down, B = h rows at out_row0, out = y
// kGateUpRaw  as kGateUp, out = FP32 [a | u] (width 2I) and out2 = h (bf16)
// kDgrad      A = W[g] stored [K][M] (map_w [G][K][M], read MN-major), B = token
//             rows at in_row0 (K-major), out = B A (width `d`)
// kWgrad      A = rows [K][M] of one buffer (map_w [1][rows][M], MN-major), B = rows
//             [K][N] of another (map_b0 [rows][N], MN-major), K = the group's 64-row
//             blocks [pad0, pad0 + pad1); out[g] = A^T B: row = M index (512 per tile,
//             `I` rows per group), col = N index (chunks of 256).  A TMEM lane holds
//             one output row, so each thread stages 64 contiguous bytes per chunk.  K is short (one
//             expert's tokens), so the output (the largest write of the backward)
//             leaves through TMA stores (map_xg = the output map) of double-buffered
//             staging tiles, and the epilogue is no longer the long pole.  (A ring of
//             two 512 x 128 accumulators in TMEM, which lets the next tile's MMAs run
//             while one drains, measured slower: it reads every A block twice as often.)
// kDgrad32    as kDgrad, out = FP32 (width `d`), stored straight from registers
enum Mode : int { kGateUp = 0, kDown = 1, kGateUpRaw = 2, kWgrad = 3, kDgrad = 4, kDgrad32 = 5 };

struct TileInfo {
  int g, mp, tok0, n, expert, brow0, out_row0;
  int k0, nk;  // K blocks of the tile: [k0, k0 + nk) (nk < 0: all K / 64)
  bool shared_b;
};

// The group of a role's previous tile.  A role's tiles only grow and consecutive
// ones mostly fall in the same group (hundreds of tiles per expert in the weight
// gradients), so the lookup is skipped then.
struct GroupCursor {
  int g = -1, lo = 0, hi = 0;
  GroupInfo gi;
};

// pair tile -> group, feature-block pair mp, token chunk
__device__ __forceinline__ bool decode_tile(const GroupInfo* __restrict__ groups, const int* __restrict__ ts,
                                            int G, int E, int tile, int mode, TileInfo& ti, GroupCursor& cur) {
  if (cur.g < 0 || tile < cur.lo || tile >= cur.hi) {
    // the largest g with ts[g] <= tile (ts[G] > tile); past the cached group if beyond it
    int lo = cur.g >= 0 && tile >= cur.hi ? cur.g + 1 : 0, hi = G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(ts + mid) <= tile) lo = mid;
      else hi = mid;
    }
    cur.g = lo;
    cur.lo = __ldg(ts + lo);
    cur.hi = __ldg(ts + lo + 1);
    cur.gi = groups[lo];
  }
  const int g = cur.g;
  const GroupInfo& gi = cur.gi;
  if (gi.nchunks <= 0) return false;
  const int local = tile - cur.lo;
  ti.g = g;
  ti.mp = local / gi.nchunks;
  const int c = local - ti.mp * gi.nchunks;
  ti.tok0 = c * gi.csize;
  ti.n = min(gi.csize, gi.n - ti.tok0);
  ti.expert = gi.expert;
  ti.out_row0 = gi.out_row0 + ti.tok0;
  ti.shared_b = (mode == kGateUp || mode == kGateUpRaw) && g >= E;
  ti.brow0 = (mode == kDown ? gi.out_row0 : gi.in_row0) + ti.tok0;
  // K range in 64-element blocks: the whole K, or (weight gradient) the group's own
  ti.k0 = mode == kWgrad ? gi.pad0 : 0;
  ti.nk = mode == kWgrad ? gi.pad1 : -1;
  return ti.n > 0;
}

// GATHER (gate/up only): routed token rows are gathered from x (map_xg: [x_rows, K]
// bf16, box 64 x 1 row) through perm_token instead of read from map_b0.  kWgrad:
// map_xg is the output map ([G][rows][cols], 64-byte swizzle, box 32 x 128).
template <int MODE, bool GATHER>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_b0,
                       const __grid_constant__ CUtensorMap map_b1, const __grid_constant__ CUtensorMap map_xg,
                       const __grid_constant__ CUtensorMap map_wp, int a_pair,
                       const GroupInfo* __restrict__ groups, const int* __restrict__ tile_start, int G, int E, int K,
                       int I, int d, const int32_t* __restrict__ perm_token, int x_rows,
                       uint16_t* __restrict__ out, uint16_t* __restrict__ out2, int* __restrict__ status) {
  static_assert(!GATHER || MODE == kGateUp, "row gather feeds the gate/up GEMM only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint16_t* stg = reinterpret_cast<uint16_t*>(smem + kStages * kStage);
  uint8_t* ctrl = smem + kStages * kStage + kStgBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);  // [kStages], used in the even CTA
  uint64_t* empty = full + kStages;                    // [kStages], both CTAs
  uint64_t* tmem_full = empty + kStages;               // [2] both CTAs
  uint64_t* tmem_empty = tmem_full + 2;                // [2] even CTA: both CTAs' epilogues arrive
  uint64_t* drain = tmem_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 132);
  volatile int* zero_flag = reinterpret_cast<volatile int*>(ctrl + 136);
  int* last_round = reinterpret_cast<int*>(ctrl + 144);  // [kStages]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0 = the CTA that issues the MMAs
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(nclusters_x());
  const int nk_all = K / 64;
  const int total = __ldg(tile_start + G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      last_round[s] = -1;
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 2 * 256);
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
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t full_leader = map_to_rank(smem_u32(full), 0);        // full[0] of the even CTA
  const uint32_t tmem_empty_leader = map_to_rank(smem_u32(tmem_empty), 0);  // + 8 * buffer
  // accumulator buffers in TMEM: one tile uses all 512 columns (the barrier and column
  // arithmetic allows a ring of two 256-column tiles)
  constexpr int kBufs = 1;

  if (warp == 0 && GATHER) {
    const int nk = nk_all;
    // ---------------- producer with row gather (whole warp): lane 0 issues the weight
    // loads (and the shared experts' contiguous token rows), lane q gathers this CTA's
    // token rows 4q .. 4q + 3 of a routed chunk
    uint32_t it = 0;
    bool ok = true;
    GroupCursor cur;
    for (int tile = pair; tile < total && ok; tile += npairs) {
      TileInfo ti;
      if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti, cur)) continue;
      const int nm = (ti.n + 15) & ~15;
      const int half = nm / 2;  // token rows per CTA (multiple of 8)
      const bool gat = !ti.shared_b;
      // shared experts' contiguous rows: one 128-row box
      const uint32_t b_mine = gat ? half * 128u : kBTile;
      const uint32_t bytes_pair = 2 * (2 * kATile + b_mine);  // both CTAs (same row count)
      const int a0_row = ti.mp * 256 + rank * 128;  // gate rows of this CTA's 128 features
      const int a1_row = I + a0_row;                // up rows of the same features
      const int brow = ti.brow0 + rank * half;
      const bool my_rows = gat && 4 * lane < half;
      int tk[4] = {0, 0, 0, 0};
      if (my_rows) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int row = rank * half + 4 * lane + u;  // padding rows repeat the chunk's first token
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
        const uint32_t fb = full_leader + s * 8;
        const int kq = (kb + ti.mp * kKStagger) % nk;
        if (lane == 0) {
          if (rank == 0) mbar_arrive_expect_tx(&full[s], bytes_pair);
          if (a_pair) {
            tma_load_4d_pair(st, &map_wp, fb, kq * 64, a0_row, 0, ti.expert);
          } else {
            tma_load_3d_pair(st, &map_w, fb, kq * 64, a0_row, ti.expert);
            tma_load_3d_pair(st + kATile, &map_w, fb, kq * 64, a1_row, ti.expert);
          }
          if (!gat) tma_load_2d_pair(st + 2 * kATile, &map_b1, fb, kq * 64, brow);
          last_round[s] = r;
        }
        if (my_rows)
          tma_gather4_pair(st + 2 * kATile + lane * 512, &map_xg, fb, kq * 64, tk[0], tk[1], tk[2], tk[3]);
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: this CTA's weight rows and half of the token rows
      uint32_t it = 0;
      bool ok = true;
      GroupCursor cur;
      for (int tile = pair; tile < total && ok; tile += npairs) {
        TileInfo ti;
        if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti, cur)) continue;
        const int nk = ti.nk >= 0 ? ti.nk : nk_all;
        const int nm = (ti.n + 15) & ~15;
        const int half = nm / 2;  // token rows per CTA (multiple of 8)
        // token operand: one 128-row K-major box (forward), 32-row K-major boxes, or (weight
        // gradient) 64-column MN-major boxes
        constexpr bool kFwd = MODE == kGateUp || MODE == kDown;
        const int nbox_mine = kFwd ? 1 : MODE == kWgrad ? half / 64 : (half + kBoxRows - 1) / kBoxRows;
        const uint32_t bytes_pair =
            2 * (2 * kATile + (kFwd ? kBTile : nbox_mine * (MODE == kWgrad ? 8192u : kBox)));
        int a0_row, a1_row;
        if (MODE == kGateUp || MODE == kGateUpRaw) {
          a0_row = ti.mp * 256 + rank * 128;        // gate rows of this CTA's 128 features
          a1_row = I + ti.mp * 256 + rank * 128;    // up rows of the same features
        } else {
          a0_row = ti.mp * 512 + rank * 128;        // channel block 0 of the pair (256 channels)
          a1_row = ti.mp * 512 + 256 + rank * 128;  // channel block 1
        }
        const CUtensorMap* mb = ti.shared_b ? &map_b1 : &map_b0;
        const int brow = ti.brow0 + rank * half;
        const int wexp = MODE == kWgrad ? 0 : ti.expert;  // weight gradient: A is one buffer
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages, r = it / kStages;
          if (!mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, status, status + 1, kSiteGemmProducer)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * kStage;
          const uint32_t fb = full_leader + s * 8;
          const int kq = ti.k0 + (kb + ti.mp * kKStagger) % nk;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], bytes_pair);
          if (MODE == kDgrad || MODE == kDgrad32 || MODE == kWgrad) {
            // MN-major A: two 64-feature x 64-k boxes per 128 rows (k rows of 128 bytes)
            tma_load_3d_pair(st, &map_w, fb, a0_row, kq * 64, wexp);
            tma_load_3d_pair(st + 8192, &map_w, fb, a0_row + 64, kq * 64, wexp);
            tma_load_3d_pair(st + kATile, &map_w, fb, a1_row, kq * 64, wexp);
            tma_load_3d_pair(st + kATile + 8192, &map_w, fb, a1_row + 64, kq * 64, wexp);
          } else if (kFwd && a_pair == 1) {  // gate and up blocks: {K, I rows, gate/up, expert}
            tma_load_4d_pair(st, &map_wp, fb, kq * 64, a0_row, 0, wexp);
          } else if (kFwd && a_pair == 2) {  // channel blocks 0 and 1: {K, 256 rows, block, tile, expert}
            tma_load_5d_pair(st, &map_wp, fb, kq * 64, static_cast<int>(rank) * 128, 0, ti.mp, wexp);
          } else {
            tma_load_3d_pair(st, &map_w, fb, kq * 64, a0_row, wexp);
            tma_load_3d_pair(st + kATile, &map_w, fb, kq * 64, a1_row, wexp);
          }
          if (kFwd) {
            tma_load_2d_pair(st + 2 * kATile, mb, fb, kq * 64, brow);
          } else if (MODE == kWgrad) {
            for (int b = 0; b < nbox_mine; ++b)
              tma_load_2d_pair(st + 2 * kATile + b * 8192, mb, fb, brow + b * 64, kq * 64);
          } else {
            for (int b = 0; b < nbox_mine; ++b)
              tma_load_2d_pair(st + 2 * kATile + b * kBox, mb, fb, kq * 64, brow + b * kBoxRows);
          }
          last_round[s] = r;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA only)
      uint32_t it = 0, tl = 0;
      bool ok = true;
      GroupCursor cur;
      for (int tile = pair; tile < total && ok; tile += npairs) {
        TileInfo ti;
        if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti, cur)) continue;
        const int nm = (ti.n + 15) & ~15;
        // MN-major operands: transpose bits 15 (A) and 16 (B) of the instruction descriptor
        const uint32_t idesc = idesc_bf16(256, nm) | (MODE == kDgrad || MODE == kDgrad32 || MODE == kWgrad ? 1u << 15 : 0u) |
                               (MODE == kWgrad ? 1u << 16 : 0u);
        const int nk = ti.nk >= 0 ? ti.nk : nk_all;
        const uint32_t buf = tl % kBufs, use = tl / kBufs;  // accumulator buffer, its earlier uses
        if (!mbar_wait(&tmem_empty[buf], (use & 1) ^ 1, abort_flag, status, status + 1, kSiteGemmMma)) break;
        tc_fence_after();
        const uint32_t acc0 = tmem + buf * 256;                             // feature block 0
        const uint32_t acc1 = acc0 + (kBufs == 1 ? 256 : 128);              // feature block 1
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages, r = it / kStages;
          if (!mbar_wait(&full[s], r & 1, abort_flag, status, status + 1, kSiteGemmMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + s * kStage);
          const uint32_t a1 = a0 + kATile;
          const uint32_t b = a0 + 2 * kATile;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // K-major: 16 k = 32 bytes along the row; MN-major: 16 k = 16 rows of 128 bytes
            const uint64_t bd = MODE == kWgrad ? sdesc_mn128(b + kk * 2048) : sdesc_k128(b + kk * 32);
            const bool amn = MODE == kDgrad || MODE == kDgrad32 || MODE == kWgrad;
            const uint64_t ad0 = amn ? sdesc_mn128(a0 + kk * 2048) : sdesc_k128(a0 + kk * 32);
            const uint64_t ad1 = amn ? sdesc_mn128(a1 + kk * 2048) : sdesc_k128(a1 + kk * 32);
            const uint32_t acc = (kb | kk) != 0;
            mma_bf16_pair(acc0, ad0, bd, idesc, acc);
            mma_bf16_pair(acc1, ad1, bd, idesc, acc);
          }
          mma_commit_pair_mc(&empty[s], 0x3);  // stage s free in both CTAs
        }
        if (!ok) break;
        mma_commit_pair_mc(&tmem_full[buf], 0x3);
        ++tl;
      }
      mma_commit_pair(drain);
      mbar_wait(drain, 0, zero_flag, status, status + 1, kSiteGemmTeardown, 100000000ull);
    }
  } else {
    // ---------------- epilogue: two groups of four warps (warps 2-5 and 6-9); warp w
    // reads TMEM lane quadrant w % 4, group g takes the 32-token column chunks
    // g, g + 2, g + 4, ... of every tile
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int f = q * 32 + lane;
    const int etid = (threadIdx.x - 64) & 127;
    uint16_t* sg = stg + grp * (32 * kStgStride);
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tl = 0;
    uint32_t spass = 0;  // weight gradient: staged passes of this group (buffer = spass & 1)
    GroupCursor cur;
    for (int tile = pair; tile < total; tile += npairs) {
      TileInfo ti;
      if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti, cur)) continue;
      const uint32_t buf = tl % kBufs, use = tl / kBufs;
      if (!mbar_wait(&tmem_full[buf], use & 1, abort_flag, status, status + 1, kSiteGemmEpi)) break;
      tc_fence_after();
      const uint32_t empty_bar = tmem_empty_leader + 8 * buf;
      const int nm = (ti.n + 15) & ~15;
      const int nchunk = (nm + 31) / 32;
      const int mine = nchunk > grp ? (nchunk - grp + 1) / 2 : 0;
      if (mine == 0) {
        tc_fence_before();
        mbar_arrive_remote(empty_bar);
      }
      for (int ci = 0; ci < mine; ++ci) {
        const int c0 = (grp + 2 * ci) * 32;
        uint32_t ra[32], rb[32];
        tmem_ld32(tmem + lane_base + buf * 256 + c0, ra);
        tmem_ld32(tmem + lane_base + buf * 256 + (kBufs == 1 ? 256 : 128) + c0, rb);
        tmem_ld_wait();
        if (ci == mine - 1) {  // this group is done with TMEM for this tile
          tc_fence_before();
          mbar_arrive_remote(empty_bar);
        }
        const int rows_here = min(32, ti.n - c0);
        const bool zero = MODE == kWgrad && ti.nk == 0;  // a group without tokens: dW = 0
#pragma unroll
        for (int pass = 0; pass < (MODE == kGateUp ? 1 : MODE == kGateUpRaw ? 3 : 2); ++pass) {
          if ((MODE == kGateUpRaw && pass < 2) || MODE == kDgrad32) {
            // FP32 rows straight from registers (a warp writes 32 consecutive features,
            // 128 bytes, of one row per store): a (pass 0) and u (pass 1) of the raw
            // gate/up into [a | u] of width 2I, or the two 256-feature blocks of kDgrad32
            const int F = MODE == kDgrad32 ? ti.mp * 512 + pass * 256 + rank * 128 + f
                                           : ti.mp * 256 + rank * 128 + f;
            const int lim = MODE == kDgrad32 ? d : I;
            const int wo = MODE == kDgrad32 ? d : 2 * I;
            if (F < lim) {
              float* o = reinterpret_cast<float*>(out) + (size_t)(ti.out_row0 + c0) * wo +
                         (MODE == kDgrad32 ? 0 : pass * I) + F;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < rows_here) o[(size_t)i * wo] = __uint_as_float(pass == 0 ? ra[i] : rb[i]);
            }
            continue;
          }
          if (MODE == kWgrad) {
            // this thread's output row (TMEM lane f), output columns tok0 + c0 .. + 31:
            // 64 bytes staged in a [128 rows][32 columns] tile with the 64-byte swizzle
            // (16-byte chunk c of row f at c ^ ((f >> 1) & 3)), then one TMA store
            uint8_t* sb = reinterpret_cast<uint8_t*>(stg) + (grp * 2 + (spass & 1)) * 8192;
            if (etid == 0) bulk_wait_read<1>();  // the store that used this buffer has read it
            named_bar_sync(1 + grp, 128);
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[j] = zero ? 0u
                           : pack_bf16x2(__uint_as_float(pass == 0 ? ra[2 * j] : rb[2 * j]),
                                         __uint_as_float(pass == 0 ? ra[2 * j + 1] : rb[2 * j + 1]));
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(sb + f * 64 + ((c ^ ((f >> 1) & 3)) * 16)) =
                  make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            fence_proxy_async_smem();
            named_bar_sync(1 + grp, 128);
            if (etid == 0) {
              const int mrow = ti.mp * 512 + pass * 256 + rank * 128;
              if (mrow < I) tma_store_3d(&map_xg, sb, ti.tok0 + c0, mrow, ti.g);
              bulk_commit();  // one group per pass, empty when nothing was stored
            }
            ++spass;
            continue;
          }
          if (MODE == kGateUp || (MODE == kGateUpRaw && pass == 2)) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = __uint_as_float(ra[i]);
              const float u = __uint_as_float(rb[i]);
              const float h = __fdividef(g, 1.0f + __expf(-g)) * u;  // silu(g) * u
              sg[i * kStgStride + f] = __bfloat16_as_ushort(__float2bfloat16_rn(h));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              sg[i * kStgStride + f] = __bfloat16_as_ushort(
                  __float2bfloat16_rn(zero ? 0.0f : __uint_as_float(pass == 0 ? ra[i] : rb[i])));
          }
          named_bar_sync(1 + grp, 128);
          // 128 features x 2 bytes = 16 x 16-byte pieces per token row
          const int ch = etid & 15;
          int col, width;
          bool in_range;
          uint16_t* dst = out;
          if (MODE == kGateUp || MODE == kGateUpRaw) {
            // raw: pass 0 a, pass 1 u (rows [a | u] of width 2I), pass 2 h into out2
            const int feat = ti.mp * 256 + rank * 128 + ch * 8;
            const bool raw_au = MODE == kGateUpRaw && pass < 2;
            col = (raw_au ? pass * I : 0) + feat;
            width = raw_au ? 2 * I : I;
            if (MODE == kGateUpRaw && pass == 2) dst = out2;
            in_range = feat < I;
          } else {
            col = ti.mp * 512 + pass * 256 + rank * 128 + ch * 8;
            width = d;
            in_range = col < d;
          }
          if (in_range) {
            for (int rr = etid >> 4; rr < rows_here; rr += 8) {
              const uint4 v = *reinterpret_cast<const uint4*>(sg + rr * kStgStride + ch * 8);
              *reinterpret_cast<uint4*>(dst + (size_t)(ti.out_row0 + c0 + rr) * width + col) = v;
            }
          }
          named_bar_sync(1 + grp, 128);
        }
      }
      ++tl;
    }
    if (MODE == kWgrad && etid == 0) bulk_wait_all();  // staging is read and the output written
  }
  __syncthreads();
  if (warp == 0 && lane == 0 && *abort_flag) {
    // this CTA's own loads completed on the even CTA's barriers; wait there (bounded)
    for (int s = 0; s < kStages; ++s)
      if (last_round[s] >= 0 && rank == 0)
        mbar_wait(&full[s], last_round[s] & 1, zero_flag, status, status + 1, kSiteGemmTeardown, 100000000ull);
  }
  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace

// One block: per group token count, chunking and the prefix sums of tiles.
__global__ void schedule_kernel(const int32_t* __restrict__ offsets, int T, int k, int E, int S, int m_gu, int m_dn,
                                int chunk_max,
                                GroupInfo* __restrict__ groups, int* __restrict__ ts_gu, int* __restrict__ ts_dn,
                                int* __restrict__ status) {
  __shared__ int sg[2][512], sd[2][512];
  __shared__ int bad;
  const int G = E + S;
  const int g = threadIdx.x;
  if (g == 0) bad = 0;
  __syncthreads();
  int tg = 0, td = 0;
  if (g < G) {
    GroupInfo gi{};
    const int Tk = T * k;
    if (g < E) {
      const int lo = offsets[g], hi = offsets[g + 1];
      if (lo < 0 || hi < lo || hi > Tk || (g == E - 1 && hi != Tk) || (g == 0 && lo != 0)) {
        bad = 1;
        gi.n = 0;
      } else {
        gi.n = hi - lo;
      }
      gi.in_row0 = lo;
      gi.out_row0 = lo;
      gi.expert = g;
    } else {
      gi.n = T;
      gi.in_row0 = 0;
      gi.out_row0 = Tk + (g - E) * T;
      gi.expert = g;
    }
    gi.nchunks = (gi.n + chunk_max - 1) / chunk_max;
    gi.csize = gi.nchunks ? (((gi.n + gi.nchunks - 1) / gi.nchunks + 15) & ~15) : 16;
    groups[g] = gi;
    tg = gi.nchunks * m_gu;
    td = gi.nchunks * m_dn;
  }
  // inclusive scan (Hillis-Steele) over up to 512 groups
  int cur = 0;
  sg[0][g] = tg;
  sd[0][g] = td;
  __syncthreads();
  for (int off = 1; off < 512; off <<= 1) {
    const int a = sg[cur][g] + (g >= off ? sg[cur][g - off] : 0);
    const int b = sd[cur][g] + (g >= off ? sd[cur][g - off] : 0);
    sg[cur ^ 1][g] = a;
    sd[cur ^ 1][g] = b;
    cur ^= 1;
    __syncthreads();
  }
  if (bad) {
    if (g == 0) set_error(status, status + 1, MOE_ERR_DEVICE, kSiteSchedule);
    if (g <= G) {
      ts_gu[g] = 0;
      ts_dn[g] = 0;
    }
    return;
  }
  if (g < G) {
    ts_gu[g + 1] = sg[cur][g];
    ts_dn[g + 1] = sd[cur][g];
  }
  if (g == 0) {
    ts_gu[0] = 0;
    ts_dn[0] = 0;
  }
}


moe_status_t launch_expert_ffn(const moe_shape_t& s, const void* x_perm, const float* x_perm_scale, const void* x,
                               const int32_t* perm_token, const int32_t* offsets, const void* w_gate_up,
                               const float* w_gu_scale, const void* w_down, const float* w_down_scale, void* y,
                               void* ws, cudaStream_t st, const WsLayout* layout) {
  if (s.T == 0) return MOE_OK;
  if (s.dtype == MOE_FP8_E4M3)
    return launch_expert_ffn_fp8(s, x_perm, x_perm_scale, x, perm_token, offsets, w_gate_up, w_gu_scale, w_down,
                                 w_down_scale, y, ws, st, layout);
  if (s.dtype == MOE_FP8_E4M3_POW2) {
    if (perm_token) return MOE_ERR_UNSUPPORTED;  // whole-tile loads of the permuted copy only
    return launch_expert_ffn_mx(s, x_perm, x_perm_scale, x, offsets, w_gate_up, w_gu_scale, w_down, w_down_scale,
                                y, ws, st, layout);
  }
  const bool gather = perm_token != nullptr;
  const WsLayout L = layout ? *layout : ws_layout(s);
  char* w = static_cast<char*>(ws);
  const int G = s.E + s.S;
  GroupInfo* groups = reinterpret_cast<GroupInfo*>(w + L.sched);
  int* ts_gu = reinterpret_cast<int*>(groups + G);
  int* ts_dn = ts_gu + (G + 1);
  uint16_t* h = reinterpret_cast<uint16_t*>(w + L.h);
  int* status = ws_status(ws);
  const int Tk = s.T * s.k;
  const int rows = Tk + s.S * s.T;
  const int m_gu = (s.I + 255) / 256;  // feature-block pairs
  const int m_dn = (s.d + 511) / 512;

  schedule_kernel<<<1, 512, 0, st>>>(offsets, s.T, s.k, s.E, s.S, m_gu, m_dn, kChunkMax, groups, ts_gu, ts_dn,
                                     status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  CUtensorMap m_wgu, m_wgu_p, m_xp, m_x, m_xg, m_wd, m_wd_p, m_h;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map_3d(&m_wgu, w_gate_up, bf, 2, s.d, 2 * (uint64_t)s.I, G, 64, 128)) return MOE_ERR_CUDA;
  // gate and up rows of a tile in one load: the up block is I rows after the gate block
  if (!make_map_pair_rows(&m_wgu_p, w_gate_up, bf, 2, s.d, s.I, s.I, G, 2 * (uint64_t)s.I, 64))
    return MOE_ERR_CUDA;
  // token rows: one 128-row box per stage (this CTA's half of <= 256 rows)
  if (!make_map_2d(&m_x, x, bf, 2, s.d, s.T, 64, 128)) return MOE_ERR_CUDA;
  if (gather) {  // routed rows gathered from x one row at a time; no permuted copy
    if (!make_map_2d(&m_xg, x, bf, 2, s.d, s.T, 64, 1)) return MOE_ERR_CUDA;
    m_xp = m_x;
  } else {
    if (!make_map_2d(&m_xp, x_perm, bf, 2, s.d, Tk, 64, 128)) return MOE_ERR_CUDA;
    m_xg = m_x;
  }
  if (!make_map_3d(&m_wd, w_down, bf, 2, s.I, s.d, G, 64, 128)) return MOE_ERR_CUDA;
  // the two channel blocks of a 512-channel tile in one load (when d is a multiple of 512)
  const int dn_pair = s.d % 512 == 0 ? 2 : 0;
  m_wd_p = m_wd;
  if (dn_pair && !make_map_pair_rows5(&m_wd_p, w_down, bf, 2, s.I, 256, 256, s.d / 512, 512, G, s.d, 64))
    return MOE_ERR_CUDA;
  if (!make_map_2d(&m_h, h, bf, 2, s.I, rows, 64, 128)) return MOE_ERR_CUDA;

  auto k_gu = gather ? expert_gemm_kernel<kGateUp, true> : expert_gemm_kernel<kGateUp, false>;
  auto k_dn = expert_gemm_kernel<kDown, false>;
  if (cudaFuncSetAttribute(k_gu, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(k_dn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int grid = pair_grid((const void*)k_gu, kThreads, kSmemBytes);
  if (grid <= 0) return MOE_ERR_CUDA;
  k_gu<<<grid, kThreads, kSmemBytes, st>>>(m_wgu, m_xp, m_x, m_xg, m_wgu_p, 1, groups, ts_gu, G, s.E, s.d, s.I, s.d,
                                          perm_token, s.T, h, nullptr, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  k_dn<<<grid, kThreads, kSmemBytes, st>>>(m_wd, m_h, m_h, m_h, m_wd_p, dn_pair, groups, ts_dn, G, s.E, s.I, s.I,
                                          s.d, nullptr, 0, static_cast<uint16_t*>(y), nullptr, status);
  return cuda_status(cudaGetLastError());
}

moe_status_t launch_gemm_bwd(GemmMode mode, const CUtensorMap& map_w, const CUtensorMap& map_b0,
                             const CUtensorMap& map_b1, const GroupInfo* groups, const int* tile_start, int G, int E,
                             int K, int I, int width, void* out, void* out2, int* status, cudaStream_t st,
                             const CUtensorMap* map_out) {
  if (mode == GemmMode::kWgrad && !map_out) return MOE_ERR_INVALID_ARG;
  const void* fn;
  switch (mode) {
    case GemmMode::kGateUpRaw: fn = (const void*)expert_gemm_kernel<kGateUpRaw, false>; break;
    case GemmMode::kDgrad: fn = (const void*)expert_gemm_kernel<kDgrad, false>; break;
    case GemmMode::kWgrad: fn = (const void*)expert_gemm_kernel<kWgrad, false>; break;
    case GemmMode::kDgrad32: fn = (const void*)expert_gemm_kernel<kDgrad32, false>; break;
    default: return MOE_ERR_INVALID_ARG;
  }
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int grid = pair_grid(fn, kThreads, kSmemBytes);
  if (grid <= 0) return MOE_ERR_CUDA;
  CUtensorMap mw = map_w, m0 = map_b0, m1 = map_b1, mg = map_out ? *map_out : map_b0, mwp = map_w;
  int a_pair = 0;  // the backward modes load their A blocks one at a time
  const int32_t* no_perm = nullptr;
  int x_rows = 0;
  uint16_t* o = static_cast<uint16_t*>(out);
  uint16_t* o2 = static_cast<uint16_t*>(out2);
  void* args[] = {&mw, &m0, &m1, &mg, &mwp, &a_pair, &groups, &tile_start, &G, &E, &K, &I, &width, &no_perm, &x_rows,
                  &o, &o2, &status};
  return cuda_status(cudaLaunchKernel(fn, dim3(grid), dim3(kThreads), args, kSmemBytes, st));
}

}  // namespace moe
