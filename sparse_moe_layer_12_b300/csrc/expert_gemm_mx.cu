// FP8 (E4M3) grouped SwiGLU expert GEMMs with power-of-two block scales, applied by
// the tensor core ("DeepSeek-V3 详解" 4.2: an independent scale per 1x128 activation
// tile and per 128x128 weight block; 4.3: FP32 accumulation).  The pages fix the
// granularity of the scales, not their number format; with every scale a power of
// two (the smallest 2^e with amax <= 448 * 2^e) the scale of a 1x128 / 128x128 block
// is one UE8M0 byte, and the block-scaled MMA (tcgen05 kind::mxf8f6f4) multiplies
// each 32-wide K slice of A and B by its row's scale before accumulating in FP32 in
// TMEM -- no per-K-block promotion through registers:
//
//   y[f, t] = sum_k  2^ea[f / 128, k / 128] q_w[f, k] * 2^eb[t, k / 128] q_a[t, k]
//
// Tile: CTA pairs (cta_group::2), M = 256 weight rows (each CTA 128: gate and up rows
// of the same 128 features, or two 128-channel blocks of W_down, as two MMAs sharing
// the token operand), N <= 224 tokens of one group, K block = 128 bytes = 4 MMAs of
// K = 32 with scale-factor ids 0..3.  TMEM (512 columns): two 224-column FP32
// accumulators and a ring of four 16-column scale slots, one per operand stage (A gate
// / first block 4, A up / second block 4, B tokens 8: two 128-row chunks).
//
// The scales travel with the operands: for every K block the producer warp writes the
// stage's 2 KB scale tile into shared memory beside the TMA data -- the UE8M0 bytes
// (the exponent field of the FP32 power-of-two scale) of the tile's two weight blocks
// and of its tokens, in the 32 x 16-byte chunk layout the MMA reads (line r holds rows
// r, r + 32, r + 64, r + 96 of a 128-row chunk, four bytes each, one per K slice) --
// and the MMA thread copies it into the stage's TMEM slot with tcgen05.cp (each CTA's
// own shared memory into its own TMEM) right before the MMAs that read it: the copy
// and the MMAs run in issue order, and the slot is free once the operand stage is.
//
// Warps: 0 producer (lane 0 issues the TMA loads, all lanes write the scale tile);
// 1 MMA issuer (even CTA); 2-9 epilogue in two groups of four (alternate 32-token
// column chunks).  The gate/up epilogue computes h = silu(g) * u and quantises it per
// token per 128 features (this CTA's 128 features: one 1x128 tile along I) to E4M3 with
// a power-of-two scale, also writing the scale's byte for the down GEMM; the down
// epilogue writes bf16 rows of y.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kStages = 4;
constexpr int kChunk = kChunkMxMax;           // tokens per tile (N)
constexpr int kMine = kChunk / 64;            // 32-column chunks per epilogue group, at most
static_assert((kChunk + 31) / 32 <= 2 * kMine, "each epilogue group holds all of its column chunks");
constexpr int kProducers = 2;                 // producer warps: 0 and 10 .. 8 + kProducers (4 measured slower)
constexpr int kThreads = 32 * (9 + kProducers);  // + MMA warp 1 and epilogue warps 2-9
static_assert(kStages % kProducers == 0, "a producer warp owns whole operand stages");
constexpr int kKStagger = 5;                  // K-block offset between consecutive feature blocks
constexpr uint32_t kATile = 128 * 128;        // 128 weight rows x 128 K bytes
constexpr int kBRows = kChunk / 2;            // this CTA's half of the tile's token rows
constexpr uint32_t kBTile = kBRows * 128;     // one kBRows-row box
constexpr uint32_t kSfTile = 2048;            // scale tile: A gate, A up, B chunk 0, B chunk 1 (512 B each)
constexpr uint32_t kStage = 2 * kATile + kBTile + kSfTile;  // 46 KB
constexpr int kStgStride = 136;               // bf16 staging row stride (elements)
constexpr uint32_t kStgBytes = 2 * 32 * kStgStride * 2;  // one [32][136] bf16 tile per epilogue group
constexpr uint32_t kCtrl = 2048;
constexpr size_t kSmemBytes = 1024 + kStages * kStage + kStgBytes + kCtrl;
constexpr uint32_t kAcc1 = kChunk;            // TMEM column of the second accumulator
constexpr uint32_t kSfBase = 2 * kChunk;      // TMEM column of scale slot 0
constexpr uint32_t kSfSlot = 16;              // columns per scale slot
static_assert(kSfBase + kStages * kSfSlot <= 512, "accumulators and scale slots fit TMEM");
static_assert(kChunk % 16 == 0 && kChunk / 2 <= 128, "token rows fit the 128-row B box");
static_assert(kChunk <= 256, "two 128-row chunks of token scales");
static_assert(kStage % 1024 == 0, "stages stay 1024-aligned for the 128-byte swizzle");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// No-swizzle shared-memory descriptor of a 32 x 16-byte scale tile (8-row x 16-byte core
// matrices 128 bytes apart) for tcgen05.cp.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 16;
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// 32 TMEM lanes x 128 bits from a 32 x 16-byte shared tile, copied into all four lane
// quadrants, in both CTAs of the pair (each from its own shared memory).
__device__ __forceinline__ void tmem_cp_sf_pair(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}

enum Mode : int { kGateUp = 0, kDown = 1 };

struct TileInfo {
  int g, mp, tok0, n, expert, brow0, out_row0;
  bool shared_b;
};

struct GroupCursor {
  int g = -1, lo = 0, hi = 0;
  GroupInfo gi;
};

__device__ __forceinline__ bool decode_tile(const GroupInfo* __restrict__ groups, const int* __restrict__ ts,
                                            int G, int E, int tile, int mode, TileInfo& ti, GroupCursor& cur) {
  if (cur.g < 0 || tile < cur.lo || tile >= cur.hi) {
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
  const GroupInfo& gi = cur.gi;
  if (gi.nchunks <= 0) return false;
  const int local = tile - cur.lo;
  ti.g = cur.g;
  ti.mp = local / gi.nchunks;
  const int c = local - ti.mp * gi.nchunks;
  ti.tok0 = c * gi.csize;
  ti.n = min(gi.csize, gi.n - ti.tok0);
  ti.expert = gi.expert;
  ti.out_row0 = gi.out_row0 + ti.tok0;
  ti.shared_b = mode == kGateUp && cur.g >= E;
  ti.brow0 = (mode == kDown ? gi.out_row0 : gi.in_row0) + ti.tok0;
  return ti.n > 0;
}

// Weight rows of this CTA's two A operands in a tile.
__device__ __forceinline__ void a_rows(int mode, int mp, uint32_t rank, int I, int& a0, int& a1) {
  if (mode == kGateUp) {
    a0 = mp * 256 + static_cast<int>(rank) * 128;  // gate rows of this CTA's 128 features
    a1 = I + a0;                                    // up rows of the same features
  } else {
    a0 = mp * 512 + static_cast<int>(rank) * 128;   // channel block 0 of the pair
    a1 = a0 + 256;                                  // channel block 1
  }
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    expert_gemm_mx_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_wp,
                          int a_pair, const __grid_constant__ CUtensorMap map_b0,
                          const __grid_constant__ CUtensorMap map_b1, const GroupInfo* __restrict__ groups,
                          const int* __restrict__ tile_start, int G, int E, int K, int I, int d,
                          const uint8_t* __restrict__ sb0, int sb0_rows, const uint8_t* __restrict__ sb1,
                          int sb1_rows, const float* __restrict__ sw, int w_rows, uint8_t* __restrict__ out,
                          float* __restrict__ out_scale, uint8_t* __restrict__ out_sb, int out_rows,
                          int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint16_t* stg = reinterpret_cast<uint16_t*>(smem + kStages * kStage);
  uint8_t* ctrl = smem + kStages * kStage + kStgBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);  // [kStages], used in the even CTA
  uint64_t* empty = full + kStages;                    // [kStages], both CTAs
  uint64_t* tmem_full = empty + kStages;               // both CTAs
  uint64_t* tmem_empty = tmem_full + 1;                // even CTA: both CTAs' epilogues arrive
  uint64_t* drain = tmem_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl + 260);
  volatile int* zero_flag = reinterpret_cast<volatile int*>(ctrl + 264);
  int* last_round = reinterpret_cast<int*>(ctrl + 272);  // [kStages]
  float* colmax = reinterpret_cast<float*>(ctrl + 512);  // [2 groups][128]
  // outcome of an epilogue group's bounded wait, published by the one thread that waited,
  // so that the group's four warps go on or stop together (double-buffered by iteration)
  volatile int* epi_ok = reinterpret_cast<volatile int*>(ctrl + 296);  // [2 groups][2]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int pair = static_cast<int>(cluster_id_x());
  const int npairs = static_cast<int>(nclusters_x());
  const int nk = K / 128;
  const int total = __ldg(tile_start + G);
  const int wblk = w_rows / 128;  // 128-row weight blocks per expert

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 2);  // the even CTA's expect_tx arrival + the odd CTA's scale-tile arrival
      mbar_init(&empty[s], 1);
      last_round[s] = -1;
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 2 * 256);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *zero_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(a_pair ? &map_wp : &map_w);
    tma_prefetch_desc(&map_b0);
    tma_prefetch_desc(&map_b1);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);
  tc_fence_before();
  cluster_sync_all();  // barriers initialised and TMEM allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t full_leader = map_to_rank(smem_u32(full), 0);
  const uint32_t tmem_empty_leader = map_to_rank(smem_u32(tmem_empty), 0);

  if (warp == 0 || warp >= 10) {
    // ---------------- producer warps: producer p (warp 0, then warps 10, 11, ...) fills the
    // operand stages s with s % kProducers = p, i.e. the K blocks whose running count is p
    // modulo kProducers; lane 0 issues the TMA loads of this CTA's 2 x 128 weight rows and
    // half of the token rows, every lane writes its line of the stage's scale tile.  Each
    // warp reads the scales of its own K blocks two of them ahead.
    const uint32_t pw = warp == 0 ? 0u : static_cast<uint32_t>(warp - 9);
    uint32_t it = 0;  // running K-block count over the tiles (both warps count every block)
    bool ok = true;
    GroupCursor cur;
    for (int tile = pair; tile < total && ok; tile += npairs) {
      TileInfo ti;
      if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti, cur)) continue;
      const int half = ((ti.n + 15) & ~15) / 2;  // token rows per CTA (multiple of 8)
      const uint32_t bytes_pair = 2 * (2 * kATile + kBTile);  // both CTAs: two A blocks, one B box
      int a0, a1;
      a_rows(MODE, ti.mp, rank, I, a0, a1);
      const CUtensorMap* mb = ti.shared_b ? &map_b1 : &map_b0;
      const int brow = ti.brow0 + static_cast<int>(rank) * half;
      const int wb0 = min(a0 / 128, wblk - 1), wb1 = min(a1 / 128, wblk - 1);
      const float* w0 = sw + ((size_t)ti.expert * wblk + wb0) * nk;
      const float* w1 = sw + ((size_t)ti.expert * wblk + wb1) * nk;
      // the tokens' UE8M0 bytes, K-block major: plane kq holds every row's byte of K
      // block kq, so a warp's 32 lanes read 32 consecutive bytes
      const uint8_t* sb = ti.shared_b ? sb1 : sb0;
      const size_t plane = static_cast<size_t>(ti.shared_b ? sb1_rows : sb0_rows);
      int trow[8];  // this lane's tokens: n = lane + 32 c (+ 128 for the second chunk)
      bool live[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int n = lane + 32 * (j & 3) + 128 * (j >> 2);
        live[j] = n < ti.n;
        trow[j] = ti.brow0 + (live[j] ? n : 0);
      }
      // raw scales of two K blocks in flight, one register set for even and one for odd
      // K blocks: a block's loads are issued two blocks before the shared-memory stores
      // that consume them, and nothing else reads the registers in between
      float ew0 = 1.0f, ew1 = 1.0f, ow0 = 1.0f, ow1 = 1.0f;
      uint32_t et[8], ot[8];
      auto load_scales = [&](int kb, float& w0v, float& w1v, uint32_t (&tv)[8]) {
        const int kq = (kb + ti.mp * kKStagger) % nk;
        w0v = __ldg(w0 + kq);
        w1v = __ldg(w1 + kq);
#pragma unroll
        for (int j = 0; j < 8; ++j) tv[j] = live[j] ? static_cast<uint32_t>(__ldg(sb + (size_t)kq * plane + trow[j])) : 127u;
      };
      // one K block: wait for the stage, write this lane's line of its scale tile, issue the loads
      auto stage = [&](int kb, uint32_t itk, float w0v, float w1v, const uint32_t (&tv)[8]) -> bool {
        const int s = itk % kStages, r = itk / kStages;
        int waited = 1;
        if (lane == 0)
          waited = mbar_wait(&empty[s], (r & 1) ^ 1, abort_flag, status, status + 1, kSiteGemmProducer) ? 1 : 0;
        waited = __shfl_sync(0xffffffffu, waited, 0);
        if (!waited) return false;
        uint8_t* st = smem + s * kStage;
        // this lane's line of the four 32 x 16-byte scale chunks
        uint8_t* sf = st + 2 * kATile + kBTile + lane * 16;
        const uint32_t a0w = ue8m0_of(w0v) * 0x01010101u, a1w = ue8m0_of(w1v) * 0x01010101u;
        *reinterpret_cast<uint4*>(sf) = make_uint4(a0w, a0w, a0w, a0w);
        *reinterpret_cast<uint4*>(sf + 512) = make_uint4(a1w, a1w, a1w, a1w);
        *reinterpret_cast<uint4*>(sf + 1024) =
            make_uint4(tv[0] * 0x01010101u, tv[1] * 0x01010101u, tv[2] * 0x01010101u, tv[3] * 0x01010101u);
        *reinterpret_cast<uint4*>(sf + 1536) =
            make_uint4(tv[4] * 0x01010101u, tv[5] * 0x01010101u, tv[6] * 0x01010101u, tv[7] * 0x01010101u);
        fence_proxy_async_smem();  // the tcgen05.cp reads the tile through the async proxy
        __syncwarp();
        if (lane == 0) {
          const uint32_t fb = full_leader + s * 8;
          const int kq = (kb + ti.mp * kKStagger) % nk;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], bytes_pair);
          else mbar_arrive_remote(fb);  // this CTA's scale tile is written
          if (a_pair == 1) {  // gate and up blocks: {K, I rows, gate/up, expert}
            tma_load_4d_pair(st, &map_wp, fb, kq * 128, a0, 0, ti.expert);
          } else if (a_pair == 2) {  // the two channel blocks: {K, 256 rows, block, 512-row tile, expert}
            tma_load_5d_pair(st, &map_wp, fb, kq * 128, static_cast<int>(rank) * 128, 0, ti.mp, ti.expert);
          } else {
            tma_load_3d_pair(st, &map_w, fb, kq * 128, a0, ti.expert);
            tma_load_3d_pair(st + kATile, &map_w, fb, kq * 128, a1, ti.expert);
          }
          // this CTA's token rows as one kBRows-row box
          tma_load_2d_pair(st + 2 * kATile, mb, fb, kq * 128, brow);
          last_round[s] = r;
        }
        return true;
      };
      // this warp's K blocks of the tile: kb0, kb0 + P, kb0 + 2P, ... (P = kProducers);
      // register set E takes kb0 + 2jP, set O kb0 + (2j + 1)P
      constexpr int P = kProducers;
      const int kb0 = static_cast<int>((pw + P - it % P) % P);
      if (kb0 < nk) load_scales(kb0, ew0, ew1, et);
      if (kb0 + P < nk) load_scales(kb0 + P, ow0, ow1, ot);
      for (int kb = kb0; kb < nk && ok; kb += 2 * P) {
        ok = stage(kb, it + kb, ew0, ew1, et);
        if (!ok) break;
        if (kb + 2 * P < nk) load_scales(kb + 2 * P, ew0, ew1, et);
        if (kb + P < nk) {
          ok = stage(kb + P, it + kb + P, ow0, ow1, ot);
          if (ok && kb + 3 * P < nk) load_scales(kb + 3 * P, ow0, ow1, ot);
        }
      }
      it += nk;
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA): 2 x 4 block-scaled MMAs per K block
      uint32_t it = 0, tl = 0;
      bool ok = true;
      GroupCursor cur;
      for (int tile = pair; tile < total && ok; tile += npairs) {
        TileInfo ti;
        if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti, cur)) continue;
        const int nm = (ti.n + 15) & ~15;
        if (!mbar_wait(tmem_empty, (tl & 1) ^ 1, abort_flag, status, status + 1, kSiteGemmMma)) break;
        tc_fence_after();
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
          const uint32_t sft = b + kBTile;  // the stage's scale tile
          const uint32_t sf = tmem + kSfBase + s * kSfSlot;
          // scales of this K block into the stage's TMEM slot, ahead of the MMAs that read them
          tmem_cp_sf_pair(sf, sdesc_sf(sft));
          tmem_cp_sf_pair(sf + 4, sdesc_sf(sft + 512));
          tmem_cp_sf_pair(sf + 8, sdesc_sf(sft + 1024));
          if (nm > 128) tmem_cp_sf_pair(sf + 12, sdesc_sf(sft + 1536));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t idesc = idesc_mx_e4m3(256, nm, kk);
            const uint64_t bd = sdesc_k128(b + kk * 32);
            const uint32_t acc = (kb | kk) != 0;
            mma_mx_pair(tmem, sdesc_k128(a0 + kk * 32), bd, idesc, sf, sf + 8, acc);
            mma_mx_pair(tmem + kAcc1, sdesc_k128(a1 + kk * 32), bd, idesc, sf + 4, sf + 8, acc);
          }
          mma_commit_pair_mc(&empty[s], 0x3);  // operand stage (and its scale slot) free in both CTAs
        }
        if (!ok) break;
        mma_commit_pair_mc(tmem_full, 0x3);
        ++tl;
      }
      mma_commit_pair(drain);
      mbar_wait(drain, 0, zero_flag, status, status + 1, kSiteGemmTeardown, 100000000ull);
    }
  } else {
    // ---------------- epilogue: two groups of four warps (warps 2-5 and 6-9); warp w
    // reads TMEM lane quadrant w % 4, group g takes the 32-token column chunks g, g + 2, ...
    const int q = warp & 3;
    const int grp = (warp - 2) >> 2;
    const int f = q * 32 + lane;
    const int etid = (threadIdx.x - 64) & 127;
    uint16_t* sg = stg + grp * (32 * kStgStride);
    float* gmax = colmax + grp * 128;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tl = 0;
    GroupCursor cur;
    for (int tile = pair; tile < total; tile += npairs) {
      TileInfo ti;
      if (!decode_tile(groups, tile_start, G, E, tile, MODE, ti, cur)) continue;
      if (etid == 0)
        epi_ok[grp * 2 + (tl & 1)] = mbar_wait(tmem_full, tl & 1, abort_flag, status, status + 1, kSiteGemmEpi);
      named_bar_sync(1 + grp, 128);
      if (!epi_ok[grp * 2 + (tl & 1)]) break;  // the group's four warps stop together
      tc_fence_after();
      const int nm = (ti.n + 15) & ~15;
      const int nchunk = (nm + 31) / 32;
      const int mine = nchunk > grp ? (nchunk - grp + 1) / 2 : 0;
      // (a) every column chunk of this group out of TMEM into registers -- gate/up: h =
      // silu(g) * u in FP32; down: y as bf16 pairs, channel block 0 then 1 -- and TMEM
      // released, so that the next tile's MMAs run under (b)
      uint32_t keep[kMine][32];
#pragma unroll
      for (int ci = 0; ci < kMine; ++ci) {
        if (ci < mine) {
          const int c0 = (grp + 2 * ci) * 32;
          uint32_t ra[32], rb[32];
          tmem_ld32(tmem + lane_base + c0, ra);
          tmem_ld32(tmem + lane_base + kAcc1 + c0, rb);
          tmem_ld_wait();
          if (MODE == kGateUp) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float g = __uint_as_float(ra[i]);
              keep[ci][i] = __float_as_uint(__fdividef(g, 1.0f + __expf(-g)) * __uint_as_float(rb[i]));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              keep[ci][i] = pack_bf16x2(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1]));
              keep[ci][16 + i] = pack_bf16x2(__uint_as_float(rb[2 * i]), __uint_as_float(rb[2 * i + 1]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive_remote(tmem_empty_leader);  // this group is done with TMEM for this tile
      // (b) per chunk: quantise h (one 1x128 tile per token: this CTA's 128 features) or
      // convert y, transposed through the staging tile into whole-row stores
#pragma unroll
      for (int ci = 0; ci < kMine; ++ci) {
        if (ci >= mine) continue;
        const int c0 = (grp + 2 * ci) * 32;
        const int rows_here = min(32, ti.n - c0);
        if (MODE == kGateUp) {
          uint32_t mx = 0;  // |h| max over this warp's 32 features, token column = lane
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint32_t m = __reduce_max_sync(0xffffffffu, keep[ci][i] & 0x7fffffffu);
            if (lane == i) mx = m;
          }
          gmax[q * 32 + lane] = __uint_as_float(mx);
          named_bar_sync(1 + grp, 128);
          const int fb0 = ti.mp * 256 + static_cast<int>(rank) * 128;  // first feature of this CTA
          if (q == 0) {
            const float amax =
                fmaxf(fmaxf(gmax[lane], gmax[32 + lane]), fmaxf(gmax[64 + lane], gmax[96 + lane]));
            const float sc = pow2_scale(amax);
            gmax[lane] = pow2_recip(sc);  // the codes below are h * (1 / sc) = h / sc exactly
            if (lane < rows_here && fb0 < I) {
              const int row = ti.out_row0 + c0 + lane;
              out_scale[(size_t)row * (I / 128) + fb0 / 128] = sc;
              out_sb[(size_t)(fb0 / 128) * out_rows + row] = static_cast<uint8_t>(ue8m0_of(sc));
            }
          }
          named_bar_sync(1 + grp, 128);
          // codes, transposed to [token][feature] bytes in the staging tile
          uint8_t* sb = reinterpret_cast<uint8_t*>(sg);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const uint16_t c2 = f32x2_to_e4m3x2(__fmul_rn(__uint_as_float(keep[ci][i]), gmax[i]),
                                                __fmul_rn(__uint_as_float(keep[ci][i + 1]), gmax[i + 1]));
            sb[i * 128 + f] = static_cast<uint8_t>(c2 & 0xff);
            sb[(i + 1) * 128 + f] = static_cast<uint8_t>(c2 >> 8);
          }
          named_bar_sync(1 + grp, 128);
          if (fb0 < I) {
            const int ch = etid & 7;  // 8 x 16 bytes per 128-byte token row
            for (int rr = etid >> 3; rr < rows_here; rr += 16) {
              const uint4 val = *reinterpret_cast<const uint4*>(sb + rr * 128 + ch * 16);
              *reinterpret_cast<uint4*>(out + (size_t)(ti.out_row0 + c0 + rr) * I + fb0 + ch * 16) = val;
            }
          }
          named_bar_sync(1 + grp, 128);
        } else {
          uint16_t* y = reinterpret_cast<uint16_t*>(out);
#pragma unroll
          for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              sg[i * kStgStride + f] = static_cast<uint16_t>(keep[ci][pass * 16 + i / 2] >> (16 * (i & 1)));
            named_bar_sync(1 + grp, 128);
            const int ch = etid & 15;
            const int col = ti.mp * 512 + pass * 256 + static_cast<int>(rank) * 128 + ch * 8;
            if (col < d) {
              for (int rr = etid >> 4; rr < rows_here; rr += 8) {
                const uint4 val = *reinterpret_cast<const uint4*>(sg + rr * kStgStride + ch * 8);
                *reinterpret_cast<uint4*>(y + (size_t)(ti.out_row0 + c0 + rr) * d + col) = val;
              }
            }
            named_bar_sync(1 + grp, 128);
          }
        }
      }
      ++tl;
    }
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

// x [T, d] bf16 -> E4M3 codes + power-of-two 1x128 scales (input of the shared experts),
// the scales also as UE8M0 bytes [d/128][T]
__global__ void __launch_bounds__(128) quant_rows_pow2_kernel(const uint4* __restrict__ x, int d, int T,
                                                              uint8_t* __restrict__ q, float* __restrict__ scale,
                                                              uint8_t* __restrict__ sb) {
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = d / 8;
  for (int v0 = warp * 32; v0 < nvec; v0 += 128) {
    const int v = v0 + lane;
    const bool valid = v < nvec;
    float f[8];
    bf16x8_to_f32(valid ? __ldg(x + (size_t)t * nvec + v) : make_uint4(0, 0, 0, 0), f);
    uint2 c;
    const float sc = quant_tile16<true>(f, c);
    if (valid) {
      *reinterpret_cast<uint2*>(q + (size_t)t * d + (size_t)v * 8) = c;
      if ((lane & 15) == 0) {
        scale[(size_t)t * (d / 128) + (v >> 4)] = sc;
        sb[(size_t)(v >> 4) * T + t] = static_cast<uint8_t>(ue8m0_of(sc));
      }
    }
  }
}

// FP32 power-of-two scales [rows, nk] -> UE8M0 bytes [nk, rows] (one block per 256 rows;
// the block's rows, nk * 1 KB at most, stay in L1 across the K blocks)
__global__ void __launch_bounds__(256) scale_bytes_kernel(const float* __restrict__ src, int rows, int nk,
                                                          uint8_t* __restrict__ dst) {
  const int r = blockIdx.x * 256 + threadIdx.x;
  if (r >= rows) return;
  for (int kb = 0; kb < nk; ++kb) dst[(size_t)kb * rows + r] = static_cast<uint8_t>(ue8m0_of(__ldg(src + (size_t)r * nk + kb)));
}

}  // namespace

moe_status_t launch_expert_ffn_mx(const moe_shape_t& s, const void* x_perm, const float* x_perm_scale, const void* x,
                                  const int32_t* offsets, const void* w_gate_up, const float* w_gu_scale,
                                  const void* w_down, const float* w_down_scale, void* y, void* ws, cudaStream_t st,
                                  const WsLayout* layout) {
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
  uint8_t* sb_xp = reinterpret_cast<uint8_t*>(w + L.sb_xp);
  uint8_t* sb_xq = reinterpret_cast<uint8_t*>(w + L.sb_xq);
  uint8_t* sb_h = reinterpret_cast<uint8_t*>(w + L.sb_h);
  int* status = ws_status(ws);
  const int Tk = s.T * s.k;
  const int rows = Tk + s.S * s.T;

  schedule_kernel<<<1, 512, 0, st>>>(offsets, s.T, s.k, s.E, s.S, (s.I + 255) / 256, (s.d + 511) / 512, kChunk,
                                     groups, ts_gu, ts_dn, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  if (s.S > 0) {  // E4M3 copy of x: the shared experts' input
    quant_rows_pow2_kernel<<<s.T, 128, 0, st>>>(static_cast<const uint4*>(x), s.d, s.T, xq, xq_scale, sb_xq);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (Tk > 0) {  // the routed rows' scales as K-block-major bytes
    scale_bytes_kernel<<<(Tk + 255) / 256, 256, 0, st>>>(x_perm_scale, Tk, s.d / 128, sb_xp);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  CUtensorMap m_wgu, m_wgu_p, m_xp, m_x, m_wd, m_wd_p, m_h;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (!make_map_3d(&m_wgu, w_gate_up, u8, 1, s.d, 2 * (uint64_t)s.I, G, 128, 128)) return MOE_ERR_CUDA;
  // gate and up rows of a tile in one load: the up block is I rows after the gate block
  if (!make_map_pair_rows(&m_wgu_p, w_gate_up, u8, 1, s.d, s.I, s.I, G, 2 * (uint64_t)s.I, 128))
    return MOE_ERR_CUDA;
  if (!make_map_2d(&m_x, xq, u8, 1, s.d, s.T, 128, kBRows)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_xp, x_perm, u8, 1, s.d, Tk, 128, kBRows)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_wd, w_down, u8, 1, s.I, s.d, G, 128, 128)) return MOE_ERR_CUDA;
  // the two channel blocks of a 512-channel tile in one load (when d is a multiple of 512)
  const int dn_pair = s.d % 512 == 0 ? 2 : 0;
  m_wd_p = m_wd;
  if (dn_pair && !make_map_pair_rows5(&m_wd_p, w_down, u8, 1, s.I, 256, 256, s.d / 512, 512, G, s.d, 128))
    return MOE_ERR_CUDA;
  if (!make_map_2d(&m_h, hq, u8, 1, s.I, rows, 128, kBRows)) return MOE_ERR_CUDA;

  auto k_gu = expert_gemm_mx_kernel<kGateUp>;
  auto k_dn = expert_gemm_mx_kernel<kDown>;
  if (cudaFuncSetAttribute(k_gu, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(k_dn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int grid = pair_grid((const void*)k_gu, kThreads, kSmemBytes);
  if (grid <= 0) return MOE_ERR_CUDA;
  k_gu<<<grid, kThreads, kSmemBytes, st>>>(m_wgu, m_wgu_p, 1, m_xp, m_x, groups, ts_gu, G, s.E, s.d, s.I, s.d, sb_xp, Tk, sb_xq,
                                           s.T, w_gu_scale, 2 * s.I, hq, h_scale, sb_h, rows, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  k_dn<<<grid, kThreads, kSmemBytes, st>>>(m_wd, m_wd_p, dn_pair, m_h, m_h, groups, ts_dn, G, s.E, s.I, s.I, s.d, sb_h, rows, sb_h,
                                           rows, w_down_scale, s.d, static_cast<uint8_t*>(y), nullptr, nullptr, 0,
                                           status);
  return cuda_status(cudaGetLastError());
}

}  // namespace moe
