// Backward pass of the layer for a fixed routing: the gradients that training the
// layer of "DeepSeek-V3 详解" 2.2-2.3 needs.  The selection bias only chooses and
// gets no gradient ("deepseek-v3-report", load-balancing paragraph), so the chosen
// set is an input here (the forward's topk_idx).  Per expert e and row r of its
// tokens, with a = x Wg^T, u = x Wu^T, h = silu(a) u, y = h Wd^T, and per token
// out = sum_shared y + sum_j g_j y_j, g_j = s_j / sum_i s_i, s = sigmoid(z):
//
//   dh_raw = dout Wd                     (dh = g dh_raw on a routed row)
//   dg_j   = <dh_raw_j, h_j>             (= <dout, y_j>; y is never recomputed)
//   ds_j   = (dg_j - sum_i g_i dg_i) / sum_i s_i,   dz_j = ds_j s_j (1 - s_j)
//   da     = dh u silu'(a),  du = dh silu(a),  dx_rows = [da du] [Wg; Wu]
//   dx[t]  = sum of dx_rows over t's rows + sum_j dz_j w_router[e_j]
//   dW_router[e] = sum over e's rows of dz x,  dW_down[e] = dy_e^T h_e,
//   dW_gate_up[e] = [da du]_e^T x_e          (dy = g dout routed, dout shared)
//
// Steps on the caller's stream:
//   1 counts and offsets of topk_idx; the permutation tables
//   2 per token: copy x and dout to the token's k rows; recompute s and g
//   3 grouped tcgen05 GEMMs: [a | u] and h (gate/up), dh_raw (W_down^T)
//   4 per row: dg, [da du]
//   5 grouped tcgen05 GEMM: dx_rows (W_gate_up^T)
//   6 per token: dz, dx
//   7 transposes of x, dy, h and [da du] into per-expert column blocks of 64
//     tokens (zero padded), with the router-gradient partial sums taken from x's
//   8 tcgen05 weight-gradient GEMMs, each expert over its own column blocks
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kTokThreads = 128;
constexpr int kRowThreads = 256;
constexpr int kTrThreads = 256;
constexpr int kTrStride = 72;  // bf16 elements per staged tile row (144 bytes, 16-byte multiple)

size_t up(size_t v, size_t a) { return (v + a - 1) / a * a; }

#define MOE_RC(expr)                  \
  do {                                \
    const moe_status_t rc_ = (expr);  \
    if (rc_ != MOE_OK) return rc_;    \
  } while (0)

__device__ __forceinline__ void bf16x8_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 f32_bf16x8(const float (&f)[8]) {
  uint4 o;
  o.x = pack_bf16x2(f[0], f[1]);
  o.y = pack_bf16x2(f[2], f[3]);
  o.z = pack_bf16x2(f[4], f[5]);
  o.w = pack_bf16x2(f[6], f[7]);
  return o;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// exclusive scan of v over the threads of one block (blockDim.x <= 1024), through buf[1024]
__device__ int block_exclusive_scan(int v, int* buf) {
  const int i = threadIdx.x;
  buf[i] = v;
  __syncthreads();
  for (int off = 1; off < (int)blockDim.x; off <<= 1) {
    const int add = i >= off ? buf[i - off] : 0;
    __syncthreads();
    buf[i] += add;
    __syncthreads();
  }
  const int inc = buf[i];
  __syncthreads();
  return inc - v;
}

// counts[e] and offsets (exclusive prefix, E + 1 entries) of the chosen experts; one block
__global__ void __launch_bounds__(1024)
    bwd_offsets_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int32_t* __restrict__ counts,
                       int32_t* __restrict__ offsets, int* __restrict__ status) {
  __shared__ int cnt[kMaxE];
  __shared__ int buf[1024];
  const int tid = threadIdx.x;
  for (int e = tid; e < kMaxE; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int n = T * k;
  for (int p = tid; p < n; p += blockDim.x) {
    const int e = idx[p];
    if (e < 0 || e >= E) set_error(status, status + 1, MOE_ERR_DEVICE, kSiteBackward);
    else atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  const int c = tid < E ? cnt[tid] : 0;
  const int ex = block_exclusive_scan(c, buf);
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = ex;
    if (tid == E - 1) offsets[E] = ex + c;
  }
}

// Per-expert weight-gradient schedules.  Expert g owns the 64-token column blocks
// [kb_start[g], kb_start[g+1]) of the transposed operands.  For dW_down (out rows
// n_a = d, features over I in m_a 512-blocks) and dW_gate_up (out rows n_b = 2I,
// features over d in m_b blocks) each group is chunked into <= 256 output rows.
__global__ void __launch_bounds__(512)
    wgrad_schedule_kernel(const int32_t* __restrict__ offsets, int T, int k, int E, int S, int n_a, int m_a, int n_b,
                          int m_b, GroupInfo* __restrict__ groups_a, int* __restrict__ ts_a,
                          GroupInfo* __restrict__ groups_b, int* __restrict__ ts_b, int* __restrict__ kb_start,
                          int* __restrict__ status) {
  __shared__ int buf[1024];
  const int G = E + S;
  const int g = threadIdx.x;
  int ntok = 0;
  if (g < E) {
    const int lo = offsets[g], hi = offsets[g + 1];
    if (lo < 0 || hi < lo || hi > T * k) set_error(status, status + 1, MOE_ERR_DEVICE, kSiteBackward);
    else ntok = hi - lo;
  } else if (g < G) {
    ntok = T;
  }
  const int nkb = (ntok + 63) / 64;
  const int kb0 = block_exclusive_scan(g < G ? nkb : 0, buf);
  GroupInfo ga{}, gb{};
  ga.n = n_a;
  ga.nchunks = (n_a + kChunkMax - 1) / kChunkMax;
  ga.csize = ((n_a + ga.nchunks - 1) / ga.nchunks + 15) & ~15;
  ga.out_row0 = g * n_a;
  gb.n = n_b;
  gb.nchunks = (n_b + kChunkMax - 1) / kChunkMax;
  gb.csize = ((n_b + gb.nchunks - 1) / gb.nchunks + 15) & ~15;
  gb.out_row0 = g * n_b;
  ga.expert = gb.expert = g;
  ga.pad0 = gb.pad0 = kb0;
  ga.pad1 = gb.pad1 = nkb;
  const int ta = block_exclusive_scan(g < G ? ga.nchunks * m_a : 0, buf);
  const int tb = block_exclusive_scan(g < G ? gb.nchunks * m_b : 0, buf);
  if (g < G) {
    groups_a[g] = ga;
    groups_b[g] = gb;
    ts_a[g] = ta;
    ts_b[g] = tb;
    kb_start[g] = kb0;
    if (g == G - 1) {
      ts_a[G] = ta + ga.nchunks * m_a;
      ts_b[G] = tb + gb.nchunks * m_b;
      kb_start[G] = kb0 + nkb;
    }
  }
}

// One block per token: copies x[t] and dout[t] to the token's k permuted rows and
// recomputes the chosen affinities s = sigmoid(x . w_router[e] (+ o_e)) (FP32 dot
// products on the CUDA cores) and gates g = s / sum s.
__global__ void __launch_bounds__(kTokThreads)
    bwd_token_fwd_kernel(const uint4* __restrict__ x, const uint4* __restrict__ dout, const uint4* __restrict__ wr,
                         const float* __restrict__ logit_offset, const int32_t* __restrict__ idx,
                         const int32_t* __restrict__ inv_pos, int d, int k, int E, int R, uint4* __restrict__ x_perm,
                         uint4* __restrict__ dout_perm, float* __restrict__ s_out, float* __restrict__ gate_out,
                         float* __restrict__ gate_row, int* __restrict__ status) {
  __shared__ int es[kMaxK], rs[kMaxK];
  __shared__ float red[kTokThreads / 32][kMaxK];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < k) {
    int e = idx[(size_t)t * k + tid];
    int r = inv_pos[(size_t)t * k + tid];
    if (e < 0 || e >= E || r < 0 || r >= R) {
      set_error(status, status + 1, MOE_ERR_DEVICE, kSiteBackward);
      e = -1;
      r = -1;
    }
    es[tid] = e;
    rs[tid] = r;
  }
  __syncthreads();
  const int nvec = d / 8;
  float acc[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) acc[j] = 0.0f;
  for (int v = tid; v < nvec; v += kTokThreads) {
    const uint4 xv = x[(size_t)t * nvec + v];
    const uint4 dv = dout[(size_t)t * nvec + v];
    float xf[8];
    bf16x8_f32(xv, xf);
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k && rs[j] >= 0) {
        x_perm[(size_t)rs[j] * nvec + v] = xv;
        dout_perm[(size_t)rs[j] * nvec + v] = dv;
        float wf[8];
        bf16x8_f32(__ldg(wr + (size_t)es[j] * nvec + v), wf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j] = fmaf(xf[i], wf[i], acc[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < k) {
      const float v = warp_sum(acc[j]);
      if (lane == 0) red[warp][j] = v;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float sv[kMaxK];
    float ssum = 0.0f;
    for (int j = 0; j < k; ++j) {
      float z = 0.0f;
      for (int w = 0; w < kTokThreads / 32; ++w) z += red[w][j];
      if (logit_offset && es[j] >= 0) z += logit_offset[es[j]];
      sv[j] = sigmoidf_(z);
      ssum += sv[j];
    }
    for (int j = 0; j < k; ++j) {
      const float g = sv[j] / ssum;
      s_out[(size_t)t * k + j] = sv[j];
      gate_out[(size_t)t * k + j] = g;
      if (rs[j] >= 0) gate_row[rs[j]] = g;
    }
  }
}

// One block per row of the expert intermediate (routed rows, then S*T shared rows):
// dg = <dh_raw, h> (routed rows), dh = g dh_raw, da = dh u silu'(a), du = dh silu(a).
__global__ void __launch_bounds__(kRowThreads)
    swiglu_bwd_kernel(const uint4* __restrict__ au, const uint4* __restrict__ h, const uint4* __restrict__ dh_raw,
                      const float* __restrict__ gate_row, int R, int I, uint4* __restrict__ dgu,
                      float* __restrict__ dgate_row) {
  __shared__ float red[kRowThreads / 32];
  const size_t r = blockIdx.x;
  const int tid = threadIdx.x;
  const bool routed = r < (size_t)R;
  const float g = routed ? gate_row[r] : 1.0f;
  const int nvec = I / 8;
  float part = 0.0f;
  for (int v = tid; v < nvec; v += kRowThreads) {
    float a[8], u[8], hh[8], dr[8], da[8], du[8];
    bf16x8_f32(au[r * 2 * nvec + v], a);
    bf16x8_f32(au[r * 2 * nvec + nvec + v], u);
    bf16x8_f32(h[r * nvec + v], hh);
    bf16x8_f32(dh_raw[r * nvec + v], dr);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      part = fmaf(dr[i], hh[i], part);
      const float dhi = g * dr[i];
      const float sa = sigmoidf_(a[i]);
      const float silu = a[i] * sa;
      da[i] = dhi * u[i] * (sa * (1.0f + a[i] * (1.0f - sa)));
      du[i] = dhi * silu;
    }
    dgu[r * 2 * nvec + v] = f32_bf16x8(da);
    dgu[r * 2 * nvec + nvec + v] = f32_bf16x8(du);
  }
  part = warp_sum(part);
  if ((tid & 31) == 0) red[tid >> 5] = part;
  __syncthreads();
  if (tid == 0 && routed) {
    float sum = 0.0f;
    for (int w = 0; w < kRowThreads / 32; ++w) sum += red[w];
    dgate_row[r] = sum;
  }
}

// One block per token: dz of its k slots, then
// dx[t] = sum_shared dx_rows + sum_j dx_rows[row j] + sum_j dz_j w_router[e_j].
__global__ void __launch_bounds__(kTokThreads)
    bwd_token_kernel(const float* __restrict__ s_in, const float* __restrict__ gate, const float* __restrict__ dgate_row,
                     const int32_t* __restrict__ idx, const int32_t* __restrict__ inv_pos,
                     const uint4* __restrict__ wr, const uint4* __restrict__ dx_rows, int T, int d, int k, int E,
                     int S, int R, float* __restrict__ dz_out, float* __restrict__ dz_row, uint4* __restrict__ dx) {
  __shared__ int es[kMaxK], rs[kMaxK];
  __shared__ float dzs[kMaxK];
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid == 0) {
    float sv[kMaxK], gv[kMaxK], dg[kMaxK];
    float ssum = 0.0f, gdg = 0.0f;
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      int r = inv_pos[(size_t)t * k + j];
      if (e < 0 || e >= E || r < 0 || r >= R) {
        e = -1;
        r = -1;
      }
      es[j] = e;
      rs[j] = r;
      sv[j] = s_in[(size_t)t * k + j];
      gv[j] = gate[(size_t)t * k + j];
      dg[j] = r >= 0 ? dgate_row[r] : 0.0f;
      ssum += sv[j];
      gdg = fmaf(gv[j], dg[j], gdg);
    }
    for (int j = 0; j < k; ++j) {
      const float ds = (dg[j] - gdg) / ssum;
      const float dz = ds * sv[j] * (1.0f - sv[j]);
      dzs[j] = dz;
      dz_out[(size_t)t * k + j] = dz;
      if (rs[j] >= 0) dz_row[rs[j]] = dz;
    }
  }
  __syncthreads();
  const int nvec = d / 8;
  for (int v = tid; v < nvec; v += kTokThreads) {
    float a[8] = {0, 0, 0, 0, 0, 0, 0, 0}, f[8];
    for (int sh = 0; sh < S; ++sh) {
      bf16x8_f32(dx_rows[((size_t)R + (size_t)sh * T + t) * nvec + v], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] += f[i];
    }
    for (int j = 0; j < k; ++j) {
      if (rs[j] < 0) continue;
      bf16x8_f32(dx_rows[(size_t)rs[j] * nvec + v], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] += f[i];
    }
    for (int j = 0; j < k; ++j) {
      if (es[j] < 0) continue;
      bf16x8_f32(__ldg(wr + (size_t)es[j] * nvec + v), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = fmaf(dzs[j], f[i], a[i]);
    }
    dx[(size_t)t * nvec + v] = f32_bf16x8(a);
  }
}

// Transposes 64 rows x 64 columns of a group's rows into dst [W, Kcap] at the
// group's column block: dst[w][kb * 64 + i] = src row i (scaled by scale_r on a
// routed row), 0 for i >= n.  Routed groups read src_r at row out_row0 + i; the
// shared experts read src_s row i when src_s is given (x, dout), else src_r at
// out_row0 + i.  With rpart: rpart[kb][w] = sum_i dz_row[out_row0 + i] src[i][w]
// over the block's rows (routed groups; the partial sums of dW_router).
__global__ void __launch_bounds__(kTrThreads)
    group_transpose_kernel(const uint4* __restrict__ src_r, const uint4* __restrict__ src_s, int W,
                           const float* __restrict__ scale_r, const GroupInfo* __restrict__ groups,
                           const int* __restrict__ kb_start, int G, int E, uint16_t* __restrict__ dst, size_t kcap,
                           const float* __restrict__ dz_row, float* __restrict__ rpart) {
  __shared__ __align__(16) uint16_t tile[64 * kTrStride];
  __shared__ float dzs[64];
  __shared__ float red[4][64];
  const int kb = blockIdx.x;  // < kcap / 64 by the launch
  if (kb >= kb_start[G]) return;
  int lo = 0, hi = G;  // kb_start[lo] <= kb < kb_start[lo + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (kb_start[mid] <= kb) lo = mid;
    else hi = mid;
  }
  const int g = lo;
  const GroupInfo gi = groups[g];
  const int i0 = (kb - kb_start[g]) * 64;
  const int w0 = blockIdx.y * 64;
  const int tid = threadIdx.x;
  const bool routed = g < E;
  const int nvec = W / 8;
  for (int v = tid; v < 512; v += kTrThreads) {
    const int row = v >> 3, c = v & 7, i = i0 + row;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (i < gi.n) {
      const uint4* src = (routed || !src_s) ? src_r + (size_t)(gi.out_row0 + i) * nvec : src_s + (size_t)i * nvec;
      val = src[w0 / 8 + c];
      if (routed && scale_r) {
        const float sc = scale_r[gi.out_row0 + i];
        float f[8];
        bf16x8_f32(val, f);
#pragma unroll
        for (int q = 0; q < 8; ++q) f[q] *= sc;
        val = f32_bf16x8(f);
      }
    }
    *reinterpret_cast<uint4*>(tile + row * kTrStride + c * 8) = val;
  }
  if (rpart && routed && tid < 64) dzs[tid] = i0 + tid < gi.n ? dz_row[gi.out_row0 + i0 + tid] : 0.0f;
  __syncthreads();
  if (rpart && routed) {
    const int f = tid & 63, part = tid >> 6;
    float sum = 0.0f;
#pragma unroll 4
    for (int rr = part * 16; rr < part * 16 + 16; ++rr)
      sum = fmaf(dzs[rr], __uint_as_float((uint32_t)tile[rr * kTrStride + f] << 16), sum);
    red[part][f] = sum;
    __syncthreads();
    if (tid < 64) rpart[(size_t)kb * W + w0 + tid] = (red[0][tid] + red[1][tid]) + (red[2][tid] + red[3][tid]);
  }
  for (int v = tid; v < 512; v += kTrThreads) {
    const int f = v & 63, q = v >> 6;
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      p[i] = (uint32_t)tile[(q * 8 + 2 * i) * kTrStride + f] |
             ((uint32_t)tile[(q * 8 + 2 * i + 1) * kTrStride + f] << 16);
    *reinterpret_cast<uint4*>(dst + (size_t)(w0 + f) * kcap + (size_t)kb * 64 + q * 8) =
        make_uint4(p[0], p[1], p[2], p[3]);
  }
}

// dW_router[e][c] = sum of rpart[kb][c] over expert e's column blocks (fixed order)
__global__ void __launch_bounds__(256)
    router_grad_kernel(const float* __restrict__ rpart, const int* __restrict__ kb_start, int nkb, int d,
                       float* __restrict__ dw_router) {
  const int e = blockIdx.x;
  const int c = blockIdx.y * 256 + threadIdx.x;
  if (c >= d) return;
  float sum = 0.0f;
  const int end = min(kb_start[e + 1], nkb);
  for (int kb = kb_start[e]; kb < end; ++kb) sum += rpart[(size_t)kb * d + c];
  dw_router[(size_t)e * d + c] = sum;
}

// w_t[g][c][r] = w[g][r][c] in 64 x 64 tiles
__global__ void __launch_bounds__(kTrThreads)
    transpose_kernel(const uint4* __restrict__ w, int R, int C, uint16_t* __restrict__ w_t) {
  __shared__ __align__(16) uint16_t tile[64 * kTrStride];
  const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
  const size_t g = blockIdx.z;
  const int tid = threadIdx.x;
  const int nvec = C / 8;
  for (int v = tid; v < 512; v += kTrThreads) {
    const int row = v >> 3, c = v & 7;
    *reinterpret_cast<uint4*>(tile + row * kTrStride + c * 8) = w[(g * R + r0 + row) * nvec + c0 / 8 + c];
  }
  __syncthreads();
  for (int v = tid; v < 512; v += kTrThreads) {
    const int f = v & 63, q = v >> 6;
    uint32_t p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      p[i] = (uint32_t)tile[(q * 8 + 2 * i) * kTrStride + f] |
             ((uint32_t)tile[(q * 8 + 2 * i + 1) * kTrStride + f] << 16);
    *reinterpret_cast<uint4*>(w_t + (g * C + c0 + f) * R + r0 + q * 8) = make_uint4(p[0], p[1], p[2], p[3]);
  }
}

}  // namespace

size_t bwd_kcap(const moe_shape_t& s) {
  const size_t R = (size_t)s.T * s.k;
  return up(R + 63 * (size_t)s.E, 64) + (size_t)s.S * up((size_t)s.T, 64);
}

BwdLayout bwd_layout(const moe_shape_t& s) {
  BwdLayout L{};
  const size_t A = 1024;
  const size_t R = (size_t)s.T * s.k;
  const size_t RS = R + (size_t)s.S * s.T;
  const size_t G = (size_t)s.E + s.S;
  const size_t d = s.d, I = s.I;
  const size_t kcap = bwd_kcap(s);
  const size_t sched = sizeof(GroupInfo) * G + sizeof(int) * 2 * (G + 1);
  size_t o = 0;
  auto take = [&](size_t& field, size_t bytes) {
    field = o;
    o = up(o + bytes, A);
  };
  take(L.status, 256);
  take(L.counts, 4 * (size_t)s.E);
  take(L.offsets, 4 * ((size_t)s.E + 1));
  take(L.perm_token, 4 * R);
  take(L.inv_pos, 4 * R);
  take(L.s, 4 * R);
  take(L.gate, 4 * R);
  take(L.gate_row, 4 * R);
  take(L.dgate_row, 4 * R);
  take(L.dz, 4 * R);
  take(L.dz_row, 4 * R);
  take(L.sched1, sched);
  take(L.sched2, sched);
  take(L.wsched_a, sched);
  take(L.wsched_b, sched);
  take(L.kb_start, 4 * (G + 1));
  take(L.x_perm, R * d * 2);
  take(L.dout_perm, R * d * 2);
  take(L.au, RS * 2 * I * 2);
  take(L.h, RS * I * 2);
  take(L.dh, RS * I * 2);
  take(L.dgu, RS * 2 * I * 2);
  take(L.dx_rows, RS * d * 2);
  take(L.xT, d * kcap * 2);
  take(L.dyT, d * kcap * 2);
  take(L.hT, I * kcap * 2);
  take(L.dguT, 2 * I * kcap * 2);
  take(L.rpart, (kcap / 64) * d * 4);
  L.total = o;
  return L;
}

moe_status_t launch_transpose_weights(int G, int R, int C, const void* w, void* w_t, cudaStream_t st) {
  if (G == 0) return MOE_OK;
  transpose_kernel<<<dim3(C / 64, R / 64, G), kTrThreads, 0, st>>>(static_cast<const uint4*>(w), R, C,
                                                                   static_cast<uint16_t*>(w_t));
  return cuda_status(cudaGetLastError());
}

moe_status_t launch_backward(const moe_shape_t& s, const void* x, const void* w_router, const float* logit_offset,
                             const void* w_gate_up, const void* w_gate_up_t, const void* w_down_t,
                             const int32_t* topk_idx, const void* dout, void* dx, float* dw_router, void* dw_gate_up,
                             void* dw_down, void* ws, cudaStream_t st) {
  const int G = s.E + s.S;
  if (s.T == 0) {  // no tokens: every weight gradient is zero
    if (cudaMemsetAsync(dw_router, 0, sizeof(float) * s.E * s.d, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(dw_gate_up, 0, (size_t)G * 2 * s.I * s.d * 2, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(dw_down, 0, (size_t)G * s.I * s.d * 2, st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const BwdLayout L = bwd_layout(s);
  char* w = static_cast<char*>(ws);
  int* status = ws_status(ws);
  const int R = s.T * s.k;
  const int RS = R + s.S * s.T;
  const size_t kcap = bwd_kcap(s);
  auto at = [&](size_t off) { return static_cast<void*>(w + off); };
  int32_t* counts = static_cast<int32_t*>(at(L.counts));
  int32_t* offsets = static_cast<int32_t*>(at(L.offsets));
  int32_t* perm_token = static_cast<int32_t*>(at(L.perm_token));
  int32_t* inv_pos = static_cast<int32_t*>(at(L.inv_pos));
  float* sv = static_cast<float*>(at(L.s));
  float* gate = static_cast<float*>(at(L.gate));
  float* gate_row = static_cast<float*>(at(L.gate_row));
  float* dgate_row = static_cast<float*>(at(L.dgate_row));
  float* dz = static_cast<float*>(at(L.dz));
  float* dz_row = static_cast<float*>(at(L.dz_row));
  auto sched = [&](size_t off, GroupInfo*& groups, int*& ts0, int*& ts1) {
    groups = static_cast<GroupInfo*>(at(off));
    ts0 = reinterpret_cast<int*>(groups + G);
    ts1 = ts0 + (G + 1);
  };
  GroupInfo *g1, *g2, *ga, *gb;
  int *ts1_gu, *ts1_dn, *ts2_gu, *ts2_dn, *ts_a, *ts_b, *unused;
  sched(L.sched1, g1, ts1_gu, ts1_dn);
  sched(L.sched2, g2, ts2_gu, ts2_dn);
  sched(L.wsched_a, ga, ts_a, unused);
  sched(L.wsched_b, gb, ts_b, unused);
  int* kb_start = static_cast<int*>(at(L.kb_start));
  void* x_perm = at(L.x_perm);
  void* dout_perm = at(L.dout_perm);
  void* au = at(L.au);
  void* h = at(L.h);
  void* dh = at(L.dh);
  void* dgu = at(L.dgu);
  void* dx_rows = at(L.dx_rows);
  uint16_t* xT = static_cast<uint16_t*>(at(L.xT));
  uint16_t* dyT = static_cast<uint16_t*>(at(L.dyT));
  uint16_t* hT = static_cast<uint16_t*>(at(L.hT));
  uint16_t* dguT = static_cast<uint16_t*>(at(L.dguT));
  float* rpart = static_cast<float*>(at(L.rpart));
  const uint4* x4 = static_cast<const uint4*>(x);
  const uint4* dout4 = static_cast<const uint4*>(dout);
  const uint4* wr4 = static_cast<const uint4*>(w_router);

  // 1 tables
  bwd_offsets_kernel<<<1, 1024, 0, st>>>(topk_idx, s.T, s.k, s.E, counts, offsets, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  moe_status_t rc = launch_permute(s, x, topk_idx, offsets, nullptr, nullptr, perm_token, inv_pos, ws, st);
  if (rc != MOE_OK) return rc;
  // 2 rows of x and dout, s and g
  bwd_token_fwd_kernel<<<s.T, kTokThreads, 0, st>>>(x4, dout4, wr4, logit_offset, topk_idx, inv_pos, s.d, s.k, s.E,
                                                    R, static_cast<uint4*>(x_perm), static_cast<uint4*>(dout_perm),
                                                    sv, gate, gate_row, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  schedule_kernel<<<1, 512, 0, st>>>(offsets, s.T, s.k, s.E, s.S, (s.I + 255) / 256, (s.I + 511) / 512, kChunkMax, g1,
                                     ts1_gu, ts1_dn, status);
  schedule_kernel<<<1, 512, 0, st>>>(offsets, s.T, s.k, s.E, s.S, 1, (s.d + 511) / 512, kChunkMax, g2, ts2_gu, ts2_dn,
                                     status);
  wgrad_schedule_kernel<<<1, 512, 0, st>>>(offsets, s.T, s.k, s.E, s.S, s.d, (s.I + 511) / 512, 2 * s.I,
                                           (s.d + 511) / 512, ga, ts_a, gb, ts_b, kb_start, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap m_wgu, m_xp, m_x, m_wdt, m_dp, m_do, m_wgut, m_dgu, m_hT, m_dyT, m_xT, m_dguT;
  if (!make_map_3d(&m_wgu, w_gate_up, bf, 2, s.d, 2 * (uint64_t)s.I, G, 64, 128)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_xp, x_perm, bf, 2, s.d, R, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_x, x, bf, 2, s.d, s.T, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_wdt, w_down_t, bf, 2, s.d, s.I, G, 64, 128)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_dp, dout_perm, bf, 2, s.d, R, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_do, dout, bf, 2, s.d, s.T, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_wgut, w_gate_up_t, bf, 2, 2 * (uint64_t)s.I, s.d, G, 64, 128)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_dgu, dgu, bf, 2, 2 * (uint64_t)s.I, RS, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_hT, hT, bf, 2, kcap, s.I, 1, 64, 128)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_dyT, dyT, bf, 2, kcap, s.d, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_xT, xT, bf, 2, kcap, s.d, 1, 64, 128)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_dguT, dguT, bf, 2, kcap, 2 * (uint64_t)s.I, 64, kBoxRows)) return MOE_ERR_CUDA;

  // 3 [a | u], h; dh_raw
  MOE_RC(launch_gemm_bwd(GemmMode::kGateUpRaw, m_wgu, m_xp, m_x, g1, ts1_gu, G, s.E, s.d, s.I, s.d, au, h, status,
                         st));
  MOE_RC(launch_gemm_bwd(GemmMode::kDgradShared, m_wdt, m_dp, m_do, g1, ts1_dn, G, s.E, s.d, s.I, s.I, dh, nullptr,
                         status, st));
  // 4 dg, [da du]
  swiglu_bwd_kernel<<<RS, kRowThreads, 0, st>>>(static_cast<const uint4*>(au), static_cast<const uint4*>(h),
                                                static_cast<const uint4*>(dh), gate_row, R, s.I,
                                                static_cast<uint4*>(dgu), dgate_row);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 5 dx_rows
  MOE_RC(launch_gemm_bwd(GemmMode::kDgradRows, m_wgut, m_dgu, m_dgu, g2, ts2_dn, G, s.E, 2 * s.I, s.I, s.d, dx_rows,
                         nullptr, status, st));
  // 6 dz, dx
  bwd_token_kernel<<<s.T, kTokThreads, 0, st>>>(sv, gate, dgate_row, topk_idx, inv_pos, wr4,
                                                static_cast<const uint4*>(dx_rows), s.T, s.d, s.k, s.E, s.S, R, dz,
                                                dz_row, static_cast<uint4*>(dx));
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 7 transposed operands (+ router-gradient partials)
  const unsigned nkb = static_cast<unsigned>(kcap / 64);
  group_transpose_kernel<<<dim3(nkb, s.d / 64), kTrThreads, 0, st>>>(
      static_cast<const uint4*>(x_perm), x4, s.d, nullptr, g1, kb_start, G, s.E, xT, kcap, dz_row, rpart);
  group_transpose_kernel<<<dim3(nkb, s.d / 64), kTrThreads, 0, st>>>(
      static_cast<const uint4*>(dout_perm), dout4, s.d, gate_row, g1, kb_start, G, s.E, dyT, kcap, nullptr, nullptr);
  group_transpose_kernel<<<dim3(nkb, s.I / 64), kTrThreads, 0, st>>>(
      static_cast<const uint4*>(h), nullptr, s.I, nullptr, g1, kb_start, G, s.E, hT, kcap, nullptr, nullptr);
  group_transpose_kernel<<<dim3(nkb, 2 * s.I / 64), kTrThreads, 0, st>>>(
      static_cast<const uint4*>(dgu), nullptr, 2 * s.I, nullptr, g1, kb_start, G, s.E, dguT, kcap, nullptr, nullptr);
  router_grad_kernel<<<dim3(s.E, (s.d + 255) / 256), 256, 0, st>>>(rpart, kb_start, (int)nkb, s.d, dw_router);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 8 weight gradients
  MOE_RC(launch_gemm_bwd(GemmMode::kWgrad, m_hT, m_dyT, m_dyT, ga, ts_a, G, s.E, (int)kcap, s.I, s.I, dw_down, nullptr,
                         status, st));
  MOE_RC(launch_gemm_bwd(GemmMode::kWgrad, m_xT, m_dguT, m_dguT, gb, ts_b, G, s.E, (int)kcap, s.I, s.d, dw_gate_up,
                         nullptr, status, st));
  return MOE_OK;
}

}  // namespace moe
