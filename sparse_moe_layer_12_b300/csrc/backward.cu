// Backward pass of the layer for a fixed routing: the gradients that training the
// layer of "DeepSeek-V3 详解" 2.2-2.3 needs.  The selection bias only chooses and
// gets no gradient ("deepseek-v3-report", load-balancing paragraph), so the chosen
// set is an input here (the forward's topk_idx).  Per expert e and row r of its
// tokens, with a = x Wg^T, u = x Wu^T, h = silu(a) u, y = h Wd^T, and per token
// out = sum_shared y + sum_j g_j y_j, g_j = s_j / sum_i s_i, s = sigmoid(z):
//
//   dy     = g dout (routed row), dout (shared expert's row)
//   dh     = dy Wd,   dg_j = <dout, y_j> = <dh_j, h_j> / g_j  (y is never formed)
//   ds_j   = (dg_j - sum_i g_i dg_i) / sum_i s_i,   dz_j = ds_j s_j (1 - s_j)
//   da     = dh u silu'(a),  du = dh silu(a),  dx_rows = [da du] [Wg; Wu]
//   dx[t]  = sum of dx_rows over t's rows + sum_j dz_j w_router[e_j]
//   dW_router[e] = sum over e's rows of dz x,  dW_down[e] = dy_e^T h_e,
//   dW_gate_up[e] = [da du]_e^T x_e
//
// Row layout: every expert's rows (routed: its tokens in token order; shared: all
// T tokens) start on a multiple of 64 and are followed by zero rows up to the next
// multiple, so the weight-gradient GEMMs contract whole 64-row blocks of one expert.
// Steps on the caller's stream:
//   1 counts, offsets, the schedules and the permutation tables
//   2 per token: x to the token's rows, s and g, then dy = g dout to the same rows
//   3 grouped tcgen05 GEMMs: FP32 [a | u] and bf16 h (gate/up); FP32 dh (W_down read
//     MN-major)
//   4 per row: <dh, h>, [da du] (the SwiGLU derivative from FP32 a, u, dh)
//   5 grouped tcgen05 GEMM: dx_rows (W_gate_up read MN-major)
//   6 per token: dg = <dh, h> / g, dz, dx; per expert: dW_router
//   7 tcgen05 weight-gradient GEMMs, both operands read MN-major from the rows
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kTokThreads = 128;

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

// Schedules of the five grouped GEMMs, one thread per group.  Group g (routed
// experts, then the shared ones) owns rows [64 kb_start[g], 64 kb_start[g+1]) of the
// row buffers, its n tokens first.  groups: the token-row GEMMs (chunks of <= 256
// tokens), with tile prefix sums for gate/up (I in 256-feature pairs), dh (I in
// 512-blocks) and dx_rows (d in 512-blocks).  groups_a / groups_b: dW_down (I columns in
// chunks of 256, d rows in 512-blocks) and dW_gate_up (d columns in chunks of 256, 2I rows
// in 512-blocks), K = the group's 64-row blocks.
__global__ void __launch_bounds__(512)
    bwd_schedule_kernel(const int32_t* __restrict__ offsets, int T, int k, int E, int S, int d, int I,
                        GroupInfo* __restrict__ groups, int* __restrict__ ts_gu, int* __restrict__ ts_dh,
                        int* __restrict__ ts_dx, GroupInfo* __restrict__ groups_a, int* __restrict__ ts_a,
                        GroupInfo* __restrict__ groups_b, int* __restrict__ ts_b, int* __restrict__ kb_start,
                        int* __restrict__ status) {
  __shared__ int buf[1024];
  const int G = E + S;
  const int g = threadIdx.x;
  const bool live = g < G;
  int ntok = 0;
  if (g < E) {
    const int lo = offsets[g], hi = offsets[g + 1];
    if (lo < 0 || hi < lo || hi > T * k) set_error(status, status + 1, MOE_ERR_DEVICE, kSiteBackward);
    else ntok = hi - lo;
  } else if (live) {
    ntok = T;
  }
  const int nkb = (ntok + 63) / 64;
  const int kb0 = block_exclusive_scan(live ? nkb : 0, buf);
  GroupInfo gi{}, ga{}, gb{};
  gi.n = ntok;
  gi.in_row0 = gi.out_row0 = kb0 * 64;
  gi.nchunks = (ntok + kChunkMax - 1) / kChunkMax;
  gi.csize = gi.nchunks ? (((ntok + gi.nchunks - 1) / gi.nchunks + 15) & ~15) : 16;
  gi.expert = g;
  ga.n = I;
  ga.csize = kChunkMax;
  ga.nchunks = (I + kChunkMax - 1) / kChunkMax;
  gb.n = d;
  gb.csize = kChunkMax;
  gb.nchunks = (d + kChunkMax - 1) / kChunkMax;
  ga.expert = gb.expert = g;
  ga.pad0 = gb.pad0 = kb0;
  ga.pad1 = gb.pad1 = nkb;
  const int n_gu = live ? gi.nchunks * ((I + 255) / 256) : 0;
  const int n_dh = live ? gi.nchunks * ((I + 511) / 512) : 0;
  const int n_dx = live ? gi.nchunks * ((d + 511) / 512) : 0;
  const int n_a = live ? ga.nchunks * ((d + 511) / 512) : 0;
  const int n_b = live ? gb.nchunks * ((2 * I + 511) / 512) : 0;
  const int t_gu = block_exclusive_scan(n_gu, buf);
  const int t_dh = block_exclusive_scan(n_dh, buf);
  const int t_dx = block_exclusive_scan(n_dx, buf);
  const int t_a = block_exclusive_scan(n_a, buf);
  const int t_b = block_exclusive_scan(n_b, buf);
  if (live) {
    groups[g] = gi;
    groups_a[g] = ga;
    groups_b[g] = gb;
    ts_gu[g] = t_gu;
    ts_dh[g] = t_dh;
    ts_dx[g] = t_dx;
    ts_a[g] = t_a;
    ts_b[g] = t_b;
    kb_start[g] = kb0;
    if (g == G - 1) {
      ts_gu[G] = t_gu + n_gu;
      ts_dh[G] = t_dh + n_dh;
      ts_dx[G] = t_dx + n_dx;
      ts_a[G] = t_a + n_a;
      ts_b[G] = t_b + n_b;
      kb_start[G] = kb0 + nkb;
    }
  }
}

// One block per token: x[t] to its k routed rows and its S shared rows, the chosen
// affinities s = sigmoid(x . w_router[e] (+ o_e)) (FP32 dot products on the CUDA
// cores) and gates g = s / sum s, then dy = g dout[t] (routed) / dout[t] (shared)
// to the same rows.  pinv[t, j] = the row of (t, j).
__global__ void __launch_bounds__(kTokThreads)
    bwd_token_fwd_kernel(const uint4* __restrict__ x, const uint4* __restrict__ dout, const uint4* __restrict__ wr,
                         const float* __restrict__ logit_offset, const int32_t* __restrict__ idx,
                         const int32_t* __restrict__ inv_pos, const int32_t* __restrict__ offsets,
                         const int* __restrict__ kb_start, int T, int d, int k, int E, int S,
                         uint4* __restrict__ xp, uint4* __restrict__ dyp, float* __restrict__ s_out,
                         float* __restrict__ gate_out, int32_t* __restrict__ pinv,
                         int* __restrict__ status) {
  __shared__ int es[kMaxK], rs[kMaxK], shr[kMaxS];
  __shared__ float gs[kMaxK];
  __shared__ float red[kTokThreads / 32][kMaxK];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < k) {
    int e = idx[(size_t)t * k + tid];
    int r = inv_pos[(size_t)t * k + tid];
    int pr = -1;
    if (e >= 0 && e < E && r >= offsets[e] && r < offsets[e + 1]) pr = r - offsets[e] + kb_start[e] * 64;
    if (pr < 0) {
      set_error(status, status + 1, MOE_ERR_DEVICE, kSiteBackward);
      e = -1;
    }
    es[tid] = e;
    rs[tid] = pr;
    pinv[(size_t)t * k + tid] = pr;
  }
  if (tid < S) shr[tid] = kb_start[E + tid] * 64 + t;
  __syncthreads();
  const int nvec = d / 8;
  float acc[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) acc[j] = 0.0f;
  for (int v = tid; v < nvec; v += kTokThreads) {
    const uint4 xv = x[(size_t)t * nvec + v];
    float xf[8];
    bf16x8_f32(xv, xf);
    for (int sh = 0; sh < S; ++sh) xp[(size_t)shr[sh] * nvec + v] = xv;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j < k && rs[j] >= 0) {
        xp[(size_t)rs[j] * nvec + v] = xv;
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
      gs[j] = g;
      s_out[(size_t)t * k + j] = sv[j];
      gate_out[(size_t)t * k + j] = g;
    }
  }
  __syncthreads();
  for (int v = tid; v < nvec; v += kTokThreads) {
    const uint4 dv = dout[(size_t)t * nvec + v];
    for (int sh = 0; sh < S; ++sh) dyp[(size_t)shr[sh] * nvec + v] = dv;
    float df[8];
    bf16x8_f32(dv, df);
    for (int j = 0; j < k; ++j) {
      if (rs[j] < 0) continue;
      float f[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = gs[j] * df[i];
      dyp[(size_t)rs[j] * nvec + v] = f32_bf16x8(f);
    }
  }
}

// Zero rows n .. 64 ceil(n / 64) - 1 of every group in x, dy, h and [da du] (the
// operands of the weight-gradient GEMMs; grid: groups x 64)
__global__ void __launch_bounds__(128)
    zero_pad_rows_kernel(const GroupInfo* __restrict__ groups, int d, int I, uint4* __restrict__ xp,
                         uint4* __restrict__ dyp, uint4* __restrict__ h, uint4* __restrict__ dgu) {
  const GroupInfo gi = groups[blockIdx.x];
  const int i = gi.n + blockIdx.y;
  if (i >= ((gi.n + 63) & ~63)) return;
  const size_t row = (size_t)gi.in_row0 + i;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int v = threadIdx.x; v < d / 8; v += 128) {
    xp[row * (d / 8) + v] = z;
    dyp[row * (d / 8) + v] = z;
  }
  for (int v = threadIdx.x; v < I / 8; v += 128) {
    h[row * (I / 8) + v] = z;
    dgu[row * (I / 4) + v] = z;
    dgu[row * (I / 4) + I / 8 + v] = z;
  }
}

// One block per row (64 kb_start[G] rows; pad rows are skipped, zero already):
// <dh, h> (routed rows), da = dh u silu'(a), du = dh silu(a) from FP32 a, u, dh.
__global__ void __launch_bounds__(256)
    swiglu_bwd_kernel(const float4* __restrict__ au, const uint2* __restrict__ h, const float4* __restrict__ dh,
                      const GroupInfo* __restrict__ groups, const int* __restrict__ kb_start, int G, int E, int I,
                      uint2* __restrict__ dgu, float* __restrict__ dhh_row) {
  __shared__ float red[8];
  const size_t r = blockIdx.x;
  const int tid = threadIdx.x;
  const int kb = static_cast<int>(r >> 6);
  if (kb >= kb_start[G]) return;
  int lo = 0, hi = G;  // kb_start[lo] <= kb < kb_start[lo + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (kb_start[mid] <= kb) lo = mid;
    else hi = mid;
  }
  if ((int)(r - (size_t)kb_start[lo] * 64) >= groups[lo].n) return;  // pad row
  const int n4 = I / 4;
  float part = 0.0f;
  for (int v = tid; v < n4; v += 256) {
    const float4 a = au[r * 2 * n4 + v], u = au[r * 2 * n4 + n4 + v], g = dh[r * n4 + v];
    const uint2 hv = h[r * n4 + v];
    const float av[4] = {a.x, a.y, a.z, a.w}, uv[4] = {u.x, u.y, u.z, u.w}, gv[4] = {g.x, g.y, g.z, g.w};
    const float hh[4] = {__uint_as_float(hv.x << 16), __uint_as_float(hv.x & 0xffff0000u),
                         __uint_as_float(hv.y << 16), __uint_as_float(hv.y & 0xffff0000u)};
    float da[4], du[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      part = fmaf(gv[i], hh[i], part);
      const float sa = sigmoidf_(av[i]);
      da[i] = gv[i] * uv[i] * (sa * (1.0f + av[i] * (1.0f - sa)));
      du[i] = gv[i] * (av[i] * sa);
    }
    dgu[r * 2 * n4 + v] = make_uint2(pack_bf16x2(da[0], da[1]), pack_bf16x2(da[2], da[3]));
    dgu[r * 2 * n4 + n4 + v] = make_uint2(pack_bf16x2(du[0], du[1]), pack_bf16x2(du[2], du[3]));
  }
  part = warp_sum(part);
  if ((tid & 31) == 0) red[tid >> 5] = part;
  __syncthreads();
  if (tid == 0 && lo < E) {
    float sum = 0.0f;
    for (int w = 0; w < 8; ++w) sum += red[w];
    dhh_row[r] = sum;
  }
}

// One block per token: dg_j = <dh, h> / g_j of its k rows, dz, then
// dx[t] = sum_shared dx_rows + sum_j dx_rows[row j] + sum_j dz_j w_router[e_j].
__global__ void __launch_bounds__(kTokThreads)
    bwd_token_kernel(const float* __restrict__ s_in, const float* __restrict__ gate,
                     const float* __restrict__ dhh_row, const int32_t* __restrict__ idx,
                     const int32_t* __restrict__ pinv, const int* __restrict__ kb_start,
                     const uint4* __restrict__ wr, const uint4* __restrict__ dx_rows, int d, int k, int E, int S,
                     float* __restrict__ dz_out, float* __restrict__ dz_prow, uint4* __restrict__ dx) {
  __shared__ int es[kMaxK], rs[kMaxK], shr[kMaxS];
  __shared__ float dzs[kMaxK];
  const int t = blockIdx.x, tid = threadIdx.x;
  if (tid < S) shr[tid] = kb_start[E + tid] * 64 + t;
  if (tid == 0) {
    float sv[kMaxK], gv[kMaxK], dg[kMaxK];
    float ssum = 0.0f, gdg = 0.0f;
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      const int r = pinv[(size_t)t * k + j];
      if (e < 0 || e >= E || r < 0) e = -1;
      es[j] = e;
      rs[j] = e < 0 ? -1 : r;
      sv[j] = s_in[(size_t)t * k + j];
      gv[j] = gate[(size_t)t * k + j];
      // dh = g dout Wd, so <dout, y> = <dh, h> / g; g = 0 means s = 0 and dz = 0 whatever dg is
      dg[j] = rs[j] >= 0 && gv[j] > 0.0f ? dhh_row[rs[j]] / gv[j] : 0.0f;
      ssum += sv[j];
      gdg = fmaf(gv[j], dg[j], gdg);
    }
    for (int j = 0; j < k; ++j) {
      const float ds = (dg[j] - gdg) / ssum;
      const float dz = ds * sv[j] * (1.0f - sv[j]);
      dzs[j] = dz;
      dz_out[(size_t)t * k + j] = dz;
      if (rs[j] >= 0) dz_prow[rs[j]] = dz;
    }
  }
  __syncthreads();
  const int nvec = d / 8;
  for (int v = tid; v < nvec; v += kTokThreads) {
    float a[8] = {0, 0, 0, 0, 0, 0, 0, 0}, f[8];
    for (int sh = 0; sh < S; ++sh) {
      bf16x8_f32(dx_rows[(size_t)shr[sh] * nvec + v], f);
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

// dW_router[e][c] = sum over expert e's rows i (in order) of dz[i] x[i][c]; eight
// columns per thread
__global__ void __launch_bounds__(128)
    router_grad_kernel(const uint4* __restrict__ xp, const float* __restrict__ dz_prow,
                       const GroupInfo* __restrict__ groups, int d, float* __restrict__ dw_router) {
  const int e = blockIdx.x;
  const int v = blockIdx.y * 128 + threadIdx.x;
  const int nvec = d / 8;
  if (v >= nvec) return;
  const GroupInfo gi = groups[e];
  float a[8] = {0, 0, 0, 0, 0, 0, 0, 0}, f[8];
  for (int i = 0; i < gi.n; ++i) {
    const size_t row = (size_t)gi.in_row0 + i;
    const float dz = dz_prow[row];
    bf16x8_f32(xp[row * nvec + v], f);
#pragma unroll
    for (int q = 0; q < 8; ++q) a[q] = fmaf(dz, f[q], a[q]);
  }
  float4* o = reinterpret_cast<float4*>(dw_router + (size_t)e * d + (size_t)v * 8);
  o[0] = make_float4(a[0], a[1], a[2], a[3]);
  o[1] = make_float4(a[4], a[5], a[6], a[7]);
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
  const size_t G = (size_t)s.E + s.S;
  const size_t d = s.d, I = s.I;
  const size_t kcap = bwd_kcap(s);
  const size_t sched = sizeof(GroupInfo) * G + sizeof(int) * 3 * (G + 1);
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
  take(L.pinv, 4 * R);
  take(L.dz, 4 * R);
  take(L.dgate_prow, 4 * kcap);
  take(L.dz_prow, 4 * kcap);
  take(L.sched, sched);
  take(L.wsched_a, sched);
  take(L.wsched_b, sched);
  take(L.kb_start, 4 * (G + 1));
  take(L.xp, kcap * d * 2);
  take(L.dyp, kcap * d * 2);
  take(L.au, kcap * 2 * I * 4);
  take(L.h, kcap * I * 2);
  take(L.dh, kcap * I * 4);
  take(L.dgu, kcap * 2 * I * 2);
  take(L.dx_rows, kcap * d * 2);
  L.total = o;
  return L;
}

moe_status_t launch_backward(const moe_shape_t& s, const void* x, const void* w_router, const float* logit_offset,
                             const void* w_gate_up, const void* w_down, const int32_t* topk_idx, const void* dout,
                             void* dx, float* dw_router, void* dw_gate_up, void* dw_down, void* ws,
                             cudaStream_t st) {
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
  const size_t kcap = bwd_kcap(s);
  auto at = [&](size_t off) { return static_cast<void*>(w + off); };
  int32_t* counts = static_cast<int32_t*>(at(L.counts));
  int32_t* offsets = static_cast<int32_t*>(at(L.offsets));
  int32_t* perm_token = static_cast<int32_t*>(at(L.perm_token));
  int32_t* inv_pos = static_cast<int32_t*>(at(L.inv_pos));
  float* sv = static_cast<float*>(at(L.s));
  float* gate = static_cast<float*>(at(L.gate));
  int32_t* pinv = static_cast<int32_t*>(at(L.pinv));
  float* dz = static_cast<float*>(at(L.dz));
  float* dhh_row = static_cast<float*>(at(L.dgate_prow));
  float* dz_prow = static_cast<float*>(at(L.dz_prow));
  GroupInfo* groups = static_cast<GroupInfo*>(at(L.sched));
  int* ts_gu = reinterpret_cast<int*>(groups + G);
  int* ts_dh = ts_gu + (G + 1);
  int* ts_dx = ts_dh + (G + 1);
  GroupInfo* ga = static_cast<GroupInfo*>(at(L.wsched_a));
  int* ts_a = reinterpret_cast<int*>(ga + G);
  GroupInfo* gb = static_cast<GroupInfo*>(at(L.wsched_b));
  int* ts_b = reinterpret_cast<int*>(gb + G);
  int* kb_start = static_cast<int*>(at(L.kb_start));
  void* xp = at(L.xp);
  void* dyp = at(L.dyp);
  void* au = at(L.au);
  void* h = at(L.h);
  void* dh = at(L.dh);
  void* dgu = at(L.dgu);
  void* dx_rows = at(L.dx_rows);
  const uint4* wr4 = static_cast<const uint4*>(w_router);

  // 1 tables and schedules
  bwd_offsets_kernel<<<1, 1024, 0, st>>>(topk_idx, s.T, s.k, s.E, counts, offsets, status);
  bwd_schedule_kernel<<<1, 512, 0, st>>>(offsets, s.T, s.k, s.E, s.S, s.d, s.I, groups, ts_gu, ts_dh, ts_dx, ga,
                                         ts_a, gb, ts_b, kb_start, status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  MOE_RC(launch_permute(s, x, topk_idx, offsets, nullptr, nullptr, perm_token, inv_pos, ws, st));
  // 2 rows of x and dy, s and g
  bwd_token_fwd_kernel<<<s.T, kTokThreads, 0, st>>>(
      static_cast<const uint4*>(x), static_cast<const uint4*>(dout), wr4, logit_offset, topk_idx, inv_pos, offsets,
      kb_start, s.T, s.d, s.k, s.E, s.S, static_cast<uint4*>(xp), static_cast<uint4*>(dyp), sv, gate, pinv,
      status);
  zero_pad_rows_kernel<<<dim3(G, 64), 128, 0, st>>>(groups, s.d, s.I, static_cast<uint4*>(xp),
                                                    static_cast<uint4*>(dyp), static_cast<uint4*>(h),
                                                    static_cast<uint4*>(dgu));
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;

  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap m_wgu, m_xp, m_wd_mn, m_dyp, m_wgu_mn, m_dgu, m_h_mn, m_dyp_mn, m_xp_mn, m_dgu_mn;
  // weight gradients: A = the rows' operand of dW (dy for dW_down, [da du] for dW_gate_up)
  // as [1][kcap][M] with 64 x 64 boxes, B = the columns' operand (h, x) as [kcap][N]
  const uint64_t I2 = 2 * (uint64_t)s.I;
  if (!make_map_3d(&m_wgu, w_gate_up, bf, 2, s.d, I2, G, 64, 128)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_xp, xp, bf, 2, s.d, kcap, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_wd_mn, w_down, bf, 2, s.I, s.d, G, 64, 64)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_dyp, dyp, bf, 2, s.d, kcap, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_wgu_mn, w_gate_up, bf, 2, s.d, I2, G, 64, 64)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_dgu, dgu, bf, 2, I2, kcap, 64, kBoxRows)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_h_mn, h, bf, 2, s.I, kcap, 64, 64)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_dyp_mn, dyp, bf, 2, s.d, kcap, 1, 64, 64)) return MOE_ERR_CUDA;
  if (!make_map_2d(&m_xp_mn, xp, bf, 2, s.d, kcap, 64, 64)) return MOE_ERR_CUDA;
  if (!make_map_3d(&m_dgu_mn, dgu, bf, 2, I2, kcap, 1, 64, 64)) return MOE_ERR_CUDA;

  // 3 [a | u] (FP32), h; dh (FP32)
  MOE_RC(launch_gemm_bwd(GemmMode::kGateUpRaw, m_wgu, m_xp, m_xp, groups, ts_gu, G, s.E, s.d, s.I, s.d, au, h, status,
                         st));
  MOE_RC(launch_gemm_bwd(GemmMode::kDgrad32, m_wd_mn, m_dyp, m_dyp, groups, ts_dh, G, s.E, s.d, s.I, s.I, dh, nullptr,
                         status, st));
  // 4 <dh, h>, [da du]
  swiglu_bwd_kernel<<<static_cast<unsigned>(kcap), 256, 0, st>>>(
      static_cast<const float4*>(au), static_cast<const uint2*>(h), static_cast<const float4*>(dh), groups, kb_start,
      G, s.E, s.I, static_cast<uint2*>(dgu), dhh_row);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 5 dx_rows
  MOE_RC(launch_gemm_bwd(GemmMode::kDgrad, m_wgu_mn, m_dgu, m_dgu, groups, ts_dx, G, s.E, 2 * s.I, s.I, s.d, dx_rows,
                         nullptr, status, st));
  // 6 dg, dz, dx; dW_router
  bwd_token_kernel<<<s.T, kTokThreads, 0, st>>>(sv, gate, dhh_row, topk_idx, pinv, kb_start, wr4,
                                                static_cast<const uint4*>(dx_rows), s.d, s.k, s.E, s.S, dz, dz_prow,
                                                static_cast<uint4*>(dx));
  router_grad_kernel<<<dim3(s.E, (s.d / 8 + 127) / 128), 128, 0, st>>>(static_cast<const uint4*>(xp), dz_prow,
                                                                       groups, s.d, dw_router);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  // 7 weight gradients
  CUtensorMap m_dwd, m_dwgu;  // outputs [G][rows][cols], stored from staged 128 x 32 tiles
  if (!make_map_3d_sw64(&m_dwd, dw_down, bf, 2, s.I, s.d, G, 32, 128)) return MOE_ERR_CUDA;
  if (!make_map_3d_sw64(&m_dwgu, dw_gate_up, bf, 2, s.d, I2, G, 32, 128)) return MOE_ERR_CUDA;
  // (the `I` argument carries the output rows per expert, `width` its columns)
  MOE_RC(launch_gemm_bwd(GemmMode::kWgrad, m_dyp_mn, m_h_mn, m_h_mn, ga, ts_a, G, s.E, (int)kcap, s.d, s.I, dw_down,
                         nullptr, status, st, &m_dwd));
  MOE_RC(launch_gemm_bwd(GemmMode::kWgrad, m_dgu_mn, m_xp_mn, m_xp_mn, gb, ts_b, G, s.E, (int)kcap, 2 * s.I, s.d,
                         dw_gate_up, nullptr, status, st, &m_dwgu));
  return MOE_OK;
}

}  // namespace moe
