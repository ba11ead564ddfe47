// Combine, bias update and FP8 weight preparation.
//
// combine      out[t] = sum_s y_shared_s[t] + sum_j gate[t, j] * y[inv_pos[t, j]]
//              (the gate-weighted sum over the chosen experts plus the always-on
//              shared expert: "deepseek-v3-report" model table "8 + 1";
//              "DeepSeek-V3 详解" 2.2).  FP32 sum in a fixed order, bf16 store.
// bias update  b_i += gamma * sign(T*k/E - count_i) ("DeepSeek-V3 详解" 2.3,
//              gamma = 0.001; "deepseek-v3-report": overloaded -> down,
//              idle -> up; "DeepSeek-V3 技术报告要点" 4.2: per batch).
// quant        per-128x128-block E4M3 quantisation of expert weights
//              ("DeepSeek-V3 详解" 4.2), scale = amax / 448.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kCombineThreads = 128;

__device__ __forceinline__ void acc_bf16x8(float (&a)[8], const uint4& v, float g) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = fmaf(g, __uint_as_float(w[i] << 16), a[2 * i]);
    a[2 * i + 1] = fmaf(g, __uint_as_float(w[i] & 0xffff0000u), a[2 * i + 1]);
  }
}

__device__ __forceinline__ void add_bf16x8(float (&a)[8], const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] += __uint_as_float(w[i] << 16);
    a[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const uint4* __restrict__ y, const float* __restrict__ gate, const int32_t* __restrict__ inv_pos,
                   int T, int d, int k, int S, uint4* __restrict__ out) {
  __shared__ int pos[kMaxK];
  __shared__ float g[kMaxK];
  const int t = blockIdx.x;
  const long long rows = (long long)T * k + (long long)S * T;
  if (threadIdx.x < k) {
    int p = inv_pos[(size_t)t * k + threadIdx.x];
    pos[threadIdx.x] = (p >= 0 && p < T * k) ? p : -1;
    g[threadIdx.x] = gate[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  const int nvec = d / 8;
  for (int v = threadIdx.x; v < nvec; v += kCombineThreads) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = 0.0f;
    for (int s = 0; s < S; ++s) {
      const long long r = (long long)T * k + (long long)s * T + t;
      if (r < rows) add_bf16x8(a, __ldg(y + r * nvec + v));
    }
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 buf[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int jj = j0 + j;
        buf[j] = (jj < k && pos[jj] >= 0) ? __ldg(y + (size_t)pos[jj] * nvec + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int jj = j0 + j;
        if (jj < k) acc_bf16x8(a, buf[j], g[jj]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(a[0], a[1]);
    o.y = pack_bf16x2(a[2], a[3]);
    o.z = pack_bf16x2(a[4], a[5]);
    o.w = pack_bf16x2(a[6], a[7]);
    out[(size_t)t * nvec + v] = o;
  }
}

__global__ void bias_update_kernel(const int32_t* __restrict__ counts, float* __restrict__ bias, int E,
                                   long long Tk, float gamma) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= E) return;
  const long long load = (long long)E * counts[i];
  const float sgn = Tk > load ? 1.0f : (Tk < load ? -1.0f : 0.0f);
  bias[i] = bias[i] + gamma * sgn;
}

// one CTA per 128x128 block of one expert matrix; scale = amax / 448, or (POW2) the
// smallest power of two with amax <= 448 * scale
template <bool POW2>
__global__ void __launch_bounds__(256)
    quant_weight_kernel(const uint16_t* __restrict__ w, uint8_t* __restrict__ wq, float* __restrict__ ws, int N,
                        int K) {
  __shared__ float red[8];
  const int kb = blockIdx.x, nb = blockIdx.y, g = blockIdx.z;
  const int nkb = K / 128;
  const size_t base = (size_t)g * N * K + (size_t)nb * 128 * K + (size_t)kb * 128;
  // thread: row r = tid / 2 (0..127), 64-element half h = tid % 2
  const int r = threadIdx.x >> 1, h = threadIdx.x & 1;
  const uint4* src = reinterpret_cast<const uint4*>(w + base + (size_t)r * K + h * 64);
  float f[64];
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint4 u = __ldg(src + v);
    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[v * 8 + 2 * i] = __uint_as_float(wd[i] << 16);
      f[v * 8 + 2 * i + 1] = __uint_as_float(wd[i] & 0xffff0000u);
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float scale = POW2 ? pow2_scale(amax) : (amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f));
  uint2* dst = reinterpret_cast<uint2*>(wq + base + (size_t)r * K + h * 64);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint32_t a = f32x2_to_e4m3x2(__fdiv_rn(f[v * 8 + 0], scale), __fdiv_rn(f[v * 8 + 1], scale));
    const uint32_t b = f32x2_to_e4m3x2(__fdiv_rn(f[v * 8 + 2], scale), __fdiv_rn(f[v * 8 + 3], scale));
    const uint32_t c = f32x2_to_e4m3x2(__fdiv_rn(f[v * 8 + 4], scale), __fdiv_rn(f[v * 8 + 5], scale));
    const uint32_t e = f32x2_to_e4m3x2(__fdiv_rn(f[v * 8 + 6], scale), __fdiv_rn(f[v * 8 + 7], scale));
    dst[v] = make_uint2(a | (b << 16), c | (e << 16));
  }
  if (threadIdx.x == 0) ws[((size_t)g * (N / 128) + nb) * nkb + kb] = scale;
}

}  // namespace

moe_status_t launch_combine(const moe_shape_t& s, const void* y, const float* gate, const int32_t* inv_pos,
                            void* out, cudaStream_t st) {
  if (s.T == 0) return MOE_OK;
  combine_kernel<<<s.T, kCombineThreads, 0, st>>>(static_cast<const uint4*>(y), gate, inv_pos, s.T, s.d, s.k, s.S,
                                                  static_cast<uint4*>(out));
  return cuda_status(cudaGetLastError());
}

moe_status_t launch_bias_update(const moe_shape_t& s, const int32_t* counts, float* bias, float gamma,
                                cudaStream_t st) {
  bias_update_kernel<<<(s.E + 255) / 256, 256, 0, st>>>(counts, bias, s.E, (long long)s.T * s.k, gamma);
  return cuda_status(cudaGetLastError());
}

moe_status_t launch_quant_weights(int G, int N, int K, const void* w, void* w_q, float* w_scale, bool pow2,
                                  cudaStream_t st) {
  if (N / 128 > 65535 || G > 65535) return MOE_ERR_UNSUPPORTED;
  dim3 grid(K / 128, N / 128, G);
  if (pow2)
    quant_weight_kernel<true><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(w), static_cast<uint8_t*>(w_q),
                                                    w_scale, N, K);
  else
    quant_weight_kernel<false><<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(w), static_cast<uint8_t*>(w_q),
                                                     w_scale, N, K);
  return cuda_status(cudaGetLastError());
}

}  // namespace moe
