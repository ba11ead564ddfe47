// moe_expert_ffn_static: the expert FFN call for callers that cannot allocate
// device memory.
//
// Some callers of this library cannot call cudaMalloc: a plugin running inside
// a host framework that owns every byte of device memory and gives its plugins
// no workspace, or a latency-critical serving loop that forbids allocation after
// start-up (cudaMalloc may synchronise the device and fragments the framework's
// pool).  For them this entry point runs the same grouped expert GEMMs as
// moe_expert_ffn, but takes its scratch (the device status word, the expert-GEMM
// schedule, the E4M3 copy of x on the FP8 path and the SwiGLU intermediate h)
// from a fixed array compiled into the library instead of a caller-provided
// workspace, packed tighter than the workspace layout (which also holds what
// moe_forward needs).
//
//   * The array is kStaticScratchBytes (64 MiB).  Every GPU that loads the
//     library holds it until the process exits.
//   * Layers whose scratch does not fit are rejected with MOE_ERR_WORKSPACE
//     before anything is enqueued.  At d=7168, 256+1 experts, top-8, I=2048 the
//     scratch is about 36 KB per token in bf16 (up to 1800 tokens) and 26 KB per
//     token in FP8 (up to 2500 tokens).
//   * The first call on a device looks up the array's device address (one
//     cudaGetSymbolAddress with that device current); make that first call
//     before any stream capture.
//   * All calls share the one array, which keeps the last call's contents.  The
//     status word is cleared at the start of every call; an error found on the
//     device (inconsistent offsets, a wait that gave up) is read back with
//     moe_get_static_device_status before the next call clears it.  Calls that
//     overlap on the GPU (different streams, or different host threads, without
//     ordering between them) race on the array and give wrong results.
//   * Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library
//     routine.
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

static constexpr size_t kStaticScratchBytes = 64ull << 20;

// The scratch itself.  In host code this name is a host-side stand-in, not a
// device address: only the address from cudaGetSymbolAddress may be passed to a
// kernel.
static __device__ __align__(256) unsigned char moe_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
moe_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, moe_static_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" MOE_API moe_status_t moe_expert_ffn_static(const moe_shape_t* shape, const void* x_perm,
                                                      const float* x_perm_scale, const void* x,
                                                      const int32_t* offsets, const void* w_gate_up,
                                                      const float* w_gu_scale, const void* w_down,
                                                      const float* w_down_scale, void* y, moe_stream_t stream) {
  if (!moe::shape_valid(shape)) return MOE_ERR_INVALID_ARG;
  const moe_shape_t& s = *shape;
  if (s.E > moe::kMaxE || s.S > moe::kMaxS || s.k > moe::kMaxK) return MOE_ERR_UNSUPPORTED;
  const long long rows_ll = (long long)s.T * s.k + (long long)s.S * s.T;
  if (rows_ll * (s.d > s.I ? s.d : s.I) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  const bool none = s.T == 0;  // no tokens: the token-sized buffers may be NULL
  if (!(x_perm || none) || !(x || none) || !offsets || !w_gate_up || !w_down || !(y || none))
    return MOE_ERR_INVALID_ARG;
  if (moe::is_fp8(s.dtype) && (!(x_perm_scale || none) || !w_gu_scale || !w_down_scale))
    return MOE_ERR_INVALID_ARG;
  if (!moe::aligned16(x_perm) || !moe::aligned16(x) || !moe::aligned16(w_gate_up) || !moe::aligned16(w_down) ||
      !moe::aligned16(y))
    return MOE_ERR_ALIGNMENT;
  const moe::WsLayout L = moe::ffn_ws_layout(s);
  if (L.total > kStaticScratchBytes) return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const moe_status_t st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  cudaStream_t cs = (cudaStream_t)stream;
  // the device status word must start clear; the rest is overwritten before use
  if (cudaMemsetAsync(scratch, 0, 256, cs) != cudaSuccess) return MOE_ERR_CUDA;
  return moe::launch_expert_ffn(s, x_perm, x_perm_scale, x, nullptr, offsets, w_gate_up, w_gu_scale, w_down, w_down_scale,
                                y, scratch, cs, &L);
}

// The status word of the static array on the current device: the same read-and-clear
// as moe_get_device_status on a workspace.
extern "C" MOE_API moe_status_t moe_get_static_device_status(moe_stream_t stream) {
  void* scratch = nullptr;
  const moe_status_t st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  return moe_get_device_status(scratch, stream);
}
