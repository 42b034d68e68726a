// ra_noalloc.cu — a backward entry point for callers that cannot allocate device memory.
//
// ra_ring_attn_bwd needs scratch memory (the per-row dot(dout, out), and float32 dq
// partial sums for its single-pass variant) that its caller passes in. Some callers cannot provide it: a plain-C
// plugin that its host framework hands only the input and output buffers, or a caller
// whose allocator forbids cudaMalloc (and its device-wide synchronisation) inside a
// training step. For them this file keeps the scratch in one file-scope device array of
// fixed size, and ra_ring_attn_bwd_noalloc runs the ordinary backward on it.
//
// The array lives as long as the library is loaded, on every GPU that loads it. Every call
// shares it: calls that overlap on the GPU (for instance on two streams) race on it. The
// backward overwrites the per-row values and clears the dq partial sums itself before
// use, so nothing from an earlier call leaks into a later one.
#include <cuda_runtime.h>

#include <mutex>

#include "ra_internal.h"

namespace {

// In host code this name is only a host-side stand-in for the device array: its address
// must be looked up with cudaGetSymbolAddress on the device that will use it.
static __device__ __align__(256) unsigned char g_scratch[RA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device and kept
// for the life of the process (a context torn down by cudaDeviceReset is not supported).
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int ra_ring_attn_bwd_noalloc(const ra_problem* p, const void* q, const void* k,
                                        const void* v, const void* out, const float* lse,
                                        const void* dout, void* dq, void* dk, void* dv,
                                        void* stream) {
  if (int e = ra_validate(p)) return e;
  const size_t need = ra_workspace_bytes(p, 1);
  if (need > RA_NOALLOC_SCRATCH_BYTES)
    return ra::record_error(RA_ERR_WORKSPACE,
                            "problem needs %zu bytes of backward scratch; the allocation-free "
                            "backward holds at most %zu (use ra_ring_attn_bwd with a workspace)",
                            need, static_cast<size_t>(RA_NOALLOC_SCRATCH_BYTES));
  void* scratch = nullptr;
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess)
    return ra::record_error(RA_ERR_CUDA, "scratch address look-up: %s", cudaGetErrorString(e));
  return ra_ring_attn_bwd(p, q, k, v, out, lse, dout, dq, dk, dv, scratch,
                          RA_NOALLOC_SCRATCH_BYTES, stream);
}
