// ra_internal.h — launchers shared between the translation units of the library (not
// exported). Each launcher enqueues on `st` and returns the CUDA status of the launch.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ra_plan.h"

namespace ra {

// Default bound of every device-side wait (nanoseconds).
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

// 3-D TMA map over a bf16 token tensor [rows, heads, head_dim]: box 64 x 1 x 128, 128B swizzle.
cudaError_t make_token_tmap(CUtensorMap* map, const void* base, int rows, int heads, int head_dim);

// Tensor-core (bf16, head_dim 64/128) kernels.
cudaError_t launch_fwd_tc(const Plan& P, const void* q, const void* k, const void* v, void* out,
                          float* lse, cudaStream_t st);
// Backward K/V-tile kernel variants: kFused (dq sums into dq_acc, dk / dv stored in the
// problem dtype), kKvOnly (dk / dv only; dq_acc unused), kBlockAccum (float32 dq, dk, dv
// added into the outputs).
enum class BwdKind { kFused, kKvOnly, kBlockAccum, kKvAccum };
cudaError_t launch_bwd_tc(const Plan& P, BwdKind kind, const void* q, const void* k, const void* v,
                          const void* dout, const float* lse, const float* delta, float* dq_acc,
                          void* dk, void* dv, cudaStream_t st);
// Query-tile-major dq of the deterministic backward (bf16, head_dim 64/128): dq written in
// the problem dtype, no atomics. The plan's items are re-numbered inside.
cudaError_t launch_bwd_dq_tc(const Plan& P, const void* q, const void* k, const void* v,
                             const void* dout, const float* lse, const float* delta, void* dq,
                             cudaStream_t st);
cudaError_t bwd_dq_status(unsigned int* value, bool reset);
cudaError_t launch_wait_timeout(uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_exp2_poly(const float* x, float* y, int n, cudaStream_t st);
cudaError_t fwd_status(unsigned int* value, bool reset);
cudaError_t bwd_status(unsigned int* value, bool reset);

// CUDA-core kernels (f32 path; bf16 inputs accepted for cross-checks).
cudaError_t launch_fwd_simt(const Plan& P, int dtype, const void* q, const void* k, const void* v,
                            void* out, float* lse, cudaStream_t st);
cudaError_t launch_bwd_simt(const Plan& P, int dtype, const void* q, const void* k,
                            const void* v, const void* dout, const float* lse,
                            const float* delta, void* dq, void* dk, void* dv, cudaStream_t st);

// Elementwise / permutation kernels (HBM-bound).
cudaError_t launch_bwd_delta(const Plan& P, int dtype, const void* out, const void* dout,
                             float* delta, cudaStream_t st);
cudaError_t launch_dq_convert(const Plan& P, const float* dq_acc, void* dq, cudaStream_t st);
cudaError_t launch_merge(const Plan& P, float* out, float* lse, const void* block_out,
                         int block_f32, const float* block_lse, cudaStream_t st);
cudaError_t launch_shard_tokens(const Plan& P, int direction, const void* src, void* dst,
                                int64_t row_bytes, cudaStream_t st);
cudaError_t launch_shard_lse(const Plan& P, int direction, const float* src, float* dst,
                             cudaStream_t st);

// Sets the thread's ra_last_error() message (printf format) and returns `code`.
int record_error(int code, const char* fmt, ...);

}  // namespace ra
