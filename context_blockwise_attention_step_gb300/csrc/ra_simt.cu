// ra_simt.cu — ring attention on the CUDA cores: the float32 path (any head_dim <= 128) and
// a plain cross-check for bf16 inputs. One warp per (query row, head) in the forward; the
// lanes split the head dimension and reduce dot products with shuffles.
//
// Forward: for every ring step s the warp walks the keys of K/V shard (r - s) mod D that
// its query may see (a prefix of the shard, from the global-position causal rule) and keeps
// the exact online-softmax state (running max m, denominator l, accumulator), i.e. the
// log-sum-exp merge of update_out_and_lse applied key by key (nanotron how-to page,
// "Forward Pass Implementation" and "Numerically-Stable Output Fusion").
//
// Backward ("Backward Pass and Gradient Accumulation"): P is recomputed from the final
// lse; dq is summed per query row over every step, dk and dv per key row over every query
// head of its group and every rank that sees it at some step. Two kernels, no atomics, so
// the result is run-to-run deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ra_internal.h"
#include "ra_plan.h"

namespace ra {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kMaxPerLane = 4;  // head_dim <= 128

template <typename T> __device__ __forceinline__ float ld(const T* p);
template <> __device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void st(T* p, float v);
template <> __device__ __forceinline__ void st<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T>
__device__ __forceinline__ void load_row(const T* p, int dh, int lane, float (&r)[kMaxPerLane]) {
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int d = lane + 32 * i;
    r[i] = d < dh ? ld<T>(p + d) : 0.f;
  }
}

template <typename T>
__device__ __forceinline__ float dot_row(const float (&x)[kMaxPerLane], const T* p, int dh, int lane) {
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    const int d = lane + 32 * i;
    if (d < dh) s += x[i] * ld<T>(p + d);
  }
  return warp_sum(s);
}

// -------------------------------------------------------------------------------- forward
template <typename T, typename OutT>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    fwd_simt_kernel(const __grid_constant__ Plan P, const T* __restrict__ q,
                    const T* __restrict__ k, const T* __restrict__ v, OutT* __restrict__ out,
                    float* __restrict__ lse) {
  const SeqDesc& sd = P.seq[blockIdx.y];
  const int L = sd.L, dh = P.head_dim, lane = threadIdx.x & 31;
  const int nr = plan_ranks(P);
  const long units = static_cast<long>(nr) * L * P.hq;
  for (long u = static_cast<long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); u < units;
       u += static_cast<long>(gridDim.x) * kWarpsPerBlock) {
    const int h = static_cast<int>(u % P.hq);
    const int a = static_cast<int>((u / P.hq) % L);
    const int r = P.rank_only >= 0 ? P.rank_only : static_cast<int>(u / (static_cast<long>(P.hq) * L));
    const int hk = h / P.group;
    const int qrow = sd.row_off + r * P.shard_stride + a;
    float qr[kMaxPerLane], acc[kMaxPerLane];
    load_row(q + (static_cast<size_t>(qrow) * P.hq + h) * dh, dh, lane, qr);
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) acc[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    const int64_t pq = layout_pos(P.layout, P.D, L, r, a);
    for (int s = P.step_begin; s < P.step_end; ++s) {
      const int j = shard_at_step(P.D, r, s);
      const int lim = P.causal ? key_limit(P.layout, P.D, L, j, pq) : L - 1;
      for (int b = 0; b <= lim; ++b) {
        const size_t krow = static_cast<size_t>(sd.row_off + j * P.shard_stride + b);
        const float x = dot_row(qr, k + (krow * P.hkv + hk) * dh, dh, lane) * P.scale;
        const float m_new = fmaxf(m, x);
        const float alpha = expf(m - m_new);  // m = -inf -> 0
        const float p = expf(x - m_new);
        l = l * alpha + p;
        const T* vr = v + (krow * P.hkv + hk) * dh;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
          const int d = lane + 32 * i;
          acc[i] = acc[i] * alpha + (d < dh ? p * ld<T>(vr + d) : 0.f);
        }
        m = m_new;
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    OutT* orow = out + (static_cast<size_t>(qrow) * P.hq + h) * dh;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int d = lane + 32 * i;
      if (d < dh) st<OutT>(orow + d, acc[i] * inv);
    }
    if (lane == 0)
      lse[sd.lse_off + static_cast<size_t>(h) * P.lse_hstride + static_cast<size_t>(r) * P.shard_stride + a] =
          l > 0.f ? m + logf(l) : -INFINITY;
  }
}

// -------------------------------------------------------------------------------- backward
// Block mode (the unfused path's per-step backward): only the steps [step_begin, step_end)
// and, if set, the rank rank_only; OutT = float with kAccum adds into the outputs.
template <typename T, typename OutT, bool kAccum>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    bwd_dq_simt_kernel(const __grid_constant__ Plan P, const T* __restrict__ q,
                       const T* __restrict__ k, const T* __restrict__ v,
                       const T* __restrict__ dout, const float* __restrict__ lse,
                       const float* __restrict__ delta, OutT* __restrict__ dq) {
  const SeqDesc& sd = P.seq[blockIdx.y];
  const int L = sd.L, dh = P.head_dim, lane = threadIdx.x & 31;
  const long units = static_cast<long>(plan_ranks(P)) * L * P.hq;
  for (long u = static_cast<long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); u < units;
       u += static_cast<long>(gridDim.x) * kWarpsPerBlock) {
    const int h = static_cast<int>(u % P.hq);
    const int a = static_cast<int>((u / P.hq) % L);
    const int r = P.rank_only >= 0 ? P.rank_only : static_cast<int>(u / (static_cast<long>(P.hq) * L));
    const int hk = h / P.group;
    const int qrow = sd.row_off + r * P.shard_stride + a;
    const size_t li = sd.lse_off + static_cast<size_t>(h) * P.lse_hstride + static_cast<size_t>(r) * P.shard_stride + a;
    const float lse_a = lse[li], delta_a = delta[li];
    float qr[kMaxPerLane], dor[kMaxPerLane], acc[kMaxPerLane];
    load_row(q + (static_cast<size_t>(qrow) * P.hq + h) * dh, dh, lane, qr);
    load_row(dout + (static_cast<size_t>(qrow) * P.hq + h) * dh, dh, lane, dor);
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) acc[i] = 0.f;
    const int64_t pq = layout_pos(P.layout, P.D, L, r, a);
    for (int s = P.step_begin; s < P.step_end; ++s) {
      const int j = shard_at_step(P.D, r, s);
      const int lim = P.causal ? key_limit(P.layout, P.D, L, j, pq) : L - 1;
      for (int b = 0; b <= lim; ++b) {
        const size_t krow = static_cast<size_t>(sd.row_off + j * P.shard_stride + b);
        const T* kr = k + (krow * P.hkv + hk) * dh;
        const float p = expf(dot_row(qr, kr, dh, lane) * P.scale - lse_a);
        const float dp = dot_row(dor, v + (krow * P.hkv + hk) * dh, dh, lane);
        const float ds = p * (dp - delta_a);
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
          const int d = lane + 32 * i;
          if (d < dh) acc[i] += ds * ld<T>(kr + d);
        }
      }
    }
    OutT* o = dq + (static_cast<size_t>(qrow) * P.hq + h) * dh;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int d = lane + 32 * i;
      if (d < dh) {
        if constexpr (kAccum) o[d] += acc[i] * P.scale;
        else st<OutT>(o + d, acc[i] * P.scale);
      }
    }
  }
}

template <typename T, typename OutT, bool kAccum>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    bwd_dkv_simt_kernel(const __grid_constant__ Plan P, const T* __restrict__ q,
                        const T* __restrict__ k, const T* __restrict__ v,
                        const T* __restrict__ dout, const float* __restrict__ lse,
                        const float* __restrict__ delta, OutT* __restrict__ dk, OutT* __restrict__ dv) {
  const SeqDesc& sd = P.seq[blockIdx.y];
  const int L = sd.L, dh = P.head_dim, lane = threadIdx.x & 31;
  const long units = static_cast<long>(plan_kv_shards(P)) * L * P.hkv;
  for (long u = static_cast<long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); u < units;
       u += static_cast<long>(gridDim.x) * kWarpsPerBlock) {
    const int hk = static_cast<int>(u % P.hkv);
    const int b = static_cast<int>((u / P.hkv) % L);
    const int j = P.kv_shard_only >= 0 ? P.kv_shard_only : static_cast<int>(u / (static_cast<long>(P.hkv) * L));
    const size_t krow = static_cast<size_t>(sd.row_off + j * P.shard_stride + b);
    float kr[kMaxPerLane], vr[kMaxPerLane], dka[kMaxPerLane], dva[kMaxPerLane];
    load_row(k + (krow * P.hkv + hk) * dh, dh, lane, kr);
    load_row(v + (krow * P.hkv + hk) * dh, dh, lane, vr);
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) dka[i] = dva[i] = 0.f;
    const int64_t pk = layout_pos(P.layout, P.D, L, j, b);
    for (int g = 0; g < P.group; ++g) {
      const int h = hk * P.group + g;
      for (int s = P.step_begin; s < P.step_end; ++s) {
        const int r = rank_at_step(P.D, j, s);
        if (P.rank_only >= 0 && r != P.rank_only) continue;
        const int a_begin = P.causal ? first_query(P.layout, P.D, L, r, pk) : 0;
        for (int a = a_begin; a < L; ++a) {
          const size_t qrow = static_cast<size_t>(sd.row_off + r * P.shard_stride + a);
          const size_t li = sd.lse_off + static_cast<size_t>(h) * P.lse_hstride + static_cast<size_t>(r) * P.shard_stride + a;
          const T* qa = q + (qrow * P.hq + h) * dh;
          const T* da = dout + (qrow * P.hq + h) * dh;
          const float p = expf(dot_row(kr, qa, dh, lane) * P.scale - lse[li]);
          const float dp = dot_row(vr, da, dh, lane);
          const float ds = p * (dp - delta[li]);
#pragma unroll
          for (int i = 0; i < kMaxPerLane; ++i) {
            const int d = lane + 32 * i;
            if (d < dh) {
              dva[i] += p * ld<T>(da + d);
              dka[i] += ds * ld<T>(qa + d);
            }
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int d = lane + 32 * i;
      if (d < dh) {
        if constexpr (kAccum) {
          dk[(krow * P.hkv + hk) * dh + d] += dka[i] * P.scale;
          dv[(krow * P.hkv + hk) * dh + d] += dva[i];
        } else {
          st<OutT>(dk + (krow * P.hkv + hk) * dh + d, dka[i] * P.scale);
          st<OutT>(dv + (krow * P.hkv + hk) * dh + d, dva[i]);
        }
      }
    }
  }
}

dim3 seq_grid(const Plan& P, long units_per_seq) {
  long blocks = (units_per_seq + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  return dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(P.n_seqs));
}

long max_len(const Plan& P) {
  long m = 0;
  for (int i = 0; i < P.n_seqs; ++i) m = P.seq[i].L > m ? P.seq[i].L : m;
  return m;
}

}  // namespace

cudaError_t launch_fwd_simt(const Plan& P, int dtype, const void* q, const void* k, const void* v,
                            void* out, float* lse, cudaStream_t st) {
  const dim3 grid = seq_grid(P, plan_ranks(P) * max_len(P) * P.hq);
  const dim3 block(32 * kWarpsPerBlock);
  if (dtype == RA_F32) {
    fwd_simt_kernel<float, float><<<grid, block, 0, st>>>(
        P, static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
        static_cast<float*>(out), lse);
  } else if (P.out_f32) {
    fwd_simt_kernel<__nv_bfloat16, float><<<grid, block, 0, st>>>(
        P, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), static_cast<float*>(out), lse);
  } else {
    fwd_simt_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, block, 0, st>>>(
        P, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), static_cast<__nv_bfloat16*>(out), lse);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const Plan& P, int dtype, const void* q, const void* k,
                            const void* v, const void* dout, const float* lse,
                            const float* delta, void* dq, void* dk, void* dv, cudaStream_t st) {
  const dim3 gq = seq_grid(P, plan_ranks(P) * max_len(P) * P.hq);
  const dim3 gk = seq_grid(P, plan_kv_shards(P) * max_len(P) * P.hkv);
  const dim3 block(32 * kWarpsPerBlock);
  if (P.bwd_accum) {
    if (dtype == RA_F32) {
      using T = float;
      bwd_dq_simt_kernel<T, float, true><<<gq, block, 0, st>>>(
          P, (const T*)q, (const T*)k, (const T*)v, (const T*)dout, lse, delta, (float*)dq);
      bwd_dkv_simt_kernel<T, float, true><<<gk, block, 0, st>>>(
          P, (const T*)q, (const T*)k, (const T*)v, (const T*)dout, lse, delta, (float*)dk, (float*)dv);
    } else {
      using T = __nv_bfloat16;
      bwd_dq_simt_kernel<T, float, true><<<gq, block, 0, st>>>(
          P, (const T*)q, (const T*)k, (const T*)v, (const T*)dout, lse, delta, (float*)dq);
      bwd_dkv_simt_kernel<T, float, true><<<gk, block, 0, st>>>(
          P, (const T*)q, (const T*)k, (const T*)v, (const T*)dout, lse, delta, (float*)dk, (float*)dv);
    }
  } else if (dtype == RA_F32) {
    using T = float;
    bwd_dq_simt_kernel<T, T, false><<<gq, block, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v,
                                                           (const T*)dout, lse, delta, (T*)dq);
    bwd_dkv_simt_kernel<T, T, false><<<gk, block, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v,
                                                            (const T*)dout, lse, delta, (T*)dk, (T*)dv);
  } else {
    using T = __nv_bfloat16;
    bwd_dq_simt_kernel<T, T, false><<<gq, block, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v,
                                                           (const T*)dout, lse, delta, (T*)dq);
    bwd_dkv_simt_kernel<T, T, false><<<gk, block, 0, st>>>(P, (const T*)q, (const T*)k, (const T*)v,
                                                            (const T*)dout, lse, delta, (T*)dk, (T*)dv);
  }
  return cudaGetLastError();
}

}  // namespace ra
