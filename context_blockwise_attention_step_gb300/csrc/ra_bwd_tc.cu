// ra_bwd_tc.cu — ring-attention backward on the 5th-generation tensor cores (sm_103a).
//
// The pages' backward ("Backward Pass and Gradient Accumulation", nanotron how-to page)
// revisits every (rank, step) block, differentiates it against the FINAL out and lse,
// adds block_dq into the rank's dq and sends block_dk / block_dv around the ring back to
// the shard that owns the K/V. On one GPU the ring of gradients becomes an accumulation in
// place: a persistent CTA owns one 128-row K/V tile (shard j, one K/V head) and walks
// every ring step s, i.e. the query shard r = (j + s) mod D that holds this K/V at step s,
// every query head of the GQA group, and every 128-row query tile of shard r that may see
// the tile (global-position causal rule). With P^T computed K/V-row-major:
//
//   S^T  = K Q^T                 tcgen05 (SS), TMEM
//   P^T  = 2^(S^T*scale*log2e - lse*log2e)  (recomputed from lse, masked), bf16 -> TMEM
//   dP^T = V dO^T                tcgen05 (SS), TMEM
//   dV  += P^T dO                tcgen05 (TS: P^T from TMEM), f32 in TMEM for the whole walk
//   dS^T = P^T * (dP^T - delta)  delta = rowsum(dO * O) from the preprocess kernel; bf16 smem
//   dK  += dS^T Q                tcgen05 (SS), f32 in TMEM for the whole walk
//   dQ   = dS K                  tcgen05 (SS, dS read MN-major), then added with vector
//                                float atomics into an f32 dq workspace
//
// dK and dV leave TMEM once per tile (times scale for dK), so they need no atomics; dq is
// scaled and converted by the postprocess kernel.
//
// Warp roles (384 threads): warp 0 TMA producer (K, V once per item; Q and dO per query
// tile, two stages), warp 1 TMEM allocator + MMA issuer, warps 4-7 the P / dS warpgroup
// (thread = K/V row) which also writes dK and dV, warps 8-11 the dQ warpgroup
// (thread = query row).
#include <cuda_runtime.h>

#include "ra_internal.h"
#include "ra_plan.h"
#include "ra_ptx.cuh"

namespace ra {

static __device__ unsigned int g_status_bwd;

namespace {

constexpr int kBwdThreads = 384;
constexpr int kSubBytes = 128 * 128;
constexpr float kLog2e = 1.4426950408889634f;

template <int DH>
struct BwdCfg {
  static constexpr int kSub = DH / 64;
  static constexpr int kTileBytes = 128 * DH * 2;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffQ = kOffV + kTileBytes;            // 2 stages: Q then dO
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffDS = kOffQ + 2 * kStageBytes;     // 128 x 128 bf16
  static constexpr int kOffLse = kOffDS + 2 * kSubBytes;     // [2][128] f32
  static constexpr int kOffDelta = kOffLse + 2 * 128 * 4;    // [2][128] f32
  static constexpr int kOffBar = kOffDelta + 2 * 128 * 4;
  static constexpr int kSmemBytes = kOffBar + 320;
  static constexpr int kKSteps = DH / 16;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColDK = 0, kColDV = DH, kColS = 2 * DH, kColDP = 2 * DH + 128;
};

struct BwdBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full, ds_empty, dq_full, dq_free;
  uint64_t acc_done, acc_free, drain;
  uint64_t lse_bar[2];
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdWalk {
  int L, b0, N, nqt;
  int64_t pk0;  // global position of the tile's first K/V row
};

__device__ __forceinline__ int qt_begin(const Plan& P, const BwdWalk& w, int r) {
  if (!P.causal) return 0;
  const int a = first_query(P.layout, P.D, w.L, r, w.pk0);
  return a >= w.L ? w.nqt : a / kQTileRows;
}

__device__ __forceinline__ BwdWalk bwd_walk(const Plan& P, const BwdItem& it) {
  BwdWalk w;
  w.L = P.seq[it.seq].L;
  w.b0 = it.kt * kKvTileRows;
  w.nqt = ceil_div(w.L, kQTileRows);
  w.pk0 = layout_pos(P.layout, P.D, w.L, it.j, w.b0);
  w.N = 0;
  for (int r = 0; r < P.D; ++r) w.N += w.nqt - qt_begin(P, w, r);
  w.N *= P.group;
  return w;
}

// Calls f(r, h, q0) for every query tile the item visits, in walk order; stops early when
// f returns false. Returns false if stopped. The query ranks are walked in the same fixed
// order 0..D-1 by every item (not in ring-step order relative to the item's shard): the
// set of (rank, step) pairs and hence the sums are the same, but CTAs that run together
// then read the same Q / dO tiles and add into the same dq rows at about the same time.
template <typename F>
__device__ __forceinline__ bool for_each_qtile(const Plan& P, const BwdItem& it, const BwdWalk& w,
                                               F&& f) {
  for (int r = 0; r < P.D; ++r) {
    const int q_begin = qt_begin(P, w, r);
    for (int g = 0; g < P.group; ++g) {
      const int h = it.hk * P.group + g;
      for (int qt = q_begin; qt < w.nqt; ++qt)
        if (!f(r, h, qt * kQTileRows)) return false;
    }
  }
  return true;
}

__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16* dst, const uint32_t (&r)[32],
                                                 float mul) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * mul, __uint_as_float(r[8 * q + 1]) * mul);
    u.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * mul, __uint_as_float(r[8 * q + 3]) * mul);
    u.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * mul, __uint_as_float(r[8 * q + 5]) * mul);
    u.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * mul, __uint_as_float(r[8 * q + 7]) * mul);
    d[q] = u;
  }
}

template <int DH>
__global__ void __launch_bounds__(kBwdThreads, 1)
    ring_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ Plan P,
                       const float* __restrict__ lse, const float* __restrict__ delta,
                       float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dk,
                       __nv_bfloat16* __restrict__ dv) {
  using C = BwdCfg<DH>;
  extern __shared__ __align__(1024) uint8_t smem[];
  BwdBars& sh = *reinterpret_cast<BwdBars*>(smem + C::kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {  // the swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicOr(&g_status_bwd, 2u);
    return;
  }
  volatile int* abort_flag = &sh.abort_flag;
  unsigned int* status = &g_status_bwd;
  const uint64_t tmo = P.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(&sh.kv_full, 1);
    mbar_init(&sh.kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.q_full[i], 1);
      mbar_init(&sh.q_empty[i], 1);
    }
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.p_full, 128);
    mbar_init(&sh.ds_full, 128);
    mbar_init(&sh.ds_empty, 1);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_free, 128);
    mbar_init(&sh.acc_done, 1);
    mbar_init(&sh.acc_free, 128);
    mbar_init(&sh.drain, 1);
    mbar_init(&sh.lse_bar[0], 128);
    mbar_init(&sh.lse_bar[1], 128);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kv_phase = 0;
      int qcount = 0;
      for (int w = blockIdx.x; w < P.n_items; w += gridDim.x) {
        const BwdItem it = decode_bwd(P, w);
        const BwdWalk wk = bwd_walk(P, it);
        if (wk.N == 0) continue;
        const SeqDesc& sd = P.seq[it.seq];
        if (!mbar_wait(&sh.kv_empty, kv_phase ^ 1, abort_flag, tmo, status)) break;
        kv_phase ^= 1;
        mbar_expect_tx(&sh.kv_full, 2 * C::kTileBytes);
        const int krow = sd.row_off + it.j * P.shard_stride + wk.b0;
        for (int d = 0; d < C::kSub; ++d) {
          tma_load_3d(smem + C::kOffK + d * kSubBytes, &tmK, &sh.kv_full, d * 64, it.hk, krow);
          tma_load_3d(smem + C::kOffV + d * kSubBytes, &tmV, &sh.kv_full, d * 64, it.hk, krow);
        }
        const bool ok = for_each_qtile(P, it, wk, [&](int r, int h, int q0) -> bool {
          const int st = qcount & 1;
          const uint32_t ph = (qcount >> 1) & 1;
          if (!mbar_wait(&sh.q_empty[st], ph ^ 1, abort_flag, tmo, status)) return false;
          mbar_expect_tx(&sh.q_full[st], 2 * C::kTileBytes);
          const int qrow = sd.row_off + r * P.shard_stride + q0;
          uint8_t* base = smem + C::kOffQ + st * C::kStageBytes;
          for (int d = 0; d < C::kSub; ++d) {
            tma_load_3d(base + d * kSubBytes, &tmQ, &sh.q_full[st], d * 64, h, qrow);
            tma_load_3d(base + C::kTileBytes + d * kSubBytes, &tmDO, &sh.q_full[st], d * 64, h, qrow);
          }
          ++qcount;
          return true;
        });
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t kv_phase = 0, af_phase = 0, p_phase = 0, ds_phase = 0, dqf_phase = 0;
      int qcount = 0;
      const uint32_t idSS = idesc_bf16_f32(128, 128, 0, 0);     // S^T, dP^T
      const uint32_t idKV = idesc_bf16_f32(128, DH, 0, 1);      // dV, dK: B MN-major
      const uint32_t idQ = idesc_bf16_f32(128, DH, 1, 1);       // dQ: A and B MN-major
      const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
      const uint32_t sQ0 = smem_u32(smem + C::kOffQ), sDS = smem_u32(smem + C::kOffDS);
      bool ok = true;
      for (int w = blockIdx.x; w < P.n_items && ok; w += gridDim.x) {
        const BwdItem it = decode_bwd(P, w);
        const BwdWalk wk = bwd_walk(P, it);
        if (wk.N == 0) continue;
        if (!(ok = mbar_wait(&sh.kv_full, kv_phase, abort_flag, tmo, status))) break;
        kv_phase ^= 1;
        // the previous item's dK / dV must be out of TMEM before accumulate = 0 overwrites
        if (!(ok = mbar_wait(&sh.acc_free, af_phase ^ 1, abort_flag, tmo, status))) break;
        af_phase ^= 1;
        tc_fence_after();
        int i = 0;
        ok = for_each_qtile(P, it, wk, [&](int, int, int) -> bool {
          const int st = qcount & 1;
          const uint32_t ph = (qcount >> 1) & 1;
          const uint32_t sQ = sQ0 + st * C::kStageBytes, sDO = sQ + C::kTileBytes;
          if (!mbar_wait(&sh.q_full[st], ph, abort_flag, tmo, status)) return false;
          tc_fence_after();
          // S^T = K Q^T
#pragma unroll
          for (int k = 0; k < C::kKSteps; ++k) {
            const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
            mma_ss(tmem + C::kColS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024),
                   idSS, k > 0);
          }
          tc_commit(&sh.s_full);
          // dP^T = V dO^T (its TMEM columns held the previous dQ)
          if (i > 0) {
            if (!mbar_wait(&sh.dq_free, dqf_phase, abort_flag, tmo, status)) return false;
            dqf_phase ^= 1;
            tc_fence_after();
          }
#pragma unroll
          for (int k = 0; k < C::kKSteps; ++k) {
            const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
            mma_ss(tmem + C::kColDP, sdesc_sw128(sV + off, 16, 1024),
                   sdesc_sw128(sDO + off, 16, 1024), idSS, k > 0);
          }
          tc_commit(&sh.dp_full);
          // dV += P^T dO
          if (!mbar_wait(&sh.p_full, p_phase, abort_flag, tmo, status)) return false;
          p_phase ^= 1;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + C::kColDV, tmem + C::kColS + 8 * k,
                   sdesc_sw128(sDO + k * 2048, kSubBytes, 1024), idKV, (i > 0 || k > 0) ? 1u : 0u);
          // dK += dS^T Q ; dQ = dS K
          if (!mbar_wait(&sh.ds_full, ds_phase, abort_flag, tmo, status)) return false;
          ds_phase ^= 1;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
            mma_ss(tmem + C::kColDK, sdesc_sw128(sDS + off, 16, 1024),
                   sdesc_sw128(sQ + k * 2048, kSubBytes, 1024), idKV, (i > 0 || k > 0) ? 1u : 0u);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ss(tmem + C::kColDP, sdesc_sw128(sDS + k * 2048, kSubBytes, 1024),
                   sdesc_sw128(sK + k * 2048, kSubBytes, 1024), idQ, k > 0);
          tc_commit(&sh.dq_full);
          tc_commit(&sh.ds_empty);
          tc_commit(&sh.q_empty[st]);
          ++qcount;
          ++i;
          return true;
        });
        if (!ok) break;
        tc_commit(&sh.acc_done);
        tc_commit(&sh.kv_empty);
        // the last dQ must be read before the next item's first dP reuses its columns
        if (!(ok = mbar_wait(&sh.dq_free, dqf_phase, abort_flag, tmo, status))) break;
        dqf_phase ^= 1;
      }
      tc_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, abort_flag, tmo, status);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------------ P / dS warpgroup
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // K/V row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS, tDP = tmem + lane_off + C::kColDP;
    const uint32_t tDK = tmem + lane_off + C::kColDK, tDV = tmem + lane_off + C::kColDV;
    float* lse_s = reinterpret_cast<float*>(smem + C::kOffLse);
    float* delta_s = reinterpret_cast<float*>(smem + C::kOffDelta);
    uint8_t* ds_tile = smem + C::kOffDS;
    const float sl2 = P.scale_log2;
    uint32_t s_phase = 0, dp_phase = 0, dse_phase = 0, ad_phase = 0;
    int iter = 0;
    for (int w = blockIdx.x; w < P.n_items; w += gridDim.x) {
      const BwdItem it = decode_bwd(P, w);
      const BwdWalk wk = bwd_walk(P, it);
      const SeqDesc& sd = P.seq[it.seq];
      const int b = wk.b0 + row;
      const bool validk = b < wk.L;
      const size_t krow = static_cast<size_t>(sd.row_off + it.j * P.shard_stride + b);
      if (wk.N == 0) {
        if (validk) {
          uint32_t z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
          for (int c = 0; c < DH / 32; ++c) {
            store_row32_bf16(dk + (krow * P.hkv + it.hk) * DH + c * 32, z, 0.f);
            store_row32_bf16(dv + (krow * P.hkv + it.hk) * DH + c * 32, z, 0.f);
          }
        }
        continue;
      }
      const int64_t pk = validk ? layout_pos(P.layout, P.D, wk.L, it.j, b) : 0;
      const bool ok = for_each_qtile(P, it, wk, [&](int r, int h, int q0) -> bool {
        // lse (log2 domain) and delta of the query tile, double-buffered in smem
        float* ls = lse_s + (iter & 1) * 128;
        float* dl = delta_s + (iter & 1) * 128;
        {
          const int a = q0 + row;
          if (a < wk.L) {
            const size_t li = sd.lse_off + static_cast<size_t>(h) * P.lse_hstride +
                              static_cast<size_t>(r) * P.shard_stride + a;
            ls[row] = lse[li] * kLog2e;
            dl[row] = delta[li];
          } else {
            ls[row] = INFINITY;  // rows beyond the piece: P = 0
            dl[row] = 0.f;
          }
        }
        // every thread of the warpgroup staged its value (bounded wait, no hang on abort)
        mbar_arrive(&sh.lse_bar[iter & 1]);
        if (!mbar_wait(&sh.lse_bar[iter & 1], (iter >> 1) & 1, abort_flag, tmo, status)) return false;
        ++iter;
        int lo = validk ? (P.causal ? first_query(P.layout, P.D, wk.L, r, pk) - q0 : 0) : 128;
        int hi = wk.L - q0;
        if (lo < 0) lo = 0;
        // P^T = 2^(S^T * scale * log2e - lse * log2e), masked; bf16 pairs over S columns
        if (!mbar_wait(&sh.s_full, s_phase, abort_flag, tmo, status)) return false;
        s_phase ^= 1;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rr[32], pk16[16];
          tmem_ld32(tS + c * 32, rr);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = c * 32 + 2 * i;
            const float p0 = (col >= lo && col < hi) ? ex2(fmaf(__uint_as_float(rr[2 * i]), sl2, -ls[col])) : 0.f;
            const float p1 = (col + 1 >= lo && col + 1 < hi) ? ex2(fmaf(__uint_as_float(rr[2 * i + 1]), sl2, -ls[col + 1])) : 0.f;
            pk16[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + c * 16, pk16);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sh.p_full);
        // dS^T = P^T * (dP^T - delta) -> bf16, 128B-swizzled K-major tile [K/V row][query]
        if (!mbar_wait(&sh.dp_full, dp_phase, abort_flag, tmo, status)) return false;
        dp_phase ^= 1;
        if (!mbar_wait(&sh.ds_empty, dse_phase ^ 1, abort_flag, tmo, status)) return false;
        dse_phase ^= 1;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t dp[32], pp[16];
          tmem_ld32(tDP + c * 32, dp);
          tmem_ld16(tS + c * 16, pp);
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = c * 32 + 2 * i;
            const __nv_bfloat162 pv = *reinterpret_cast<const __nv_bfloat162*>(&pp[i]);
            const float d0 = __low2float(pv) * (__uint_as_float(dp[2 * i]) - dl[col]);
            const float d1 = __high2float(pv) * (__uint_as_float(dp[2 * i + 1]) - dl[col + 1]);
            o[i] = pack_bf16x2(d0, d1);
          }
          // columns c*32 .. c*32+31 = four 16-byte chunks of sub-tile (c >> 1)
          uint8_t* rowp = ds_tile + (c >> 1) * kSubBytes + row * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = (c & 1) * 4 + q;
            uint4 v;
            v.x = o[4 * q + 0];
            v.y = o[4 * q + 1];
            v.z = o[4 * q + 2];
            v.w = o[4 * q + 3];
            *reinterpret_cast<uint4*>(rowp + ((chunk ^ (row & 7)) << 4)) = v;
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sh.ds_full);
        return true;
      });
      if (!ok) break;
      // dK (times scale) and dV of this tile
      if (!mbar_wait(&sh.acc_done, ad_phase, abort_flag, tmo, status)) break;
      ad_phase ^= 1;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tDK + c * 32, rr);
        if (validk) store_row32_bf16(dk + (krow * P.hkv + it.hk) * DH + c * 32, rr, P.scale);
        tmem_ld32(tDV + c * 32, rr);
        if (validk) store_row32_bf16(dv + (krow * P.hkv + it.hk) * DH + c * 32, rr, 1.f);
      }
      tc_fence_before();
      mbar_arrive(&sh.acc_free);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------------ dQ warpgroup
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row within the tile = TMEM lane
    const uint32_t tDQ = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + C::kColDP;
    uint32_t dqf_phase = 0;
    for (int w = blockIdx.x; w < P.n_items; w += gridDim.x) {
      const BwdItem it = decode_bwd(P, w);
      const BwdWalk wk = bwd_walk(P, it);
      if (wk.N == 0) continue;
      const SeqDesc& sd = P.seq[it.seq];
      const bool ok = for_each_qtile(P, it, wk, [&](int r, int h, int q0) -> bool {
        if (!mbar_wait(&sh.dq_full, dqf_phase, abort_flag, tmo, status)) return false;
        dqf_phase ^= 1;
        tc_fence_after();
        const int a = q0 + row;
        const bool valid = a < wk.L;
        float4* dst = reinterpret_cast<float4*>(
            dq_acc + (static_cast<size_t>(sd.row_off + r * P.shard_stride + a) * P.hq + h) * DH);
#pragma unroll
        for (int c = 0; c < DH / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(tDQ + c * 32, rr);
          if (valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              atomicAdd(dst + c * 8 + q,
                        make_float4(__uint_as_float(rr[4 * q]), __uint_as_float(rr[4 * q + 1]),
                                    __uint_as_float(rr[4 * q + 2]), __uint_as_float(rr[4 * q + 3])));
          }
        }
        tc_fence_before();
        mbar_arrive(&sh.dq_free);
        return true;
      });
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int DH>
cudaError_t launch_one(const Plan& P, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, const float* lse,
                       const float* delta, float* dq_acc, void* dk, void* dv, int n_sm,
                       cudaStream_t st) {
  using C = BwdCfg<DH>;
  auto kern = ring_bwd_tc_kernel<DH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = P.n_items < n_sm ? P.n_items : n_sm;
  kern<<<grid, kBwdThreads, C::kSmemBytes, st>>>(mq, mk, mv, mdo, P, lse, delta, dq_acc,
                                                 static_cast<__nv_bfloat16*>(dk),
                                                 static_cast<__nv_bfloat16*>(dv));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_tc(const Plan& P, const void* q, const void* k, const void* v,
                          const void* dout, const float* lse, const float* delta, float* dq_acc,
                          void* dk, void* dv, cudaStream_t st) {
  if (P.n_items == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv, mdo;
  cudaError_t e = make_token_tmap(&mq, q, P.n_rows, P.hq, P.head_dim);
  if (e == cudaSuccess) e = make_token_tmap(&mk, k, P.n_rows, P.hkv, P.head_dim);
  if (e == cudaSuccess) e = make_token_tmap(&mv, v, P.n_rows, P.hkv, P.head_dim);
  if (e == cudaSuccess) e = make_token_tmap(&mdo, dout, P.n_rows, P.hq, P.head_dim);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (P.head_dim == 128)
    return launch_one<128>(P, mq, mk, mv, mdo, lse, delta, dq_acc, dk, dv, n_sm, st);
  return launch_one<64>(P, mq, mk, mv, mdo, lse, delta, dq_acc, dk, dv, n_sm, st);
}

cudaError_t bwd_status(unsigned int* value, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_status_bwd, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_status_bwd, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace ra
