// ra_bwd_dq_tc.cu — the dq half of the deterministic ring-attention backward (sm_103a).
//
// The fused backward adds every (K/V tile, query tile) contribution to dq with float
// reductions, whose order varies from run to run. For `deterministic` problems (nanotron
// how-to page, "Calling the Ring Attention Function Directly": the `deterministic` flag)
// dq is instead computed query-tile-major: one CTA owns a 128-row query tile of one rank
// and one query head and walks the ring like the forward — step s = 0..D-1 against K/V
// shard (r - s) mod D, and of each shard only the K/V tiles some row may see — with dq
// accumulated in TMEM in a fixed order ("Backward Pass and Gradient Accumulation": dq
// accumulates over the steps on its own rank). dk and dv come from the K/V-tile kernel
// without its dq part, which writes each K/V row from one CTA, so the whole backward is
// free of atomics. Per K/V tile:
//
//   S  = Q K^T                 tcgen05 (SS), TMEM (two buffers)
//   P  = 2^(S*scale*log2e - lse*log2e)   one thread per query row, masked by key counts
//   dP = dO V^T                tcgen05 (SS), TMEM
//   dS = P * (dP - delta)      bf16, written over the tile's S buffer (columns [32, 96))
//   dQ += dS K                 tcgen05 (TS: dS from TMEM, K MN-major), f32 in TMEM
//
// MMA order: S(0) dP(0) S(1) | dP(1) dQ(0) S(2) | dP(2) dQ(1) S(3) | ...: once dS(n) is
// written, dP(n+1) goes first, so the softmax threads compute dS(n+1) (into the other S
// buffer) while dQ(n) runs, and S(n+2) is ready while dS(n+1) is computed. K stays in
// shared memory from S(n) to dQ(n), which now trails dP(n+1): three K stages let the load
// of K(n+2) start before dQ(n) ends. Items (query tiles) come from a counter in the
// caller's workspace, passed from the producer thread to the other roles through a two-slot
// ring in shared memory. Warp roles (384 threads): warp 0 TMA producer, warp 1 TMEM
// allocator + MMA issuer, warps 4-7 and 8-11 the P / dS warpgroups (thread = query row;
// key columns 0-63 and 64-127; they also write dq).
#include <cuda_runtime.h>

#include "ra_internal.h"
#include "ra_plan.h"
#include "ra_ptx.cuh"

namespace ra {

static __device__ unsigned int g_status_dq;

namespace {

constexpr int kDqThreads = 384;
// Of every 8 pairs of recomputed exponentials, this many are evaluated on the FMA pipe
// (exp2_poly2) and the rest on the MUFU unit.
#ifndef RA_DQ_POLY_PAIRS
#define RA_DQ_POLY_PAIRS 0
#endif
constexpr int kSubBytes = 128 * 128;
constexpr float kLog2e = 1.4426950408889634f;

template <int DH>
struct DqCfg {
  static constexpr int kSub = DH / 64;
  static constexpr int kTileBytes = 128 * DH * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTileBytes;
  static constexpr int kKStages = 3;  // K is held from S(n) to dQ(n), which trails dP(n+1)
  static constexpr int kOffK = 2 * kTileBytes;                // kKStages stages
  static constexpr int kOffV = kOffK + kKStages * kTileBytes; // 2 stages
  static constexpr int kOffBar = kOffV + 2 * kTileBytes;
  static constexpr int kSmemBytes = kOffBar + 256;
  static constexpr int kKSteps = DH / 16;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: S0 | S1 | dP | dQ
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColDP = 256, kColDQ = 384;
};

struct DqBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full[2], dp_full, ds_full[2], dq_done, dq_free;
  uint64_t drain;
  uint64_t item_full[2], item_empty[2];  // the CTA's item queue
  int item[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(DqBars) <= 256, "barrier block");
static_assert(DqCfg<128>::kSmemBytes <= 232448, "shared memory budget");

// Query-tile items: K/V heads outermost (CTAs that run together share K/V in L2), then
// the last query tile first (causal: it sees the most keys), then ranks, then the query
// heads of the group.
struct DqItem { int seq, h, r, qt; };

RA_HD int dq_items_of(const Plan& P, int L) { return ceil_div(L, kQTileRows) * plan_ranks(P) * P.hq; }

__device__ __forceinline__ DqItem decode_dq(const Plan& P, int w) {
  DqItem it;
  it.seq = find_seq(P, w);
  const SeqDesc& s = P.seq[it.seq];
  const int nqt = ceil_div(s.L, kQTileRows), nr = plan_ranks(P);
  int x = w - s.item_start;
  const int g = x % P.group;
  x /= P.group;
  it.r = P.rank_only >= 0 ? P.rank_only : x % nr;
  x /= nr;
  it.qt = nqt - 1 - x % nqt;
  const int hk = x / nqt;
  it.h = hk * P.group + g;
  return it;
}

__device__ __forceinline__ int dq_walk_tiles(const Plan& P, const DqItem& it, int L) {
  const int a_last = min(L, (it.qt + 1) * kQTileRows) - 1;
  int n = 0;
  for (int s = P.step_begin; s < P.step_end; ++s)
    n += kv_tiles_for(P, L, it.r, shard_at_step(P.D, it.r, s), a_last);
  return n;
}

// The CTA's item queue (two slots), as in the K/V-tile pass: the producer thread takes the
// next item from the shared counter (or by the static stride when there is none) and
// publishes it; the MMA thread and the softmax threads read it from the ring.
__device__ __forceinline__ int dq_item_publish(DqBars& sh, const Plan& P, int k,
                                               volatile int* abort_flag, uint64_t tmo,
                                               unsigned int* status) {
  const int slot = k & 1;
  if (!mbar_wait(&sh.item_empty[slot], ((k >> 1) & 1) ^ 1, abort_flag, tmo, status)) return -1;
  const int w = P.work_counter ? atomicAdd(P.work_counter, 1)
                               : static_cast<int>(blockIdx.x + static_cast<unsigned>(k) * gridDim.x);
  sh.item[slot] = w;
  mbar_arrive(&sh.item_full[slot]);
  return w;
}
__device__ __forceinline__ int dq_item_take(DqBars& sh, int k, volatile int* abort_flag,
                                            uint64_t tmo, unsigned int* status) {
  const int slot = k & 1;
  if (!mbar_wait(&sh.item_full[slot], (k >> 1) & 1, abort_flag, tmo, status)) return -1;
  const int w = *reinterpret_cast<volatile int*>(&sh.item[slot]);
  mbar_arrive(&sh.item_empty[slot]);
  return w;
}

template <int DH>
__global__ void __launch_bounds__(kDqThreads, 1)
    ring_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ Plan P,
                          const float* __restrict__ lse, const float* __restrict__ delta,
                          void* __restrict__ dq) {
  using C = DqCfg<DH>;
  extern __shared__ __align__(1024) uint8_t smem[];
  DqBars& sh = *reinterpret_cast<DqBars*>(smem + C::kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(&g_status_dq, 2u);
    return;
  }
  volatile int* abort_flag = &sh.abort_flag;
  unsigned int* status = &g_status_dq;
  const uint64_t tmo = P.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.v_empty[i], 1);
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.ds_full[i], 256);
    }
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.dq_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.item_full[i], 1);
      mbar_init(&sh.item_empty[i], 1 + 256);
    }
    mbar_init(&sh.dq_free, 256);
    mbar_init(&sh.drain, 1);
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
      uint32_t q_phase = 0;
      int kc = 0;
      for (int kq = 0;; ++kq) {
        const int w = dq_item_publish(sh, P, kq, abort_flag, tmo, status);
        if (w < 0 || w >= P.n_items) break;
        const DqItem it = decode_dq(P, w);
        const SeqDesc& sd = P.seq[it.seq];
        const int L = sd.L;
        const int N = dq_walk_tiles(P, it, L);
        if (N == 0) continue;
        if (!mbar_wait(&sh.q_empty, q_phase ^ 1, abort_flag, tmo, status)) break;
        q_phase ^= 1;
        mbar_expect_tx(&sh.q_full, 2 * C::kTileBytes);
        const int qrow = sd.row_off + it.r * P.shard_stride + it.qt * kQTileRows;
        for (int d = 0; d < C::kSub; ++d) {
          tma_load_3d(smem + C::kOffQ + d * kSubBytes, &tmQ, &sh.q_full, d * 64, it.h, qrow);
          tma_load_3d(smem + C::kOffDO + d * kSubBytes, &tmDO, &sh.q_full, d * 64, it.h, qrow);
        }
        const int hk = it.h / P.group;
        const int a_last = min(L, (it.qt + 1) * kQTileRows) - 1;
        bool ok = true;
        for (int s = P.step_begin; s < P.step_end && ok; ++s) {
          const int j = shard_at_step(P.D, it.r, s);
          const int nb = kv_tiles_for(P, L, it.r, j, a_last);
          const int krow = sd.row_off + j * P.shard_stride;
          for (int b = 0; b < nb; ++b, ++kc) {
            const int st = kc & 1;
            const uint32_t ph = (kc >> 1) & 1;
            const int kst = kc % C::kKStages;
            const uint32_t kph = (kc / C::kKStages) & 1;
            if (!(ok = mbar_wait(&sh.k_empty[kst], kph ^ 1, abort_flag, tmo, status))) break;
            mbar_expect_tx(&sh.k_full[kst], C::kTileBytes);
            for (int d = 0; d < C::kSub; ++d)
              tma_load_3d(smem + C::kOffK + kst * C::kTileBytes + d * kSubBytes, &tmK, &sh.k_full[kst],
                          d * 64, hk, krow + b * kKvTileRows);
            if (!(ok = mbar_wait(&sh.v_empty[st], ph ^ 1, abort_flag, tmo, status))) break;
            mbar_expect_tx(&sh.v_full[st], C::kTileBytes);
            for (int d = 0; d < C::kSub; ++d)
              tma_load_3d(smem + C::kOffV + st * C::kTileBytes + d * kSubBytes, &tmV, &sh.v_full[st],
                          d * 64, hk, krow + b * kKvTileRows);
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t q_phase = 0, dqf_phase = 0;
      uint32_t ds_phase[2] = {0, 0};
      int kc = 0;
      const uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);  // S, dP: A and B K-major
      const uint32_t idQ = idesc_bf16_f32(128, DH, 0, 1);   // dQ: A from TMEM, B MN-major
      const uint32_t sQ = smem_u32(smem + C::kOffQ), sDO = smem_u32(smem + C::kOffDO);
      const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
      bool ok = true;
      for (int kq = 0; ok; ++kq) {
        const int w = dq_item_take(sh, kq, abort_flag, tmo, status);
        if (w < 0) ok = false;
        if (w < 0 || w >= P.n_items) break;
        const DqItem it = decode_dq(P, w);
        const int N = dq_walk_tiles(P, it, P.seq[it.seq].L);
        if (N == 0) continue;
        if (!(ok = mbar_wait(&sh.q_full, q_phase, abort_flag, tmo, status))) break;
        q_phase ^= 1;
        tc_fence_after();
        auto issue_S = [&](int n) -> bool {
          const int c = kc + n, st = c % C::kKStages;
          if (!mbar_wait(&sh.k_full[st], (c / C::kKStages) & 1, abort_flag, tmo, status)) return false;
          tc_fence_after();
          const uint32_t ka = sK + st * C::kTileBytes;
#pragma unroll
          for (int k = 0; k < C::kKSteps; ++k) {
            const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
            mma_ss(tmem + (n & 1 ? C::kColS1 : C::kColS0), sdesc_sw128(sQ + off, 16, 1024),
                   sdesc_sw128(ka + off, 16, 1024), idS, k > 0);
          }
          tc_commit(&sh.s_full[n & 1]);
          return true;
        };
        auto issue_dP = [&](int n) -> bool {
          const int c = kc + n, st = c & 1;
          if (!mbar_wait(&sh.v_full[st], (c >> 1) & 1, abort_flag, tmo, status)) return false;
          tc_fence_after();
          const uint32_t va = sV + st * C::kTileBytes;
#pragma unroll
          for (int k = 0; k < C::kKSteps; ++k) {
            const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
            mma_ss(tmem + C::kColDP, sdesc_sw128(sDO + off, 16, 1024), sdesc_sw128(va + off, 16, 1024),
                   idS, k > 0);
          }
          tc_commit(&sh.dp_full);
          tc_commit(&sh.v_empty[st]);
          return true;
        };
        ok = issue_S(0) && issue_dP(0) && (N == 1 || issue_S(1));
        // the previous item's dq must be out of TMEM before the first dQ overwrites it
        if (ok) {
          ok = mbar_wait(&sh.dq_free, dqf_phase ^ 1, abort_flag, tmo, status);
          dqf_phase ^= 1;
          tc_fence_after();
        }
        for (int n = 0; n < N && ok; ++n) {
          const int c = kc + n, st = c % C::kKStages;
          if (!(ok = mbar_wait(&sh.ds_full[n & 1], ds_phase[n & 1], abort_flag, tmo, status))) break;
          ds_phase[n & 1] ^= 1;
          tc_fence_after();
          // dP(n+1) first: dP(n) has been read (ds_full), and dS(n+1) goes to the other S
          // buffer, so the softmax threads can compute it while dQ(n) runs
          if (n + 1 < N && !(ok = issue_dP(n + 1))) break;
          const uint32_t ka = sK + st * C::kTileBytes;
          const uint32_t tds = tmem + (n & 1 ? C::kColS1 : C::kColS0) + 32;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + C::kColDQ, tds + 8 * k, sdesc_sw128(ka + k * 2048, kSubBytes, 1024), idQ,
                   (n > 0 || k > 0) ? 1u : 0u);
          tc_commit(&sh.k_empty[st]);
          if (n + 2 < N) ok = issue_S(n + 2);
        }
        if (!ok) break;
        tc_commit(&sh.dq_done);
        tc_commit(&sh.q_empty);
        kc += N;
      }
      tc_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, abort_flag, tmo, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ P / dS warpgroups
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // query row within the tile = TMEM lane
    const int c0 = wg * 64;               // this warpgroup's key columns
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = P.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    uint32_t s_phase[2] = {0, 0}, dp_phase = 0, dd_phase = 0;
    for (int kq = 0;; ++kq) {
      const int w = dq_item_take(sh, kq, abort_flag, tmo, status);
      if (w < 0 || w >= P.n_items) break;
      const DqItem it = decode_dq(P, w);
      const SeqDesc& sd = P.seq[it.seq];
      const int L = sd.L;
      const int a = it.qt * kQTileRows + row;
      const bool valid = a < L;
      const size_t qrow = static_cast<size_t>(sd.row_off + it.r * P.shard_stride + a);
      const int N = dq_walk_tiles(P, it, L);
      if (N == 0) {  // no key visible: dq = 0 (nothing to add for bwd_accum)
        if (valid && !P.bwd_accum) {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(dq) + (qrow * P.hq + it.h) * DH;
#pragma unroll
          for (int c = wg * DH / 64; c < (wg + 1) * DH / 64; ++c) {
            uint4* d = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) d[q] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      float nl = -INFINITY, dl = 0.f;
      int64_t pq = 0;
      if (valid) {
        const size_t li = sd.lse_off + static_cast<size_t>(it.h) * P.lse_hstride +
                          static_cast<size_t>(it.r) * P.shard_stride + a;
        const float l = lse[li];
        nl = l == -INFINITY ? -INFINITY : -l * kLog2e;
        dl = delta[li];
        pq = layout_pos(P.layout, P.D, L, it.r, a);
      }
      const uint64_t nl2 = f2(nl, nl), dl2 = f2(dl, dl);
      const int a_last = min(L, (it.qt + 1) * kQTileRows) - 1;
      int n = 0;
      bool ok = true;
      for (int s = P.step_begin; s < P.step_end && ok; ++s) {
        const int j = shard_at_step(P.D, it.r, s);
        const int nb = kv_tiles_for(P, L, it.r, j, a_last);
        const int lim = !valid ? -1 : (P.causal ? key_limit(P.layout, P.D, L, j, pq) : L - 1);
        for (int b = 0; b < nb; ++b, ++n) {
          const int buf = n & 1;
          const uint32_t tS = tmem + lane_off + (buf ? C::kColS1 : C::kColS0);
          int cnt = lim + 1 - b * kKvTileRows;  // visible keys of this tile (a prefix)
          cnt = cnt < 0 ? 0 : (cnt > kKvTileRows ? kKvTileRows : cnt);
          if (!(ok = mbar_wait(&sh.s_full[buf], s_phase[buf], abort_flag, tmo, status))) break;
          s_phase[buf] ^= 1;
          tc_fence_after();
          uint32_t pp[32], sv2[2][32];
          tmem_ld32_nowait(tS + c0, sv2[0]);  // both chunks in flight, one wait
          tmem_ld32_nowait(tS + c0 + 32, sv2[1]);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const int cs = c0 + 32 * ch;
            const uint32_t (&sv)[32] = sv2[ch];
            const bool full = __all_sync(0xffffffffu, cnt >= cs + 32);
            // staged: every FMA, then every exponential, then masking and packing
            uint64_t xv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              xv[i] = fma2(f2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), sl2x2, nl2);
            float ev[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 e = f2_split((i & 7) < RA_DQ_POLY_PAIRS ? exp2_poly2(xv[i]) : xv[i]);
              ev[2 * i] = (i & 7) < RA_DQ_POLY_PAIRS ? e.x : ex2(e.x);  // poly: x <= 0 if visible
              ev[2 * i + 1] = (i & 7) < RA_DQ_POLY_PAIRS ? e.y : ex2(e.y);
            }
            if (!full) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (cs + i >= cnt) ev[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) pp[16 * ch + i] = pack_bf16x2(ev[2 * i], ev[2 * i + 1]);
          }
          if (!(ok = mbar_wait(&sh.dp_full, dp_phase, abort_flag, tmo, status))) break;
          dp_phase ^= 1;
          tc_fence_after();
          uint32_t dp2[2][32];
          tmem_ld32_nowait(tmem + lane_off + C::kColDP + c0, dp2[0]);
          tmem_ld32_nowait(tmem + lane_off + C::kColDP + c0 + 32, dp2[1]);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const uint32_t (&dp)[32] = dp2[ch];
            uint32_t o[16];
            uint64_t xv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              xv[i] = sub2(f2(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1])), dl2);
#pragma unroll
            for (int i = 0; i < 16; ++i) xv[i] = mul2(xv[i], f2_of_bf16x2(pp[16 * ch + i]));
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = bf16x2_of(xv[i]);
            // dS (bf16) into columns [32, 96) of this tile's S buffer (read into registers
            // above): the A operand of dQ += dS K
            tmem_st16(tS + 32 + c0 / 2 + 16 * ch, o);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&sh.ds_full[buf]);
        }
      }
      if (!ok) break;
      // dq = scale * dQ (or dq += scale * dQ into float32 sums for bwd_accum, the per-step
      // block backward): warpgroup 0 takes columns [0, DH/2), warpgroup 1 the rest
      if (!mbar_wait(&sh.dq_done, dd_phase, abort_flag, tmo, status)) break;
      dd_phase ^= 1;
      tc_fence_after();
      const size_t qoff = (qrow * P.hq + it.h) * DH;
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(dq) + qoff;
      float* dst_acc = static_cast<float*>(dq) + qoff;
#pragma unroll
      for (int c = 0; c < DH / 64; ++c) {
        const int col = wg * (DH / 2) + 32 * c;
        uint32_t rr[32];
        tmem_ld32(tmem + lane_off + C::kColDQ + col, rr);
        if (valid && P.bwd_accum) {
          float4* d = reinterpret_cast<float4*>(dst_acc + col);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 u = d[q];
            u.x += __uint_as_float(rr[4 * q + 0]) * P.scale;
            u.y += __uint_as_float(rr[4 * q + 1]) * P.scale;
            u.z += __uint_as_float(rr[4 * q + 2]) * P.scale;
            u.w += __uint_as_float(rr[4 * q + 3]) * P.scale;
            d[q] = u;
          }
        } else if (valid) {
          uint4* d = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(rr[8 * q + 0]) * P.scale, __uint_as_float(rr[8 * q + 1]) * P.scale);
            u.y = pack_bf16x2(__uint_as_float(rr[8 * q + 2]) * P.scale, __uint_as_float(rr[8 * q + 3]) * P.scale);
            u.z = pack_bf16x2(__uint_as_float(rr[8 * q + 4]) * P.scale, __uint_as_float(rr[8 * q + 5]) * P.scale);
            u.w = pack_bf16x2(__uint_as_float(rr[8 * q + 6]) * P.scale, __uint_as_float(rr[8 * q + 7]) * P.scale);
            d[q] = u;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sh.dq_free);
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
                       const float* delta, void* dq, int n_items, int n_sm, cudaStream_t st) {
  using C = DqCfg<DH>;
  auto kern = ring_bwd_dq_tc_kernel<DH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = n_items < n_sm ? n_items : n_sm;
  kern<<<grid, kDqThreads, C::kSmemBytes, st>>>(mq, mk, mv, mdo, P, lse, delta, dq);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_tc(const Plan& P0, const void* q, const void* k, const void* v,
                             const void* dout, const float* lse, const float* delta, void* dq,
                             cudaStream_t st) {
  Plan P = P0;  // re-number the items for query tiles; the next counter of the block
  P.work_counter = P0.work_counter ? P0.work_counter + 1 : nullptr;
  int items = 0;
  for (int i = 0; i < P.n_seqs; ++i) {
    P.seq[i].item_start = items;
    items += dq_items_of(P, P.seq[i].L);
  }
  P.n_items = items;
  if (items == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv, mdo;
  cudaError_t e = make_token_tmap(&mq, q, P.n_rows, P.hq, P.head_dim);
  if (e == cudaSuccess) e = make_token_tmap(&mk, k, P.n_rows, P.hkv, P.head_dim);
  if (e == cudaSuccess) e = make_token_tmap(&mv, v, P.n_rows, P.hkv, P.head_dim);
  if (e == cudaSuccess) e = make_token_tmap(&mdo, dout, P.n_rows, P.hq, P.head_dim);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (P.head_dim == 128) return launch_one<128>(P, mq, mk, mv, mdo, lse, delta, dq, items, n_sm, st);
  return launch_one<64>(P, mq, mk, mv, mdo, lse, delta, dq, items, n_sm, st);
}

cudaError_t bwd_dq_status(unsigned int* value, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_status_dq, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_status_dq, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace ra
