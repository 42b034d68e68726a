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
//   S^T  = K Q^T                 tcgen05 (SS), TMEM buffer X
//   P^T  = 2^(S^T*scale*log2e - lse*log2e)  (recomputed from lse, masked), bf16 -> X
//                                (columns [32, 96), over S^T columns already consumed)
//   dP^T = V dO^T                tcgen05 (SS), TMEM buffer Y
//   dV  += P^T dO                tcgen05 (TS: P^T from X), f32 in TMEM for the whole walk
//   dS^T = P^T * (dP^T - delta)  delta = rowsum(dO * O) from the preprocess kernel; bf16,
//                                written to a 128B-swizzled smem tile
//   dK  += dS^T Q                tcgen05 (SS: dS^T K-major), f32 in TMEM for the whole walk
//   dQ   = dS K                  tcgen05 (SS, dS read MN-major from smem) into Y, then
//                                added with vector float reductions into f32 dq sums
//
// With dQ the MMA warp issues, per query tile i: dV(i), dP(i), S(i+1), dK(i), dQ(i). P(i)
// stays in the registers of the threads that computed it, so X is free for S(i+1) as soon
// as dV(i) is issued, and the softmax threads compute P(i+1) while the tensor core runs
// dK(i) and dQ(i); the drain of dQ(i) overlaps dV(i+1). Without dQ the order is dK(i-1),
// dP(i), dV(i), S(i+1): dP(i) runs while P(i) is computed, S(i+1) while dS(i) is. The lse
// and delta of each query tile are staged in shared memory ahead of use by a loader warp.
// The items (K/V tiles) come from a counter in the caller's workspace, passed from the
// producer thread to the other roles through a two-slot ring in shared memory.
//
// Variants (template): kWithDQ = false leaves dq out (the K/V pass of the two-pass
// backward); kAccum = true adds float32 dk / dv into the outputs instead of storing them
// in the problem dtype (the per-step block backward of the unfused path).
//
// Warp roles (512 threads; 384 without dQ): warp 0 TMA producer (K, V once per item; Q and
// dO per query tile, two stages), warp 1 TMEM allocator + MMA issuer, warp 2 lse / delta
// loader, warps 4-7 and 8-11 the P / dS warpgroups (thread = K/V row; query columns 0-63
// and 64-127; at the end of an item they write dK and dV respectively), warps 12-15 the dQ
// warpgroup (thread = query row).
#include <cuda_runtime.h>

#include "ra_internal.h"
#include "ra_plan.h"
#include "ra_ptx.cuh"

namespace ra {

static __device__ unsigned int g_status_bwd;

namespace {

// Of every 8 pairs of recomputed exponentials, this many are evaluated on the FMA pipe
// (exp2_poly2) and the rest on the MUFU unit.
#ifndef RA_BWD_POLY_PAIRS
#define RA_BWD_POLY_PAIRS 0
#endif
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
  static constexpr int kOffLs = kOffDS + 2 * kSubBytes;      // [2 slots][-lse*log2e | delta][128]
  static constexpr int kOffBar = kOffLs + 2 * 2 * 128 * 4;
  static constexpr int kSmemBytes = kOffBar + 256;
  static constexpr int kKSteps = DH / 16;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColDK = 0, kColDV = DH, kColX = 2 * DH, kColY = 2 * DH + 128;
};

struct BwdBars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], do_full[2], q_empty[2];  // Q and dO of a stage land separately
  uint64_t ls_full[2], ls_empty[2];
  uint64_t s_full, p_full, dp_full, ds_full, dq_full, dq_free;
  uint64_t acc_done, drain;
  uint64_t item_full[2], item_empty[2];  // the CTA's item queue
  int item[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block");
static_assert(BwdCfg<128>::kSmemBytes <= 232448, "shared memory budget");

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
  for (int r = 0; r < P.D; ++r)
    if (rank_in_walk(P, it.j, r)) w.N += w.nqt - qt_begin(P, w, r);
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
    if (!rank_in_walk(P, it.j, r)) continue;
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

__device__ __forceinline__ void add_row32_f32(float* dst, const uint32_t (&r)[32], float mul) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float4 o = d[q];
    o.x += __uint_as_float(r[4 * q + 0]) * mul;
    o.y += __uint_as_float(r[4 * q + 1]) * mul;
    o.z += __uint_as_float(r[4 * q + 2]) * mul;
    o.w += __uint_as_float(r[4 * q + 3]) * mul;
    d[q] = o;
  }
}

// 8 x 8 transpose of 16-byte pieces inside each group of 8 lanes: on entry lane t of a
// group holds pieces 0..7 (r[4j..4j+3]) of its own row; on exit it holds piece t of the
// group's rows 0..7 (r[4j..4j+3] = piece t of row j). Three butterfly stages (lane
// distance 4, 2, 1): at distance s the lanes with bit s clear keep the pieces whose index
// has bit s clear and take the partner's, and the other lanes the reverse.
__device__ __forceinline__ void transpose8_f4(uint32_t (&r)[32], int t) {
#pragma unroll
  for (int s = 4; s >= 1; s >>= 1) {
    const bool hi = (t & s) != 0;
#pragma unroll
    for (int j0 = 0; j0 < 8; ++j0) {
      if (j0 & s) continue;
      const int j1 = j0 | s;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t send = hi ? r[4 * j0 + e] : r[4 * j1 + e];
        const uint32_t got = __shfl_xor_sync(0xffffffffu, send, s);
        if (hi) r[4 * j0 + e] = got;
        else r[4 * j1 + e] = got;
      }
    }
  }
}

// dS^T = P^T * (dP^T - delta) for the 32 query columns [c0 + 32*CH, +32) of this thread's
// K/V row, from their dP^T registers: the bf16 result goes to the 128B-swizzled smem tile
// [K/V row][query], the A operand of the dK MMA (K-major) and of the dQ MMA (MN-major).
// (Kept out of TMEM: MMAs that read an operand from TMEM slow down while the softmax
// warps load and store TMEM.)
template <int CH, bool kWithDQ>
__device__ __forceinline__ void ds_from(const uint32_t (&dp)[32], uint32_t tY, int c0, const float* dl,
                                        const uint32_t (&pp)[32], uint8_t* ds_row, int row) {
  const int cs = c0 + 32 * CH;
  uint32_t o[16];
  uint64_t xv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 d2 = *reinterpret_cast<const float2*>(dl + cs + 2 * i);
    xv[i] = sub2(f2(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1])), f2(d2.x, d2.y));
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) xv[i] = mul2(xv[i], f2_of_bf16x2(pp[16 * CH + i]));
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = bf16x2_of(xv[i]);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int chunk = 4 * CH + q;
    uint4 v;
    v.x = o[4 * q + 0];
    v.y = o[4 * q + 1];
    v.z = o[4 * q + 2];
    v.w = o[4 * q + 3];
    *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (row & 7)) << 4)) = v;
  }
}

// One chunk at a time.
template <int CH, bool kWithDQ>
__device__ __forceinline__ void ds_chunk(uint32_t tY, int c0, const float* dl,
                                         const uint32_t (&pp)[32], uint8_t* ds_row, int row) {
  uint32_t dp[32];
  tmem_ld32(tY + c0 + 32 * CH, dp);
  ds_from<CH, kWithDQ>(dp, tY, c0, dl, pp, ds_row, row);
}

// P^T = 2^(S^T * scale*log2e - lse*log2e) for the query columns [c0 + 32*CH, +32), from
// their S^T registers: columns before `lo` (queries that may not see this key) are zero;
// columns past the sequence piece have -lse*log2e = -inf from the loader and give 0. The
// bf16 result goes to X columns [32 + c0/2 + 16*CH, +16): inside the S^T columns this
// warpgroup reads itself (the other warpgroup may still be reading its own).
template <int CH>
__device__ __forceinline__ void p_from(const uint32_t (&sv)[32], uint32_t tX, int c0, const float* nl,
                                       uint64_t sl2x2, int lo, uint32_t (&pp)[32]) {
  const int cs = c0 + 32 * CH;
  uint32_t pk[16];
  const bool full = __all_sync(0xffffffffu, lo <= cs);
  // staged: every FMA, then every exponential, then masking and packing
  uint64_t xv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 n2 = *reinterpret_cast<const float2*>(nl + cs + 2 * i);
    xv[i] = fma2(f2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), sl2x2,
                 f2(n2.x, n2.y));
  }
  float ev[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {  // poly: visible entries have x <= 0; hidden ones are zeroed
    const float2 e = f2_split((i & 7) < RA_BWD_POLY_PAIRS ? exp2_poly2(xv[i]) : xv[i]);
    ev[2 * i] = (i & 7) < RA_BWD_POLY_PAIRS ? e.x : ex2(e.x);
    ev[2 * i + 1] = (i & 7) < RA_BWD_POLY_PAIRS ? e.y : ex2(e.y);
  }
  if (!full) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (cs + i < lo) ev[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    pk[i] = pack_bf16x2(ev[2 * i], ev[2 * i + 1]);
    pp[16 * CH + i] = pk[i];
  }
  tmem_st16(tX + 32 + c0 / 2 + 16 * CH, pk);
}

// One chunk at a time, on columns of a chunk this thread has already read (hence the
// per-warpgroup chunk order).
template <int CH>
__device__ __forceinline__ void p_chunk(uint32_t tX, int c0, const float* nl, uint64_t sl2x2,
                                        int lo, uint32_t (&pp)[32]) {
  uint32_t sv[32];
  tmem_ld32(tX + c0 + 32 * CH, sv);
  p_from<CH>(sv, tX, c0, nl, sl2x2, lo, pp);
}

// Threads per block: the dQ warpgroup only exists when dq is computed; without it the
// P / dS warpgroups get 170 registers a thread and load both of their chunks at once.
template <bool kWithDQ>
constexpr int bwd_threads() { return kWithDQ ? 512 : 384; }

// The CTA's item queue (two slots). The producer thread takes the next item, from the shared
// counter when there is one (dynamic: a CTA that finishes early takes more items, in index
// order, so the CTAs running together still hold neighbouring items), else by the static
// stride, and publishes it; every other role reads it from the ring, so all roles walk the
// same items. A value >= n_items ends the walk.
__device__ __forceinline__ int item_publish(BwdBars& sh, const Plan& P, int k,
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
__device__ __forceinline__ int item_take(BwdBars& sh, int k, volatile int* abort_flag,
                                         uint64_t tmo, unsigned int* status) {
  const int slot = k & 1;
  if (!mbar_wait(&sh.item_full[slot], (k >> 1) & 1, abort_flag, tmo, status)) return -1;
  const int w = *reinterpret_cast<volatile int*>(&sh.item[slot]);
  mbar_arrive(&sh.item_empty[slot]);
  return w;
}

template <int DH, bool kWithDQ, bool kAccum>
__global__ void __launch_bounds__(bwd_threads<kWithDQ>(), 1)
    ring_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ Plan P,
                       const float* __restrict__ lse, const float* __restrict__ delta,
                       float* __restrict__ dq_acc, void* __restrict__ dk_out,
                       void* __restrict__ dv_out) {
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
      mbar_init(&sh.do_full[i], 1);
      mbar_init(&sh.q_empty[i], 1);
      mbar_init(&sh.ls_full[i], 32);
      mbar_init(&sh.ls_empty[i], 256);
    }
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.p_full, 256);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.ds_full, 256);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_free, 128);
    mbar_init(&sh.acc_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.item_full[i], 1);
      mbar_init(&sh.item_empty[i], 1 + 32 + 256 + (kWithDQ ? 128 : 0));
    }
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
      uint32_t kv_phase = 0;
      int qcount = 0;
      for (int kq = 0;; ++kq) {
        const int w = item_publish(sh, P, kq, abort_flag, tmo, status);
        if (w < 0 || w >= P.n_items) break;
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
          // Q first, on its own barrier: S of this tile needs only Q, and is issued well
          // before dP needs dO
          const int qrow = sd.row_off + r * P.shard_stride + q0;
          uint8_t* base = smem + C::kOffQ + st * C::kStageBytes;
          mbar_expect_tx(&sh.q_full[st], C::kTileBytes);
          for (int d = 0; d < C::kSub; ++d)
            tma_load_3d(base + d * kSubBytes, &tmQ, &sh.q_full[st], d * 64, h, qrow);
          mbar_expect_tx(&sh.do_full[st], C::kTileBytes);
          for (int d = 0; d < C::kSub; ++d)
            tma_load_3d(base + C::kTileBytes + d * kSubBytes, &tmDO, &sh.do_full[st], d * 64, h, qrow);
          ++qcount;
          return true;
        });
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t kv_phase = 0, p_phase = 0, ds_phase = 0, dqf_phase = 0;
      int qc = 0;
      bool dq_pending = false;
      const uint32_t idSS = idesc_bf16_f32(128, 128, 0, 0);     // S^T, dP^T
      const uint32_t idKV = idesc_bf16_f32(128, DH, 0, 1);      // dV, dK: A from TMEM, B MN-major
      const uint32_t idQ = idesc_bf16_f32(128, DH, 1, 1);       // dQ: A and B MN-major
      const uint32_t sK = smem_u32(smem + C::kOffK), sV = smem_u32(smem + C::kOffV);
      const uint32_t sQ0 = smem_u32(smem + C::kOffQ), sDS = smem_u32(smem + C::kOffDS);
      const uint32_t tX = tmem + C::kColX, tY = tmem + C::kColY;
      auto issue_S = [&](uint32_t sQ) {
#pragma unroll
        for (int k = 0; k < C::kKSteps; ++k) {
          const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
          mma_ss(tX, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), idSS, k > 0);
        }
        tc_commit(&sh.s_full);
      };
      bool ok = true;
      for (int kq = 0; ok; ++kq) {
        const int w = item_take(sh, kq, abort_flag, tmo, status);
        if (w < 0) ok = false;
        if (w < 0 || w >= P.n_items) break;
        const BwdItem it = decode_bwd(P, w);
        const BwdWalk wk = bwd_walk(P, it);
        if (wk.N == 0) continue;
        if (!(ok = mbar_wait(&sh.kv_full, kv_phase, abort_flag, tmo, status))) break;
        kv_phase ^= 1;
        {
          const int st = qc & 1;
          if (!(ok = mbar_wait(&sh.q_full[st], (qc >> 1) & 1, abort_flag, tmo, status))) break;
          tc_fence_after();
          issue_S(sQ0 + st * C::kStageBytes);
        }
        int i = 0;
        if constexpr (!kWithDQ) {
          // Without dQ the order per tile is [dS(i-1)] dK(i-1), dP(i), [P(i)] dV(i), S(i+1):
          // dP(i) needs no P, so it runs while P(i) is computed, and S(i+1) runs while
          // dS(i) is computed.
          ok = for_each_qtile(P, it, wk, [&](int, int, int) -> bool {
            const int qi = qc + i;
            const int st = qi & 1;
            const uint32_t sQ = sQ0 + st * C::kStageBytes, sDO = sQ + C::kTileBytes;
            if (i > 0) {
              if (!mbar_wait(&sh.ds_full, ds_phase, abort_flag, tmo, status)) return false;
              ds_phase ^= 1;
              tc_fence_after();
              const uint32_t sQp = sQ0 + ((qi - 1) & 1) * C::kStageBytes;
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
                mma_ss(tmem + C::kColDK, sdesc_sw128(sDS + off, 16, 1024),
                       sdesc_sw128(sQp + k * 2048, kSubBytes, 1024), idKV, (i > 1 || k > 0) ? 1u : 0u);
              }
              tc_commit(&sh.q_empty[(qi - 1) & 1]);
            }
            if (!mbar_wait(&sh.do_full[st], (qi >> 1) & 1, abort_flag, tmo, status)) return false;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < C::kKSteps; ++k) {
              const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
              mma_ss(tY, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), idSS, k > 0);
            }
            tc_commit(&sh.dp_full);
            if (!mbar_wait(&sh.p_full, p_phase, abort_flag, tmo, status)) return false;
            p_phase ^= 1;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ts(tmem + C::kColDV, tX + 32 + 8 * k, sdesc_sw128(sDO + k * 2048, kSubBytes, 1024),
                     idKV, (i > 0 || k > 0) ? 1u : 0u);
            if (i + 1 < wk.N) {
              const int st1 = (qi + 1) & 1;
              if (!mbar_wait(&sh.q_full[st1], ((qi + 1) >> 1) & 1, abort_flag, tmo, status)) return false;
              tc_fence_after();
              issue_S(sQ0 + st1 * C::kStageBytes);
            }
            ++i;
            return true;
          });
          if (ok) {  // the last tile's dK
            const int ql = qc + wk.N - 1;
            ok = mbar_wait(&sh.ds_full, ds_phase, abort_flag, tmo, status);
            ds_phase ^= 1;
            tc_fence_after();
            const uint32_t sQl = sQ0 + (ql & 1) * C::kStageBytes;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
              mma_ss(tmem + C::kColDK, sdesc_sw128(sDS + off, 16, 1024),
                     sdesc_sw128(sQl + k * 2048, kSubBytes, 1024), idKV, (wk.N > 1 || k > 0) ? 1u : 0u);
            }
            tc_commit(&sh.q_empty[ql & 1]);
          }
          if (!ok) break;
          qc += wk.N;
          tc_commit(&sh.acc_done);
          tc_commit(&sh.kv_empty);
          continue;
        }
        ok = for_each_qtile(P, it, wk, [&](int, int, int) -> bool {
          const int qi = qc + i;
          const int st = qi & 1;
          const uint32_t sQ = sQ0 + st * C::kStageBytes, sDO = sQ + C::kTileBytes;
          // dV += P^T dO (P^T from X columns [32, 96)). dV is overwritten at the first tile:
          // the previous item's dK / dV were read by the P / dS threads before they
          // signalled P(0).
          if (!mbar_wait(&sh.do_full[st], (qi >> 1) & 1, abort_flag, tmo, status)) return false;
          if (!mbar_wait(&sh.p_full, p_phase, abort_flag, tmo, status)) return false;
          p_phase ^= 1;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + C::kColDV, tX + 32 + 8 * k, sdesc_sw128(sDO + k * 2048, kSubBytes, 1024),
                   idKV, (i > 0 || k > 0) ? 1u : 0u);
          // dP^T = V dO^T into Y, once the previous dQ has been read out of Y
          if (dq_pending) {
            if (!mbar_wait(&sh.dq_free, dqf_phase, abort_flag, tmo, status)) return false;
            dqf_phase ^= 1;
            dq_pending = false;
            tc_fence_after();
          }
#pragma unroll
          for (int k = 0; k < C::kKSteps; ++k) {
            const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
            mma_ss(tY, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), idSS, k > 0);
          }
          tc_commit(&sh.dp_full);
          // S(i+1) into X: P(i) has been read by dV(i) (issued above, executed in order)
          if (i + 1 < wk.N) {
            const int st1 = (qi + 1) & 1;
            if (!mbar_wait(&sh.q_full[st1], ((qi + 1) >> 1) & 1, abort_flag, tmo, status)) return false;
            tc_fence_after();
            issue_S(sQ0 + st1 * C::kStageBytes);
          }
          // dK += dS^T Q ; dQ = dS K into Y (dS^T from smem, K-major / MN-major)
          if (!mbar_wait(&sh.ds_full, ds_phase, abort_flag, tmo, status)) return false;
          ds_phase ^= 1;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
            mma_ss(tmem + C::kColDK, sdesc_sw128(sDS + off, 16, 1024),
                   sdesc_sw128(sQ + k * 2048, kSubBytes, 1024), idKV, (i > 0 || k > 0) ? 1u : 0u);
          }
          if constexpr (kWithDQ) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(tY, sdesc_sw128(sDS + k * 2048, kSubBytes, 1024),
                     sdesc_sw128(sK + k * 2048, kSubBytes, 1024), idQ, k > 0);
            tc_commit(&sh.dq_full);
            dq_pending = true;
          }
          tc_commit(&sh.q_empty[st]);
          ++i;
          return true;
        });
        if (!ok) break;
        qc += wk.N;
        tc_commit(&sh.acc_done);
        tc_commit(&sh.kv_empty);
      }
      tc_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, abort_flag, tmo, status);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ lse / delta loader
    float* ls_base = reinterpret_cast<float*>(smem + C::kOffLs);
    int t = 0;
    for (int kq = 0;; ++kq) {
      const int w = item_take(sh, kq, abort_flag, tmo, status);
      if (w < 0 || w >= P.n_items) break;
      const BwdItem it = decode_bwd(P, w);
      const BwdWalk wk = bwd_walk(P, it);
      if (wk.N == 0) continue;
      const SeqDesc& sd = P.seq[it.seq];
      const bool ok = for_each_qtile(P, it, wk, [&](int r, int h, int q0) -> bool {
        const int slot = t & 1;
        if (!mbar_wait(&sh.ls_empty[slot], ((t >> 1) & 1) ^ 1, abort_flag, tmo, status)) return false;
        float* nl = ls_base + slot * 256;
        const size_t li0 = sd.lse_off + static_cast<size_t>(h) * P.lse_hstride +
                           static_cast<size_t>(r) * P.shard_stride + q0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = lane + 32 * k;
          float n = -INFINITY, d = 0.f;
          if (q0 + c < wk.L) {
            const float l = lse[li0 + c];
            n = l == -INFINITY ? -INFINITY : -l * kLog2e;
            d = delta[li0 + c];
          }
          nl[c] = n;
          nl[128 + c] = d;
        }
        mbar_arrive(&sh.ls_full[slot]);
        ++t;
        return true;
      });
      if (!ok) break;
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------------ P / dS warpgroups
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // K/V row within the tile = TMEM lane
    const int c0 = wg * 64;               // this warpgroup's query columns
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tX = tmem + lane_off + C::kColX, tY = tmem + lane_off + C::kColY;
    const float* ls_base = reinterpret_cast<const float*>(smem + C::kOffLs);
    uint8_t* ds_row = smem + C::kOffDS + wg * kSubBytes + row * 128;
    const uint64_t sl2x2 = f2(P.scale_log2, P.scale_log2);
    uint32_t s_phase = 0, dp_phase = 0, ad_phase = 0;
    int t = 0;
    for (int kq = 0;; ++kq) {
      const int w = item_take(sh, kq, abort_flag, tmo, status);
      if (w < 0 || w >= P.n_items) break;
      const BwdItem it = decode_bwd(P, w);
      const BwdWalk wk = bwd_walk(P, it);
      const SeqDesc& sd = P.seq[it.seq];
      const int b = wk.b0 + row;
      const bool validk = b < wk.L;
      const size_t krow = static_cast<size_t>(sd.row_off + it.j * P.shard_stride + b);
      const size_t out_off = (krow * P.hkv + it.hk) * DH;
      if (wk.N == 0) {
        if constexpr (!kAccum) {
          if (validk) {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(wg == 0 ? dk_out : dv_out) + out_off;
#pragma unroll
            for (int c = 0; c < DH / 32; ++c) store_row32_bf16(dst + c * 32, z, 0.f);
          }
        }
        continue;
      }
      const int64_t pk = validk ? layout_pos(P.layout, P.D, wk.L, it.j, b) : 0;
      const bool ok = for_each_qtile(P, it, wk, [&](int r, int, int q0) -> bool {
        const int slot = t & 1;
        const int lo = validk ? (P.causal ? first_query(P.layout, P.D, wk.L, r, pk) - q0 : 0) : 128;
        if (!mbar_wait(&sh.ls_full[slot], (t >> 1) & 1, abort_flag, tmo, status)) return false;
        const float* nl = ls_base + slot * 256;
        const float* dl = nl + 128;
        // P^T into X (bf16), kept in registers for dS^T
        if (!mbar_wait(&sh.s_full, s_phase, abort_flag, tmo, status)) return false;
        s_phase ^= 1;
        tc_fence_after();
        uint32_t pp[32];
        if constexpr (!kWithDQ) {  // both chunks in registers before any write
          uint32_t s0[32], s1[32];
          tmem_ld32_nowait(tX + c0, s0);
          tmem_ld32_nowait(tX + c0 + 32, s1);
          tmem_wait_ld();
          p_from<0>(s0, tX, c0, nl, sl2x2, lo, pp);
          p_from<1>(s1, tX, c0, nl, sl2x2, lo, pp);
        } else if (wg == 0) {
          p_chunk<1>(tX, c0, nl, sl2x2, lo, pp);
          p_chunk<0>(tX, c0, nl, sl2x2, lo, pp);
        } else {
          p_chunk<0>(tX, c0, nl, sl2x2, lo, pp);
          p_chunk<1>(tX, c0, nl, sl2x2, lo, pp);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sh.p_full);
        // dS^T = P^T * (dP^T - delta). Each chunk's output lands on dP^T columns this thread
        // has already read, so the chunk order differs between the two warpgroups.
        if (!mbar_wait(&sh.dp_full, dp_phase, abort_flag, tmo, status)) return false;
        dp_phase ^= 1;
        tc_fence_after();
        if constexpr (!kWithDQ) {
          uint32_t d0[32], d1[32];
          tmem_ld32_nowait(tY + c0, d0);
          tmem_ld32_nowait(tY + c0 + 32, d1);
          tmem_wait_ld();
          ds_from<0, kWithDQ>(d0, tY, c0, dl, pp, ds_row, row);
          ds_from<1, kWithDQ>(d1, tY, c0, dl, pp, ds_row, row);
        } else if (wg == 0) {
          ds_chunk<1, kWithDQ>(tY, c0, dl, pp, ds_row, row);
          ds_chunk<0, kWithDQ>(tY, c0, dl, pp, ds_row, row);
        } else {
          ds_chunk<0, kWithDQ>(tY, c0, dl, pp, ds_row, row);
          ds_chunk<1, kWithDQ>(tY, c0, dl, pp, ds_row, row);
        }
        mbar_arrive(&sh.ls_empty[slot]);
        ++t;
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sh.ds_full);
        return true;
      });
      if (!ok) break;
      // dK (times scale; warpgroup 0) and dV (warpgroup 1) of this tile
      if (!mbar_wait(&sh.acc_done, ad_phase, abort_flag, tmo, status)) break;
      ad_phase ^= 1;
      tc_fence_after();
      const uint32_t tacc = tmem + lane_off + (wg == 0 ? C::kColDK : C::kColDV);
      const float mul = wg == 0 ? P.scale : 1.f;
#pragma unroll
      for (int c = 0; c < DH / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(tacc + c * 32, rr);
        if (validk) {
          if constexpr (kAccum)
            add_row32_f32(static_cast<float*>(wg == 0 ? dk_out : dv_out) + out_off + c * 32, rr, mul);
          else
            store_row32_bf16(static_cast<__nv_bfloat16*>(wg == 0 ? dk_out : dv_out) + out_off + c * 32,
                             rr, mul);
        }
      }
      tc_fence_before();
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------------ dQ warpgroup
    if constexpr (kWithDQ) {
      const int quarter = warp & 3;  // TMEM lanes = query rows quarter*32 .. +31
      const uint32_t tQ = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + C::kColY;
      const float mul = P.dq_mul;
      uint32_t dqf_phase = 0;
      for (int kq = 0;; ++kq) {
        const int w = item_take(sh, kq, abort_flag, tmo, status);
        if (w < 0 || w >= P.n_items) break;
        const BwdItem it = decode_bwd(P, w);
        const BwdWalk wk = bwd_walk(P, it);
        if (wk.N == 0) continue;
        const SeqDesc& sd = P.seq[it.seq];
        const bool ok = for_each_qtile(P, it, wk, [&](int r, int h, int q0) -> bool {
          if (!mbar_wait(&sh.dq_full, dqf_phase, abort_flag, tmo, status)) return false;
          dqf_phase ^= 1;
          tc_fence_after();
          // Lane 8g + t ends up with 16-byte piece t of rows 8g .. 8g+7 of its warp's 32
          // rows, so each reduction instruction covers four rows x 128 contiguous bytes.
          const int t8 = lane & 7;
          const int row0 = q0 + quarter * 32 + (lane & ~7);  // first row of this lane's group
          const size_t base = static_cast<size_t>(sd.row_off + r * P.shard_stride);
#pragma unroll
          for (int c = 0; c < DH / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(tQ + c * 32, rr);
            if (c == DH / 32 - 1) {  // every column of Y has been read: release it
              tc_fence_before();
              mbar_arrive(&sh.dq_free);
            }
            transpose8_f4(rr, t8);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int a = row0 + j;
              if (a < wk.L) {
                float* dst = dq_acc + ((base + a) * P.hq + h) * DH + c * 32 + 4 * t8;
                red_add_v4(dst, __uint_as_float(rr[4 * j]) * mul, __uint_as_float(rr[4 * j + 1]) * mul,
                           __uint_as_float(rr[4 * j + 2]) * mul, __uint_as_float(rr[4 * j + 3]) * mul);
              }
            }
          }
          return true;
        });
        if (!ok) break;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int DH, bool kWithDQ, bool kAccum>
cudaError_t launch_one(const Plan& P, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, const CUtensorMap& mdo, const float* lse,
                       const float* delta, float* dq_acc, void* dk, void* dv, int n_sm,
                       cudaStream_t st) {
  using C = BwdCfg<DH>;
  auto kern = ring_bwd_tc_kernel<DH, kWithDQ, kAccum>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = P.n_items < n_sm ? P.n_items : n_sm;
  kern<<<grid, bwd_threads<kWithDQ>(), C::kSmemBytes, st>>>(mq, mk, mv, mdo, P, lse, delta, dq_acc,
                                                            dk, dv);
  return cudaGetLastError();
}

template <bool kWithDQ, bool kAccum>
cudaError_t launch_dh(const Plan& P, const CUtensorMap& mq, const CUtensorMap& mk,
                      const CUtensorMap& mv, const CUtensorMap& mdo, const float* lse,
                      const float* delta, float* dq_acc, void* dk, void* dv, int n_sm,
                      cudaStream_t st) {
  if (P.head_dim == 128)
    return launch_one<128, kWithDQ, kAccum>(P, mq, mk, mv, mdo, lse, delta, dq_acc, dk, dv, n_sm, st);
  return launch_one<64, kWithDQ, kAccum>(P, mq, mk, mv, mdo, lse, delta, dq_acc, dk, dv, n_sm, st);
}

}  // namespace

cudaError_t launch_bwd_tc(const Plan& P, BwdKind kind, const void* q, const void* k, const void* v,
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
  switch (kind) {
    case BwdKind::kFused:
      return launch_dh<true, false>(P, mq, mk, mv, mdo, lse, delta, dq_acc, dk, dv, n_sm, st);
    case BwdKind::kKvOnly:
      return launch_dh<false, false>(P, mq, mk, mv, mdo, lse, delta, dq_acc, dk, dv, n_sm, st);
    case BwdKind::kBlockAccum:
      return launch_dh<true, true>(P, mq, mk, mv, mdo, lse, delta, dq_acc, dk, dv, n_sm, st);
    case BwdKind::kKvAccum:
      return launch_dh<false, true>(P, mq, mk, mv, mdo, lse, delta, dq_acc, dk, dv, n_sm, st);
  }
  return cudaErrorInvalidValue;
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
