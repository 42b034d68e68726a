// ra_fwd_tc.cu — fused ring-attention forward on the 5th-generation tensor cores (sm_103a).
//
// One persistent CTA per SM takes work items (256 query rows of one rank and one query
// head) and walks the ring: for step s = begin..end-1 it reads the K/V shard
// j = (r - s) mod D (Ring Attention concept page, "Sequence sharding and the ring
// topology") and, of that shard, only the 128-row K/V tiles that some query of the block
// may see under the global-position causal rule ("Watch Out For"). For each tile:
//
//   S = Q K^T          tcgen05.mma, Q and K tiles TMA-loaded into 128B-swizzled smem,
//                      S (128 x 128 f32) accumulated in TMEM
//   online softmax     two threads per query row (64 columns each) read the S row from
//                      TMEM, mask the columns beyond the key count, update the running max
//                      m and denominator l, write P = 2^(S*scale*log2e - m) as bf16 back
//                      into TMEM over consumed S columns
//   O += P V           tcgen05.mma with A = P from TMEM, B = V tile (MN-major) from smem
//
// The running (m, l, O) persists across all tiles and all ring steps of the block, which
// is the log-sum-exp merge of update_out_and_lse (nanotron how-to page, "Numerically-
// Stable Output Fusion"; interview question page: rescale the old partial by
// exp(old_max - new_max)) fused into the tile loop. O is rescaled only when a row max grows
// by more than 2^8: with a stale reference value every exponent stays <= 2^8, and the final
// out = O / l and lse = m + log l are the same quantities (an exact identity, not an
// approximation). Finally out = O / l (bf16, or f32 for block outputs) and lse (natural
// log, f32) are written; a row that saw no key gets out = 0, lse = -inf.
//
// Warp roles (640 threads): warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 4-11 = softmax of query tile 0, warps 12-19 = softmax of query tile 1. Each tile's
// rows are split between two warpgroups of 64 key columns, which exchange their partial
// row maxima every K/V tile and their partial sums at the end through shared memory; P
// goes to S columns [32, 96), each half on its own S columns. The two tiles ping-pong: the
// MMA order S0(n) S1(n) | O0(n) S0(n+1) O1(n) S1(n+1) | ... lets one tile's softmax run
// while the tensor core works on the other tile.
#include <cuda_runtime.h>

#include "ra_internal.h"
#include "ra_plan.h"
#include "ra_ptx.cuh"

namespace ra {

static __device__ unsigned int g_status_fwd;

namespace {

constexpr int kFwdThreads = 640;  // 4 control warps + 4 softmax warpgroups (2 per query tile)
constexpr int kSubBytes = 128 * 128;  // 128 rows x 64 bf16: one 128B-swizzled sub-tile

template <int DH>
struct FwdCfg {
  static constexpr int kStages = DH == 128 ? 2 : 4;
  static constexpr int kSub = DH / 64;
  static constexpr int kTileBytes = 128 * DH * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kSmemBytes = kOffV + kStages * kTileBytes + 1024;
  static constexpr int kKSteps = DH / 16;
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: S0 | S1 | O0 | O1 (P of tile t overwrites the first 64 columns of S_t)
  __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __device__ static constexpr uint32_t col_o(int t) { return t ? 256u + DH : 256u; }
};

struct FwdShared {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t drain;
  uint64_t xmax_bar[2][2], xl_bar[2];  // half-row exchanges: [tile][slot], [tile]
  uint64_t item_full[2], item_empty[2];  // the CTA's item queue
  int item[2];
  uint32_t tmem_base;
  int abort_flag;
  float xmax[2][2][2][128];  // [tile][slot][half][row]: partial row maxima
  float xl[2][2][128];       // [tile][half][row]: partial row sums
};

// Total K/V tiles a forward item walks, and its first/last valid query rows.
struct FwdWalk {
  int L, a0, a_last, N;
  bool two;
};

__device__ __forceinline__ FwdWalk fwd_walk(const Plan& P, const FwdItem& it) {
  FwdWalk w;
  w.L = P.seq[it.seq].L;
  w.a0 = it.blk * kFwdBlockRows;
  const int a_end = min(w.L, w.a0 + kFwdBlockRows);
  w.a_last = a_end - 1;
  w.two = (a_end - w.a0) > kQTileRows;
  w.N = 0;
  for (int s = P.step_begin; s < P.step_end; ++s)
    w.N += kv_tiles_for(P, w.L, it.r, shard_at_step(P.D, it.r, s), w.a_last);
  return w;
}

template <typename OutT>
__device__ __forceinline__ void store_row32(OutT* dst, const float (&v)[32]);

template <>
__device__ __forceinline__ void store_row32<__nv_bfloat16>(__nv_bfloat16* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    d[q] = u;
  }
}
template <>
__device__ __forceinline__ void store_row32<float>(float* dst, const float (&v)[32]) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// The CTA's item queue (two slots): the producer thread takes the next item from the shared
// counter when the caller passed a workspace (a CTA that finishes early takes more items,
// in index order), else by the static stride, and publishes it; the MMA thread and the
// softmax threads read it from the ring. A value >= n_items ends the walk.
__device__ __forceinline__ int fwd_item_publish(FwdShared& sh, const Plan& P, int k,
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
__device__ __forceinline__ int fwd_item_take(FwdShared& sh, int k, volatile int* abort_flag,
                                             uint64_t tmo, unsigned int* status) {
  const int slot = k & 1;
  if (!mbar_wait(&sh.item_full[slot], (k >> 1) & 1, abort_flag, tmo, status)) return -1;
  const int w = *reinterpret_cast<volatile int*>(&sh.item[slot]);
  mbar_arrive(&sh.item_empty[slot]);
  return w;
}

template <int DH, typename OutT>
__global__ void __launch_bounds__(kFwdThreads, 1)
    ring_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ Plan P,
                       OutT* __restrict__ out, float* __restrict__ lse) {
  using C = FwdCfg<DH>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh.abort_flag;
  unsigned int* status = &g_status_fwd;
  const uint64_t tmo = P.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(&sh.q_full, 1);
    mbar_init(&sh.q_empty, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&sh.k_full[i], 1);
      mbar_init(&sh.k_empty[i], 1);
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sh.s_full[t], 1);
      mbar_init(&sh.p_full[t], 256);
      mbar_init(&sh.o_done[t], 1);
      mbar_init(&sh.o_free[t], 256);
      mbar_init(&sh.xmax_bar[t][0], 256);
      mbar_init(&sh.xmax_bar[t][1], 256);
      mbar_init(&sh.xl_bar[t], 256);
    }
    mbar_init(&sh.drain, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.item_full[i], 1);
      mbar_init(&sh.item_empty[i], 1 + (kFwdThreads - 128));  // MMA thread + softmax warps
    }
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
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
      int kv_count = 0;
      uint32_t q_phase = 0;
      for (int kq = 0;; ++kq) {
        const int w = fwd_item_publish(sh, P, kq, abort_flag, tmo, status);
        if (w < 0 || w >= P.n_items) break;
        const FwdItem it = decode_fwd(P, w);
        const FwdWalk wk = fwd_walk(P, it);
        if (wk.N == 0) continue;
        const SeqDesc& sd = P.seq[it.seq];
        if (!mbar_wait(&sh.q_empty, q_phase ^ 1, abort_flag, tmo, status)) goto producer_done;
        q_phase ^= 1;
        mbar_expect_tx(&sh.q_full, (wk.two ? 2 : 1) * C::kTileBytes);
        {
          const int qrow = sd.row_off + it.r * P.shard_stride + wk.a0;
          for (int t = 0; t < (wk.two ? 2 : 1); ++t)
            for (int d = 0; d < C::kSub; ++d)
              tma_load_3d(smem + C::kOffQ + t * C::kTileBytes + d * kSubBytes, &tmQ, &sh.q_full,
                          d * 64, it.h, qrow + t * kQTileRows);
        }
        const int hk = it.h / P.group;
        for (int s = P.step_begin; s < P.step_end; ++s) {
          const int j = shard_at_step(P.D, it.r, s);
          const int nb = kv_tiles_for(P, wk.L, it.r, j, wk.a_last);
          const int krow = sd.row_off + j * P.shard_stride;
          for (int b = 0; b < nb; ++b, ++kv_count) {
            const int st = kv_count % C::kStages;
            const uint32_t ph = (kv_count / C::kStages) & 1;
            if (!mbar_wait(&sh.k_empty[st], ph ^ 1, abort_flag, tmo, status)) goto producer_done;
            mbar_expect_tx(&sh.k_full[st], C::kTileBytes);
            for (int d = 0; d < C::kSub; ++d)
              tma_load_3d(smem + C::kOffK + st * C::kTileBytes + d * kSubBytes, &tmK,
                          &sh.k_full[st], d * 64, hk, krow + b * kKvTileRows);
            if (!mbar_wait(&sh.v_empty[st], ph ^ 1, abort_flag, tmo, status)) goto producer_done;
            mbar_expect_tx(&sh.v_full[st], C::kTileBytes);
            for (int d = 0; d < C::kSub; ++d)
              tma_load_3d(smem + C::kOffV + st * C::kTileBytes + d * kSubBytes, &tmV,
                          &sh.v_full[st], d * 64, hk, krow + b * kKvTileRows);
          }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int kv_count = 0;
      uint32_t q_phase = 0, p_phase[2] = {0, 0}, of_phase[2] = {0, 0};
      const uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);
      const uint32_t idO = idesc_bf16_f32(128, DH, 0, 1);
      const uint32_t sQ = smem_u32(smem + C::kOffQ);
      const uint32_t sK = smem_u32(smem + C::kOffK);
      const uint32_t sV = smem_u32(smem + C::kOffV);
      bool ok = true;
      for (int kq = 0; ok; ++kq) {
        const int w = fwd_item_take(sh, kq, abort_flag, tmo, status);
        if (w < 0) ok = false;
        if (w < 0 || w >= P.n_items) break;
        const FwdItem it = decode_fwd(P, w);
        const FwdWalk wk = fwd_walk(P, it);
        const int N = wk.N;
        if (N == 0) continue;
        const int nt = wk.two ? 2 : 1;
        if (!(ok = mbar_wait(&sh.q_full, q_phase, abort_flag, tmo, status))) break;
        q_phase ^= 1;
        tc_fence_after();
        auto issue_S = [&](int t, int n) -> bool {
          const int c = kv_count + n;
          const int st = c % C::kStages;
          const uint32_t ph = (c / C::kStages) & 1;
          if (t == 0) {
            if (!mbar_wait(&sh.k_full[st], ph, abort_flag, tmo, status)) return false;
            tc_fence_after();
          }
          const uint32_t qa = sQ + t * C::kTileBytes, ka = sK + st * C::kTileBytes;
#pragma unroll
          for (int k = 0; k < C::kKSteps; ++k) {
            const uint32_t off = (k >> 2) * kSubBytes + (k & 3) * 32;
            mma_ss(tmem + C::col_s(t), sdesc_sw128(qa + off, 16, 1024),
                   sdesc_sw128(ka + off, 16, 1024), idS, k > 0);
          }
          tc_commit(&sh.s_full[t]);
          if (t == nt - 1) tc_commit(&sh.k_empty[st]);
          return true;
        };
        auto issue_O = [&](int t, int n) -> bool {
          const int c = kv_count + n;
          const int st = c % C::kStages;
          const uint32_t ph = (c / C::kStages) & 1;
          if (t == 0) {
            if (!mbar_wait(&sh.v_full[st], ph, abort_flag, tmo, status)) return false;
          }
          if (!mbar_wait(&sh.p_full[t], p_phase[t], abort_flag, tmo, status)) return false;
          p_phase[t] ^= 1;
          if (n == 0) {
            if (!mbar_wait(&sh.o_free[t], of_phase[t] ^ 1, abort_flag, tmo, status)) return false;
            of_phase[t] ^= 1;
          }
          tc_fence_after();
          const uint32_t va = sV + st * C::kTileBytes;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts(tmem + C::col_o(t), tmem + C::col_s(t) + 32 + 8 * k,
                   sdesc_sw128(va + k * 2048, kSubBytes, 1024), idO, (n > 0 || k > 0) ? 1u : 0u);
          if (n == N - 1) tc_commit(&sh.o_done[t]);
          if (t == nt - 1) tc_commit(&sh.v_empty[st]);
          return true;
        };
        ok = issue_S(0, 0) && (nt == 1 || issue_S(1, 0));
        for (int n = 0; n < N && ok; ++n) {
          ok = issue_O(0, n) && (n + 1 >= N || issue_S(0, n + 1));
          if (ok && nt == 2) ok = issue_O(1, n) && (n + 1 >= N || issue_S(1, n + 1));
        }
        tc_commit(&sh.q_empty);
        kv_count += N;
      }
      // let every MMA issued so far finish before TMEM is released
      tc_commit(&sh.drain);
      mbar_wait(&sh.drain, 0, abort_flag, tmo, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax + epilogue
    // Query tile t = (warp - 4) / 8; its rows are split in two halves of 64 key columns
    // (hf), each held by one warpgroup; the halves exchange partial maxima per tile and
    // partial sums at the end through shared memory (bounded mbarrier waits).
    const int t = (warp - 4) >> 3;
    const int hf = ((warp - 4) >> 2) & 1;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int c0 = hf * 64;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::col_s(t);
    const uint32_t tO = tmem + lane_off + C::col_o(t);
    const float sl2 = P.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    uint32_t s_phase = 0, od_phase = 0, xl_phase = 0;
    uint32_t xm_phase[2] = {0, 0};
    int xn = 0;  // max exchanges done (slot = xn & 1)
    for (int kq = 0;; ++kq) {
      const int w = fwd_item_take(sh, kq, abort_flag, tmo, status);
      if (w < 0 || w >= P.n_items) break;
      const FwdItem it = decode_fwd(P, w);
      const FwdWalk wk = fwd_walk(P, it);
      if (t == 1 && !wk.two) continue;
      const SeqDesc& sd = P.seq[it.seq];
      const int a = wk.a0 + t * kQTileRows + row;
      const bool valid = a < wk.L;
      const int orow = sd.row_off + it.r * P.shard_stride + a;
      OutT* orow_ptr = out + (static_cast<size_t>(orow) * P.hq + it.h) * DH;
      float* lse_ptr = lse + sd.lse_off + static_cast<size_t>(it.h) * P.lse_hstride +
                       static_cast<size_t>(it.r) * P.shard_stride + a;
      if (wk.N == 0) {  // a block with no visible key at these steps
        if (valid) {
          float z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0.f;
#pragma unroll
          for (int c = 0; c < DH / 64; ++c) store_row32<OutT>(orow_ptr + hf * (DH / 2) + c * 32, z);
          if (hf == 0) *lse_ptr = -INFINITY;
        }
        continue;
      }
      const int64_t pq = valid ? layout_pos(P.layout, P.D, wk.L, it.r, a) : 0;
      float m = -INFINITY, l = 0.f;
      int n = 0;
      bool ok = true;
      for (int s = P.step_begin; s < P.step_end && ok; ++s) {
        const int j = shard_at_step(P.D, it.r, s);
        const int nb = kv_tiles_for(P, wk.L, it.r, j, wk.a_last);
        const int lim = !valid ? -1 : (P.causal ? key_limit(P.layout, P.D, wk.L, j, pq) : wk.L - 1);
        for (int b = 0; b < nb; ++b, ++n) {
          if (!(ok = mbar_wait(&sh.s_full[t], s_phase, abort_flag, tmo, status))) break;
          s_phase ^= 1;
          tc_fence_after();
          int cnt = lim + 1 - b * kKvTileRows;
          cnt = cnt < 0 ? 0 : (cnt > kKvTileRows ? kKvTileRows : cnt);
          const bool full = __all_sync(0xffffffffu, cnt == kKvTileRows);  // no mask needed
          // pass 1: partial row max over this half's visible columns, then both halves'
          uint32_t r2[2][32];
          tmem_ld32_nowait(tS + c0, r2[0]);
          tmem_ld32_nowait(tS + c0 + 32, r2[1]);
          tmem_wait_ld();
          float mx;
          {  // four independent max chains (one chain of 32 dependent max ops is slow)
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (full) {
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                  mq[2 * h] = max3(mq[2 * h], __uint_as_float(r2[h][i]), __uint_as_float(r2[h][i + 1]));
                  mq[2 * h + 1] =
                      max3(mq[2 * h + 1], __uint_as_float(r2[h][i + 2]), __uint_as_float(r2[h][i + 3]));
                }
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const float v = (c0 + 32 * h + i < cnt) ? __uint_as_float(r2[h][i]) : -INFINITY;
                  mq[2 * h + (i & 1)] = fmaxf(mq[2 * h + (i & 1)], v);
                }
            }
            mx = fmaxf(max3(mq[0], mq[1], mq[2]), mq[3]);
          }
          {
            const int slot = xn & 1;
            sh.xmax[t][slot][hf][row] = mx;
            mbar_arrive(&sh.xmax_bar[t][slot]);
            if (!(ok = mbar_wait(&sh.xmax_bar[t][slot], xm_phase[slot], abort_flag, tmo, status))) break;
            xm_phase[slot] ^= 1;
            mx = fmaxf(mx, sh.xmax[t][slot][hf ^ 1][row]);
            ++xn;
          }
          mx *= sl2;
          const float m_new = fmaxf(m, mx);
          const bool grow = m_new > m + 8.f;  // also true for the first visible key
          const bool need = grow && n > 0 && m != -INFINITY;
          if (__any_sync(0xffffffffu, need)) {  // rescale this half's output columns
            const float alpha = need ? ex2(m - m_new) : 1.f;
#pragma unroll
            for (int c = 0; c < DH / 64; ++c) {
              uint32_t r[32];
              tmem_ld32(tO + hf * (DH / 2) + c * 32, r);
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tmem_st32(tO + hf * (DH / 2) + c * 32, r);
            }
            if (need) l *= alpha;
          }
          if (grow) m = m_new;
          const float mref = (m == -INFINITY) ? 0.f : m;
          // pass 2: P = 2^(S*scale*log2e - m) as bf16 pairs into S columns [32 + c0/2, +32),
          // inside this half's own S columns; both chunks are in registers before any P is
          // written.
          const uint64_t nm2 = f2(-mref, -mref);
          uint64_t l2 = f2(0.f, 0.f);
          uint32_t rr[2][32];
          tmem_ld32_nowait(tS + c0, rr[0]);
          tmem_ld32_nowait(tS + c0 + 32, rr[1]);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const int cs = c0 + 32 * ch;
            uint32_t (&r)[32] = rr[ch];
            uint32_t pk[16];
            // staged: every FMA, then every exponential (independent, so they issue back to
            // back), then packing and two partial sums
            uint64_t xv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              xv[i] = fma2(f2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sl2x2, nm2);
            float ev[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 e = f2_split(xv[i]);
              ev[2 * i] = ex2(e.x);
              ev[2 * i + 1] = ex2(e.y);
            }
            if (!full) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (cs + i >= cnt) ev[i] = 0.f;
            }
            uint64_t la = f2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint64_t p2 = f2(ev[2 * i], ev[2 * i + 1]);
              if (i & 1) la = add2(la, p2); else l2 = add2(l2, p2);
              pk[i] = bf16x2_of(p2);
            }
            l2 = add2(l2, la);
            tmem_st16(tS + 32 + c0 / 2 + 16 * ch, pk);
          }
          {
            const float2 ls = f2_split(l2);
            l += ls.x + ls.y;
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&sh.p_full[t]);
        }
      }
      if (!ok) break;
      // epilogue: both halves' sums, out = O / l for this half's columns, lse
      sh.xl[t][hf][row] = l;
      mbar_arrive(&sh.xl_bar[t]);
      if (!mbar_wait(&sh.xl_bar[t], xl_phase, abort_flag, tmo, status)) break;
      xl_phase ^= 1;
      l += sh.xl[t][hf ^ 1][row];
      if (!mbar_wait(&sh.o_done[t], od_phase, abort_flag, tmo, status)) break;
      od_phase ^= 1;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < DH / 64; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + hf * (DH / 2) + c * 32, r);
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * inv_l;
        if (valid) store_row32<OutT>(orow_ptr + hf * (DH / 2) + c * 32, v);
      }
      if (valid && hf == 0) *lse_ptr = l > 0.f ? (m + lg2(l)) * 0.69314718055994531f : -INFINITY;
      tc_fence_before();
      mbar_arrive(&sh.o_free[t]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// One CTA waits on a barrier nothing completes, with a bounded wait (failure-path test).
__global__ void wait_timeout_kernel(uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, timeout_ns, &g_status_fwd);
  __syncthreads();
}

// exp2_poly2 on n values (test hook for its error bound).
__global__ void exp2_poly_kernel(const float* __restrict__ x, float* __restrict__ y, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x1 = i + 1 < n ? x[i + 1] : 0.f;
  const float2 r = f2_split(exp2_poly2(f2(x[i], x1)));
  y[i] = r.x;
  if (i + 1 < n) y[i + 1] = r.y;
}

template <int DH, typename OutT>
cudaError_t launch_one(const Plan& P, const CUtensorMap& mq, const CUtensorMap& mk,
                       const CUtensorMap& mv, OutT* out, float* lse, int n_sm, cudaStream_t st) {
  using C = FwdCfg<DH>;
  auto kern = ring_fwd_tc_kernel<DH, OutT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = P.n_items < n_sm ? P.n_items : n_sm;
  kern<<<grid, kFwdThreads, C::kSmemBytes, st>>>(mq, mk, mv, P, out, lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const Plan& P, const void* q, const void* k, const void* v, void* out,
                          float* lse, cudaStream_t st) {
  if (P.n_items == 0) return cudaSuccess;
  CUtensorMap mq, mk, mv;
  cudaError_t e = make_token_tmap(&mq, q, P.n_rows, P.hq, P.head_dim);
  if (e == cudaSuccess) e = make_token_tmap(&mk, k, P.n_rows, P.hkv, P.head_dim);
  if (e == cudaSuccess) e = make_token_tmap(&mv, v, P.n_rows, P.hkv, P.head_dim);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (P.head_dim == 128) {
    return P.out_f32 ? launch_one<128, float>(P, mq, mk, mv, static_cast<float*>(out), lse, n_sm, st)
                     : launch_one<128, __nv_bfloat16>(P, mq, mk, mv, static_cast<__nv_bfloat16*>(out), lse, n_sm, st);
  }
  return P.out_f32 ? launch_one<64, float>(P, mq, mk, mv, static_cast<float*>(out), lse, n_sm, st)
                   : launch_one<64, __nv_bfloat16>(P, mq, mk, mv, static_cast<__nv_bfloat16*>(out), lse, n_sm, st);
}

cudaError_t launch_exp2_poly(const float* x, float* y, int n, cudaStream_t st) {
  const int pairs = (n + 1) / 2;
  exp2_poly_kernel<<<(pairs + 255) / 256, 256, 0, st>>>(x, y, n);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(uint64_t timeout_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(timeout_ns);
  return cudaGetLastError();
}

cudaError_t fwd_status(unsigned int* value, bool reset) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_status_fwd, sizeof(unsigned int));
  if (e == cudaSuccess && reset) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_status_fwd, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace ra
