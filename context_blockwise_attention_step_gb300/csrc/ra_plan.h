// ra_plan.h — the launch plan every kernel receives by value: problem constants, the
// per-sequence table (the varlen tile scheduler's input) and the work-item decoding.
//
// Varlen mode packs several sequences (cu_seqlens); batch mode is the special case of B
// equal sequences. Each sequence i is split into D pieces of L_i = len_i/D local tokens;
// the shard-major row of local token a of rank r is row_off_i + r*shard_stride + a and its
// natural row is nat_off_i + layout_pos(r, a). The host sorts the table by length
// (longest first) so that a persistent grid starts with the biggest work.
#pragma once
#include <stdint.h>

#include "ra_layout.h"
#include "../../include/ringattn.h"

namespace ra {

constexpr int kFwdBlockRows = 256;  // query rows per forward work item (two 128-row tiles)
constexpr int kKvTileRows = 128;    // K/V rows per tile (and per backward work item)
constexpr int kQTileRows = 128;

struct SeqDesc {
  int32_t row_off;      // shard-major row of (rank 0, local token 0)
  int32_t nat_off;      // natural row of the sequence's first token
  int32_t L;            // local length len_i / D
  int32_t lse_off;      // shard-major lse index of (rank 0, local 0), head 0
  int32_t lse_nat_off;  // natural lse index of the sequence's first token, head 0
  int32_t item_start;   // first work item of this sequence in the launched kernel
};

struct Plan {
  int32_t layout, causal, D;
  int32_t hq, hkv, group, head_dim;
  int32_t shard_stride;  // rows between rank r and rank r+1 of one sequence piece
  int32_t lse_hstride;   // lse elements between heads
  int32_t n_rows;        // rows of the token axis (B*S or T)
  int32_t n_seqs, n_items;
  int32_t step_begin, step_end;  // ring steps covered by a launch: [begin, end)
  int32_t rank_only;             // >= 0: only this rank's query rows (block mode)
  int32_t kv_shard_only;         // backward, >= 0: only this K/V shard's tiles are items
  int32_t out_f32;               // forward output stored as float32 (else problem dtype)
  int32_t bwd_accum;             // backward: add float32 gradients into the outputs
  int32_t bwd_kt_inner;          // backward items: K/V tiles innermost (see decode_bwd)
  float scale, scale_log2;
  float dq_mul;                  // factor on dS K before it is added to the dq sums
  uint64_t timeout_ns;
  int32_t* work_counter;         // backward K/V pass: shared item counter (null: static stride)
  SeqDesc seq[RA_MAX_SEQS];
};

RA_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

RA_HD int plan_ranks(const Plan& P) { return P.rank_only >= 0 ? 1 : P.D; }

// Forward items of one sequence: one per (256-row query block, rank, query head).
RA_HD int fwd_items_of(const Plan& P, int L) {
  return ceil_div(L, kFwdBlockRows) * plan_ranks(P) * P.hq;
}
RA_HD int plan_kv_shards(const Plan& P) { return P.kv_shard_only >= 0 ? 1 : P.D; }

// Backward items of one sequence: one per (128-row K/V tile, K/V shard, K/V head).
RA_HD int bwd_items_of(const Plan& P, int L) {
  return ceil_div(L, kKvTileRows) * plan_kv_shards(P) * P.hkv;
}

// Whether the backward walk of K/V shard j visits query rank r: the ring step at which
// r holds shard j, (r - j) mod D, must lie in [step_begin, step_end), and r must be the
// selected rank when one is selected.
RA_HD bool rank_in_walk(const Plan& P, int j, int r) {
  const int s = ((r - j) % P.D + P.D) % P.D;
  return s >= P.step_begin && s < P.step_end && (P.rank_only < 0 || r == P.rank_only);
}

RA_HD int find_seq(const Plan& P, int w) {
  int lo = 0, hi = P.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.seq[mid].item_start <= w) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct FwdItem { int seq, h, r, blk; };
struct BwdItem { int seq, hk, j, kt; };

// Forward decode: the last query block first (for causal layouts it sees the most keys),
// then K/V heads, ranks, and the query heads of a GQA group innermost (they read the same
// K/V tiles at about the same time, from L2). The CTAs running together then cover a few
// K/V heads of one query block. Measured on GB300 against the alternatives: K/V heads
// outermost 1013, query heads innermost over all heads 1094, this order 1093 TFLOP/s at
// 131072 tokens (32/8 heads, D = 16); at 32768 tokens (16 heads) 1039 against 973.
RA_HD FwdItem decode_fwd(const Plan& P, int w) {
  FwdItem it;
  it.seq = find_seq(P, w);
  const SeqDesc& s = P.seq[it.seq];
  const int nr = plan_ranks(P);
  int x = w - s.item_start;
  const int g = x % P.group;
  x /= P.group;
  it.r = P.rank_only >= 0 ? P.rank_only : x % nr;
  x /= nr;
  const int hk = x % P.hkv;
  x /= P.hkv;
  it.h = hk * P.group + g;
  it.blk = ceil_div(s.L, kFwdBlockRows) - 1 - x;
  return it;
}

// Backward decode: K/V heads outermost, so that the CTAs running at the same time share
// one K/V head and therefore the same query heads' Q, dO (and dq rows). Within a head,
// either K/V tiles in increasing order (early keys are seen by the most queries) with the
// shards innermost, or, when one K/V head group's Q and dO are larger than the L2
// (bwd_kt_inner), shards in order with the K/V tiles innermost: the CTAs running together
// then hold neighbouring tiles of one shard, whose walks visit nearly the same query tiles
// in the same order, so each Q / dO tile is read from DRAM about once per pass of that
// group instead of once per CTA. (Measured on GB300: 3 % faster K/V pass at 131072 tokens,
// 32/8 heads; 3-5 % slower where the group's Q and dO fit in L2.)
RA_HD BwdItem decode_bwd(const Plan& P, int w) {
  BwdItem it;
  it.seq = find_seq(P, w);
  const SeqDesc& s = P.seq[it.seq];
  const int ns = plan_kv_shards(P);
  const int nkt = ceil_div(s.L, kKvTileRows);
  const int per_head = nkt * ns;
  int x = w - s.item_start;
  it.hk = x / per_head;
  x %= per_head;
  if (P.bwd_kt_inner) {
    it.kt = x % nkt;
    it.j = P.kv_shard_only >= 0 ? P.kv_shard_only : x / nkt;
  } else {
    it.j = P.kv_shard_only >= 0 ? P.kv_shard_only : x % ns;
    it.kt = x / ns;
  }
  return it;
}

// Number of K/V tiles of shard j that a query block of rank r whose last valid local row
// is a_last must visit (a prefix of the shard's tiles).
RA_HD int kv_tiles_for(const Plan& P, int L, int r, int j, int a_last) {
  if (!P.causal) return ceil_div(L, kKvTileRows);
  const int lim = key_limit(P.layout, P.D, L, j, layout_pos(P.layout, P.D, L, r, a_last));
  return lim < 0 ? 0 : lim / kKvTileRows + 1;
}

// Number of keys of K/V tile b (shard j) that the query at local row a of rank r sees.
RA_HD int row_key_count(const Plan& P, int L, int r, int a, int j, int b) {
  if (a >= L) return 0;
  const int lim = P.causal ? key_limit(P.layout, P.D, L, j, layout_pos(P.layout, P.D, L, r, a))
                           : L - 1;
  int c = lim + 1 - b * kKvTileRows;
  return c < 0 ? 0 : (c > kKvTileRows ? kKvTileRows : c);
}

// Rank that holds K/V shard j at ring step s, and the shard rank r holds at step s.
RA_HD int rank_at_step(int D, int j, int s) { return (j + s) % D; }
RA_HD int shard_at_step(int D, int r, int s) { return ((r - s) % D + D) % D; }

}  // namespace ra
