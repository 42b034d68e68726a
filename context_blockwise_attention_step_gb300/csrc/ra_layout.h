// ra_layout.h — shard layouts and causal key limits, shared by host and device code.
//
// A sequence of len tokens is split into D shards of L = len/D local tokens. Local token a
// of rank r holds a global position (ring-flash-attn package card, "What it is and what it
// does": basic, zigzag, stripe; Ring Attention concept page, "Sequence sharding and the
// ring topology"):
//   basic : r*L + a                       (contiguous blocks)
//   zigzag: a < c ? r*c + a : (2D-1-r)*c + (a - c),  c = L/2  (chunks r and 2D-1-r)
//   stripe: a*D + r                       (token t on rank t mod D)
// In every layout the position grows with a, so the keys of shard j that a query at global
// position p may see under the causal rule (concept page, "Watch Out For": mask by global
// position) are a prefix of shard j's local tokens. key_limit() returns its last index.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

enum Layout : int { kBasic = 0, kZigzag = 1, kStripe = 2 };

// Global position of local token a of rank r.
RA_HD int64_t layout_pos(int layout, int D, int L, int r, int a) {
  if (layout == kBasic) return (int64_t)r * L + a;
  if (layout == kStripe) return (int64_t)a * D + r;
  const int c = L >> 1;
  return a < c ? (int64_t)r * c + a : (int64_t)(2 * D - 1 - r) * c + (a - c);
}

// Largest local index b of rank j with layout_pos(j, b) <= p, or -1 if none; at most L-1.
RA_HD int key_limit(int layout, int D, int L, int j, int64_t p) {
  if (p < 0) return -1;
  int64_t b;
  if (layout == kBasic) {
    b = p - (int64_t)j * L;
  } else if (layout == kStripe) {
    if (p < j) return -1;
    b = (p - j) / D;
  } else {
    const int64_t c = L >> 1;
    const int64_t second = (int64_t)(2 * D - 1 - j) * c;  // first position of chunk 2D-1-j
    if (p >= second) {
      b = c + (p - second);
    } else {
      b = p - (int64_t)j * c;
      if (b > c - 1) b = c - 1;
    }
  }
  if (b < 0) return -1;
  return b > L - 1 ? L - 1 : (int)b;
}

// Smallest local index a of rank r with layout_pos(r, a) >= p (L if none).
RA_HD int first_query(int layout, int D, int L, int r, int64_t p) {
  return key_limit(layout, D, L, r, p - 1) + 1;
}

}  // namespace ra
