// ra_api.cu — the exported C ABI (include/ringattn.h): validation, launch plans, dispatch.
//
// Every entry point validates its arguments on the host first and launches nothing when
// they are invalid. Launch plans carry the per-sequence table of the varlen tile scheduler:
// sequences sorted longest first, each with its shard-major / natural offsets and the index
// of its first work item.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

#include "ra_internal.h"
#include "ra_plan.h"

using ra::Plan;
using ra::SeqDesc;

namespace {

thread_local std::string g_last_error;
thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr, g_prof_mid = nullptr;

// Records the profiling events (if set) around the launch done by `launch`.
template <typename F>
cudaError_t profiled(cudaStream_t st, F&& launch) {
  if (g_prof_start) cudaEventRecord(g_prof_start, st);
  const cudaError_t e = launch();
  if (g_prof_stop) cudaEventRecord(g_prof_stop, st);
  return e;
}

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return RA_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool is_varlen(const ra_problem* p) { return p->batch == 0; }

// Natural-order sequence lengths (batch: B copies of S).
std::vector<int64_t> lengths_of(const ra_problem* p) {
  std::vector<int64_t> len;
  if (!is_varlen(p)) {
    len.assign(p->batch, p->seqlen);
  } else {
    for (int i = 0; i < p->n_seqs; ++i) len.push_back(int64_t(p->cu_seqlens[i + 1]) - p->cu_seqlens[i]);
  }
  return len;
}

int validate(const ra_problem* p) {
  if (p == nullptr) return fail(RA_ERR_INVALID_ARG, "problem is NULL");
  if (p->dtype != RA_F32 && p->dtype != RA_BF16) return fail(RA_ERR_INVALID_ARG, "bad dtype %d", p->dtype);
  if (p->layout < RA_LAYOUT_BASIC || p->layout > RA_LAYOUT_STRIPE)
    return fail(RA_ERR_INVALID_ARG, "bad layout %d", p->layout);
  if (p->D < 1) return fail(RA_ERR_INVALID_ARG, "D must be >= 1 (got %d)", p->D);
  if (p->hq < 1 || p->hkv < 1 || p->head_dim < 1)
    return fail(RA_ERR_INVALID_ARG, "heads and head_dim must be >= 1");
  if (p->hq % p->hkv) return fail(RA_ERR_UNSUPPORTED, "hq (%d) must be a multiple of hkv (%d)", p->hq, p->hkv);
  if (std::isnan(p->scale) || std::isinf(p->scale)) return fail(RA_ERR_INVALID_ARG, "scale is not finite");
  if (p->dtype == RA_BF16 && p->head_dim != 64 && p->head_dim != 128)
    return fail(RA_ERR_UNSUPPORTED, "bf16 supports head_dim 64 or 128 (got %d)", p->head_dim);
  if (p->dtype == RA_F32 && p->head_dim > 128)
    return fail(RA_ERR_UNSUPPORTED, "f32 supports head_dim <= 128 (got %d)", p->head_dim);
  if (p->batch < 0) return fail(RA_ERR_INVALID_ARG, "batch must be >= 0");
  const int64_t div = p->layout == RA_LAYOUT_ZIGZAG ? 2LL * p->D : p->D;
  int64_t rows = 0;
  if (!is_varlen(p)) {
    if (p->cu_seqlens != nullptr) return fail(RA_ERR_INVALID_ARG, "cu_seqlens must be NULL in batch mode");
    if (p->seqlen < 1) return fail(RA_ERR_SHAPE, "seqlen must be >= 1");
    if (p->batch > RA_MAX_SEQS) return fail(RA_ERR_UNSUPPORTED, "batch > %d", RA_MAX_SEQS);
    if (p->seqlen % div)
      return fail(RA_ERR_SHAPE, "seqlen %d not divisible by %lld", p->seqlen, (long long)div);
    rows = int64_t(p->batch) * p->seqlen;
  } else {
    if (p->cu_seqlens == nullptr) return fail(RA_ERR_INVALID_ARG, "varlen mode needs cu_seqlens (host)");
    if (p->n_seqs < 0) return fail(RA_ERR_INVALID_ARG, "n_seqs must be >= 0");
    if (p->n_seqs > RA_MAX_SEQS) return fail(RA_ERR_UNSUPPORTED, "n_seqs > %d", RA_MAX_SEQS);
    if (p->cu_seqlens[0] != 0) return fail(RA_ERR_SHAPE, "cu_seqlens[0] must be 0");
    for (int i = 0; i < p->n_seqs; ++i) {
      const int64_t len = int64_t(p->cu_seqlens[i + 1]) - p->cu_seqlens[i];
      if (len < 0) return fail(RA_ERR_SHAPE, "cu_seqlens decreases at %d", i);
      if (len % div)
        return fail(RA_ERR_SHAPE, "sequence %d length %lld not divisible by %lld", i, (long long)len,
                    (long long)div);
    }
    rows = p->cu_seqlens[p->n_seqs];
    if (rows % p->D) return fail(RA_ERR_SHAPE, "total tokens not divisible by D");
  }
  if (rows * int64_t(p->hq) >= (int64_t(1) << 31))
    return fail(RA_ERR_UNSUPPORTED, "tokens x query heads must stay below 2^31");
  return RA_OK;
}

// which: 0 forward items, 1 backward items, 2 no items (elementwise kernels).
Plan* make_plan(const ra_problem* p, int which, int step_begin, int step_end, int rank_only,
                int out_f32, std::vector<int>* natural_index = nullptr, int kv_shard_only = -1) {
  Plan* P = static_cast<Plan*>(calloc(1, sizeof(Plan)));
  P->layout = p->layout;
  P->causal = p->causal ? 1 : 0;
  P->D = p->D;
  P->hq = p->hq;
  P->hkv = p->hkv;
  P->group = p->hq / p->hkv;
  P->head_dim = p->head_dim;
  P->step_begin = step_begin;
  P->step_end = step_end;
  P->rank_only = rank_only;
  P->kv_shard_only = kv_shard_only;
  P->out_f32 = out_f32;
  P->bwd_accum = 0;
  P->scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt(static_cast<float>(p->head_dim));
  P->scale_log2 = P->scale * 1.4426950408889634f;
  P->dq_mul = P->scale;
  P->timeout_ns = ra::kDefaultTimeoutNs;
  const std::vector<int64_t> len = lengths_of(p);
  const int n = static_cast<int>(len.size());
  std::vector<int> order(n);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return len[a] > len[b]; });
  int64_t T = 0;
  for (int64_t x : len) T += x;
  P->n_rows = static_cast<int32_t>(T);
  if (!is_varlen(p)) {
    P->shard_stride = p->seqlen / p->D;
    P->lse_hstride = p->seqlen;
  } else {
    P->shard_stride = static_cast<int32_t>(T / p->D);
    P->lse_hstride = static_cast<int32_t>(T);
  }
  int items = 0, ns = 0;
  for (int k = 0; k < n; ++k) {
    const int i = order[k];
    if (len[i] == 0) continue;
    SeqDesc& s = P->seq[ns++];
    s.L = static_cast<int32_t>(len[i] / p->D);
    if (!is_varlen(p)) {
      s.row_off = s.nat_off = i * p->seqlen;
      s.lse_off = s.lse_nat_off = i * p->hq * p->seqlen;
    } else {
      s.row_off = s.lse_off = p->cu_seqlens[i] / p->D;
      s.nat_off = s.lse_nat_off = p->cu_seqlens[i];
    }
    s.item_start = items;
    if (natural_index) natural_index->push_back(i);
    if (which == 0) items += ra::fwd_items_of(*P, s.L);
    else if (which == 1) items += ra::bwd_items_of(*P, s.L);
  }
  P->n_seqs = ns;
  P->n_items = items;
  // Walk order of the backward items: K/V tiles innermost when one K/V head group's Q and
  // dO of the longest sequence (all ranks) are larger than this device's L2.
  if (which == 1 && n > 0) {
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) == cudaSuccess && l2 > 0) {
      const int64_t elem = p->dtype == RA_F32 ? 4 : 2;
      const int64_t group_qdo = len[order[0]] * P->group * p->head_dim * elem * 2;
      P->bwd_kt_inner = group_qdo > static_cast<int64_t>(l2) ? 1 : 0;
    } else {
      cudaGetLastError();  // no device: keep the default order
    }
  }
  return P;
}

struct PlanHolder {
  Plan* p;
  explicit PlanHolder(Plan* q) : p(q) {}
  ~PlanHolder() { free(p); }
};

bool force_simt() {
  const char* e = getenv("RA_IMPL");
  return e != nullptr && strcmp(e, "simt") == 0;
}

bool use_tc(const ra_problem* p) { return p->dtype == RA_BF16 && !force_simt(); }

// The tensor-core backward runs as two atomic-free passes (K/V tiles for dk / dv, query
// tiles for dq), which is both faster and run-to-run deterministic. RA_BWD=fused selects
// the single K/V-tile pass that adds dq with float reductions instead (for comparison;
// never used for problems that ask for determinism).
bool fused_bwd(const ra_problem* p) {
  const char* e = getenv("RA_BWD");
  return use_tc(p) && !p->deterministic && e != nullptr && strcmp(e, "fused") == 0;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t delta_bytes(const ra_problem* p) {
  int64_t rows = 0;
  for (int64_t x : lengths_of(p)) rows += x;
  return align256(size_t(rows) * p->hq * sizeof(float));
}

// The shared item counters of the K/V-tile pass and of the dq pass (dynamic scheduling),
// one 256-byte block.
size_t sched_bytes(const ra_problem* p) { return use_tc(p) ? 256 : 0; }

size_t dq_acc_bytes(const ra_problem* p) {
  if (!fused_bwd(p)) return 0;
  int64_t rows = 0;
  for (int64_t x : lengths_of(p)) rows += x;
  return align256(size_t(rows) * p->hq * p->head_dim * sizeof(float));
}

}  // namespace

int ra::record_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

extern "C" {

int ra_version(void) { return RA_VERSION; }

const char* ra_last_error(void) { return g_last_error.c_str(); }

int ra_validate(const ra_problem* p) {
  const int v = validate(p);
  return v == RA_OK ? ok() : v;
}

int ra_ring_attn_fwd(const ra_problem* p, const void* q, const void* k, const void* v, void* out,
                     float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (int e = validate(p)) return e;
  if (!q || !k || !v || !out || !lse) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (workspace != nullptr && reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(RA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  PlanHolder P(make_plan(p, 0, 0, p->D, -1, p->dtype == RA_F32));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // With a workspace the CTAs take their items from a counter in it; without, by stride.
  if (workspace != nullptr && use_tc(p) && workspace_bytes >= sched_bytes(p)) {
    P.p->work_counter = static_cast<int32_t*>(workspace);
    const cudaError_t c = cudaMemsetAsync(workspace, 0, sizeof(int32_t), st);
    if (c != cudaSuccess) return cuda_fail(c, "item counter clear");
  }
  const cudaError_t e = profiled(st, [&] {
    return use_tc(p) ? ra::launch_fwd_tc(*P.p, q, k, v, out, lse, st)
                     : ra::launch_fwd_simt(*P.p, p->dtype, q, k, v, out, lse, st);
  });
  return e == cudaSuccess ? ok() : cuda_fail(e, "ring forward launch");
}

int ra_block_attn_fwd(const ra_problem* p, int rank, int step, const void* q, const void* k,
                      const void* v, void* block_out, int block_out_dtype, float* block_lse,
                      void* stream) {
  if (int e = validate(p)) return e;
  if (!q || !k || !v || !block_out || !block_lse) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (rank >= p->D || rank < -1) return fail(RA_ERR_INVALID_ARG, "rank %d out of range", rank);
  if (step < 0 || step >= p->D) return fail(RA_ERR_INVALID_ARG, "step %d out of range", step);
  if (block_out_dtype != RA_F32 && block_out_dtype != RA_BF16)
    return fail(RA_ERR_INVALID_ARG, "bad block_out dtype %d", block_out_dtype);
  if (p->dtype == RA_F32 && block_out_dtype != RA_F32)
    return fail(RA_ERR_UNSUPPORTED, "f32 problems produce f32 block outputs");
  PlanHolder P(make_plan(p, 0, step, step + 1, rank < 0 ? -1 : rank, block_out_dtype == RA_F32));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = use_tc(p)
                            ? ra::launch_fwd_tc(*P.p, q, k, v, block_out, block_lse, st)
                            : ra::launch_fwd_simt(*P.p, p->dtype, q, k, v, block_out, block_lse, st);
  return e == cudaSuccess ? ok() : cuda_fail(e, "block forward launch");
}

int ra_update_out_and_lse(const ra_problem* p, int rank, float* out, float* lse,
                          const void* block_out, int block_out_dtype, const float* block_lse,
                          void* stream) {
  if (int e = validate(p)) return e;
  if (!out || !lse || !block_out || !block_lse) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (rank >= p->D || rank < -1) return fail(RA_ERR_INVALID_ARG, "rank %d out of range", rank);
  if (block_out_dtype != RA_F32 && block_out_dtype != RA_BF16)
    return fail(RA_ERR_INVALID_ARG, "bad block_out dtype %d", block_out_dtype);
  PlanHolder P(make_plan(p, 2, 0, p->D, rank < 0 ? -1 : rank, 1));
  const cudaError_t e = ra::launch_merge(*P.p, out, lse, block_out, block_out_dtype == RA_F32,
                                         block_lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "merge launch");
}

size_t ra_workspace_bytes(const ra_problem* p, int which) {
  if (validate(p) != RA_OK) return 0;
  if (which == 0) return sched_bytes(p);
  if (which == 1) return delta_bytes(p) + dq_acc_bytes(p) + sched_bytes(p);
  if (which == 2) return delta_bytes(p) + sched_bytes(p);
  return 0;
}

int ra_ring_attn_bwd(const ra_problem* p, const void* q, const void* k, const void* v,
                     const void* out, const float* lse, const void* dout, void* dq, void* dk,
                     void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  if (int e = validate(p)) return e;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv)
    return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  const size_t need = delta_bytes(p) + dq_acc_bytes(p) + sched_bytes(p);
  if (workspace_bytes < need)
    return fail(RA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (need > 0 && (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256))
    return fail(RA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* delta = static_cast<float*>(workspace);
  PlanHolder E(make_plan(p, 2, 0, p->D, -1, 0));
  cudaError_t e = ra::launch_bwd_delta(*E.p, p->dtype, out, dout, delta, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  int32_t* counter = nullptr;  // the K/V-tile pass takes its items from counter[0], dq from [1]
  if (use_tc(p)) {
    counter = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + delta_bytes(p) +
                                         dq_acc_bytes(p));
    e = cudaMemsetAsync(counter, 0, 2 * sizeof(int32_t), st);  // K/V pass, dq pass
    if (e != cudaSuccess) return cuda_fail(e, "item counter clear");
  }
  if (use_tc(p) && !fused_bwd(p)) {
    // dk, dv from the K/V-tile kernel without its dq part; dq query-tile-major
    PlanHolder P(make_plan(p, 1, 0, p->D, -1, 0));
    P.p->work_counter = counter;
    e = profiled(st, [&] {
      cudaError_t r = ra::launch_bwd_tc(*P.p, ra::BwdKind::kKvOnly, q, k, v, dout, lse, delta, nullptr,
                                        dk, dv, st);
      if (r != cudaSuccess) return r;
      if (g_prof_mid) cudaEventRecord(g_prof_mid, st);
      return ra::launch_bwd_dq_tc(*P.p, q, k, v, dout, lse, delta, dq, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  } else if (use_tc(p)) {
    float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + delta_bytes(p));
    e = cudaMemsetAsync(dq_acc, 0, dq_acc_bytes(p), st);
    if (e != cudaSuccess) return cuda_fail(e, "dq workspace clear");
    PlanHolder P(make_plan(p, 1, 0, p->D, -1, 0));
    P.p->work_counter = counter;
    e = profiled(st, [&] {
      return ra::launch_bwd_tc(*P.p, ra::BwdKind::kFused, q, k, v, dout, lse, delta, dq_acc, dk, dv, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    e = ra::launch_dq_convert(*E.p, dq_acc, dq, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward postprocess launch");
  } else {
    e = profiled(st, [&] { return ra::launch_bwd_simt(*E.p, p->dtype, q, k, v, dout, lse, delta, dq, dk, dv, st); });
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  }
  return ok();
}

int ra_block_attn_bwd(const ra_problem* p, int rank, int step, const void* q, const void* k,
                      const void* v, const void* out, const float* lse, const void* dout,
                      float* dq_acc, float* dk_acc, float* dv_acc, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (int e = validate(p)) return e;
  if (!q || !k || !v || !out || !lse || !dout || !dq_acc || !dk_acc || !dv_acc)
    return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (rank >= p->D || rank < -1) return fail(RA_ERR_INVALID_ARG, "rank %d out of range", rank);
  if (step < 0 || step >= p->D) return fail(RA_ERR_INVALID_ARG, "step %d out of range", step);
  const size_t need = delta_bytes(p) + sched_bytes(p);
  if (workspace_bytes < need)
    return fail(RA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(RA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* delta = static_cast<float*>(workspace);
  const int r_only = rank < 0 ? -1 : rank;
  const int kv_only = rank < 0 ? -1 : ((rank - step) % p->D + p->D) % p->D;
  PlanHolder E(make_plan(p, 2, step, step + 1, r_only, 0));
  cudaError_t e = ra::launch_bwd_delta(*E.p, p->dtype, out, dout, delta, st);
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  int32_t* counter = nullptr;  // item counters of the two passes, as in ra_ring_attn_bwd
  if (use_tc(p)) {
    counter = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + delta_bytes(p));
    e = cudaMemsetAsync(counter, 0, 2 * sizeof(int32_t), st);
    if (e != cudaSuccess) return cuda_fail(e, "item counter clear");
  }
  if (use_tc(p) && !fused_bwd(p)) {
    // the two passes of the deterministic backward, restricted to (rank, step), adding into
    // the float32 sums: dk, dv from the K/V-tile kernel, dq from the query-tile kernel
    PlanHolder P(make_plan(p, 1, step, step + 1, r_only, 0, nullptr, kv_only));
    P.p->bwd_accum = 1;
    P.p->work_counter = counter;
    e = ra::launch_bwd_tc(*P.p, ra::BwdKind::kKvAccum, q, k, v, dout, lse, delta, nullptr, dk_acc,
                          dv_acc, st);
    if (e == cudaSuccess) e = ra::launch_bwd_dq_tc(*P.p, q, k, v, dout, lse, delta, dq_acc, st);
  } else if (use_tc(p)) {
    PlanHolder P(make_plan(p, 1, step, step + 1, r_only, 0, nullptr, kv_only));
    P.p->bwd_accum = 1;
    P.p->work_counter = counter;
    e = ra::launch_bwd_tc(*P.p, ra::BwdKind::kBlockAccum, q, k, v, dout, lse, delta, dq_acc, dk_acc,
                          dv_acc, st);
  } else {
    PlanHolder P(make_plan(p, 2, step, step + 1, r_only, 0, nullptr, kv_only));
    P.p->bwd_accum = 1;
    e = ra::launch_bwd_simt(*P.p, p->dtype, q, k, v, dout, lse, delta, dq_acc, dk_acc, dv_acc, st);
  }
  return e == cudaSuccess ? ok() : cuda_fail(e, "block backward launch");
}

int ra_shard_tokens(const ra_problem* p, int direction, const void* src, void* dst,
                    int64_t row_bytes, void* stream) {
  if (int e = validate(p)) return e;
  if (!src || !dst) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (direction != 0 && direction != 1) return fail(RA_ERR_INVALID_ARG, "direction must be 0 or 1");
  if (row_bytes < 1 || row_bytes > (int64_t(1) << 30)) return fail(RA_ERR_INVALID_ARG, "bad row_bytes");
  PlanHolder P(make_plan(p, 2, 0, p->D, -1, 0));
  const cudaError_t e =
      ra::launch_shard_tokens(*P.p, direction, src, dst, row_bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "shard launch");
}

int ra_shard_lse(const ra_problem* p, int direction, const float* src, float* dst, void* stream) {
  if (int e = validate(p)) return e;
  if (!src || !dst) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (direction != 0 && direction != 1) return fail(RA_ERR_INVALID_ARG, "direction must be 0 or 1");
  PlanHolder P(make_plan(p, 2, 0, p->D, -1, 0));
  const cudaError_t e = ra::launch_shard_lse(*P.p, direction, src, dst, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "shard launch");
}

int ra_layout_positions(const ra_problem* p, int seq, int64_t* pos_out) {
  if (int e = validate(p)) return e;
  const std::vector<int64_t> len = lengths_of(p);
  if (seq < 0 || seq >= static_cast<int>(len.size())) return fail(RA_ERR_INVALID_ARG, "bad sequence index");
  if (!pos_out) return fail(RA_ERR_INVALID_ARG, "null output");
  const int L = static_cast<int>(len[seq] / p->D);
  for (int r = 0; r < p->D; ++r)
    for (int a = 0; a < L; ++a) pos_out[int64_t(r) * L + a] = ra::layout_pos(p->layout, p->D, L, r, a);
  return ok();
}

int ra_step_counts(const ra_problem* p, int seq, int rank, int step, int32_t* count_out,
                   int32_t* active_out) {
  if (int e = validate(p)) return e;
  const std::vector<int64_t> len = lengths_of(p);
  if (seq < 0 || seq >= static_cast<int>(len.size())) return fail(RA_ERR_INVALID_ARG, "bad sequence index");
  if (rank < 0 || rank >= p->D || step < 0 || step >= p->D) return fail(RA_ERR_INVALID_ARG, "bad rank/step");
  if (!count_out) return fail(RA_ERR_INVALID_ARG, "null output");
  const int L = static_cast<int>(len[seq] / p->D);
  const int j = ra::shard_at_step(p->D, rank, step);
  int any = 0;
  for (int a = 0; a < L; ++a) {
    const int lim = p->causal ? ra::key_limit(p->layout, p->D, L, j, ra::layout_pos(p->layout, p->D, L, rank, a))
                              : L - 1;
    count_out[a] = lim + 1;
    any |= lim >= 0;
  }
  if (active_out) *active_out = any;
  return ok();
}

int ra_work_items(const ra_problem* p, int which, int32_t* items_out, int max_items) {
  if (int e = validate(p)) return e;
  if (which != 0 && which != 1) return fail(RA_ERR_INVALID_ARG, "which must be 0 or 1");
  std::vector<int> nat;
  PlanHolder P(make_plan(p, which, 0, p->D, -1, 0, &nat));
  const int n = P.p->n_items;
  for (int w = 0; w < n && w < max_items && items_out; ++w) {
    if (which == 0) {
      const ra::FwdItem it = ra::decode_fwd(*P.p, w);
      items_out[4 * w + 0] = nat[it.seq];
      items_out[4 * w + 1] = it.h;
      items_out[4 * w + 2] = it.r;
      items_out[4 * w + 3] = it.blk;
    } else {
      const ra::BwdItem it = ra::decode_bwd(*P.p, w);
      items_out[4 * w + 0] = nat[it.seq];
      items_out[4 * w + 1] = it.hk;
      items_out[4 * w + 2] = it.j;
      items_out[4 * w + 3] = it.kt;
    }
  }
  ok();
  return n;
}

int ra_check_device_status(int reset) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
  unsigned int f = 0, b = 0, d = 0;
  e = ra::fwd_status(&f, reset != 0);
  if (e == cudaSuccess) e = ra::bwd_status(&b, reset != 0);
  if (e == cudaSuccess) e = ra::bwd_dq_status(&d, reset != 0);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (f | b | d)
    return fail(RA_ERR_DEVICE_TIMEOUT, "device status: forward 0x%x backward 0x%x dq 0x%x", f, b, d);
  return ok();
}

int ra_profile_events(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr))
    return fail(RA_ERR_INVALID_ARG, "pass both events or neither");
  g_prof_start = static_cast<cudaEvent_t>(start_event);
  g_prof_stop = static_cast<cudaEvent_t>(stop_event);
  return ok();
}

int ra_profile_split_event(void* mid_event) {
  g_prof_mid = static_cast<cudaEvent_t>(mid_event);
  return ok();
}

int ra_test_wait_timeout(uint64_t timeout_ns, void* stream) {
  if (timeout_ns == 0 || timeout_ns > 10ull * 1000000000ull)
    return fail(RA_ERR_INVALID_ARG, "timeout must be in (0, 10 s]");
  const cudaError_t e = ra::launch_wait_timeout(timeout_ns, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "wait-timeout launch");
}

int ra_test_exp2_poly(const float* x, float* y, int n, void* stream) {
  if (!x || !y || n < 0) return fail(RA_ERR_INVALID_ARG, "bad arguments");
  if (n == 0) return ok();
  const cudaError_t e = ra::launch_exp2_poly(x, y, n, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "exp2 test launch");
}

}  // extern "C"
