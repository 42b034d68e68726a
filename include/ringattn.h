/*
 * ringattn.h — C ABI of the single-GPU ring attention hot path (GB300, sm_103a).
 *
 * Ring attention splits one sequence of N tokens into D shards of N/D tokens. Rank r keeps
 * its query shard; the K/V shards travel around a ring, so at step s rank r holds the K/V
 * shard of rank (r - s) mod D, computes local attention against it and folds the block
 * result into its running (out, lse) with the log-sum-exp merge (Ring Attention concept
 * page, "Sequence sharding and the ring topology" and "Online softmax across ring steps";
 * nanotron how-to page, "Forward Pass Implementation"). On one GPU the D ranks are virtual:
 * all shards sit in HBM and a ring step is the choice of which K/V shard a query tile reads.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller. The library allocates no
 *   device memory and never synchronises the device (except ra_check_device_status); all
 *   work is enqueued on the caller's CUDA stream, passed as `void* stream` (a cudaStream_t,
 *   NULL = legacy default stream).
 * - Token tensors (q, k, v, out, dout, dq, dk, dv) are row-major with the head dimension
 *   innermost: batch mode [B, S, H, Dh], varlen mode packed [T, H, Dh].
 *   Their token axis is SHARD-MAJOR: the D local shard buffers concatenated. Batch mode:
 *   token (b, r, a) — local index a of rank r — is row b*S + r*(S/D) + a. Varlen mode:
 *   every sequence i is split on its own into D pieces of len_i/D tokens, and rank r's
 *   buffer (rows [r*T/D, (r+1)*T/D)) holds its pieces of all sequences in order, i.e.
 *   token (i, r, a) is row r*T/D + cu_seqlens[i]/D + a. ra_shard_tokens / ra_shard_lse
 *   convert from and to natural order.
 * - Which global position a local token holds depends on the layout (ring-flash-attn
 *   package card, "What it is and what it does"): BASIC: r*L + a; ZIGZAG (2D chunks of
 *   c = L/2, rank r holds chunks r and 2D-1-r): a < c ? r*c + a : (2D-1-r)*c + a - c;
 *   STRIPE (token t on rank t mod D): a*D + r. L = len/D is the local length.
 * - lse is float32, natural log: batch mode [B, Hq, S], varlen mode [Hq, T], with the
 *   token axis shard-major like the token tensors.
 * - Causal masking uses global positions: query at position p sees keys at positions
 *   <= p of the same sequence (concept page, "Watch Out For"). With the basic layout this
 *   is the pages' rule "attend only if step <= rank" plus a triangular diagonal block.
 * - Grouped-query attention: query head h reads K/V head h / (Hq/Hkv).
 * - Return value: RA_OK (0) or a negative ra_status. On error nothing was launched (except
 *   RA_ERR_CUDA, which reports a failed launch) and ra_last_error() returns a message.
 *
 * Supported: bf16 with head_dim 64 or 128 (tensor-core path); f32 with head_dim 1..128
 * (CUDA-core path). D >= 1 and every sequence length divisible by D (2D for zigzag).
 * Up to RA_MAX_SEQS sequences (batch elements or varlen sequences) per call.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RA_VERSION 1
#define RA_MAX_SEQS 1024

typedef enum ra_status {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad enum                     */
  RA_ERR_UNSUPPORTED = -2,   /* dtype / head_dim / hq % hkv / option not implemented      */
  RA_ERR_SHAPE = -3,         /* a length not divisible by D (2D for zigzag), bad cu_seqlens */
  RA_ERR_WORKSPACE = -4,     /* workspace smaller than ra_workspace_bytes()               */
  RA_ERR_CUDA = -5,          /* a CUDA call or kernel launch failed                       */
  RA_ERR_DEVICE_TIMEOUT = -6 /* a kernel gave up a bounded wait (see ra_check_device_status) */
} ra_status;

typedef enum ra_dtype { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

typedef enum ra_layout {
  RA_LAYOUT_BASIC = 0,
  RA_LAYOUT_ZIGZAG = 1,
  RA_LAYOUT_STRIPE = 2
} ra_layout;

/* One ring-attention problem (nanotron how-to page, "Calling the Ring Attention Function
 * Directly": q, k, v, cu_seqlens, max_seqlen, scaling, causal, deterministic; ring-flash-attn
 * package card: batch and varlen modes, basic / zigzag / stripe). */
typedef struct ra_problem {
  int32_t dtype;              /* ra_dtype of q, k, v, out, dout, dq, dk, dv                  */
  int32_t layout;             /* ra_layout                                                  */
  int32_t causal;             /* 1: global-position causal mask; 0: full attention          */
  int32_t D;                  /* ring size: number of virtual shards                        */
  int32_t batch;              /* batch mode: B > 0.  Varlen mode: 0                          */
  int32_t seqlen;             /* batch mode: S (per batch element). Varlen mode: ignored     */
  int32_t n_seqs;             /* varlen mode: number of packed sequences                     */
  const int32_t* cu_seqlens;  /* varlen mode: HOST array of n_seqs+1 natural-order offsets,
                                 cu_seqlens[0] = 0, non-decreasing. NULL in batch mode.      */
  int32_t hq;                 /* query heads                                                */
  int32_t hkv;                /* K/V heads (hq % hkv == 0)                                   */
  int32_t head_dim;           /* Dh                                                         */
  float scale;                /* softmax scale; <= 0 selects 1/sqrt(head_dim) (the pages'
                                 default for scaling=None)                                  */
  int32_t deterministic;      /* 1: the backward must be run-to-run bit-identical (no
                                 floating-point atomics). 0: no such promise is asked for;
                                 the bf16 backward is atomic-free and deterministic anyway,
                                 the f32 one always is                                      */
} ra_problem;

/* Fused ring forward: every rank r, every step s = 0..D-1 against K/V shard (r-s) mod D,
 * with the log-sum-exp merge fused (running max and denominator kept across steps).
 * q [.., Hq, Dh], k/v [.., Hkv, Dh] in the problem dtype; out like q; lse float32.
 * The workspace is optional: NULL (any workspace_bytes) runs with a static work split;
 * a device buffer of >= ra_workspace_bytes(p, 0) bytes, 256-byte aligned, holds a counter
 * from which the CTAs take their work items (a CTA that finishes early takes more), and is
 * overwritten. (nanotron how-to page, "Forward Pass Implementation".) */
int ra_ring_attn_fwd(const ra_problem* p, const void* q, const void* k, const void* v,
                     void* out, float* lse, void* workspace, size_t workspace_bytes,
                     void* stream);

/* One ring step of the unfused path: rank `rank` (or every rank if rank < 0) attends with
 * its query shard to the K/V shard it holds at step `step`, i.e. shard (rank-step) mod D.
 * Writes the NORMALISED block_out (like q, in dtype `block_out_dtype` = RA_F32 or RA_BF16)
 * and block_lse (lse layout) for the rows of the selected rank(s) only. A row that sees no
 * key gets block_lse = -inf and block_out = 0. (How-to page, step 2: local attention of
 * the rank's queries against the received K/V slice.) */
int ra_block_attn_fwd(const ra_problem* p, int rank, int step, const void* q,
                      const void* k, const void* v, void* block_out, int block_out_dtype,
                      float* block_lse, void* stream);

/* The log-sum-exp merge of update_out_and_lse (how-to page, "Numerically-Stable Output
 * Fusion"), in place on float32 out / lse, for the rows of rank `rank` (all if < 0):
 *   lse' = log(exp(lse) + exp(block_lse))
 *   out' = exp(lse - lse') * out + exp(block_lse - lse') * block_out
 * lse = -inf with out = 0 is the identity (start state of a ring). block_out is float32 or
 * bf16 (block_out_dtype); out is always float32, in the token layout with Hq heads. */
int ra_update_out_and_lse(const ra_problem* p, int rank, float* out, float* lse,
                          const void* block_out, int block_out_dtype, const float* block_lse,
                          void* stream);

/* Bytes of device workspace: which = 0 for ra_ring_attn_fwd (optional there), which = 1
 * for ra_ring_attn_bwd, which = 2 for ra_block_attn_bwd; 0 for which = 0 on the f32 path. Returns 0 for an invalid problem as well;
 * call ra_validate to tell the two apart. */
size_t ra_workspace_bytes(const ra_problem* p, int which);

/* Ring backward (how-to page, "Backward Pass and Gradient Accumulation"): the blocks of
 * every (rank, step) pair again, each differentiated against the FINAL out and lse of the
 * forward (P recomputed from lse, never stored); dq accumulates per query rank, dk and dv
 * accumulate into the K/V shard that owns the block, summed over the query heads of a
 * group. Inputs: q, k, v, out, lse as from the forward, dout like out. Outputs dq (like q),
 * dk, dv (like k) in the problem dtype; every element is written. The bf16 path runs two
 * passes without atomics (K/V tiles: dk, dv; query tiles: dq), so results are run-to-run
 * bit-identical. The workspace (device, >= ra_workspace_bytes(p, 1), 256-byte aligned)
 * holds the per-row dot(dout, out), the counter from which the K/V-tile pass's CTAs take
 * their work items (and, only when the environment variable RA_BWD=fused selects the
 * single-pass variant with float reductions, float32 dq sums); it is overwritten. */
int ra_ring_attn_bwd(const ra_problem* p, const void* q, const void* k, const void* v,
                     const void* out, const float* lse, const void* dout, void* dq,
                     void* dk, void* dv, void* workspace, size_t workspace_bytes,
                     void* stream);

/* One ring step of the unfused backward (how-to page, "Backward Pass and Gradient
 * Accumulation": per step, the block is differentiated against the FINAL out and lse, then
 * dq += block_dq on the rank and block_dk / block_dv are added into the K/V shard's
 * gradients). Rank `rank` (every rank if rank < 0) at step `step` holds K/V shard
 * (rank - step) mod D; this call ADDS, in float32:
 *   dq_acc rows of rank `rank`                     += block_dq   (layout like q)
 *   dk_acc, dv_acc rows of shard (rank-step) mod D += block_dk, block_dv (layout like k)
 * Summing the calls of steps 0..D-1 into zeroed accumulators gives the full backward.
 * Inputs as for ra_ring_attn_bwd (out, lse: the final forward results). The workspace
 * (device, >= ra_workspace_bytes(p, 2), 256-byte aligned) receives the per-row
 * dot(dout, out) of the selected rank(s) and the passes' item counters; it is overwritten. Rows outside the selection are
 * not touched. Calls must not overlap on the GPU when they add into the same rows. The bf16
 * path runs the two atomic-free passes of ra_ring_attn_bwd restricted to the step (each
 * accumulator row is added by one thread), so results are run-to-run bit-identical;
 * RA_BWD=fused selects the single pass that adds block_dq with float reductions. */
int ra_block_attn_bwd(const ra_problem* p, int rank, int step, const void* q, const void* k,
                      const void* v, const void* out, const float* lse, const void* dout,
                      float* dq_acc, float* dk_acc, float* dv_acc, void* workspace,
                      size_t workspace_bytes, void* stream);

/* The same backward for callers that cannot allocate device memory (a plain-C plugin
 * handed only its input and output buffers, or a caller that must keep cudaMalloc and its
 * device-wide synchronisation out of a training step). The pages have no counterpart: on
 * the pages every rank allocates its own buffers. Instead of a caller workspace, the
 * scratch (the per-row dot(dout, out), plus float32 dq sums when RA_BWD=fused selects the
 * single-pass variant) lives in one static device
 * array of RA_NOALLOC_SCRATCH_BYTES that every GPU loading the library keeps until exit.
 * Arguments as for ra_ring_attn_bwd minus the workspace. Problems whose
 * ra_workspace_bytes(p, 1) exceeds the array are rejected with RA_ERR_WORKSPACE and nothing
 * is launched. The first call on a device looks the array's address up on that device
 * and keeps it for the life of the process (make that first call before any stream
 * capture; a cudaDeviceReset after it is not supported, since the kept address would then
 * be stale). Every call shares the array and the
 * backward clears what must start at zero, but calls that overlap on the GPU race on it:
 * order them on one stream. Allocates nothing. */
#define RA_NOALLOC_SCRATCH_BYTES (64u << 20)
int ra_ring_attn_bwd_noalloc(const ra_problem* p, const void* q, const void* k, const void* v,
                             const void* out, const float* lse, const void* dout, void* dq,
                             void* dk, void* dv, void* stream);

/* Natural order <-> shard-major order of a token tensor (row = one token, `row_bytes`
 * bytes: H*Dh*element size), bit-exact copy. direction 0: natural -> shard-major (shard);
 * 1: shard-major -> natural (unshard). src and dst must not overlap. */
int ra_shard_tokens(const ra_problem* p, int direction, const void* src, void* dst,
                    int64_t row_bytes, void* stream);

/* The same permutation for an lse tensor (float32, [B, Hq, S] or [Hq, T]). */
int ra_shard_lse(const ra_problem* p, int direction, const float* src, float* dst,
                 void* stream);

/* ---- host-side integer helpers (no GPU needed; the kernels use the same arithmetic) ---- */

/* 0 if the problem is valid, else the ra_status the compute calls would return. */
int ra_validate(const ra_problem* p);

/* Global positions of sequence `seq` (natural order index; batch element in batch mode):
 * pos_out[r*L + a] = global position of local token a of rank r, L = len/D. */
int ra_layout_positions(const ra_problem* p, int seq, int64_t* pos_out);

/* Per-row key counts of one (rank, step) block of sequence `seq`: the keys a local query
 * row may see in K/V shard (rank-step) mod D always form a prefix [0, count) of that
 * shard's local tokens (positions grow with the local index in every layout). Writes L
 * counts; count 0 = row sees nothing at this step, L = full row. *active_out (may be NULL)
 * is 1 if any row sees a key, i.e. the step is not skipped. */
int ra_step_counts(const ra_problem* p, int seq, int rank, int step, int32_t* count_out,
                   int32_t* active_out);

/* The work list the kernels run, in launch order. which = 0: forward (one item per
 * 256-query-row block of one rank and one query head); which = 1: backward (one item per
 * 128-row K/V tile of one rank and one K/V head). Each item is 4 int32: sequence, head,
 * rank, block index. Writes at most max_items items; returns the item count (or < 0). */
int ra_work_items(const ra_problem* p, int which, int32_t* items_out, int max_items);

/* ---- status ---- */

/* Synchronises the current device, then reports whether any kernel of this library gave
 * up a bounded wait since the last reset: RA_OK or RA_ERR_DEVICE_TIMEOUT (RA_ERR_CUDA if the
 * synchronisation itself failed). reset != 0 clears the flag. */
int ra_check_device_status(int reset);

/* Test hook for the bounded-wait path: launches one CTA that waits, with a limit of
 * `timeout_ns` nanoseconds, on a shared-memory barrier that nothing completes, then gives
 * up, records RA_ERR_DEVICE_TIMEOUT in the device status and returns. */
int ra_test_wait_timeout(uint64_t timeout_ns, void* stream);

/* Test hook for the softmax's FMA-pipe exponential: y[i] = 2^x[i] for n device floats
 * x[i] <= 127, computed the way the forward kernel computes part of its exponentials
 * (range split and a degree-3 polynomial; relative error below 8e-5; inputs below -125
 * give 2^-125). */
int ra_test_exp2_poly(const float* x, float* y, int n, void* stream);

/* Profiling hook: while set (non-NULL), ra_ring_attn_fwd and ra_ring_attn_bwd record
 * `start_event` immediately before and `stop_event` immediately after their main kernels
 * (the fused forward; the backward's K/V-tile pass and query-tile dq pass, or its single
 * pass) on the call's stream, so a caller can time them alone with cudaEventElapsedTime.
 * Both are cudaEvent_t handles owned by the caller; pass NULL, NULL to switch the hook off.
 * Per calling thread. */
int ra_profile_events(void* start_event, void* stop_event);

/* Companion of ra_profile_events: while set (non-NULL), the two-pass backward records
 * `mid_event` between its K/V-tile pass and its dq pass. NULL switches it off. Per
 * calling thread. */
int ra_profile_split_event(void* mid_event);

/* Thread-local message describing the last error of this thread ("" if none). */
const char* ra_last_error(void);

/* RA_VERSION. */
int ra_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
