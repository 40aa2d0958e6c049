/*
 * prhs.h - C ABI of the GB300 (sm_103a) Pre-hoc Sparsity decode path.
 *
 * Source of the operations: "Near-Oracle KV Selection via Pre-hoc Sparsity
 * for Long-Context Inference" (arXiv 2602.08329): the abstract (top-k oracle
 * selection before attention, dropped mass delta), Table I (notation: K, V,
 * t, N, S_t, tau(.), delta(.)), Fig. 2 / Fig. 8 (sharing between queries
 * whose similarity is >= tau = 0.8), Fig. 4 and Table VIII (critical-index
 * set dilation, radius r) and the Table V caption (a fused sparse-attention
 * kernel over the selected KV entries).
 *
 * Conventions shared by every call:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    allocates no device memory. Scratch comes from a caller workspace sized
 *    by prhs_workspace_size() and zero-filled once by prhs_workspace_init().
 *  - Calls are asynchronous on the given stream. Arguments are checked on
 *    the host before any launch; a bad argument returns PRHS_EINVAL (or
 *    PRHS_EUNSUPPORTED for a valid but unbuilt shape) and launches nothing.
 *    prhs_last_message() then describes the failure.
 *  - Errors found by kernels (an index outside [0, t_b), a page number
 *    outside the pool, a wait that timed out, a set larger than its row
 *    capacity) set bits in a device error word; the offending element is
 *    skipped, nothing faults. prhs_last_error() synchronises the device,
 *    reads and clears that word.
 *  - Layouts (row-major, innermost last):
 *      q, q_anchor   [B][Hq][d]      same element type as the cache, 16-byte aligned
 *      K, V          contiguous [B][Hkv][t_max][d]
 *                    or paged   [num_blocks][Hkv][block_size][d]
 *      idx           [B][Hq][cap]    int32, ascending, n_sel valid entries
 *      n_sel, n_budget, anchor_n     int32 [B][Hq] (n_budget: [B])
 *      reuse         uint8 [B][Hq];  delta, lse float [B][Hq]; out float [B][Hq][d]
 *    Query head h reads KV head h / (Hq / Hkv).
 *  - Inputs must be finite; NaN or Inf in q, K or V gives undefined results.
 *  - No call is thread-safe against another call using the same workspace.
 *    prhs_decode_step keeps one internal side stream (and fork/join events)
 *    per caller stream, created by the first decode step on that stream:
 *    make that first step outside stream capture. Steps on different caller
 *    streams, each with its own workspace and buffers, may run concurrently.
 */
#ifndef PRHS_H
#define PRHS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PRHS_OK = 0,
  PRHS_EINVAL = 1,        /* bad argument (null pointer, size, alignment, capacity) */
  PRHS_EUNSUPPORTED = 2,  /* head dim / dtype / group size not built */
  PRHS_EWORKSPACE = 3,    /* workspace null or smaller than prhs_workspace_size() */
  PRHS_ECUDA = 4,         /* a CUDA runtime call failed (launch, attribute, encode) */
  PRHS_EDEVICE = 5        /* a kernel reported a data error (see prhs_device_error_bits) */
} prhs_status;

typedef enum { PRHS_F32 = 0, PRHS_BF16 = 1 } prhs_dtype;

/* device error word bits (prhs_device_error_bits) */
#define PRHS_DEV_TIMEOUT   1u   /* a bounded barrier wait gave up */
#define PRHS_DEV_BAD_INDEX 2u   /* idx / anchor entry outside [0, t_b) or not ascending */
#define PRHS_DEV_BAD_LEN   4u   /* seq_lens[b] outside [0, t_max] */
#define PRHS_DEV_BAD_BLOCK 8u   /* block_table entry outside [0, num_blocks) */
#define PRHS_DEV_CAPACITY  16u  /* a result set did not fit its row capacity */

/* KV cache descriptor (Table I: K, V, t; H heads of dimension d).
 * Host struct; its pointers are device pointers, borrowed for the call only. */
typedef struct prhs_kv {
  prhs_dtype dtype;            /* element type of K, V and q */
  int B;                       /* sequences in the batch */
  int Hq;                      /* query heads per sequence */
  int Hkv;                     /* KV heads per sequence; Hq % Hkv == 0, Hq/Hkv in {1,2,4,8} */
  int d;                       /* head dimension: 64 or 128 */
  const void* k;               /* K rows, 16-byte aligned */
  const void* v;               /* V rows, same layout as K */
  int t_max;                   /* contiguous: keys per (b, kv head) row stride.
                                  paged: ignored (max_blocks * block_size is used) */
  const int32_t* seq_lens;     /* [B] cache length t_b of each sequence, 0 <= t_b <= t_max */
  const int32_t* block_table;  /* NULL: contiguous. else [B][max_blocks] physical page ids */
  int block_size;              /* paged: keys per page, a positive multiple of 16 */
  int max_blocks;              /* paged: columns of block_table */
  int num_blocks;              /* paged: pages in the pool (bounds check) */
} prhs_kv;

/* Bytes of workspace that every call below needs for this cache and a
 * per-head set capacity `cap` (scores [B][Hq][t_max] f32 plus split-K
 * partials and counters). Returns 0 for an invalid descriptor. */
size_t prhs_workspace_size(const prhs_kv* kv, int cap);

/* Zero-fill the workspace's completion counters (required once after the
 * workspace is allocated; every later call leaves them zero again). */
prhs_status prhs_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Top-N oracle selector (abstract: "near-oracle top-k KV selection"; Table I:
 * S_t, N, delta). For every query head not flagged in head_skip:
 *   s_i = scale * <q, k_i>, i < t_b;  A = softmax(s);
 *   S = the N largest s_i (ties -> lowest index), written ascending to idx;
 *   delta = sum_{i not in S} A_i.
 * N is `N`, or n_budget[b] when n_budget != NULL. When N >= t_b the set is
 * all of [0, t_b) and delta = 0. cap >= max budget is required.
 * head_skip [B][Hq] uint8 (nullable): heads with a nonzero flag are left
 * untouched (their idx, n_sel and delta rows are not written).
 * anchor_idx / anchor_n / q_anchor (all nullable together): also copy each
 * written set, its size and the query into these anchor buffers (the CIS
 * anchor, row capacity anchor_cap).
 * Forced keys (Fig. 11: attention sinks and the recent window), n_sink >= 0
 * and window >= 0, 0 and 0 for none: the first n_sink and the last `window`
 * keys of each cache are left out of the ranking; the N largest are taken
 * among the keys between them, and the written set is the forced keys, those
 * N and nothing else (ascending); delta is its dropped mass; the anchor row
 * gets only the N ranked keys. Forced keys need the anchor buffers and a
 * t_max of at most 131072; cap >= N + n_sink + window. */
prhs_status prhs_score_select(const prhs_kv* kv, const void* q, float scale, int N,
                              const int32_t* n_budget, int n_sink, int window,
                              const uint8_t* head_skip, int32_t* idx, int32_t* n_sel, int cap,
                              float* delta, int32_t* anchor_idx, int32_t* anchor_n,
                              int anchor_cap, void* q_anchor, void* ws, size_t ws_bytes,
                              cudaStream_t stream);

/* Retrieval for the query heads not flagged in head_skip (in a decode step,
 * the heads that do not reuse an anchor): the set, its size, delta and the
 * anchor copies exactly as prhs_score_select writes them (same arguments),
 * and the attention over that set as prhs_sparse_attn computes it,
 *   out[b][h] = sum_{i in S} A_i v_i / sum_{i in S} A_i  (fp32, [B][Hq][d]),
 *   lse[b][h] = log sum_{i in S} exp(s_i)                 ([B][Hq]),
 * out = 0 and lse = -inf for an empty set. Rows of flagged heads are left
 * untouched. A cache of t_max <= 8192 without forced keys takes one kernel
 * launch (logits, selection and attention in one thread-block cluster per
 * head); otherwise it is scoring, selection (with the forced keys' passes)
 * and an attention launch that weights each selected V row by the logit the
 * scoring left in the workspace (K rows are read once, by the scoring).
 * out and lse must be non-null. */
prhs_status prhs_retrieve(const prhs_kv* kv, const void* q, float scale, int N,
                          const int32_t* n_budget, int n_sink, int window,
                          const uint8_t* head_skip, int32_t* idx, int32_t* n_sel, int cap,
                          float* delta, int32_t* anchor_idx, int32_t* anchor_n, int anchor_cap,
                          void* q_anchor, float* out, float* lse, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

/* The two halves of prhs_score_select, for callers that time or reuse them
 * separately. prhs_score writes the logits s_i = scale * <q, k_i> of every
 * query head not flagged in head_skip into the workspace; prhs_select then
 * selects from the logits the last prhs_score call on the same workspace left
 * there (same q, kv and head_skip), with the arguments and results of
 * prhs_score_select. */
prhs_status prhs_score(const prhs_kv* kv, const void* q, float scale, const uint8_t* head_skip,
                       void* ws, size_t ws_bytes, cudaStream_t stream);
prhs_status prhs_select(const prhs_kv* kv, const void* q, int N, const int32_t* n_budget,
                        int n_sink, int window, const uint8_t* head_skip, int32_t* idx,
                        int32_t* n_sel, int cap, float* delta, int32_t* anchor_idx,
                        int32_t* anchor_n, int anchor_cap, void* q_anchor, void* ws,
                        size_t ws_bytes, cudaStream_t stream);

/* Critical-index-set reuse with dilation (Fig. 2, Fig. 4, Fig. 8, Table VIII).
 * Per query head: c = <q, q_anchor> / (|q| |q_anchor|); the decision is the
 * one of that formula in float64 (an fp32 estimate decides when it is more
 * than 1e-4 away from tau, its error being below 2e-6; float64 otherwise);
 * reuse = anchor_n > 0 and |q| |q_anchor| > 0 and c >= tau, and, when
 * max_run > 0, anchor_age < max_run - 1: the CIS block size s of Tables IV,
 * V and VIII read as the most consecutive queries one retrieval serves.
 * anchor_age [B][Hq] int32 counts reuses since the anchor retrieved; it is
 * required when max_run > 0 (nullable otherwise) and is updated to
 * reuse ? age + 1 : 0.
 * When reuse: idx = union over anchor entries a of [a - w, a + w] clipped to
 * [0, t_b), ascending without repeats, n_sel its size (<= cap required).
 * Budgeted dilation (Fig. 9a, dilation strength m = floor(k / n_den)): with
 * n_den > 0 only m = floor(anchor_n / n_den) of those neighbours are added to
 * the anchor entries, the nearest to an anchor entry first and, at equal
 * distance, the lowest position first (n_den = 0: all of them; m = 0: the
 * anchor set itself).
 * When not: idx and n_sel rows are left untouched. reuse [B][Hq] is always
 * written. anchor_idx rows must be ascending and inside [0, t_b).
 * q is the vectors the gate compares with q_anchor: the queries, or for the
 * "Key" similarity design of Table IX the current tokens' keys (one per query
 * head, [B][Hq][d]).
 * Forced keys (n_sink, window as in prhs_score_select): the dilated set is
 * united with [0, n_sink) and [t_b - window, t_b) (clipped), still ascending
 * without repeats; cap >= min(t_max, anchor_cap * (2w + 1) + n_sink + window). */
prhs_status prhs_cis_dilate(const prhs_kv* kv, const int32_t* anchor_idx,
                            const int32_t* anchor_n, int anchor_cap, const void* q,
                            const void* q_anchor, int w, int n_den, int n_sink, int window,
                            double tau, int max_run, int32_t* anchor_age, int32_t* idx,
                            int32_t* n_sel, int cap, uint8_t* reuse, cudaStream_t stream);

/* Dropped attention mass of given index sets under the current query (a
 * diagnostic for reuse steps, whose set was not selected under this query;
 * abstract: the attention mass of discarded entries; Table I: delta(.)).
 * Per query head with n = n_sel entries of idx (ascending, inside [0, t_b)):
 *   s_i = scale * <q, k_i>, i < t_b;  delta = sum_{i < t_b, i not in idx} softmax(s)_i.
 * n = 0 gives 1 (0 when t_b = 0). Scores every head through the workspace
 * (ws from prhs_workspace_size(kv, 0)); entries out of range or not
 * ascending are flagged in the device error word and skipped. */
prhs_status prhs_set_mass(const prhs_kv* kv, const void* q, float scale, const int32_t* idx,
                          const int32_t* n_sel, int cap, float* delta, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

/* Sparse attention over the selected rows (Table V caption: sparse-attention
 * kernel over the selected KV): per query head with n = n_sel entries of idx,
 *   lse = log sum_{i in S} exp(s_i),  out = sum_{i in S} exp(s_i - lse) v_i,
 * s_i = scale * <q, k_i>; natural log; fp32 accumulation. n = 0 gives
 * out = 0, lse = -inf. Entries outside [0, t_b) are skipped and flagged. */
prhs_status prhs_sparse_attn(const prhs_kv* kv, const void* q, float scale,
                             const int32_t* idx, const int32_t* n_sel, int cap,
                             float* out, float* lse, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/* Sparse attention that allocates nothing, for callers that cannot call
 * cudaMalloc and so cannot hand the library a workspace (a plugin host that
 * owns all device memory, a serving loop that may not take cudaMalloc's
 * device synchronisation). The paper has no counterpart: this is a library
 * convenience. Same arguments and results as prhs_sparse_attn minus the
 * workspace; the split-K scratch is a fixed device array of
 * PRHS_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that
 * loads it until the process exits. A batch whose scratch (256-byte-rounded
 * B*Hq tickets plus (ctas + B*Hq)*(d+4) floats, ctas <= 4 per SM) exceeds
 * that size returns PRHS_EINVAL. The first call on each device resolves the array's device
 * address (cudaGetSymbolAddress), so make that first call before any stream
 * capture. Every call shares the array: calls that overlap on the GPU (other
 * streams, other threads) race and give wrong results; serialise them. Each
 * call clears its tickets with cudaMemsetAsync before the kernel runs; it
 * calls no cudaMalloc, cudaFree or allocating routine. */
#define PRHS_NOALLOC_SCRATCH_BYTES (4u << 20)
prhs_status prhs_sparse_attn_noalloc(const prhs_kv* kv, const void* q, float scale,
                                     const int32_t* idx, const int32_t* n_sel, int cap,
                                     float* out, float* lse, cudaStream_t stream);

/* Dense attention over all t_b keys (the dense baseline of Table IV), with
 * the same outputs as prhs_sparse_attn over idx = [0, t_b). One query head per
 * KV head (MHA): the row-gather attention kernel over [0, t_b). Grouped heads:
 * K and V tiles are staged in shared memory by TMA and every query head of the
 * group is computed from the same tile, so each row is read from HBM once.
 * Errors as prhs_sparse_attn; ws from prhs_workspace_size(kv, 0). */
prhs_status prhs_dense_attn(const prhs_kv* kv, const void* q, float scale, float* out,
                            float* lse, void* ws, size_t ws_bytes, cudaStream_t stream);

/* One decode step with CIS reuse, stream-ordered, no host round trip:
 *   prhs_cis_dilate(anchor -> idx, reuse);
 *   the reusing heads: prhs_sparse_attn(idx) on an internal side stream;
 *   the others: prhs_retrieve(head_skip = reuse, anchor outputs = the anchor
 *   buffers) on `stream`, which then waits for the side stream (when the
 *   retrieving branch is small, its scoring runs before the side stream
 *   forks and the rest beside the side stream; results are the same).
 * Heads that reuse attend the dilated anchor set; the others retrieve a fresh
 * top-N set, attend it and make it (with the gated vector) the new anchor.
 * delta is written for retrieving heads only. Start a sequence with anchor_n
 * (and anchor_age) all zero; max_run, anchor_age and n_den (budgeted
 * dilation) as in prhs_cis_dilate; n_sink and window (forced keys) as in
 * prhs_score_select and prhs_cis_dilate.
 * gate (nullable, [B][Hq][d], the cache's element type, 16-byte aligned):
 * the vectors the CIS gate compares, in place of q; the "Key" similarity
 * design of Table IX passes the key each sequence appended for this token
 * (its KV head's row for every query head of the group). q_anchor then holds
 * the gate vector of each head's anchor. */
prhs_status prhs_decode_step(const prhs_kv* kv, const void* q, const void* gate, float scale, int N,
                             const int32_t* n_budget, int n_sink, int window, int w, int n_den,
                             double tau, int max_run, int32_t* anchor_age, int32_t* anchor_idx,
                             int32_t* anchor_n, int anchor_cap, void* q_anchor, int32_t* idx,
                             int32_t* n_sel, int cap, uint8_t* reuse, float* delta, float* out,
                             float* lse, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Grow the cache by one key per sequence (decoding appends the current
 * token's key and value before it attends): for every sequence b and KV head
 * h, k_new[b][h][:] and v_new[b][h][:] (device, [B][Hkv][d], the cache's
 * element type, 16-byte aligned) are written at position seq_lens[b] of the cache, then
 * seq_lens[b] (the descriptor's device array) is advanced by one. A paged
 * cache must already map that position to a page. A sequence whose length
 * is already t_max is left as it is and flagged (PRHS_DEV_CAPACITY). */
prhs_status prhs_append_kv(const prhs_kv* kv, const void* k_new, const void* v_new,
                           cudaStream_t stream);

/* Self-test of the kernels' failure path (no counterpart in the paper): one
 * warp waits on a shared-memory mbarrier that nothing arrives on, through the
 * same bounded wait every TMA pipeline of the library uses, but giving up
 * after limit_us microseconds (1 <= limit_us <= 1000000) instead of about a
 * second. The wait runs out, PRHS_DEV_TIMEOUT is set in the device error word
 * and the kernel returns; no fault, the context stays usable. A following
 * prhs_last_error() returns PRHS_EDEVICE with that bit. */
prhs_status prhs_selftest_wait_timeout(unsigned limit_us, cudaStream_t stream);

/* Synchronise the current device, read and clear the device error word.
 * PRHS_OK when it was zero, PRHS_EDEVICE otherwise, PRHS_ECUDA when the
 * synchronisation itself failed. */
prhs_status prhs_last_error(void);

/* Bits of the device error word seen by the last prhs_last_error(). */
unsigned prhs_device_error_bits(void);

/* Text of a status code; text of the calling thread's last host-side failure. */
const char* prhs_status_str(prhs_status s);
const char* prhs_last_message(void);

/* Launch geometry the library picks for this device (for benchmarks and
 * tests): SM count and split-K factors of the attention kernels. */
int prhs_num_sms(void);

/* Kernels this library has issued (launched, or recorded into a CUDA graph
 * being captured) since it was loaded, over all threads. Read it before and
 * after a call to count that call's launches. */
unsigned long long prhs_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* PRHS_H */
