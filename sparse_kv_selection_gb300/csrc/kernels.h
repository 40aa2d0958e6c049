// Internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace prhs {

// Keys per TMA stage of the scoring kernel, and rows per TMA box when the
// cache is paged (one box never crosses a page: block_size % 16 == 0).
constexpr int SCORE_TILE = 128;
constexpr int PAGED_BOX_ROWS = 16;

// Scores cached in shared memory by the selection kernel (floats).
constexpr int SELECT_CACHE_FLOATS = 48 * 1024;
constexpr int SELECT_THREADS = 1024;
// Logits held in shared memory per CTA by the cluster selection kernel: one
// CTA takes up to SELECT_SLICE_ONE, a cluster of 2..8 CTAs up to
// SELECT_SLICE_MAX each; longer caches use the single-CTA kernel that streams
// them from L2.
constexpr int SELECT_SLICE_ONE = 44032;
constexpr int SELECT_SLICE_MAX = 16384;
// Score-and-select kernel: a cluster of up to SELECT_FUSED_CL CTAs per query
// head, each computing the logits of about SELECT_FUSED_ROWS keys (at most
// SELECT_FUSED_MAX_ROWS) straight from K; longer caches go through the
// separate scoring and selection kernels.
constexpr int SELECT_FUSED_ROWS = 256;
constexpr int SELECT_FUSED_MAX_ROWS = 512;
constexpr int SELECT_FUSED_CL = 16;

struct ScoreLaunch {
  KVView kv;
  const void* q;
  float scale;
  const uint8_t* head_skip;  // [B][Hq] or null
  float* scores;             // [B][Hq][t_max]
  int ctas;                  // CTAs sharing the key tiles of all retrieving KV heads
  bool paged;
};

struct SelectLaunch {
  KVView kv;
  const float* scores;
  int N;
  const int32_t* n_budget;
  const uint8_t* head_skip;
  int32_t* idx;
  int32_t* n_sel;
  int cap;
  float* delta;
  int32_t* anchor_idx;  // all three null or all three set
  int32_t* anchor_n;
  int anchor_cap;
  const void* q;
  void* q_anchor;
  const void* q_src;  // what the anchor copies into q_anchor: q, or the vectors gated on
  int n_sink;  // forced keys are left out of the ranking (the caller adds them)
  int window;
  // score-and-select kernel only: the logits' scale, and where to leave the
  // logits (null: kept in shared memory only)
  float scale;
  float* logits_out;
  // score-and-select kernel only, no forced keys: attention over the selected
  // set into out [B][Hq][d] and lse [B][Hq] (null: selection only)
  float* out;
  float* lse;
};

struct CisLaunch {
  KVView kv;
  const int32_t* anchor_idx;
  const int32_t* anchor_n;
  int anchor_cap;
  const void* q;          // the vectors gated on (queries, or the current tokens' keys)
  const void* q_anchor;
  int w;
  int n_den;              // > 0: budgeted dilation, floor(anchor_n / n_den) positions added
  double tau;
  int max_run;           // 0: reuse runs are unbounded
  int32_t* anchor_age;   // [B][Hq] reuses since the anchor retrieved (null when max_run == 0)
  int32_t* idx;
  int32_t* n_sel;
  int cap;
  uint8_t* reuse;
  int n_sink;            // forced keys: the first n_sink and the last `window` of each cache
  int window;
};

// A CTA of the attention kernels takes at least this many rows: below it the
// fixed per-CTA cost (prefix, index staging, partial record, merge) outweighs
// the extra parallelism.
constexpr int ATTN_MIN_ROWS = 64;
// CTAs per SM of the V-only (logit-source) attention: its register budget
// allows six 128-thread CTAs where the K-and-V form fits four.
constexpr int ATTN_LG_CTAS_PER_SM = 6;
// The same floor for the reusing heads' branch of a decode step, which runs
// beside the retrieving heads' scoring and selection: when the reused sets
// are small, fewer and fuller CTAs leave room on the SMs for those kernels.
constexpr int ATTN_SIDE_MIN_ROWS = 192;

struct AttnLaunch {
  KVView kv;
  const void* q;
  float scale;
  const int32_t* idx;    // sparse: [B][Hq][cap]; dense: null
  const int32_t* n_sel;  // sparse: [B][Hq]
  const uint8_t* unit_mask;  // sparse, nullable: attend only units u with (mask[u] != 0) == mask_want
  int mask_want;
  int cap;
  float* out;
  float* lse;
  float* partials;       // [ctas + units][G][d + 4]
  unsigned* counters;    // [units], zero on entry, left zero
  int ctas;              // CTAs sharing the rows of all units
  int min_rows;          // fewest rows a CTA takes (fewer CTAs join small batches)
  int cluster = 0;       // sparse only: > 0 runs the cluster kernel with this many CTAs per head
  // sparse only, nullable: the logits scale * <q, k_i> of every query head
  // ([B][Hq][t_max], as the scoring kernel leaves them); the attention then
  // takes each selected row's weight from there and reads only its V row
  const float* logits = nullptr;
};

// Dropped mass of given sets over the logits in `scores` ([B][Hq][t_max]).
struct MassLaunch {
  KVView kv;
  const float* scores;
  const int32_t* idx;
  const int32_t* n_sel;
  int cap;
  float* delta;
  const uint8_t* head_skip = nullptr;  // heads with a nonzero flag are left untouched
  float* partials = nullptr;   // [units][parts][4] when a head is split (workspace)
  unsigned* counters = nullptr;  // [units], zero at rest
  int chunk = 0;               // keys per part (set by launch_mass)
};
// A head's keys are split into parts of MASS_CHUNK keys, at most
// MASS_PARTS_MAX (4 floats per part must fit a unit's attention partial record).
constexpr int MASS_CHUNK = 8192;
constexpr int MASS_PARTS_MAX = 16;
int mass_parts(int t_max);
cudaError_t launch_mass(const MassLaunch& a, cudaStream_t s);

// Attended set of a retrieving head with forced keys: the first n_sink keys,
// the head's middle top-N set (its anchor row) and the last `window` keys.
struct ComposeLaunch {
  KVView kv;
  const uint8_t* head_skip;
  const int32_t* anchor_idx;
  const int32_t* anchor_n;
  int anchor_cap;
  int32_t* idx;
  int32_t* n_sel;
  int cap;
  int n_sink;
  int window;
};
cudaError_t launch_compose(const ComposeLaunch& a, cudaStream_t s);

// Appends one key and value row per (sequence, KV head) at position
// seq_lens[b] and increments seq_lens[b].
struct AppendLaunch {
  KVView kv;
  const void* k_new;  // [B][Hkv][d]
  const void* v_new;
  int32_t* seq_lens;
};
cudaError_t launch_append(const AppendLaunch& a, cudaStream_t s);

// Units of the attention split (query heads when sparse, KV heads when dense)
// and the floats of partial records the kernel may write for `ctas` CTAs.
int attn_units(const KVView& kv, bool sparse);
size_t attn_partial_floats(const KVView& kv, bool sparse, int ctas);

cudaError_t launch_score(const ScoreLaunch& a, const CUtensorMap* tmap, cudaStream_t s);
cudaError_t launch_select(const SelectLaunch& a, cudaStream_t s);
cudaError_t launch_select_global(const SelectLaunch& a, cudaStream_t s);
// Logits and selection in one launch (a.scale, a.logits_out; a.scores unused),
// and the attention over the selected set when a.out is set (no forced keys).
// Returns cudaErrorNotSupported when the cache is too long for it.
bool score_select_fits(const KVView& kv);
cudaError_t launch_score_select(const SelectLaunch& a, cudaStream_t s);
// The cluster size and slice length of the score-and-select kernels (false:
// the cache is too long for them), and their launch: one cluster of cl CTAs
// per query head, with programmatic dependent launch when the view allows it.
bool score_select_geometry(const KVView& kv, int* cl, int* chunk);
cudaError_t launch_select_grid(void (*k)(const SelectLaunch, int), const SelectLaunch& a, int cl,
                               int chunk, size_t smem, cudaStream_t s);
// Retrieval in one launch (logits, selection spread over the cluster, the
// attention over the set): a.out and a.lse set, no forced keys.
cudaError_t launch_retrieve(const SelectLaunch& a, cudaStream_t s);
cudaError_t launch_cis(const CisLaunch& a, cudaStream_t s);
cudaError_t launch_attn(const AttnLaunch& a, bool sparse, cudaStream_t s);
// Sparse attention with one thread-block cluster of a.cluster CTAs per query
// head (batches with few heads; no workspace).
constexpr int ATTN_CLUSTER_MAX = 8;
// The decode step's reusing-heads branch runs beside the retrieval's
// 16-CTA clusters; clusters of at most this many CTAs leave the SM room both
// need (measured on the llama shape: 1.515 -> 1.597 M query-heads/s, though
// the attention alone is 9.2 us with 8-CTA clusters against 11.3 with 4).
constexpr int ATTN_SIDE_CLUSTER_MAX = 4;
cudaError_t launch_attn_cluster(const AttnLaunch& a, cudaStream_t s);

// Hooks into the C ABI layer for the library's other entry-point files:
// descriptor checks, per-device facts (error word, SM count), the failure
// message of prhs_last_message, and the CTA count of the attention kernels.
prhs_status abi_check_kv(const prhs_kv* kv);
prhs_status abi_device(unsigned** err, int* sms);
prhs_status abi_fail(prhs_status s, const char* msg);
void abi_count_launch();  // one more kernel issued (entry points outside the ABI file)
KVView abi_view(const prhs_kv& kv, unsigned* err);
int abi_attn_ctas(const prhs_kv& kv, bool sparse, int cap, int sms);

// Dense attention through TMA-staged K/V tiles (one launch per call).
cudaError_t launch_dense(const KVView& kv, const void* q, float scale, float* out, float* lse,
                         float* partials, unsigned* counters, int ctas, bool paged,
                         const CUtensorMap* kmap, const CUtensorMap* vmap, cudaStream_t st);
size_t dense_partial_floats(const KVView& kv, int ctas);
int dense_rows_per_stage(const KVView& kv);

// Bytes of dynamic shared memory the scoring kernel needs for this shape.
size_t score_smem_bytes(prhs_dtype dt, int d);

}  // namespace prhs
