// C ABI of the PrHS decode path: argument checks, workspace layout, TMA
// descriptor encoding and kernel launches. Declarations and the contract of
// every entry point are in include/prhs.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.h"

namespace prhs {

__device__ unsigned int g_error_word = 0;

namespace {

thread_local std::string t_message;
unsigned g_last_bits = 0;

prhs_status fail(prhs_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
prhs_status fail(prhs_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_message = buf;
  return s;
}

prhs_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PRHS_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The second branch of prhs_decode_step for one caller stream: its own side
// stream and fork/join events, so that decode steps issued on different
// caller streams (other host threads, other workspaces) never share an event
// or land on a stream another caller is capturing. `mu` keeps one step's
// record/wait sequence whole when several threads use the same caller stream.
struct SideBranch {
  cudaStream_t caller = nullptr;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};

constexpr int MAX_DEVICES = 64;
struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  unsigned* err = nullptr;
  std::vector<std::unique_ptr<SideBranch>> branches;  // one per caller stream seen
};
DeviceInfo g_dev[MAX_DEVICES];
std::mutex g_dev_mu;

// Per-device facts resolved once, with that device current.
prhs_status device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= MAX_DEVICES) return fail(PRHS_ECUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    di.err = static_cast<unsigned*>(p);
    di.ready = true;
  }
  *out = &di;
  return PRHS_OK;
}

// The side branch of `caller` on the current device, created on first use.
prhs_status side_branch(DeviceInfo* di, cudaStream_t caller, SideBranch** out) {
  std::lock_guard<std::mutex> lock(g_dev_mu);
  for (auto& b : di->branches)
    if (b->caller == caller) {
      *out = b.get();
      return PRHS_OK;
    }
  std::unique_ptr<SideBranch> b(new SideBranch);
  b->caller = caller;
  cudaError_t e = cudaStreamCreateWithFlags(&b->side, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreateWithFlags (decode side stream)");
  e = cudaEventCreateWithFlags(&b->fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b->join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cudaStreamDestroy(b->side);
    return cuda_fail(e, "cudaEventCreateWithFlags (decode fork/join)");
  }
  *out = b.get();
  di->branches.push_back(std::move(b));
  return PRHS_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// ---------------------------------------------------------------------------
// descriptor checks
// ---------------------------------------------------------------------------
constexpr int MAX_UNITS = 16384;  // B * Hq: bounds the kernels' shared prefix arrays

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int t_max_of(const prhs_kv& kv) {
  return kv.block_table != nullptr ? kv.max_blocks * kv.block_size : kv.t_max;
}

prhs_status check_kv(const prhs_kv* kv) {
  if (kv == nullptr) return fail(PRHS_EINVAL, "kv descriptor is null");
  if (kv->dtype != PRHS_F32 && kv->dtype != PRHS_BF16)
    return fail(PRHS_EINVAL, "unknown dtype %d", (int)kv->dtype);
  if (kv->B <= 0 || kv->Hq <= 0 || kv->Hkv <= 0)
    return fail(PRHS_EINVAL, "B, Hq, Hkv must be positive (got %d, %d, %d)", kv->B, kv->Hq, kv->Hkv);
  if (kv->Hq % kv->Hkv != 0) return fail(PRHS_EINVAL, "Hq %% Hkv != 0");
  if ((long long)kv->B * kv->Hq > MAX_UNITS)
    return fail(PRHS_EUNSUPPORTED, "B * Hq = %lld above %d", (long long)kv->B * kv->Hq, MAX_UNITS);
  const int G = kv->Hq / kv->Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(PRHS_EUNSUPPORTED, "query group Hq/Hkv = %d not built (1, 2, 4, 8)", G);
  if (kv->d != 64 && kv->d != 128) return fail(PRHS_EUNSUPPORTED, "head dim %d not built (64, 128)", kv->d);
  if (kv->k == nullptr || kv->v == nullptr || kv->seq_lens == nullptr)
    return fail(PRHS_EINVAL, "k, v and seq_lens must be non-null");
  if (!aligned16(kv->k) || !aligned16(kv->v)) return fail(PRHS_EINVAL, "k and v must be 16-byte aligned");
  if (kv->block_table != nullptr) {
    if (kv->block_size <= 0 || kv->block_size % 16 != 0)
      return fail(PRHS_EINVAL, "block_size must be a positive multiple of 16 (got %d)", kv->block_size);
    if (kv->max_blocks <= 0 || kv->num_blocks <= 0)
      return fail(PRHS_EINVAL, "max_blocks and num_blocks must be positive");
    const long long rows = (long long)kv->num_blocks * kv->Hkv * kv->block_size;
    if (rows >= (1ll << 31)) return fail(PRHS_EINVAL, "paged pool too large (%lld rows)", rows);
    if ((long long)kv->max_blocks * kv->block_size >= (1ll << 30))
      return fail(PRHS_EINVAL, "max_blocks * block_size too large");
  } else {
    if (kv->t_max <= 0) return fail(PRHS_EINVAL, "t_max must be positive (got %d)", kv->t_max);
    const long long rows = (long long)kv->B * kv->Hkv * kv->t_max;
    if (rows >= (1ll << 31)) return fail(PRHS_EINVAL, "cache too large (%lld rows)", rows);
  }
  return PRHS_OK;
}

KVView view_of(const prhs_kv& kv, unsigned* err) {
  KVView v;
  v.dtype = kv.dtype;
  v.k = kv.k;
  v.v = kv.v;
  v.seq_lens = kv.seq_lens;
  v.block_table = kv.block_table;
  v.B = kv.B;
  v.Hq = kv.Hq;
  v.Hkv = kv.Hkv;
  v.d = kv.d;
  v.t_max = t_max_of(kv);
  v.block_size = kv.block_table ? kv.block_size : 1;
  v.max_blocks = kv.block_table ? kv.max_blocks : 0;
  v.num_blocks = kv.block_table ? kv.num_blocks : 0;
  v.err = err;
  v.pdl = v.t_max <= PDL_MAX_KEYS;
  return v;
}

size_t elem_size(prhs_dtype dt) { return dt == PRHS_BF16 ? 2 : 4; }

// ---------------------------------------------------------------------------
// launch geometry and workspace layout
// ---------------------------------------------------------------------------
constexpr int ATTN_CTAS_PER_SM = 4;
constexpr int SCORE_CTAS_PER_SM = 2;

// CTAs of the attention kernels: enough for every SM to hold per_sm (four
// for the K-and-V form, ATTN_LG_CTAS_PER_SM for the V-only one), fewer when
// the rows can be bounded from the host (about 32 rows per CTA).
int attn_ctas(const prhs_kv& kv, bool sparse, int cap, int sms, int per_sm = ATTN_CTAS_PER_SM) {
  const long long units = (long long)kv.B * kv.Hq;  // both kernels split by query head
  const long long rows = units * (sparse ? cap : t_max_of(kv));
  long long c = (rows + 31) / 32;
  const long long most = (long long)per_sm * sms;
  if (c > most) c = most;
  return c < 1 ? 1 : (int)c;
}

// CTAs per query head of the cluster attention kernel, or 0 for the balanced
// kernel. Clusters pay off when the whole launch is small (at most 256 rows
// per CTA slot, rows_hint rows per head at most) and the heads are few enough
// that each can have at least two CTAs within ATTN_CTAS_PER_SM CTAs per SM;
// then as many CTAs per head (a power of two up to ATTN_CLUSTER_MAX) as fit,
// each with at least 64 of rows_hint rows. Large launches keep the balanced
// kernel, which fills every SM whatever the number of heads.
int attn_cluster_size(const prhs_kv& kv, int rows_hint, int sms) {
  const long long units = (long long)kv.B * kv.Hq;
  const long long slots = (long long)ATTN_CTAS_PER_SM * sms;
  if (units * 2 > slots || units * rows_hint > slots * 256) return 0;
  int cl = 1;
  while (cl * 2 <= ATTN_CLUSTER_MAX && units * cl * 2 <= slots && rows_hint >= 64ll * cl * 2) cl *= 2;
  return cl;
}

struct Layout {
  size_t counters, partials, partials2, scores, total;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

Layout layout_of(const prhs_kv& kv, int sms) {
  Layout L;
  const KVView v = view_of(kv, nullptr);
  const int most = (ATTN_CTAS_PER_SM > ATTN_LG_CTAS_PER_SM ? ATTN_CTAS_PER_SM : ATTN_LG_CTAS_PER_SM) * sms;
  const size_t ps = attn_partial_floats(v, true, most);
  const size_t pd0 = dense_partial_floats(v, sms);
  const size_t pd = pd0 > ps ? pd0 : ps;
  const size_t units = (size_t)kv.B * kv.Hq;  // >= B * Hkv
  L.counters = 0;
  L.partials = round_up(units * sizeof(unsigned), 256);
  L.partials2 = round_up(L.partials + (ps > pd ? ps : pd) * sizeof(float), 256);
  L.scores = round_up(L.partials2 + ps * sizeof(float), 256);
  L.total = round_up(L.scores + (size_t)kv.B * kv.Hq * t_max_of(kv) * sizeof(float), 256);
  return L;
}

prhs_status check_ws(const prhs_kv& kv, int sms, void* ws, size_t ws_bytes, Layout* L) {
  *L = layout_of(kv, sms);
  if (ws == nullptr) return fail(PRHS_EWORKSPACE, "workspace is null");
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(PRHS_EWORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < L->total)
    return fail(PRHS_EWORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, L->total);
  return PRHS_OK;
}

// TMA descriptor over K viewed as [rows][d*esize/128][128 bytes] with the
// 128-byte swizzle; boxes of `box_rows` rows.
prhs_status make_tmap(const prhs_kv& kv, int box_rows, CUtensorMap* map, const void* base = nullptr) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(PRHS_ECUDA, "cuTensorMapEncodeTiled unavailable");
  const size_t es = elem_size(kv.dtype);
  const cuuint64_t inner = 128 / es;
  const cuuint64_t segs = kv.d * es / 128;
  const cuuint64_t rows = kv.block_table != nullptr
                              ? (cuuint64_t)kv.num_blocks * kv.Hkv * kv.block_size
                              : (cuuint64_t)kv.B * kv.Hkv * kv.t_max;
  const cuuint64_t dims[3] = {inner, segs, rows};
  const cuuint64_t strides[2] = {128, (cuuint64_t)kv.d * es};  // bytes, dims 1 and 2
  const cuuint32_t box[3] = {(cuuint32_t)inner, (cuuint32_t)segs, (cuuint32_t)box_rows};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, kv.dtype == PRHS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                   3, const_cast<void*>(base != nullptr ? base : kv.k), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PRHS_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return PRHS_OK;
}

std::atomic<unsigned long long> g_launches{0};  // kernels issued since load

prhs_status launch_result(cudaError_t e, const char* what) {
  if (e == cudaSuccess) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return PRHS_OK;
  }
  if (e == cudaErrorNotSupported) return fail(PRHS_EUNSUPPORTED, "%s: shape not built", what);
  return cuda_fail(e, what);
}

prhs_status do_score(const prhs_kv& kv, DeviceInfo* di, const Layout& L, void* ws, const void* q,
                     float scale, const uint8_t* head_skip, cudaStream_t st) {
  CUtensorMap map;
  const bool paged = kv.block_table != nullptr;
  prhs_status s = make_tmap(kv, paged ? PAGED_BOX_ROWS : SCORE_TILE, &map);
  if (s != PRHS_OK) return s;
  ScoreLaunch sl;
  sl.kv = view_of(kv, di->err);
  sl.q = q;
  sl.scale = scale;
  sl.head_skip = head_skip;
  sl.scores = reinterpret_cast<float*>(static_cast<char*>(ws) + L.scores);
  sl.paged = paged;
  sl.ctas = SCORE_CTAS_PER_SM * di->sms;
  return launch_result(launch_score(sl, &map, st), "score kernel");
}

prhs_status do_select(const prhs_kv& kv, DeviceInfo* di, const Layout& L, void* ws,
                      const void* q, int N, const int32_t* n_budget, int n_sink, int window,
                      const uint8_t* head_skip,
                      int32_t* idx, int32_t* n_sel, int cap, float* delta, int32_t* anchor_idx,
                      int32_t* anchor_n, int anchor_cap, void* q_anchor, cudaStream_t st,
                      const void* q_src = nullptr) {
  SelectLaunch se;
  se.kv = view_of(kv, di->err);
  se.scores = reinterpret_cast<float*>(static_cast<char*>(ws) + L.scores);
  se.N = N;
  se.n_budget = n_budget;
  se.head_skip = head_skip;
  se.idx = idx;
  se.n_sel = n_sel;
  se.cap = cap;
  se.delta = delta;
  se.anchor_idx = anchor_idx;
  se.anchor_n = anchor_n;
  se.anchor_cap = anchor_cap;
  se.q = q;
  se.q_anchor = q_anchor;
  se.q_src = q_src != nullptr ? q_src : q;
  se.n_sink = n_sink;
  se.window = window;
  se.scale = 0.f;
  se.logits_out = nullptr;
  se.out = nullptr;
  se.lse = nullptr;
  return launch_result(launch_select(se, st), "select kernel");
}

prhs_status do_score_select(const prhs_kv& kv, DeviceInfo* di, const Layout& L, void* ws,
                            const void* q, float scale, int N, const int32_t* n_budget,
                            int n_sink, int window, const uint8_t* head_skip, int32_t* idx, int32_t* n_sel, int cap,
                            float* delta, int32_t* anchor_idx, int32_t* anchor_n, int anchor_cap,
                            void* q_anchor, cudaStream_t st, float* out = nullptr,
                            float* lse = nullptr, const void* q_src = nullptr) {
  const KVView v = view_of(kv, di->err);
  if (score_select_fits(v)) {  // short caches: logits computed into shared memory, one launch
    SelectLaunch se;
    se.kv = v;
    se.scores = nullptr;
    se.N = N;
    se.n_budget = n_budget;
    se.head_skip = head_skip;
    se.idx = idx;
    se.n_sel = n_sel;
    se.cap = cap;
    se.delta = delta;
    se.anchor_idx = anchor_idx;
    se.anchor_n = anchor_n;
    se.anchor_cap = anchor_cap;
    se.q = q;
    se.q_anchor = q_anchor;
    se.q_src = q_src != nullptr ? q_src : q;
    se.n_sink = n_sink;
    se.window = window;
    se.scale = scale;
    // with forced keys the set-mass pass that follows reads the logits
    se.logits_out = n_sink > 0 || window > 0 ? reinterpret_cast<float*>(static_cast<char*>(ws) + L.scores)
                                             : nullptr;
    se.out = out;  // with out: the attention over the set too (no forced keys)
    se.lse = lse;
    return launch_result(launch_score_select(se, st), "score-select kernel");
  }
  prhs_status s = do_score(kv, di, L, ws, q, scale, head_skip, st);
  if (s != PRHS_OK) return s;
  return do_select(kv, di, L, ws, q, N, n_budget, n_sink, window, head_skip, idx, n_sel, cap, delta,
                   anchor_idx, anchor_n, anchor_cap, q_anchor, st, q_src);
}

// Host checks shared by the selection entry points.
prhs_status check_select_args(const prhs_kv& kv, const void* q, int N, const int32_t* n_budget,
                              int32_t* idx, int32_t* n_sel, int cap, float* delta,
                              int32_t* anchor_idx, int32_t* anchor_n, int anchor_cap,
                              void* q_anchor) {
  if (q == nullptr || idx == nullptr || n_sel == nullptr || delta == nullptr)
    return fail(PRHS_EINVAL, "q, idx, n_sel and delta must be non-null");
  if (!aligned16(q) || !aligned16(q_anchor)) return fail(PRHS_EINVAL, "q and q_anchor must be 16-byte aligned");
  if (n_budget == nullptr && N <= 0) return fail(PRHS_EINVAL, "N must be positive (got %d)", N);
  if (cap <= 0) return fail(PRHS_EINVAL, "cap must be positive");
  const int tmax = t_max_of(kv);
  if (n_budget == nullptr && cap < (N < tmax ? N : tmax))
    return fail(PRHS_EINVAL, "cap %d < budget %d", cap, N < tmax ? N : tmax);
  const bool any_anchor = anchor_idx || anchor_n || q_anchor;
  if (any_anchor && !(anchor_idx && anchor_n && q_anchor))
    return fail(PRHS_EINVAL, "anchor_idx, anchor_n and q_anchor must be all set or all null");
  if (any_anchor && n_budget == nullptr && anchor_cap < (N < tmax ? N : tmax))
    return fail(PRHS_EINVAL, "anchor_cap %d < budget", anchor_cap);
  return PRHS_OK;
}

prhs_status do_attn(const prhs_kv& kv, DeviceInfo* di, const Layout& L, void* ws, const void* q,
                    float scale, const int32_t* idx, const int32_t* n_sel, int cap, float* out,
                    float* lse, bool sparse, cudaStream_t st, const uint8_t* unit_mask = nullptr,
                    int mask_want = 0, bool second_region = false, int max_ctas = 0,
                    int min_rows = ATTN_MIN_ROWS, int rows_hint = 0,
                    const float* logits = nullptr) {
  // the kernels index the concatenated rows of all units with 32-bit integers
  if ((long long)kv.B * kv.Hq * (sparse ? cap : t_max_of(kv)) >= (1ll << 30))
    return fail(PRHS_EUNSUPPORTED, "B * Hq * %s = %lld rows above 2^30", sparse ? "cap" : "t_max",
                (long long)kv.B * kv.Hq * (sparse ? cap : t_max_of(kv)));
  AttnLaunch a;
  a.kv = view_of(kv, di->err);
  a.q = q;
  a.scale = scale;
  a.idx = idx;
  a.n_sel = n_sel;
  a.unit_mask = unit_mask;
  a.mask_want = mask_want;
  a.cap = cap;
  a.out = out;
  a.lse = lse;
  a.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + (second_region ? L.partials2 : L.partials));
  a.counters = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + L.counters);
  a.ctas = attn_ctas(kv, sparse, cap, di->sms);
  a.min_rows = min_rows;
  a.cluster = sparse ? attn_cluster_size(kv, rows_hint > 0 ? rows_hint : cap, di->sms) : 0;
  if (second_region && a.cluster > ATTN_SIDE_CLUSTER_MAX) a.cluster = ATTN_SIDE_CLUSTER_MAX;  // a decode step's side branch
  a.logits = sparse ? logits : nullptr;
  if (a.logits != nullptr) a.ctas = attn_ctas(kv, sparse, cap, di->sms, ATTN_LG_CTAS_PER_SM);
  if (max_ctas > 0 && a.ctas > max_ctas) a.ctas = max_ctas;
  return launch_result(launch_attn(a, sparse, st), sparse ? "sparse attention" : "dense attention");
}

prhs_status do_cis(const prhs_kv& kv, DeviceInfo* di, const int32_t* anchor_idx,
                   const int32_t* anchor_n, int anchor_cap, const void* q, const void* q_anchor,
                   int w, int n_den, int n_sink, int window, double tau, int max_run,
                   int32_t* anchor_age, int32_t* idx, int32_t* n_sel, int cap, uint8_t* reuse,
                   cudaStream_t st) {
  CisLaunch c;
  c.kv = view_of(kv, di->err);
  c.anchor_idx = anchor_idx;
  c.anchor_n = anchor_n;
  c.anchor_cap = anchor_cap;
  c.q = q;
  c.q_anchor = q_anchor;
  c.w = w;
  c.n_den = n_den;
  c.tau = tau;
  c.max_run = max_run;
  c.anchor_age = anchor_age;
  c.idx = idx;
  c.n_sel = n_sel;
  c.cap = cap;
  c.reuse = reuse;
  c.n_sink = n_sink;
  c.window = window;
  return launch_result(launch_cis(c, st), "cis kernel");
}

bool dilated_fits(long long anchor_cap, int w, int tmax, int cap, int forced = 0) {
  long long need = anchor_cap * (2ll * w + 1) + forced;
  if (need > tmax) need = tmax;
  return need <= cap;
}

// Forced keys (sinks and window): non-negative, and selection with forced
// keys runs only where a head's logits fit one CTA or a cluster.
prhs_status check_forced(const prhs_kv& kv, int n_sink, int window) {
  if (n_sink < 0 || window < 0)
    return fail(PRHS_EINVAL, "n_sink and window must be >= 0 (got %d, %d)", n_sink, window);
  if ((n_sink > 0 || window > 0) && (long long)t_max_of(kv) > 8ll * SELECT_SLICE_MAX)
    return fail(PRHS_EUNSUPPORTED, "forced keys with t_max above %d", 8 * SELECT_SLICE_MAX);
  return PRHS_OK;
}

// After a selection with forced keys: the attended set (sinks, the middle
// top-N kept in the anchor rows, window) into idx / n_sel, and its dropped
// mass over the logits still in the workspace into delta.
prhs_status forced_finish(const prhs_kv& kv, DeviceInfo* di, const Layout& L, void* ws,
                          const uint8_t* head_skip, const int32_t* anchor_idx,
                          const int32_t* anchor_n, int anchor_cap, int32_t* idx, int32_t* n_sel,
                          int cap, float* delta, int n_sink, int window, cudaStream_t st) {
  ComposeLaunch c;
  c.kv = view_of(kv, di->err);
  c.head_skip = head_skip;
  c.anchor_idx = anchor_idx;
  c.anchor_n = anchor_n;
  c.anchor_cap = anchor_cap;
  c.idx = idx;
  c.n_sel = n_sel;
  c.cap = cap;
  c.n_sink = n_sink;
  c.window = window;
  prhs_status s = launch_result(launch_compose(c, st), "compose kernel");
  if (s != PRHS_OK) return s;
  MassLaunch m;
  m.kv = view_of(kv, di->err);
  m.scores = reinterpret_cast<const float*>(static_cast<const char*>(ws) + L.scores);
  m.idx = idx;
  m.n_sel = n_sel;
  m.cap = cap;
  m.delta = delta;
  m.head_skip = head_skip;
  // the retrieving heads' tickets and the first partial region: the reusing
  // heads' attention, which may run beside this, uses the second region
  m.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + L.partials);
  m.counters = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + L.counters);
  return launch_result(launch_mass(m, st), "set mass kernel");
}

// The retrieving heads (not flagged in head_skip): top-N set, delta and the
// attention over the set into out/lse. Short caches without forced keys take
// one launch (score, select and attend); otherwise scoring, selection, the
// forced keys' composition and set mass, and sparse attention over the heads
// with head_skip == 0, which weights each selected V row by the logit the
// scoring left in the workspace (K is not read again). rows_hint bounds the
// rows of one head's set.
prhs_status do_retrieve(const prhs_kv& kv, DeviceInfo* di, const Layout& L, void* ws, const void* q,
                        float scale, int N, const int32_t* n_budget, int n_sink, int window,
                        const uint8_t* head_skip, int32_t* idx, int32_t* n_sel, int cap, float* delta,
                        int32_t* anchor_idx, int32_t* anchor_n, int anchor_cap, void* q_anchor,
                        float* out, float* lse, int rows_hint, cudaStream_t st,
                        const void* q_src = nullptr) {
  const bool forced = n_sink > 0 || window > 0;
  const bool one = !forced && score_select_fits(view_of(kv, di->err));
  prhs_status s = do_score_select(kv, di, L, ws, q, scale, N, n_budget, n_sink, window, head_skip, idx,
                                  n_sel, cap, delta, anchor_idx, anchor_n, anchor_cap, q_anchor, st,
                                  one ? out : nullptr, one ? lse : nullptr, q_src);
  if (s != PRHS_OK || one) return s;
  if (forced && (s = forced_finish(kv, di, L, ws, head_skip, anchor_idx, anchor_n, anchor_cap, idx,
                                   n_sel, cap, delta, n_sink, window, st)) != PRHS_OK)
    return s;
  return do_attn(kv, di, L, ws, q, scale, idx, n_sel, cap, out, lse, true, st, head_skip, 0, false, 0,
                 ATTN_MIN_ROWS, rows_hint,
                 reinterpret_cast<const float*>(static_cast<const char*>(ws) + L.scores));
}

// One warp waits on an mbarrier that nothing ever arrives on: the bounded
// wait of the other kernels gives up after limit_ns, raises PRHS_DEV_TIMEOUT
// and the kernel returns (nothing else is in flight on the barrier).
__global__ void __launch_bounds__(32) wait_selftest_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  mbar_wait(&bar, 0, err, limit_ns);
}

}  // namespace

// Internal hooks for other translation units of the library (no C linkage).
prhs_status abi_check_kv(const prhs_kv* kv) { return check_kv(kv); }
prhs_status abi_device(unsigned** err, int* sms) {
  DeviceInfo* di = nullptr;
  prhs_status s = device_info(&di);
  if (s != PRHS_OK) return s;
  *err = di->err;
  *sms = di->sms;
  return PRHS_OK;
}
prhs_status abi_fail(prhs_status s, const char* msg) { return fail(s, "%s", msg); }
void abi_count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
KVView abi_view(const prhs_kv& kv, unsigned* err) { return view_of(kv, err); }
int abi_attn_ctas(const prhs_kv& kv, bool sparse, int cap, int sms) {
  return attn_ctas(kv, sparse, cap, sms);
}

}  // namespace prhs

using namespace prhs;

extern "C" {

size_t prhs_workspace_size(const prhs_kv* kv, int cap) {
  (void)cap;
  if (check_kv(kv) != PRHS_OK) return 0;
  DeviceInfo* di = nullptr;
  if (device_info(&di) != PRHS_OK) return 0;
  return layout_of(*kv, di->sms).total;
}

prhs_status prhs_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (ws == nullptr || ws_bytes == 0) return fail(PRHS_EWORKSPACE, "workspace is null or empty");
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, stream);
  return e == cudaSuccess ? PRHS_OK : cuda_fail(e, "cudaMemsetAsync");
}

prhs_status prhs_score_select(const prhs_kv* kv, const void* q, float scale, int N,
                              const int32_t* n_budget, int n_sink, int window,
                              const uint8_t* head_skip, int32_t* idx, int32_t* n_sel, int cap,
                              float* delta, int32_t* anchor_idx, int32_t* anchor_n, int anchor_cap,
                              void* q_anchor, void* ws, size_t ws_bytes, cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if ((s = check_select_args(*kv, q, N, n_budget, idx, n_sel, cap, delta, anchor_idx, anchor_n,
                             anchor_cap, q_anchor)) != PRHS_OK)
    return s;
  if ((s = check_forced(*kv, n_sink, window)) != PRHS_OK) return s;
  const bool forced = n_sink > 0 || window > 0;
  if (forced && anchor_idx == nullptr) return fail(PRHS_EINVAL, "forced keys need the anchor buffers");
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  Layout L;
  if ((s = check_ws(*kv, di->sms, ws, ws_bytes, &L)) != PRHS_OK) return s;
  if ((s = do_score_select(*kv, di, L, ws, q, scale, N, n_budget, n_sink, window, head_skip, idx,
                           n_sel, cap, delta, anchor_idx, anchor_n, anchor_cap, q_anchor,
                           stream)) != PRHS_OK)
    return s;
  if (!forced) return PRHS_OK;
  return forced_finish(*kv, di, L, ws, head_skip, anchor_idx, anchor_n, anchor_cap, idx, n_sel, cap,
                       delta, n_sink, window, stream);
}

prhs_status prhs_retrieve(const prhs_kv* kv, const void* q, float scale, int N, const int32_t* n_budget,
                          int n_sink, int window, const uint8_t* head_skip, int32_t* idx,
                          int32_t* n_sel, int cap, float* delta, int32_t* anchor_idx,
                          int32_t* anchor_n, int anchor_cap, void* q_anchor, float* out, float* lse,
                          void* ws, size_t ws_bytes, cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if ((s = check_select_args(*kv, q, N, n_budget, idx, n_sel, cap, delta, anchor_idx, anchor_n,
                             anchor_cap, q_anchor)) != PRHS_OK)
    return s;
  if (out == nullptr || lse == nullptr) return fail(PRHS_EINVAL, "out and lse must be non-null");
  if ((s = check_forced(*kv, n_sink, window)) != PRHS_OK) return s;
  const bool forced = n_sink > 0 || window > 0;
  if (forced && anchor_idx == nullptr) return fail(PRHS_EINVAL, "forced keys need the anchor buffers");
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  Layout L;
  if ((s = check_ws(*kv, di->sms, ws, ws_bytes, &L)) != PRHS_OK) return s;
  return do_retrieve(*kv, di, L, ws, q, scale, N, n_budget, n_sink, window, head_skip, idx, n_sel, cap,
                     delta, anchor_idx, anchor_n, anchor_cap, q_anchor, out, lse, cap, stream);
}

prhs_status prhs_score(const prhs_kv* kv, const void* q, float scale, const uint8_t* head_skip,
                       void* ws, size_t ws_bytes, cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if (q == nullptr) return fail(PRHS_EINVAL, "q must be non-null");
  if (!aligned16(q)) return fail(PRHS_EINVAL, "q must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  Layout L;
  if ((s = check_ws(*kv, di->sms, ws, ws_bytes, &L)) != PRHS_OK) return s;
  return do_score(*kv, di, L, ws, q, scale, head_skip, stream);
}

prhs_status prhs_set_mass(const prhs_kv* kv, const void* q, float scale, const int32_t* idx,
                          const int32_t* n_sel, int cap, float* delta, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if (!q || !idx || !n_sel || !delta) return fail(PRHS_EINVAL, "set_mass: null pointer argument");
  if (!aligned16(q)) return fail(PRHS_EINVAL, "q must be 16-byte aligned");
  if (cap <= 0) return fail(PRHS_EINVAL, "cap must be positive");
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  Layout L;
  if ((s = check_ws(*kv, di->sms, ws, ws_bytes, &L)) != PRHS_OK) return s;
  if ((s = do_score(*kv, di, L, ws, q, scale, nullptr, stream)) != PRHS_OK) return s;
  MassLaunch m;
  m.kv = view_of(*kv, di->err);
  m.scores = reinterpret_cast<const float*>(static_cast<const char*>(ws) + L.scores);
  m.idx = idx;
  m.n_sel = n_sel;
  m.cap = cap;
  m.delta = delta;
  m.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + L.partials);
  m.counters = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + L.counters);
  return launch_result(launch_mass(m, stream), "set mass kernel");
}

prhs_status prhs_select(const prhs_kv* kv, const void* q, int N, const int32_t* n_budget,
                        int n_sink, int window, const uint8_t* head_skip, int32_t* idx,
                        int32_t* n_sel, int cap, float* delta, int32_t* anchor_idx,
                        int32_t* anchor_n, int anchor_cap, void* q_anchor, void* ws,
                        size_t ws_bytes, cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if ((s = check_select_args(*kv, q, N, n_budget, idx, n_sel, cap, delta, anchor_idx, anchor_n,
                             anchor_cap, q_anchor)) != PRHS_OK)
    return s;
  if ((s = check_forced(*kv, n_sink, window)) != PRHS_OK) return s;
  const bool forced = n_sink > 0 || window > 0;
  if (forced && anchor_idx == nullptr) return fail(PRHS_EINVAL, "forced keys need the anchor buffers");
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  Layout L;
  if ((s = check_ws(*kv, di->sms, ws, ws_bytes, &L)) != PRHS_OK) return s;
  if ((s = do_select(*kv, di, L, ws, q, N, n_budget, n_sink, window, head_skip, idx, n_sel, cap,
                     delta, anchor_idx, anchor_n, anchor_cap, q_anchor, stream)) != PRHS_OK)
    return s;
  if (!forced) return PRHS_OK;
  return forced_finish(*kv, di, L, ws, head_skip, anchor_idx, anchor_n, anchor_cap, idx, n_sel, cap,
                       delta, n_sink, window, stream);
}

prhs_status prhs_cis_dilate(const prhs_kv* kv, const int32_t* anchor_idx, const int32_t* anchor_n,
                            int anchor_cap, const void* q, const void* q_anchor, int w, int n_den,
                            int n_sink, int window, double tau, int max_run, int32_t* anchor_age,
                            int32_t* idx, int32_t* n_sel, int cap, uint8_t* reuse,
                            cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if ((q && !aligned16(q)) || (q_anchor && !aligned16(q_anchor)))
    return fail(PRHS_EINVAL, "q and q_anchor must be 16-byte aligned");
  if (!anchor_idx || !anchor_n || !q || !q_anchor || !idx || !n_sel || !reuse)
    return fail(PRHS_EINVAL, "cis: null pointer argument");
  if (w < 0) return fail(PRHS_EINVAL, "w must be >= 0 (got %d)", w);
  if (n_den < 0) return fail(PRHS_EINVAL, "n_den must be >= 0 (got %d)", n_den);
  if (max_run < 0) return fail(PRHS_EINVAL, "max_run must be >= 0 (got %d)", max_run);
  if (max_run > 0 && anchor_age == nullptr) return fail(PRHS_EINVAL, "max_run > 0 needs anchor_age");
  if (anchor_cap <= 0 || cap <= 0) return fail(PRHS_EINVAL, "capacities must be positive");
  if (n_sink < 0 || window < 0)
    return fail(PRHS_EINVAL, "n_sink and window must be >= 0 (got %d, %d)", n_sink, window);
  if (!dilated_fits(anchor_cap, w, t_max_of(*kv), cap, n_sink + window))
    return fail(PRHS_EINVAL, "cap %d < min(t_max, anchor_cap * (2w + 1) + n_sink + window)", cap);
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  return do_cis(*kv, di, anchor_idx, anchor_n, anchor_cap, q, q_anchor, w, n_den, n_sink, window, tau,
                max_run, anchor_age, idx, n_sel, cap, reuse, stream);
}

prhs_status prhs_sparse_attn(const prhs_kv* kv, const void* q, float scale, const int32_t* idx,
                             const int32_t* n_sel, int cap, float* out, float* lse, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if (!q || !idx || !n_sel || !out || !lse) return fail(PRHS_EINVAL, "sparse: null pointer argument");
  if (!aligned16(q)) return fail(PRHS_EINVAL, "q must be 16-byte aligned");
  if (cap <= 0) return fail(PRHS_EINVAL, "cap must be positive");
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  Layout L;
  if ((s = check_ws(*kv, di->sms, ws, ws_bytes, &L)) != PRHS_OK) return s;
  return do_attn(*kv, di, L, ws, q, scale, idx, n_sel, cap, out, lse, true, stream);
}

prhs_status prhs_dense_attn(const prhs_kv* kv, const void* q, float scale, float* out, float* lse,
                            void* ws, size_t ws_bytes, cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if (!q || !out || !lse) return fail(PRHS_EINVAL, "dense: null pointer argument");
  if (!aligned16(q)) return fail(PRHS_EINVAL, "q must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  Layout L;
  if ((s = check_ws(*kv, di->sms, ws, ws_bytes, &L)) != PRHS_OK) return s;
  if (kv->Hq == kv->Hkv)  // no query group to share K/V tiles: the gather kernel streams faster
    return do_attn(*kv, di, L, ws, q, scale, nullptr, nullptr, 0, out, lse, false, stream);
  const bool paged = kv->block_table != nullptr;
  const KVView v = view_of(*kv, di->err);
  const int box = paged ? PAGED_BOX_ROWS : dense_rows_per_stage(v);
  CUtensorMap kmap, vmap;
  if ((s = make_tmap(*kv, box, &kmap, kv->k)) != PRHS_OK) return s;
  if ((s = make_tmap(*kv, box, &vmap, kv->v)) != PRHS_OK) return s;
  float* partials = reinterpret_cast<float*>(static_cast<char*>(ws) + L.partials);
  unsigned* counters = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + L.counters);
  return launch_result(launch_dense(v, q, scale, out, lse, partials, counters, di->sms, paged,
                                    &kmap, &vmap, stream),
                       "dense attention");
}

prhs_status prhs_decode_step(const prhs_kv* kv, const void* q, const void* gate, float scale, int N,
                             const int32_t* n_budget, int n_sink, int window, int w, int n_den,
                             double tau, int max_run,
                             int32_t* anchor_age, int32_t* anchor_idx,
                             int32_t* anchor_n, int anchor_cap, void* q_anchor, int32_t* idx,
                             int32_t* n_sel, int cap, uint8_t* reuse, float* delta, float* out,
                             float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if (!q || !anchor_idx || !anchor_n || !q_anchor || !idx || !n_sel || !reuse || !delta || !out || !lse)
    return fail(PRHS_EINVAL, "decode: null pointer argument");
  if (!aligned16(q) || !aligned16(q_anchor) || !aligned16(gate))
    return fail(PRHS_EINVAL, "q, gate and q_anchor must be 16-byte aligned");
  if (n_budget == nullptr && N <= 0) return fail(PRHS_EINVAL, "N must be positive (got %d)", N);
  if (w < 0) return fail(PRHS_EINVAL, "w must be >= 0 (got %d)", w);
  if (n_den < 0) return fail(PRHS_EINVAL, "n_den must be >= 0 (got %d)", n_den);
  if (max_run < 0) return fail(PRHS_EINVAL, "max_run must be >= 0 (got %d)", max_run);
  if (max_run > 0 && anchor_age == nullptr) return fail(PRHS_EINVAL, "max_run > 0 needs anchor_age");
  const int tmax = t_max_of(*kv);
  if (anchor_cap <= 0 || cap <= 0) return fail(PRHS_EINVAL, "capacities must be positive");
  if (n_budget == nullptr && anchor_cap < (N < tmax ? N : tmax))
    return fail(PRHS_EINVAL, "anchor_cap %d < budget", anchor_cap);
  if ((s = check_forced(*kv, n_sink, window)) != PRHS_OK) return s;
  const bool forced = n_sink > 0 || window > 0;
  if (!dilated_fits(anchor_cap, w, tmax, cap, n_sink + window))
    return fail(PRHS_EINVAL, "cap %d < min(t_max, anchor_cap * (2w + 1) + n_sink + window)", cap);
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  Layout L;
  if ((s = check_ws(*kv, di->sms, ws, ws_bytes, &L)) != PRHS_OK) return s;
  // the gate compares `gate` (or q) with the anchor's copy of it
  const void* gv = gate != nullptr ? gate : q;
  if ((s = do_cis(*kv, di, anchor_idx, anchor_n, anchor_cap, gv, q_anchor, w, n_den, n_sink, window,
                  tau, max_run, anchor_age, idx, n_sel, cap, reuse, stream)) != PRHS_OK)
    return s;
  // Two branches after the gate: heads that reuse their anchor only need the
  // dilated sets and attend on the side stream, while the retrieving heads
  // score, select and attend on the caller's stream; the caller's stream then
  // waits for the side branch.
  SideBranch* br = nullptr;
  if ((s = side_branch(di, stream, &br)) != PRHS_OK) return s;
  std::lock_guard<std::mutex> branch_lock(br->mu);
  // Scoring first, on its own, when what follows it on the retrieving branch
  // is small beside the reusing heads' attention: a one-CTA selection per head
  // with at most one head per SM, and a V-only attention without clusters.
  // Their CTAs then run beside that attention instead of after it. Larger
  // retrieving branches keep the order below: the attention splits its rows
  // evenly over one wave of CTAs, so kernels that take SM room at its start
  // hold back the CTAs they displace and the whole launch ends later.
  const KVView vv = view_of(*kv, di->err);
  const bool fused = !forced && score_select_fits(vv);
  const bool score_first = !forced && !fused && vv.t_max <= SELECT_SLICE_ONE &&
                           (long long)kv->B * kv->Hq <= di->sms &&
                           attn_cluster_size(*kv, anchor_cap, di->sms) == 0;
  if (score_first && (s = do_score(*kv, di, L, ws, q, scale, reuse, stream)) != PRHS_OK) return s;
  cudaError_t e = cudaEventRecord(br->fork, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(br->side, br->fork, 0);
  if (e != cudaSuccess) return cuda_fail(e, "decode: fork");
  // The branch more likely to be the longer one is issued first, so its CTAs
  // are placed first: the one-launch retrieval on short caches, the reusing
  // heads' attention otherwise (measured both ways on 4K-, 32K- and 128K-key
  // caches); after scoring first, the selection and V-only attention, which
  // take few SMs. The retrieving heads' sets hold at most anchor_cap (+ forced) rows.
  const bool retrieve_first = fused || score_first;
  for (int branch = 0; branch < 2 && s == PRHS_OK; branch++) {
    if ((branch == 0) == retrieve_first && score_first) {
      s = do_select(*kv, di, L, ws, q, N, n_budget, n_sink, window, reuse, idx, n_sel, cap, delta,
                    anchor_idx, anchor_n, anchor_cap, q_anchor, stream, gv);
      if (s == PRHS_OK)
        s = do_attn(*kv, di, L, ws, q, scale, idx, n_sel, cap, out, lse, true, stream, reuse, 0, false,
                    0, ATTN_MIN_ROWS, anchor_cap,
                    reinterpret_cast<const float*>(static_cast<const char*>(ws) + L.scores));
    } else if ((branch == 0) == retrieve_first) {
      s = do_retrieve(*kv, di, L, ws, q, scale, N, n_budget, n_sink, window, reuse, idx, n_sel, cap,
                      delta, anchor_idx, anchor_n, anchor_cap, q_anchor, out, lse,
                      anchor_cap + n_sink + window, stream, gv);
    } else {
      s = do_attn(*kv, di, L, ws, q, scale, idx, n_sel, cap, out, lse, true, br->side, reuse, 1, true, 0,
                  ATTN_SIDE_MIN_ROWS);
    }
  }
  // The join is recorded even after a failed launch, so the side stream never
  // stays forked (a capture would otherwise end unjoined); the first failure
  // is what the caller sees.
  const std::string first_message = t_message;
  e = cudaEventRecord(br->join, br->side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, br->join, 0);
  if (s != PRHS_OK) {
    t_message = first_message;
    return s;
  }
  return e == cudaSuccess ? PRHS_OK : cuda_fail(e, "decode: join");
}

prhs_status prhs_append_kv(const prhs_kv* kv, const void* k_new, const void* v_new,
                           cudaStream_t stream) {
  prhs_status s = check_kv(kv);
  if (s != PRHS_OK) return s;
  if (!k_new || !v_new) return fail(PRHS_EINVAL, "append: null pointer argument");
  if (!aligned16(k_new) || !aligned16(v_new)) return fail(PRHS_EINVAL, "k_new and v_new must be 16-byte aligned");
  DeviceInfo* di = nullptr;
  if ((s = device_info(&di)) != PRHS_OK) return s;
  AppendLaunch a;
  a.kv = view_of(*kv, di->err);
  a.k_new = k_new;
  a.v_new = v_new;
  a.seq_lens = const_cast<int32_t*>(kv->seq_lens);
  return launch_result(launch_append(a, stream), "append kernel");
}

prhs_status prhs_selftest_wait_timeout(unsigned limit_us, cudaStream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u)
    return fail(PRHS_EINVAL, "limit_us must be in [1, 1000000] (got %u)", limit_us);
  DeviceInfo* di = nullptr;
  prhs_status s = device_info(&di);
  if (s != PRHS_OK) return s;
  wait_selftest_kernel<<<1, 32, 0, stream>>>(di->err, 1000ull * limit_us);
  return launch_result(cudaGetLastError(), "wait self-test kernel");
}

prhs_status prhs_last_error(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned bits = 0;
  e = cudaMemcpyFromSymbol(&bits, g_error_word, sizeof(bits));
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  const unsigned zero = 0;
  e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  g_last_bits = bits;
  if (bits != 0) return fail(PRHS_EDEVICE, "device error bits 0x%x", bits);
  return PRHS_OK;
}

unsigned prhs_device_error_bits(void) { return g_last_bits; }

unsigned long long prhs_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* prhs_status_str(prhs_status s) {
  switch (s) {
    case PRHS_OK: return "ok";
    case PRHS_EINVAL: return "invalid argument";
    case PRHS_EUNSUPPORTED: return "unsupported shape";
    case PRHS_EWORKSPACE: return "workspace missing or too small";
    case PRHS_ECUDA: return "CUDA runtime error";
    case PRHS_EDEVICE: return "device-side data error";
  }
  return "unknown status";
}

const char* prhs_last_message(void) { return t_message.c_str(); }

int prhs_num_sms(void) {
  DeviceInfo* di = nullptr;
  if (device_info(&di) != PRHS_OK) return 0;
  return di->sms;
}

}  // extern "C"
