// Retrieval of one query head in one launch, for caches of up to 8192 keys:
// the logits straight from K, the exact top-N set with its dropped mass, and
// the attention over that set, with the selection spread over a thread-block
// cluster. "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context
// Inference": abstract (the top-k oracle picks the KV entries before the
// attention; the dropped mass delta), Table I (S_t, N, tau(.), delta(.)) and
// the Table V caption (attention over the selected KV entries only).
//
// Each of the cluster's CL CTAs keeps the logits of its own slice of keys in
// its shared memory, one key per thread. Every exchange between the CTAs is a
// push: a CTA writes what the others need into each of their shared memories
// (distributed shared memory stores, no remote atomics or loads) and one
// cluster barrier later every CTA reads it locally. The rounds:
//   1. logits of the slice; its logit range to every rank.
//   2. a 64-bin value histogram of the slice over the head's range to every
//      rank; each CTA finds the bin of the N-th largest logit, the keys above
//      that bin (kept for sure) and below it (dropped), and the counts of the
//      lower ranks. A bin holding more than RT_CANDS keys is narrowed further:
//      the exact range of its keys (one value: heavy ties, decided at once),
//      then another 64-bin round inside it.
//   3. the final bin's keys (the candidates) to every rank, each rank's at an
//      offset fixed by the lower ranks' counts; every CTA then ranks them
//      exactly. The V rows of the keys kept for sure, and of the CTA's own
//      candidates, are loaded while this barrier completes.
//   4. each CTA compacts its slice in index order (ties to the lowest index),
//      adds up the weighted V rows of its kept keys with weights exp(s - max)
//      (the largest logit is always kept, so the CTAs' sums add without
//      rescaling) and pushes its sums and its dropped weight to CTA 0, which
//      writes out, lse and delta.
// Bins that stay full after RT_ROUNDS rounds fall back to radix passes over
// the order-preserving key that CTA 0 runs over every CTA's logits in place.
#include <cooperative_groups.h>

#include "kernels.h"

namespace cg = cooperative_groups;

namespace prhs {
namespace {

constexpr int RT_THREADS = 512;
constexpr int RT_WARPS = RT_THREADS / 32;
constexpr int RT_SLICE = SELECT_FUSED_MAX_ROWS;  // keys per CTA at most
constexpr int RT_HB = 64;        // bins of a histogram round
constexpr int RT_CANDS = 256;    // candidates the cluster ranks exactly
constexpr int UD_ROWS = 2;       // waves of kept rows loaded during the candidate barrier
constexpr int RT_ROUNDS = 4;     // histogram rounds before the radix fallback
// A contiguous cache's slice of K rows comes in by one bulk copy into shared
// memory when it takes at most this many bytes (else by 16-byte loads).
constexpr int RT_STAGE_BYTES = 64 * 1024;
static_assert(RT_SLICE <= RT_THREADS, "one key of a slice per thread");
static_assert(RT_HB == 64, "two bins per lane");

template <int DK>
struct RetrieveShared {
  float lg[RT_SLICE];                   // this CTA's logits
  int32_t kept[RT_SLICE];               // this CTA's kept keys, ascending
  int32_t dl[RT_SLICE];                 // keys above the final bin (slice positions)
  int32_t cl[RT_SLICE];                 // this CTA's candidates (slice positions)
  unsigned char take[RT_SLICE];         // whether each key of the slice is kept
  __align__(16) unsigned tab[SELECT_FUSED_CL][RT_HB];  // each rank's counts of the round
  __align__(16) unsigned lh[RT_HB];     // this CTA's counts of the round
  __align__(16) unsigned cand[RT_CANDS];  // every rank's candidates, rank by rank
  float rmin[SELECT_FUSED_CL], rmax[SELECT_FUSED_CL];  // each rank's logit range
  float part[SELECT_FUSED_CL][DK + 2];  // rank 0: each rank's sum w v, sum w, dropped weight
  float wsum[RT_WARPS * DK > 2048 ? RT_WARPS * DK : 2048];  // warps' V sums; fallback counts
  unsigned fgt[SELECT_FUSED_CL], feq[SELECT_FUSED_CL];      // fallback: counts per rank
  float red[RT_WARPS], red2[RT_WARPS];
  unsigned scan[RT_WARPS];
  unsigned bin, krem, cnt_bin, above_lo, inb_lo;  // the round's bin and counts
  unsigned thr, keq, carry_gt, carry_eq;          // the decision, the lower ranks' counts
};

template <bool ONE>
__device__ __forceinline__ void cluster_barrier(cg::cluster_group& cluster) {
  if (ONE) __syncthreads(); else cluster.sync();
}

// The cluster barrier in two halves, with work between them that the other
// CTAs need not wait for.
template <bool ONE>
__device__ __forceinline__ void cluster_arrive() {
  if (!ONE) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
template <bool ONE>
__device__ __forceinline__ void cluster_wait() {
  if (ONE) __syncthreads();
  else asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <bool ONE, typename S>
__device__ __forceinline__ S* at_rank(cg::cluster_group& cluster, S& sh, int r) {
  if (ONE) return &sh;
  return cluster.map_shared_rank(&sh, r);
}

// Bin of s among NB equal bins from lo (inv = bins per unit), clamped;
// monotone non-decreasing in s. Every rank evaluates it with the same
// arguments, so a bin computed for a key and one computed for a trial value
// agree exactly.
template <int NB>
__device__ __forceinline__ int bin_of(float s, float lo, float inv) {
  const float x = (s - lo) * inv;
  return x <= 0.f ? 0 : (x >= (float)(NB - 1) ? NB - 1 : (int)x);
}


// One histogram round: each CTA counts its keys still in play (bin c >= 0),
// pushes the counts to every rank and, after the barrier, finds the bin
// holding the krem-th largest of them, that bin's count, and the lower ranks'
// counts in that bin and above it.
template <int DK, bool ONE>
__device__ __forceinline__ void hist_round(cg::cluster_group& cluster, RetrieveShared<DK>& sh, int CL,
                                           int rank, int c, unsigned krem) {
  const int tid = threadIdx.x;
  if (tid < RT_HB) sh.lh[tid] = 0;
  __syncthreads();
  if (c >= 0) atomicAdd(&sh.lh[c], 1u);
  __syncthreads();
  if (tid < CL * (RT_HB / 4)) {
    const int dst = tid / (RT_HB / 4), q4 = tid % (RT_HB / 4);
    reinterpret_cast<uint4*>(at_rank<ONE>(cluster, sh, dst)->tab[rank])[q4] =
        reinterpret_cast<const uint4*>(sh.lh)[q4];
  }
  cluster_barrier<ONE>(cluster);
  if (tid < 32) {
    const int lane = tid;
    const int bh = RT_HB - 1 - 2 * lane, bl = bh - 1;  // two bins per lane, highest first
    unsigned th = 0, tl = 0, lh = 0, ll = 0;
#pragma unroll
    for (int r = 0; r < SELECT_FUSED_CL; r++) {  // every slot exists; ranks >= CL masked
      const unsigned x = r < CL ? sh.tab[r][bh] : 0u, y = r < CL ? sh.tab[r][bl] : 0u;
      th += x;
      tl += y;
      lh += r < rank ? x : 0u;
      ll += r < rank ? y : 0u;
    }
    const unsigned sum = th + tl;
    unsigned inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned nx = __shfl_up_sync(FULL_MASK, inc, o);
      if (lane >= o) inc += nx;
    }
    const unsigned exc = inc - sum;
    const unsigned ball = __ballot_sync(FULL_MASK, exc < krem && inc >= krem);
    const int src = ball ? __ffs(ball) - 1 : 0;
    unsigned bsel = 0, kr = 0, cb = 0, inb = 0;
    if (lane == src) {
      if (exc + th >= krem) {
        bsel = bh;
        kr = krem - exc;
        cb = th;
        inb = lh;
      } else {
        bsel = bl;
        kr = krem - exc - th;
        cb = tl;
        inb = ll;
      }
    }
    bsel = __shfl_sync(FULL_MASK, bsel, src);
    kr = __shfl_sync(FULL_MASK, kr, src);
    cb = __shfl_sync(FULL_MASK, cb, src);
    inb = __shfl_sync(FULL_MASK, inb, src);
    unsigned ab = ((unsigned)bh > bsel ? lh : 0u) + ((unsigned)bl > bsel ? ll : 0u);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ab += __shfl_xor_sync(FULL_MASK, ab, o);
    if (lane == 0) {
      sh.bin = bsel;
      sh.krem = kr;
      sh.cnt_bin = cb;
      sh.inb_lo = inb;
      sh.above_lo = ab;
    }
  }
  __syncthreads();
}

// Heavy ties: rank 0 finds the threshold key and how many ties at it to keep
// by three radix passes (11, 11 and 10 bits of the order-preserving key) over
// the logits of every rank, read in place, then leaves in each rank's shared
// memory the decision and the counts of the ranks below it.
template <int DK, bool ONE>
__device__ void radix_decide(cg::cluster_group& cluster, RetrieveShared<DK>& sh, int CL, int chunk,
                             int t, unsigned Nb) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned prefix = 0, mask = 0, krem = Nb;
  unsigned* hist = reinterpret_cast<unsigned*>(sh.wsum);
  for (int pass = 0; pass < 3; pass++) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass == 2 ? 1024 : 2048;
    for (int i = tid; i < nb; i += RT_THREADS) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < t; i += RT_THREADS) {
      const int r = i / chunk;
      const unsigned u = order_key(at_rank<ONE>(cluster, sh, r)->lg[i - r * chunk]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    // the bin of the krem-th largest: each thread sums `per` bins, highest first
    const int per = nb / RT_THREADS;
    const int top = nb - 1 - per * tid;
    unsigned c[4] = {0u, 0u, 0u, 0u}, sum = 0;
    for (int k = 0; k < per; k++) {
      c[k] = hist[top - k];
      sum += c[k];
    }
    unsigned v = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned nx = __shfl_up_sync(FULL_MASK, v, o);
      if (lane >= o) v += nx;
    }
    if (lane == 31) sh.scan[warp] = v;
    __syncthreads();
    unsigned run = v - sum;
    for (int w = 0; w < warp; w++) run += sh.scan[w];
    for (int k = 0; k < per; k++) {
      if (run < krem && run + c[k] >= krem) {
        sh.bin = (unsigned)(top - k);
        sh.krem = krem - run;
      }
      run += c[k];
    }
    __syncthreads();
    prefix |= sh.bin << shift;
    mask |= (unsigned)(nb - 1) << shift;
    krem = sh.krem;
    __syncthreads();
  }
  if (tid < CL) {
    sh.fgt[tid] = 0;
    sh.feq[tid] = 0;
  }
  __syncthreads();
  for (int i = tid; i < t; i += RT_THREADS) {
    const int r = i / chunk;
    const unsigned u = order_key(at_rank<ONE>(cluster, sh, r)->lg[i - r * chunk]);
    if (u > prefix) atomicAdd(&sh.fgt[r], 1u);
    else if (u == prefix) atomicAdd(&sh.feq[r], 1u);
  }
  __syncthreads();
  if (tid < CL) {
    unsigned g = 0, e = 0;
    for (int r = 0; r < tid; r++) {
      g += sh.fgt[r];
      e += sh.feq[r];
    }
    RetrieveShared<DK>* rs = at_rank<ONE>(cluster, sh, tid);
    rs->thr = prefix;
    rs->keq = krem;
    rs->carry_gt = g;
    rs->carry_eq = e;
  }
}

// acc += w v over the rows at positions [p0, p1) of list (slice positions of
// keys), weights exp(logit - smax); with check, only the rows marked kept.
// LPR lanes share a row; UV rows per lane group are in flight at a time.
template <typename T, int DK>
__device__ __forceinline__ void gather_rows(const KVView& kv, const RetrieveShared<DK>& sh,
                                            const int32_t* list, int p0, int p1, bool check, int b,
                                            int kvh, int lo, int t, float smax, float* acc,
                                            float& lsum) {
  constexpr int EPC = Elem<T>::per16, LPR = DK / EPC, RPW = RT_THREADS / LPR, UV = 4;
  const int j = threadIdx.x & (LPR - 1), rsub = threadIdx.x / LPR;
  const char* vb = static_cast<const char*>(kv.v);
  for (int pb = p0; pb < p1; pb += RPW * UV) {
    float ww[UV];
    uint4 raw[UV];
#pragma unroll
    for (int k = 0; k < UV; k++) {
      const int p = pb + k * RPW + rsub;
      const int i = p < p1 ? list[p] : -1;
      long long r = -1;
      ww[k] = 0.f;
      if (i >= 0 && i < RT_SLICE && lo + i < t && (!check || sh.take[i])) {
        ww[k] = expf(sh.lg[i] - smax);
        r = kv_row(kv, b, kvh, lo + i);
        if (r < 0 && j == 0) raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
      }
      raw[k] = r >= 0 ? ldg_stream(vb + r * (long long)(DK * sizeof(T)) + 16 * j)
                      : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < UV; k++) {
      float f[EPC];
      Elem<T>::unpack(raw[k], f);
#pragma unroll
      for (int e = 0; e < EPC; e++) acc[e] = fmaf(ww[k], f[e], acc[e]);
      lsum += ww[k];
    }
  }
}

// V rows of the candidate path, loaded while its barrier completes.
template <int UD>
struct CandRound {
  bool on = false;      // the candidate exchange decided: the loads below are valid
  int nd = 0, ncl = 0;  // this CTA's keys kept for sure / candidates
  int di[UD], ci = -1;  // slice positions of the rows loaded (-1: none)
  uint4 dv[UD], cv;
  __device__ CandRound() {
#pragma unroll
    for (int k = 0; k < UD; k++) {
      di[k] = -1;
      dv[k] = make_uint4(0u, 0u, 0u, 0u);
    }
    cv = make_uint4(0u, 0u, 0u, 0u);
  }
};

// The candidate exchange that ends the histogram rounds. Keys with st == 1
// are kept for sure, st == 2 are the candidates (every key equal to the
// threshold is one); each CTA writes its candidates into every rank's row
// from inb_lo on (the lower ranks' candidates, known from the histogram), nc
// of them in all. While the barrier completes, each lane group loads the V
// rows of the first kept keys and of one candidate.
template <typename T, int DK, bool ONE>
__device__ void candidate_round(const KVView& kv, cg::cluster_group& cluster, RetrieveShared<DK>& sh,
                                CandRound<UD_ROWS>& cr, int CL, int rank, int b, int kvh, int lo,
                                int st, float s, unsigned inb_lo, unsigned nc, unsigned krem,
                                unsigned carry_above, unsigned& thr, unsigned& keq, unsigned& carry_gt,
                                unsigned& carry_eq) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int EPC = Elem<T>::per16, LPR = DK / EPC, RPW = RT_THREADS / LPR;
  const int j = tid & (LPR - 1), rsub = tid / LPR;
  const unsigned below = (1u << lane) - 1u;
  const unsigned bd = __ballot_sync(FULL_MASK, st == 1), bc = __ballot_sync(FULL_MASK, st == 2);
  __syncthreads();  // sh.scan may still be read
  if (lane == 0) sh.scan[warp] = ((unsigned)__popc(bd) << 16) | (unsigned)__popc(bc);
  __syncthreads();
  unsigned before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < RT_WARPS; w++) {
    const unsigned x = sh.scan[w];
    before += w < warp ? x : 0u;
    tot += x;
  }
  const int nd = (int)(tot >> 16), ncl = (int)(tot & 0xffffu);
  if (st == 1) sh.dl[(before >> 16) + __popc(bd & below)] = tid;
  if (st == 2) {
    const unsigned pc = (before & 0xffffu) + __popc(bc & below);
    sh.cl[pc] = tid;
    const unsigned slot = inb_lo + pc;  // the lower ranks' candidates come first
    if (slot < (unsigned)RT_CANDS) {
      const unsigned key = order_key(s);
      for (int r = 0; r < CL; r++) at_rank<ONE>(cluster, sh, r)->cand[slot] = key;
    }
  }
  if (tid == 0) {  // no match below (inconsistent counts) keeps nothing at the threshold
    sh.thr = 0xffffffffu;
    sh.keq = 0u;
  }
  __syncthreads();  // the lists are complete
  cluster_arrive<ONE>();
  const char* vb = static_cast<const char*>(kv.v);
#pragma unroll
  for (int k = 0; k < UD_ROWS; k++) {
    const int p = k * RPW + rsub;
    cr.di[k] = p < nd ? sh.dl[p] : -1;
    const long long r = cr.di[k] >= 0 ? kv_row(kv, b, kvh, lo + cr.di[k]) : -1;
    if (cr.di[k] >= 0 && r < 0 && j == 0) raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
    if (r >= 0) cr.dv[k] = ldg_stream(vb + r * (long long)(DK * sizeof(T)) + 16 * j);
  }
  {
    cr.ci = rsub < ncl ? sh.cl[rsub] : -1;
    const long long r = cr.ci >= 0 ? kv_row(kv, b, kvh, lo + cr.ci) : -1;
    if (cr.ci >= 0 && r < 0 && j == 0) raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
    if (r >= 0) cr.cv = ldg_stream(vb + r * (long long)(DK * sizeof(T)) + 16 * j);
  }
  cluster_wait<ONE>();  // every candidate is in every rank
  const unsigned nlow = min(inb_lo, nc);
  cr.on = true;
  cr.nd = nd;
  cr.ncl = ncl;
  // pad the row to whole 16-byte groups with a key below every logit
  if (tid < 4 && nc + tid < (unsigned)RT_CANDS && ((nc + tid) & 3u) != 0u) sh.cand[nc + tid] = 0u;
  __syncthreads();
  if (tid < (int)nc) {  // exact rank of each candidate among all of them
    const unsigned my = sh.cand[tid];
    const uint4* c4 = reinterpret_cast<const uint4*>(sh.cand);
    unsigned g = 0, e = 0;
#pragma unroll 4
    for (unsigned q4 = 0; q4 < (nc + 3u) / 4u; q4++) {
      const uint4 x = c4[q4];
      g += (x.x > my) + (x.y > my) + (x.z > my) + (x.w > my);
      e += (x.x == my) + (x.y == my) + (x.z == my) + (x.w == my);
    }
    if (g < krem && g + e >= krem) {
      sh.thr = my;
      sh.keq = krem - g;
    }
  }
  __syncthreads();
  thr = sh.thr;
  keq = sh.keq;
  unsigned cgt = 0, ceq = 0;  // the lower ranks' candidates above and at the threshold
  for (unsigned q = (unsigned)lane; q < nlow; q += 32) {
    cgt += sh.cand[q] > thr;
    ceq += sh.cand[q] == thr;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cgt += __shfl_xor_sync(FULL_MASK, cgt, o);
    ceq += __shfl_xor_sync(FULL_MASK, ceq, o);
  }
  carry_gt = carry_above + cgt;
  carry_eq = ceq;
}

template <typename T, int DK>
__host__ __device__ constexpr bool stage_by_copy(bool paged, int chunk) {
  return !paged && (long long)chunk * DK * sizeof(T) <= RT_STAGE_BYTES;
}

template <typename T, int DK, bool ONE>
__global__ void __launch_bounds__(RT_THREADS, 2) retrieve_kernel(const SelectLaunch a, int chunk) {
  __shared__ RetrieveShared<DK> sh;
  __shared__ __align__(8) uint64_t kbar;     // the bulk copy of the K slice
  extern __shared__ __align__(128) unsigned char kst[];  // that slice, when staged
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = ONE ? 1 : (int)cluster.num_blocks();
  const int rank = ONE ? 0 : (int)cluster.block_rank();
  const bool staged = stage_by_copy<T, DK>(a.kv.block_table != nullptr, chunk);
  if (staged && threadIdx.x == 0) {
    mbar_init(&kbar, 1);
    fence_barrier_init();
  }
  pdl_wait();
  pdl_trigger();

  const KVView& kv = a.kv;
  const int qh = blockIdx.x / CL;
  const int b = qh / kv.Hq;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int EPC = Elem<T>::per16;       // elements per 16-byte piece
  constexpr int LPR = DK / EPC;             // lanes per row: 8, 16 or 32
  constexpr int RPW = RT_THREADS / LPR;     // rows per CTA-wide wave of loads
  static_assert(LPR >= 8 && LPR <= 32 && (LPR & (LPR - 1)) == 0, "row split");
  const int j = tid & (LPR - 1), rsub = tid / LPR;

  // the head's inputs, all in flight before the first is used
  const unsigned skip = a.head_skip != nullptr ? a.head_skip[qh] : 0u;
  int t = kv.seq_lens[b];
  const int nb_in = a.n_budget != nullptr ? a.n_budget[b] : a.N;
  const uint4 qraw = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.q) +
                                                          (long long)qh * DK * sizeof(T)) + j);
  const bool anchor_row = rank == 0 && a.q_anchor != nullptr && tid < LPR;  // stored at the end
  uint4 qsrc = make_uint4(0u, 0u, 0u, 0u);
  if (anchor_row)
    qsrc = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.q_src) +
                                                (long long)qh * DK * sizeof(T)) + tid);
  if (skip != 0) return;  // uniform over the cluster
  if (t < 0 || t > kv.t_max) {
    if (tid == 0) raise_error(kv.err, PRHS_DEV_BAD_LEN);
    t = t < 0 ? 0 : kv.t_max;
  }
  int Nb = nb_in < 0 ? 0 : nb_in;
  const int lim = a.anchor_idx != nullptr ? min(a.cap, a.anchor_cap) : a.cap;
  if (min(Nb, t) > lim) {
    if (tid == 0 && rank == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    Nb = lim;
  }
  const int n = min(Nb, t);
  int32_t* out = a.idx + (long long)qh * a.cap;
  int32_t* aout = a.anchor_idx != nullptr ? a.anchor_idx + (long long)qh * a.anchor_cap : nullptr;
  const int lo = min(t, rank * chunk), cnt = min(t, lo + chunk) - lo;
  uint4* qa_dst = anchor_row ? reinterpret_cast<uint4*>(static_cast<char*>(a.q_anchor) +
                                                        (long long)qh * DK * sizeof(T)) + tid
                             : nullptr;

  if (n == 0) {  // zero budget or empty cache: the empty set (uniform over the cluster)
    if (rank == 0) {
      if (tid == 0) {
        a.n_sel[qh] = 0;
        a.delta[qh] = t == 0 ? 0.f : 1.f;
        if (a.anchor_n) a.anchor_n[qh] = 0;
        a.lse[qh] = -INFINITY;
      }
      for (int e = tid; e < DK; e += RT_THREADS) a.out[(long long)qh * DK + e] = 0.f;
      if (qa_dst) *qa_dst = qsrc;
    }
    return;
  }

  // ---- round 1: logits of this CTA's slice, and its range to every rank ----
  const int kvh = (qh % kv.Hq) / (kv.Hq / kv.Hkv);
  {
    float qf[EPC];
    Elem<T>::unpack(qraw, qf);
    const char* kb = static_cast<const char*>(kv.k);
    constexpr long long ROW = DK * sizeof(T);
    float vmin = INFINITY, vmax = -INFINITY;
    constexpr int U = 8;  // rows in flight per thread
    if (staged) {
      __syncthreads();  // the barrier's initialisation is visible
      if (tid == 0 && cnt > 0) {
        const uint32_t bytes = (uint32_t)(cnt * ROW);
        mbar_arrive_expect_tx(&kbar, bytes);
        bulk_load(kst, kb + kv_row(kv, b, kvh, lo) * ROW, bytes, &kbar);
      }
      const bool ok = cnt == 0 || mbar_wait(&kbar, 0, kv.err);
      constexpr int US = 4;  // shared memory: few rows in flight suffice
      for (int r0 = 0; r0 < cnt; r0 += RPW * US) {
        uint4 raw[US];
#pragma unroll
        for (int u = 0; u < US; u++) {
          const int r = r0 + u * RPW + rsub;
          raw[u] = ok && r < cnt ? *reinterpret_cast<const uint4*>(kst + r * ROW + 16 * j)
                                 : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < US; u++) {
          float f[EPC];
          Elem<T>::unpack(raw[u], f);
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < EPC; e++) acc = fmaf(qf[e], f[e], acc);
#pragma unroll
          for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, o);
          const int r = r0 + u * RPW + rsub;
          if (j == 0 && r < cnt) {
            const float v = acc * a.scale;
            sh.lg[r] = v;
            vmin = fminf(vmin, v);
            vmax = fmaxf(vmax, v);
          }
        }
      }
    }
    for (int r0 = 0; !staged && r0 < cnt; r0 += RPW * U) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int r = r0 + u * RPW + rsub;
        long long row = -1;
        if (r < cnt) {
          row = kv_row(kv, b, kvh, lo + r);
          if (row < 0 && j == 0) raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
        }
        raw[u] = row >= 0 ? ldg_stream(kb + row * (long long)(DK * sizeof(T)) + 16 * j)
                          : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; u++) {
        float f[EPC];
        Elem<T>::unpack(raw[u], f);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EPC; e++) acc = fmaf(qf[e], f[e], acc);
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, o);
        const int r = r0 + u * RPW + rsub;
        if (j == 0 && r < cnt) {
          const float v = acc * a.scale;
          sh.lg[r] = v;
          vmin = fminf(vmin, v);
          vmax = fmaxf(vmax, v);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      vmin = fminf(vmin, __shfl_xor_sync(FULL_MASK, vmin, o));
      vmax = fmaxf(vmax, __shfl_xor_sync(FULL_MASK, vmax, o));
    }
    if (lane == 0) {
      sh.red[warp] = vmin;
      sh.red2[warp] = vmax;
    }
    __syncthreads();
    if (tid < CL) {
      float m0 = INFINITY, m1 = -INFINITY;
#pragma unroll
      for (int w = 0; w < RT_WARPS; w++) {
        m0 = fminf(m0, sh.red[w]);
        m1 = fmaxf(m1, sh.red2[w]);
      }
      RetrieveShared<DK>* rs = at_rank<ONE>(cluster, sh, tid);
      rs->rmin[rank] = m0;
      rs->rmax[rank] = m1;
    }
  }
  cluster_barrier<ONE>(cluster);  // every rank's range in every rank
  float smin = INFINITY, smax = -INFINITY;
#pragma unroll
  for (int r = 0; r < SELECT_FUSED_CL; r++) {  // every slot exists; ranks >= CL masked
    const float x0 = sh.rmin[r], x1 = sh.rmax[r];
    smin = r < CL ? fminf(smin, x0) : smin;
    smax = r < CL ? fmaxf(smax, x1) : smax;
  }

  const bool mine = tid < cnt;
  const float s = mine ? sh.lg[tid] : -INFINITY;

  // candidate path: the V rows loaded while its barrier completes
  CandRound<UD_ROWS> cr;

  // ---- the decision: threshold key thr, ties kept keq, lower ranks' counts ----
  unsigned thr = 0, keq = 0, carry_gt = 0, carry_eq = 0;
  if (Nb >= t) {  // every key: all count as above a zero threshold
    keq = 0xffffffffu;
    carry_gt = (unsigned)lo;
  } else if (!(smax > smin)) {  // every logit equal: the lowest indices win
    thr = order_key(smax);
    keq = (unsigned)Nb;
    carry_eq = (unsigned)lo;
  } else {
    // ---- round 2: 64-bin histograms until the final bin is small or one value ----
    int st = mine ? 2 : 0;  // 0 dropped, 1 kept (above the final bin), 2 in the current bin
    unsigned krem = (unsigned)Nb, carry_above = 0;
    {
      float blo = smin, bw = smax - smin;
      unsigned inb_lo = 0;
      int path = 0;  // 0 candidates, 1 one value, 2 radix fallback
      for (int round = 0;; round++) {
        const int c = st == 2 ? bin_of<RT_HB>(s, blo, (float)RT_HB / bw) : -1;
        hist_round<DK, ONE>(cluster, sh, CL, rank, c, krem);
        const int bsel = (int)sh.bin;
        krem = sh.krem;
        carry_above += sh.above_lo;
        inb_lo = sh.inb_lo;
        if (st == 2) st = c > bsel ? 1 : (c < bsel ? 0 : 2);
        if (sh.cnt_bin <= (unsigned)RT_CANDS) break;
        // the bin is full: its exact range (ties show as a single value)
        float m0 = st == 2 ? s : INFINITY, m1 = st == 2 ? s : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          m0 = fminf(m0, __shfl_xor_sync(FULL_MASK, m0, o));
          m1 = fmaxf(m1, __shfl_xor_sync(FULL_MASK, m1, o));
        }
        if (lane == 0) {
          sh.red[warp] = m0;
          sh.red2[warp] = m1;
        }
        __syncthreads();
        if (tid < CL) {
          float x0 = INFINITY, x1 = -INFINITY;
#pragma unroll
          for (int w = 0; w < RT_WARPS; w++) {
            x0 = fminf(x0, sh.red[w]);
            x1 = fmaxf(x1, sh.red2[w]);
          }
          RetrieveShared<DK>* rs = at_rank<ONE>(cluster, sh, tid);
          rs->rmin[rank] = x0;
          rs->rmax[rank] = x1;
        }
        cluster_barrier<ONE>(cluster);
        float g0 = INFINITY, g1 = -INFINITY;
#pragma unroll
        for (int r = 0; r < SELECT_FUSED_CL; r++) {
          const float x0 = sh.rmin[r], x1 = sh.rmax[r];
          g0 = r < CL ? fminf(g0, x0) : g0;
          g1 = r < CL ? fmaxf(g1, x1) : g1;
        }
        if (!(g1 > g0)) {
          path = 1;
          thr = order_key(g1);
          break;
        }
        if (round + 1 >= RT_ROUNDS) {
          path = 2;
          break;
        }
        blo = g0;
        bw = g1 - g0;
      }
      if (path == 1) {  // every key of the final bin has the same logit
        keq = krem;
        carry_gt = carry_above;
        carry_eq = inb_lo;
      } else if (path == 2) {
        if (rank == 0) radix_decide<DK, ONE>(cluster, sh, CL, chunk, t, (unsigned)Nb);
        cluster_barrier<ONE>(cluster);
        thr = sh.thr;
        keq = sh.keq;
        carry_gt = sh.carry_gt;
        carry_eq = sh.carry_eq;
      } else {
        candidate_round<T, DK, ONE>(kv, cluster, sh, cr, CL, rank, b, kvh, lo, st, s, inb_lo,
                                    min(sh.cnt_bin, (unsigned)RT_CANDS), krem, carry_above, thr, keq,
                                    carry_gt, carry_eq);
      }
    }
  }

  // ---- round 4: index-ordered compaction of the slice (one key per thread) ----
  const unsigned below = (1u << lane) - 1u;
  const unsigned u = order_key(s);
  const unsigned mgt = __ballot_sync(FULL_MASK, mine && u > thr);
  const unsigned meq = __ballot_sync(FULL_MASK, mine && u == thr);
  __syncthreads();  // sh.scan may still be read by the decision's counts
  if (lane == 0) sh.scan[warp] = ((unsigned)__popc(mgt) << 16) | (unsigned)__popc(meq);
  __syncthreads();
  unsigned before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < RT_WARPS; w++) {
    const unsigned c = sh.scan[w];
    before += w < warp ? c : 0u;
    tot += c;
  }
  const unsigned g = carry_gt + (before >> 16) + __popc(mgt & below);
  const unsigned q = carry_eq + (before & 0xffffu) + __popc(meq & below);
  const unsigned base = carry_gt + min(carry_eq, keq);
  const unsigned n_own = (tot >> 16) + min(carry_eq + (tot & 0xffffu), keq) - min(carry_eq, keq);
  bool take = false;
  unsigned pos = 0;
  if ((mgt >> lane) & 1u) {
    take = true;
    pos = g + min(q, keq);
  } else if (((meq >> lane) & 1u) && q < keq) {
    take = true;
    pos = g + q;
  }
  float dsum = 0.f;
  if (take) {
    if (pos < (unsigned)n && pos - base < (unsigned)RT_SLICE) {
      sh.kept[pos - base] = lo + tid;
      if (!cr.on) sh.dl[pos - base] = tid;  // the rows to gather
    } else {
      raise_error(kv.err, PRHS_DEV_CAPACITY);
    }
  } else if (mine) {
    dsum = expf(s - smax);
  }
  if (mine) sh.take[tid] = take ? 1 : 0;
  __syncthreads();
  const int nown = (int)min(n_own, (unsigned)RT_SLICE);

  // ---- V rows of this CTA's kept keys, weighted; sums to rank 0 ----
  float acc[EPC];
#pragma unroll
  for (int e = 0; e < EPC; e++) acc[e] = 0.f;
  float lsum = 0.f;
  if (cr.on) {
#pragma unroll
    for (int k = 0; k < UD_ROWS; k++) {
      const float w = cr.di[k] >= 0 ? expf(sh.lg[cr.di[k]] - smax) : 0.f;
      float f[EPC];
      Elem<T>::unpack(cr.dv[k], f);
#pragma unroll
      for (int e = 0; e < EPC; e++) acc[e] = fmaf(w, f[e], acc[e]);
      lsum += w;
    }
    gather_rows<T, DK>(kv, sh, sh.dl, UD_ROWS * RPW, cr.nd, false, b, kvh, lo, t, smax, acc, lsum);
    if (cr.ci >= 0 && sh.take[cr.ci]) {
      const float w = expf(sh.lg[cr.ci] - smax);
      float f[EPC];
      Elem<T>::unpack(cr.cv, f);
#pragma unroll
      for (int e = 0; e < EPC; e++) acc[e] = fmaf(w, f[e], acc[e]);
      lsum += w;
    }
    gather_rows<T, DK>(kv, sh, sh.cl, RPW, cr.ncl, true, b, kvh, lo, t, smax, acc, lsum);
  } else {
    gather_rows<T, DK>(kv, sh, sh.dl, 0, nown, false, b, kvh, lo, t, smax, acc, lsum);
  }
  // over the rows of a warp (lanes with the same j), then over the warps
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < EPC; e++) acc[e] += __shfl_xor_sync(FULL_MASK, acc[e], o);
    lsum += __shfl_xor_sync(FULL_MASK, lsum, o);
  }
  dsum = warp_sum(dsum);
  if (lane < LPR)
#pragma unroll
    for (int e = 0; e < EPC; e++) sh.wsum[warp * DK + j * EPC + e] = acc[e];
  if (lane == 0) {
    sh.red[warp] = lsum;
    sh.red2[warp] = dsum;
  }
  __syncthreads();
  RetrieveShared<DK>* root = at_rank<ONE>(cluster, sh, 0);
  for (int e = tid; e < DK; e += RT_THREADS) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < RT_WARPS; w++) o += sh.wsum[w * DK + e];
    root->part[rank][e] = o;
  }
  if (tid == 0) {
    float l = 0.f, dd = 0.f;
#pragma unroll
    for (int w = 0; w < RT_WARPS; w++) {
      l += sh.red[w];
      dd += sh.red2[w];
    }
    root->part[rank][DK] = l;
    root->part[rank][DK + 1] = dd;
  }
  cluster_barrier<ONE>(cluster);  // every rank's sums are in rank 0

  // ---- the set (each rank its own part, coalesced) and, in rank 0, the outputs ----
  for (int p = tid; p < nown && base + p < (unsigned)n; p += RT_THREADS) {
    out[base + p] = sh.kept[p];
    if (aout) aout[base + p] = sh.kept[p];
  }
  if (rank != 0) return;
  float L = 0.f, D = 0.f;
#pragma unroll
  for (int r = 0; r < SELECT_FUSED_CL; r++) {  // every slot exists; ranks >= CL masked
    const float x = sh.part[r][DK], y = sh.part[r][DK + 1];
    L += r < CL ? x : 0.f;
    D += r < CL ? y : 0.f;
  }
  for (int e = tid; e < DK; e += RT_THREADS) {
    float o = 0.f;
#pragma unroll
    for (int r = 0; r < SELECT_FUSED_CL; r++) {
      const float x = sh.part[r][e];
      o += r < CL ? x : 0.f;
    }
    a.out[(long long)qh * DK + e] = L > 0.f ? o / L : 0.f;
  }
  if (tid == 0) {
    a.lse[qh] = L > 0.f ? smax + logf(L) : -INFINITY;
    a.n_sel[qh] = n;
    a.delta[qh] = D + L > 0.f ? D / (D + L) : 0.f;
    if (a.anchor_n) a.anchor_n[qh] = n;
  }
  if (qa_dst) *qa_dst = qsrc;
}

template <typename T, int DK>
cudaError_t dispatch_d(const SelectLaunch& a, int cl, int chunk, cudaStream_t st) {
  void (*k)(const SelectLaunch, int) =
      cl == 1 ? retrieve_kernel<T, DK, true> : retrieve_kernel<T, DK, false>;
  const size_t smem =
      stage_by_copy<T, DK>(a.kv.block_table != nullptr, chunk) ? (size_t)chunk * DK * sizeof(T) : 0;
  return launch_select_grid(k, a, cl, chunk, smem, st);
}

template <typename T>
cudaError_t dispatch(const SelectLaunch& a, int cl, int chunk, cudaStream_t st) {
  if (a.kv.d == 128) return dispatch_d<T, 128>(a, cl, chunk, st);
  if (a.kv.d == 64) return dispatch_d<T, 64>(a, cl, chunk, st);
  return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_retrieve(const SelectLaunch& a, cudaStream_t st) {
  int cl = 1, chunk = 0;
  if (!score_select_geometry(a.kv, &cl, &chunk)) return cudaErrorNotSupported;
  if (a.out == nullptr || a.lse == nullptr || a.n_sink > 0 || a.window > 0) return cudaErrorInvalidValue;
  return a.kv.dtype == PRHS_BF16 ? dispatch<__nv_bfloat16>(a, cl, chunk, st)
                                 : dispatch<float>(a, cl, chunk, st);
}

}  // namespace prhs
