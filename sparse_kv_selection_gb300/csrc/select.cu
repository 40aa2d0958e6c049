// Top-N selection and dropped mass, one thread-block cluster per query head:
// from the logits of prhs_score (select_cluster_kernel), or with the logits
// computed from K in the same launch (score_select_kernel, caches of up to
// 8192 keys; the retrieval with its attention is in retrieve.cu).
// "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference":
// abstract (top-k oracle selection before attention; the dropped mass delta),
// Table I (S_t, N, tau(.), delta(.)) and the Table V caption (attention over
// the selected KV entries only).
//
// select_cluster_kernel: the CL CTAs of a cluster (often one) each hold a
// contiguous slice of the head's logits in shared memory (one read of the
// logits from L2/HBM). The threshold is found on value bins: the logit
// range, a 2048-bin histogram over it summed into CTA 0 through distributed
// shared memory, a second 2048 bins inside the threshold bin when it holds
// more than SEL_CANDS logits, then the candidates of the final bin ranked
// exactly; heavy ties fall back to three
// radix passes (11, 11, 10 bits of an order-preserving key). Every CTA takes
// the same decision. The index-ordered compaction gets each CTA's output
// offset from the counts of the lower ranks, so the set comes out ascending
// with ties resolved to the lowest index, and the dropped mass is the cluster
// sum of the unselected weights. Forced keys (sinks, window) are ranked below
// every other key and left to the caller. score_select_kernel runs the same
// one-CTA selection in CTA 0 of its cluster after the cluster has scored.
#include <cooperative_groups.h>

#include "kernels.h"

namespace cg = cooperative_groups;

namespace prhs {

constexpr int SEL_THREADS = 512;
constexpr int SEL_WARPS = SEL_THREADS / 32;

// Candidates ranked exactly after the bin passes. The ranking costs
// candidates^2 / threads steps, so a bin holding more runs the second, finer
// bin pass first.
constexpr int SEL_CANDS = 64;

struct SelClusterShared {
  unsigned hist[2048];        // this CTA's histogram of the current bin pass
  unsigned histg[2][2048];    // rank 0: cluster totals of the two value-bin passes
  unsigned fb[2][2048];       // fallback radix passes: this CTA's histograms
  unsigned cand[SEL_CANDS];   // rank 0: gathered candidate keys; every rank: a copy
  unsigned lcand[SEL_CANDS];  // this CTA's own candidate keys
  unsigned candi[SEL_CANDS];  // one CTA: each candidate's position in the slice
  unsigned lcandi[SEL_CANDS]; // cluster: each own candidate's position in the slice
  unsigned ncand, nlcand;
  unsigned scan[32];
  float red[SEL_WARPS], red2[SEL_WARPS];
  float lmin, lmax;           // this CTA's logit range
  float Zp;                   // this CTA's sum of exp(s - max) over all its logits
  unsigned cnt_gt, cnt_eq;    // this CTA's logits above / equal to the threshold
  float dsum;                 // this CTA's dropped weight
  unsigned digit, krem, cnt_bin, thr, keq;
  float rmin[SELECT_FUSED_CL], rmax[SELECT_FUSED_CL];  // score-and-select: each rank's logit range
};

__device__ __forceinline__ void merge_mz(float& m, float& z, float m2, float z2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  z = (m == -INFINITY ? 0.f : z * expf(m - M)) + (m2 == -INFINITY ? 0.f : z2 * expf(m2 - M));
  m = M;
}

// Block-wide inclusive scan of one unsigned per thread.
__device__ __forceinline__ unsigned scan_block(unsigned v, unsigned* warp_tot, unsigned& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned n = __shfl_up_sync(FULL_MASK, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned w = lane < nw ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned n = __shfl_up_sync(FULL_MASK, w, o);
      if (lane >= o) w += n;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  total = warp_tot[nw - 1];
  const unsigned add = warp > 0 ? warp_tot[warp - 1] : 0u;
  __syncthreads();
  return v + add;
}

template <typename T>
__device__ __forceinline__ void mirror_query(const SelectLaunch& a, int qh) {
  for (int i = threadIdx.x; i < a.kv.d; i += blockDim.x)
    copy_elem<T>(a.q_anchor, a.q_src, (long long)qh * a.kv.d + i);
}

// Bin of a histogram (nb bins, highest first) holding the krem-th largest
// element; `h` may live in another CTA's shared memory. Sets sh.digit, the
// rank sh.krem inside that bin and its count sh.cnt_bin.
__device__ __forceinline__ void find_bin_counts(const unsigned (&c)[4], int per, int top,
                                                unsigned krem, SelClusterShared& sh) {
  unsigned sum = 0;
  for (int k = 0; k < per; k++) sum += c[k];
  unsigned total;
  unsigned run = scan_block(sum, sh.scan, total) - sum;
  for (int k = 0; k < per; k++) {
    if (run < krem && run + c[k] >= krem) {
      sh.digit = (unsigned)(top - k);
      sh.krem = krem - run;
      sh.cnt_bin = c[k];
    }
    run += c[k];
  }
  __syncthreads();
}

__device__ __forceinline__ void find_bin(const unsigned* h, int nb, unsigned krem,
                                         SelClusterShared& sh) {
  const int per = nb / SEL_THREADS;  // 4 or 2
  const int top = nb - 1 - per * threadIdx.x;
  unsigned c[4] = {0u, 0u, 0u, 0u};
  for (int k = 0; k < per; k++) c[k] = h[top - k];
  find_bin_counts(c, per, top, krem, sh);
}

// A cluster's histogram: every rank writes its 2048 counts, as 16-bit values
// (a slice holds at most SELECT_SLICE_MAX keys), into its row of a table in
// rank 0's shared memory (the cluster totals and fallback counters, unused
// until the bins are found): 256 16-byte stores, no atomics. The caller then
// passes a cluster barrier.
constexpr int SEL_ROWS_MAX = 8;  // ranks a table holds: 8 rows of 2048 16-bit counts
static_assert(SELECT_SLICE_MAX < 65536, "slice counts fit 16 bits");
__device__ __forceinline__ void push_hist_row(cg::cluster_group& cluster, const SelClusterShared& sh,
                                              int rank) {
  const int t = threadIdx.x;
  if (t < 2048 / 8) {
    const unsigned* h = sh.hist + 8 * t;
    const uint4 v = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                               h[6] | (h[7] << 16));
    SelClusterShared* root = cluster.map_shared_rank(const_cast<SelClusterShared*>(&sh), 0);
    reinterpret_cast<uint4*>(&root->histg[0][0])[rank * (2048 / 8) + t] = v;
  }
}

// The bin of the krem-th largest in a cluster's 2048-bin histogram: rank 0
// adds the ranks' rows of its table as it scans them and writes the result
// into every rank's shared memory (remote reads of 2048 counters by every rank
// cost several microseconds); one cluster barrier.
template <bool ONE>
__device__ __forceinline__ void find_bin_cluster(cg::cluster_group& cluster, SelClusterShared& sh,
                                                 unsigned krem, int CL, int rank) {
  if (rank == 0) {
    // Each thread adds its four bins (top-3 .. top, one 8-byte word of a row)
    // over the ranks' rows.
    static_assert(2048 / SEL_THREADS == 4, "four bins a thread");
    const uint2* tab = reinterpret_cast<const uint2*>(&sh.histg[0][0]);
    const int top = 2047 - 4 * (int)threadIdx.x;
    unsigned c[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int r = 0; r < SEL_ROWS_MAX; r++) {
      if (r < CL) {
        const uint2 w = tab[r * (2048 / 4) + (top - 3) / 4];
        c[3] += w.x & 0xffffu;
        c[2] += w.x >> 16;
        c[1] += w.y & 0xffffu;
        c[0] += w.y >> 16;
      }
    }
    find_bin_counts(c, 4, top, krem, sh);
    if (threadIdx.x < CL) {
      SelClusterShared* rs = cluster.map_shared_rank(&sh, (int)threadIdx.x);
      rs->digit = sh.digit;
      rs->krem = sh.krem;
      rs->cnt_bin = sh.cnt_bin;
    }
  }
  cluster.sync();
}

__device__ __forceinline__ float float_of_key(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Value bins: monotone non-decreasing in s, clamped to [0, 2047].
__device__ __forceinline__ int vbin(float s, float lo, float inv) {
  const float x = (s - lo) * inv;
  return x <= 0.f ? 0 : (x >= 2047.f ? 2047 : (int)x);
}

// Barrier over the head's CTAs: the cluster when the head is split, the block
// otherwise (a one-CTA cluster barrier would add a cluster-scope fence).
template <bool ONE>
__device__ __forceinline__ void head_sync(cg::cluster_group& cluster) {
  if (ONE) __syncthreads(); else cluster.sync();
}

template <bool ONE>
__device__ __forceinline__ SelClusterShared* rank_shared(cg::cluster_group& cluster,
                                                         SelClusterShared& sh, int r) {
  if (ONE) return &sh;
  return cluster.map_shared_rank(&sh, r);
}

// Logits s_i = scale * <q, k_i> of keys [lo, lo + cnt) of query head qh,
// computed from 16-byte pieces of the K rows (LPR lanes per row, all of a
// thread's loads issued before the first is used), into a.logits_out when set
// and into cache (forced keys as -inf) when cache is set, with the range of
// the unforced ones.
template <typename T, int DK>
__device__ __forceinline__ void slice_logits(const SelectLaunch& a, int qh, int b, int lo, int cnt,
                                             int ns, int we, float* cache, float& vmin, float& vmax) {
  const KVView& kv = a.kv;
  constexpr int EPC = Elem<T>::per16;       // elements per 16-byte piece
  constexpr int LPR = DK / EPC;             // lanes per K row: 8, 16 or 32
  constexpr int RPW = SEL_THREADS / LPR;    // rows per CTA-wide wave of loads
  constexpr int U = 8;                      // waves in flight per thread
  static_assert(LPR >= 8 && LPR <= 32 && (LPR & (LPR - 1)) == 0, "row split");
  const int tid = threadIdx.x;
  const int j = tid & (LPR - 1);
  const int kvh = (qh % kv.Hq) / (kv.Hq / kv.Hkv);
  float qf[EPC];
  Elem<T>::unpack(__ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.q) +
                                                       (long long)qh * DK * sizeof(T)) + j), qf);
  const char* kb = static_cast<const char*>(kv.k);
  float* lout = a.logits_out != nullptr ? a.logits_out + (long long)qh * kv.t_max + lo : nullptr;
  for (int r0 = 0; r0 < cnt; r0 += RPW * U) {
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int r = r0 + u * RPW + tid / LPR;
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
      const int r = r0 + u * RPW + tid / LPR;
      if (j == 0 && r < cnt) {
        const float v = acc * a.scale;
        if (lout != nullptr) lout[r] = v;
        if (cache != nullptr) {
          const bool forced = lo + r < ns || lo + r >= we;  // ranked below every middle key
          cache[r] = forced ? -INFINITY : v;
          if (!forced) {
            vmin = fminf(vmin, v);
            vmax = fmaxf(vmax, v);
          }
        }
      }
    }
  }
}

// Selection over logits already in shared memory: this CTA holds keys
// [lo, lo + cnt) of query head qh in cache (forced keys as -inf), and vmin,
// vmax is its thread's share of their range. The CL CTAs of the cluster call
// it together (CL = 1 when ONE).
template <typename T, bool ONE>
__device__ __forceinline__ void select_in_shared(const SelectLaunch& a, SelClusterShared& sh,
                                                 const float* cache, cg::cluster_group& cluster,
                                                 const int CL, const int rank, const int qh, const int Nb,
                                                 int32_t* out, int32_t* aout, const int lo, const int cnt,
                                                 float vmin, float vmax) {
  const KVView& kv = a.kv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 2048; i += SEL_THREADS) sh.hist[i] = 0;
  if (tid == 0) {
    sh.ncand = 0;
    sh.nlcand = 0;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    vmin = fminf(vmin, __shfl_xor_sync(FULL_MASK, vmin, o));
    vmax = fmaxf(vmax, __shfl_xor_sync(FULL_MASK, vmax, o));
  }
  if (lane == 0) {
    sh.red[warp] = vmin;
    sh.scan[warp] = __float_as_uint(vmax);
  }
  __syncthreads();
  float smin = INFINITY, smax = -INFINITY;  // every thread reads the warp results
#pragma unroll
  for (int w = 0; w < SEL_WARPS; w++) {
    smin = fminf(smin, sh.red[w]);
    smax = fmaxf(smax, __uint_as_float(sh.scan[w]));
  }
  if (!ONE) {
    if (tid == 0) {
      sh.lmin = smin;
      sh.lmax = smax;
    }
    __syncthreads();
    head_sync<ONE>(cluster);  // ranges published; rank 0's accumulators are zero
    smin = INFINITY;
    smax = -INFINITY;
    for (int r = 0; r < CL; r++) {
      const SelClusterShared* rs = rank_shared<ONE>(cluster, sh, r);
      smin = fminf(smin, rs->lmin);
      smax = fmaxf(smax, rs->lmax);
    }
  }
  SelClusterShared* root = rank_shared<ONE>(cluster, sh, 0);
  const bool flat = !(smax > smin);
  const float w1 = (smax - smin) * (1.f / 2048.f);
  const float inv1 = flat ? 0.f : 2048.f / (smax - smin);

  // ---- pass 1: value histogram over [smin, smax]; this thread's share of the
  // CTA's total weight sum exp(s - max) (delta's denominator) ----
  float zacc = 0.f;
  if (!flat) {
    for (int i = tid; i < cnt; i += SEL_THREADS) {
      const float s = cache[i];
      atomicAdd(&sh.hist[vbin(s, smin, inv1)], 1u);
      zacc += __expf(s - smax);  // weights for delta only: few-ulp error, 1e-4 tolerance
    }
    if (!ONE) {
      __syncthreads();
      push_hist_row(cluster, sh, rank);
    }
  }
  __syncthreads();
  if (!ONE) head_sync<ONE>(cluster);

  // ---- threshold: the key of the N-th largest logit, and how many ties to keep ----
  unsigned thr = 0, keq = 0, cta_gt = 0, cta_eq = 0;
  bool fallback = false;
  if (flat) {  // every logit of the head is equal: the lowest indices win
    thr = order_key(smax);
    keq = (unsigned)Nb;
    cta_eq = (unsigned)cnt;
  } else {
    if (ONE) find_bin(sh.hist, 2048, (unsigned)Nb, sh);
    else find_bin_cluster<ONE>(cluster, sh, (unsigned)Nb, CL, rank);
    const int b1 = (int)sh.digit;
    unsigned krem = sh.krem;
    const float lo1 = smin + (float)b1 * w1;
    const float inv2 = w1 > 0.f ? 2048.f / w1 : 0.f;
    int b2 = -1;  // -1: the candidates are all of bin b1
    if (sh.cnt_bin > SEL_CANDS) {
      // pass 2: second value histogram inside bin b1
      for (int i = tid; i < 2048; i += SEL_THREADS) sh.hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < cnt; i += SEL_THREADS) {
        const float s = cache[i];
        if (vbin(s, smin, inv1) == b1) atomicAdd(&sh.hist[vbin(s, lo1, inv2)], 1u);
      }
      __syncthreads();
      if (!ONE) {
        push_hist_row(cluster, sh, rank);
        __syncthreads();
        head_sync<ONE>(cluster);
      }
      if (ONE) find_bin(sh.hist, 2048, krem, sh);
      else find_bin_cluster<ONE>(cluster, sh, krem, CL, rank);
      b2 = (int)sh.digit;
      krem = sh.krem;
    }
    if (sh.cnt_bin <= SEL_CANDS) {
      // pass 3: gather the candidates; count the logits above them and mark
      // them in a bitmap of the slice (one ballot word per warp and 32 keys, in
      // sh.hist, free after the bin passes)
      unsigned dgt = 0;
      unsigned* bits = sh.hist;
      constexpr int UC = 4;  // rows of 512 keys per iteration, read before the first is used
      for (int r0 = 0; r0 < cnt; r0 += SEL_THREADS * UC) {
        float sv[UC];
#pragma unroll
        for (int k = 0; k < UC; k++) {
          const int i = r0 + k * SEL_THREADS + tid;
          sv[k] = i < cnt ? cache[i] : -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < UC; k++) {
        const int i0 = r0 + k * SEL_THREADS;
        if (i0 >= cnt) break;  // uniform over the block
        const int i = i0 + tid;
        const float s = sv[k];
        const int c1 = vbin(s, smin, inv1);
        bool cand = false, above = false;
        if (i < cnt) {
          if (c1 > b1) {
            above = true;
          } else if (c1 == b1) {
            if (b2 < 0) {
              cand = true;
            } else {
              const int c2 = vbin(s, lo1, inv2);
              above = c2 > b2;
              cand = c2 == b2;
            }
          }
        }
        dgt += above;
        const unsigned word = __ballot_sync(FULL_MASK, above);
        if (lane == 0) bits[(i0 >> 5) + warp] = word;
        if (cand) {
          const unsigned u = order_key(s);
          const unsigned slot = atomicAdd(&root->ncand, 1u);
          if (slot < SEL_CANDS) {
            root->cand[slot] = u;
            if (ONE) root->candi[slot] = (unsigned)i;
          }
          if (!ONE) {
            const unsigned ls = atomicAdd(&sh.nlcand, 1u);
            if (ls < SEL_CANDS) {
              sh.lcand[ls] = u;
              sh.lcandi[ls] = (unsigned)i;
            }
          }
        }
        }
      }
      // a single CTA needs no count of its own: nothing follows it
      unsigned dgt_cta = 0;
      if (!ONE) scan_block(dgt, sh.scan, dgt_cta);
      head_sync<ONE>(cluster);
      const unsigned nc = min(root->ncand, (unsigned)SEL_CANDS);
      unsigned myc = 0;
      if (tid < (int)nc) myc = root->cand[tid];
      if (!ONE) {
        __syncthreads();
        if (tid < (int)nc) sh.cand[tid] = myc;
        __syncthreads();
      }
      if (tid < (int)nc) {  // exact rank of each candidate among all candidates
        unsigned g = 0, e = 0;
        for (unsigned jj = 0; jj < nc; jj++) {
          g += sh.cand[jj] > myc;
          e += sh.cand[jj] == myc;
        }
        if (g < krem && g + e >= krem) {
          sh.thr = myc;
          sh.keq = krem - g;
        }
      }
      __syncthreads();
      thr = sh.thr;
      keq = sh.keq;
      if (!ONE) {
        const unsigned nl = min(sh.nlcand, (unsigned)SEL_CANDS);
        cta_gt = dgt_cta;
        for (unsigned jj = 0; jj < nl; jj++) {
          cta_gt += sh.lcand[jj] > thr;
          cta_eq += sh.lcand[jj] == thr;
        }
      }
    } else {
      fallback = true;  // heavy ties or a very dense spot: exact radix over all logits
    }
  }
  if (fallback) {
    unsigned prefix = 0, mask = 0, krem = (unsigned)Nb;
    for (int pass = 0; pass < 3; pass++) {
      const int buf = pass & 1;
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int nb = pass == 2 ? 1024 : 2048;
      for (int i = tid; i < nb; i += SEL_THREADS) sh.fb[buf][i] = 0;
      __syncthreads();
      for (int i = tid; i < cnt; i += SEL_THREADS) {
        const unsigned u = order_key(cache[i]);
        if ((u & mask) == prefix) atomicAdd(&sh.fb[buf][(u >> shift) & (nb - 1)], 1u);
      }
      __syncthreads();
      head_sync<ONE>(cluster);
      for (int i = tid; i < nb; i += SEL_THREADS) {
        unsigned tot = 0;
        for (int r = 0; r < CL; r++) tot += rank_shared<ONE>(cluster, sh, r)->fb[buf][i];
        sh.hist[i] = tot;
      }
      __syncthreads();
      find_bin(sh.hist, nb, krem, sh);
      prefix |= sh.digit << shift;
      mask |= (unsigned)(nb - 1) << shift;
      krem = sh.krem;
    }
    thr = prefix;
    keq = krem;
    unsigned lgt = 0, leq = 0;
    for (int i = tid; i < cnt; i += SEL_THREADS) {
      const unsigned u = order_key(cache[i]);
      lgt += u > thr;
      leq += u == thr;
    }
    scan_block(lgt, sh.scan, cta_gt);
    scan_block(leq, sh.scan, cta_eq);
  }
  unsigned carry_gt = 0, carry_eq = 0;  // counts in the lower ranks' slices
  if (!ONE) {
    if (tid == 0) {
      sh.cnt_gt = cta_gt;
      sh.cnt_eq = cta_eq;
    }
    __syncthreads();
    head_sync<ONE>(cluster);
    for (int r = 0; r < rank; r++) {
      const SelClusterShared* rs = rank_shared<ONE>(cluster, sh, r);
      carry_gt += rs->cnt_gt;
      carry_eq += rs->cnt_eq;
    }
  }

  // ---- index-ordered compaction; dropped weight of the rest ----
  // Warp w takes keys [base + 256 w, base + 256 (w + 1)) of each tile of 4096
  // keys, lane l the keys base + 256 w + 32 e + l (e < 8, conflict-free
  // reads): ballots give each key's counts of keys above / at the threshold
  // before it inside its warp, one prefix over the warps' totals the rest.
  constexpr int E = 8;
  constexpr int WSPAN = 32 * E;
  constexpr int TILE = SEL_THREADS * E;
  float dsum = 0.f, ssum = 0.f;  // weights exp(s - max) of dropped / kept logits
  const unsigned below = (1u << lane) - 1u;
  if (!flat && !fallback) {
    // The candidate path: the bitmap holds the keys above the threshold's bin;
    // the kept candidates join it (ties in index order, after the lower
    // ranks' ties), then positions come from a prefix over the words' counts
    // and only the kept keys are written and weighed (dropped weight = this
    // CTA's total minus the kept one).
    unsigned* bits = sh.hist;
    const unsigned* ck = ONE ? sh.cand : sh.lcand;
    const unsigned* cix = ONE ? sh.candi : sh.lcandi;
    const unsigned ncl = min(ONE ? sh.ncand : sh.nlcand, (unsigned)SEL_CANDS);
    if (tid < (int)ncl) {
      const unsigned u = ck[tid], i = cix[tid];
      bool keep = u > thr;
      if (u == thr) {
        unsigned r = carry_eq;  // equal keys before this one, in index order
        for (unsigned jj = 0; jj < ncl; jj++) r += ck[jj] == thr && cix[jj] < i;
        keep = r < keq;
      }
      if (keep && (int)i < cnt) atomicOr(&bits[i >> 5], 1u << (i & 31));
    }
    __syncthreads();
    // rounds of one word per thread (kept keys cluster in index order, so
    // contiguous ranges per thread would leave a few threads most of them)
    const int nw = (cnt + 31) >> 5;
    unsigned carry_pos = carry_gt + min(carry_eq, keq);
    for (int w0 = 0; w0 < nw; w0 += SEL_THREADS) {
      const int w = w0 + tid;
      unsigned m = w < nw ? bits[w] : 0u;
      const unsigned c = __popc(m);
      unsigned tot_kept;
      unsigned pos = carry_pos + scan_block(c, sh.scan, tot_kept) - c;
      carry_pos += tot_kept;
      while (m != 0u) {
        const int i = (w << 5) + __ffs(m) - 1;
        m &= m - 1u;
        if (pos < (unsigned)Nb) {
          out[pos] = lo + i;
          if (aout) aout[pos] = lo + i;
        } else {
          raise_error(kv.err, PRHS_DEV_CAPACITY);
        }
        pos++;
        ssum += __expf(cache[i] - smax);
      }
    }
    dsum = zacc - ssum;
  } else
  for (int base = 0; base < cnt; base += TILE) {
    const int wbase = base + warp * WSPAN;
    float sv[E];
    unsigned mgt[E], meq[E];
    unsigned ngt = 0, neq = 0;
#pragma unroll
    for (int e = 0; e < E; e++) {
      const int i = wbase + e * 32 + lane;
      sv[e] = i < cnt ? cache[i] : -INFINITY;
    }
#pragma unroll
    for (int e = 0; e < E; e++) {
      const int i = wbase + e * 32 + lane;
      const unsigned u = order_key(sv[e]);
      mgt[e] = __ballot_sync(FULL_MASK, i < cnt && u > thr);
      meq[e] = __ballot_sync(FULL_MASK, i < cnt && u == thr);
      ngt += __popc(mgt[e]);
      neq += __popc(meq[e]);
    }
    if (lane == 0) sh.scan[warp] = (ngt << 16) | neq;  // at most 4096 each
    __syncthreads();
    unsigned before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < SEL_WARPS; w++) {
      const unsigned c = sh.scan[w];
      before += w < warp ? c : 0u;
      tot += c;
    }
    unsigned gt_before = carry_gt + (before >> 16);
    unsigned eq_before = carry_eq + (before & 0xffffu);
#pragma unroll
    for (int e = 0; e < E; e++) {
      const int i = wbase + e * 32 + lane;
      const unsigned g = gt_before + __popc(mgt[e] & below);
      const unsigned q = eq_before + __popc(meq[e] & below);
      gt_before += __popc(mgt[e]);
      eq_before += __popc(meq[e]);
      if (i >= cnt) continue;
      bool take = false;
      int pos = 0;
      if ((mgt[e] >> lane) & 1u) {
        take = true;
        pos = (int)(g + min(q, keq));
      } else if (((meq[e] >> lane) & 1u) && q < keq) {
        take = true;
        pos = (int)(g + q);
      }
      // weights for delta only (dropped / total mass): the fast exponential's
      // few-ulp error is far inside the 1e-4 tolerance of delta
      const float wgt = __expf(sv[e] - smax);
      if (take) {
        ssum += wgt;
        if (pos < Nb) {
          out[pos] = lo + i;
          if (aout) aout[pos] = lo + i;
        } else {
          raise_error(kv.err, PRHS_DEV_CAPACITY);
        }
      } else {
        dsum += wgt;
      }
    }
    carry_gt += tot >> 16;
    carry_eq += tot & 0xffffu;
    if (base + TILE < cnt) __syncthreads();  // the next tile rewrites the warp totals
  }
  dsum = warp_sum(dsum);
  ssum = warp_sum(ssum);
  if (lane == 0) {
    sh.red[warp] = dsum;
    sh.red2[warp] = ssum;
  }
  __syncthreads();
  if (tid == 0) {
    float s = 0.f, s2 = 0.f;
    for (int w = 0; w < SEL_WARPS; w++) {
      s += sh.red[w];
      s2 += sh.red2[w];
    }
    sh.dsum = s;
    sh.Zp = s + s2;
  }
  if (!ONE) {
    __syncthreads();
    head_sync<ONE>(cluster);
  }
  if (rank == 0) {
    if (tid == 0) {
      float s = 0.f, Z = 0.f;
      for (int r = 0; r < CL; r++) {
        const SelClusterShared* rs = rank_shared<ONE>(cluster, sh, r);
        s += rs->dsum;
        Z += rs->Zp;
      }
      a.n_sel[qh] = Nb;
      a.delta[qh] = s / Z;
      if (a.anchor_n) a.anchor_n[qh] = Nb;
    }
    if (a.q_anchor) mirror_query<T>(a, qh);
  }
  if (!ONE) head_sync<ONE>(cluster);  // shared memory stays valid until every remote read is done
}

// The c-th query head not flagged in skip (c = blockIdx.x), or -1 when fewer
// heads are left: every thread reads up to SEL_ORDER_PER flags, the block
// counts the unflagged ones and the thread holding the c-th names it. Heads
// with work then take the lowest block indices, which the block scheduler
// places first, and the CTAs past them exit without holding a slot long.
constexpr int SEL_ORDER_PER = 8;
__device__ __forceinline__ int nth_unskipped(const uint8_t* skip, int units, int c, unsigned* warp_tot,
                                             int* found) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j0 = tid * SEL_ORDER_PER;
  unsigned mine = 0;  // bit k: unit j0 + k has work
#pragma unroll
  for (int k = 0; k < SEL_ORDER_PER; k++)
    if (j0 + k < units && skip[j0 + k] == 0) mine |= 1u << k;
  const unsigned cnt = __popc(mine);
  unsigned total;
  const unsigned before = scan_block(cnt, warp_tot, total) - cnt;
  if (tid == 0) *found = -1;
  __syncthreads();
  if ((unsigned)c >= before && (unsigned)c < before + cnt) {
    unsigned m = mine;
    for (unsigned r = (unsigned)c - before; r > 0; r--) m &= m - 1;  // drop the lower set bits
    *found = j0 + __ffs(m) - 1;
  }
  __syncthreads();
  (void)lane;
  (void)warp;
  return *found;
}

template <typename T, bool ONE>
__global__ void __launch_bounds__(SEL_THREADS, 2) select_cluster_kernel(const SelectLaunch a, int chunk) {
  extern __shared__ __align__(16) float cache[];
  __shared__ SelClusterShared sh;
  __shared__ __align__(8) uint64_t lbar;  // the bulk copy of the logits
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = ONE ? 1 : (int)cluster.num_blocks();
  const int rank = ONE ? 0 : (int)cluster.block_rank();
  // a row stride of whole 16-byte groups lets one bulk copy bring the slice in
  const bool bulk = (a.kv.t_max & 3) == 0;
  if (bulk && threadIdx.x == 0) {
    mbar_init(&lbar, 1);
    fence_barrier_init();
  }
  pdl_wait();
  pdl_trigger();

  const KVView& kv = a.kv;
  int qh = blockIdx.x / CL;  // the cluster's query head (b * Hq + h)
  if (ONE && a.head_skip != nullptr && kv.B * kv.Hq <= SEL_THREADS * SEL_ORDER_PER) {
    __shared__ int found;
    qh = nth_unskipped(a.head_skip, kv.B * kv.Hq, qh, sh.scan, &found);
    if (qh < 0) return;
  } else if (a.head_skip != nullptr && a.head_skip[qh] != 0) {
    return;  // uniform over the cluster
  }
  const int b = qh / kv.Hq;
  const int tid = threadIdx.x;
  const int t = seq_len(kv, b);
  int Nb = a.n_budget != nullptr ? a.n_budget[b] : a.N;
  if (Nb < 0) Nb = 0;
  const int lim = a.anchor_idx != nullptr ? min(a.cap, a.anchor_cap) : a.cap;
  if (min(Nb, t) > lim) {
    if (tid == 0 && rank == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    Nb = lim;
  }
  int32_t* out = a.idx + (long long)qh * a.cap;
  int32_t* aout = a.anchor_idx != nullptr ? a.anchor_idx + (long long)qh * a.anchor_cap : nullptr;
  const int lo = min(t, rank * chunk), hi = min(t, lo + chunk), cnt = hi - lo;
  // forced keys [0, ns) and [we, t) are left out of the ranking: the set is
  // the top Nb of the middle keys [ns, we), written from position 0
  const int ns = min(max(a.n_sink, 0), t);
  const int we = max(ns, t - max(a.window, 0));
  const int tmid = we - ns;

  if (Nb >= tmid || Nb == 0) {  // keep every middle key (delta = 0 without forced keys) or none
    const int n = Nb >= tmid ? tmid : 0;
    for (int i = max(lo, ns) + tid; i < min(hi, ns + n); i += SEL_THREADS) {
      out[i - ns] = i;
      if (aout) aout[i - ns] = i;
    }
    if (rank == 0) {
      if (tid == 0) {
        a.n_sel[qh] = n;
        a.delta[qh] = n == t ? 0.f : 1.f;  // recomputed over the whole set when keys are forced
        if (a.anchor_n) a.anchor_n[qh] = n;
      }
      if (a.q_anchor) mirror_query<T>(a, qh);
    }
    return;
  }

  // ---- load this CTA's slice; its logit range ----
  const float* src = a.scores + (long long)qh * kv.t_max + lo;
  float vmin = INFINITY, vmax = -INFINITY;
  if (bulk) {
    __syncthreads();  // the barrier's initialisation is visible
    const int cnt4 = (cnt + 3) & ~3;  // whole 16-byte groups, inside the row (t_max % 4 == 0)
    if (tid == 0 && cnt4 > 0) {
      mbar_arrive_expect_tx(&lbar, (uint32_t)(cnt4 * sizeof(float)));
      bulk_load(cache, src, (uint32_t)(cnt4 * sizeof(float)), &lbar);
    }
    const bool ok = cnt4 == 0 || mbar_wait(&lbar, 0, kv.err);
    for (int i = tid; i < cnt; i += SEL_THREADS) {
      const float v = ok ? cache[i] : 0.f;
      const bool forced = lo + i < ns || lo + i >= we;  // ranked below every middle key
      cache[i] = forced ? -INFINITY : v;
      if (!forced) {
        vmin = fminf(vmin, v);
        vmax = fmaxf(vmax, v);
      }
    }
  }
  constexpr int PRE = 8;  // loads in flight per thread before the first is used
  for (int i0 = 0; !bulk && i0 < cnt; i0 += SEL_THREADS * PRE) {
    float v[PRE];
#pragma unroll
    for (int k = 0; k < PRE; k++) {
      const int i = i0 + k * SEL_THREADS + tid;
      v[k] = i < cnt ? src[i] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < PRE; k++) {
      const int i = i0 + k * SEL_THREADS + tid;
      if (i < cnt) {
        const bool forced = lo + i < ns || lo + i >= we;  // ranked below every middle key
        cache[i] = forced ? -INFINITY : v[k];
        if (!forced) {
          vmin = fminf(vmin, v[k]);
          vmax = fmaxf(vmax, v[k]);
        }
      }
    }
  }
  select_in_shared<T, ONE>(a, sh, cache, cluster, CL, rank, qh, Nb, out, aout, lo, cnt, vmin, vmax);
}

// Logits and top-N selection of one query head in one launch (the retrieval
// with its attention is retrieve_kernel). The cluster's CL CTAs each compute
// the logits of one slice of keys straight from K and store them into CTA 0's
// shared memory (distributed shared memory), with the slice's logit range;
// after one cluster barrier CTA 0 alone selects from the whole row, as the
// one-CTA selection does, and the other CTAs are done.
template <typename T, int DK, bool ONE>
__global__ void __launch_bounds__(SEL_THREADS, 2) score_select_kernel(const SelectLaunch a, int chunk) {
  extern __shared__ float cache[];  // CTA 0: the head's logits (t_max)
  __shared__ SelClusterShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = ONE ? 1 : (int)cluster.num_blocks();
  const int rank = ONE ? 0 : (int)cluster.block_rank();
  pdl_wait();
  pdl_trigger();

  const KVView& kv = a.kv;
  const int qh = blockIdx.x / CL;
  const int b = qh / kv.Hq;
  if (a.head_skip != nullptr && a.head_skip[qh] != 0) return;  // uniform over the cluster
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = seq_len(kv, b);
  int Nb = a.n_budget != nullptr ? a.n_budget[b] : a.N;
  if (Nb < 0) Nb = 0;
  const int lim = a.anchor_idx != nullptr ? min(a.cap, a.anchor_cap) : a.cap;
  if (min(Nb, t) > lim) {
    if (tid == 0 && rank == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    Nb = lim;
  }
  int32_t* out = a.idx + (long long)qh * a.cap;
  int32_t* aout = a.anchor_idx != nullptr ? a.anchor_idx + (long long)qh * a.anchor_cap : nullptr;
  const int lo = min(t, rank * chunk), hi = min(t, lo + chunk), cnt = hi - lo;
  const int ns = min(max(a.n_sink, 0), t);   // forced keys [0, ns) and [we, t)
  const int we = max(ns, t - max(a.window, 0));
  const int tmid = we - ns;

  // every middle key or none, without ranking (uniform over the cluster)
  if (Nb == 0 || Nb >= tmid) {
    const int n = Nb >= tmid ? tmid : 0;
    for (int i = max(lo, ns) + tid; i < min(hi, ns + n); i += SEL_THREADS) {
      out[i - ns] = i;
      if (aout) aout[i - ns] = i;
    }
    if (a.logits_out != nullptr) {  // the caller's set-mass pass reads every logit
      float u0 = 0.f, u1 = 0.f;
      slice_logits<T, DK>(a, qh, b, lo, cnt, ns, we, nullptr, u0, u1);
    }
    if (rank == 0) {
      if (tid == 0) {
        a.n_sel[qh] = n;
        a.delta[qh] = n == t ? 0.f : 1.f;  // recomputed over the whole set when keys are forced
        if (a.anchor_n) a.anchor_n[qh] = n;
      }
      if (a.q_anchor) mirror_query<T>(a, qh);
    }
    return;
  }

  // ---- this CTA's slice of logits, into CTA 0's row; the slice's range ----
  float* row = ONE ? cache : cluster.map_shared_rank(cache, 0);
  float vmin = INFINITY, vmax = -INFINITY;
  slice_logits<T, DK>(a, qh, b, lo, cnt, ns, we, row + lo, vmin, vmax);
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
  if (tid == 0) {
    float m0 = INFINITY, m1 = -INFINITY;
    for (int w = 0; w < SEL_WARPS; w++) {
      m0 = fminf(m0, sh.red[w]);
      m1 = fmaxf(m1, sh.red2[w]);
    }
    SelClusterShared* root = ONE ? &sh : cluster.map_shared_rank(&sh, 0);
    root->rmin[rank] = m0;
    root->rmax[rank] = m1;
  }
  if (ONE) {
    __syncthreads();
  } else {
    cluster.sync();  // every slice and range is in CTA 0
    if (rank != 0) return;
  }
  float smin = INFINITY, smax = -INFINITY;
  for (int r = 0; r < CL; r++) {
    smin = fminf(smin, sh.rmin[r]);
    smax = fmaxf(smax, sh.rmax[r]);
  }
  __syncthreads();  // sh.red is reused by the selection
  select_in_shared<T, true>(a, sh, cache, cluster, 1, 0, qh, Nb, out, aout, 0, t, smin, smax);
}

// Cluster size and slice length: one CTA holds up to SELECT_SLICE_ONE logits;
// longer caches spread a head over 2..8 CTAs. (Splitting shorter caches to
// fill the GPU costs more in cluster barriers than it saves.)
static void select_geometry(const KVView& kv, int sms, int* cl, int* chunk) {
  const int tmax = kv.t_max;
  int c = 1;
  if (tmax > SELECT_SLICE_ONE) {
    c = 2;
    while (c < 8 && (tmax + c - 1) / c > SELECT_SLICE_MAX) c *= 2;
  }
  (void)sms;
  *cl = c;
  *chunk = ((tmax + c - 1) / c + 3) / 4 * 4;
}

// One cluster of cl CTAs per query head, smem bytes of dynamic shared memory each.
cudaError_t launch_select_grid(void (*k)(const SelectLaunch, int), const SelectLaunch& a, int cl,
                               int chunk, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (cl > 8) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const int U = a.kv.B * a.kv.Hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(U * cl);
  cfg.blockDim = dim3(SEL_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = cl == 1 ? attr + 1 : attr;  // no cluster attribute for a single CTA
  cfg.numAttrs = (cl == 1 ? 0 : 1) + (a.kv.pdl ? 1 : 0);
  return cudaLaunchKernelEx(&cfg, k, a, chunk);
}

cudaError_t launch_select(const SelectLaunch& a, cudaStream_t st) {
  int sms = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int cl = 1, chunk = 0;
  select_geometry(a.kv, sms, &cl, &chunk);
  if (chunk > (cl == 1 ? SELECT_SLICE_ONE : SELECT_SLICE_MAX)) return launch_select_global(a, st);
  void (*k)(const SelectLaunch, int);
  if (a.kv.dtype == PRHS_BF16)
    k = cl == 1 ? select_cluster_kernel<__nv_bfloat16, true> : select_cluster_kernel<__nv_bfloat16, false>;
  else
    k = cl == 1 ? select_cluster_kernel<float, true> : select_cluster_kernel<float, false>;
  return launch_select_grid(k, a, cl, chunk, (size_t)chunk * sizeof(float), st);
}

// Score-and-select geometry: the fewest CTAs (a power of two up to
// SELECT_FUSED_CL) whose slices hold at most SELECT_FUSED_ROWS keys each, or
// SELECT_FUSED_CL CTAs of up to SELECT_FUSED_MAX_ROWS.
bool score_select_geometry(const KVView& kv, int* cl, int* chunk) {
  int c = 1;
  while (c < SELECT_FUSED_CL && (kv.t_max + c - 1) / c > SELECT_FUSED_ROWS) c *= 2;
  if ((kv.t_max + c - 1) / c > SELECT_FUSED_MAX_ROWS) return false;
  *cl = c;
  *chunk = ((kv.t_max + c - 1) / c + 3) / 4 * 4;
  return true;
}

bool score_select_fits(const KVView& kv) {
  int cl, chunk;
  return (kv.d == 64 || kv.d == 128) && score_select_geometry(kv, &cl, &chunk);
}

template <typename T, int DK>
static cudaError_t score_select_dispatch_d(const SelectLaunch& a, int cl, int chunk, cudaStream_t st) {
  void (*k)(const SelectLaunch, int) =
      cl == 1 ? score_select_kernel<T, DK, true> : score_select_kernel<T, DK, false>;
  // CTA 0 holds the whole row of logits
  return launch_select_grid(k, a, cl, chunk, (size_t)a.kv.t_max * sizeof(float), st);
}

template <typename T>
static cudaError_t score_select_dispatch(const SelectLaunch& a, int cl, int chunk, cudaStream_t st) {
  if (a.kv.d == 128) return score_select_dispatch_d<T, 128>(a, cl, chunk, st);
  if (a.kv.d == 64) return score_select_dispatch_d<T, 64>(a, cl, chunk, st);
  return cudaErrorNotSupported;
}

cudaError_t launch_score_select(const SelectLaunch& a, cudaStream_t st) {
  int cl = 1, chunk = 0;
  if (!score_select_geometry(a.kv, &cl, &chunk)) return cudaErrorNotSupported;
  if (a.out != nullptr) return launch_retrieve(a, st);
  return a.kv.dtype == PRHS_BF16 ? score_select_dispatch<__nv_bfloat16>(a, cl, chunk, st)
                                 : score_select_dispatch<float>(a, cl, chunk, st);
}

}  // namespace prhs
