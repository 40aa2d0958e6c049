// Critical-index-set (CIS) reuse with dilation.
// "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference":
// Fig. 2 (adjacent queries with cosine similarity above 0.8 share critical
// indices), Fig. 8 (sharing triggers when sim(q, q') >= tau), Fig. 4 and
// Table VIII (the shared set is dilated; radius r), and the CIS block size s
// of Tables IV, V and VIII read as a bound on consecutive reuses.
//
// One CTA per query head. The gate takes the decision of the float64 formula
// c = <q, q_a> / (sqrt(|q|^2) sqrt(|q_a|^2)) >= tau. Its first warp forms the
// three sums in fp32 (on bf16 caches the products are exact in fp32, on fp32
// ones each adds one rounding; tree sums of d <= 128 terms stay within 8
// roundings, so the fp32 cosine is within a few 1e-6 of the exact one, far
// inside the margin) and decides from them when that cosine lies farther than
// CIS_MARGIN = 1e-4 from tau; otherwise, or when a sum is not finite or a norm
// is tiny, the same warp recomputes the sums and the ratio in float64. fp64 is
// slow on this part, so the common case avoids it. The dilated set
//   union_{a in anchor} [a - w, a + w] clipped to [0, t_b)
// is produced without sorting: the anchor row is ascending, so interval j
// contributes the positions after max(lo_j, hi_{j-1} + 1); a block-wide
// exclusive scan of those counts gives every write position directly and the
// output comes out ascending and free of repeats.
#include <cooperative_groups.h>

#include "kernels.h"

namespace cg = cooperative_groups;

namespace prhs {

constexpr int CIS_THREADS = 256;
constexpr int CIS_CLUSTER_MAX = 8;  // CTAs per head at most

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}

constexpr int CIS_PER = 4;  // anchor entries per thread per chunk
// Dilated positions of one chunk staged in dynamic shared memory before they
// are written: room for CIS_THREADS * CIS_PER anchor entries of 2w + 1
// positions each, at most CIS_STAGE_MAX (a chunk with more positions, w > 4,
// is written directly). Sized by w so that short radii leave room for more
// CTAs per SM.
constexpr int CIS_STAGE_MAX = CIS_THREADS * CIS_PER * 9;
__host__ __device__ __forceinline__ int cis_stage(int w, int n_den) {
  if (n_den > 0) return 0;  // budgeted dilation writes directly
  const long long s = (long long)CIS_THREADS * CIS_PER * (2ll * (w < 0 ? 0 : w) + 1);
  return s < CIS_STAGE_MAX ? (int)s : CIS_STAGE_MAX;
}
constexpr float CIS_MARGIN = 1e-4f;

// Block-wide sum (all CIS_THREADS threads call it; `tot` is shared scratch
// of CIS_THREADS / 32 ints, free again on return).
__device__ __forceinline__ int block_sum(int v, int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  if (lane == 0) tot[warp] = v;
  __syncthreads();
  int s = 0;
#pragma unroll
  for (int w2 = 0; w2 < CIS_THREADS / 32; w2++) s += tot[w2];
  __syncthreads();
  return s;
}

// Block-wide exclusive scan; *total gets the sum. Same calling rules.
__device__ __forceinline__ int block_excl_scan(int v, int* tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL_MASK, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tot[warp] = x;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w2 = 0; w2 < CIS_THREADS / 32; w2++) {
    before += w2 < warp ? tot[w2] : 0;
    all += tot[w2];
  }
  __syncthreads();
  *total = all;
  return before + x - v;
}

// Budgeted dilation (Fig. 9a: dilation strength m = floor(k / n_den)): the
// anchor set and at most m of its +-w neighbours, nearest first, the lowest
// position first at equal distance; forced sinks before and the window after,
// as in the unbounded rule. Unit j of the anchor row (ascending x_j) owns the
// neighbours between x_{j-1} and x_j (those of the first anchor below it; the
// last unit also those above the last anchor). A candidate p of unit j lies
// at distance min(p - x_{j-1}, x_j - p) (x_j - p for j = 0, p - x_last above
// the last anchor). Pass 1 finds the distance D at which the budget runs out
// (C(d), the candidates within d, for d = 1, 2, ...) and how many of the
// candidates at exactly D fit; pass 2 writes, unit by unit, the gap's chosen
// candidates, the anchor and (last unit) the chosen candidates above it, with
// every write position from a block scan.
__device__ void dilate_budgeted(const CisLaunch& a, const int32_t* anc, int n, int t, int ns,
                                int32_t* out, int qh, int* tot) {
  const KVView& kv = a.kv;
  const int w = a.w, tid = threadIdx.x;
  // the anchor row must be ascending inside [0, t): otherwise it is flagged
  // and the head attends its forced keys only
  {
    int bad = 0;
    for (int j = tid; j < n; j += CIS_THREADS) {
      const int x = anc[j];
      bad += x < 0 || x >= t || (j > 0 && anc[j - 1] >= x);
    }
    if (block_sum(bad, tot) > 0) {
      if (tid == 0) raise_error(kv.err, PRHS_DEV_BAD_INDEX);
      n = 0;
    }
  }
  const int m = n / a.n_den;
  const int wlo = max(ns, t - max(a.window, 0));  // the forced window [wlo, t)
  // candidates of unit j within distance d of the anchors
  auto unit_within = [&](int j, int d) {
    const int x = anc[j];
    int c;
    if (j == 0) {
      c = min(d, x);
    } else {
      const int g = x - anc[j - 1] - 1;
      c = min(g, 2 * d);
    }
    if (j == n - 1) c += min(d, t - 1 - x);
    return c;
  };
  // ---- pass 1: the cut distance D and the candidates taken at exactly D ----
  int D = 0, take_at_D = 0, below = 0;  // below = C(D - 1)
  if (m > 0) {
    for (int d = 1; d <= w; d++) {
      int loc = 0;
      for (int j = tid; j < n; j += CIS_THREADS) loc += unit_within(j, d);
      const int cd = block_sum(loc, tot);
      D = d;
      take_at_D = min(m, cd) - below;
      if (cd >= m) break;
      below = cd;
    }
  }
  // ---- pass 2: write ----
  for (int i = tid; i < ns; i += CIS_THREADS) {
    if (i < a.cap) out[i] = i;
    else raise_error(kv.err, PRHS_DEV_CAPACITY);
  }
  int carry = ns, rank0 = 0;  // entries written so far; candidates at distance D in earlier chunks
  for (int base = 0; base < n; base += CIS_THREADS) {
    const int j = base + tid;
    const bool has = j < n;
    const int x = has ? anc[j] : 0;
    const bool first = j == 0;
    const int xp = has && !first ? anc[j - 1] : 0;
    // the unit's candidates, ascending: [lo1, hi1] near x_{j-1}, [lo2, x - 1]
    // near x_j, and for the last unit [x + 1, hi3] above it
    const int lo1 = xp + 1, hi1 = first ? xp : min(xp + w, x - 1);
    const int lo2 = max(first ? x - w : max(hi1 + 1, x - w), 0);
    const int hi3 = has && j == n - 1 ? min(t - 1, x + w) : x;
    auto dist = [&](int p) { return p > x ? p - x : (first ? x - p : min(p - xp, x - p)); };
    int atD = 0;
    if (has && D > 0) {
      for (int p = lo1; p <= hi1; p++) atD += dist(p) == D;
      for (int p = lo2; p < x; p++) atD += dist(p) == D;
      for (int p = x + 1; p <= hi3; p++) atD += dist(p) == D;
    }
    int at_total;
    const int rank_first = rank0 + block_excl_scan(atD, tot, &at_total);
    // a candidate is kept if nearer than D, or at D within the budget's
    // remainder (rank counted over all candidates at D, ascending); kept
    // positions among the sinks or in the window are written with them
    auto keep = [&](int p, int& rank) {
      const int dd = dist(p);
      const bool c = dd < D || (dd == D && rank++ < take_at_D);
      return c && p >= ns && p < wlo;
    };
    int k = 0;
    if (has) {
      int rank = rank_first;
      for (int p = lo1; p <= hi1; p++) k += keep(p, rank);
      for (int p = lo2; p < x; p++) k += keep(p, rank);
      k += x >= ns && x < wlo;
      for (int p = x + 1; p <= hi3; p++) k += keep(p, rank);
    }
    int total;
    int pos = carry + block_excl_scan(k, tot, &total);
    if (has) {
      int rank = rank_first;
      auto emit = [&](int p) {
        if (pos < a.cap) out[pos] = p;
        else raise_error(kv.err, PRHS_DEV_CAPACITY);
        pos++;
      };
      for (int p = lo1; p <= hi1; p++) if (keep(p, rank)) emit(p);
      for (int p = lo2; p < x; p++) if (keep(p, rank)) emit(p);
      if (x >= ns && x < wlo) emit(x);
      for (int p = x + 1; p <= hi3; p++) if (keep(p, rank)) emit(p);
    }
    carry += total;
    rank0 += at_total;
  }
  // the window, whole: kept positions stop below it
  for (int i = tid; i < t - wlo; i += CIS_THREADS) {
    if (carry + i < a.cap) out[carry + i] = wlo + i;
    else raise_error(kv.err, PRHS_DEV_CAPACITY);
  }
  carry += t - wlo;
  if (tid == 0) a.n_sel[qh] = min(carry, a.cap);
}

// Intervals of the anchor entries j0 .. j0 + CIS_PER - 1 below `end` (x: their
// positions, prev: the entry before j0, -1 for the first): entry j adds the
// positions from max(x_j - w, the previous interval's end + 1, ns) to
// min(x_j + w, wlo - 1), the forced sinks [0, ns) and window [wlo, t) being
// written whole beside them. Returns their count; err (null: not checked)
// gets PRHS_DEV_BAD_INDEX for an entry outside [0, t) or not ascending.
__device__ __forceinline__ int chunk_intervals(const int* x, int prev, int j0, int end, int t, int w,
                                               int ns, int wlo, unsigned* err, int* start, int* cnt) {
  int local = 0;
#pragma unroll
  for (int k = 0; k < CIS_PER; k++) {
    start[k] = 0;
    cnt[k] = 0;
    if (j0 + k < end) {
      const int xv = x[k];
      if (xv < 0 || xv >= t || xv <= prev) {
        if (err != nullptr) raise_error(err, PRHS_DEV_BAD_INDEX);
      } else {
        const int lo = max(0, xv - w);
        const int hi = min(min(t - 1, xv + w), wlo - 1);
        const int prev_hi = max(ns - 1, j0 + k > 0 ? min(t - 1, prev + w) : -1);
        start[k] = max(lo, prev_hi + 1);
        cnt[k] = max(0, hi - start[k] + 1);
      }
      prev = xv;
    }
    local += cnt[k];
  }
  return local;
}

// One CTA per query head, or (CLU) a cluster of CL CTAs per head when heads
// are few and anchor rows long: CTA r then dilates the anchor entries
// [r * seg, (r + 1) * seg), after one round in which every CTA counts its
// segment's positions and writes the count into every CTA's shared memory, so
// each knows where its part of the ascending output starts.
template <typename T, bool CLU>
__global__ void __launch_bounds__(CIS_THREADS) cis_kernel(const CisLaunch a) {
  __shared__ int sh_reuse;
  __shared__ int warp_tot[CIS_THREADS / 32];
  __shared__ int seg_cnt[CIS_CLUSTER_MAX];  // CLU: every rank's count of dilated positions
  extern __shared__ int stage[];            // one chunk's dilated positions (cis_stage ints)
  cg::cluster_group cluster = cg::this_cluster();
  const int CL = CLU ? (int)cluster.num_blocks() : 1;
  const int rank = CLU ? (int)cluster.block_rank() : 0;
  pdl_wait();
  pdl_trigger();
  const KVView& kv = a.kv;
  const int qh = blockIdx.x / CL;
  const int b = qh / kv.Hq;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = kv.d;
  constexpr int CHUNK = CIS_THREADS * CIS_PER;
  constexpr int EPC = Elem<T>::per16;

  // every input of the first chunk is requested before any result is used:
  // the anchor row is read up to this CTA's part of its capacity, whatever
  // anchor_n turns out to be, and the entries past anchor_n are ignored below
  int n = a.anchor_n[qh];
  const int age = a.anchor_age != nullptr ? a.anchor_age[qh] : 0;
  const int t = seq_len(kv, b);
  const int32_t* anc = a.anchor_idx + (long long)qh * a.anchor_cap;
  const int seg = (a.anchor_cap + CL - 1) / CL;
  const int seg_lo = rank * seg, seg_cap_hi = min(a.anchor_cap, seg_lo + seg);
  int x[CIS_PER];
  int prev0;
  {
    const int j0 = seg_lo + tid * CIS_PER;
#pragma unroll
    for (int k = 0; k < CIS_PER; k++) x[k] = j0 + k < seg_cap_hi ? anc[j0 + k] : 0;
    prev0 = j0 > 0 && j0 - 1 < a.anchor_cap ? anc[j0 - 1] : -1;
  }
  if (warp == 0) {
    // the gated vectors in 16-byte pieces, one round trip: lanes below d / EPC
    // hold EPC elements each of g and of the anchor's copy
    float u[EPC], v[EPC];
    const int lpr = d / EPC;
    if (lane < lpr) {
      const uint4 ru = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.q) +
                                                            (long long)qh * d * sizeof(T)) + lane);
      const uint4 rv = __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.q_anchor) +
                                                            (long long)qh * d * sizeof(T)) + lane);
      Elem<T>::unpack(ru, u);
      Elem<T>::unpack(rv, v);
    } else {
#pragma unroll
      for (int e = 0; e < EPC; e++) u[e] = v[e] = 0.f;
    }
    float df = 0.f, qq = 0.f, aa = 0.f;
#pragma unroll
    for (int e = 0; e < EPC; e++) {
      df = fmaf(u[e], v[e], df);
      qq = fmaf(u[e], u[e], qq);
      aa = fmaf(v[e], v[e], aa);
    }
    df = warp_sum(df);
    qq = warp_sum(qq);
    aa = warp_sum(aa);
    int pass = -1;  // -1: not decided in fp32
    if (isfinite(df) && isfinite(qq) && isfinite(aa) && qq > 1e-30f && aa > 1e-30f) {
      const float c = df * rsqrtf(qq) * rsqrtf(aa);
      const float tf = (float)a.tau;
      if (fabsf(c - tf) > CIS_MARGIN) pass = c > tf;
    }
    pass = __shfl_sync(FULL_MASK, pass, 0);  // one decision for the warp
    if (pass < 0) {  // near the threshold: the float64 formula, from the same elements
      double dot = 0.0, nq = 0.0, na = 0.0;
#pragma unroll
      for (int e = 0; e < EPC; e++) {
        dot = fma((double)u[e], (double)v[e], dot);
        nq = fma((double)u[e], (double)u[e], nq);
        na = fma((double)v[e], (double)v[e], na);
      }
      dot = warp_sum_f64(dot);
      nq = warp_sum_f64(nq);
      na = warp_sum_f64(na);
      const double den = sqrt(nq) * sqrt(na);
      pass = den > 0.0 && dot / den >= a.tau;
    }
    if (lane == 0) {  // every rank takes the same decision; rank 0 records it
      const int reuse = n > 0 && pass && (a.max_run <= 0 || age < a.max_run - 1);
      sh_reuse = reuse;
      if (rank == 0) {
        a.reuse[qh] = (uint8_t)reuse;
        if (a.anchor_age != nullptr) a.anchor_age[qh] = reuse ? age + 1 : 0;
      }
    }
  }
  __syncthreads();
  if (!sh_reuse) return;  // uniform over the cluster

  // ---- dilation of the anchor set: CIS_PER consecutive entries per thread ----
  if (n > a.anchor_cap) {
    if (tid == 0 && rank == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    n = a.anchor_cap;
  }
  int32_t* out = a.idx + (long long)qh * a.cap;
  const int w = a.w;
  // forced keys: sinks [0, ns) first, the window after the dilated entries
  const int ns = min(max(a.n_sink, 0), t);
  const int wlo = max(ns, t - max(a.window, 0));  // the window [wlo, t)
  if (a.n_den > 0) {  // uniform over the block; the launch gives it one CTA per head
    dilate_budgeted(a, anc, n, t, ns, out, qh, warp_tot);
    return;
  }
  const int seg_hi = min(n, seg_lo + seg);  // this CTA's entries [seg_lo, seg_hi)
  int offset = 0, grand = 0;                // positions of the lower ranks' entries, of all
  if (CLU) {
    int local = 0;
    for (int base = seg_lo; base < seg_hi; base += CHUNK) {
      const int j0 = base + tid * CIS_PER;
      int y[CIS_PER], prev = prev0;
      if (base == seg_lo) {
#pragma unroll
        for (int k = 0; k < CIS_PER; k++) y[k] = x[k];
      } else {
#pragma unroll
        for (int k = 0; k < CIS_PER; k++) y[k] = j0 + k < seg_hi ? anc[j0 + k] : 0;
        prev = j0 - 1 < seg_hi ? anc[j0 - 1] : -1;
      }
      int start[CIS_PER], cnt[CIS_PER];
      local += chunk_intervals(y, prev, j0, seg_hi, t, w, ns, wlo, nullptr, start, cnt);
    }
    const int total = block_sum(local, warp_tot);
    if (tid < CL) cluster.map_shared_rank(seg_cnt, tid)[rank] = total;
    cluster.sync();  // every rank's count is in every rank
#pragma unroll
    for (int r = 0; r < CIS_CLUSTER_MAX; r++) {
      const int c = r < CL ? seg_cnt[r] : 0;
      offset += r < rank ? c : 0;
      grand += c;
    }
  }
  if (rank == 0)
    for (int i = tid; i < ns; i += CIS_THREADS) {
      if (i < a.cap) out[i] = i;
      else raise_error(kv.err, PRHS_DEV_CAPACITY);
    }
  int carry = ns + offset;
  for (int base = seg_lo; base < seg_hi; base += CHUNK) {
    const int j0 = base + tid * CIS_PER;
    if (base > seg_lo) {
#pragma unroll
      for (int k = 0; k < CIS_PER; k++) x[k] = j0 + k < seg_hi ? anc[j0 + k] : 0;
      prev0 = j0 - 1 < seg_hi ? anc[j0 - 1] : -1;
    }
    int start[CIS_PER], cnt[CIS_PER];
    const int local = chunk_intervals(x, prev0, j0, seg_hi, t, w, ns, wlo, kv.err, start, cnt);
    int total;
    int pos = carry + block_excl_scan(local, warp_tot, &total);
    if (total <= cis_stage(w, a.n_den)) {
      // the chunk's positions are laid out in shared memory, then written
      // by consecutive threads (each thread's runs written directly would
      // scatter every warp store over several times the bytes it carries)
      int lp = pos - carry;
#pragma unroll
      for (int k = 0; k < CIS_PER; k++)
        for (int e = 0; e < cnt[k]; e++) stage[lp++] = start[k] + e;
      __syncthreads();
      const int room = max(0, min(total, a.cap - carry));
      for (int i = tid; i < room; i += CIS_THREADS) out[carry + i] = stage[i];
      if (tid == 0 && room < total) raise_error(kv.err, PRHS_DEV_CAPACITY);
      __syncthreads();  // the stage is free for the next chunk
    } else {
#pragma unroll
      for (int k = 0; k < CIS_PER; k++) {
        for (int e = 0; e < cnt[k]; e++) {
          if (pos + e < a.cap) {
            out[pos + e] = start[k] + e;
          } else {
            raise_error(kv.err, PRHS_DEV_CAPACITY);
            break;
          }
        }
        pos += cnt[k];
      }
    }
    carry += total;
  }
  if (CLU) carry = ns + grand;
  if (rank != 0) return;
  // the window, whole: the dilated intervals stop below it
  for (int i = tid; i < t - wlo; i += CIS_THREADS) {
    if (carry + i < a.cap) out[carry + i] = wlo + i;
    else raise_error(kv.err, PRHS_DEV_CAPACITY);
  }
  carry += t - wlo;
  if (tid == 0) a.n_sel[qh] = min(carry, a.cap);
}

// CTAs per head: a cluster only when the heads are few and the anchor rows
// long (at least 1024 entries per CTA), never for budgeted dilation.
static int cis_cluster(const CisLaunch& a, int sms) {
  if (a.n_den > 0) return 1;
  const long long heads = (long long)a.kv.B * a.kv.Hq;
  int cl = 1;
  while (cl < CIS_CLUSTER_MAX && a.anchor_cap / (cl * 2) >= 1024 && heads * cl * 2 <= 2ll * sms) cl *= 2;
  return cl;
}

template <typename T>
static cudaError_t launch_cis_t(const CisLaunch& a, int cl, cudaStream_t st) {
  void (*k)(const CisLaunch) = cl == 1 ? cis_kernel<T, false> : cis_kernel<T, true>;
  const size_t smem = (size_t)cis_stage(a.w, a.n_den) * sizeof(int);
  if (cl == 1) return launch_pdl(k, dim3(a.kv.B * a.kv.Hq), dim3(CIS_THREADS), smem, st, a.kv.pdl, a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.kv.B * a.kv.Hq * cl);
  cfg.blockDim = dim3(CIS_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.kv.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k, a);
}

cudaError_t launch_cis(const CisLaunch& a, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int cl = cis_cluster(a, sms);
  return a.kv.dtype == PRHS_BF16 ? launch_cis_t<__nv_bfloat16>(a, cl, st) : launch_cis_t<float>(a, cl, st);
}

}  // namespace prhs
