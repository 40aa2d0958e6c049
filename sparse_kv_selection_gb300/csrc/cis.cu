// Critical-index-set (CIS) reuse with dilation.
// "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference":
// Fig. 2 (adjacent queries with cosine similarity above 0.8 share critical
// indices), Fig. 8 (sharing triggers when sim(q, q') >= tau), Fig. 4 and
// Table VIII (the shared set is dilated; radius r), and the CIS block size s
// of Tables IV, V and VIII read as a bound on consecutive reuses.
//
// One CTA per query head. The gate takes the decision of the float64 formula
// c = <q, q_a> / (sqrt(|q|^2) sqrt(|q_a|^2)) >= tau. Its first warp forms the
// three sums in fp32 (bf16 products are exact in fp32; tree sums of d <= 128
// terms stay within 8 roundings, so the fp32 cosine is within about 2e-6 of
// the exact one) and decides from them when that cosine lies farther than
// CIS_MARGIN = 1e-4 from tau; otherwise, or when a sum is not finite or a norm
// is tiny, the same warp recomputes the sums and the ratio in float64. fp64 is
// slow on this part, so the common case avoids it. The dilated set
//   union_{a in anchor} [a - w, a + w] clipped to [0, t_b)
// is produced without sorting: the anchor row is ascending, so interval j
// contributes the positions after max(lo_j, hi_{j-1} + 1); a block-wide
// exclusive scan of those counts gives every write position directly and the
// output comes out ascending and free of repeats.
#include "kernels.h"

namespace prhs {

constexpr int CIS_THREADS = 256;

__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}

constexpr int CIS_PER = 4;  // anchor entries per thread per chunk
constexpr float CIS_MARGIN = 1e-4f;

template <typename T>
__global__ void __launch_bounds__(CIS_THREADS) cis_kernel(const CisLaunch a) {
  __shared__ int sh_reuse;
  __shared__ int warp_tot[CIS_THREADS / 32];
  pdl_wait();
  pdl_trigger();
  const KVView& kv = a.kv;
  const int qh = blockIdx.x;
  const int b = qh / kv.Hq;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d = kv.d;
  constexpr int CHUNK = CIS_THREADS * CIS_PER;

  // every input of the first chunk is requested before any result is used:
  // the anchor row is read up to its capacity, whatever anchor_n turns out
  // to be, and the entries past anchor_n are ignored below
  int n = a.anchor_n[qh];
  const int age = a.anchor_age != nullptr ? a.anchor_age[qh] : 0;
  const int t = seq_len(kv, b);
  const int32_t* anc = a.anchor_idx + (long long)qh * a.anchor_cap;
  int x[CIS_PER];
  int prev0;
  {
    const int j0 = tid * CIS_PER;
#pragma unroll
    for (int k = 0; k < CIS_PER; k++) x[k] = j0 + k < a.anchor_cap ? anc[j0 + k] : 0;
    prev0 = j0 > 0 && j0 - 1 < a.anchor_cap ? anc[j0 - 1] : -1;
  }
  if (warp == 0) {
    float df = 0.f, qq = 0.f, aa = 0.f;
    for (int i = lane; i < d; i += 32) {
      const float u = Elem<T>::load1(a.q, (long long)qh * d + i);
      const float v = Elem<T>::load1(a.q_anchor, (long long)qh * d + i);
      df = fmaf(u, v, df);
      qq = fmaf(u, u, qq);
      aa = fmaf(v, v, aa);
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
    if (pass < 0) {  // near the threshold: the float64 formula
      double dot = 0.0, nq = 0.0, na = 0.0;
      for (int i = lane; i < d; i += 32) {
        const double u = (double)Elem<T>::load1(a.q, (long long)qh * d + i);
        const double v = (double)Elem<T>::load1(a.q_anchor, (long long)qh * d + i);
        dot = fma(u, v, dot);
        nq = fma(u, u, nq);
        na = fma(v, v, na);
      }
      dot = warp_sum_f64(dot);
      nq = warp_sum_f64(nq);
      na = warp_sum_f64(na);
      const double den = sqrt(nq) * sqrt(na);
      pass = den > 0.0 && dot / den >= a.tau;
    }
    if (lane == 0) {
      const int reuse = n > 0 && pass && (a.max_run <= 0 || age < a.max_run - 1);
      sh_reuse = reuse;
      a.reuse[qh] = (uint8_t)reuse;
      if (a.anchor_age != nullptr) a.anchor_age[qh] = reuse ? age + 1 : 0;
    }
  }
  __syncthreads();
  if (!sh_reuse) return;

  // ---- dilation of the anchor set: CIS_PER consecutive entries per thread ----
  if (n > a.anchor_cap) {
    if (tid == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    n = a.anchor_cap;
  }
  int32_t* out = a.idx + (long long)qh * a.cap;
  const int w = a.w;
  // forced keys: sinks [0, ns) first, the window after the dilated entries
  const int ns = min(max(a.n_sink, 0), t);
  for (int i = tid; i < ns; i += CIS_THREADS) {
    if (i < a.cap) out[i] = i;
    else raise_error(kv.err, PRHS_DEV_CAPACITY);
  }
  int carry = ns;
  for (int base = 0; base < n; base += CHUNK) {
    const int j0 = base + tid * CIS_PER;
    if (base > 0) {
#pragma unroll
      for (int k = 0; k < CIS_PER; k++) x[k] = j0 + k < n ? anc[j0 + k] : 0;
      prev0 = j0 - 1 < n ? anc[j0 - 1] : -1;
    }
    int start[CIS_PER], cnt[CIS_PER];
    int local = 0;
    int prev = prev0;
#pragma unroll
    for (int k = 0; k < CIS_PER; k++) {
      start[k] = 0;
      cnt[k] = 0;
      if (j0 + k < n) {
        const int xv = x[k];
        if (xv < 0 || xv >= t || xv <= prev) {
          raise_error(kv.err, PRHS_DEV_BAD_INDEX);
        } else {
          const int lo = max(0, xv - w);
          const int hi = min(t - 1, xv + w);
          const int prev_hi = max(ns - 1, j0 + k > 0 ? min(t - 1, prev + w) : -1);
          start[k] = max(lo, prev_hi + 1);
          cnt[k] = max(0, hi - start[k] + 1);
        }
        prev = xv;
      }
      local += cnt[k];
    }
    // block exclusive scan of the per-thread counts
    int v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w2 = 0; w2 < CIS_THREADS / 32; w2++) {
      before += w2 < warp ? warp_tot[w2] : 0;
      total += warp_tot[w2];
    }
    int pos = carry + before + v - local;
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
    carry += total;
    if (base + CHUNK < n) __syncthreads();  // warp_tot is reused by the next chunk
  }
  // the window: past both the sinks and the last dilated interval
  int last = ns - 1;
  if (n > 0) {
    const int xl = anc[n - 1];
    if (xl >= 0 && xl < t) last = max(last, min(t - 1, xl + w));
  }
  const int wstart = max(max(ns, t - max(a.window, 0)), last + 1);
  for (int i = tid; i < t - wstart; i += CIS_THREADS) {
    if (carry + i < a.cap) out[carry + i] = wstart + i;
    else raise_error(kv.err, PRHS_DEV_CAPACITY);
  }
  carry += max(0, t - wstart);
  if (tid == 0) a.n_sel[qh] = min(carry, a.cap);
}

cudaError_t launch_cis(const CisLaunch& a, cudaStream_t st) {
  void (*k)(const CisLaunch) = a.kv.dtype == PRHS_BF16 ? cis_kernel<__nv_bfloat16> : cis_kernel<float>;
  return launch_pdl(k, dim3(a.kv.B * a.kv.Hq), dim3(CIS_THREADS), 0, st, a.kv.pdl, a);
}

}  // namespace prhs
