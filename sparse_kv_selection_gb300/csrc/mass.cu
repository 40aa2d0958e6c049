// Dropped attention mass of a given index set under the current query: a
// diagnostic for reuse steps, whose attended set was not selected under this
// query, and the delta of a retrieving head when keys are forced into its
// set. "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context
// Inference": abstract (the attention mass of discarded entries) and Table I
// (tau(.) retained and delta(.) = 1 - tau(.) dropped mass).
//
// Over the logits prhs_score left in the workspace, CTA (u, p) of a head
// takes keys [p*chunk, (p+1)*chunk): m_p = their largest logit, z_p = the sum
// of exp(s_i - m_p) and k_p the same sum over the set's entries in that range.
// With one part it writes delta = (z - k) / z; with more, it stores (m_p, z_p,
// k_p) and the last part to arrive (atomic ticket) rescales them to the
// overall maximum, writes delta and resets the ticket. An entry outside
// [0, t_b) or not above its predecessor is flagged and skipped.
#include "kernels.h"

namespace prhs {

constexpr int MASS_THREADS = 256;

__global__ void __launch_bounds__(MASS_THREADS) mass_kernel(const MassLaunch a) {
  __shared__ float red[MASS_THREADS / 32];
  __shared__ float red2[MASS_THREADS / 32];
  __shared__ int sh_last;
  pdl_wait();
  pdl_trigger();
  const KVView& kv = a.kv;
  const int qh = blockIdx.x, part = blockIdx.y, P = gridDim.y, b = qh / kv.Hq;
  if (a.head_skip != nullptr && a.head_skip[qh] != 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = seq_len(kv, b);
  const int lo = min(t, part * a.chunk), hi = min(t, lo + a.chunk);
  const float* s = a.scores + (long long)qh * kv.t_max;
  int n = a.n_sel[qh];
  if (n < 0 || n > a.cap) {
    if (tid == 0 && part == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    n = n < 0 ? 0 : a.cap;
  }
  float mx = -INFINITY;
  for (int i = lo + tid; i < hi; i += MASS_THREADS) mx = fmaxf(mx, s[i]);
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < MASS_THREADS / 32; w++) m = fmaxf(m, red[w]);
  float z = 0.f, kept = 0.f;
  if (m != -INFINITY) {
    for (int i = lo + tid; i < hi; i += MASS_THREADS) z += expf(s[i] - m);
    const int32_t* row = a.idx + (long long)qh * a.cap;
    for (int j = tid; j < n; j += MASS_THREADS) {
      const int i = row[j];
      const int prev = j > 0 ? row[j - 1] : -1;
      if (i < 0 || i >= t || i <= prev) {
        if (part == 0) raise_error(kv.err, PRHS_DEV_BAD_INDEX);
        continue;
      }
      if (i >= lo && i < hi) kept += expf(s[i] - m);
    }
  }
  z = warp_sum(z);
  kept = warp_sum(kept);
  __syncthreads();  // red is reused
  if (lane == 0) {
    red[warp] = z;
    red2[warp] = kept;
  }
  __syncthreads();
  if (tid == 0) {
    float Z = 0.f, K = 0.f;
    for (int w = 0; w < MASS_THREADS / 32; w++) {
      Z += red[w];
      K += red2[w];
    }
    if (P == 1) {
      a.delta[qh] = Z > 0.f ? fmaxf(0.f, (Z - K) / Z) : (t == 0 ? 0.f : 1.f);
      return;
    }
    float* rec = a.partials + ((long long)qh * P + part) * 4;
    rec[0] = m;
    rec[1] = Z;
    rec[2] = K;
    __threadfence();
    sh_last = atomicAdd(&a.counters[qh], 1u) == (unsigned)(P - 1);
    if (sh_last) {
      __threadfence();
      const float* r0 = a.partials + (long long)qh * P * 4;
      float M = -INFINITY;
      for (int p = 0; p < P; p++) M = fmaxf(M, __ldcg(r0 + p * 4));
      float Zt = 0.f, Kt = 0.f;
      if (M != -INFINITY)
        for (int p = 0; p < P; p++) {
          const float c = expf(__ldcg(r0 + p * 4) - M);
          Zt += c * __ldcg(r0 + p * 4 + 1);
          Kt += c * __ldcg(r0 + p * 4 + 2);
        }
      a.delta[qh] = Zt > 0.f ? fmaxf(0.f, (Zt - Kt) / Zt) : (t == 0 ? 0.f : 1.f);
      a.counters[qh] = 0u;
    }
  }
}

int mass_parts(int t_max) {
  const int p = (t_max + MASS_CHUNK - 1) / MASS_CHUNK;
  return p < 1 ? 1 : (p > MASS_PARTS_MAX ? MASS_PARTS_MAX : p);
}

cudaError_t launch_mass(const MassLaunch& a, cudaStream_t st) {
  const int P = mass_parts(a.kv.t_max);
  MassLaunch m = a;
  m.chunk = (a.kv.t_max + P - 1) / P;
  if (P > 1 && (a.partials == nullptr || a.counters == nullptr)) return cudaErrorInvalidValue;
  return launch_pdl(mass_kernel, dim3(a.kv.B * a.kv.Hq, P), dim3(MASS_THREADS), 0, st, a.kv.pdl, m);
}

}  // namespace prhs
