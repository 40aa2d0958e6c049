// Dropped attention mass of a given index set under the current query: a
// diagnostic for reuse steps, whose attended set was not selected under this
// query. "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context
// Inference": abstract (the attention mass of discarded entries) and Table I
// (tau(.) retained and delta(.) = 1 - tau(.) dropped mass).
//
// One CTA per query head over the logits prhs_score left in the workspace:
// m = max_i s_i and Z = sum_i exp(s_i - m) over [0, t_b), kept = sum over the
// set's entries of exp(s_i - m), delta = (Z - kept) / Z. An entry outside
// [0, t_b) or not above its predecessor is flagged and skipped.
#include "kernels.h"

namespace prhs {

constexpr int MASS_THREADS = 256;

__global__ void __launch_bounds__(MASS_THREADS) mass_kernel(const MassLaunch a) {
  __shared__ float red[MASS_THREADS / 32];
  __shared__ float red2[MASS_THREADS / 32];
  pdl_wait();
  pdl_trigger();
  const KVView& kv = a.kv;
  const int qh = blockIdx.x, b = qh / kv.Hq;
  if (a.head_skip != nullptr && a.head_skip[qh] != 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = seq_len(kv, b);
  const float* s = a.scores + (long long)qh * kv.t_max;
  int n = a.n_sel[qh];
  if (n < 0 || n > a.cap) {
    if (tid == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    n = n < 0 ? 0 : a.cap;
  }
  float mx = -INFINITY;
  for (int i = tid; i < t; i += MASS_THREADS) mx = fmaxf(mx, s[i]);
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < MASS_THREADS / 32; w++) m = fmaxf(m, red[w]);
  float z = 0.f, kept = 0.f;
  if (m != -INFINITY) {
    for (int i = tid; i < t; i += MASS_THREADS) z += expf(s[i] - m);
    const int32_t* row = a.idx + (long long)qh * a.cap;
    for (int j = tid; j < n; j += MASS_THREADS) {
      const int i = row[j];
      const int prev = j > 0 ? row[j - 1] : -1;
      if (i < 0 || i >= t || i <= prev) {
        raise_error(kv.err, PRHS_DEV_BAD_INDEX);
        continue;
      }
      kept += expf(s[i] - m);
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
    a.delta[qh] = Z > 0.f ? fmaxf(0.f, (Z - K) / Z) : (t == 0 ? 0.f : 1.f);
  }
}

cudaError_t launch_mass(const MassLaunch& a, cudaStream_t st) {
  return launch_pdl(mass_kernel, dim3(a.kv.B * a.kv.Hq), dim3(MASS_THREADS), 0, st, a);
}

}  // namespace prhs
