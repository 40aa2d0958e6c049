// Split-K decode attention over a selected index set (sparse) or over the
// whole cache (dense baseline).
// "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference":
// the Table V caption's sparse-attention kernel over the selected KV entries,
// and Table IV's dense ("Flash") operator as the baseline.
//
// Each CTA (4 warps) takes a contiguous slice of one head's rows. Eight lanes
// share a row: lane j reads 16-byte chunks j, j+8, ... of the K and V rows
// (128 contiguous bytes per 8 lanes per load), so every gathered row is read
// with full cache lines. A warp has 4 rows in flight per step and UNROLL steps
// per iteration. Softmax is online in fp32, in base 2 (logits pre-scaled by
// log2 e). The dense kernel computes all G query heads of a KV head from the
// same loaded rows. The last CTA of a head (atomic ticket, no waiting) merges
// the per-CTA partials into out and lse and resets the ticket.
#include "kernels.h"

namespace prhs {

constexpr int ATTN_THREADS = 128;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

template <typename T, int D>
struct AttnShape {
  static constexpr int RB = D * (int)sizeof(T);
  static constexpr int CPR = RB / 16;          // 16-byte chunks per row
  static constexpr int CPL = CPR / 8;          // chunks per lane
  static constexpr int EPC = 16 / (int)sizeof(T);
  static constexpr int EL = CPL * EPC;         // elements per lane
  static_assert(CPR % 8 == 0, "row must be a multiple of 128 bytes");
};

template <typename T, int D, int G, bool SPARSE, int UNROLL>
__global__ void __launch_bounds__(ATTN_THREADS) attn_kernel(const AttnLaunch a) {
  using S = AttnShape<T, D>;
  const KVView& kv = a.kv;
  const int unit = blockIdx.y;  // sparse: b * Hq + h;  dense: b * Hkv + kv head
  const int split = blockIdx.x;
  const int group = kv.Hq / kv.Hkv;
  int b, kvh, qh0;
  if (SPARSE) {
    b = unit / kv.Hq;
    qh0 = unit;
    kvh = (unit % kv.Hq) / group;
  } else {
    b = unit / kv.Hkv;
    kvh = unit % kv.Hkv;
    qh0 = b * kv.Hq + kvh * G;
  }
  const int t = seq_len(kv, b);
  int n;
  const int32_t* rows = nullptr;
  if (SPARSE) {
    n = a.n_sel[unit];
    if (n < 0 || n > a.cap) {
      if (threadIdx.x == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
      n = n < 0 ? 0 : a.cap;
    }
    rows = a.idx + (long long)unit * a.cap;
  } else {
    n = t;
  }
  const int chunk = (n + a.splits - 1) / a.splits;
  const int r0 = min(n, split * chunk);
  const int r1 = min(n, r0 + chunk);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sg = lane >> 3, j = lane & 7;
  const float qscale = a.scale * LOG2E;

  float qf[G][S::EL];
#pragma unroll
  for (int g = 0; g < G; g++)
#pragma unroll
    for (int c = 0; c < S::CPL; c++)
#pragma unroll
      for (int e = 0; e < S::EPC; e++)
        qf[g][c * S::EPC + e] =
            Elem<T>::load1(a.q, (long long)(qh0 + g) * D + (c * 8 + j) * S::EPC + e) * qscale;

  float m[G], l[G], o[G][S::EL];
#pragma unroll
  for (int g = 0; g < G; g++) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < S::EL; e++) o[g][e] = 0.f;
  }

  const char* kbase = static_cast<const char*>(kv.k);
  const char* vbase = static_cast<const char*>(kv.v);
  constexpr int STEP = 16 * UNROLL;  // rows per CTA iteration
  for (int base = r0; base < r1; base += STEP) {
    long long row[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; u++) {
      const int r = base + u * 16 + warp * 4 + sg;
      row[u] = -1;
      if (r < r1) {
        const int key = SPARSE ? rows[r] : r;
        if ((unsigned)key < (unsigned)t) {
          row[u] = kv_row(kv, b, kvh, key);
          if (row[u] < 0) raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
        } else {
          raise_error(kv.err, PRHS_DEV_BAD_INDEX);
        }
      }
    }
    uint4 kc[UNROLL][S::CPL], vc[UNROLL][S::CPL];
#pragma unroll
    for (int u = 0; u < UNROLL; u++)
#pragma unroll
      for (int c = 0; c < S::CPL; c++) {
        if (row[u] >= 0) {
          kc[u][c] = ldg_stream(kbase + row[u] * S::RB + (c * 8 + j) * 16);
          vc[u][c] = ldg_stream(vbase + row[u] * S::RB + (c * 8 + j) * 16);
        } else {
          kc[u][c] = make_uint4(0, 0, 0, 0);
          vc[u][c] = make_uint4(0, 0, 0, 0);
        }
      }
    float s[UNROLL][G];
#pragma unroll
    for (int u = 0; u < UNROLL; u++) {
      float kf[S::EL];
#pragma unroll
      for (int c = 0; c < S::CPL; c++) Elem<T>::unpack(kc[u][c], kf + c * S::EPC);
#pragma unroll
      for (int g = 0; g < G; g++) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < S::EL; e++) acc = fmaf(qf[g][e], kf[e], acc);
        acc += __shfl_xor_sync(FULL_MASK, acc, 1);
        acc += __shfl_xor_sync(FULL_MASK, acc, 2);
        acc += __shfl_xor_sync(FULL_MASK, acc, 4);
        s[u][g] = row[u] >= 0 ? acc : -INFINITY;
      }
    }
    float vf[UNROLL][S::EL];
#pragma unroll
    for (int u = 0; u < UNROLL; u++)
#pragma unroll
      for (int c = 0; c < S::CPL; c++) Elem<T>::unpack(vc[u][c], vf[u] + c * S::EPC);
#pragma unroll
    for (int g = 0; g < G; g++) {
      float mx = m[g];
#pragma unroll
      for (int u = 0; u < UNROLL; u++) mx = fmaxf(mx, s[u][g]);
      if (mx == -INFINITY) continue;
      const float corr = exp2f(m[g] - mx);
      l[g] *= corr;
#pragma unroll
      for (int e = 0; e < S::EL; e++) o[g][e] *= corr;
#pragma unroll
      for (int u = 0; u < UNROLL; u++) {
        const float p = exp2f(s[u][g] - mx);
        l[g] += p;
#pragma unroll
        for (int e = 0; e < S::EL; e++) o[g][e] = fmaf(p, vf[u][e], o[g][e]);
      }
      m[g] = mx;
    }
  }

  // ---- merge the 4 row groups of the warp (lanes j, j+8, j+16, j+24) ----
#pragma unroll
  for (int g = 0; g < G; g++) {
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
      const float m2 = __shfl_xor_sync(FULL_MASK, m[g], off);
      const float l2 = __shfl_xor_sync(FULL_MASK, l[g], off);
      const float M = fmaxf(m[g], m2);
      const float c1 = M == -INFINITY ? 0.f : exp2f(m[g] - M);
      const float c2 = M == -INFINITY ? 0.f : exp2f(m2 - M);
      l[g] = l[g] * c1 + l2 * c2;
#pragma unroll
      for (int e = 0; e < S::EL; e++) {
        const float o2 = __shfl_xor_sync(FULL_MASK, o[g][e], off);
        o[g][e] = o[g][e] * c1 + o2 * c2;
      }
      m[g] = M;
    }
  }

  // ---- merge the 4 warps through shared memory, write this CTA's partial ----
  __shared__ float sm_m[4][G], sm_l[4][G];
  __shared__ float sm_o[4][G][D];
  __shared__ int sh_last;
  if (lane < 8) {
#pragma unroll
    for (int g = 0; g < G; g++) {
      if (lane == 0) {
        sm_m[warp][g] = m[g];
        sm_l[warp][g] = l[g];
      }
#pragma unroll
      for (int c = 0; c < S::CPL; c++)
#pragma unroll
        for (int e = 0; e < S::EPC; e++) sm_o[warp][g][(c * 8 + j) * S::EPC + e] = o[g][c * S::EPC + e];
    }
  }
  __syncthreads();
  constexpr int PW = D + 2;  // partial record: m, l, o[D]
  float* part = a.partials + ((long long)unit * G * a.splits) * PW;
  for (int x = threadIdx.x; x < G * D; x += ATTN_THREADS) {
    const int g = x / D, e = x % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; w++) M = fmaxf(M, sm_m[w][g]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; w++) {
        const float c = exp2f(sm_m[w][g] - M);
        L += c * sm_l[w][g];
        O += c * sm_o[w][g][e];
      }
    }
    float* rec = part + ((long long)g * a.splits + split) * PW;
    rec[2 + e] = O;
    if (e == 0) {
      rec[0] = M;
      rec[1] = L;
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) sh_last = atomicAdd(&a.counters[unit], 1u) == (unsigned)(a.splits - 1);
  __syncthreads();
  if (!sh_last) return;
  __threadfence();

  // ---- last CTA of this unit: combine every split ----
  for (int x = threadIdx.x; x < G * D; x += ATTN_THREADS) {
    const int g = x / D, e = x % D;
    const float* recs = part + (long long)g * a.splits * PW;
    float M = -INFINITY;
    for (int sp = 0; sp < a.splits; sp++) M = fmaxf(M, __ldcg(recs + (long long)sp * PW));
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int sp = 0; sp < a.splits; sp++) {
        const float* rec = recs + (long long)sp * PW;
        const float c = exp2f(__ldcg(rec) - M);
        L += c * __ldcg(rec + 1);
        O += c * __ldcg(rec + 2 + e);
      }
    }
    const long long qh = qh0 + g;
    a.out[qh * D + e] = L > 0.f ? O / L : 0.f;
    if (e == 0) a.lse[qh] = L > 0.f ? (M + log2f(L)) * LN2 : -INFINITY;
  }
  if (threadIdx.x == 0) a.counters[unit] = 0u;
}

template <typename T, int D, int G, bool SPARSE>
static cudaError_t attn_go(const AttnLaunch& a, int units, cudaStream_t st) {
  dim3 grid(a.splits, units);
  attn_kernel<T, D, G, SPARSE, 2><<<grid, ATTN_THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t attn_dispatch(const AttnLaunch& a, bool sparse, cudaStream_t st) {
  const KVView& kv = a.kv;
  if (sparse) return attn_go<T, D, 1, true>(a, kv.B * kv.Hq, st);
  const int units = kv.B * kv.Hkv;
  switch (kv.Hq / kv.Hkv) {
    case 1: return attn_go<T, D, 1, false>(a, units, st);
    case 2: return attn_go<T, D, 2, false>(a, units, st);
    case 4: return attn_go<T, D, 4, false>(a, units, st);
    case 8: return attn_go<T, D, 8, false>(a, units, st);
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_attn(const AttnLaunch& a, bool sparse, cudaStream_t st) {
  if (a.kv.dtype == PRHS_BF16) {
    if (a.kv.d == 128) return attn_dispatch<__nv_bfloat16, 128>(a, sparse, st);
    if (a.kv.d == 64) return attn_dispatch<__nv_bfloat16, 64>(a, sparse, st);
  } else {
    if (a.kv.d == 128) return attn_dispatch<float, 128>(a, sparse, st);
    if (a.kv.d == 64) return attn_dispatch<float, 64>(a, sparse, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace prhs
