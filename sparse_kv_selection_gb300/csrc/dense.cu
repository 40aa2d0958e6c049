// Dense decode attention (the baseline of Table IV, "Near-Oracle KV Selection
// via Pre-hoc Sparsity for Long-Context Inference"): every cached key of a KV
// head, for all G query heads that read it.
//
// K and V tiles of one KV head stream through a TMA -> shared-memory ring
// (128-byte swizzle, mbarrier-paced, one producer warp). The consumer warps
// form two groups of four, each holding GH = G / 2 query heads of the KV
// head: both groups read the same shared-memory tiles,
// computes its heads' logits as the scoring kernel does (8 lanes per key,
// transposed shuffle reduction), keeps a warp-uniform online softmax per head
// in base 2 and accumulates p * v from the same V tile. Each K and V byte
// leaves HBM once for the whole group, and the SM runs 8 consumer warps
// instead of 4 with the registers of G / 2 heads each. CTAs take
// equal shares of the key tiles of all KV heads; a KV head split over several
// CTAs is merged by the last one to finish (atomic ticket, no waiting).
#include "kernels.h"

namespace prhs {

template <typename T, int D>
struct DenseShape {
  static constexpr int RB = D * (int)sizeof(T);     // bytes per row
  static constexpr int NH = RB / 128;               // 128-byte segments per row
  static constexpr int EPC = 16 / (int)sizeof(T);   // elements per 16-byte chunk
  static constexpr int EL = NH * EPC;               // elements per lane (one d-slice)
  static constexpr int TK = RB <= 256 ? 128 : 64;   // keys per stage
  static constexpr int NW = TK / 32;                // consumer warps
  static constexpr int TILE = TK * RB;              // bytes of one K (or V) tile
  static constexpr int STAGE = 2 * TILE;            // K tile then V tile
  static constexpr int STAGES = (192 * 1024) / STAGE;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE + 2 * STAGES * 8 + 1024;
};

constexpr float D_LOG2E = 1.4426950408889634f;
constexpr float D_LN2 = 0.6931471805599453f;

__device__ __forceinline__ float transpose_reduce8_d(const float (&v)[8], int j) {
  float a[4], b[2];
  const bool h4 = j & 4, h2 = j & 2, h1 = j & 1;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const float send = h4 ? v[i] : v[i + 4];
    const float keep = h4 ? v[i + 4] : v[i];
    a[i] = keep + __shfl_xor_sync(FULL_MASK, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; i++) {
    const float send = h2 ? a[i] : a[i + 2];
    const float keep = h2 ? a[i + 2] : a[i];
    b[i] = keep + __shfl_xor_sync(FULL_MASK, send, 2);
  }
  const float send = h1 ? b[0] : b[1];
  const float keep = h1 ? b[1] : b[0];
  return keep + __shfl_xor_sync(FULL_MASK, send, 1);
}

__device__ __forceinline__ void consumer_bar(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

struct DenseLaunch {
  KVView kv;
  const void* q;
  float scale;
  float* out;
  float* lse;
  float* partials;     // [ctas + units][G][d + 2]
  unsigned* counters;  // [units]
  int ctas;
  bool paged;
  long long n_partial;  // floats available at partials (bounds check)
};

// Guarded global accesses: an index outside its array is reported and skipped.
__device__ __forceinline__ bool in_range(long long i, long long n, unsigned* err) {
  if (i >= 0 && i < n) return true;
  raise_error(err, PRHS_DEV_BAD_INDEX);
  return false;
}

// Query heads per consumer group and consumer warps of the dense kernel.
// Two consumer groups of G / 2 heads (one group when G = 1): 9 warps per SM,
// at most 3 per scheduler, whose 16K registers then allow 168 per thread.
template <int G> struct DenseGroups {
  static constexpr int GH = G >= 2 ? G / 2 : 1;
  static constexpr int NGR = G / GH;
  static constexpr int REGS = 168;
};

template <typename T, int D, int G>
__global__ void __maxnreg__(DenseGroups<G>::REGS)
    dense_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const DenseLaunch a) {
  using S = DenseShape<T, D>;
  constexpr int PW = D + 2;
  constexpr int GH = DenseGroups<G>::GH;     // query heads per consumer group
  constexpr int NCW = S::NW * DenseGroups<G>::NGR;  // consumer warps
  constexpr int NC = NCW * 32;                // consumer threads
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::STAGES * S::STAGE);
  uint64_t* empty = full + S::STAGES;
  int* tprefix = reinterpret_cast<int*>(empty + S::STAGES);  // [units + 1]
  __shared__ int sh_wsum[32];
  __shared__ float sm_m[S::NW][G], sm_l[S::NW][G];
  __shared__ float sm_o[S::NW][G][D];
  __shared__ int sh_last;

  pdl_wait();
  pdl_trigger();

  const KVView& kv = a.kv;
  const int U = kv.B * kv.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nthr = blockDim.x;
  const long long n_heads = (long long)kv.B * kv.Hq;
  const long long n_out = n_heads * D;

  // ---- key tiles of every KV head and their prefix sums ----
  {
    const int per_t = (U + nthr - 1) / nthr;
    const int u0 = threadIdx.x * per_t;
    int loc = 0;
    for (int k = 0; k < per_t; k++) {
      const int u = u0 + k;
      if (u >= U) break;
      const int tiles = (seq_len(kv, u / kv.Hkv) + S::TK - 1) / S::TK;
      tprefix[u] = tiles;
      loc += tiles;
    }
    int v = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, v, o);
      if (lane >= o) v += y;
    }
    if (lane == 31) sh_wsum[warp] = v;
    __syncthreads();
    int run = v - loc;
    for (int w = 0; w < warp; w++) run += sh_wsum[w];
    for (int k = 0; k < per_t; k++) {
      const int u = u0 + k;
      if (u >= U) break;
      const int tl = tprefix[u];
      tprefix[u] = run;
      run += tl;
    }
    if (threadIdx.x == nthr - 1) tprefix[U] = run;
    __syncthreads();
  }
  const int total = tprefix[U];
  const int C = gridDim.x, c = blockIdx.x;

  // KV heads without keys: out = 0, lse = -inf
  for (int u = c; u < U; u += C) {
    if (tprefix[u + 1] != tprefix[u]) continue;
    const int qh0 = (u / kv.Hkv) * kv.Hq + (u % kv.Hkv) * G;
    for (int x = threadIdx.x; x < G * D; x += nthr) {
      const long long oi = (long long)(qh0 + x / D) * D + x % D;
      if (in_range(oi, n_out, kv.err)) a.out[oi] = 0.f;
      if (x % D == 0 && in_range(qh0 + x / D, n_heads, kv.err)) a.lse[qh0 + x / D] = -INFINITY;
    }
  }
  const int per = (total + C - 1) / C;
  const int g0 = c * per;
  const int ntiles = min(total, g0 + per) - g0;
  if (total == 0 || ntiles <= 0) return;

  auto tile_at = [&](int it, int& u, int& key0) {
    const int g = g0 + it;
    int lo = 0, hi = U - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tprefix[mid] <= g) lo = mid; else hi = mid - 1;
    }
    u = lo;
    key0 = (g - tprefix[lo]) * S::TK;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::STAGES; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == NCW) {
    // ------- producer warp: K and V tiles of each stage -------
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&vmap);
    }
    int issued = 0;
    for (int it = 0; it < ntiles; it++) {
      const int s = it % S::STAGES;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&empty[s], ((it / S::STAGES) & 1) ^ 1, kv.err);
      if (!__shfl_sync(FULL_MASK, ok, 0)) break;
      int u, tile0;
      tile_at(it, u, tile0);
      const int b = u / kv.Hkv, kvh = u % kv.Hkv;
      uint8_t* dst = smem + s * S::STAGE;
      if (!a.paged) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[s], S::STAGE);
          tma_load_3d(dst, &kmap, 0, 0, u * kv.t_max + tile0, &full[s]);
          tma_load_3d(dst + S::TILE, &vmap, 0, 0, u * kv.t_max + tile0, &full[s]);
        }
      } else {
        const int k1 = min(seq_len(kv, b), tile0 + S::TK);
        const int nbox = min(S::TK / PAGED_BOX_ROWS, (k1 - tile0 + PAGED_BOX_ROWS - 1) / PAGED_BOX_ROWS);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], 2 * nbox * PAGED_BOX_ROWS * S::RB);
        __syncwarp();
        if (lane < nbox) {
          long long row = kv_row(kv, b, kvh, tile0 + lane * PAGED_BOX_ROWS);
          if (row < 0) {
            raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
            row = 0;
          }
          tma_load_3d(dst + lane * PAGED_BOX_ROWS * S::RB, &kmap, 0, 0, (int)row, &full[s]);
          tma_load_3d(dst + S::TILE + lane * PAGED_BOX_ROWS * S::RB, &vmap, 0, 0, (int)row, &full[s]);
        }
      }
      __syncwarp();
      issued = it + 1;
    }
    if (lane == 0)
      for (int it = max(0, issued - S::STAGES); it < issued; it++)
        mbar_wait(&full[it % S::STAGES], (it / S::STAGES) & 1, kv.err);
    return;
  }

  // ---------------- consumers ----------------
  const int r = lane >> 3;  // key slot (8 keys)
  const int j = lane & 7;   // 16-byte chunk of each 128-byte segment: this lane's d-slice
  const int wl = warp % S::NW;       // this warp's 32 keys of each stage
  const int hg = (warp / S::NW) * GH;  // this warp's first query head in the group
  const float qscale = a.scale * D_LOG2E;
  float qf[GH][S::EL], o[GH][S::EL], m[GH], l[GH];
  int cur_u = -1, k1 = 0, qh0 = 0;
  bool dead = false;  // a wait timed out: keep step with the other warps, compute nothing

  // merge this CTA's state for unit u into out/lse (or a partial + ticket)
  auto finalize = [&](int u) {
#pragma unroll
    for (int gg = 0; gg < GH; gg++) {
#pragma unroll
      for (int e = 0; e < S::EL; e++) {  // the warp's m is uniform: slots add up
        o[gg][e] += __shfl_xor_sync(FULL_MASK, o[gg][e], 8);
        o[gg][e] += __shfl_xor_sync(FULL_MASK, o[gg][e], 16);
      }
      const float L = warp_sum(l[gg]);
      if (lane == 0) {
        sm_m[wl][hg + gg] = m[gg];
        sm_l[wl][hg + gg] = L;
      }
      if (lane < 8) {
#pragma unroll
        for (int h = 0; h < S::NH; h++)
#pragma unroll
          for (int e = 0; e < S::EPC; e++)
            sm_o[wl][hg + gg][h * (128 / (int)sizeof(T)) + j * S::EPC + e] = o[gg][h * S::EPC + e];
      }
    }
    consumer_bar(NC);
    const int cf = tprefix[u] / per, cl = (tprefix[u + 1] - 1) / per;
    for (int x = threadIdx.x; x < G * D; x += NC) {
      const int g = x / D, e = x % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < S::NW; w++) M = fmaxf(M, sm_m[w][g]);
      float Lt = 0.f, Ot = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < S::NW; w++) {
          const float cw = exp2f(sm_m[w][g] - M);
          Lt += cw * sm_l[w][g];
          Ot += cw * sm_o[w][g][e];
        }
      }
      if (cf == cl) {
        const long long oi = (long long)(qh0 + g) * D + e;
        if (in_range(oi, n_out, kv.err)) a.out[oi] = Lt > 0.f ? Ot / Lt : 0.f;
        if (e == 0 && in_range(qh0 + g, n_heads, kv.err))
          a.lse[qh0 + g] = Lt > 0.f ? (M + log2f(Lt)) * D_LN2 : -INFINITY;
      } else {
        const long long ri = ((long long)(c + u) * G + g) * PW;
        if (in_range(ri + PW - 1, a.n_partial, kv.err)) {
          float* rec = a.partials + ri;
          rec[2 + e] = Ot;
          if (e == 0) {
            rec[0] = M;
            rec[1] = Lt;
          }
        }
      }
    }
    if (cf != cl) {
      __threadfence();
      consumer_bar(NC);
      if (threadIdx.x == 0) sh_last = atomicAdd(&a.counters[u], 1u) == (unsigned)(cl - cf);
      consumer_bar(NC);
      if (sh_last) {
        __threadfence();
        for (int x = threadIdx.x; x < G * D; x += NC) {
          const int g = x / D, e = x % D;
          float M = -INFINITY;
          for (int cs = cf; cs <= cl; cs++) {
            const long long ri = ((long long)(cs + u) * G + g) * PW;
            if (in_range(ri + PW - 1, a.n_partial, kv.err)) M = fmaxf(M, __ldcg(a.partials + ri));
          }
          float Lt = 0.f, Ot = 0.f;
          if (M != -INFINITY) {
            for (int cs = cf; cs <= cl; cs++) {
              const long long ri = ((long long)(cs + u) * G + g) * PW;
              if (!in_range(ri + PW - 1, a.n_partial, kv.err)) continue;
              const float* rec = a.partials + ri;
              const float cw = exp2f(__ldcg(rec) - M);
              Lt += cw * __ldcg(rec + 1);
              Ot += cw * __ldcg(rec + 2 + e);
            }
          }
          const long long oi = (long long)(qh0 + g) * D + e;
          if (in_range(oi, n_out, kv.err)) a.out[oi] = Lt > 0.f ? Ot / Lt : 0.f;
          if (e == 0 && in_range(qh0 + g, n_heads, kv.err))
            a.lse[qh0 + g] = Lt > 0.f ? (M + log2f(Lt)) * D_LN2 : -INFINITY;
        }
        if (threadIdx.x == 0) a.counters[u] = 0u;
      }
    }
    consumer_bar(NC);  // shared partial state is free again
  };

  for (int it = 0; it < ntiles; it++) {
    int u, tile0;
    tile_at(it, u, tile0);
    if (u != cur_u) {
      if (cur_u >= 0) finalize(cur_u);
      cur_u = u;
      const int b = u / kv.Hkv, kvh = u % kv.Hkv;
      qh0 = b * kv.Hq + kvh * G;
      k1 = seq_len(kv, b);
#pragma unroll
      for (int gg = 0; gg < GH; gg++) {
        m[gg] = -INFINITY;
        l[gg] = 0.f;
#pragma unroll
        for (int h = 0; h < S::NH; h++)
#pragma unroll
          for (int e = 0; e < S::EPC; e++) {
            const long long qi =
                (long long)(qh0 + hg + gg) * D + h * (128 / (int)sizeof(T)) + j * S::EPC + e;
            qf[gg][h * S::EPC + e] = in_range(qi, n_out, kv.err) ? Elem<T>::load1(a.q, qi) * qscale : 0.f;
            o[gg][h * S::EPC + e] = 0.f;
          }
      }
    }
    const int s = it % S::STAGES;
    if (dead || !mbar_wait(&full[s], (it / S::STAGES) & 1, kv.err)) {
      dead = true;
      continue;
    }
    const uint8_t* kt = smem + s * S::STAGE;
    const uint8_t* vt = kt + S::TILE;
    float acc[GH][8];
#pragma unroll
    for (int gg = 0; gg < GH; gg++)
#pragma unroll
      for (int p = 0; p < 8; p++) acc[gg][p] = 0.f;
#pragma unroll
    for (int p = 0; p < 8; p++) {
      const int key = wl * 32 + r * 8 + p;
#pragma unroll
      for (int h = 0; h < S::NH; h++) {
        const int line = key * S::NH + h;
        const uint4 cw = *reinterpret_cast<const uint4*>(kt + line * 128 + ((j ^ (line & 7)) << 4));
        float f[S::EPC];
        Elem<T>::unpack(cw, f);
#pragma unroll
        for (int gg = 0; gg < GH; gg++)
#pragma unroll
          for (int e = 0; e < S::EPC; e++) acc[gg][p] = fmaf(qf[gg][h * S::EPC + e], f[e], acc[gg][p]);
      }
    }
    const bool valid = tile0 + wl * 32 + lane < k1;
    float pr[GH];
#pragma unroll
    for (int gg = 0; gg < GH; gg++) {
      const float red = transpose_reduce8_d(acc[gg], j);  // every lane takes part
      const float sc = valid ? red : -INFINITY;
      const float mx = fmaxf(m[gg], warp_max(sc));
      const float corr = m[gg] == -INFINITY ? 0.f : exp2f(m[gg] - mx);
      pr[gg] = mx == -INFINITY ? 0.f : exp2f(sc - mx);
      l[gg] = l[gg] * corr + pr[gg];
#pragma unroll
      for (int e = 0; e < S::EL; e++) o[gg][e] *= corr;
      m[gg] = mx;
    }
    // p * v: lane (r, j) adds the keys of slot r into its d-slice j. On a
    // head's last tile the rows past t_b were not loaded on a paged cache
    // (whatever the shared memory held, possibly not finite): their weight
    // is 0 and their row is taken as 0, so they add nothing.
    const bool partial = tile0 + S::TK > k1;
#pragma unroll
    for (int p = 0; p < 8; p++) {
      const int key = wl * 32 + r * 8 + p;
      float vf[S::EL];
#pragma unroll
      for (int h = 0; h < S::NH; h++) {
        const int line = key * S::NH + h;
        const uint4 cw = *reinterpret_cast<const uint4*>(vt + line * 128 + ((j ^ (line & 7)) << 4));
        Elem<T>::unpack(cw, vf + h * S::EPC);
      }
      if (partial && tile0 + key >= k1) {
#pragma unroll
        for (int e = 0; e < S::EL; e++) vf[e] = 0.f;
      }
#pragma unroll
      for (int gg = 0; gg < GH; gg++) {
        const float pk = __shfl_sync(FULL_MASK, pr[gg], r * 8 + p);
#pragma unroll
        for (int e = 0; e < S::EL; e++) o[gg][e] = fmaf(pk, vf[e], o[gg][e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (cur_u >= 0) finalize(cur_u);
}

template <typename T, int D, int G>
static cudaError_t dense_go(const DenseLaunch& a, const CUtensorMap* km, const CUtensorMap* vm,
                            cudaStream_t st) {
  using S = DenseShape<T, D>;
  auto k = dense_kernel<T, D, G>;
  const size_t smem = S::SMEM + ((size_t)a.kv.B * a.kv.Hkv + 1) * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(a.ctas), dim3(32 * (S::NW * DenseGroups<G>::NGR + 1)), smem, st, a.kv.pdl, *km, *vm, a);
}

template <typename T, int D>
static cudaError_t dense_dispatch(const DenseLaunch& a, const CUtensorMap* km,
                                  const CUtensorMap* vm, cudaStream_t st) {
  switch (a.kv.Hq / a.kv.Hkv) {
    case 1: return dense_go<T, D, 1>(a, km, vm, st);
    case 2: return dense_go<T, D, 2>(a, km, vm, st);
    case 4: return dense_go<T, D, 4>(a, km, vm, st);
    case 8: return dense_go<T, D, 8>(a, km, vm, st);
  }
  return cudaErrorNotSupported;
}

size_t dense_partial_floats(const KVView& kv, int ctas);

cudaError_t launch_dense(const KVView& kv, const void* q, float scale, float* out, float* lse,
                         float* partials, unsigned* counters, int ctas, bool paged,
                         const CUtensorMap* kmap, const CUtensorMap* vmap, cudaStream_t st) {
  DenseLaunch a;
  a.kv = kv;
  a.q = q;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.partials = partials;
  a.counters = counters;
  a.ctas = ctas;
  a.paged = paged;
  a.n_partial = (long long)dense_partial_floats(kv, ctas);
  if (kv.dtype == PRHS_BF16) {
    if (kv.d == 128) return dense_dispatch<__nv_bfloat16, 128>(a, kmap, vmap, st);
    if (kv.d == 64) return dense_dispatch<__nv_bfloat16, 64>(a, kmap, vmap, st);
  } else {
    if (kv.d == 128) return dense_dispatch<float, 128>(a, kmap, vmap, st);
    if (kv.d == 64) return dense_dispatch<float, 64>(a, kmap, vmap, st);
  }
  return cudaErrorNotSupported;
}

size_t dense_partial_floats(const KVView& kv, int ctas) {
  return ((size_t)ctas + (size_t)kv.B * kv.Hkv) * (kv.Hq / kv.Hkv) * (kv.d + 2);
}

int dense_rows_per_stage(const KVView& kv) {
  return kv.dtype == PRHS_F32 && kv.d == 128 ? 64 : 128;
}

}  // namespace prhs
