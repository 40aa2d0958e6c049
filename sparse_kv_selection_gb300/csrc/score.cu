// Top-N oracle selector: logits s_i = scale * <q, k_i> over the whole cache,
// then the N largest (lowest index on ties) and the dropped mass
//   delta = sum_{i not in S} softmax(s)_i.
// "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference",
// abstract (top-k oracle selection before attention scoring, dropped mass)
// and Table I (S_t, N, tau(.), delta(.)).
//
// Two kernels:
//  * score_kernel  streams K once per KV head through a TMA -> shared-memory
//    ring (128-byte swizzled tiles, mbarrier-pipelined, one producer warp,
//    four consumer warps) and writes fp32 logits for the G query heads of
//    the group. HBM-bound: t * d * sizeof(T) bytes per KV head.
//  * select_kernel one CTA per query head: softmax statistics, a three-digit
//    radix select for the N-th largest logit, then an index-ordered compaction
//    that emits the set ascending and sums the dropped mass.
#include "kernels.h"

namespace prhs {

// -------------------------------------------------------------------------- //
// scoring
// -------------------------------------------------------------------------- //
constexpr int SCORE_PB = 8;  // KV heads whose lengths and skip flags a thread loads at once

template <typename T, int D>
struct ScoreShape {
  static constexpr int RB = D * (int)sizeof(T);        // bytes per key row
  static constexpr int NH = RB / 128;                  // 128-byte segments per row
  static constexpr int EPC = 16 / (int)sizeof(T);      // elements per 16-byte chunk
  static constexpr int EL = NH * EPC;                  // q elements per lane
  static constexpr int TK = SCORE_TILE;                // keys per stage
  static constexpr int NW = 4;                         // consumer warps (32 keys each)
  static constexpr int STAGE_BYTES = TK * RB;
  static constexpr int STAGES = RB == 128 ? 6 : (RB == 256 ? 3 : 2);
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 2 * STAGES * 8 + 1024;
  static_assert(RB % 128 == 0, "row must be a whole number of 128-byte segments");
};

// Eight partial dot products per lane (one per key p) held by the 8 lanes of
// a key slot; afterwards lane j of the slot holds the full sum for key p = j.
__device__ __forceinline__ float transpose_reduce8(const float (&v)[8], int j) {
  float a[4], b[2];
  const bool h4 = j & 4, h2 = j & 2, h1 = j & 1;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    float send = h4 ? v[i] : v[i + 4];
    float keep = h4 ? v[i + 4] : v[i];
    a[i] = keep + __shfl_xor_sync(FULL_MASK, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; i++) {
    float send = h2 ? a[i] : a[i + 2];
    float keep = h2 ? a[i + 2] : a[i];
    b[i] = keep + __shfl_xor_sync(FULL_MASK, send, 2);
  }
  float send = h1 ? b[0] : b[1];
  float keep = h1 ? b[1] : b[0];
  return keep + __shfl_xor_sync(FULL_MASK, send, 1);
}

// Tensor-core pieces of the grouped scoring: a 16x16 bf16 tile of K (keys as
// rows) from shared memory into the A fragment of mma.m16n8k16, and the mma
// itself (bf16 inputs, fp32 accumulation).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(160) score_kernel(const __grid_constant__ CUtensorMap tmap,
                                                    const ScoreLaunch a) {
  using S = ScoreShape<T, D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::STAGES * S::STAGE_BYTES);
  uint64_t* empty = full + S::STAGES;
  int* tprefix = reinterpret_cast<int*>(empty + S::STAGES);  // [units + 1] tile prefix
  __shared__ int sh_wsum[5];

  pdl_wait();
  pdl_trigger();

  const KVView& kv = a.kv;
  const int U = kv.B * kv.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nthr = blockDim.x;

  // ---- key tiles of every retrieving KV head, and their prefix sums ----
  {
    const int per_t = (U + nthr - 1) / nthr;
    const int u0 = threadIdx.x * per_t;
    // SCORE_PB units per batch, all their loads issued before any is used
    int loc = 0;
    for (int k0 = 0; k0 < per_t; k0 += SCORE_PB) {
      int len[SCORE_PB];
      bool need[SCORE_PB];
#pragma unroll
      for (int i = 0; i < SCORE_PB; i++) {
        const int u = u0 + k0 + i;
        const bool in = k0 + i < per_t && u < U;
        const int b = u / kv.Hkv, kvh = u % kv.Hkv;
        len[i] = in ? __ldg(kv.seq_lens + b) : 0;
        need[i] = a.head_skip == nullptr;
        if (in && !need[i]) {
          const int qh0 = b * kv.Hq + kvh * G;
#pragma unroll
          for (int g = 0; g < G; g++) need[i] |= __ldg(a.head_skip + qh0 + g) == 0;
        }
      }
#pragma unroll
      for (int i = 0; i < SCORE_PB; i++) {
        const int u = u0 + k0 + i;
        if (k0 + i >= per_t || u >= U) break;
        const int tiles = need[i] ? (checked_len(kv, len[i]) + S::TK - 1) / S::TK : 0;
        tprefix[u] = tiles;
        loc += tiles;
      }
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
  const int per = (total + gridDim.x - 1) / gridDim.x;
  const int g0 = blockIdx.x * per;
  const int ntiles = min(total, g0 + per) - g0;
  if (ntiles <= 0) return;

  // unit and first key of the it-th tile of this CTA
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
      mbar_init(&empty[s], S::NW);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == S::NW) {
    // ------- producer warp: lane 0 paces the ring, lanes issue the TMA boxes -------
    if (lane == 0) prefetch_tmap(&tmap);
    int issued = 0;
    if (!a.paged) {
      // contiguous caches: one 3-D box per tile
      for (int it = 0; it < ntiles; it++) {
        const int s = it % S::STAGES;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&empty[s], ((it / S::STAGES) & 1) ^ 1, kv.err);
        if (!__shfl_sync(FULL_MASK, ok, 0)) break;
        int u, tile0;
        tile_at(it, u, tile0);
        if (lane == 0) {
          uint8_t* dst = smem + s * S::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], S::STAGE_BYTES);
          tma_load_3d(dst, &tmap, 0, 0, u * kv.t_max + tile0, &full[s]);
        }
        __syncwarp();
        issued = it + 1;
      }
    } else {
      // paged caches: one 16-row box per page, one lane per box. The tiles of
      // a CTA are consecutive: the next tile follows the current one in its
      // head (a search only where a head ends), and its page rows are looked
      // up before the wait for the free slot, so those loads overlap the wait.
      int u, tile0;
      tile_at(0, u, tile0);
      int len = seq_len(kv, u / kv.Hkv);
      auto box_row = [&](int uu, int t0, int ln) -> long long {
        const int nb = min(S::TK / PAGED_BOX_ROWS, (min(ln, t0 + S::TK) - t0 + PAGED_BOX_ROWS - 1) / PAGED_BOX_ROWS);
        if (lane >= nb) return 0;
        long long row = kv_row(kv, uu / kv.Hkv, uu % kv.Hkv, t0 + lane * PAGED_BOX_ROWS);
        if (row < 0) {
          raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
          row = 0;
        }
        return row;
      };
      long long row_next = box_row(u, tile0, len);
      for (int it = 0; it < ntiles; it++) {
        const int s = it % S::STAGES;
        const int ct0 = tile0, clen = len;
        const long long row = row_next;
        if (it + 1 < ntiles) {
          tile0 += S::TK;
          if (tile0 >= len) {
            tile_at(it + 1, u, tile0);
            len = seq_len(kv, u / kv.Hkv);
          }
          row_next = box_row(u, tile0, len);
        }
        int ok = 1;
        if (lane == 0) ok = mbar_wait(&empty[s], ((it / S::STAGES) & 1) ^ 1, kv.err);
        if (!__shfl_sync(FULL_MASK, ok, 0)) break;
        uint8_t* dst = smem + s * S::STAGE_BYTES;
        const int k1 = min(clen, ct0 + S::TK);
        const int nbox = min(S::TK / PAGED_BOX_ROWS, (k1 - ct0 + PAGED_BOX_ROWS - 1) / PAGED_BOX_ROWS);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], nbox * PAGED_BOX_ROWS * S::RB);
        __syncwarp();
        if (lane < nbox) tma_load_3d(dst + lane * PAGED_BOX_ROWS * S::RB, &tmap, 0, 0, (int)row, &full[s]);
        __syncwarp();
        issued = it + 1;
      }
    }
    // never leave while a copy into this CTA's shared memory is in flight
    if (lane == 0)
      for (int it = max(0, issued - S::STAGES); it < issued; it++)
        mbar_wait(&full[it % S::STAGES], (it / S::STAGES) & 1, kv.err);
    return;
  }

  // ---------------- consumers: 32 keys per warp per stage ----------------
  // A bf16 cache read by a group of query heads is a real contraction: the
  // stage's keys times the group's queries, on the tensor cores (keys as the
  // M dimension, 16 per tile; the group as N, padded to 8; d as K). fp32
  // caches and single heads take the CUDA-core form below.
  constexpr bool MMA = sizeof(T) == 2 && G >= 2;
  if constexpr (MMA) {
    constexpr int KS = D / 16;           // k-steps of 16 dimensions
    constexpr int EPS = 128 / 2;         // bf16 elements per 128-byte segment
    uint32_t bq[KS][2];                  // B fragments: q[n][k], n = lane / 4
    const int n_b = lane >> 2, kq = (lane & 3) * 2;
    int cur_u = -1, qh0 = 0, k1 = 0;
    for (int it = 0; it < ntiles; it++) {
      int u, tile0;
      tile_at(it, u, tile0);
      if (u != cur_u) {
        cur_u = u;
        const int b = u / kv.Hkv, kvh = u % kv.Hkv;
        qh0 = b * kv.Hq + kvh * G;
        k1 = seq_len(kv, b);
        const uint16_t* qb = static_cast<const uint16_t*>(a.q) + (long long)(qh0 + n_b) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ks++) {
          bq[ks][0] = n_b < G ? *reinterpret_cast<const uint32_t*>(qb + ks * 16 + kq) : 0u;
          bq[ks][1] = n_b < G ? *reinterpret_cast<const uint32_t*>(qb + ks * 16 + 8 + kq) : 0u;
        }
      }
      const int s = it % S::STAGES;
      if (!mbar_wait(&full[s], (it / S::STAGES) & 1, kv.err)) break;
      const uint32_t stage = smem_addr(smem + s * S::STAGE_BYTES);
      float c[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; mt++) {
#pragma unroll
        for (int e = 0; e < 4; e++) c[mt][e] = 0.f;
        // lane l addresses row (l % 16) of the 16-key tile, dims +8 (l / 16)
        const int key = warp * 32 + mt * 16 + (lane & 15);
#pragma unroll
        for (int ks = 0; ks < KS; ks++) {
          const int kd = ks * 16 + (lane >> 4) * 8;
          const int line = key * S::NH + kd / EPS;           // 128-byte line of the stage
          const int ch = (kd % EPS) / 8;                     // its 16-byte chunk, swizzled
          uint32_t af[4];
          ldsm_x4(stage + line * 128 + ((ch ^ (line & 7)) << 4), af);
          mma_16816_bf16(c[mt], af, bq[ks][0], bq[ks][1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      // c[mt][0..1]: key (lane / 4), heads 2 (lane % 4) + {0, 1}; c[mt][2..3]: key + 8
      const int n0 = (lane & 3) * 2;
#pragma unroll
      for (int mt = 0; mt < 2; mt++) {
        const int key = tile0 + warp * 32 + mt * 16 + (lane >> 2);
#pragma unroll
        for (int h = 0; h < 2; h++) {
          const int kk = key + 8 * h;
          if (kk >= k1) continue;
          if (n0 < G) a.scores[(long long)(qh0 + n0) * kv.t_max + kk] = c[mt][2 * h] * a.scale;
          if (n0 + 1 < G) a.scores[(long long)(qh0 + n0 + 1) * kv.t_max + kk] = c[mt][2 * h + 1] * a.scale;
        }
      }
    }
    return;
  }
  const int r = lane >> 3;  // key slot 0..3 (8 keys each)
  const int j = lane & 7;   // 16-byte chunk within each 128-byte segment
  float qf[G][S::EL];
  int cur_u = -1, qh0 = 0, k1 = 0;

  for (int it = 0; it < ntiles; it++) {
    int u, tile0;
    tile_at(it, u, tile0);
    if (u != cur_u) {
      cur_u = u;
      const int b = u / kv.Hkv, kvh = u % kv.Hkv;
      qh0 = b * kv.Hq + kvh * G;
      k1 = seq_len(kv, b);
#pragma unroll
      for (int g = 0; g < G; g++) {
        const long long qbase = (long long)(qh0 + g) * D;
#pragma unroll
        for (int h = 0; h < S::NH; h++)
#pragma unroll
          for (int e = 0; e < S::EPC; e++)
            qf[g][h * S::EPC + e] =
                Elem<T>::load1(a.q, qbase + h * (128 / (int)sizeof(T)) + j * S::EPC + e);
      }
    }
    const int s = it % S::STAGES;
    if (!mbar_wait(&full[s], (it / S::STAGES) & 1, kv.err)) break;
    const uint8_t* stage = smem + s * S::STAGE_BYTES;
    float acc[G][8];
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
      for (int p = 0; p < 8; p++) acc[g][p] = 0.f;
#pragma unroll
    for (int p = 0; p < 8; p++) {
      const int key = warp * 32 + r * 8 + p;
#pragma unroll
      for (int h = 0; h < S::NH; h++) {
        const int line = key * S::NH + h;  // 128-byte line in the stage
        const uint4 c = *reinterpret_cast<const uint4*>(stage + line * 128 + ((j ^ (line & 7)) << 4));
        float f[S::EPC];
        Elem<T>::unpack(c, f);
#pragma unroll
        for (int g = 0; g < G; g++)
#pragma unroll
          for (int e = 0; e < S::EPC; e++) acc[g][p] = fmaf(qf[g][h * S::EPC + e], f[e], acc[g][p]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    const int key = tile0 + warp * 32 + lane;
#pragma unroll
    for (int g = 0; g < G; g++) {
      const float sc = transpose_reduce8(acc[g], j) * a.scale;
      if (key < k1) a.scores[(long long)(qh0 + g) * kv.t_max + key] = sc;
    }
  }
}

template <typename T, int D>
static cudaError_t score_dispatch_g(const ScoreLaunch& a, const CUtensorMap* tmap, int G,
                                   cudaStream_t st) {
  using S = ScoreShape<T, D>;
  void (*k)(const CUtensorMap, const ScoreLaunch) = nullptr;
  switch (G) {
    case 1: k = score_kernel<T, D, 1>; break;
    case 2: k = score_kernel<T, D, 2>; break;
    case 4: k = score_kernel<T, D, 4>; break;
    case 8: k = score_kernel<T, D, 8>; break;
    default: return cudaErrorInvalidValue;
  }
  const size_t smem = S::SMEM + ((size_t)a.kv.B * a.kv.Hkv + 1) * sizeof(int);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(a.ctas), dim3(32 * (S::NW + 1)), smem, st, a.kv.pdl, *tmap, a);
}

size_t score_smem_bytes(prhs_dtype dt, int d) {
  if (dt == PRHS_BF16) return d == 64 ? ScoreShape<__nv_bfloat16, 64>::SMEM : ScoreShape<__nv_bfloat16, 128>::SMEM;
  return d == 64 ? ScoreShape<float, 64>::SMEM : ScoreShape<float, 128>::SMEM;
}

// -------------------------------------------------------------------------- //
// selection
// -------------------------------------------------------------------------- //
struct SelShared {
  unsigned hist[2048];
  unsigned scan[32];
  float red_m[32];
  float red_z[32];
  unsigned digit, krem;
  float M, Z;
};

// Block-wide inclusive scan of one unsigned per thread (1024 threads).
__device__ __forceinline__ unsigned block_inclusive_scan(unsigned v, unsigned* warp_tot,
                                                         unsigned& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    unsigned n = __shfl_up_sync(FULL_MASK, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      unsigned n = __shfl_up_sync(FULL_MASK, w, o);
      if (lane >= o) w += n;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  total = warp_tot[(blockDim.x >> 5) - 1];
  const unsigned add = warp > 0 ? warp_tot[warp - 1] : 0u;
  __syncthreads();  // warp_tot may be reused right after
  return v + add;
}

__device__ __forceinline__ void combine_mz(float& m, float& z, float m2, float z2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  z = (m == -INFINITY ? 0.f : z * expf(m - M)) + (m2 == -INFINITY ? 0.f : z2 * expf(m2 - M));
  m = M;
}

template <typename T>
__device__ __forceinline__ void copy_query(const SelectLaunch& a, int qh) {
  const int d = a.kv.d;
  for (int i = threadIdx.x; i < d; i += blockDim.x)
    copy_elem<T>(a.q_anchor, a.q_src, (long long)qh * d + i);
}

template <typename T>
__global__ void __launch_bounds__(SELECT_THREADS) select_kernel(const SelectLaunch a) {
  extern __shared__ float cache[];
  __shared__ SelShared sh;
  pdl_wait();
  pdl_trigger();
  const KVView& kv = a.kv;
  const int qh = blockIdx.x;  // b * Hq + query head
  const int b = qh / kv.Hq;
  if (a.head_skip != nullptr && a.head_skip[qh] != 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x;
  const int t = seq_len(kv, b);
  int Nb = a.n_budget != nullptr ? a.n_budget[b] : a.N;
  if (Nb < 0) Nb = 0;
  const int lim = a.anchor_idx != nullptr ? min(a.cap, a.anchor_cap) : a.cap;
  if (min(Nb, t) > lim) {
    if (tid == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    Nb = lim;
  }
  int32_t* out = a.idx + (long long)qh * a.cap;
  int32_t* aout = a.anchor_idx != nullptr ? a.anchor_idx + (long long)qh * a.anchor_cap : nullptr;

  if (Nb >= t || Nb == 0) {  // keep everything (delta = 0) or nothing (delta = 1)
    const int n = Nb >= t ? t : 0;
    for (int i = tid; i < n; i += nthreads) {
      out[i] = i;
      if (aout) aout[i] = i;
    }
    if (tid == 0) {
      a.n_sel[qh] = n;
      a.delta[qh] = n == t ? 0.f : 1.f;
      if (a.anchor_n) a.anchor_n[qh] = n;
    }
    if (a.q_anchor) copy_query<T>(a, qh);
    return;
  }

  // ---- stage the logits (shared memory when they fit) ----
  const float* src = a.scores + (long long)qh * kv.t_max;
  const float* sp = src;
  if (t <= SELECT_CACHE_FLOATS) {
    for (int i = tid; i < t; i += nthreads) cache[i] = src[i];
    sp = cache;
  }
  for (int i = tid; i < 2048; i += nthreads) sh.hist[i] = 0;
  __syncthreads();

  // ---- pass 1: softmax statistics (m, Z) and histogram of the top 11 bits ----
  float m = -INFINITY, z = 0.f;
  const int rounds = (t + nthreads - 1) / nthreads;
  for (int rd = 0; rd < rounds; rd++) {
    const int i = rd * nthreads + tid;
    const bool in = i < t;
    const float s = in ? sp[i] : -INFINITY;
    if (in) {
      if (s > m) {
        z = z * expf(m - s) + 1.f;
        m = s;
      } else {
        z += expf(s - m);
      }
    }
    if (in) atomicAdd(&sh.hist[order_key(s) >> 21], 1u);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(FULL_MASK, m, o);
    const float z2 = __shfl_xor_sync(FULL_MASK, z, o);
    combine_mz(m, z, m2, z2);
  }
  if (lane == 0) {
    sh.red_m[warp] = m;
    sh.red_z[warp] = z;
  }
  if (tid == 0) sh.krem = (unsigned)Nb;
  __syncthreads();
  if (warp == 0) {  // one warp merges the per-warp softmax statistics
    float m2 = lane < (nthreads >> 5) ? sh.red_m[lane] : -INFINITY;
    float z2 = lane < (nthreads >> 5) ? sh.red_z[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m3 = __shfl_xor_sync(FULL_MASK, m2, o);
      const float z3 = __shfl_xor_sync(FULL_MASK, z2, o);
      combine_mz(m2, z2, m3, z3);
    }
    if (lane == 0) {
      sh.M = m2;
      sh.Z = z2;
    }
  }

  // ---- radix select: digits of 11, 11 and 10 bits from the top ----
  unsigned prefix = 0, mask = 0;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; pass++) {
    const int sh_ = shifts[pass];
    const int nb = 1 << widths[pass];
    if (pass > 0) {
      for (int i = tid; i < nb; i += nthreads) sh.hist[i] = 0;
      __syncthreads();
      for (int rd = 0; rd < rounds; rd++) {
        const int i = rd * nthreads + tid;
        bool in = i < t;
        const unsigned u = in ? order_key(sp[i]) : 0u;
        in = in && (u & mask) == prefix;
        if (in) atomicAdd(&sh.hist[(u >> sh_) & (nb - 1)], 1u);
      }
      __syncthreads();
    }
    // descending cumulative counts: thread i owns bins nb-1-2i and nb-2-2i
    const unsigned krem = sh.krem;
    const int per = nb / nthreads;  // 2 or 1
    unsigned c0 = 0, c1 = 0;
    const int bin0 = nb - 1 - per * tid;
    c0 = sh.hist[bin0];
    if (per == 2) c1 = sh.hist[bin0 - 1];
    unsigned tot;
    const unsigned incl = block_inclusive_scan(c0 + c1, sh.scan, tot);
    const unsigned excl = incl - c0 - c1;
    // the bin holding the krem-th largest among the candidates
    if (excl < krem && excl + c0 >= krem) {
      sh.digit = (unsigned)bin0;
      sh.krem = krem - excl;
    } else if (per == 2 && excl + c0 < krem && excl + c0 + c1 >= krem) {
      sh.digit = (unsigned)(bin0 - 1);
      sh.krem = krem - excl - c0;
    }
    __syncthreads();
    prefix |= sh.digit << sh_;
    mask |= (unsigned)(nb - 1) << sh_;
    __syncthreads();
  }
  const unsigned thr = prefix;        // key of the N-th largest logit
  const unsigned keq = sh.krem;       // how many logits equal to it are kept
  const float M = sh.M, Z = sh.Z;     // written before the radix passes' barriers
  __syncthreads();

  // ---- compaction in index order; dropped mass of the rest ----
  constexpr int E = 4;
  const int tile = nthreads * E;
  unsigned carry_gt = 0, carry_eq = 0;
  float dsum = 0.f;
  for (int base = 0; base < t; base += tile) {
    unsigned u[E];
    float sv[E];
    unsigned cgt = 0, ceq = 0;
#pragma unroll
    for (int e = 0; e < E; e++) {
      const int i = base + tid * E + e;
      sv[e] = i < t ? sp[i] : -INFINITY;
      u[e] = i < t ? order_key(sv[e]) : 0u;
      cgt += u[e] > thr;
      ceq += (i < t) && u[e] == thr;
    }
    unsigned tot;
    const unsigned packed = (cgt << 16) | ceq;
    const unsigned incl = block_inclusive_scan(packed, sh.scan, tot);
    const unsigned excl = incl - packed;
    unsigned gt_before = carry_gt + (excl >> 16);
    unsigned eq_before = carry_eq + (excl & 0xffffu);
#pragma unroll
    for (int e = 0; e < E; e++) {
      const int i = base + tid * E + e;
      if (i >= t) break;
      bool take = false;
      int pos = 0;
      if (u[e] > thr) {
        take = true;
        pos = (int)(gt_before + min(eq_before, keq));
        gt_before++;
      } else if (u[e] == thr) {
        if (eq_before < keq) {
          take = true;
          pos = (int)(gt_before + eq_before);
        }
        eq_before++;
      }
      if (take) {
        if (pos < Nb) {
          out[pos] = i;
          if (aout) aout[pos] = i;
        } else {
          raise_error(kv.err, PRHS_DEV_CAPACITY);
        }
      } else {
        dsum += expf(sv[e] - M);
      }
    }
    carry_gt += tot >> 16;
    carry_eq += tot & 0xffffu;
  }
  dsum = warp_sum(dsum);
  if (lane == 0) sh.red_z[warp] = dsum;
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
    for (int w = 0; w < (nthreads >> 5); w++) tot += sh.red_z[w];
    a.n_sel[qh] = Nb;
    a.delta[qh] = tot / Z;
    if (a.anchor_n) a.anchor_n[qh] = Nb;
  }
  if (a.q_anchor) copy_query<T>(a, qh);
}

cudaError_t launch_score(const ScoreLaunch& a, const CUtensorMap* tmap, cudaStream_t st) {
  const int G = a.kv.Hq / a.kv.Hkv;
  if (a.kv.dtype == PRHS_BF16) {
    if (a.kv.d == 128) return score_dispatch_g<__nv_bfloat16, 128>(a, tmap, G, st);
    if (a.kv.d == 64) return score_dispatch_g<__nv_bfloat16, 64>(a, tmap, G, st);
  } else {
    if (a.kv.d == 128) return score_dispatch_g<float, 128>(a, tmap, G, st);
    if (a.kv.d == 64) return score_dispatch_g<float, 64>(a, tmap, G, st);
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_select_global(const SelectLaunch& a, cudaStream_t st) {
  const size_t smem = (size_t)min(a.kv.t_max, SELECT_CACHE_FLOATS) * sizeof(float);
  void (*k)(const SelectLaunch) = a.kv.dtype == PRHS_BF16 ? select_kernel<__nv_bfloat16>
                                                          : select_kernel<float>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(a.kv.B * a.kv.Hq), dim3(SELECT_THREADS), smem, st, a.kv.pdl, a);
}

}  // namespace prhs
