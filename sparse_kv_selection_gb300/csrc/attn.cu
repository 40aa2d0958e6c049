// Decode attention over a selected index set (sparse) or over the whole
// cache (dense baseline), split over CTAs with equal row counts.
// "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference":
// the Table V caption's sparse-attention kernel over the selected KV entries,
// and Table IV's dense ("Flash") operator as the baseline.
//
// Work split. A unit is a query head (sparse) or a KV head with its G query
// heads (dense); unit u owns rows(u) rows (n_sel or t_b). Every CTA reads
// all rows(u), forms their prefix sums P and takes rows [c*per, (c+1)*per)
// of the concatenation, per = max(ceil(total / CTAs), ATTN_MIN_ROWS): each
// CTA gets the same number of rows whatever the mix of set sizes (small
// batches leave the surplus CTAs idle), and a CTA may cover the end of one
// unit and the start of the next. A unit covered by one CTA is written
// directly; otherwise each covering CTA writes a partial softmax state into
// slot c + u and the last one to arrive (atomic ticket, no waiting) merges
// them, with all its threads at once, into out and lse and resets the ticket.
//
// Gather. Eight lanes share a row: lane j reads 16-byte chunks j, j+8, ... of
// the K and V rows (128 contiguous bytes per 8 lanes per load), so every
// gathered row arrives as full cache lines. A warp keeps 4 rows per step and
// several steps in flight; the row numbers of a segment are staged in shared
// memory first. Softmax is online in fp32 and base 2 (logits pre-scaled by
// log2 e). Units are query heads in both kernels; the kernel template can
// also give one unit the G query heads of a KV head (registers per thread
// grow with G, which costs more occupancy than the L2 re-reads it saves).
//
// Logit source (LG). After a fresh selection the logits of every key are
// still in the workspace: the retrieving heads' attention then reads each
// selected row's logit (4 bytes) and its V row only, not its K row.
#include <type_traits>

#include "kernels.h"

namespace prhs {

constexpr int ATTN_THREADS = 128;
constexpr int ATTN_IDX_STAGE = 2048;
constexpr int MERGE_CH = 32;  // partial records merged per shared-memory pass
constexpr int ATTN_ALIGN_UNITS = 2048;  // most units for the unit-aligned split
constexpr int ATTN_PB = 8;  // units whose counts a thread loads at once

// Slot of unit u in the per-unit prefix arrays: one spare word after every 32,
// so that threads owning runs of 2, 4, 8, 16 or 32 consecutive units reach 32
// different banks.
__host__ __device__ __forceinline__ int attn_sk(int u) { return u + (u >> 5); }

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}
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

template <int CPL, int G>
struct AttnUnroll {
  static constexpr int base = G <= 2 ? 4 : (G == 4 ? 2 : 1);
  static constexpr int value = CPL >= 4 ? (base > 1 ? base / 2 : 1) : base;
};

// Merge two online-softmax states (m, l, o) in base 2.
__device__ __forceinline__ void merge_coeffs(float m1, float m2, float& M, float& c1, float& c2) {
  M = fmaxf(m1, m2);
  c1 = M == -INFINITY ? 0.f : exp2f(m1 - M);
  c2 = M == -INFINITY ? 0.f : exp2f(m2 - M);
}

template <typename T, int D, int G, bool SPARSE, bool LG>
__global__ void __launch_bounds__(ATTN_THREADS, LG ? ATTN_LG_CTAS_PER_SM : 4) attn_kernel(const AttnLaunch a) {
  using S = AttnShape<T, D>;
  static_assert(!LG || (SPARSE && G == 1), "logit source: sparse, one query head per unit");
  constexpr int PW = D + 4;          // partial record: m, l, 2 pad, o[D] (16-byte aligned)
  static_assert(D <= ATTN_THREADS && D % 64 == 0, "merge maps one thread per output element");
  // one buffer: the row numbers of a segment, or a chunk of partial records
  // while a unit is merged
  constexpr int BUF_FLOATS = (SPARSE && ATTN_IDX_STAGE > MERGE_CH * PW) ? ATTN_IDX_STAGE : MERGE_CH * PW;
  // [units + 1] row prefix, then (aligned split) [units + 1] CTA prefix,
  // both indexed through attn_sk
  extern __shared__ int sh_prefix[];
  __shared__ __align__(16) float sh_buf[BUF_FLOATS];
  int* const sh_idx = reinterpret_cast<int*>(sh_buf);
  __shared__ float sm_m[4][G], sm_l[4][G];
  __shared__ float sm_o[4][G][D];
  __shared__ int sh_wsum[ATTN_THREADS / 32], sh_wact[ATTN_THREADS / 32];
  __shared__ int sh_last;

  pdl_wait();
  pdl_trigger();

  const KVView& kv = a.kv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sg = lane >> 3, j = lane & 7;
  // units are query heads unless G query heads share one dense unit
  constexpr bool PER_QUERY = SPARSE || G == 1;
  const int U = PER_QUERY ? kv.B * kv.Hq : kv.B * kv.Hkv;
  const int C = gridDim.x, c = blockIdx.x;
  const int group = kv.Hq / kv.Hkv;

  // Exclusive prefix over units of per-unit counts: thread tid owns units
  // [u0, u0 + per_t), whose counts are in arr[] on entry; also returns the
  // number of units with a non-zero count. Ends with a barrier.
  const int per_t = (U + ATTN_THREADS - 1) / ATTN_THREADS;
  const int u0 = tid * per_t;
  auto block_scan = [&](int* arr, int loc, int act) -> int {
    int v = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, v, o);
      if (lane >= o) v += y;
    }
    act = warp_sum_int(act);
    if (lane == 31) sh_wsum[warp] = v;
    if (lane == 0) sh_wact[warp] = act;
    __syncthreads();
    int before = 0, nact = 0;
    for (int w = 0; w < ATTN_THREADS / 32; w++) {
      if (w < warp) before += sh_wsum[w];
      nact += sh_wact[w];
    }
    int run = before + v - loc;
    for (int k = 0; k < per_t; k++) {
      const int u = u0 + k;
      if (u >= U) break;
      const int r = arr[attn_sk(u)];
      arr[attn_sk(u)] = run;
      run += r;
    }
    if (tid == ATTN_THREADS - 1) arr[attn_sk(U)] = run;
    __syncthreads();
    return nact;
  };

  // ---- rows per unit and their prefix sums (every CTA computes the same) ----
  int nact;
  {
    // ATTN_PB units per batch, all their loads issued before any is used (one
    // round trip per batch instead of two dependent ones per unit)
    int loc = 0, act = 0;
    for (int k0 = 0; k0 < per_t; k0 += ATTN_PB) {
      int cnt[ATTN_PB];
      bool skip[ATTN_PB];
#pragma unroll
      for (int i = 0; i < ATTN_PB; i++) {
        const int u = u0 + k0 + i;
        const bool in = k0 + i < per_t && u < U;
        cnt[i] = !in ? 0 : SPARSE ? __ldg(a.n_sel + u) : __ldg(kv.seq_lens + (PER_QUERY ? u / kv.Hq : u / kv.Hkv));
        // another launch attends the units the mask leaves out
        skip[i] = SPARSE && in && a.unit_mask != nullptr &&
                  (__ldg(a.unit_mask + u) != 0) != (a.mask_want != 0);
      }
#pragma unroll
      for (int i = 0; i < ATTN_PB; i++) {
        const int u = u0 + k0 + i;
        if (k0 + i >= per_t || u >= U) break;
        int r = cnt[i];
        if (!SPARSE) {
          r = checked_len(kv, r);
        } else if (skip[i]) {
          r = 0;
        } else if (r < 0 || r > a.cap) {
          raise_error(kv.err, PRHS_DEV_CAPACITY);
          r = r < 0 ? 0 : a.cap;
        }
        sh_prefix[attn_sk(u)] = r;  // temporarily the count
        loc += r;
        act += r > 0;
      }
    }
    nact = block_scan(sh_prefix, loc, act);
  }
  const int total = sh_prefix[attn_sk(U)];

  // ---- units with no rows: out = 0, lse = -inf ----
  for (int u = c; u < U; u += C) {
    if (sh_prefix[attn_sk(u + 1)] != sh_prefix[attn_sk(u)]) continue;
    if (SPARSE && a.unit_mask != nullptr && (a.unit_mask[u] != 0) != (a.mask_want != 0)) continue;
    const int qh0 = PER_QUERY ? u : (u / kv.Hkv) * kv.Hq + (u % kv.Hkv) * G;
    for (int x = tid; x < G * D; x += ATTN_THREADS) {
      a.out[(long long)(qh0 + x / D) * D + x % D] = 0.f;
      if (x % D == 0) a.lse[qh0 + x / D] = -INFINITY;
    }
  }
  if (total == 0) return;

  // ---- the split ----
  // Aligned (few active units): every CTA takes rows of one unit only, unit u
  // getting ceil(rows_u / per) CTAs with its rows shared evenly; with per =
  // ceil(total / (C - nact)) those counts add up to at most C. Otherwise the
  // concatenated rows are cut into C equal ranges, and a CTA may cover the
  // end of one unit and the start of the next.
  const int min_rows = max(a.min_rows, 1);
  const bool aligned = U <= ATTN_ALIGN_UNITS && 2 * nact <= C;
  int per;
  int* const sh_cpre = sh_prefix + attn_sk(U) + 1;
  if (aligned) {
    per = max(min_rows, (total + (C - nact) - 1) / (C - nact));
    int loc = 0;
    for (int k = 0; k < per_t; k++) {
      const int u = u0 + k;
      if (u >= U) break;
      const int n = (sh_prefix[attn_sk(u + 1)] - sh_prefix[attn_sk(u)] + per - 1) / per;
      sh_cpre[attn_sk(u)] = n;
      loc += n;
    }
    block_scan(sh_cpre, loc, 0);
  } else {
    per = max((total + C - 1) / C, min_rows);
  }

  const char* kbase = static_cast<const char*>(kv.k);
  const char* vbase = static_cast<const char*>(kv.v);
  const float qscale = a.scale * LOG2E;

  // Rows [r0, r1) of unit u, one of the CTAs cf..cl that cover it.
  auto process = [&](const int u, const int r0, const int r1, const int cf, const int cl) {
    int b, kvh, qh0;
    if (PER_QUERY) {
      b = u / kv.Hq;
      qh0 = u;
      kvh = (u % kv.Hq) / group;
    } else {
      b = u / kv.Hkv;
      kvh = u % kv.Hkv;
      qh0 = b * kv.Hq + kvh * G;
    }
    const int t = seq_len(kv, b);

    // the query's 16-byte pieces and the first segment's row numbers are
    // requested together
    uint4 qraw[G][S::CPL];
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
      for (int cc = 0; cc < S::CPL; cc++)
        qraw[g][cc] = LG ? make_uint4(0, 0, 0, 0)
                         : __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.q) +
                                                                ((long long)(qh0 + g) * D) * sizeof(T)) +
                                 cc * 8 + j);
    const float* lrow = LG ? a.logits + (long long)u * kv.t_max : nullptr;
    const int32_t* rows = SPARSE ? a.idx + (long long)u * a.cap : nullptr;
    if (SPARSE) {
      __syncthreads();  // earlier readers of the buffer are done
      const int se0 = min(r1, r0 + ATTN_IDX_STAGE);
      for (int x = tid; x < se0 - r0; x += ATTN_THREADS) sh_idx[x] = rows[r0 + x];
      __syncthreads();
    }
    float qf[G][S::EL];
#pragma unroll
    for (int g = 0; g < G; g++) {
#pragma unroll
      for (int cc = 0; cc < S::CPL; cc++) Elem<T>::unpack(qraw[g][cc], qf[g] + cc * S::EPC);
#pragma unroll
      for (int e = 0; e < S::EL; e++) qf[g][e] *= qscale;
    }
    float m[G], l[G], o[G][S::EL];
#pragma unroll
    for (int g = 0; g < G; g++) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int e = 0; e < S::EL; e++) o[g][e] = 0.f;
    }

    // Rows [sb, se) of the staged segment, weights from K (LGU false) or
    // from the logits (LGU true); UR rows per lane group in flight. One body
    // per weight source, so each keeps its loads together. (The V-only form
    // runs ATTN_LG_CTAS_PER_SM CTAs per SM at the same UR: more warps hide
    // its short chains better than twice the rows per warp at four CTAs.)
    auto run_rows = [&](auto lg_tag, const int sb, const int se) {
      constexpr bool LGU = decltype(lg_tag)::value;
      constexpr int UR = AttnUnroll<S::CPL, G>::value;
      for (int base = sb; base < se; base += 16 * UR) {
        long long row[UR];
        int keyv[UR];
#pragma unroll
        for (int uu = 0; uu < UR; uu++) {
          const int r = base + uu * 16 + warp * 4 + sg;
          row[uu] = -1;
          keyv[uu] = 0;
          if (r < se) {
            const int key = SPARSE ? sh_idx[r - sb] : r;
            if ((unsigned)key < (unsigned)t) {
              row[uu] = kv_row(kv, b, kvh, key);
              keyv[uu] = key;
              if (row[uu] < 0) raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
            } else {
              raise_error(kv.err, PRHS_DEV_BAD_INDEX);
            }
          }
        }
        uint4 kc[LGU ? 1 : UR][S::CPL], vc[UR][S::CPL];
        float lg[LGU ? UR : 1];
#pragma unroll
        for (int uu = 0; uu < UR; uu++) {
          if constexpr (LGU) lg[uu] = row[uu] >= 0 ? __ldg(lrow + keyv[uu]) : 0.f;
#pragma unroll
          for (int cc = 0; cc < S::CPL; cc++) {
            if (row[uu] >= 0) {
              if constexpr (!LGU) kc[uu][cc] = ldg_stream(kbase + row[uu] * S::RB + (cc * 8 + j) * 16);
              vc[uu][cc] = ldg_stream(vbase + row[uu] * S::RB + (cc * 8 + j) * 16);
            } else {
              if constexpr (!LGU) kc[uu][cc] = make_uint4(0, 0, 0, 0);
              vc[uu][cc] = make_uint4(0, 0, 0, 0);
            }
          }
        }
        float s[UR][G];
#pragma unroll
        for (int uu = 0; uu < UR; uu++) {
          if constexpr (LGU) {
            s[uu][0] = row[uu] >= 0 ? lg[uu] * LOG2E : -INFINITY;
          } else {
            float kf[S::EL];
#pragma unroll
            for (int cc = 0; cc < S::CPL; cc++) Elem<T>::unpack(kc[uu][cc], kf + cc * S::EPC);
#pragma unroll
            for (int g = 0; g < G; g++) {
              float acc = 0.f;
#pragma unroll
              for (int e = 0; e < S::EL; e++) acc = fmaf(qf[g][e], kf[e], acc);
              acc += __shfl_xor_sync(FULL_MASK, acc, 1);
              acc += __shfl_xor_sync(FULL_MASK, acc, 2);
              acc += __shfl_xor_sync(FULL_MASK, acc, 4);
              s[uu][g] = row[uu] >= 0 ? acc : -INFINITY;
            }
          }
        }
        float vf[UR][S::EL];
#pragma unroll
        for (int uu = 0; uu < UR; uu++)
#pragma unroll
          for (int cc = 0; cc < S::CPL; cc++) Elem<T>::unpack(vc[uu][cc], vf[uu] + cc * S::EPC);
#pragma unroll
        for (int g = 0; g < G; g++) {
          float mx = m[g];
#pragma unroll
          for (int uu = 0; uu < UR; uu++) mx = fmaxf(mx, s[uu][g]);
          if (mx == -INFINITY) continue;
          const float corr = exp2f(m[g] - mx);
          l[g] *= corr;
#pragma unroll
          for (int e = 0; e < S::EL; e++) o[g][e] *= corr;
#pragma unroll
          for (int uu = 0; uu < UR; uu++) {
            const float p = exp2f(s[uu][g] - mx);
            l[g] += p;
#pragma unroll
            for (int e = 0; e < S::EL; e++) o[g][e] = fmaf(p, vf[uu][e], o[g][e]);
          }
          m[g] = mx;
        }
      }
    };

    for (int sb = r0; sb < r1; sb += (SPARSE ? ATTN_IDX_STAGE : (r1 - r0))) {
      const int se = SPARSE ? min(r1, sb + ATTN_IDX_STAGE) : r1;
      if (SPARSE && sb != r0) {
        __syncthreads();
        for (int x = tid; x < se - sb; x += ATTN_THREADS) sh_idx[x] = rows[sb + x];
        __syncthreads();
      }
      run_rows(std::integral_constant<bool, LG>{}, sb, se);
    }

    // ---- merge the 4 row groups of each warp, then the 4 warps ----
#pragma unroll
    for (int g = 0; g < G; g++) {
#pragma unroll
      for (int off = 8; off <= 16; off <<= 1) {
        const float m2 = __shfl_xor_sync(FULL_MASK, m[g], off);
        const float l2 = __shfl_xor_sync(FULL_MASK, l[g], off);
        float M, c1, c2;
        merge_coeffs(m[g], m2, M, c1, c2);
        l[g] = l[g] * c1 + l2 * c2;
#pragma unroll
        for (int e = 0; e < S::EL; e++) {
          const float o2 = __shfl_xor_sync(FULL_MASK, o[g][e], off);
          o[g][e] = o[g][e] * c1 + o2 * c2;
        }
        m[g] = M;
      }
    }
    __syncthreads();  // shared state of the previous segment fully consumed
    if (lane < 8) {
#pragma unroll
      for (int g = 0; g < G; g++) {
        if (lane == 0) {
          sm_m[warp][g] = m[g];
          sm_l[warp][g] = l[g];
        }
#pragma unroll
        for (int cc = 0; cc < S::CPL; cc++)
#pragma unroll
          for (int e = 0; e < S::EPC; e++)
            sm_o[warp][g][(cc * 8 + j) * S::EPC + e] = o[g][cc * S::EPC + e];
      }
    }
    __syncthreads();

    if (cf == cl) {
      // the whole unit is in this CTA: final result
      for (int x = tid; x < G * D; x += ATTN_THREADS) {
        const int g = x / D, e = x % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; w++) M = fmaxf(M, sm_m[w][g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < 4; w++) {
            const float cw = exp2f(sm_m[w][g] - M);
            L += cw * sm_l[w][g];
            O += cw * sm_o[w][g][e];
          }
        }
        a.out[(long long)(qh0 + g) * D + e] = L > 0.f ? O / L : 0.f;
        if (e == 0) a.lse[qh0 + g] = L > 0.f ? (M + log2f(L)) * LN2 : -INFINITY;
      }
      return;
    }
    for (int x = tid; x < G * D; x += ATTN_THREADS) {
      const int g = x / D, e = x % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; w++) M = fmaxf(M, sm_m[w][g]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 4; w++) {
          const float cw = exp2f(sm_m[w][g] - M);
          L += cw * sm_l[w][g];
          O += cw * sm_o[w][g][e];
        }
      }
      float* rec = a.partials + ((long long)(c + u) * G + g) * PW;
      rec[4 + e] = O;
      if (e == 0) {
        rec[0] = M;
        rec[1] = L;
      }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) sh_last = atomicAdd(&a.counters[u], 1u) == (unsigned)(cl - cf);
    __syncthreads();
    if (!sh_last) return;
    __threadfence();
    // Merge the ncov partial records of this unit: chunks of MERGE_CH records
    // are copied to shared memory by the whole block in one pass (16-byte
    // loads, all independent), then folded into a running (M, L, O) state,
    // thread e owning output element e.
    const int ncov = cl - cf + 1;
    constexpr int V4 = PW / 4;  // 16-byte pieces per record
    for (int g = 0; g < G; g++) {
      const float* rec0 = a.partials + ((long long)(cf + u) * G + g) * PW;
      const long long RS = (long long)G * PW;  // floats between consecutive records
      float M = -INFINITY, L = 0.f, O = 0.f;
      for (int i0 = 0; i0 < ncov; i0 += MERGE_CH) {
        const int nb = min(MERGE_CH, ncov - i0);
        __syncthreads();  // the buffer is free
        for (int x = tid; x < nb * V4; x += ATTN_THREADS) {
          const int i = x / V4, k = x % V4;
          reinterpret_cast<float4*>(sh_buf)[x] =
              __ldcg(reinterpret_cast<const float4*>(rec0 + (i0 + i) * RS) + k);
        }
        __syncthreads();
        float mc = M;
        for (int i = 0; i < nb; i++) mc = fmaxf(mc, sh_buf[i * PW]);
        if (mc != -INFINITY) {
          const float r = exp2f(M - mc);  // 0 while M is still -inf
          L *= r;
          O *= r;
          for (int i = 0; i < nb; i++) {
            const float wgt = exp2f(sh_buf[i * PW] - mc);
            L = fmaf(wgt, sh_buf[i * PW + 1], L);
            if (tid < D) O = fmaf(wgt, sh_buf[i * PW + 4 + tid], O);
          }
          M = mc;
        }
      }
      if (tid < D) {
        a.out[(long long)(qh0 + g) * D + tid] = L > 0.f ? O / L : 0.f;
        if (tid == 0) a.lse[qh0 + g] = L > 0.f ? (M + log2f(L)) * LN2 : -INFINITY;
      }
    }
    if (tid == 0) a.counters[u] = 0u;
  };

  if (aligned) {
    if (c >= sh_cpre[attn_sk(U)]) return;  // more CTAs than the split needs
    int ulo = 0, uhi = U - 1;     // the unit: largest u with CP[u] <= c
    while (ulo < uhi) {
      const int mid = (ulo + uhi + 1) >> 1;
      if (sh_cpre[attn_sk(mid)] <= c) ulo = mid; else uhi = mid - 1;
    }
    const int cf = sh_cpre[attn_sk(ulo)], n = sh_cpre[attn_sk(ulo + 1)] - cf, k = c - cf;
    const int ru = sh_prefix[attn_sk(ulo + 1)] - sh_prefix[attn_sk(ulo)];
    process(ulo, (int)((long long)k * ru / n), (int)((long long)(k + 1) * ru / n), cf, cf + n - 1);
    return;
  }
  const int lo = c * per, hi = min(total, lo + per);
  if (lo >= hi) return;
  // first unit with rows overlapping [lo, hi): largest u with P[u] <= lo
  int ulo = 0, uhi = U - 1;
  while (ulo < uhi) {
    const int mid = (ulo + uhi + 1) >> 1;
    if (sh_prefix[attn_sk(mid)] <= lo) ulo = mid; else uhi = mid - 1;
  }
  for (int u = ulo; u < U && sh_prefix[attn_sk(u)] < hi; u++) {
    const int P0 = sh_prefix[attn_sk(u)], P1 = sh_prefix[attn_sk(u + 1)];
    const int r0 = max(lo, P0) - P0, r1 = min(hi, P1) - P0;
    if (r0 < r1) process(u, r0, r1, P0 / per, (P1 - 1) / per);
  }
}

// Units are query heads, sparse or dense (the dense path here serves one
// query head per KV head; grouped heads go to the TMA dense kernel).
int attn_units(const KVView& kv, bool sparse) { (void)sparse; return kv.B * kv.Hq; }

size_t attn_partial_floats(const KVView& kv, bool sparse, int ctas) {
  return ((size_t)ctas + attn_units(kv, sparse)) * (kv.d + 4);
}

template <typename T, int D, int G, bool SPARSE, bool LG>
static cudaError_t attn_go(const AttnLaunch& a, cudaStream_t st) {
  const size_t units = (size_t)attn_units(a.kv, SPARSE);
  const size_t smem = ((size_t)attn_sk((int)units) + 1) * sizeof(int) * (units <= (size_t)ATTN_ALIGN_UNITS ? 2 : 1);
  auto k = attn_kernel<T, D, G, SPARSE, LG>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(k, dim3(a.ctas), dim3(ATTN_THREADS), smem, st, a.kv.pdl, a);
}

template <typename T, int D>
static cudaError_t attn_dispatch(const AttnLaunch& a, bool sparse, cudaStream_t st) {
  if (sparse && a.logits != nullptr) return attn_go<T, D, 1, true, true>(a, st);
  if (sparse) return attn_go<T, D, 1, true, false>(a, st);
  return attn_go<T, D, 1, false, false>(a, st);
}

cudaError_t launch_attn(const AttnLaunch& a, bool sparse, cudaStream_t st) {
  if (sparse && a.cluster > 0) return launch_attn_cluster(a, st);
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
