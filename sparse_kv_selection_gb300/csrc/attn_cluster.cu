// Sparse decode attention for batches with few query heads: one
// thread-block cluster of CL CTAs per query head.
// "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference":
// the Table V caption's sparse-attention kernel over the selected KV entries.
//
// CTA r of the cluster of head u takes the selected positions r, r + CL,
// r + 2 CL, ... of that head's index row. Because the positions do not depend
// on the set size, the CTA requests the set size, its query and its first
// segment of row numbers (read up to the row capacity, the entries past the
// set size ignored) in one round trip. The gather is the one of the balanced
// kernel: eight lanes per row, 16-byte streaming loads, fp32 online softmax
// in base 2. Each CTA folds its four warps into one partial state (m, l, o)
// and stores it into CTA 0's shared memory through distributed shared
// memory; after one cluster barrier CTA 0 merges the CL states from its own
// shared memory and writes out and lse. No workspace and no global-memory
// round trip take part in the merge. With a logit source (LG: the logits
// the scoring kernel left in the workspace, after a fresh selection) a row
// costs its 4-byte logit and its V row; its K row is not read.
#include <cooperative_groups.h>

#include "kernels.h"

namespace cg = cooperative_groups;

namespace prhs {

constexpr int ACL_THREADS = 256;  // 8 warps: 32 rows per step in flight per CTA
constexpr int ACL_WARPS = ACL_THREADS / 32;
constexpr int ACL_STAGE = 2048;  // row numbers staged in shared memory at a time
constexpr float ACL_LOG2E = 1.4426950408889634f;
constexpr float ACL_LN2 = 0.6931471805599453f;

template <typename T, int D, bool LG>
__global__ void __launch_bounds__(ACL_THREADS, 2) attn_cluster_kernel(const AttnLaunch a) {
  constexpr int RB = D * (int)sizeof(T);  // bytes per row
  constexpr int CPL = RB / 16 / 8;        // 16-byte chunks per lane
  constexpr int EPC = 16 / (int)sizeof(T);
  constexpr int EL = CPL * EPC;           // elements per lane
  constexpr int UP = (CPL >= 4 ? 1 : 2) * (LG ? 2 : 1);  // rows per 8-lane group per batch
  constexpr int STEP = 4 * ACL_WARPS * UP;       // rows per batch per CTA
  static_assert(RB % 128 == 0 && D <= ACL_THREADS, "row of whole 128-byte lines, one thread per output");
  __shared__ int sh_idx[ACL_STAGE];
  __shared__ float sm_m[ACL_WARPS], sm_l[ACL_WARPS];
  __shared__ float sm_o[ACL_WARPS][D];
  __shared__ float part[ATTN_CLUSTER_MAX][D + 2];  // CTA 0: every CTA's state m, l, o[D]

  pdl_wait();
  pdl_trigger();

  const KVView& kv = a.kv;
  const int CL = gridDim.x, rank = blockIdx.x, u = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sg = lane >> 3, j = lane & 7;
  // uniform over the cluster: every CTA of it has the same u
  if (a.unit_mask != nullptr && (a.unit_mask[u] != 0) != (a.mask_want != 0)) return;
  const int b = u / kv.Hq;
  const int kvh = (u % kv.Hq) / (kv.Hq / kv.Hkv);

  // ---- one round trip: set size, query, first segment of row numbers ----
  int n = a.n_sel[u];
  const int t = seq_len(kv, b);
  uint4 qraw[CPL];
#pragma unroll
  for (int cc = 0; cc < CPL; cc++)
    qraw[cc] = LG ? make_uint4(0, 0, 0, 0)
                  : __ldg(reinterpret_cast<const uint4*>(static_cast<const char*>(a.q) + (long long)u * RB) +
                          cc * 8 + j);
  const float* lrow = LG ? a.logits + (long long)u * kv.t_max : nullptr;
  const int32_t* rows = a.idx + (long long)u * a.cap;
  const int mine_cap = a.cap > rank ? (a.cap - rank + CL - 1) / CL : 0;
  const int spec = min(ACL_STAGE, mine_cap);
  for (int x = tid; x < spec; x += ACL_THREADS) sh_idx[x] = rows[rank + (long long)CL * x];
  __syncthreads();
  if (n < 0 || n > a.cap) {
    if (tid == 0 && rank == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    n = n < 0 ? 0 : a.cap;
  }
  if (n == 0) {  // uniform over the cluster: nothing to attend
    if (rank == 0)
      for (int e = tid; e < D; e += ACL_THREADS) {
        a.out[(long long)u * D + e] = 0.f;
        if (e == 0) a.lse[u] = -INFINITY;
      }
    return;
  }
  const int mine = n > rank ? (n - rank + CL - 1) / CL : 0;  // positions rank + CL * i, i < mine

  const float qscale = a.scale * ACL_LOG2E;
  float qf[EL];
#pragma unroll
  for (int cc = 0; cc < CPL; cc++) Elem<T>::unpack(qraw[cc], qf + cc * EPC);
#pragma unroll
  for (int e = 0; e < EL; e++) qf[e] *= qscale;
  float m = -INFINITY, l = 0.f, o[EL];
#pragma unroll
  for (int e = 0; e < EL; e++) o[e] = 0.f;

  const char* kbase = static_cast<const char*>(kv.k);
  const char* vbase = static_cast<const char*>(kv.v);
  for (int sb = 0; sb < mine; sb += ACL_STAGE) {
    const int se = min(mine, sb + ACL_STAGE);
    if (sb > 0) {
      __syncthreads();
      for (int x = tid; x < se - sb; x += ACL_THREADS) sh_idx[x] = rows[rank + (long long)CL * (sb + x)];
      __syncthreads();
    }
    // Two batches of UP rows per 8-lane group in flight: the loads of the
    // next batch are issued before the current one is consumed, so a CTA
    // never waits a full memory round trip between batches.
    constexpr int UK = LG ? 1 : UP;  // K pieces are kept only when the logits are computed here
    long long rowA[UP], rowB[UP];
    uint4 kA[UK][CPL], vA[UP][CPL], kB[UK][CPL], vB[UP][CPL];
    float lA[UP], lB[UP];
    auto issue = [&](int base, long long (&row)[UP], uint4 (&kc)[UK][CPL], uint4 (&vc)[UP][CPL],
                     float (&lg)[UP]) {
      int keyv[UP];
#pragma unroll
      for (int uu = 0; uu < UP; uu++) {
        const int r = base + uu * 4 * ACL_WARPS + warp * 4 + sg;
        row[uu] = -1;
        keyv[uu] = 0;
        if (r < se) {
          const int key = sh_idx[r - sb];
          if ((unsigned)key < (unsigned)t) {
            row[uu] = kv_row(kv, b, kvh, key);
            keyv[uu] = key;
            if (row[uu] < 0) raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
          } else {
            raise_error(kv.err, PRHS_DEV_BAD_INDEX);
          }
        }
      }
#pragma unroll
      for (int uu = 0; uu < UP; uu++) {
        lg[uu] = LG && row[uu] >= 0 ? __ldg(lrow + keyv[uu]) : 0.f;
#pragma unroll
        for (int cc = 0; cc < CPL; cc++) {
          if (row[uu] >= 0) {
            if (!LG) kc[LG ? 0 : uu][cc] = ldg_stream(kbase + row[uu] * RB + (cc * 8 + j) * 16);
            vc[uu][cc] = ldg_stream(vbase + row[uu] * RB + (cc * 8 + j) * 16);
          } else {
            if (!LG) kc[LG ? 0 : uu][cc] = make_uint4(0, 0, 0, 0);
            vc[uu][cc] = make_uint4(0, 0, 0, 0);
          }
        }
      }
    };
    auto consume = [&](const long long (&row)[UP], const uint4 (&kc)[UK][CPL],
                       const uint4 (&vc)[UP][CPL], const float (&lg)[UP]) {
      float s[UP];
#pragma unroll
      for (int uu = 0; uu < UP; uu++) {
        if (LG) {
          s[uu] = row[uu] >= 0 ? lg[uu] * ACL_LOG2E : -INFINITY;
          continue;
        }
        float kf[EL];
#pragma unroll
        for (int cc = 0; cc < CPL; cc++) Elem<T>::unpack(kc[LG ? 0 : uu][cc], kf + cc * EPC);
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EL; e++) acc = fmaf(qf[e], kf[e], acc);
        acc += __shfl_xor_sync(FULL_MASK, acc, 1);
        acc += __shfl_xor_sync(FULL_MASK, acc, 2);
        acc += __shfl_xor_sync(FULL_MASK, acc, 4);
        s[uu] = row[uu] >= 0 ? acc : -INFINITY;
      }
      float mx = m;
#pragma unroll
      for (int uu = 0; uu < UP; uu++) mx = fmaxf(mx, s[uu]);
      if (mx == -INFINITY) return;
      const float corr = exp2f(m - mx);
      l *= corr;
#pragma unroll
      for (int e = 0; e < EL; e++) o[e] *= corr;
#pragma unroll
      for (int uu = 0; uu < UP; uu++) {
        float vf[EL];
#pragma unroll
        for (int cc = 0; cc < CPL; cc++) Elem<T>::unpack(vc[uu][cc], vf + cc * EPC);
        const float p = exp2f(s[uu] - mx);
        l += p;
#pragma unroll
        for (int e = 0; e < EL; e++) o[e] = fmaf(p, vf[e], o[e]);
      }
      m = mx;
    };
    issue(sb, rowA, kA, vA, lA);
    for (int base = sb; base < se; base += 2 * STEP) {  // uniform over the CTA
      const bool more = base + STEP < se;
      if (more) issue(base + STEP, rowB, kB, vB, lB);
      consume(rowA, kA, vA, lA);
      if (!more) break;
      if (base + 2 * STEP < se) issue(base + 2 * STEP, rowA, kA, vA, lA);
      consume(rowB, kB, vB, lB);
    }
  }

  // ---- this CTA's state: the 4 row groups of each warp, then the warps ----
#pragma unroll
  for (int off = 8; off <= 16; off <<= 1) {
    const float m2 = __shfl_xor_sync(FULL_MASK, m, off);
    const float l2 = __shfl_xor_sync(FULL_MASK, l, off);
    const float M = fmaxf(m, m2);
    const float c1 = M == -INFINITY ? 0.f : exp2f(m - M);
    const float c2 = M == -INFINITY ? 0.f : exp2f(m2 - M);
    l = l * c1 + l2 * c2;
#pragma unroll
    for (int e = 0; e < EL; e++) {
      const float o2 = __shfl_xor_sync(FULL_MASK, o[e], off);
      o[e] = o[e] * c1 + o2 * c2;
    }
    m = M;
  }
  if (lane < 8) {
    if (lane == 0) {
      sm_m[warp] = m;
      sm_l[warp] = l;
    }
#pragma unroll
    for (int cc = 0; cc < CPL; cc++)
#pragma unroll
      for (int e = 0; e < EPC; e++) sm_o[warp][(cc * 8 + j) * EPC + e] = o[cc * EPC + e];
  }
  __syncthreads();
  if (tid < D) {
    float M = sm_m[0];
#pragma unroll
    for (int w = 1; w < ACL_WARPS; w++) M = fmaxf(M, sm_m[w]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < ACL_WARPS; w++) {
        const float cw = exp2f(sm_m[w] - M);
        L += cw * sm_l[w];
        O += cw * sm_o[w][tid];
      }
    }
    if (CL == 1) {
      a.out[(long long)u * D + tid] = L > 0.f ? O / L : 0.f;
      if (tid == 0) a.lse[u] = L > 0.f ? (M + log2f(L)) * ACL_LN2 : -INFINITY;
    } else {
      // this CTA's state into row `rank` of CTA 0's table
      cg::cluster_group cluster = cg::this_cluster();
      float* dst = cluster.map_shared_rank(&part[0][0], 0) + rank * (D + 2);
      dst[2 + tid] = O;
      if (tid == 0) {
        dst[0] = M;
        dst[1] = L;
      }
    }
  }
  if (CL == 1) return;

  // ---- CTA 0 merges the cluster's states from its own shared memory ----
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();  // every CTA's stores into CTA 0 are visible
  if (rank == 0 && tid < D) {
    float M = -INFINITY;
    for (int r = 0; r < CL; r++) M = fmaxf(M, part[r][0]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int r = 0; r < CL; r++) {
        const float cw = exp2f(part[r][0] - M);
        L += cw * part[r][1];
        O += cw * part[r][2 + tid];
      }
    }
    a.out[(long long)u * D + tid] = L > 0.f ? O / L : 0.f;
    if (tid == 0) a.lse[u] = L > 0.f ? (M + log2f(L)) * ACL_LN2 : -INFINITY;
  }
}

template <typename T, int D>
static cudaError_t cluster_go(const AttnLaunch& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.cluster, a.kv.B * a.kv.Hq);
  cfg.blockDim = dim3(ACL_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a.cluster == 1 ? attr + 1 : attr;
  cfg.numAttrs = (a.cluster == 1 ? 0 : 1) + (a.kv.pdl ? 1 : 0);
  if (a.logits != nullptr) return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<T, D, true>, a);
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<T, D, false>, a);
}

cudaError_t launch_attn_cluster(const AttnLaunch& a, cudaStream_t st) {
  if (a.cluster < 1 || a.cluster > ATTN_CLUSTER_MAX) return cudaErrorInvalidValue;
  if (a.kv.dtype == PRHS_BF16) {
    if (a.kv.d == 128) return cluster_go<__nv_bfloat16, 128>(a, st);
    if (a.kv.d == 64) return cluster_go<__nv_bfloat16, 64>(a, st);
  } else {
    if (a.kv.d == 128) return cluster_go<float, 128>(a, st);
    if (a.kv.d == 64) return cluster_go<float, 64>(a, st);
  }
  return cudaErrorNotSupported;
}

}  // namespace prhs
