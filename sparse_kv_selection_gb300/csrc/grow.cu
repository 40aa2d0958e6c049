// Decode on a growing cache with forced keys.
// "Near-Oracle KV Selection via Pre-hoc Sparsity for Long-Context Inference":
// Fig. 11 (attention sinks and the most recent positions take attention mass
// for every query), read as a deterministic set that every query attends on
// top of its selected or shared keys, while the cache gains one key per
// decode query.
//
// compose_kernel: the attended set of a retrieving head = the first n_sink
// keys, the head's middle top-N set (kept in its anchor row by selection,
// which ranks only the keys between the forced ones), and the last `window`
// keys; ascending because the three ranges are disjoint and ordered.
// append_kernel: one CTA per sequence writes its new key and value rows for
// every KV head at position seq_lens[b] in 16-byte pieces (all loads of a
// thread issued before its stores), then advances seq_lens[b].
#include "kernels.h"

namespace prhs {

constexpr int GROW_THREADS = 128;

__global__ void __launch_bounds__(GROW_THREADS) compose_kernel(const ComposeLaunch a) {
  pdl_wait();
  pdl_trigger();
  const KVView& kv = a.kv;
  const int qh = blockIdx.x, b = qh / kv.Hq;
  if (a.head_skip != nullptr && a.head_skip[qh] != 0) return;
  const int t = seq_len(kv, b);
  const int ns = min(max(a.n_sink, 0), t);
  const int we = max(ns, t - max(a.window, 0));
  int nm = a.anchor_n[qh];
  if (nm < 0 || nm > a.anchor_cap || nm > we - ns) {
    if (threadIdx.x == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    nm = max(0, min(nm, min(a.anchor_cap, we - ns)));
  }
  const int total = ns + nm + (t - we);
  if (total > a.cap && threadIdx.x == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
  const int32_t* mid = a.anchor_idx + (long long)qh * a.anchor_cap;
  int32_t* out = a.idx + (long long)qh * a.cap;
  for (int p = threadIdx.x; p < min(total, a.cap); p += GROW_THREADS) {
    int key;
    if (p < ns) key = p;
    else if (p < ns + nm) key = mid[p - ns];
    else key = we + (p - ns - nm);
    out[p] = key;
  }
  if (threadIdx.x == 0) a.n_sel[qh] = min(total, a.cap);
}

constexpr int APPEND_THREADS = 256;
constexpr int APPEND_PER = 4;  // 16-byte pieces per thread, loaded before any is stored

template <typename T>
__global__ void __launch_bounds__(APPEND_THREADS) append_kernel(const AppendLaunch a) {
  pdl_wait();
  pdl_trigger();
  __shared__ int sh_pos;
  const KVView& kv = a.kv;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) sh_pos = a.seq_lens[b];
  __syncthreads();
  const int pos = sh_pos;
  if (pos < 0 || pos >= kv.t_max) {  // no room: flagged, nothing written
    if (threadIdx.x == 0) raise_error(kv.err, PRHS_DEV_CAPACITY);
    return;
  }
  const int cpr = kv.d * (int)sizeof(T) / 16;  // 16-byte pieces per row
  const int pieces = kv.Hkv * cpr;
  const uint4* kn = static_cast<const uint4*>(a.k_new) + (long long)b * pieces;
  const uint4* vn = static_cast<const uint4*>(a.v_new) + (long long)b * pieces;
  uint4* kc = static_cast<uint4*>(const_cast<void*>(kv.k));
  uint4* vc = static_cast<uint4*>(const_cast<void*>(kv.v));
  for (int x0 = 0; x0 < pieces; x0 += APPEND_THREADS * APPEND_PER) {
    uint4 kk[APPEND_PER], vv[APPEND_PER];
    long long dst[APPEND_PER];
#pragma unroll
    for (int u = 0; u < APPEND_PER; u++) {
      const int x = x0 + u * APPEND_THREADS + threadIdx.x;
      dst[u] = -1;
      if (x < pieces) {
        const long long row = kv_row(kv, b, x / cpr, pos);
        if (row < 0) {
          raise_error(kv.err, PRHS_DEV_BAD_BLOCK);
          continue;
        }
        dst[u] = row * cpr + x % cpr;
        kk[u] = kn[x];
        vv[u] = vn[x];
      }
    }
#pragma unroll
    for (int u = 0; u < APPEND_PER; u++)
      if (dst[u] >= 0) {
        kc[dst[u]] = kk[u];
        vc[dst[u]] = vv[u];
      }
  }
  __syncthreads();  // every piece of this sequence is written before its length moves
  if (threadIdx.x == 0) a.seq_lens[b] = pos + 1;
}

cudaError_t launch_compose(const ComposeLaunch& a, cudaStream_t st) {
  return launch_pdl(compose_kernel, dim3(a.kv.B * a.kv.Hq), dim3(GROW_THREADS), 0, st, a.kv.pdl, a);
}

cudaError_t launch_append(const AppendLaunch& a, cudaStream_t st) {
  if (a.kv.dtype == PRHS_BF16)
    return launch_pdl(append_kernel<__nv_bfloat16>, dim3(a.kv.B), dim3(APPEND_THREADS), 0, st, a.kv.pdl, a);
  return launch_pdl(append_kernel<float>, dim3(a.kv.B), dim3(APPEND_THREADS), 0, st, a.kv.pdl, a);
}

}  // namespace prhs
