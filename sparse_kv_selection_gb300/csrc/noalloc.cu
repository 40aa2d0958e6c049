// Sparse attention for callers that cannot allocate device memory.
//
// prhs_sparse_attn takes its split-K scratch (per-CTA partial softmax
// states and completion tickets) from a workspace the caller allocates.
// Some callers cannot call cudaMalloc at all, so they cannot provide one:
// for example a plugin host that owns every byte of device memory and
// forbids the libraries it loads to allocate, or a serving loop that may
// not take cudaMalloc's implicit device synchronisation. For them,
// prhs_sparse_attn_noalloc runs the same kernel with its scratch in the
// file-scope device array below, which every GPU that loads this library
// holds until the process exits.
#include <mutex>
#include <string>

#include "kernels.h"

namespace prhs {
namespace {

// Fixed scratch: completion tickets first, then the partial records. Every
// call on a device shares it, and it keeps the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PRHS_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
void* g_scratch_ptr[MAX_DEVICES] = {};
std::mutex g_mu;

// Device address of the scratch array on the current device, resolved once
// per device with that device current (in host code the array's name is
// only a host-side stand-in, not a device address).
prhs_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return abi_fail(PRHS_ECUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= MAX_DEVICES) return abi_fail(PRHS_ECUDA, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      std::string m = std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e);
      return abi_fail(PRHS_ECUDA, m.c_str());
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PRHS_OK;
}

}  // namespace
}  // namespace prhs

using namespace prhs;

extern "C" prhs_status prhs_sparse_attn_noalloc(const prhs_kv* kv, const void* q, float scale,
                                                const int32_t* idx, const int32_t* n_sel, int cap,
                                                float* out, float* lse, cudaStream_t stream) {
  prhs_status s = abi_check_kv(kv);
  if (s != PRHS_OK) return s;
  if (!q || !idx || !n_sel || !out || !lse)
    return abi_fail(PRHS_EINVAL, "sparse_attn_noalloc: null pointer argument");
  if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0)
    return abi_fail(PRHS_EINVAL, "sparse_attn_noalloc: q must be 16-byte aligned");
  if (cap <= 0) return abi_fail(PRHS_EINVAL, "sparse_attn_noalloc: cap must be positive");
  if ((long long)kv->B * kv->Hq * cap >= (1ll << 30))
    return abi_fail(PRHS_EUNSUPPORTED, "sparse_attn_noalloc: B * Hq * cap above 2^30 rows");
  unsigned* err = nullptr;
  int sms = 0;
  if ((s = abi_device(&err, &sms)) != PRHS_OK) return s;
  void* scratch = nullptr;
  if ((s = scratch_address(&scratch)) != PRHS_OK) return s;

  const int units = kv->B * kv->Hq;
  const KVView view = abi_view(*kv, err);
  const int ctas = abi_attn_ctas(*kv, true, cap, sms);
  const size_t tickets = ((size_t)units * sizeof(unsigned) + 255) / 256 * 256;
  const size_t need = tickets + attn_partial_floats(view, true, ctas) * sizeof(float);
  if (need > (size_t)PRHS_NOALLOC_SCRATCH_BYTES) {
    std::string m = "sparse_attn_noalloc: this batch needs " + std::to_string(need) +
                    " bytes of scratch, more than the fixed " +
                    std::to_string((size_t)PRHS_NOALLOC_SCRATCH_BYTES);
    return abi_fail(PRHS_EINVAL, m.c_str());
  }
  // the tickets must start at zero, whatever an earlier call left there
  cudaError_t e = cudaMemsetAsync(scratch, 0, tickets, stream);
  if (e != cudaSuccess) return abi_fail(PRHS_ECUDA, cudaGetErrorString(e));

  AttnLaunch a;
  a.kv = view;
  a.q = q;
  a.scale = scale;
  a.idx = idx;
  a.n_sel = n_sel;
  a.unit_mask = nullptr;
  a.mask_want = 0;
  a.cap = cap;
  a.out = out;
  a.lse = lse;
  a.counters = static_cast<unsigned*>(scratch);
  a.partials = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + tickets);
  a.ctas = ctas;
  a.min_rows = ATTN_MIN_ROWS;
  e = launch_attn(a, true, stream);
  if (e != cudaSuccess) return abi_fail(PRHS_ECUDA, cudaGetErrorString(e));
  abi_count_launch();
  return PRHS_OK;
}
