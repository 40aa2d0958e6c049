// Shared device helpers of the PrHS decode kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/prhs.h"

namespace prhs {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Kernels OR PRHS_DEV_* bits into the library's device error word, whose
// address every launch receives; prhs_last_error() reads and clears it.
__device__ __forceinline__ void raise_error(unsigned* err, unsigned bits) { atomicOr(err, bits); }

// -------------------------------------------------------------------------- //
// Cache descriptor as the kernels see it
// -------------------------------------------------------------------------- //
struct KVView {
  prhs_dtype dtype;
  const void* k;
  const void* v;
  const int32_t* seq_lens;
  const int32_t* block_table;  // null: contiguous
  int B, Hq, Hkv, d;
  int t_max;                   // contiguous row stride, or max_blocks * block_size
  int block_size, max_blocks, num_blocks;
  unsigned* err;               // device error word
  bool pdl;                    // launches overlap their stream predecessor's tail
};

// A loaded sequence length clamped to [0, t_max] (out-of-range lengths are
// flagged). Loops that read many lengths load them all first and check them
// after, so that the loads are not held behind a possible error write.
__device__ __forceinline__ int checked_len(const KVView& kv, int t) {
  if (t < 0 || t > kv.t_max) {
    raise_error(kv.err, PRHS_DEV_BAD_LEN);
    t = t < 0 ? 0 : kv.t_max;
  }
  return t;
}

// Length of sequence b, clamped to [0, t_max] (out-of-range lengths are flagged).
__device__ __forceinline__ int seq_len(const KVView& kv, int b) {
  return checked_len(kv, kv.seq_lens[b]);
}

// Row number (in units of d elements) of key i of (b, kv head h); -1 when the
// page id is outside the pool.
__device__ __forceinline__ long long kv_row(const KVView& kv, int b, int h, int i) {
  if (kv.block_table == nullptr) return ((long long)b * kv.Hkv + h) * kv.t_max + i;
  int page = kv.block_table[(long long)b * kv.max_blocks + i / kv.block_size];
  if ((unsigned)page >= (unsigned)kv.num_blocks) return -1;
  return ((long long)page * kv.Hkv + h) * kv.block_size + (i % kv.block_size);
}

// -------------------------------------------------------------------------- //
// element conversion
// -------------------------------------------------------------------------- //
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int per16 = 4;  // elements per 16-byte chunk
  __device__ static __forceinline__ void unpack(const uint4& c, float* f) {
    f[0] = __uint_as_float(c.x); f[1] = __uint_as_float(c.y);
    f[2] = __uint_as_float(c.z); f[3] = __uint_as_float(c.w);
  }
  __device__ static __forceinline__ float load1(const void* p, long long i) {
    return static_cast<const float*>(p)[i];
  }
  __device__ static __forceinline__ void store1(void* p, long long i, float v) {
    static_cast<float*>(p)[i] = v;
  }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int per16 = 8;
  __device__ static __forceinline__ void unpack(const uint4& c, float* f) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static __forceinline__ float load1(const void* p, long long i) {
    return __uint_as_float(uint32_t(static_cast<const uint16_t*>(p)[i]) << 16);
  }
};

// Raw copy of one element (used to mirror q into the anchor buffer).
template <typename T>
__device__ __forceinline__ void copy_elem(void* dst, const void* src, long long i) {
  static_cast<T*>(dst)[i] = static_cast<const T*>(src)[i];
}

// -------------------------------------------------------------------------- //
// global loads that bypass L1 allocation (streamed once)
// -------------------------------------------------------------------------- //
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// -------------------------------------------------------------------------- //
// mbarrier / TMA (inline PTX)
// -------------------------------------------------------------------------- //
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `parity` to complete, giving up after limit_ns (about
// a second unless a caller asks for less). On timeout the error word gets
// PRHS_DEV_TIMEOUT and false is returned.
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned* err,
                                          uint64_t limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (unsigned n = 1;; n++) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255u) == 0 && globaltimer_ns() - t0 > limit_ns) {
      raise_error(err, PRHS_DEV_TIMEOUT);
      return false;
    }
  }
}

// 3-D tiled TMA load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Plain bulk copy of `bytes` contiguous bytes (a multiple of 16; both
// addresses 16-byte aligned) into this CTA's shared memory, completion
// counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// -------------------------------------------------------------------------- //
// programmatic dependent launch: every kernel of the path waits for its
// stream predecessor before touching memory the predecessor may write or
// read, then lets its own successor start launching. The launch attribute is
// set only when `pdl` is (caches of up to PDL_MAX_KEYS keys: short kernels
// back to back, whose launch latency it hides); on longer caches the two
// branches of a decode step overlap better without it (measured 4-6% faster
// steps on 32K-131K-key caches). Without the attribute the wait and the
// trigger are no-ops.
// -------------------------------------------------------------------------- //
constexpr int PDL_MAX_KEYS = 8192;
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// -------------------------------------------------------------------------- //
// small reductions
// -------------------------------------------------------------------------- //
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL_MASK, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL_MASK, v, o);
  return v;
}

// Order-preserving map of a float to uint32 (larger float -> larger key);
// -0.0 is folded onto +0.0 so that the two compare equal.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace prhs
