// dspark_common.cuh -- device helpers shared by the libdspark kernels (sm_103a).
//
// Inline PTX for the asynchronous-copy path: mbarrier initialisation,
// expect-tx arrival and bounded parity waits, and the 1-D bulk copy
// (cp.async.bulk, the TMA engine's untiled form) from global memory into the
// issuing CTA's own shared memory. No multicast form is used anywhere.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark_testing.h"

namespace dspark {

// Every bounded wait gives up after about a second of wall time (the
// device's global timer): far beyond any legitimate copy or barrier latency,
// short enough that a lost completion ends the kernel with DSPARK_ERR_TIMEOUT
// instead of hanging the GPU. The clock is read once every 1,024 failed
// tries, so a wait that succeeds soon never reads it.
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

struct WaitClock {
  uint64_t t0 = 0;
  uint32_t n = 0;
  // call after each failed try; true once the wait has lasted kWaitNs
  __device__ __forceinline__ bool expired() {
    if ((++n & 1023u) != 0u) return false;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) {
      t0 = now;
      return false;
    }
    return now - t0 > kWaitNs;
  }
};

__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, (int32_t)DSPARK_OK, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the asynchronous proxy (the copy engine).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later asynchronous-proxy writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t addr = smem_addr(bar);
  WaitClock clock;
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
    if (clock.expired()) return false;
  }
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction count on
// `bar`. src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Per-thread asynchronous 16-byte copy global -> shared (the thread's own
// copies complete in commit-group order; cp.async.wait_group N leaves at most
// N of its groups in flight and makes the completed ones visible to it).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch. Every kernel of the library is launched with
// programmatic stream serialization, so the next kernel on the stream may be
// scheduled before this one ends. pdl_wait() blocks until the preceding grid
// has completed and its memory is visible; each kernel calls it before its
// first global-memory access, so reads and writes stay ordered exactly as
// without the attribute. pdl_trigger() then lets the following grid launch
// early, hiding its launch latency behind this kernel.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 2^x, hardware approximation (flush-to-zero for results below the normal range).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T>
__device__ __forceinline__ float to_float(T v);
template <>
__device__ __forceinline__ float to_float<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_float<uint16_t>(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// A value carried as an unevaluated sum of two floats (about 48 significant
// bits): double-like precision on the float pipes.
struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff ff_norm(float s, float e) {
  const float hi = s + e;
  return ff{hi, e - (hi - s)};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const float s = a.hi + b.hi;
  const float bp = s - a.hi;
  const float err = (a.hi - (s - bp)) + (b.hi - bp) + a.lo + b.lo;
  return ff_norm(s, err);
}

__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff{-b.hi, -b.lo}); }

__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return ff_norm(p, e);
}

// sign of a - b (-1, 0, 1)
__device__ __forceinline__ int ff_cmp(ff a, ff b) {
  const ff d = ff_sub(a, b);
  const float v = d.hi != 0.f ? d.hi : d.lo;
  return (v > 0.f) - (v < 0.f);
}

__device__ __forceinline__ ff shfl_up_ff(ff v, int o) {
  return ff{__shfl_up_sync(0xFFFFFFFFu, v.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.lo, o)};
}

__device__ __forceinline__ ff shfl_ff(ff v, int src) {
  return ff{__shfl_sync(0xFFFFFFFFu, v.hi, src), __shfl_sync(0xFFFFFFFFu, v.lo, src)};
}

// Kahan-compensated float accumulator.
struct KahanF {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  __device__ __forceinline__ double value() const {
    return static_cast<double>(s) - static_cast<double>(c);
  }
};

// Launch `kernel` on `stream` with programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace dspark
