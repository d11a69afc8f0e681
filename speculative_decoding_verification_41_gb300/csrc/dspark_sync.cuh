// dspark_sync.cuh -- GPU-scope acquire / release accesses and a bounded
// grid barrier, shared by the kernels whose CTAs wait on one another
// (sm_103a). Every wait is bounded by wall time (WaitClock): a barrier that a
// CTA never reaches ends with DSPARK_ERR_TIMEOUT instead of a hang.
#pragma once

#include "dspark_common.cuh"

namespace dspark {

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_gpu64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// One thread per CTA. sync[0] counts arrivals and is 0 between uses (zeroed
// before the launch, reset by the last arrival); sync[1] is a generation that
// every CTA reads before its first arrival. Returns false if the wait gave up.
__device__ inline bool grid_barrier(uint32_t* sync, uint32_t nctas, uint32_t& gen) {
  const uint32_t g = gen;
  __threadfence();
  if (atom_add_acq_rel_gpu(&sync[0], 1u) == nctas - 1) {
    atomicExch(&sync[0], 0u);
    __threadfence();
    st_release_gpu(&sync[1], g + 1u);
  } else {
    WaitClock clock;
    while (ld_acquire_gpu(&sync[1]) == g) {
      if (clock.expired()) return false;
      __nanosleep(128);
    }
  }
  gen = g + 1u;
  __threadfence();
  return true;
}

}  // namespace dspark
