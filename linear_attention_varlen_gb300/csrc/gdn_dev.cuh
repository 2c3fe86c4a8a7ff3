// Device helpers shared by the forward and backward kernels: bounded waits, publication
// flags, status word, and copies between shared and global memory.
#pragma once
#include <cstdint>

#include "bw_prims.cuh"
#include "gdn_common.cuh"

namespace gdn {

constexpr long long kWaitBudget = 4000000000LL;  // clock cycles (about two seconds)

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void set_status(Header* hd, int code) { atomicCAS(&hd->status, 0, code); }
__device__ __forceinline__ int get_status(const Header* hd) {
  return *reinterpret_cast<const volatile int*>(&hd->status);
}

// Bounded wait on a publication flag; false on timeout (status set) or on an earlier error.
__device__ __forceinline__ bool wait_flag(const int* flag, Header* hd) {
  const long long t0 = clock64();
  while (ld_acquire(flag) == 0) {
    if (get_status(hd) != 0) return false;
    if (clock64() - t0 > kWaitBudget) {
      set_status(hd, kErrTimeout);
      return false;
    }
    __nanosleep(128);
  }
  return true;
}

// All threads of the CTA wait on `bar`; the outcome is made uniform with a vote so that no
// thread leaves while others still expect a barrier. On failure each thread waits once more
// (bounded) so that copies or MMAs still in flight can land before the caller gives up.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
  const bool ok = bw::mbar_wait(bar, parity, kWaitBudget);
  if (__syncthreads_or(!ok)) {
    bw::mbar_wait(bar, parity, kWaitBudget);
    return false;
  }
  return true;
}

template <class T, class P>
__device__ __forceinline__ T* ws_ptr(const P& p, size_t off) {
  return reinterpret_cast<T*>(p.ws + off);
}

// Copy `bytes` (multiple of 16 * 256) of shared memory to global memory with all 256 threads.
__device__ __forceinline__ void copy_smem_to_global(uint8_t* dst, const uint8_t* src, int bytes, int tid) {
  for (int o = tid * 16; o < bytes; o += 256 * 16)
    *reinterpret_cast<uint4*>(dst + o) = *reinterpret_cast<const uint4*>(src + o);
}

// Make generic-proxy shared-memory writes visible to tcgen05 / TMA and order TMEM accesses
// across a CTA barrier.
__device__ __forceinline__ void sync_generic_to_async() {
  bw::fence_proxy_async_smem();
  bw::tc_fence_before();
  __syncthreads();
  bw::tc_fence_after();
}

}  // namespace gdn
