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

// Bounded wait (`budget` clock cycles) on a publication flag; false on timeout (status set) or on
// an earlier error.
__device__ __forceinline__ bool wait_flag(const int* flag, Header* hd, long long budget) {
  const long long t0 = clock64();
  while (ld_acquire(flag) == 0) {
    if (get_status(hd) != 0) return false;
    if (clock64() - t0 > budget) {
      set_status(hd, kErrTimeout);
      return false;
    }
    __nanosleep(128);
  }
  return true;
}

// Waits (bounded as wait_flag) until the counter *ctr reaches `target`.
__device__ __forceinline__ bool wait_count(const int* ctr, int target, Header* hd, long long budget) {
  const long long t0 = clock64();
  while (ld_acquire(ctr) < target) {
    if (get_status(hd) != 0) return false;
    if (clock64() - t0 > budget) {
      set_status(hd, kErrTimeout);
      return false;
    }
    __nanosleep(64);
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

// Exact split: a segment boundary needs no published state when the decay between the state it
// neglects and the chunk it starts at is below fp32 resolution. Per token the transition is
// e^{g_t} (I - beta_t k_t k_t^T), whose spectral norm is at most e^{g_t} while
// 0 <= beta_t |k_t|^2 <= 2 (the chunk's flag in `contr`, written by kkt_solve). Over a window
// whose summed log-decay is below kExactCut the neglected term is therefore below
// e^{-30} (about 2^-43, 19 bits under fp32's unit roundoff of 2^-24) times the norm of the state it
// neglects, while every chunk step of the chain itself rounds that state at 2^-24: the chain can
// start from zero at the window's far end (a warm-up) instead of waiting for the neighbouring
// segment, and the result is the exact recurrence to fp32 resolution.
constexpr float kExactCut = -30.f;
constexpr int kWarmCap = 32;  // longest warm-up window, chunks: one per lane of the warp that evaluates it

// One warp evaluates a window in one round trip: lane i takes chunk `first + step * i`, an
// inclusive prefix sum of the chunks' log-decays gives the window ending at lane i, and the window
// is the shortest one below kExactCut whose chunks all lie in [lo, hi) and contract. Every lane
// returns the same value; call with the whole warp (the chain kernels call it with all threads).
__device__ __forceinline__ int warm_window(const float* gam, const int32_t* contr, int Hv, int h, int first, int step,
                                           int lo, int hi) {
  const int lane = threadIdx.x & 31;
  const int w = first + step * lane;
  const bool in = w >= lo && w < hi;
  float acc = in ? __ldg(gam + ((size_t)w * Hv + h) * kChunk + kChunk - 1) : 0.f;
  const bool good = in && __ldg(contr + (size_t)w * Hv + h) != 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, acc, o);
    if (lane >= o) acc += t;
  }
  const unsigned bad = __ballot_sync(0xffffffffu, !good);
  const unsigned hit = __ballot_sync(0xffffffffu, good && acc < kExactCut);
  if (!hit) return -1;
  const int i = __ffs(hit) - 1;
  const unsigned upto = (i == 31) ? 0xffffffffu : ((1u << (i + 1)) - 1u);
  return (bad & upto) ? -1 : w - step * lane + step * i;
}

// Backward-looking window for a forward chain that starts at chunk c (document chunks from dc0):
// the first chunk of the warm-up, or -1 when no window of at most kWarmCap chunks qualifies.
__device__ __forceinline__ int warm_back(const float* gam, const int32_t* contr, int Hv, int h, int c, int dc0) {
  return warm_window(gam, contr, Hv, h, c - 1, -1, dc0, c);
}

// Forward-looking window for a reverse chain that ends at chunk c (exclusive; document chunks up
// to dcn): one past the last chunk of the warm-up, or -1.
__device__ __forceinline__ int warm_fwd(const float* gam, const int32_t* contr, int Hv, int h, int c, int dcn) {
  const int w = warm_window(gam, contr, Hv, h, c, 1, c, dcn);
  return w < 0 ? -1 : w + 1;
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
