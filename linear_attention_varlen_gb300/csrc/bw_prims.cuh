// Blackwell (sm_100a / sm_103a) primitives used by the GDN kernels, as inline PTX:
// mbarriers, TMA (tiled tensor copies and 1-D bulk copies), tcgen05 tensor-memory
// allocation, UMMA (tcgen05.mma kind::f16) with shared-memory descriptors, and
// tcgen05.ld readback. Every wait is bounded: a wait that runs out returns false
// and the caller records an error status instead of spinning forever.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace gdn {
namespace bw {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 1024-byte aligned start of the dynamic shared memory. It is derived from the __shared__ array
// by pointer arithmetic (not through an integer round trip), so the compiler still knows that
// accesses through it are shared-memory accesses and emits LDS/STS instead of generic loads.
__device__ __forceinline__ uint8_t* smem_align1024(uint8_t* raw) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(raw));
  return raw + ((1024u - (a & 1023u)) & 1023u);
}

// ------------------------------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Raise the current phase's expected transaction count without arriving (copies that are issued
// ahead of the arrival that arms the rest of the phase).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete; false after `budget` clock cycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > budget) return false;
  }
  return true;
}

// ------------------------------------------------------------------------------------------ fences

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Order this thread's generic-proxy view of global memory before its later async-proxy accesses
// (a bulk copy of data that another thread published).
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------------------ dependent launch

// A kernel launched with programmatic stream serialization may start while the kernel before it
// in the stream still runs: it waits here (before touching anything that kernel writes) until
// that kernel has completed and its memory is visible. A no-op for a plain launch.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel of the stream (if it was launched that way) to start early.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------------------------ TMA

// 3-D tiled load of one box into shared memory; completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
// Tiled TMA store shared -> global (3-D map; the box must lie inside the tensor: the caller
// only stores whole boxes). Completion is tracked with the bulk async-group of this thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until at most N of this thread's committed bulk groups have not finished reading their source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 1-D bulk copy shared -> global, tracked with the bulk async-group of this thread (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}

// Ask for the 128-byte line holding p to be brought into L2.
// Bring a tiled TMA box (3-D map, same coordinates as a load) into L2 ahead of its load.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// Bring `bytes` (16-byte aligned address, multiple of 16) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------------------------------ TMEM

// Allocate `ncols` (power of two >= 32) tensor-memory columns; one full warp calls it.
__device__ __forceinline__ void tmem_alloc(uint32_t* holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets lane (warp's quarter) + i.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 16 TMEM lanes (taddr's lane field: the first of them) x 32 columns over the whole warp:
// thread t gets rows t/4 and t/4 + 8 of the 16 and columns 8k + 2(t%4) + {0, 1}, k = 0..3, in
// the order v[4k] = (t/4, c), v[4k+1] = (t/4, c+1), v[4k+2] = (t/4+8, c), v[4k+3] = (t/4+8, c+1)
// with c = 8k + 2(t%4) (shape 16x256b, repeated 4 times). This is how an M = 64 accumulator
// (16 valid lanes per 32-lane quarter) is read with all 32 threads of a warp.
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 32 bits, 32 consecutive columns (thread i: lane quarter + i, v[c] = column c).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// Store 16 / 32 consecutive 32-bit columns of this thread's lane (the 32x32b shape of tmem_ld16).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Sum over the four threads of a row group of the 16x256b layout (lanes 4g .. 4g + 3).
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}
// Byte offset of the bf16 pair (row r, columns c, c + 1; c even) in a 64-column SW128 block.
// 4 x 4 transpose across the four lanes of a group (qa = lane & 3): lane qa's x[m] becomes the
// x[qa] of lane m. Two exchange rounds (lane ^ 1, lane ^ 2) of two shuffles each.
__device__ __forceinline__ void quad_transpose4(uint32_t* x, int qa) {
  {
    const bool o = qa & 1;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, o ? x[0] : x[1], 1);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, o ? x[2] : x[3], 1);
    if (o) {
      x[0] = r0;
      x[2] = r1;
    } else {
      x[1] = r0;
      x[3] = r1;
    }
  }
  {
    const bool o = qa & 2;
    const uint32_t r0 = __shfl_xor_sync(0xffffffffu, o ? x[0] : x[2], 2);
    const uint32_t r1 = __shfl_xor_sync(0xffffffffu, o ? x[1] : x[3], 2);
    if (o) {
      x[0] = r0;
      x[1] = r1;
    } else {
      x[2] = r0;
      x[3] = r1;
    }
  }
}
__device__ __forceinline__ uint32_t sw128_pair(int r, int c) {
  return r * 128 + ((((c >> 3) ^ r) & 7) << 4) + ((c & 7) << 1);
}

// ------------------------------------------------------------------------------------------ UMMA

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulate.
// a_mn / b_mn: 0 = K-major operand, 1 = MN-major operand.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                           // D format: f32
         | (1u << 7)                         // A format: bf16
         | (1u << 10)                        // B format: bf16
         | (uint32_t(a_mn & 1) << 15)        // A major
         | (uint32_t(b_mn & 1) << 16)        // B major
         | (uint32_t(N >> 3) << 17)          // N / 8
         | (uint32_t(M >> 4) << 24);         // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle, tcgen05 version bits.
// lbo: leading-dimension byte offset; sbo: stride-dimension byte offset (both multiples of 16).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// D[tmem] (+)= A * B, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A * B with A in tensor memory (row m of A in lane m, K packed two bf16 per 32-bit
// column, the lower K index in the low half; A is K-major, so the instruction descriptor's A-major
// bit is 0) and B described in shared memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on `bar` when all previously issued tcgen05.mma of this thread have completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------------------------------------------ SW128 tiles
//
// A "tile" below is a block of R rows x 64 bf16 (128 bytes per row) laid out the way a
// 128-byte-swizzled TMA box lands in shared memory: row r at byte r*128, its 16-byte chunk c
// stored at chunk position (c ^ (r % 8)). Blocks start on 1024-byte boundaries.

// Byte offset of element (row, col) (col < 64) inside a 128B-swizzled block.
__host__ __device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t col) {
  return row * 128u + ((((col >> 3) ^ (row & 7u)) & 7u) << 4) + ((col & 7u) << 1);
}

// K-major operand: rows = M (or N) index, 64-wide K blocks `kblk_stride` bytes apart.
// Descriptor for k-step ks (16 elements of K each).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, uint32_t kblk_stride, int ks) {
  return sdesc_sw128(base + (uint32_t)(ks >> 2) * kblk_stride + (uint32_t)(ks & 3) * 32u, 16u, 1024u);
}
// Descriptor of k-step ks from that of k-step 0 (no address arithmetic in the issue loop): the
// start-address field holds bits 4-17 of the address, and every operand lies below 256 KB of
// shared memory, so adding the step's offset never carries out of the field.
__device__ __forceinline__ uint64_t kmajor_step(uint64_t d0, uint32_t kblk_stride, int ks) {
  return d0 + (((uint32_t)(ks >> 2) * kblk_stride + (uint32_t)(ks & 3) * 32u) >> 4);
}
__device__ __forceinline__ uint64_t mnmajor_step(uint64_t d0, int ks) { return d0 + (uint64_t)ks * (2048u >> 4); }
// MN-major operand: rows = K index (128 bytes per row = 64 MN elements), MN blocks of 64
// elements `mn_stride` bytes apart. Descriptor for k-step ks (16 rows of K each).
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, uint32_t mn_stride, int ks) {
  return sdesc_sw128(base + (uint32_t)ks * 2048u, mn_stride, 1024u);
}

// Two fp32 values in one 64-bit register for the packed fp32x2 arithmetic of sm_100 and later
// (one instruction, each lane rounded as its scalar counterpart).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(uint64_t v) {
  float lo;
  asm("{\n .reg .f32 t;\n mov.b64 {%0, t}, %1;\n}" : "=f"(lo) : "l"(v));
  return lo;
}
__device__ __forceinline__ float f2_hi(uint64_t v) {
  float hi;
  asm("{\n .reg .f32 t;\n mov.b64 {t, %0}, %1;\n}" : "=f"(hi) : "l"(v));
  return hi;
}
__device__ __forceinline__ float f2_sum(uint64_t v) { return f2_lo(v) + f2_hi(v); }
// a * b, lane by lane
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// a * b + c, lane by lane
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace bw
}  // namespace gdn
