// Backward of the chunked Gated DeltaNet (sm_103a).
//
// The backward recomputes the forward chunk states ("How to Speed Up GDN Kernels for Qwen
// Models", section "Lever 2": the per-chunk states are rebuilt by a single pass of their own
// rather than kept from the forward),
// or finds them in the workspace when the forward of a training step kept them (the same
// recompute, run by the forward, which then forms o from the records), then runs the
// state-gradient chain in reverse and the per-chunk gradients in parallel:
//
//   1. forward recompute (plan, kkt_solve, chain in record mode): for every chunk c and value
//      head, S_c (state at the chunk start, bf16), V'_c = U - W S_c (bf16) and T_c (fp32).
//   2. rev_chain_kernel, per (document, value head), chunks in reverse:
//        dV' = K~ dS_{c+1} + P^T dO,    dS_c = e^{gamma_C} dS_{c+1} + Q~^T dO - W^T dV'
//      (K~ = diag(e^{gamma_C - gamma}) K, Q~ = diag(e^{gamma}) Q, P = (Q K^T) o E); records
//      dS_{c+1} and dV' per chunk, and dL/dS at the document start; segments warm up from zero
//      over the following chunks when the decay there provably hides the later gradient, as in
//      the forward. A document whose final
//      state was forked first collects the d(initial state) of every document that started from
//      it ("Musings on long-context fine-tuning", section "Backward through P": the gradients of
//      the branches add up at the shared state).
//   3. grad_kernel, per (chunk, key head), looping over the value heads of the group: dk
//      (summed over the group in tensor memory), dv, dbeta and dg from S_c, dS_{c+1}, V', dV'
//      and T, through the reverse mode of the chunk algebra (T = (I + A)^{-1}, W = T diag(beta
//      e^gamma) K, U = T diag(beta) V, O = Q~ S + P V', S_{c+1} = e^{gamma_C} S + K~^T V').
//      dq_kernel computes dq the same way with compensated bf16 operands (see there), and adds
//      to dg its term through the state part of o, which needs S_c at that accuracy.
//   4. dinit_reduce_kernel: d(initial_state) of each pool entry = the sum, in document order,
//      over the documents that start from it.
//
// Precision: the recompute keeps T diag(beta e^gamma), T diag(beta) and diag(e^{gamma_C-gamma}) V'
// as compensated bf16 pairs (x = hi + lo, two MMAs), so that the recorded states and V' carry
// fp32-level accuracy into the gradients; all gradients are written in fp32.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "bw_prims.cuh"
#include "gdn_bwd.h"
#include "gdn_common.cuh"
#include "gdn_dev.cuh"
#include "gdn_fwd.h"
#include "gdn_host.h"
#include "tmap.h"

namespace gdn {
using namespace bw;

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  const float* g;
  const float* beta;
  const int32_t* cu;
  const int32_t* init_idx;
  const float* dfinal;
  float* dq;
  float* dk;
  float* dv;
  float* dg;
  float* dbeta;
  float* dinit;
  uint8_t* ws;
  PlanDims d;
  BwdLayout L;
  float scale;
  long long flag_budget;  // limit of a wait on another item's publication flag, SM clock cycles
};

__device__ __forceinline__ uint4 pack8(const float* x) {
  return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                    pack_bf16x2(x[6], x[7]));
}
__device__ __forceinline__ float bf16_at(const uint8_t* blk, int row, int col) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(blk + sw128_off(row, col)));
}
// Scale row r of a [64 x 64] bf16 SW128 block (8 KB) in place; 256 threads, one 16-byte piece each pass.
__device__ __forceinline__ void scale_rows(uint8_t* blk, const float* rs, int tid) {
  for (int o = tid * 16; o < 8192; o += 256 * 16) {
    const float sc = rs[o >> 7];
    uint4 raw = *reinterpret_cast<uint4*>(blk + o);
    __nv_bfloat162* x = reinterpret_cast<__nv_bfloat162*>(&raw);
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float2 f = __bfloat1622float2(x[u]);
      w[u] = pack_bf16x2(f.x * sc, f.y * sc);
    }
    *reinterpret_cast<uint4*>(blk + o) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}
struct Ctx {
  uint64_t* bar_ld;
  uint64_t* bar_mma;
  uint32_t tmem, ph_ld, ph_mma;
  int tid, warp, lane, q4, half;
  __device__ bool wait_ld() {
    if (!wait_all(bar_ld, ph_ld)) return false;
    ph_ld ^= 1;
    tc_fence_after();
    return true;
  }
  __device__ bool commit_wait() {
    if (tid == 0) umma_commit(bar_mma);
    if (!wait_all(bar_mma, ph_mma)) return false;
    ph_mma ^= 1;
    tc_fence_after();
    return true;
  }
  __device__ uint32_t lane_base() const { return (uint32_t)(32 * q4) << 16; }
};

__device__ __forceinline__ void ctx_init(Ctx& c, uint64_t* bl, uint64_t* bm) {
  c.bar_ld = bl;
  c.bar_mma = bm;
  c.tid = threadIdx.x;
  c.warp = c.tid >> 5;
  c.lane = c.tid & 31;
  c.q4 = c.warp & 3;
  c.half = c.warp >> 2;
  c.ph_ld = 0;
  c.ph_mma = 0;
}

// ===================================================================================== reverse chain
//
// The reverse chain per (segment, value head) in one CTA of 10 warps, chunks in reverse order:
//   warp 8      TMA producer: K, Q, dO, T diag(beta e^gamma), P = scale (Q K^T o E) (formed by
//               kkt_solve) and gamma of chunk j into stage j & 1.
//   warp 9      MMA issuer (one lane): chunk j + 1's W = T_w K as soon as its operands have
//               landed; A: Q~^T dO into the dS accumulator (M = 128) and dV' = K~ dS + P^T dO
//               (M = 64); B: dS accumulator += -W^T dV' (M = 128).
//   warps 0-7   epilogue: Q~, K~ and -W of chunk j + 1 staged while chunk j runs;
//               dV' (zero rows beyond the chunk) in bf16, dS = e^{gamma_C} dS + accumulator in fp32
//               registers (row 32 q4 + lane, columns 64 half ..), its bf16 copy the next chunk's
//               operand; records (dL/dS at each chunk end, dV') go out by bulk stores.
// Hand-offs are mbarriers: tcgen05.commit from the issuer, one elected arrival after a named
// barrier from the epilogue, TMA transaction counts from the producer.

struct RevSmem {
  uint8_t k[2][16384];    // [stage] K rows t, two dk blocks (B K-major: Q K^T; B MN-major: T_w K)
  uint8_t q[2][16384];    // [stage] Q rows t                 (A K-major: Q K^T)
  uint8_t dout[2][16384]; // [stage] dO rows t, two dv blocks (B MN-major)
  uint8_t tw[2][8192];    // [stage] T diag(beta e^gamma)     (A K-major: W = T_w K)
  uint8_t qt[16384];      // Q~ = scale diag(e^gamma) Q, rows >= n zero (A MN-major: Q~^T dO)
  uint8_t kt[16384];      // K~ = diag(e^{gamma_C - gamma}) K            (A K-major: K~ dS)
  uint8_t wn[16384];      // -W rows t                                    (A MN-major: -W^T dV')
  uint8_t p[2][8192];     // [stage] P = scale (Q K^T) o E                (A MN-major: P^T dO)
  uint8_t dvp[16384];     // dV' rows t, two dv blocks                    (B MN-major)
  uint8_t ds[32768];      // dS bf16 rows dk, two dv blocks               (B MN-major)
  float gam[2][64];
  float fsc[2][64];       // row factors of Q~ (scale e^gamma, zero beyond the chunk) and K~ (e^{gamma_C - gamma})
};
constexpr size_t kRevSmemBytes = sizeof(RevSmem) + 1024;
static_assert(kRevSmemBytes <= 227 * 1024, "shared memory of the reverse chain");
constexpr int kRevThreads = 320;
constexpr uint32_t kRtW = 0, kRtA = 256, kRtC = 384;  // TMEM columns: W (M = 64), dV' (M = 64), dS (M = 128)

struct RevBars {
  uint64_t full[2], empty[2], pre_done, staged1, staged2, a_done, epi1, b_done, epi2;
};
struct RevPhase {
  uint32_t full[2], empty[2], pre_done, staged1, staged2, a_done, epi1, b_done, epi2;
};

// Bounded wait that never diverges: after the first failure (recorded in *abort) every later
// wait returns at once, so all threads keep executing the same barriers.
__device__ __forceinline__ void rrole_wait(uint64_t* bar, uint32_t& ph, volatile int* abort) {
  if (!*abort && !mbar_wait(bar, ph, kWaitBudget)) *abort = 1;
  ph ^= 1;
  tc_fence_after();
}
__device__ __forceinline__ void r_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// Epilogue hand-off: shared-memory writes visible to the async proxy, TMEM reads ordered, the 256
// epilogue threads meet, one of them arrives.
__device__ __forceinline__ void r_handoff(int tid, uint64_t* b1, uint64_t* b2 = nullptr) {
  fence_proxy_async_smem();
  tc_fence_before();
  r_sync();
  if (tid == 0) {
    mbar_arrive(b1);
    if (b2) mbar_arrive(b2);
  }
  __syncwarp();
}

// Write this thread's 64 dS values (row 32 q4 + lane, columns 64 half ..) as bf16 into sm.ds.
__device__ __forceinline__ void rev_store_ds(const Ctx& cx, RevSmem& sm, const float* dS) {
  const int r = 32 * cx.q4 + cx.lane;
  uint8_t* blk = sm.ds + cx.half * 16384;
#pragma unroll
  for (int cj = 0; cj < 8; ++cj) *reinterpret_cast<uint4*>(blk + r * 128 + ((cj ^ (r & 7)) << 4)) = pack8(dS + 8 * cj);
}

// Chunks [gc0, gc1) of one document for value head h, in reverse, from dS (epilogue registers;
// its bf16 copy is already in sm.ds): dS becomes dL/dS at the start of chunk gc0. kRecord: also
// store dL/dS at each chunk end and dV' (bf16 images) for the gradient kernels, for the chunks
// below gc_rec (the ones above are a warm-up). All 320 threads call this; returns false after a
// failed wait.
template <bool kRecord>
__device__ bool run_rev_ws(const BwdParams& p, Ctx& cx, RevSmem& sm, RevBars& bb, RevPhase& ph, volatile int* abort,
                           float* dS, int gc0, int gc1, int h, int hk, int gc_rec) {
  const int n = gc1 - gc0;
  if (n <= 0) return true;
  const int Hv = p.d.Hv;
  const int32_t* ctok = reinterpret_cast<const int32_t*>(p.ws + p.L.f.chunk_tok0);
  const int32_t* clen = reinterpret_cast<const int32_t*>(p.ws + p.L.f.chunk_len);
  const uint32_t tm = cx.tmem;
  auto chunk_of = [&](int j) { return gc1 - 1 - j; };

  if (cx.warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (cx.lane == 0) {
      for (int j = 0; j < n; ++j) {
        const int gc = chunk_of(j), st = j & 1, tok0 = ctok[gc];
        const size_t rec = (size_t)gc * Hv + h;
        if (j + 2 < n) {  // chunk j + 2 into L2 while its stage is still in use
          const int g2 = chunk_of(j + 2), t2 = ctok[g2];
          const size_t r2 = (size_t)g2 * Hv + h;
          tma_prefetch_3d(&p.tm_k, 0, hk, t2);
          tma_prefetch_3d(&p.tm_k, 64, hk, t2);
          tma_prefetch_3d(&p.tm_q, 0, hk, t2);
          tma_prefetch_3d(&p.tm_q, 64, hk, t2);
          tma_prefetch_3d(&p.tm_do, 0, h, t2);
          tma_prefetch_3d(&p.tm_do, 64, h, t2);
          bulk_prefetch_l2(p.ws + p.L.f.tw + r2 * 8192, 8192);
          bulk_prefetch_l2(p.ws + p.L.f.pimg + r2 * 8192, 8192);
          bulk_prefetch_l2(p.ws + p.L.f.gam + r2 * 256, 256);
        }
        if (j >= 2) rrole_wait(&bb.empty[st], ph.empty[st], abort);
        if (*abort) break;
        mbar_arrive_expect_tx(&bb.full[st], 3 * 16384 + 2 * 8192 + 256);
        tma_load_3d(sm.k[st], &p.tm_k, 0, hk, tok0, &bb.full[st]);
        tma_load_3d(sm.k[st] + 8192, &p.tm_k, 64, hk, tok0, &bb.full[st]);
        tma_load_3d(sm.q[st], &p.tm_q, 0, hk, tok0, &bb.full[st]);
        tma_load_3d(sm.q[st] + 8192, &p.tm_q, 64, hk, tok0, &bb.full[st]);
        tma_load_3d(sm.dout[st], &p.tm_do, 0, h, tok0, &bb.full[st]);
        tma_load_3d(sm.dout[st] + 8192, &p.tm_do, 64, h, tok0, &bb.full[st]);
        bulk_load(sm.tw[st], p.ws + p.L.f.tw + rec * 8192, 8192, &bb.full[st]);
        bulk_load(sm.p[st], p.ws + p.L.f.pimg + rec * 8192, 8192, &bb.full[st]);
        bulk_load(sm.gam[st], p.ws + p.L.f.gam + rec * 256, 256, &bb.full[st]);
      }
      for (int j = (n >= 2 ? n - 2 : 0); j < n; ++j) rrole_wait(&bb.empty[j & 1], ph.empty[j & 1], abort);
    }
    return !*abort;
  }
  if (cx.warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    if (cx.lane == 0) {
      auto prep = [&](int j) {  // W = T_w K of chunk j
        const int st = j & 1;
        #pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tm + kRtW, kmajor_step(kmajor_desc(smem_u32(sm.tw[st]), 8192, 0), 8192, ks),
                    mnmajor_step(mnmajor_desc(smem_u32(sm.k[st]), 8192, 0), ks),
                    idesc_bf16(64, 128, 0, 1), ks > 0);
        umma_commit(&bb.pre_done);
      };
      rrole_wait(&bb.full[0], ph.full[0], abort);
      if (!*abort) prep(0);
      for (int j = 0; j < n && !*abort; ++j) {
        const int st = j & 1;
        // A: needs Q~, K~ of chunk j (staged1), dS of chunk j (epi2 of j - 1, or the initial
        // hand-off) and the dV' accumulator read (epi1 of j - 1)
        rrole_wait(&bb.staged1, ph.staged1, abort);
        rrole_wait(&bb.epi2, ph.epi2, abort);
        if (*abort) break;
        // Q~^T dO first: a_done then also covers it, so that the epilogue may restage Q~ right after
        #pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tm + kRtC, mnmajor_step(mnmajor_desc(smem_u32(sm.qt), 8192, 0), ks),
                    mnmajor_step(mnmajor_desc(smem_u32(sm.dout[st]), 8192, 0), ks),
                    idesc_bf16(128, 128, 1, 1), ks > 0);
        #pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tm + kRtA, kmajor_step(kmajor_desc(smem_u32(sm.kt), 8192, 0), 8192, ks),
                    mnmajor_step(mnmajor_desc(smem_u32(sm.ds), 16384, 0), ks),
                    idesc_bf16(64, 128, 0, 1), ks > 0);
        #pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tm + kRtA, mnmajor_step(mnmajor_desc(smem_u32(sm.p[st]), 8192, 0), ks),
                    mnmajor_step(mnmajor_desc(smem_u32(sm.dout[st]), 8192, 0), ks),
                    idesc_bf16(64, 128, 1, 1), 1);
        umma_commit(&bb.a_done);
        // B as soon as dV' and -W are staged; chunk j + 1's W as soon as its operands have landed
        // and W of chunk j has been read (staged2 of j), whichever comes first
        bool need_prep = j + 1 < n, b_issued = false, w_read = false;
        const long long t0 = clock64();
        while (!b_issued && !*abort) {
          if (!w_read && mbar_test(&bb.staged2, ph.staged2)) {
            ph.staged2 ^= 1;
            tc_fence_after();
            w_read = true;
          }
          if (need_prep && w_read && mbar_test(&bb.full[st ^ 1], ph.full[st ^ 1])) {
            ph.full[st ^ 1] ^= 1;
            tc_fence_after();
            prep(j + 1);
            need_prep = false;
          }
          if (w_read && mbar_test(&bb.epi1, ph.epi1)) {
            ph.epi1 ^= 1;
            tc_fence_after();
            #pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_bf16(tm + kRtC, mnmajor_step(mnmajor_desc(smem_u32(sm.wn), 8192, 0), ks),
                        mnmajor_step(mnmajor_desc(smem_u32(sm.dvp), 8192, 0), ks),
                        idesc_bf16(128, 128, 1, 1), 1);
            umma_commit(&bb.b_done);
            umma_commit(&bb.empty[st]);
            b_issued = true;
          } else if (clock64() - t0 > kWaitBudget) {
            *abort = 1;
          } else {
            __nanosleep(64);  // leave the issue slots of this SM sub-partition to the epilogue warps
          }
        }
        if (*abort) break;
        if (need_prep) {
          rrole_wait(&bb.full[st ^ 1], ph.full[st ^ 1], abort);
          if (*abort) break;
          prep(j + 1);
        }
      }
      rrole_wait(&bb.epi2, ph.epi2, abort);  // the epilogue's last dS hand-off
    }
    return !*abort;
  }
  // -------------------------------------------------------------------- epilogue warps 0-7
  const uint32_t lane_base = (uint32_t)(32 * cx.q4) << 16;
  // Q~, K~ of chunk j (from the stage)
  auto staging1 = [&](int j) {
    const int gc = chunk_of(j), st = j & 1, nn = clen[gc];
    rrole_wait(&bb.full[st], ph.full[st], abort);
    if (cx.tid < 128) {
      const float* gm = sm.gam[st];
      const int r = cx.tid & 63;
      sm.fsc[cx.tid >> 6][r] = (cx.tid < 64) ? ((r < nn) ? __expf(gm[r]) * p.scale : 0.f) : __expf(gm[63] - gm[r]);
    }
    r_sync();
    for (int e = cx.tid; e < 2 * 2 * 64 * 8; e += 256) {
      const int which = e >> 10, b = (e >> 9) & 1, r = (e >> 3) & 63, cj = e & 7;
      const uint32_t off = b * 8192 + r * 128 + ((cj ^ (r & 7)) << 4);
      const float sc = sm.fsc[which][r];
      uint4 raw = *reinterpret_cast<const uint4*>((which == 0 ? sm.q[st] : sm.k[st]) + off);
      __nv_bfloat162* x = reinterpret_cast<__nv_bfloat162*>(&raw);
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float2 f = __bfloat1622float2(x[u]);
        w[u] = pack_bf16x2(f.x * sc, f.y * sc);
      }
      *reinterpret_cast<uint4*>((which == 0 ? sm.qt : sm.kt) + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    r_handoff(cx.tid, &bb.staged1);
  };
  // -W of chunk j
  auto staging2 = [&]() {
    rrole_wait(&bb.pre_done, ph.pre_done, abort);
    // all 32 lanes: rows r0 = 16 q4 + lane / 4 and r0 + 8 of W (M = 64), column pairs
    const int c2 = 2 * (cx.lane & 3), r0 = 16 * cx.q4 + (cx.lane >> 2);
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      float v[16];
      tmem_ld16x256_x4(tm + kRtW + lane_base + 64 * cx.half + 32 * hc, v);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = 32 * hc + 8 * k + c2;
        *reinterpret_cast<uint32_t*>(sm.wn + cx.half * 8192 + sw128_pair(r0, c)) = pack_bf16x2(-v[4 * k], -v[4 * k + 1]);
        *reinterpret_cast<uint32_t*>(sm.wn + cx.half * 8192 + sw128_pair(r0 + 8, c)) =
            pack_bf16x2(-v[4 * k + 2], -v[4 * k + 3]);
      }
    }
    r_handoff(cx.tid, &bb.staged2);
  };
  // dL/dS at the end of chunk j (the bf16 image in sm.ds) goes to the records
  auto record_ds = [&](int j) {
    if (kRecord && cx.tid == 0 && chunk_of(j) < gc_rec) {
      bulk_wait_read_all();
      bulk_store(p.ws + p.L.ds_img + ((size_t)chunk_of(j) * Hv + h) * 32768, sm.ds, 32768);
      bulk_commit_group();
    }
    __syncwarp();
  };
  r_handoff(cx.tid, &bb.epi2);  // dS of the first chunk is staged
  staging1(0);
  staging2();
  record_ds(0);
  for (int j = 0; j < n; ++j) {
    const int gc = chunk_of(j), st = j & 1, nn = clen[gc];
    const float gC = sm.gam[st][63];
    rrole_wait(&bb.a_done, ph.a_done, abort);
    // dV' (rows beyond the chunk are zero), bf16
    if (kRecord && cx.tid == 0) bulk_wait_read_all();  // the previous dV' record has read sm.dvp
    __syncwarp();
    r_sync();
    {
      // all 32 lanes: rows t0 = 16 q4 + lane / 4 and t0 + 8 of dV' (M = 64), column pairs
      const int c2 = 2 * (cx.lane & 3), t0 = 16 * cx.q4 + (cx.lane >> 2);
      const float m0 = t0 < nn ? 1.f : 0.f, m1 = t0 + 8 < nn ? 1.f : 0.f;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float v[16];
        tmem_ld16x256_x4(tm + kRtA + lane_base + 64 * cx.half + 32 * hc, v);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 32 * hc + 8 * k + c2;
          *reinterpret_cast<uint32_t*>(sm.dvp + cx.half * 8192 + sw128_pair(t0, c)) =
              pack_bf16x2(v[4 * k] * m0, v[4 * k + 1] * m0);
          *reinterpret_cast<uint32_t*>(sm.dvp + cx.half * 8192 + sw128_pair(t0 + 8, c)) =
              pack_bf16x2(v[4 * k + 2] * m1, v[4 * k + 3] * m1);
        }
      }
    }
    r_handoff(cx.tid, &bb.epi1);
    if (kRecord && cx.tid == 0 && gc < gc_rec) {
      bulk_store(p.ws + p.L.dvp_img + ((size_t)gc * Hv + h) * 16384, sm.dvp, 16384);
      bulk_commit_group();
    }
    __syncwarp();
    if (j + 1 < n) staging1(j + 1);
    rrole_wait(&bb.b_done, ph.b_done, abort);
    {
      const float GC = __expf(gC);
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float v[32];
        tmem_ld16(tm + kRtC + lane_base + 64 * cx.half + 32 * hc, v);
        tmem_ld16(tm + kRtC + lane_base + 64 * cx.half + 32 * hc + 16, v + 16);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; x += 2) {  // two values per instruction
          const uint64_t r = f2_fma(f2_pack(GC, GC), f2_pack(dS[32 * hc + x], dS[32 * hc + x + 1]), f2_pack(v[x], v[x + 1]));
          dS[32 * hc + x] = f2_lo(r);
          dS[32 * hc + x + 1] = f2_hi(r);
        }
      }
      if (kRecord && cx.tid == 0) bulk_wait_read_all();  // the dS record of chunk j has read sm.ds
      __syncwarp();
      r_sync();
      rev_store_ds(cx, sm, dS);
    }
    r_handoff(cx.tid, &bb.epi2, &bb.empty[st]);
    if (j + 1 < n) {
      staging2();
      record_ds(j + 1);
    }
  }
  if (kRecord && cx.tid == 0) bulk_wait_all();
  return !*abort;
}

// This thread's row piece (row 32 q4 + lane, columns 64 half ... +63) of a 128x128 fp32 matrix.
__device__ __forceinline__ void rev_load(const Ctx& cx, const float* src, float* dS, bool add) {
  const float* row = src + (size_t)(32 * cx.q4 + cx.lane) * kDim + 64 * cx.half;
#pragma unroll
  for (int c = 0; c < 64; c += 4) {
    const float4 f = __ldcg(reinterpret_cast<const float4*>(row + c));
    if (add) {
      dS[c] += f.x;
      dS[c + 1] += f.y;
      dS[c + 2] += f.z;
      dS[c + 3] += f.w;
    } else {
      dS[c] = f.x;
      dS[c + 1] = f.y;
      dS[c + 2] = f.z;
      dS[c + 3] = f.w;
    }
  }
}
__device__ __forceinline__ void rev_save(const Ctx& cx, float* dst, const float* dS) {
  float* row = dst + (size_t)(32 * cx.q4 + cx.lane) * kDim + 64 * cx.half;
#pragma unroll
  for (int c = 0; c < 64; c += 4) *reinterpret_cast<float4*>(row + c) = make_float4(dS[c], dS[c + 1], dS[c + 2], dS[c + 3]);
}

// out = M^T dS + B on the tensor cores with compensated bf16 operands (x = hi + lo):
// M hi^T dS hi + M hi^T dS lo + M lo^T dS hi. M is the forward transition of a segment (fp32,
// row-major [dk][dk]); the reverse chain carries dL/dS through M^T. M's rows go unchanged into
// MN-major A blocks (row k of M = row k of the block, 64 m-values per block), which is M^T as
// the A operand. dS hi is in sm.ds (rev_store_ds). Staging (idle at the start of an item): M hi in
// sm.q, M lo in sm.k, dS lo in sm.dout (two 16 KB blocks each), the fp32 product in qt | kt. The
// epilogue threads (tid < 256) hold dS; all threads of the CTA call this.
__device__ bool rev_affine(Ctx& cx, RevSmem& sm, const float* Mm, const float* Bm, const float* dS, float* out) {
  uint8_t* mhi = sm.q[0];
  uint8_t* mlo = sm.k[0];
  uint8_t* dlo = sm.dout[0];
  if (cx.tid < 256) {
    // M hi / lo from coalesced loads (16 threads per 512-byte row), four 32-byte pieces in flight
#pragma unroll
    for (int k0 = 0; k0 < 8; k0 += 4) {
      float4 mv[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = cx.tid + 256 * (k0 + k);
        const float* src = Mm + (size_t)(e >> 4) * kDim + 8 * (e & 15);
        mv[2 * k] = __ldcg(reinterpret_cast<const float4*>(src));
        mv[2 * k + 1] = __ldcg(reinterpret_cast<const float4*>(src + 4));
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = cx.tid + 256 * (k0 + k), r = e >> 4, c8 = e & 15, cj = c8 & 7;
        const float x[8] = {mv[2 * k].x, mv[2 * k].y, mv[2 * k].z, mv[2 * k].w,
                            mv[2 * k + 1].x, mv[2 * k + 1].y, mv[2 * k + 1].z, mv[2 * k + 1].w};
        float lo[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) lo[u] = x[u] - __bfloat162float(__float2bfloat16_rn(x[u]));
        const uint32_t off = (c8 >> 3) * 16384 + r * 128 + ((cj ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(mhi + off) = pack8(x);
        *reinterpret_cast<uint4*>(mlo + off) = pack8(lo);
      }
    }
    const int rr = 32 * cx.q4 + cx.lane;
    uint8_t* dl = dlo + cx.half * 16384;
#pragma unroll
    for (int cj = 0; cj < 8; ++cj) {
      float lo[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) lo[u] = dS[8 * cj + u] - __bfloat162float(__float2bfloat16_rn(dS[8 * cj + u]));
      *reinterpret_cast<uint4*>(dl + rr * 128 + ((cj ^ (rr & 7)) << 4)) = pack8(lo);
    }
  }
  sync_generic_to_async();
  if (cx.tid == 0) {
    #pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma_bf16(cx.tmem + kRtC, mnmajor_step(mnmajor_desc(smem_u32(mhi), 16384, 0), ks),
                mnmajor_step(mnmajor_desc(smem_u32(sm.ds), 16384, 0), ks),
                idesc_bf16(128, 128, 1, 1), ks > 0);
    #pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma_bf16(cx.tmem + kRtC, mnmajor_step(mnmajor_desc(smem_u32(mhi), 16384, 0), ks),
                mnmajor_step(mnmajor_desc(smem_u32(dlo), 16384, 0), ks),
                idesc_bf16(128, 128, 1, 1), 1);
    #pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma_bf16(cx.tmem + kRtC, mnmajor_step(mnmajor_desc(smem_u32(mlo), 16384, 0), ks),
                mnmajor_step(mnmajor_desc(smem_u32(sm.ds), 16384, 0), ks),
                idesc_bf16(128, 128, 1, 1), 1);
  }
  if (!cx.commit_wait()) return false;
  // the product goes through a 32 KB fp32 stage, 64 rows at a time, with granule g of local row
  // rl at rl * 128 + 4 (g XOR rl mod 32), so that B is read and out written with coalesced accesses
  float* stg = reinterpret_cast<float*>(sm.qt);
  for (int pass = 0; pass < 2; ++pass) {
    if (cx.tid < 256 && (cx.q4 >> 1) == pass) {
      const int rl = 32 * (cx.q4 & 1) + cx.lane;
#pragma unroll
      for (int cc = 0; cc < 64; cc += 16) {
        float v[16];
        tmem_ld16(cx.tmem + kRtC + cx.lane_base() + 64 * cx.half + cc, v);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int g = (64 * cx.half + cc) / 4 + x;
          *reinterpret_cast<float4*>(stg + rl * 128 + 4 * ((g ^ rl) & 31)) =
              make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
        }
      }
    }
    __syncthreads();
    if (cx.tid < 256) {
      float4 b[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int e = cx.tid + 256 * k, r = 64 * pass + (e >> 5), g = e & 31;
        b[k] = __ldcg(reinterpret_cast<const float4*>(Bm + (size_t)r * kDim + 4 * g));
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int e = cx.tid + 256 * k, rl = e >> 5, g = e & 31;
        const float4 v = *reinterpret_cast<const float4*>(stg + rl * 128 + 4 * ((g ^ rl) & 31));
        *reinterpret_cast<float4*>(out + (size_t)(64 * pass + rl) * kDim + 4 * g) =
            make_float4(v.x + b[k].x, v.y + b[k].y, v.z + b[k].z, v.w + b[k].w);
      }
    }
    __syncthreads();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return true;
}

// Bring a 128x128 fp32 matrix into L2 ahead of its use (every thread of the CTA takes a share).
__device__ __forceinline__ void prefetch_state_l2(const float* m, int tid) {
  for (int l = tid; l < kDim * kDim * 4 / 128; l += kRevThreads) prefetch_l2(reinterpret_cast<const uint8_t*>(m) + 128 * l);
}

// Does some later document of the call start from document seq's final state (a fork)?
__device__ __forceinline__ bool doc_has_forks(const BwdParams& p, int seq) {
  if (!p.init_idx) return false;
  for (int x = seq + 1; x < p.d.N; ++x)
    if (p.init_idx[x] == p.d.n_init + seq) return true;
  return false;
}

__device__ __forceinline__ void rev_publish(int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    st_release(flag, 1);
  }
  __syncthreads();
}

// Reverse chain over the segments of the forward plan, exact split (the mirror of the forward's):
// with M_s the forward transition of segment s (S_end = M_s S_start + B_s), the gradient obeys
//   dL/dS_start(s) = M_s^T dL/dS_end(s) + Br_s,   Br_s = the reverse chain over s from zero.
//   kPass 1, per (segment, value head), no dependencies: Br_s for the inner segments of a split
//            document (neither first nor last); for its last segment, when no document forks from
//            it, dL/dS at the segment start directly (published at once).
//   kPass 2, per (segment, value head) in descending segment order: the end gradient is dfinal
//            (+ the forked documents' start gradients) for a last segment, else the published start
//            gradient of segment s + 1 (or Br_{s+1} when M_{s+1} is exactly zero); an inner segment
//            publishes its start gradient M_s^T dS_end + Br_s before it runs; then the chunks in
//            reverse with records; a first segment writes dL/dS at the document start.
// Every wait is on an item with a smaller ticket, so the queue cannot deadlock.
template <int kPass>
__global__ void __launch_bounds__(kRevThreads, 1) rev_chain_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  RevSmem& sm = *reinterpret_cast<RevSmem*>(smem_align1024(smem_raw));
  __shared__ uint64_t bar_ld, bar_mma;
  __shared__ RevBars rbars;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_item, s_ok, s_abort;
  griddep_launch_dependents();
  griddep_wait();  // everything the kernels before this one write
  Header* hd = reinterpret_cast<Header*>(p.ws + p.L.f.header);
  Header* h2 = reinterpret_cast<Header*>(p.ws + p.L.hdr2);
  const int N = p.d.N, Hv = p.d.Hv, G = p.d.Hv / p.d.Hk;
  const int n_segs = hd->n_segs;
  const int n_items = n_segs * Hv;
  if (blockIdx.x >= n_items || get_status(hd) != 0) return;
  Ctx cx;
  ctx_init(cx, &bar_ld, &bar_mma);
  const bool epi = cx.tid < 256;  // threads that hold dS rows
  RevPhase ph;
  memset(&ph, 0, sizeof(ph));
  if (cx.tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&rbars.full[0], 1);
    mbar_init(&rbars.full[1], 1);
    mbar_init(&rbars.empty[0], 2);
    mbar_init(&rbars.empty[1], 2);
    mbar_init(&rbars.pre_done, 1);
    mbar_init(&rbars.staged1, 1);
    mbar_init(&rbars.staged2, 1);
    mbar_init(&rbars.a_done, 1);
    mbar_init(&rbars.epi1, 1);
    mbar_init(&rbars.b_done, 1);
    mbar_init(&rbars.epi2, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (cx.warp == 0) tmem_alloc(&tmem_holder, 512);
  sync_generic_to_async();
  cx.tmem = tmem_holder;
  const int32_t* seq_seg0 = reinterpret_cast<const int32_t*>(p.ws + p.L.f.seq_seg0);
  const int32_t* si = reinterpret_cast<const int32_t*>(p.ws + p.L.f.seg_info);
  const int32_t* slot = reinterpret_cast<const int32_t*>(p.ws + p.L.f.seg_slot);
  const int* mzero = reinterpret_cast<const int*>(p.ws + p.L.f.mzero);
  const float* mmat = reinterpret_cast<const float*>(p.ws + p.L.f.mmat);
  const float* gam_ws = reinterpret_cast<const float*>(p.ws + p.L.f.gam);
  const int32_t* contr = reinterpret_cast<const int32_t*>(p.ws + p.L.f.contr);
  const int32_t* dch = reinterpret_cast<const int32_t*>(p.ws + p.L.f.seq_chunk0);
  float* ds0 = reinterpret_cast<float*>(p.ws + p.L.ds0);
  float* rpub = reinterpret_cast<float*>(p.ws + p.L.rpub);
  float* rb = reinterpret_cast<float*>(p.ws + p.L.rb);
  int* flags = reinterpret_cast<int*>(p.ws + p.L.flags_ds0);
  int* rflags = reinterpret_cast<int*>(p.ws + p.L.flags_rseg);
  const size_t st = (size_t)kDim * kDim;
  float dS[64];
  // wait for `flag` (uniform outcome)
  auto wait_uniform = [&](const int* flag) -> bool {
    if (cx.tid == 0) {
      s_ok = wait_flag(flag, hd, p.flag_budget) ? 1 : 0;
      __threadfence();
    }
    __syncthreads();
    const bool ok = s_ok != 0;
    __syncthreads();
    return ok;
  };
  // dL/dS at a document's end: dfinal plus the start gradients of the documents forked from it
  auto doc_end_grad = [&](int seq, int h) -> bool {
    if (epi) {
      if (p.dfinal)
        rev_load(cx, p.dfinal + ((size_t)seq * Hv + h) * st, dS, false);
      else
        for (int c = 0; c < 64; ++c) dS[c] = 0.f;
    }
    if (p.init_idx)
      for (int x = seq + 1; x < N; ++x) {
        if (p.init_idx[x] != p.d.n_init + seq) continue;
        if (!wait_uniform(&flags[x * Hv + h])) return false;
        if (epi) rev_load(cx, ds0 + ((size_t)x * Hv + h) * st, dS, true);
      }
    return true;
  };
  // chunks [c0, c0 + nch) in reverse; with `record`, records for the chunks below rec_end
  auto run = [&](int c0, int nch, int h, int hk, bool record, int rec_end) -> bool {
    if (epi) rev_store_ds(cx, sm, dS);
    sync_generic_to_async();
    if (record)
      run_rev_ws<true>(p, cx, sm, rbars, ph, &s_abort, dS, c0, c0 + nch, h, hk, rec_end);
    else
      run_rev_ws<false>(p, cx, sm, rbars, ph, &s_abort, dS, c0, c0 + nch, h, hk, c0);
    __syncthreads();
    return s_abort == 0;
  };
  for (;;) {
    if (cx.tid == 0) {
      const int it = (int)atomicAdd(kPass == 1 ? &h2->q_p1 : &h2->q_chain, 1u);
      s_item = (get_status(hd) != 0) ? n_items : it;
    }
    __syncthreads();
    const int item = s_item;
    __syncthreads();  // s_item is rewritten by the next ticket
    if (item >= n_items) break;
    const int s = (kPass == 1) ? item / Hv : n_segs - 1 - item / Hv;
    const int h = item % Hv, hk = h / G;
    const int seq = si[4 * s], c0 = si[4 * s + 1], nch = si[4 * s + 2];
    const int first = seq_seg0[seq], last = seq_seg0[seq + 1] - 1;
    bool ok = true;
    // exact split, reversed: the previous segment's item needs this segment's start gradient only
    // when it cannot warm up over this segment's first chunks; this item warms up the same way
    const bool prev_warms = s > first && warm_fwd(gam_ws, contr, Hv, h, c0, dch[seq + 1]) >= 0;
    if (kPass == 1) {
      if (first == last || s == first || prev_warms) continue;  // nothing to precompute
      if (s < last) {
        if (epi)
          for (int c = 0; c < 64; ++c) dS[c] = 0.f;
        ok = run(c0, nch, h, hk, false, c0);
        if (!ok) break;
        if (epi) rev_save(cx, rb + ((size_t)slot[s] * Hv + h) * st, dS);
        __syncthreads();
        continue;
      }
      if (doc_has_forks(p, seq)) continue;  // its end gradient waits for the forked documents
      ok = doc_end_grad(seq, h) && run(c0, nch, h, hk, false, c0);
      if (!ok) break;
      if (epi) rev_save(cx, rpub + ((size_t)slot[s - 1] * Hv + h) * st, dS);
      rev_publish(&rflags[s * Hv + h]);
      continue;
    }
    // ----------------------------------------------------------------- pass 2
    const bool pub_prev = first < s && s < last && !prev_warms && !mzero[slot[s] * Hv + h];
    if (pub_prev) {  // early publication below
      const size_t o = ((size_t)slot[s] * Hv + h) * st;
      prefetch_state_l2(mmat + o, cx.tid);
      prefetch_state_l2(rb + o, cx.tid);
    }
    const int wf = s < last ? warm_fwd(gam_ws, contr, Hv, h, c0 + nch, dch[seq + 1]) : -1;
    if (s == last) {
      ok = doc_end_grad(seq, h);
    } else if (wf >= 0) {
      // the decay over chunks [c0 + nch, wf) leaves the later gradient below fp32 resolution:
      // warm up from zero over them (a run of its own: a lighter path than the recording one,
      // and the early publication below needs dL/dS at the segment end)
      if (epi)
        for (int c = 0; c < 64; ++c) dS[c] = 0.f;
      ok = run(c0 + nch, wf - (c0 + nch), h, hk, false, c0);
    } else if (s + 1 != last && mzero[slot[s + 1] * Hv + h]) {
      if (epi) rev_load(cx, rb + ((size_t)slot[s + 1] * Hv + h) * st, dS, false);  // M_{s+1} = 0: no wait
    } else {
      ok = wait_uniform(&rflags[(s + 1) * Hv + h]);
      if (ok && epi) rev_load(cx, rpub + ((size_t)slot[s] * Hv + h) * st, dS, false);
    }
    if (!ok) break;
    if (pub_prev) {
      // early publication of this segment's start gradient
      if (epi) rev_store_ds(cx, sm, dS);
      sync_generic_to_async();
      const size_t o = ((size_t)slot[s] * Hv + h) * st;
      if (!rev_affine(cx, sm, mmat + o, rb + o, dS, rpub + ((size_t)slot[s - 1] * Hv + h) * st)) {
        set_status(hd, kErrTimeout);
        break;
      }
      rev_publish(&rflags[s * Hv + h]);
    }
    if (!run(c0, nch, h, hk, true, c0 + nch)) {
      set_status(hd, kErrTimeout);
      break;
    }
    if (first < s && s == last && !prev_warms && doc_has_forks(p, seq)) {
      if (epi) rev_save(cx, rpub + ((size_t)slot[s - 1] * Hv + h) * st, dS);
      rev_publish(&rflags[s * Hv + h]);
    }
    if (s == first) {
      if (epi) rev_save(cx, ds0 + ((size_t)seq * Hv + h) * st, dS);
      rev_publish(&flags[seq * Hv + h]);
    }
    __syncthreads();
  }
  if (s_abort && cx.tid == 0) set_status(hd, kErrTimeout);
  if (cx.tid == 0) {
    umma_commit(&bar_mma);
    mbar_wait(&bar_mma, cx.ph_mma, kWaitBudget);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (cx.warp == 0) tmem_dealloc(cx.tmem, 512);
}

// ===================================================================================== gradients

struct GradSmem {
  uint8_t q[2][8192];
  uint8_t k[2][8192];
  uint8_t tb[24576];       // T fp32 [0, 16K) (fz layout), T bf16 image [16K, 24K)
  uint8_t bS[2][16384];    // S_c image (the next head's once (b) has read it)
  uint8_t bdS[2][16384];   // dS_{c+1} image  | phase 2: T_w [0, 8K), T_u [8K, 16K), dT [16K, 24K), R [24K, 32K)
  uint8_t bVp[2][8192];    // V' -> V'_s (then the next head's V')
  uint8_t bdVp[2][8192];   // dV'             | fp32 64x64 scratch (kx products)
  uint8_t bdO[2][8192];    // dO              | phase 2: V
  uint8_t bW[2][8192];     // fp32 scratch (dEg) | dW rows t
  uint8_t bP[8192];        // scale dQK, then L = dA o diag(beta) E (strictly lower)
  float scr[4096];         // fp32 64x64 scratch (fz): vy products, then L o KK
  float gam[2][64];        // [head parity] gamma
  float beta[64], Gm[64], Gi[64];  // beta, e^{gamma}, e^{-gamma}
  float part[8][64];
  float vy[64], kx[64], cA[64], db3[2][64];
  float red4[2][4][64];    // partial column sums (two matrices x four row quarters)
  float red[8];
};
constexpr size_t kGradSmemBytes = sizeof(GradSmem) + 1024;
// Chunk decay above which e^{gamma_i} and e^{-gamma_j} both stay finite in fp32 (gamma is the
// chunk-local cumulative log-decay, nonincreasing, so gamma_63 is its minimum).
constexpr float kFactorMin = -80.f;
// TMEM: K K^T and Q K^T of the key head (kept for the whole CTA), dk, two working accumulators
constexpr uint32_t kGtC = 0, kGtK = 128, kGt1 = 256, kGt2 = 384;

// Column sums of one or two fp32 64x64 fz matrices over rows [0, 64) with all 256 threads:
// out[j] = sum_i X[i][j]. Ends with the result visible to every thread.
__device__ __forceinline__ void col_sums(GradSmem& sm, const float* X, const float* Y, float* outx, float* outy,
                                         int tid) {
  const int j = tid & 63, q = tid >> 6;
  float a = 0.f, b = 0.f;
#pragma unroll 4
  for (int i = 16 * q; i < 16 * q + 16; ++i) {
    a += X[fz(i, j)];
    if (Y) b += Y[fz(i, j)];
  }
  sm.red4[0][q][j] = a;
  sm.red4[1][q][j] = b;
  __syncthreads();
  if (tid < 64) {
    outx[tid] = (sm.red4[0][0][tid] + sm.red4[0][1][tid]) + (sm.red4[0][2][tid] + sm.red4[0][3][tid]);
    if (Y) outy[tid] = (sm.red4[1][0][tid] + sm.red4[1][1][tid]) + (sm.red4[1][2][tid] + sm.red4[1][3][tid]);
  }
  __syncthreads();
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(256, 1) grad_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  GradSmem& sm = *reinterpret_cast<GradSmem*>(smem_align1024(smem_raw));
  __shared__ uint64_t bar_ld, bar_mma, bar_p1, bar_v, bar_tw;
  __shared__ uint32_t tmem_holder;
  griddep_launch_dependents();
  griddep_wait();  // the records and the reverse chain's state gradients
  Header* hd = reinterpret_cast<Header*>(p.ws + p.L.f.header);
  const int chunk = blockIdx.x, hk = blockIdx.y;
  if (chunk >= hd->n_chunks || get_status(hd) != 0) return;
  const int Hv = p.d.Hv, Hk = p.d.Hk, G = Hv / Hk;
  const int tok0 = reinterpret_cast<const int32_t*>(p.ws + p.L.f.chunk_tok0)[chunk];
  const int n = reinterpret_cast<const int32_t*>(p.ws + p.L.f.chunk_len)[chunk];
  Ctx cx;
  ctx_init(cx, &bar_ld, &bar_mma);
  const int tid = cx.tid;
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_p1, 1);
    mbar_init(&bar_v, 1);
    mbar_init(&bar_tw, 1);
    fence_mbar_init();
  }
  uint32_t ph_p1 = 0, ph_v = 0, ph_tw = 0;
  bool p1_seen = false;  // the first head's record phase has been waited for
  // bounded wait of every thread on one of the load barriers (uniform outcome)
  auto wait_bar = [&](uint64_t* bar, uint32_t& ph) -> bool {
    if (!wait_all(bar, ph)) return false;
    ph ^= 1;
    tc_fence_after();
    return true;
  };
  // Loads of one value head's records, in the order their buffers become free. The phase-1 set
  // (S, dS, V', dV', dO images and gamma) lands on bar_p1: its transaction count is armed by the
  // first piece, the other pieces follow as the previous head releases their buffers.
  const uint32_t kP1Bytes = 32768 + 16384 + 2 * 8192;  // gamma, V' and S are counted where issued
  auto rec_of = [&](int hh2) { return (size_t)chunk * Hv + hk * G + hh2; };
  auto load_do_gam = [&](int hh2) {  // thread 0; arms bar_p1
    mbar_expect_tx(&bar_p1, 256);
    bulk_load(sm.gam[hh2 & 1], p.ws + p.L.f.gam + rec_of(hh2) * 256, 256, &bar_p1);
    mbar_arrive_expect_tx(&bar_p1, kP1Bytes);
    tma_load_3d(sm.bdO[0], &p.tm_do, 0, hk * G + hh2, tok0, &bar_p1);
    tma_load_3d(sm.bdO[1], &p.tm_do, 64, hk * G + hh2, tok0, &bar_p1);
  };
  auto load_dvp = [&](int hh2) { bulk_load(sm.bdVp[0], p.ws + p.L.dvp_img + rec_of(hh2) * 16384, 16384, &bar_p1); };
  auto load_s = [&](int hh2) {
    mbar_expect_tx(&bar_p1, 32768);
    bulk_load(sm.bS[0], p.ws + p.L.st_img + rec_of(hh2) * 32768, 32768, &bar_p1);
  };
  auto load_ds = [&](int hh2) { bulk_load(sm.bdS[0], p.ws + p.L.ds_img + rec_of(hh2) * 32768, 32768, &bar_p1); };
  auto load_vp = [&](int hh2) {
    mbar_expect_tx(&bar_p1, 16384);
    bulk_load(sm.bVp[0], p.ws + p.L.vp_img + rec_of(hh2) * 16384, 16384, &bar_p1);
  };
  if (cx.warp == 0) tmem_alloc(&tmem_holder, 512);
  sync_generic_to_async();
  cx.tmem = tmem_holder;
  const uint32_t tm = cx.tmem;
  bool ok = true;
  const int i_row = 16 * cx.q4 + cx.lane;  // row held by this thread in M = 64 accumulators (lane < 16)
  const bool has_row = cx.lane < 16;

  // ---- per key head: Q, K, K K^T, Q K^T (the first head's records are already on their way: their
  // buffers are free at the start)
  if (tid == 0) {
    // the pieces with their own expect_tx first: the arrival in load_do_gam must come last
    load_s(0);
    load_vp(0);
    load_do_gam(0);
    load_dvp(0);
    load_ds(0);
    mbar_arrive_expect_tx(&bar_ld, 4 * 8192);
    tma_load_3d(sm.q[0], &p.tm_q, 0, hk, tok0, &bar_ld);
    tma_load_3d(sm.q[1], &p.tm_q, 64, hk, tok0, &bar_ld);
    tma_load_3d(sm.k[0], &p.tm_k, 0, hk, tok0, &bar_ld);
    tma_load_3d(sm.k[1], &p.tm_k, 64, hk, tok0, &bar_ld);
  }
  ok = cx.wait_ld();
  if (ok) {
    if (tid == 0) {
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        umma_bf16(tm + kGtC, kmajor_step(kmajor_desc(smem_u32(sm.k[0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.k[0]), 8192, 0), 8192, ks),
                  idesc_bf16(64, 64, 0, 0), ks > 0);
        umma_bf16(tm + kGtC + 64, kmajor_step(kmajor_desc(smem_u32(sm.q[0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.k[0]), 8192, 0), 8192, ks),
                  idesc_bf16(64, 64, 0, 0), ks > 0);
      }
    }
    ok = cx.commit_wait();  // K K^T and Q K^T stay in TMEM, read where needed
  }
  __syncthreads();

  bool first_k = true;
  for (int hh = 0; hh < G && ok; ++hh) {
    const int h = hk * G + hh;
    const size_t rec = (size_t)chunk * Hv + h;
    const bool next = hh + 1 < G;
    if (tid == 224) {  // a thread that issues neither loads nor MMAs
      // this head's later loads and the next head's records into L2 now: each buffer is refilled
      // only once the previous use frees it, and the fill then waits on L2 instead of HBM
      bulk_prefetch_l2(p.ws + p.L.t_f32 + rec * 16384, 16384);
      bulk_prefetch_l2(p.ws + p.L.f.tw + rec * 8192, 8192);
      bulk_prefetch_l2(p.ws + p.L.f.tu + rec * 8192, 8192);
      tma_prefetch_3d(&p.tm_v, 0, h, tok0);
      tma_prefetch_3d(&p.tm_v, 64, h, tok0);
      if (next) {
        const size_t r1 = rec + 1;
        tma_prefetch_3d(&p.tm_do, 0, h + 1, tok0);
        tma_prefetch_3d(&p.tm_do, 64, h + 1, tok0);
        bulk_prefetch_l2(p.ws + p.L.dvp_img + r1 * 16384, 16384);
        bulk_prefetch_l2(p.ws + p.L.st_img + r1 * 32768, 32768);
        bulk_prefetch_l2(p.ws + p.L.ds_img + r1 * 32768, 32768);
        bulk_prefetch_l2(p.ws + p.L.vp_img + r1 * 16384, 16384);
      }
    }
    if (tid < 64) sm.beta[tid] = (tid < n) ? p.beta[(size_t)(tok0 + tid) * Hv + h] : 0.f;
    p1_seen = true;
    if (!(ok = wait_bar(&bar_p1, ph_p1))) break;
    const float* gam = sm.gam[hh & 1];
    if (tid == 0 && next) {  // the next head's gamma, into the other buffer, on the next phase
      mbar_expect_tx(&bar_p1, 256);
      bulk_load(sm.gam[(hh + 1) & 1], p.ws + p.L.f.gam + rec_of(hh + 1) * 256, 256, &bar_p1);
    }
    if (tid < 64) {
      sm.Gm[tid] = __expf(gam[tid]);
      sm.Gi[tid] = __expf(-gam[tid]);
    }
    __syncthreads();
    const float gC = gam[63], GC = __expf(gC);
    float* dEg = reinterpret_cast<float*>(sm.bW[0]);
    // ---------------- (a) dP = dO V'^T ; K dS
    if (tid == 0) {
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kGt1, kmajor_step(kmajor_desc(smem_u32(sm.bdO[0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.bVp[0]), 8192, 0), 8192, ks),
                  idesc_bf16(64, 64, 0, 0), ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kGt2, kmajor_step(kmajor_desc(smem_u32(sm.k[0]), 8192, 0), 8192, ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.bdS[0]), 16384, 0), ks),
                  idesc_bf16(64, 128, 0, 1), ks > 0);
    }
    if (!(ok = cx.commit_wait())) break;
    {
      // all 32 lanes: rows r0 = 16 q4 + lane / 4 and r0 + 8, column pairs (tmem_ld16x256_x4)
      const int c2 = 2 * (cx.lane & 3);
      const int rw[2] = {16 * cx.q4 + (cx.lane >> 2), 16 * cx.q4 + (cx.lane >> 2) + 8};
      // e^{gamma_i - gamma_j} as e^{gamma_i} e^{-gamma_j} while both factors stay finite
      const bool factored = gam[63] > kFactorMin;
      float rs[2] = {0.f, 0.f};
      {
        float v[16], ev[16], qkv[16];
        tmem_ld16x256_x4(tm + kGt1 + cx.lane_base() + 32 * cx.half, v);
        tmem_ld16x256_x4(tm + kGtC + 64 + cx.lane_base() + 32 * cx.half, qkv);
        if (factored) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              ev[4 * k + q] = sm.Gm[rw[q >> 1]] * sm.Gi[32 * cx.half + 8 * k + c2 + (q & 1)];
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              ev[4 * k + q] = __expf(gam[rw[q >> 1]] - gam[32 * cx.half + 8 * k + c2 + (q & 1)]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int r = rw[rr], j = 32 * cx.half + 8 * k + c2;
            const float d0 = (j <= r && r < n) ? v[4 * k + 2 * rr] * ev[4 * k + 2 * rr] : 0.f;
            const float d1 = (j + 1 <= r && r < n) ? v[4 * k + 2 * rr + 1] * ev[4 * k + 2 * rr + 1] : 0.f;
            *reinterpret_cast<uint32_t*>(sm.bP + sw128_pair(r, j)) = pack_bf16x2(d0 * p.scale, d1 * p.scale);
            const float e0 = d0 * qkv[4 * k + 2 * rr] * p.scale, e1 = d1 * qkv[4 * k + 2 * rr + 1] * p.scale;
            *reinterpret_cast<float2*>(dEg + fz(r, j)) = make_float2(e0, e1);
            rs[rr] += e0 + e1;
          }
      }
      rs[0] = quad_sum(rs[0]);
      rs[1] = quad_sum(rs[1]);
      if ((cx.lane & 3) == 0) {
        sm.part[0 + cx.half][rw[0]] = rs[0];
        sm.part[0 + cx.half][rw[1]] = rs[1];
      }
      float kt[2] = {0.f, 0.f};
#pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        float v[16];
        tmem_ld16x256_x4(tm + kGt2 + cx.lane_base() + 64 * cx.half + cc, v);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(
                sm.bVp[cx.half] + sw128_pair(rw[rr], cc + 8 * k + c2)));
            kt[rr] += a.x * v[4 * k + 2 * rr] + a.y * v[4 * k + 2 * rr + 1];
          }
      }
      kt[0] = quad_sum(kt[0]);
      kt[1] = quad_sum(kt[1]);
      if ((cx.lane & 3) == 0) {
        sm.part[2 + cx.half][rw[0]] = kt[0];
        sm.part[2 + cx.half][rw[1]] = kt[1];
      }
    }
    __syncthreads();
    col_sums(sm, dEg, nullptr, sm.part[4], nullptr, tid);
    // ---------------- (b) dV' S^T (-> dW) ; <dS, S>  (the term of dgamma in q S dO is dq_kernel's)
    if (tid == 0) {
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kGt2, kmajor_step(kmajor_desc(smem_u32(sm.bdVp[0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.bS[0]), 16384, 0), 16384, ks),
                  idesc_bf16(64, 128, 0, 0), ks > 0);
    }
    {
      // Frobenius product of the two state images (same layout, so element-by-element)
      float fr = 0.f;
      for (int o = tid * 16; o < 32768; o += 256 * 16) {
        uint4 a = *reinterpret_cast<const uint4*>(sm.bS[0] + o);
        uint4 b = *reinterpret_cast<const uint4*>(sm.bdS[0] + o);
        const __nv_bfloat162* xa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* xb = reinterpret_cast<const __nv_bfloat162*>(&b);
        for (int u = 0; u < 4; ++u) {
          float2 fa = __bfloat1622float2(xa[u]), fb = __bfloat1622float2(xb[u]);
          fr += fa.x * fb.x + fa.y * fb.y;
        }
      }
      fr = warp_sum(fr);
      if (cx.lane == 0) sm.red[cx.warp] = fr;
    }
    if (!(ok = cx.commit_wait())) break;
    if (tid == 0) {  // T (fp32) into its buffer (phase 2); S is read: the next head's S
      mbar_arrive_expect_tx(&bar_v, 16384 + 2 * 8192);
      bulk_load(sm.tb, p.ws + p.L.t_f32 + rec * 16384, 16384, &bar_v);
      if (next) load_s(hh + 1);
    }
    {
      // all 32 lanes: rows r0 = 16 q4 + lane / 4 and r0 + 8, column pairs (tmem_ld16x256_x4)
      const int c2 = 2 * (cx.lane & 3);
      const int rw[2] = {16 * cx.q4 + (cx.lane >> 2), 16 * cx.q4 + (cx.lane >> 2) + 8};
#pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        float w[16];
        tmem_ld16x256_x4(tm + kGt2 + cx.lane_base() + 64 * cx.half + cc, w);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int c = cc + 8 * k + c2, x = 4 * k + 2 * rr;
            *reinterpret_cast<uint32_t*>(sm.bW[cx.half] + sw128_pair(rw[rr], c)) = pack_bf16x2(-w[x], -w[x + 1]);
          }
      }
    }
    // ---------------- (c) V'_s = diag(e^{gamma_C - gamma}) V' ; dk accumulation (dq has its own kernel)
    if (tid < 64) sm.cA[tid] = __expf(gC - gam[tid]);
    __syncthreads();
    if (tid == 0) {  // dO is read: V into its buffer (phase 2)
      tma_load_3d(sm.bdO[0], &p.tm_v, 0, h, tok0, &bar_v);
      tma_load_3d(sm.bdO[1], &p.tm_v, 64, h, tok0, &bar_v);
    }
    scale_rows(sm.bVp[0], sm.cA, tid);
    scale_rows(sm.bVp[1], sm.cA, tid);
    sync_generic_to_async();
    if (tid == 0) {
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kGtK, kmajor_step(kmajor_desc(smem_u32(sm.bVp[0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.bdS[0]), 16384, 0), 16384, ks),
                  idesc_bf16(64, 128, 0, 0), (!first_k || ks > 0) ? 1 : 0);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kGtK, mnmajor_step(mnmajor_desc(smem_u32(sm.bP), 8192, 0), ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.q[0]), 8192, 0), ks),
                  idesc_bf16(64, 128, 1, 1), 1);
    }
    first_k = false;
    const float fro = ((sm.red[0] + sm.red[1]) + (sm.red[2] + sm.red[3])) + ((sm.red[4] + sm.red[5]) + (sm.red[6] + sm.red[7]));
    if (!(ok = cx.commit_wait())) break;
    if (tid == 0 && next) load_vp(hh + 1);  // V'_s is read: the next head's V'
    // ---------------- phase 2 loads: T_w, T_u (dS is read); V and T were issued earlier
    if (tid == 0) {
      mbar_arrive_expect_tx(&bar_tw, 2 * 8192);
      bulk_load(sm.bdS[0], p.ws + p.L.f.tw + rec * 8192, 8192, &bar_tw);
      bulk_load(sm.bdS[0] + 8192, p.ws + p.L.f.tu + rec * 8192, 8192, &bar_tw);
    }
    if (!(ok = wait_bar(&bar_v, ph_v))) break;
    if (!(ok = wait_bar(&bar_tw, ph_tw))) break;
    const float* Tf = reinterpret_cast<const float*>(sm.tb);
    uint8_t* Tb = sm.tb + 16384;            // T bf16 image
    uint8_t* Tw = sm.bdS[0];
    uint8_t* Tu = sm.bdS[0] + 8192;
    uint8_t* dTt = sm.bdS[1];
    uint8_t* Rt = sm.bdS[1] + 8192;
    for (int e = tid; e < 64 * 8; e += 256) {
      const int r = e >> 3, cj = e & 7;
      const float4 t0 = *reinterpret_cast<const float4*>(Tf + fz(r, 8 * cj));
      const float4 t1 = *reinterpret_cast<const float4*>(Tf + fz(r, 8 * cj + 4));
      const float x[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
      *reinterpret_cast<uint4*>(Tb + r * 128 + ((cj ^ (r & 7)) << 4)) = pack8(x);
    }
    sync_generic_to_async();
    // ---------------- (d) dv = T_u^T dV' ; D1 = dV' V^T ; D2 = dW K^T ; dk += T_w^T dW
    if (tid == 0) {
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kGt1, mnmajor_step(mnmajor_desc(smem_u32(Tu), 8192, 0), ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.bdVp[0]), 8192, 0), ks),
                  idesc_bf16(64, 128, 1, 1), ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kGt2, kmajor_step(kmajor_desc(smem_u32(sm.bdVp[0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.bdO[0]), 8192, 0), 8192, ks),
                  idesc_bf16(64, 64, 0, 0), ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kGt2 + 64, kmajor_step(kmajor_desc(smem_u32(sm.bW[0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.k[0]), 8192, 0), 8192, ks),
                  idesc_bf16(64, 64, 0, 0), ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kGtK, mnmajor_step(mnmajor_desc(smem_u32(Tw), 8192, 0), ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.bW[0]), 8192, 0), ks),
                  idesc_bf16(64, 128, 1, 1), 1);
    }
    if (!(ok = cx.commit_wait())) break;
    if (tid == 0 && next) {  // V is read: the next head's dO (gamma follows once (h) is done)
      mbar_arrive_expect_tx(&bar_p1, kP1Bytes);
      tma_load_3d(sm.bdO[0], &p.tm_do, 0, h + 1, tok0, &bar_p1);
      tma_load_3d(sm.bdO[1], &p.tm_do, 64, h + 1, tok0, &bar_p1);
    }
    float* vyM = sm.scr;
    float* kxM = reinterpret_cast<float*>(sm.bdVp[0]);
    {
      // all 32 lanes: rows r0 = 16 q4 + lane / 4 and r0 + 8, column pairs (tmem_ld16x256_x4)
      const int c2 = 2 * (cx.lane & 3);
      const int rw[2] = {16 * cx.q4 + (cx.lane >> 2), 16 * cx.q4 + (cx.lane >> 2) + 8};
#pragma unroll
      for (int cc = 0; cc < 64; cc += 32) {
        float v[16];
        tmem_ld16x256_x4(tm + kGt1 + cx.lane_base() + 64 * cx.half + cc, v);
        tmem_ld_wait();
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
          if (rw[rr] < n) {
            float* dvrow = p.dv + ((size_t)(tok0 + rw[rr]) * Hv + h) * kDim + 64 * cx.half + cc + c2;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              *reinterpret_cast<float2*>(dvrow + 8 * k) = make_float2(v[4 * k + 2 * rr], v[4 * k + 2 * rr + 1]);
          }
      }
      {
        float d1[16], d2[16];
        tmem_ld16x256_x4(tm + kGt2 + cx.lane_base() + 32 * cx.half, d1);
        tmem_ld16x256_x4(tm + kGt2 + 64 + cx.lane_base() + 32 * cx.half, d2);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int j = 32 * cx.half + 8 * k + c2;
          const float b0 = sm.beta[j], b1 = sm.beta[j + 1];
          const float bg0 = b0 * sm.Gm[j], bg1 = b1 * sm.Gm[j + 1];
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const int r = rw[rr], x = 4 * k + 2 * rr;
            const float2 tf = *reinterpret_cast<const float2*>(Tf + fz(r, j));
            *reinterpret_cast<uint32_t*>(dTt + sw128_pair(r, j)) =
                pack_bf16x2(d1[x] * b0 + d2[x] * bg0, d1[x + 1] * b1 + d2[x + 1] * bg1);
            *reinterpret_cast<float2*>(vyM + fz(r, j)) = make_float2(tf.x * d1[x], tf.y * d1[x + 1]);
            *reinterpret_cast<float2*>(kxM + fz(r, j)) = make_float2(tf.x * d2[x], tf.y * d2[x + 1]);
          }
        }
      }
    }
    sync_generic_to_async();
    // ---------------- (e) R = dT T^T (the column sums of vy / kx run meanwhile)
    if (tid == 0)
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kGt1, kmajor_step(kmajor_desc(smem_u32(dTt), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(Tb), 8192, 0), 8192, ks),
                  idesc_bf16(64, 64, 0, 0), ks > 0);
    col_sums(sm, vyM, kxM, sm.vy, sm.kx, tid);
    if (tid == 0 && next) load_dvp(hh + 1);  // the kx scratch is summed: the next head's dV'
    if (!(ok = cx.commit_wait())) break;
    {
      const int c2 = 2 * (cx.lane & 3), r0 = 16 * cx.q4 + (cx.lane >> 2);
      float v[16];
      tmem_ld16x256_x4(tm + kGt1 + cx.lane_base() + 32 * cx.half, v);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = 32 * cx.half + 8 * k + c2;
        *reinterpret_cast<uint32_t*>(Rt + sw128_pair(r0, j)) = pack_bf16x2(v[4 * k], v[4 * k + 1]);
        *reinterpret_cast<uint32_t*>(Rt + sw128_pair(r0 + 8, j)) = pack_bf16x2(v[4 * k + 2], v[4 * k + 3]);
      }
    }
    sync_generic_to_async();
    // ---------------- (f) dA = -(T^T R), strictly lower and inside the chunk. With E_ij = e^{gamma_i -
    // gamma_j}: L = dA o diag(beta) E (bf16, for dk += (L + L^T) K), the row sums of dA o E o KK
    // (dbeta) and the matrix L o KK for its column sums (dgamma).
    if (tid == 0)
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kGt1, mnmajor_step(mnmajor_desc(smem_u32(Tb), 8192, 0), ks),
                  mnmajor_step(mnmajor_desc(smem_u32(Rt), 8192, 0), ks),
                  idesc_bf16(64, 64, 1, 1), ks > 0);
    if (!(ok = cx.commit_wait())) break;
    if (tid == 0 && next) load_ds(hh + 1);  // R, T_w, T_u, dT are read: the next head's dS
    float* LK = vyM;  // vy / kx column sums are done
    {
      // all 32 lanes: rows r0 = 16 q4 + lane / 4 and r0 + 8, column pairs (tmem_ld16x256_x4)
      const int c2 = 2 * (cx.lane & 3);
      const int rw[2] = {16 * cx.q4 + (cx.lane >> 2), 16 * cx.q4 + (cx.lane >> 2) + 8};
      const bool factored = gam[63] > kFactorMin;
      float v[16], ev[16], kkv[16];
      tmem_ld16x256_x4(tm + kGt1 + cx.lane_base() + 32 * cx.half, v);
      tmem_ld16x256_x4(tm + kGtC + cx.lane_base() + 32 * cx.half, kkv);
      if (factored) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int q = 0; q < 4; ++q) ev[4 * k + q] = sm.Gm[rw[q >> 1]] * sm.Gi[32 * cx.half + 8 * k + c2 + (q & 1)];
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ev[4 * k + q] = __expf(gam[rw[q >> 1]] - gam[32 * cx.half + 8 * k + c2 + (q & 1)]);
      }
      tmem_ld_wait();
      float b3[2] = {0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int r = rw[rr], j = 32 * cx.half + 8 * k + c2, x = 4 * k + 2 * rr;
          const float bi = sm.beta[r];
          const float2 kk = make_float2(kkv[x], kkv[x + 1]);
          // dA = -v, strictly lower and inside the chunk; L = dA o diag(beta) E
          const float dae0 = (j < r && r < n) ? -v[x] * ev[x] : 0.f;
          const float dae1 = (j + 1 < r && r < n) ? -v[x + 1] * ev[x + 1] : 0.f;
          b3[rr] += dae0 * kk.x + dae1 * kk.y;
          const float l0 = dae0 * bi, l1 = dae1 * bi;
          *reinterpret_cast<float2*>(LK + fz(r, j)) = make_float2(l0 * kk.x, l1 * kk.y);
          *reinterpret_cast<uint32_t*>(sm.bP + sw128_pair(r, j)) = pack_bf16x2(l0, l1);
        }
      b3[0] = quad_sum(b3[0]);
      b3[1] = quad_sum(b3[1]);
      if ((cx.lane & 3) == 0) {
        sm.db3[cx.half][rw[0]] = b3[0];
        sm.db3[cx.half][rw[1]] = b3[1];
      }
    }
    sync_generic_to_async();
    // ---------------- (g) dk += (L + L^T) K: the image of L read K-major (L) and MN-major (L^T)
    if (tid == 0) {
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kGtK, kmajor_step(kmajor_desc(smem_u32(sm.bP), 8192, 0), 8192, ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.k[0]), 8192, 0), ks),
                  idesc_bf16(64, 128, 0, 1), 1);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kGtK, mnmajor_step(mnmajor_desc(smem_u32(sm.bP), 8192, 0), ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.k[0]), 8192, 0), ks),
                  idesc_bf16(64, 128, 1, 1), 1);
    }
    col_sums(sm, LK, nullptr, sm.cA, nullptr, tid);
    // ---------------- (h) dgamma -> dg (reverse cumulative sum in the chunk), dbeta
    if (tid < 64) {
      const int i = tid;
      const float ktd = (i < n) ? __expf(gC - gam[i]) * (sm.part[2][i] + sm.part[3][i]) : 0.f;
      const float kts = warp_sum(ktd);
      if (cx.lane == 0) sm.red[cx.warp] = kts;  // warps 0 and 1 (the Frobenius partials are consumed)
      float dgam = 0.f;
      if (i < n) {
        const float b3 = sm.db3[0][i] + sm.db3[1][i];
        dgam = sm.part[0][i] + sm.part[1][i] - sm.part[4][i] - ktd +
               sm.beta[i] * sm.Gm[i] * sm.kx[i] + sm.beta[i] * b3 - sm.cA[i];
      }
      sm.part[7][i] = dgam;
    }
    __syncthreads();
    if (tid < 64) {
      // suffix sums over the chunk (two warps), the last token also takes the chunk-end terms
      const int i = tid;
      float x = sm.part[7][i];
      if (i == n - 1) x += GC * fro + (sm.red[0] + sm.red[1]);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, o);
        if (cx.lane + o < 32) x += y;
      }
      sm.red4[0][0][i] = x;
    }
    __syncthreads();
    if (tid < n) {
      const float s = sm.red4[0][0][tid] + (tid < 32 ? sm.red4[0][0][32] : 0.f);
      p.dg[(size_t)(tok0 + tid) * Hv + h] = s;
      p.dbeta[(size_t)(tok0 + tid) * Hv + h] = sm.vy[tid] + sm.Gm[tid] * sm.kx[tid] + sm.db3[0][tid] + sm.db3[1][tid];
    }
    __syncthreads();
    if (!(ok = cx.commit_wait())) break;  // (g) done before the next head reuses bP
  }
  if (ok) {
    // dk: sum over the value heads of this key head
    const size_t row = ((size_t)(tok0 + i_row) * Hk + hk) * kDim + 64 * cx.half;
    for (int cc = 0; cc < 64; cc += 16) {
      float b[16];
      tmem_ld16(tm + kGtK + cx.lane_base() + 64 * cx.half + cc, b);
      tmem_ld_wait();
      if (has_row && i_row < n)
        for (int x = 0; x < 16; x += 4)
          *reinterpret_cast<float4*>(p.dk + row + cc + x) = make_float4(b[x], b[x + 1], b[x + 2], b[x + 3]);
    }
  } else if (tid == 0) {
    set_status(hd, kErrTimeout);
  }
  // a CTA that gave up before its first head lets that head's record copies land before it leaves
  if (tid == 0 && !p1_seen) mbar_wait(&bar_p1, 0, kWaitBudget);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (cx.warp == 0) tmem_dealloc(tm, 512);
}

// ============================================================================================ dq
//
// dq = sum over the value heads h of the key head of
//        scale diag(e^gamma) dO S_c^T  +  (scale (dO V'^T) o E) K
// with S_c and V' in compensated bf16 (hi + lo, two MMAs each) so that dq, whose entries reach
// O(10) at these shapes, keeps the accuracy of the other gradients; the per-row e^gamma scaling is
// applied in fp32 and the sum over value heads is kept in fp32 registers.
//
// The same compensated dO S^T also gives the term of dgamma_t through the state part of o_t,
// scale e^{gamma_t} q_t . (S_c dO_t): its suffix sums over the chunk are added to dg, which
// grad_kernel (launched before, on the same stream) has written with all the other terms. With
// S_c in bf16 alone this term dominated the error of dg on long slowly decaying documents.

struct DqSmem {
  uint8_t k[2][8192];    // K tile                  (B MN-major: dQK K)
  uint8_t dout[2][2][8192];  // [head parity] dO tile (A K-major)
  uint8_t sh[2][16384];  // S_c high part           (B K-major: dO S^T)
  uint8_t sl[2][16384];  // S_c low part
  uint8_t vh[2][8192];   // V' high part            (B K-major: dO V'^T)
  uint8_t vl[2][8192];   // V' low part
  uint8_t qh[8192];      // scale dQK high part     (A K-major)
  uint8_t ql[8192];      // scale dQK low part
  uint8_t q[2][8192];    // Q tile (read by the threads: the dgamma term)
  float gam[2][64];      // [head parity]
  float eg[64], egi[64]; // e^{gamma}, e^{-gamma}
  float qd[2][2][64];    // [head parity][column half] row partials of the dgamma term
};
constexpr size_t kDqSmemBytes = sizeof(DqSmem) + 1024;
constexpr uint32_t kDtP = 0, kDt1 = 128, kDt2 = 256;

__global__ void __launch_bounds__(256, 1) dq_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  DqSmem& sm = *reinterpret_cast<DqSmem*>(smem_align1024(smem_raw));
  __shared__ uint64_t bar_ld, bar_mma, bar_a, bar_b;
  __shared__ uint32_t tmem_holder;
  griddep_launch_dependents();
  griddep_wait();  // grad_kernel's dg (and the records)
  Header* hd = reinterpret_cast<Header*>(p.ws + p.L.f.header);
  const int chunk = blockIdx.x, hk = blockIdx.y;
  if (chunk >= hd->n_chunks || get_status(hd) != 0) return;
  const int Hv = p.d.Hv, Hk = p.d.Hk, G = Hv / Hk;
  const int tok0 = reinterpret_cast<const int32_t*>(p.ws + p.L.f.chunk_tok0)[chunk];
  const int n = reinterpret_cast<const int32_t*>(p.ws + p.L.f.chunk_len)[chunk];
  Ctx cx;
  ctx_init(cx, &bar_ld, &bar_mma);
  const int tid = cx.tid;
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_b, 1);
    fence_mbar_init();
  }
  if (cx.warp == 0) tmem_alloc(&tmem_holder, 512);
  sync_generic_to_async();
  const uint32_t tm = tmem_holder;
  cx.tmem = tm;
  // all 32 lanes of each warp: rows rw[0] = 16 q4 + lane / 4 and rw[1] = rw[0] + 8 of the M = 64
  // accumulators, column pairs c2 + 8k of each 32-column group (tmem_ld16x256_x4)
  const int c2 = 2 * (cx.lane & 3);
  const int rw[2] = {16 * cx.q4 + (cx.lane >> 2), 16 * cx.q4 + (cx.lane >> 2) + 8};
  float dq[32];  // [32-column group ci][16 values in the tmem_ld16x256_x4 order]
  for (int c = 0; c < 32; ++c) dq[c] = 0.f;
  bool ok = true;
  // Two load groups per value head, each issued as soon as the previous head frees its buffers:
  // A (dO into the head's parity buffer, V' hi / lo, gamma) once dP = dO V'^T has run, B (S hi / lo)
  // once dO S^T has run. Head hh + 1's A then lands during head hh's second half, and its B
  // during its own dP and epilogue.
  uint32_t ph_a = 0, ph_b = 0;
  auto issue_a = [&](int hh2) {  // thread 0
    const int h2 = hk * G + hh2, b2 = hh2 & 1;
    const size_t r2 = (size_t)chunk * Hv + h2;
    mbar_arrive_expect_tx(&bar_a, (hh2 == 0 ? 4 * 8192 : 0) + 2 * 8192 + 2 * 16384 + 256);
    if (hh2 == 0) {
      tma_load_3d(sm.k[0], &p.tm_k, 0, hk, tok0, &bar_a);
      tma_load_3d(sm.k[1], &p.tm_k, 64, hk, tok0, &bar_a);
      tma_load_3d(sm.q[0], &p.tm_q, 0, hk, tok0, &bar_a);
      tma_load_3d(sm.q[1], &p.tm_q, 64, hk, tok0, &bar_a);
    }
    tma_load_3d(sm.dout[b2][0], &p.tm_do, 0, h2, tok0, &bar_a);
    tma_load_3d(sm.dout[b2][1], &p.tm_do, 64, h2, tok0, &bar_a);
    bulk_load(sm.vh[0], p.ws + p.L.vp_img + r2 * 16384, 16384, &bar_a);
    bulk_load(sm.vl[0], p.ws + p.L.vp_lo + r2 * 16384, 16384, &bar_a);
    bulk_load(sm.gam[b2], p.ws + p.L.f.gam + r2 * 256, 256, &bar_a);
  };
  auto issue_b = [&](int hh2) {  // thread 0
    const size_t r2 = (size_t)chunk * Hv + hk * G + hh2;
    mbar_arrive_expect_tx(&bar_b, 2 * 32768);
    bulk_load(sm.sh[0], p.ws + p.L.st_img + r2 * 32768, 32768, &bar_b);
    bulk_load(sm.sl[0], p.ws + p.L.st_lo + r2 * 32768, 32768, &bar_b);
  };
  if (tid == 0) {
    issue_a(0);
    issue_b(0);
  }
  for (int hh = 0; hh < G && ok; ++hh) {
    const int h = hk * G + hh, bp = hh & 1;
    const size_t rec = (size_t)chunk * Hv + h;
    // warps 2-3 add the dgamma term of this head to dg at its end: grad_kernel's value, read now
    const int gi = tid - 64;
    float dg_old = 0.f;
    if (gi >= 0 && gi < 64 && gi < n) dg_old = p.dg[(size_t)(tok0 + gi) * Hv + h];
    if (tid == 224 && hh + 1 < G) {  // the next head's records into L2 (a thread off the load path)
      const size_t r1 = rec + 1;
      tma_prefetch_3d(&p.tm_do, 0, h + 1, tok0);
      tma_prefetch_3d(&p.tm_do, 64, h + 1, tok0);
      bulk_prefetch_l2(p.ws + p.L.st_img + r1 * 32768, 32768);
      bulk_prefetch_l2(p.ws + p.L.st_lo + r1 * 32768, 32768);
      bulk_prefetch_l2(p.ws + p.L.vp_img + r1 * 16384, 16384);
      bulk_prefetch_l2(p.ws + p.L.vp_lo + r1 * 16384, 16384);
    }
    if (!(ok = wait_all(&bar_a, ph_a))) break;
    ph_a ^= 1;
    tc_fence_after();
    if (tid < 64) {
      sm.eg[tid] = __expf(sm.gam[bp][tid]);
      sm.egi[tid] = __expf(-sm.gam[bp][tid]);
    }
    // dP = dO V'^T (hi + lo)
    if (tid == 0) {
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kDtP, kmajor_step(kmajor_desc(smem_u32(sm.dout[bp][0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.vh[0]), 8192, 0), 8192, ks),
                  idesc_bf16(64, 64, 0, 0), ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kDtP, kmajor_step(kmajor_desc(smem_u32(sm.dout[bp][0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.vl[0]), 8192, 0), 8192, ks),
                  idesc_bf16(64, 64, 0, 0), 1);
    }
    if (!(ok = cx.commit_wait())) break;  // (its barrier also publishes eg / egi)
    if (tid == 0 && hh + 1 < G) issue_a(hh + 1);  // V' is read; the other dO buffer is free
    // e^{gamma_i - gamma_j} as e^{gamma_i} e^{-gamma_j} while both factors stay finite
    const bool factored = sm.gam[bp][63] > kFactorMin;
    {
      // all 32 lanes: rows rw[0], rw[1], column pairs (tmem_ld16x256_x4)
      float v[16], ev[16];
      tmem_ld16x256_x4(tm + kDtP + cx.lane_base() + 32 * cx.half, v);
      if (factored) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ev[4 * k + q] = sm.eg[rw[q >> 1]] * p.scale * sm.egi[32 * cx.half + 8 * k + c2 + (q & 1)];
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ev[4 * k + q] = __expf(sm.gam[bp][rw[q >> 1]] - sm.gam[bp][32 * cx.half + 8 * k + c2 + (q & 1)]) * p.scale;
      }
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int r = rw[rr], j = 32 * cx.half + 8 * k + c2, x = 4 * k + 2 * rr;
          const float d0 = (j <= r && r < n) ? v[x] * ev[x] : 0.f;
          const float d1 = (j + 1 <= r && r < n) ? v[x + 1] * ev[x + 1] : 0.f;
          const float h0 = __bfloat162float(__float2bfloat16_rn(d0)), h1 = __bfloat162float(__float2bfloat16_rn(d1));
          const uint32_t off = sw128_pair(r, j);
          *reinterpret_cast<uint32_t*>(sm.qh + off) = pack_bf16x2(h0, h1);
          *reinterpret_cast<uint32_t*>(sm.ql + off) = pack_bf16x2(d0 - h0, d1 - h1);
        }
    }
    sync_generic_to_async();
    if (!(ok = wait_all(&bar_b, ph_b))) break;
    ph_b ^= 1;
    tc_fence_after();
    // dO S^T (hi + lo) and dQK K (hi + lo)
    if (tid == 0) {
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kDt1, kmajor_step(kmajor_desc(smem_u32(sm.dout[bp][0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.sh[0]), 16384, 0), 16384, ks),
                  idesc_bf16(64, 128, 0, 0), ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm + kDt1, kmajor_step(kmajor_desc(smem_u32(sm.dout[bp][0]), 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(smem_u32(sm.sl[0]), 16384, 0), 16384, ks),
                  idesc_bf16(64, 128, 0, 0), 1);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kDt2, kmajor_step(kmajor_desc(smem_u32(sm.qh), 8192, 0), 8192, ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.k[0]), 8192, 0), ks),
                  idesc_bf16(64, 128, 0, 1), ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm + kDt2, kmajor_step(kmajor_desc(smem_u32(sm.ql), 8192, 0), 8192, ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.k[0]), 8192, 0), ks),
                  idesc_bf16(64, 128, 0, 1), 1);
    }
    if (!(ok = cx.commit_wait())) break;
    if (tid == 0 && hh + 1 < G) issue_b(hh + 1);  // S is read
    {
      const float sc0 = sm.eg[rw[0]] * p.scale, sc1 = sm.eg[rw[1]] * p.scale;
      float qd[2] = {0.f, 0.f};  // q_t . (S_c dO_t) over this thread's columns, rows rw[0], rw[1]
#pragma unroll
      for (int ci = 0; ci < 2; ++ci) {
        float a[16], b[16];
        tmem_ld16x256_x4(tm + kDt1 + cx.lane_base() + 64 * cx.half + 32 * ci, a);
        tmem_ld16x256_x4(tm + kDt2 + cx.lane_base() + 64 * cx.half + 32 * ci, b);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 16; ++x) dq[16 * ci + x] += ((x & 2) ? sc1 : sc0) * a[x] + b[x];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const float2 qv = __bfloat1622float2(
                *reinterpret_cast<const __nv_bfloat162*>(sm.q[cx.half] + sw128_pair(rw[rr], 32 * ci + 8 * k + c2)));
            qd[rr] += qv.x * a[4 * k + 2 * rr] + qv.y * a[4 * k + 2 * rr + 1];
          }
      }
      qd[0] = quad_sum(qd[0]);
      qd[1] = quad_sum(qd[1]);
      if ((cx.lane & 3) == 0) {
        sm.qd[bp][cx.half][rw[0]] = qd[0] * sc0;
        sm.qd[bp][cx.half][rw[1]] = qd[1] * sc1;
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (gi >= 0 && gi < 64) {
      // dg += suffix sums of the term over the chunk: warp 2 rows 0-31 (plus the total of rows
      // 32-63), warp 3 rows 32-63; the other warps go on to the next head, which writes the other
      // parity of qd
      const int i = gi;
      float x = (i < n) ? sm.qd[bp][0][i] + sm.qd[bp][1][i] : 0.f;
      float tail = 0.f;
      if (cx.warp == 2) tail = warp_sum((i + 32 < n) ? sm.qd[bp][0][i + 32] + sm.qd[bp][1][i + 32] : 0.f);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, o);
        if (cx.lane + o < 32) x += y;
      }
      if (i < n) p.dg[(size_t)(tok0 + i) * Hv + h] = dg_old + (x + tail);
    }
  }
  if (ok) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
      if (rw[rr] < n) {
        float* row = p.dq + ((size_t)(tok0 + rw[rr]) * Hk + hk) * kDim + 64 * cx.half + c2;
#pragma unroll
        for (int ci = 0; ci < 2; ++ci)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            *reinterpret_cast<float2*>(row + 32 * ci + 8 * k) =
                make_float2(dq[16 * ci + 4 * k + 2 * rr], dq[16 * ci + 4 * k + 2 * rr + 1]);
      }
  } else if (tid == 0) {
    set_status(hd, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (cx.warp == 0) tmem_dealloc(tm, 512);
}

// d(initial_state)[x][h] = sum over documents i (in order) with init_idx[i] == x of dL/dS_start(i, h).
__global__ void __launch_bounds__(256) dinit_reduce_kernel(const __grid_constant__ BwdParams p) {
  griddep_wait();  // the start-state gradients
  const int x = blockIdx.x / p.d.Hv, h = blockIdx.x % p.d.Hv;
  const float* ds0 = reinterpret_cast<const float*>(p.ws + p.L.ds0);
  const size_t st = (size_t)kDim * kDim;
  float* dst = p.dinit + ((size_t)x * p.d.Hv + h) * st;
  for (int e = threadIdx.x; e < kDim * kDim; e += 256) {
    float acc = 0.f;
    if (p.init_idx)
      for (int i = 0; i < p.d.N; ++i)
        if (p.init_idx[i] == x) acc += ds0[((size_t)i * p.d.Hv + h) * st + e];
    dst[e] = acc;
  }
}

// ============================================================================================ launch

namespace {

// The recording forward over the backward's workspace layout: tensor maps of the inputs, the
// inputs, and the record pointers. Shared by the backward's recompute and by a forward that keeps
// its records for the backward.
int setup_record_fwd(const BwdArgs& a, const BwdLayout& L, FwdParams& f) {
  std::memset(&f, 0, sizeof(f));
  const PlanDims& d = a.d;
  f.d = d;
  f.L = L.f;
  if (d.T > 0) {
    const uint64_t row_k = (uint64_t)d.Hk * kDim * 2, row_v = (uint64_t)d.Hv * kDim * 2;
    if (!make_tmap_bf16_3d(&f.tm_q, a.q, kDim, d.Hk, d.T, kDim * 2, row_k, 64, 1, 64) ||
        !make_tmap_bf16_3d(&f.tm_k, a.k, kDim, d.Hk, d.T, kDim * 2, row_k, 64, 1, 64) ||
        !make_tmap_bf16_3d(&f.tm_v, a.v, kDim, d.Hv, d.T, kDim * 2, row_v, 64, 1, 64))
      return kErrCuda;
  }
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.ws);
  f.g = a.g;
  f.beta = a.beta;
  f.cu = a.cu;
  f.init_idx = a.init_idx;
  f.initial_state = a.initial_state;
  f.out = nullptr;
  f.final_state = reinterpret_cast<float*>(ws + L.fin);
  f.ws = ws;
  f.trunc_thr = a.trunc_thr;
  f.scale = a.scale;
  f.flag_budget = a.flag_budget;
  f.withhold_fin = a.withhold_fin;
  f.st_img = ws + L.st_img;
  f.vp_img = ws + L.vp_img;
  f.p_img = ws + L.f.pimg;  // kkt_solve also forms P = scale (Q K^T o E) for the reverse chain
  f.t_f32 = reinterpret_cast<float*>(ws + L.t_f32);
  f.tw_lo = ws + L.tw_lo;
  f.tu_lo = ws + L.tu_lo;
  f.st_lo_img = ws + L.st_lo;
  f.vp_lo_img = ws + L.vp_lo;
  return kOk;
}

}  // namespace

int launch_fwd_save(const BwdArgs& a, void* out, float* final_state, cudaStream_t stream, cudaEvent_t* ev) {
  const BwdLayout L = bwd_layout(a.d);
  if (a.ws_bytes < L.total) return kErrWorkspace;
  FwdParams f;
  const int rc = setup_record_fwd(a, L, f);
  if (rc != kOk) return rc;
  if (a.d.T > 0 && !make_tmap_bf16_3d(&f.tm_o, out, kDim, a.d.Hv, a.d.T, kDim * 2, (uint64_t)a.d.Hv * kDim * 2,
                                      64, 1, 64))
    return kErrCuda;
  f.out = reinterpret_cast<__nv_bfloat16*>(out);
  f.final_state = final_state;
  return launch_fwd(f, stream, ev);
}

int launch_bwd(const BwdArgs& a, bool reuse, cudaStream_t stream, cudaEvent_t* ev) {
  static PerDevice attr_done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kErrCuda;
  if (!attr_done.done(dev)) {
    if (cudaFuncSetAttribute(rev_chain_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRevSmemBytes) !=
            cudaSuccess ||
        cudaFuncSetAttribute(rev_chain_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRevSmemBytes) !=
            cudaSuccess)
      return kErrCuda;
    if (cudaFuncSetAttribute(grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGradSmemBytes) !=
        cudaSuccess)
      return kErrCuda;
    if (cudaFuncSetAttribute(dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDqSmemBytes) !=
        cudaSuccess)
      return kErrCuda;
    attr_done.mark(dev);
  }
  const PlanDims& d = a.d;
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.d = d;
  p.L = bwd_layout(d);
  if (a.ws_bytes < p.L.total) return kErrWorkspace;
  uint8_t* ws = reinterpret_cast<uint8_t*>(a.ws);
  // the forward with per-chunk records (only its maps when a forward left the records here)
  FwdParams f;
  int rc = setup_record_fwd(a, p.L, f);
  if (rc != kOk) return rc;
  if (d.T > 0 && !make_tmap_bf16_3d(&p.tm_do, a.dout, kDim, d.Hv, d.T, kDim * 2, (uint64_t)d.Hv * kDim * 2, 64, 1, 64))
    return kErrCuda;
  p.tm_q = f.tm_q;
  p.tm_k = f.tm_k;
  p.tm_v = f.tm_v;
  // the backward's own flags, reset before the forward so that its kernels and the reverse chain
  // follow one another as kernels (dependent launches)
  if (cudaMemsetAsync(ws + p.L.flags_ds0, 0, (size_t)d.N * d.Hv * 4, stream) != cudaSuccess) return kErrCuda;
  if (cudaMemsetAsync(ws + p.L.hdr2, 0, sizeof(Header), stream) != cudaSuccess) return kErrCuda;
  if (cudaMemsetAsync(ws + p.L.flags_rseg, 0, (size_t)p.L.f.smax * d.Hv * 4, stream) != cudaSuccess) return kErrCuda;
  rc = launch_fwd(f, stream, ev, reuse);
  if (rc != kOk) return rc;
  p.g = a.g;
  p.beta = a.beta;
  p.cu = a.cu;
  p.init_idx = a.init_idx;
  p.dfinal = a.dfinal;
  p.dq = reinterpret_cast<float*>(a.dq);
  p.dk = reinterpret_cast<float*>(a.dk);
  p.dv = reinterpret_cast<float*>(a.dv);
  p.dg = a.dg;
  p.dbeta = a.dbeta;
  p.dinit = a.dinit;
  p.ws = ws;
  p.scale = a.scale;
  p.flag_budget = a.flag_budget;
  auto mark = [&](int i) {
    if (ev && ev[i]) cudaEventRecord(ev[i], stream);
  };
  mark(8);
  {
    const int64_t items = p.L.f.smax * d.Hv;
    const int grid = (int)(items < d.num_sms ? items : d.num_sms);
    if (p.L.f.slots > 0 && d.T > 0) launch_early(rev_chain_kernel<1>, grid, kRevThreads, kRevSmemBytes, stream, p);
    launch_early(rev_chain_kernel<2>, grid, kRevThreads, kRevSmemBytes, stream, p);
  }
  mark(9);
  mark(10);
  if (d.T > 0) launch_early(grad_kernel, dim3((unsigned)p.L.f.cmax, (unsigned)d.Hk), 256, kGradSmemBytes, stream, p);
  mark(11);
  mark(14);
  if (d.T > 0) launch_early(dq_kernel, dim3((unsigned)p.L.f.cmax, (unsigned)d.Hk), 256, kDqSmemBytes, stream, p);
  mark(15);
  mark(12);
  if (d.n_init > 0) launch_early(dinit_reduce_kernel, dim3(d.n_init * d.Hv), 256, 0, stream, p);
  mark(13);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace gdn
