// Forward kernels of the chunked Gated DeltaNet over packed varlen batches (sm_103a).
//
//   plan_kernel       chunk map, segment map, dependencies, queue and flag reset (device planner)
//   kkt_solve_kernel  per (chunk, key head): K K^T (and Q K^T) on tcgen05, then per value head of
//                     the group the chunk-local cumulative gate gamma, T = (I + A)^{-1} with
//                     A = diag(beta) (e^{gamma_i-gamma_j} o K K^T) (strictly lower) by forward
//                     substitution, T diag(beta e^gamma), T diag(beta) and P = scale (Q K^T o E) in
//                     bf16, and a per-chunk flag for the warm-up bound below ("How to Speed Up GDN
//                     Kernels for Qwen Models", sections "What GDN actually computes" (kkt_solve, one
//                     64x64 system per chunk per head) and "Lever 2" (gate cumsum once per chunk;
//                     one inverse per chunk serves both o and the state recurrence)).
//   chain_kernel<OUT> persistent over (segment, value head) items in dependency order: the state S
//                     (fp32, 128x128) lives transposed in registers across 8 warps; per chunk, tcgen05
//                     MMAs with the value index on the accumulator lanes compute U^T = V^T T_u^T,
//                     V'^T = U^T - S^T W^T (W^T = K^T T_w^T), S^T += V'_s^T K with V'_s = diag(
//                     e^{gamma_C - gamma}) V', and O^T = S^T Q^T + V'^T P''^T, the bf16 operands S^T and
//                     V'^T kept in tensor memory. A segment starts from the state published by the
//                     previous one, or from a warm-up from zero when the decay in between provably
//                     leaves the earlier state below fp32 resolution.
//   chain_kernel<P1>  pass 1 of the exact segment split: per segment, the end state from zero (B) and
//                     the segment transition (M, started from I) -- or, for a first segment with a known
//                     start, its end state directly -- so that segment end states can be published as
//                     soon as the start state is known ("Lever 1": a sequence is split into segments
//                     that run in parallel; here the carry is exact instead of truncated). Units that
//                     no segment reads (the next one warms up) are skipped.
//   chain_kernel<·, record> the same chain in compensated bf16 writing per-chunk records (chunk-start
//                     S, V') for the backward: its recompute, or the forward of a training step,
//                     which then forms o from the records in out_kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bw_prims.cuh"
#include "gdn_common.cuh"
#include "gdn_dev.cuh"
#include "gdn_fwd.h"
#include "gdn_host.h"

namespace gdn {
using namespace bw;

// ============================================================================================ plan

// keep_mzero: a backward that reuses a forward's records keeps that forward's pass-1 findings
// (which segment transitions are exactly zero); the maps it rebuilds are the same.
constexpr int kPlanThreads = 256;  // one block; the scans run in tiles of this many documents / segments

// Inclusive prefix sum over the 256 threads of the block: a shuffle scan per warp, then one over the
// eight warp totals (two barriers). The caller synchronises before the next call reuses s_tot.
__device__ __forceinline__ int block_inclusive_scan(int v, int* s_tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) s_tot[w] = v;
  __syncthreads();
  if (w == 0) {
    int t = lane < kPlanThreads / 32 ? s_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < kPlanThreads / 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    if (lane < kPlanThreads / 32) s_tot[lane] = t;
  }
  __syncthreads();
  return w > 0 ? v + s_tot[w - 1] : v;
}
constexpr int kPlanSmemDocs = 2048;  // per-document offsets kept in shared memory up to this many documents
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ FwdParams p, int keep_mzero) {
  griddep_launch_dependents();  // kkt_solve may start; it waits for the maps below
  Header* hd = ws_ptr<Header>(p, p.L.header);
  const int N = p.d.N;
  const int tid = threadIdx.x, nt = blockDim.x;
  __shared__ int s_bad, s_L, s_longest;
  __shared__ int s_carry[2];
  __shared__ int s_scan[kPlanThreads];
  __shared__ int32_t s_c0[kPlanSmemDocs + 1], s_s0[kPlanSmemDocs + 1];
  // the lookups below read these offsets many times: from shared memory when they fit
  const bool in_smem = N <= kPlanSmemDocs;
  int32_t* seq_chunk0 = in_smem ? s_c0 : ws_ptr<int32_t>(p, p.L.seq_chunk0);
  int32_t* seq_seg0 = in_smem ? s_s0 : ws_ptr<int32_t>(p, p.L.seq_seg0);
  if (tid == 0) {
    s_bad = 0;
    s_longest = 0;
  }
  __syncthreads();
  // validation
  if (tid == 0 && (p.cu[0] != 0 || p.cu[N] != p.d.T)) s_bad = 1;
  for (int i = tid; i < N; i += nt)
    if (plan_check_doc(i, p.cu, p.init_idx, p.d.n_init) != kOk) s_bad = 1;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      hd->status = kErrInvalid;
      hd->n_chunks = 0;
      hd->n_segs = 0;
      hd->n_p1 = 0;
      hd->n_walk = 0;
      hd->q_p1 = 0;
      hd->q_chain = 0;
    }
    return;
  }
  // exclusive scan of chunk counts -> seq_chunk0 (tiles of nt documents)
  if (tid == 0) s_carry[0] = 0;
  __syncthreads();
  for (int base = 0; base < N; base += nt) {
    const int i = base + tid;
    const int c = (i < N) ? doc_chunks(i, p.cu) : 0;
    if (i < N) atomicMax(&s_longest, c);
    const int incl = block_inclusive_scan(c, s_scan);
    if (i < N) seq_chunk0[i] = s_carry[0] + incl - c;
    __syncthreads();
    if (tid == nt - 1) s_carry[0] += incl;
    __syncthreads();
  }
  const int total_chunks = s_carry[0];
  if (tid == 0) {
    seq_chunk0[N] = total_chunks;
    s_L = plan_seg_len(p.d, total_chunks, s_longest);
  }
  __syncthreads();
  const int L = s_L;
  // exclusive scan of segment counts -> seq_seg0
  if (tid == 0) s_carry[1] = 0;
  __syncthreads();
  for (int base = 0; base < N; base += nt) {
    const int i = base + tid;
    const int c = (i < N) ? doc_segs(doc_chunks(i, p.cu), L) : 0;
    const int incl = block_inclusive_scan(c, s_scan);
    if (i < N) seq_seg0[i] = s_carry[1] + incl - c;
    __syncthreads();
    if (tid == nt - 1) s_carry[1] += incl;
    __syncthreads();
  }
  const int total_segs = s_carry[1];
  if (tid == 0) seq_seg0[N] = total_segs;
  __syncthreads();
  if (in_smem) {  // the other kernels read the offsets from the workspace
    int32_t* gc0 = ws_ptr<int32_t>(p, p.L.seq_chunk0);
    int32_t* gs0 = ws_ptr<int32_t>(p, p.L.seq_seg0);
    for (int i = tid; i <= N; i += nt) {
      gc0[i] = s_c0[i];
      gs0[i] = s_s0[i];
    }
  }
  // chunk and segment tables
  int32_t* cs = ws_ptr<int32_t>(p, p.L.chunk_seq);
  int32_t* ct = ws_ptr<int32_t>(p, p.L.chunk_tok0);
  int32_t* cl = ws_ptr<int32_t>(p, p.L.chunk_len);
  for (int c = tid; c < total_chunks; c += nt) plan_chunk(c, seq_chunk0, N, p.cu, cs + c, ct + c, cl + c);
  int32_t* si = ws_ptr<int32_t>(p, p.L.seg_info);
  for (int s = tid; s < total_segs; s += nt)
    plan_segment(s, seq_seg0, seq_chunk0, N, p.cu, L, p.init_idx, p.d.n_init, si + 4 * s);
  // flags
  int32_t* fs = ws_ptr<int32_t>(p, p.L.flags_seg);
  int32_t* ff = ws_ptr<int32_t>(p, p.L.flags_fin);
  for (int e = tid; e < total_segs * p.d.Hv; e += nt) fs[e] = 0;
  for (int e = tid; e < N * p.d.Hv; e += nt) ff[e] = 0;
  int32_t* wc = ws_ptr<int32_t>(p, p.L.walk_ctr);
  for (int e = tid; e < 2 * N * p.d.Hv; e += nt) wc[e] = 0;
  int32_t* fp1 = ws_ptr<int32_t>(p, p.L.flags_p1);
  for (int e = tid; e < (int)p.L.slots * p.d.Hv; e += nt) fp1[e] = 0;
  int32_t* mz = ws_ptr<int32_t>(p, p.L.mzero);
  if (!keep_mzero)
    for (int e = tid; e < (int)p.L.slots * p.d.Hv; e += nt) mz[e] = 0;
  // slots and pass-1 units: only split segments other than the last of their document get them
  // (exact mode), numbered in segment order; a document whose first segment starts from a known
  // state and that has middle segments also gets a walk (its first segment's unit)
  int32_t* slot = ws_ptr<int32_t>(p, p.L.seg_slot);
  int32_t* p1 = ws_ptr<int32_t>(p, p.L.p1_list);
  int32_t* walks = ws_ptr<int32_t>(p, p.L.walk_list);
  if (tid == 0) {
    s_carry[0] = 0;
    s_carry[1] = 0;
  }
  __syncthreads();
  for (int base = 0; base < total_segs; base += nt) {
    const int s = base + tid;
    int need = 0, walk = 0, known_start = 0;
    if (s < total_segs) {
      // the segment's document and dependency, recomputed (the table above is in global memory)
      int32_t info[4];
      plan_segment(s, seq_seg0, seq_chunk0, N, p.cu, L, p.init_idx, p.d.n_init, info);
      const int i = info[0];
      const bool last = (s + 1 == seq_seg0[i + 1]);
      const bool split = (seq_seg0[i + 1] - seq_seg0[i]) > 1;
      need = (split && !last && p.d.mode == 0) ? 1 : 0;
      known_start = info[3] == -1 ? 1 : 0;
      walk = (need && known_start && s == seq_seg0[i] && seq_seg0[i + 1] - seq_seg0[i] >= 3) ? 1 : 0;
    }
    const int mine = (need << 16) | walk;  // a tile holds at most nt segments: no carry between the halves
    const int incl = block_inclusive_scan(mine, s_scan);
    const int excl = incl - mine;
    if (s < total_segs) {
      const int u = s_carry[0] + (excl >> 16);  // the unit and the slot of the segment
      slot[s] = (need && u < p.L.slots) ? u : -1;
      if (need && u < p.L.slots) {
        p1[2 * u] = s;
        // 2: the end state from the document's known start; 0: the transition M and the end state
        // B from zero, or, when the segment's own start warms up, its end state directly
        p1[2 * u + 1] = known_start ? 2 : 0;
        if (walk) walks[s_carry[1] + (excl & 0xFFFF)] = u;
      }
    }
    __syncthreads();
    if (tid == nt - 1) {
      s_carry[0] += incl >> 16;
      s_carry[1] += incl & 0xFFFF;
    }
    __syncthreads();
  }
  if (tid == 0) {
    const int out_of_slots = s_carry[0] > p.L.slots ? 1 : 0;
    hd->status = out_of_slots ? kErrWorkspace : 0;
    hd->n_chunks = out_of_slots ? 0 : total_chunks;
    hd->n_segs = out_of_slots ? 0 : total_segs;
    hd->seg_chunks = L;
    hd->n_p1 = out_of_slots ? 0 : s_carry[0];
    hd->n_walk = out_of_slots ? 0 : s_carry[1];
    hd->q_p1 = 0;
    hd->q_chain = 0;
  }
}

// ======================================================================================= kkt_solve

// kkt_solve: one CTA of 256 threads per (chunk, key head). K K^T runs once on the tensor cores;
// the value heads of the group are then processed four at a time, one group of 64 threads per
// value head: the chunk-local cumulative gate gamma, A = diag(beta) (e^{gamma_i - gamma_j} o K K^T)
// (strictly lower), T = (I + A)^{-1} (32 x 32 diagonal blocks by forward substitution with one
// thread per column, x_r = [r == c] - sum_{m<r} A_rm x_m in registers, then the off-diagonal block
// from two block products), and the outputs T diag(beta e^gamma), T diag(beta) as bf16 images
// (plus T in fp32 and the low bf16 parts in record mode).
// A plain forward also computes Q K^T once per key head (tensor cores) and writes P = scale
// (Q K^T o E) per value head as a bf16 image, so that the state chain never forms it.
// The decay factors e^{gamma_i - gamma_j} (j <= i) are taken as e^{gamma_i} e^{-gamma_j} when the
// chunk's total decay is above -80 (both factors then stay finite in fp32), else one exp each.
constexpr int kKktHeads = 4;   // value heads solved concurrently
constexpr int kAStride = 68;   // fp32 row stride of A / T (16-byte aligned rows for vector loads)
constexpr float kFactorMin = -80.f;
struct KktSmem {
  uint8_t k_tile[2][8192];               // K rows, two 64-wide dk blocks, SW128; then Q K^T fp32 (fz)
  float a[kKktHeads][64][kAStride];      // A, then T (per concurrent value head); before the solve
                                         // the first 16 KB hold the Q tile (forward: Q K^T)
  float kk[64][kAStride];                // K K^T (16-byte aligned rows for vector loads)
  float gam[kKktHeads][64];
  float beta[kKktHeads][64];
  float eg[kKktHeads][64];               // e^{gamma}
  float egi[kKktHeads][64];              // e^{-gamma} (factored path only)
  float be[kKktHeads][64];               // beta e^{gamma}
  int contr[kKktHeads][2];               // per warp of a group: every token has 0 <= beta |k|^2 <= 2
};

// Named barrier of one 64-thread value-head group (ids 1-4; literal ids keep the count of
// hardware barriers the kernel reserves at five).
__device__ __forceinline__ void group_sync(int group) {
  switch (group) {
    case 0: asm volatile("bar.sync 1, 64;" ::: "memory"); break;
    case 1: asm volatile("bar.sync 2, 64;" ::: "memory"); break;
    case 2: asm volatile("bar.sync 3, 64;" ::: "memory"); break;
    default: asm volatile("bar.sync 4, 64;" ::: "memory"); break;
  }
}

// T21 = -T22 X for one column c of the lower-left 32 x 32 block (rows 32 + j, j = 2 i + kOdd):
// T22 is unit lower triangular (rows and columns 32-63 of A's buffer, zeros above the diagonal),
// x2 holds X's column in packed pairs; a row's sum runs to the next multiple of four.
template <int kOdd>
__device__ __forceinline__ void kkt_t21_rows(float (*A)[kAStride], const uint64_t* x2, int c) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int j = 2 * i + kOdd;
    uint64_t s01 = 0ull, s23 = 0ull;
#pragma unroll
    for (int m = 0; m <= j; m += 4) {
      const ulonglong2 tv = *reinterpret_cast<const ulonglong2*>(&A[32 + j][32 + m]);
      s01 = f2_fma(tv.x, x2[m / 2], s01);
      s23 = f2_fma(tv.y, x2[m / 2 + 1], s23);
    }
    A[32 + j][c] = -(f2_sum(s01) + f2_sum(s23));
  }
}

__global__ void __launch_bounds__(256, 2) kkt_solve_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  KktSmem& sm = *reinterpret_cast<KktSmem*>(smem_align1024(smem_raw));
  __shared__ uint64_t bar_ld, bar_mma;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_ld_ok;
  griddep_launch_dependents();
  griddep_wait();  // the maps of plan_kernel
  Header* hd = ws_ptr<Header>(p, p.L.header);
  const int chunk = blockIdx.x, hk = blockIdx.y;
  if (chunk >= hd->n_chunks || get_status(hd) != 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tok0 = ws_ptr<int32_t>(p, p.L.chunk_tok0)[chunk];
  const int n = ws_ptr<int32_t>(p, p.L.chunk_len)[chunk];
  const int Hv = p.d.Hv, G = p.d.Hv / p.d.Hk;
  // value-head group (warps g and g + 4) and its thread (token / column): the warp of columns 0-31
  // carries about four times the substitution work of the other, and warps g and g + 4 share a
  // sub-partition, so every sub-partition gets one of each per group
  const int grp = warp & 3, t = 32 * (warp >> 2) + lane;
  // the first round's gate and beta, loaded while the K and Q tiles and their products are in flight
  float g_first = 0.f, b_first = 0.f;
  if (grp < G && t < n) {
    const size_t at = (size_t)(tok0 + t) * Hv + hk * G + grp;
    g_first = p.g[at];
    b_first = p.beta[at];
  }

  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  const bool want_p = p.p_img != nullptr;
  if (warp == 0) tmem_alloc(&tmem_holder, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  bool ok = true;
  uint8_t* q_tile = reinterpret_cast<uint8_t*>(&sm.a[0][0][0]);
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar_ld, want_p ? 32768 : 16384);
    tma_load_3d(sm.k_tile[0], &p.tm_k, 0, hk, tok0, &bar_ld);
    tma_load_3d(sm.k_tile[1], &p.tm_k, 64, hk, tok0, &bar_ld);
    if (want_p) {
      tma_load_3d(q_tile, &p.tm_q, 0, hk, tok0, &bar_ld);
      tma_load_3d(q_tile + 8192, &p.tm_q, 64, hk, tok0, &bar_ld);
    }
    ok = mbar_wait(&bar_ld, 0, kWaitBudget);
    if (!ok) mbar_wait(&bar_ld, 0, kWaitBudget);  // let a late copy land before the CTA can exit
    if (ok) {
      tc_fence_after();
      const uint32_t kt = smem_u32(sm.k_tile[0]);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tmem, kmajor_step(kmajor_desc(kt, 8192, 0), 8192, ks),
                  kmajor_step(kmajor_desc(kt, 8192, 0), 8192, ks), idesc_bf16(64, 64, 0, 0), ks > 0);
      if (want_p)
        #pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(tmem + 64, kmajor_step(kmajor_desc(smem_u32(q_tile), 8192, 0), 8192, ks),
                    kmajor_step(kmajor_desc(kt, 8192, 0), 8192, ks),
                    idesc_bf16(64, 64, 0, 0), ks > 0);
      umma_commit(&bar_mma);
    }
    s_ld_ok = ok ? 1 : 0;
  }
  __syncthreads();
  bool ok_mma = false;
  if (s_ld_ok) ok_mma = wait_all(&bar_mma, 0);
  tc_fence_after();
  float* qk = reinterpret_cast<float*>(sm.k_tile[0]);  // the K tile is dead once the products are done
  if (!ok_mma) {
    if (tid == 0) set_status(hd, kErrTimeout);
  } else {
    // readback (M = 64: row 16q + l sits in lane 32q + l, l < 16): warps 0-3 K K^T, warps 4-7 Q K^T
    const int q4 = warp & 3;
    if (warp < 4 || want_p)
      for (int c = 0; c < 64; c += 16) {
        float v[16];
        tmem_ld16(tmem + ((uint32_t)(32 * q4) << 16) + (warp < 4 ? 0 : 64) + c, v);
        tmem_ld_wait();
        if (lane < 16) {
          const int r = 16 * q4 + lane;
          if (warp < 4)
            for (int i = 0; i < 16; ++i) sm.kk[r][c + i] = v[i];
          else
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<float4*>(qk + fz(r, c + i)) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
      }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
  if (!ok_mma) return;

  float* gam_ws = ws_ptr<float>(p, p.L.gam);
  uint8_t* tw_ws = ws_ptr<uint8_t>(p, p.L.tw);
  uint8_t* tu_ws = ws_ptr<uint8_t>(p, p.L.tu);
  float(*A)[kAStride] = sm.a[grp];
  float* gam = sm.gam[grp];
  float* bet = sm.beta[grp];
  float* eg = sm.eg[grp];
  float* egi = sm.egi[grp];
  float* be = sm.be[grp];
  const int sub = t >> 5;  // warp of the group: columns 32 sub ..; rows and terms below 32 sub are zero
  for (int hb = 0; hb < G; hb += kKktHeads) {
    if (hb + grp < G) {  // groups without a head this round skip to the CTA barrier below
      const int h = hk * G + hb + grp;
      const size_t rec = (size_t)chunk * Hv + h;
      // chunk-local cumulative gate: inclusive scan over the 64 tokens in the group's two warps
      {
        const float gi = hb == 0 ? g_first : ((t < n) ? p.g[(size_t)(tok0 + t) * Hv + h] : 0.f);
        const float bi = hb == 0 ? b_first : ((t < n) ? p.beta[(size_t)(tok0 + t) * Hv + h] : 0.f);
        float sc = gi;
        for (int off = 1; off < 32; off <<= 1) {
          const float o = __shfl_up_sync(0xffffffffu, sc, off);
          if (lane >= off) sc += o;
        }
        gam[t] = sc;
        bet[t] = bi;
        // contraction check of the chunk's token transitions (padding rows have beta = 0)
        const float bk = bi * sm.kk[t][t];
        const int all_ok = __all_sync(0xffffffffu, bk >= 0.f && bk <= 2.f);
        if (lane == 0) sm.contr[grp][sub] = all_ok;
        group_sync(grp);
        if (t == 0) ws_ptr<int32_t>(p, p.L.contr)[rec] = (sm.contr[grp][0] && sm.contr[grp][1]) ? 1 : 0;
        if (t >= 32) sc += gam[31];
        gam_ws[rec * 64 + t] = sc;
        eg[t] = __expf(sc);
        egi[t] = __expf(-sc);
        be[t] = bi * eg[t];
        group_sync(grp);
        if (t >= 32) gam[t] = sc;
        group_sync(grp);
      }
      if (p.p_factored) {
        // the inference chain's per-token factors: e^{gamma_C - gamma_t} (V'_s), the output row
        // factor scale e^{gamma_t} (1 for a row past the cut, whose P'' row is the plain P), e^{gamma_C}
        float* f = ws_ptr<float>(p, p.L.fac) + rec * kFacFloats;
        const float gt = gam[t], gC = gam[63];
        f[t] = __expf(gC - gt);
        f[64 + t] = gt >= kExactCut ? p.scale * __expf(gt) : 1.f;
        if (t == 0) f[128] = __expf(gC);
      }
      const bool factored = gam[63] > kFactorMin;  // gamma is nonincreasing: gam[63] is the minimum
      if (factored) {
        // T = (I + A)^{-1} with A_rm = (beta_r e^{gamma_r}) (K K^T)_rm e^{-gamma_m} for m < r, in 32 x 32
        // blocks: T11 = (I + A11)^{-1} (columns 0-31, first warp of the group) and T22 (columns
        // 32-63, second warp) by forward substitution on y_m = e^{-gamma_m} x_m, one thread per
        // column, reading K K^T itself (no A matrix); then X = A21 T11 and T21 = -T22 X with both
        // warps on columns 0-31 (halves of the rows each), so that neither warp carries the whole
        // column-0 substitution. T goes to A's buffer.
        // y_m = e^{-gamma_m} x_m in packed pairs (lane pairs of the fp32x2 products): entries not yet
        // solved are zero, so a row's sum may run to the next multiple of four
        uint64_t y2[16];
        {
          // both warps run the same code on their diagonal block (offset o): the instruction stream
          // is shared, and the rows come in groups of four whose beta e^{gamma} and e^{-gamma} take
          // two vector loads
          const int o = 32 * sub;
          const float(*kkb)[kAStride] = reinterpret_cast<const float(*)[kAStride]>(&sm.kk[o][o]);
          float(*Ab)[kAStride] = reinterpret_cast<float(*)[kAStride]>(&A[o][o]);
          if (sub)
#pragma unroll
            for (int r = 0; r < 32; ++r) A[r][t] = 0.f;
#pragma unroll
          for (int m = 0; m < 16; ++m) y2[m] = 0ull;
#define GDN_KKT_ROW(R)                                                                     \
  {                                                                                        \
    uint64_t s01 = 0ull, s23 = 0ull;                                                       \
    _Pragma("unroll") for (int m = 0; m < (R); m += 4) {                                   \
      const ulonglong2 kv = *reinterpret_cast<const ulonglong2*>(&kkb[(R)][m]);            \
      s01 = f2_fma(kv.x, y2[m / 2], s01);                                                  \
      s23 = f2_fma(kv.y, y2[m / 2 + 1], s23);                                              \
    }                                                                                      \
    const float xr = (((R) == lane) ? 1.f : 0.f) - cq[(R) & 3] * (f2_sum(s01) + f2_sum(s23)); \
    Ab[(R)][lane] = xr;                                                                    \
    const float yr = eq[(R) & 3] * xr;                                                     \
    y2[(R) / 2] = ((R) & 1) ? f2_pack(f2_lo(y2[(R) / 2]), yr) : f2_pack(yr, 0.f);          \
  }
#pragma unroll
          for (int rb = 0; rb < 32; rb += 4) {
            const float4 c4 = *reinterpret_cast<const float4*>(&be[o + rb]);
            const float4 e4 = *reinterpret_cast<const float4*>(&egi[o + rb]);
            const float cq[4] = {c4.x, c4.y, c4.z, c4.w}, eq[4] = {e4.x, e4.y, e4.z, e4.w};
            GDN_KKT_ROW(rb)
            GDN_KKT_ROW(rb + 1)
            GDN_KKT_ROW(rb + 2)
            GDN_KKT_ROW(rb + 3)
          }
        }
#undef GDN_KKT_ROW
        group_sync(grp);
        {
          // X = A21 T11 = diag(beta e^gamma) (K K^T)_21 (diag(e^{-gamma}) T11): column c = lane, rows
          // 32 + 16 sub .. + 15, into the T21 block
          const int c = lane;
#pragma unroll
          for (int m = 0; m < 32; m += 2) y2[m / 2] = f2_pack(egi[m] * A[m][c], egi[m + 1] * A[m + 1][c]);
          const int r0 = 32 + 16 * sub;
#pragma unroll 2
          for (int i = 0; i < 16; ++i) {
            const int r = r0 + i;
            uint64_t s01 = 0ull, s23 = 0ull;
#pragma unroll
            for (int m = 0; m < 32; m += 4) {
              const ulonglong2 kv = *reinterpret_cast<const ulonglong2*>(&sm.kk[r][m]);
              s01 = f2_fma(kv.x, y2[m / 2], s01);
              s23 = f2_fma(kv.y, y2[m / 2 + 1], s23);
            }
            A[r][c] = be[r] * (f2_sum(s01) + f2_sum(s23));
          }
        }
        group_sync(grp);
        {
          // T21 = -T22 X: column c = lane, the even rows (first warp) or the odd rows (second)
          const int c = lane;
#pragma unroll
          for (int m = 0; m < 32; m += 2) y2[m / 2] = f2_pack(A[32 + m][c], A[33 + m][c]);
          group_sync(grp);  // X is read: T21 replaces it
          if (sub == 0)
            kkt_t21_rows<0>(A, y2, c);
          else
            kkt_t21_rows<1>(A, y2, c);
        }
        group_sync(grp);
      } else {
        // A, column t (rows below the diagonal), one exponential per entry
        {
          const float gt = gam[t];
#pragma unroll 4
          for (int r = t + 1; r < 64; ++r) A[r][t] = bet[r] * __expf(gam[r] - gt) * sm.kk[r][t];
        }
        group_sync(grp);
        // T = (I + A)^{-1}, column t: forward substitution (entries above the diagonal come out 0);
        // the second warp of the group (columns 32-63) skips rows and terms below 32, which are zero
        float x[64];
        if (sub == 0) {
#pragma unroll
          for (int r = 0; r < 64; ++r) {
            // four independent partial sums keep the FMA chain of row r about r/4 long
            float a0 = (r == t) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int m = 0; m + 4 <= r; m += 4) {
              const float4 av = *reinterpret_cast<const float4*>(&A[r][m]);
              a0 -= av.x * x[m];
              a1 -= av.y * x[m + 1];
              a2 -= av.z * x[m + 2];
              a3 -= av.w * x[m + 3];
            }
#pragma unroll
            for (int m = r & ~3; m < r; ++m) a0 -= A[r][m] * x[m];
            x[r] = (a0 + a1) + (a2 + a3);
          }
        } else {
#pragma unroll
          for (int r = 0; r < 32; ++r) x[r] = 0.f;
#pragma unroll
          for (int r = 32; r < 64; ++r) {
            float a0 = (r == t) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int m = 32; m + 4 <= r; m += 4) {
              const float4 av = *reinterpret_cast<const float4*>(&A[r][m]);
              a0 -= av.x * x[m];
              a1 -= av.y * x[m + 1];
              a2 -= av.z * x[m + 2];
              a3 -= av.w * x[m + 3];
            }
#pragma unroll
            for (int m = r & ~3; m < r; ++m) a0 -= A[r][m] * x[m];
            x[r] = (a0 + a1) + (a2 + a3);
          }
        }
        group_sync(grp);  // every thread is done reading A
#pragma unroll
        for (int r = 0; r < 64; ++r) A[r][t] = x[r];
        group_sync(grp);
      }
      // outputs, row by row (8 threads per 128-byte row of the bf16 images): a thread keeps its
      // 16-byte column group cj = t mod 8 in every row, so its beta and e^{gamma} (and e^{-gamma}
      // for P'') are loaded once
      const int cjt = t & 7;
      float bcol[8], ecol[8], eicol[8];
      {
        const float4 b0 = *reinterpret_cast<const float4*>(&bet[8 * cjt]);
        const float4 b1 = *reinterpret_cast<const float4*>(&bet[8 * cjt + 4]);
        const float4 e0 = *reinterpret_cast<const float4*>(&eg[8 * cjt]);
        const float4 e1 = *reinterpret_cast<const float4*>(&eg[8 * cjt + 4]);
        const float4 i0 = *reinterpret_cast<const float4*>(&egi[8 * cjt]);
        const float4 i1 = *reinterpret_cast<const float4*>(&egi[8 * cjt + 4]);
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        const float iv[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          bcol[u] = bv[u];
          ecol[u] = ev[u];
          eicol[u] = iv[u];
        }
      }
      uint8_t* dw = tw_ws + rec * 8192;
      uint8_t* du = tu_ws + rec * 8192;
      float* tdst = p.t_f32 ? p.t_f32 + rec * 4096 : nullptr;
#pragma unroll 2
      for (int e = t; e < 64 * 8; e += 64) {
        const int r = e >> 3, cj = cjt;
        const float4 t0 = *reinterpret_cast<const float4*>(&A[r][8 * cj]);
        const float4 t1 = *reinterpret_cast<const float4*>(&A[r][8 * cj + 4]);
        const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
        if (tdst) {  // fz layout (the gradient kernel's fp32 scratch layout)
          *reinterpret_cast<float4*>(tdst + fz(r, 8 * cj)) = t0;
          *reinterpret_cast<float4*>(tdst + fz(r, 8 * cj + 4)) = t1;
        }
        float xw[8], xu[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          xu[u] = tv[u] * bcol[u];
          xw[u] = xu[u] * ecol[u];
        }
        const uint32_t off = r * 128 + ((cj ^ (r & 7)) << 4);
        uint32_t w[4], wl[4], uu[4], ul[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          w[u] = pack_bf16x2(xw[2 * u], xw[2 * u + 1]);
          uu[u] = pack_bf16x2(xu[2 * u], xu[2 * u + 1]);
          const float2 hw = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[u]));
          const float2 hu = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uu[u]));
          wl[u] = pack_bf16x2(xw[2 * u] - hw.x, xw[2 * u + 1] - hw.y);
          ul[u] = pack_bf16x2(xu[2 * u] - hu.x, xu[2 * u + 1] - hu.y);
        }
        *reinterpret_cast<uint4*>(dw + off) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(du + off) = make_uint4(uu[0], uu[1], uu[2], uu[3]);
        if (p.tw_lo) {
          *reinterpret_cast<uint4*>(p.tw_lo + rec * 8192 + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
          *reinterpret_cast<uint4*>(p.tu_lo + rec * 8192 + off) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
        }
      }
      // P = scale (Q K^T o E): rows i < n, j <= i, 8 threads per 128-byte row. In the factored
      // form of the inference forward the row factor scale e^{gamma_i} is left to the chain, which
      // applies it to (Q S + P'' V') as a whole: P''_ij = (Q K^T)_ij e^{-gamma_j}, finite for every
      // row whose decay since the chunk start stays above kExactCut; a row below it keeps P and
      // drops its Q S term in the chain (that term is below e^{kExactCut} of the chunk-start state).
      if (want_p && p.p_factored) {
        uint8_t* dp = p.p_img + rec * 8192;
#pragma unroll 2
        for (int e = t; e < 64 * 8; e += 64) {
          const int i = e >> 3, cj = cjt;
          const float4 q0 = *reinterpret_cast<const float4*>(qk + fz(i, 8 * cj));
          const float4 q1 = *reinterpret_cast<const float4*>(qk + fz(i, 8 * cj + 4));
          const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
          const float gi = gam[i];
          float pv[8];
          if (gi >= kExactCut) {
#pragma unroll
            for (int u = 0; u < 8; ++u) pv[u] = (8 * cj + u <= i && i < n) ? eicol[u] * qv[u] : 0.f;
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int j = 8 * cj + u;
              pv[u] = (j <= i && i < n) ? __expf(gi - gam[j]) * p.scale * qv[u] : 0.f;
            }
          }
          *reinterpret_cast<uint4*>(dp + i * 128 + ((cj ^ (i & 7)) << 4)) =
              make_uint4(pack_bf16x2(pv[0], pv[1]), pack_bf16x2(pv[2], pv[3]), pack_bf16x2(pv[4], pv[5]),
                         pack_bf16x2(pv[6], pv[7]));
        }
      } else if (want_p) {
        uint8_t* dp = p.p_img + rec * 8192;
        for (int e = t; e < 64 * 8; e += 64) {
          const int i = e >> 3, cj = e & 7;
          const float4 q0 = *reinterpret_cast<const float4*>(qk + fz(i, 8 * cj));
          const float4 q1 = *reinterpret_cast<const float4*>(qk + fz(i, 8 * cj + 4));
          const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
          const float gi = gam[i], ei = eg[i] * p.scale;
          float pv[8];
          if (factored) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int j = 8 * cj + u;
              pv[u] = (j <= i && i < n) ? ei * egi[j] * qv[u] : 0.f;
            }
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int j = 8 * cj + u;
              pv[u] = (j <= i && i < n) ? __expf(gi - gam[j]) * p.scale * qv[u] : 0.f;
            }
          }
          *reinterpret_cast<uint4*>(dp + i * 128 + ((cj ^ (i & 7)) << 4)) =
              make_uint4(pack_bf16x2(pv[0], pv[1]), pack_bf16x2(pv[2], pv[3]), pack_bf16x2(pv[4], pv[5]),
                         pack_bf16x2(pv[6], pv[7]));
        }
      }
      group_sync(grp);  // A / gam / beta are rewritten by the next head of this group
    }
  }
}

// =========================================================================================== chain

enum ChainMode { kModeOut = 0, kModeP1 = 1 };


struct ChainCtx {
  uint8_t* base;   // 1024-aligned dynamic shared memory (every layout starts here)
  uint64_t* bar_ld;
  uint64_t* bar_mma;
  uint32_t tmem;
  uint32_t ph_ld, ph_mma;
  int tid, warp, lane, q4, half;
};

// Compensated bf16 pair: hi = bf16(a, b), lo = bf16 of what the rounding left out.
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(a - bf16_round(a), b - bf16_round(b));
}

// Load a 128x128 fp32 state (row-major [dk][dv]) into this thread's registers.
__device__ __forceinline__ void load_state(const ChainCtx& cx, const float* src, float* S, bool cg) {
  const float* row = src + (size_t)(32 * cx.q4 + cx.lane) * kDim + 64 * cx.half;
  for (int c = 0; c < 64; c += 4) {
    float4 f = cg ? __ldcg(reinterpret_cast<const float4*>(row + c)) : *reinterpret_cast<const float4*>(row + c);
    S[c] = f.x;
    S[c + 1] = f.y;
    S[c + 2] = f.z;
    S[c + 3] = f.w;
  }
}
__device__ __forceinline__ void save_state(const ChainCtx& cx, float* dst, const float* S) {
  float* row = dst + (size_t)(32 * cx.q4 + cx.lane) * kDim + 64 * cx.half;
  for (int c = 0; c < 64; c += 4) *reinterpret_cast<float4*>(row + c) = make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);
}
// The inference chain keeps S transposed over its epilogue threads: thread (q4, half, lane) holds
// S(a, b) for b = 32 q4 + lane (its tensor-memory lane) and a = 64 half + c, c < 64. A warp reads
// and writes 128-byte rows of the row-major state.
__device__ __forceinline__ void load_state_t(const ChainCtx& cx, const float* src, float* S, bool cg) {
  const float* col = src + (size_t)(64 * cx.half) * kDim + 32 * cx.q4 + cx.lane;
#pragma unroll
  for (int c = 0; c < 64; ++c) S[c] = cg ? __ldcg(col + (size_t)c * kDim) : col[(size_t)c * kDim];
}
// The 64 values a thread holds (its row r = 32 q4 + lane of block `half`) as compensated bf16
// operand images hi (dst) and lo (dst + 32 KB): 128-byte rows, two blocks of 128 rows 16 KB apart,
// 16-byte granules swizzled by the row (the SW128 pattern). From the transposed layout (column b of
// S) this is S^T-as-operand MN-major (row b); from the record chain's row layout, K-major (row a).
__device__ __forceinline__ void store_images(const ChainCtx& cx, uint8_t* dst, const float* S) {
  const int r = 32 * cx.q4 + cx.lane;
  uint8_t* hi = dst + cx.half * 16384 + r * 128;
#pragma unroll
  for (int cj = 0; cj < 8; ++cj) {
    float lo[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) lo[u] = S[8 * cj + u] - __bfloat162float(__float2bfloat16_rn(S[8 * cj + u]));
    const uint32_t g = (cj ^ (r & 7)) << 4;
    *reinterpret_cast<uint4*>(hi + g) =
        make_uint4(pack_bf16x2(S[8 * cj], S[8 * cj + 1]), pack_bf16x2(S[8 * cj + 2], S[8 * cj + 3]),
                   pack_bf16x2(S[8 * cj + 4], S[8 * cj + 5]), pack_bf16x2(S[8 * cj + 6], S[8 * cj + 7]));
    *reinterpret_cast<uint4*>(hi + 32768 + g) = make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                                                           pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
  }
}
__device__ __forceinline__ void save_state_t(const ChainCtx& cx, float* dst, const float* S) {
  float* col = dst + (size_t)(64 * cx.half) * kDim + 32 * cx.q4 + cx.lane;
#pragma unroll
  for (int c = 0; c < 64; ++c) col[(size_t)c * kDim] = S[c];
}

// Shared-memory buffers that affine_apply borrows; at the start of an item every staging buffer
// of the chain except S hi is idle.
struct AffineBufs {
  uint8_t* mhi;         // M hi: two dk blocks of 128 rows, 16 KB apart (A K-major, M = 128)
  uint8_t* mlo;         // M lo, dk block 0 (block 1 at mlo + mlo_stride)
  uint32_t mlo_stride;
  uint8_t* slo;         // S_start lo, dv block 0 (block 1 at slo + slo_stride) (B MN-major)
  uint32_t slo_stride;
  uint8_t* shi;         // S_start hi: two blocks, 16 KB apart (staged by the record chain)
  float* stage;         // 32 KB of fp32 staging for the product
};

// M (row-major fp32, 128 x 128) as compensated bf16 images hi / lo, K-major with rows a and two
// 64-column blocks 16 KB apart (hi) or mlo_stride apart (lo): 256 threads, 16 per 512-byte row,
// four 32-byte pieces in flight.
__device__ __forceinline__ void stage_m_hilo(const float* Mm, uint8_t* mhi, uint8_t* mlo, uint32_t mlo_stride,
                                           int tid) {
#pragma unroll
  for (int k0 = 0; k0 < 8; k0 += 4) {
    float4 mv[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = tid + 256 * (k0 + k);
      const float* src = Mm + (size_t)(e >> 4) * kDim + 8 * (e & 15);
      mv[2 * k] = __ldcg(reinterpret_cast<const float4*>(src));
      mv[2 * k + 1] = __ldcg(reinterpret_cast<const float4*>(src + 4));
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int e = tid + 256 * (k0 + k), r = e >> 4, c8 = e & 15, cj = c8 & 7;
      const float x[8] = {mv[2 * k].x, mv[2 * k].y, mv[2 * k].z, mv[2 * k].w,
                          mv[2 * k + 1].x, mv[2 * k + 1].y, mv[2 * k + 1].z, mv[2 * k + 1].w};
      float lo[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) lo[u] = x[u] - __bfloat162float(__float2bfloat16_rn(x[u]));
      const uint32_t off = r * 128 + ((cj ^ (r & 7)) << 4);
      *reinterpret_cast<uint4*>(mhi + (c8 >> 3) * 16384 + off) = make_uint4(
          pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
      *reinterpret_cast<uint4*>(mlo + (c8 >> 3) * mlo_stride + off) = make_uint4(
          pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]), pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
    }
  }
}

// out = M S_start + B (B may be null) on the tensor cores with compensated bf16 operands (x = hi + lo):
// M hi S hi + M hi S lo + M lo S hi, accumulated in the TMEM columns d_col .. d_col + 127. kT: S is
// held transposed (the inference chain) and both of its images are written here, K-major (row b,
// 64 values of a per dk block); otherwise S hi is the chain's staged image and S lo is written
// MN-major (row a).
template <bool kT>
__device__ bool affine_apply(const FwdParams& p, ChainCtx& cx, const AffineBufs& sm, const float* Mm,
                             const float* Bm, const float* S, float* out, uint32_t d_col) {
  if (cx.tid < 256) {
    stage_m_hilo(Mm, sm.mhi, sm.mlo, sm.mlo_stride, cx.tid);
    // S lo (and for kT S hi): this thread's 64 values, row rr of the image's block `half`
    const int rr = 32 * cx.q4 + cx.lane;  // (threads below 256 only)
    uint8_t* slo = sm.slo + cx.half * sm.slo_stride;
    uint8_t* shi = sm.shi + cx.half * 16384;
    for (int cj = 0; cj < 8; ++cj) {
      float lo[8];
      for (int u = 0; u < 8; ++u) lo[u] = S[8 * cj + u] - __bfloat162float(__float2bfloat16_rn(S[8 * cj + u]));
      const uint32_t off = rr * 128 + ((cj ^ (rr & 7)) << 4);
      *reinterpret_cast<uint4*>(slo + off) = make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                                                        pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
      if constexpr (kT)
        *reinterpret_cast<uint4*>(shi + off) =
            make_uint4(pack_bf16x2(S[8 * cj], S[8 * cj + 1]), pack_bf16x2(S[8 * cj + 2], S[8 * cj + 3]),
                       pack_bf16x2(S[8 * cj + 4], S[8 * cj + 5]), pack_bf16x2(S[8 * cj + 6], S[8 * cj + 7]));
    }
  }
  sync_generic_to_async();
  if (cx.tid == 0) {
    // S as the B operand: K-major (kT) or MN-major rows of a
    auto sdesc = [&](const uint8_t* base, uint32_t stride, int ks) {
      return kT ? kmajor_step(kmajor_desc(smem_u32(base), stride, 0), stride, ks)
                : mnmajor_step(mnmajor_desc(smem_u32(base), stride, 0), ks);
    };
    const uint32_t id = idesc_bf16(128, 128, 0, kT ? 0 : 1);
    #pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma_bf16(cx.tmem + d_col, kmajor_step(kmajor_desc(smem_u32(sm.mhi), 16384, 0), 16384, ks),
                sdesc(sm.shi, 16384, ks), id, ks > 0);
    #pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma_bf16(cx.tmem + d_col, kmajor_step(kmajor_desc(smem_u32(sm.mhi), 16384, 0), 16384, ks),
                sdesc(sm.slo, sm.slo_stride, ks), id, 1);
    #pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma_bf16(cx.tmem + d_col, kmajor_step(kmajor_desc(smem_u32(sm.mlo), sm.mlo_stride, 0), sm.mlo_stride, ks),
                sdesc(sm.shi, 16384, ks), id, 1);
    umma_commit(cx.bar_mma);
  }
  if (!wait_all(cx.bar_mma, cx.ph_mma)) return false;
  cx.ph_mma ^= 1;
  tc_fence_after();
  // M S_start + B: the product goes through a 32 KB fp32 stage, 64 rows at a time (granule g of
  // local row rl at rl * 128 + 4 (g XOR rl mod 32): conflict-free both for a thread per row and for
  // a warp per row), so that B is read and out written with coalesced accesses.
  float* stg = sm.stage;
  for (int pass = 0; pass < 2; ++pass) {
    if (cx.tid < 256 && (cx.q4 >> 1) == pass) {
      const uint32_t lane_base = (uint32_t)(32 * cx.q4) << 16;
      const int rl = 32 * (cx.q4 & 1) + cx.lane;
#pragma unroll
      for (int cc = 0; cc < 64; cc += 16) {
        float v[16];
        tmem_ld16(cx.tmem + d_col + lane_base + 64 * cx.half + cc, v);
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
        b[k] = Bm ? __ldcg(reinterpret_cast<const float4*>(Bm + (size_t)r * kDim + 4 * g)) : make_float4(0.f, 0.f, 0.f, 0.f);
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
__device__ __forceinline__ void prefetch_state_l2(const float* m, int tid, int nthreads) {
  for (int l = tid; l < kDim * kDim * 4 / 128; l += nthreads) prefetch_l2(reinterpret_cast<const uint8_t*>(m) + 128 * l);
}

// =========================================================================== warp-specialized chain
//
// The forward chain (inference output pass and pass 1) in transposed form. Every per-chunk product
// has the value index b (for W^T: the key index a) on the 128 accumulator lanes, so that each
// epilogue spreads over the four lane quarters of all eight epilogue warps, and the chunk-to-chunk
// operands S^T, V'^T and V'_s^T stay in tensor memory as bf16 A operands (written by tcgen05.st).
// Per chunk j of one value head:
//   W^T  = K^T T_w^T               formed one chunk ahead (A: K; B: T_w)
//   D_V  = V^T T_u^T               = U^T, issued while the previous state is staged
//   D_V += S^T (-W^T)              the state product, alone on the critical path: D_V = V'^T
//   O^T  = S^T Q^T                 then O^T += V'^T P''^T
//   D_2  = V'_s^T K                V'_s = diag(e^{gamma_C - gamma}) V'
//   S^T <- e^{gamma_C} S^T + D_2   in fp32 registers, staged as bf16 for the next chunk
// The query enters unscaled: P''_ij = (Q K^T)_ij e^{-gamma_j}, and O_i = scale e^{gamma_i} (Q S +
// P'' V')_i with the per-token factors written by kkt_solve. A row whose decay since the chunk
// start is below kExactCut keeps the plain P and has its query row zeroed instead: its Q S term is
// below e^{kExactCut} of the chunk-start state (the cut of the exact split's warm-ups).
// Roles in one CTA of 11 warps:
//   warp 8    TMA producer, three lanes with one ring each: A = K, T_w, gamma and the factors
//             (three slots, since W^T runs a chunk ahead), B = V, T_u (two slots, released by the
//             U product), C = Q, P'' of the output chunks (two slots).
//   warp 9    MMA issuer of the two state products (one lane).
//   warp 10   MMA issuer of W^T, U^T, Q S and P'' V' (one lane).
//   warps 0-7 epilogue: V'^T and V'_s^T into tensor memory, -W^T of the next chunk into shared
//             memory, the state update, O.
// Hand-offs are mbarriers only: tcgen05.commit from the issuer, one arrival per epilogue warp,
// TMA transaction counts from the producer.

// TMEM columns of the chain (512 allocated).
constexpr uint32_t kTtS = 0;     // S^T bf16 (A operand: lane b, column c holds a = 2c, 2c + 1)    64 cols
constexpr uint32_t kTtDV = 64;   // D_V = (U - W S)^T fp32 (lane b, column t)                      64 cols
constexpr uint32_t kTtVp = 128;  // V'^T bf16 (A operand: lane b, column c holds t = 2c, 2c + 1)   32 cols
constexpr uint32_t kTtVs = 160;  // V'_s^T bf16 (A operand)                                        32 cols
constexpr uint32_t kTtW = 192;   // W^T fp32 (lane a, column t)                                    64 cols
constexpr uint32_t kTtD2 = 256;  // D_2 = (K^T V'_s)^T fp32 (lane b, column a)                     128 cols
constexpr uint32_t kTtO = 384;   // O^T fp32 (lane b, column t), two buffers of 64 columns         128 cols

// bf16 S^T into this thread's lane of the A operand: column 32 half + i holds a = 64 half + 2i, 2i + 1.
__device__ __forceinline__ void stage_state_t(const ChainCtx& cx, const float* S) {
  const uint32_t base = cx.tmem + ((uint32_t)(32 * cx.q4) << 16) + kTtS + 32 * cx.half;
  uint32_t r[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = pack_bf16x2(S[2 * i], S[2 * i + 1]);
  tmem_st16(base, r);
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = pack_bf16x2(S[32 + 2 * i], S[33 + 2 * i]);
  tmem_st16(base + 16, r);
}

constexpr int kRingA = 3;
struct WtSmem {
  uint8_t k[kRingA][16384];  // K rows t, two dk blocks      (A MN-major for W^T, B MN-major for D_2)
  uint8_t tw[kRingA][8192];  // T diag(beta e^gamma) rows t   (B K-major)
  uint8_t v[2][16384];       // V rows t, two dv blocks      (A MN-major)
  uint8_t tu[2][8192];       // T diag(beta) rows t           (B K-major)
  uint8_t q[2][16384];       // Q rows t, two dk blocks      (B K-major)
  uint8_t pp[2][8192];       // P'' rows t                    (B K-major)
  uint8_t wn[16384];         // -W^T rows dk, 64 t per row   (B MN-major)
  uint8_t ostage[2][16384];  // O rows t, two dv blocks (bf16, 128B-swizzled), the source of its TMA store
  float gam[kRingA][64];     // chunk-local cumulative gate
  float fac[kRingA][kFacFloats];
};
constexpr int kWsThreads = 352;
// Buffers affine_apply borrows (all idle between chain runs): M hi in K slots 0-1, S_start lo in K
// slot 2 and the T_w slots, M lo in the V slots, S_start hi in the Q slots, the fp32 stage in the
// P'' slots and -W^T.
__device__ __forceinline__ AffineBufs affine_bufs(WtSmem& sm) {
  return {sm.k[0], sm.v[0], 16384u, sm.k[2], 16384u, sm.q[0], reinterpret_cast<float*>(sm.pp[0])};
}
static_assert(offsetof(WtSmem, tw) == offsetof(WtSmem, k) + 3 * 16384, "S lo block 1 follows K slot 2");
static_assert(offsetof(WtSmem, wn) == offsetof(WtSmem, pp) + 16384, "the fp32 stage spans P'' and -W^T");

struct WtBars {
  uint64_t full_a[kRingA], empty_a[kRingA], full_b[2], empty_b[2], full_c[2], empty_c[2];
  uint64_t a_done, pre_done, b_done, o_done, qs_done, u_done, staged, epi1, epi2, o_read[2];
};
// Phase parities of these barriers as the bits of one register (slots indexed at run time would
// otherwise put them in local memory).
enum WtBit : int {
  kBitFullA = 0, kBitEmptyA = 3, kBitFullB = 6, kBitEmptyB = 8, kBitFullC = 10, kBitEmptyC = 12, kBitADone = 14,
  kBitPreDone = 15, kBitBDone = 16, kBitODone = 17, kBitStaged = 18, kBitEpi1 = 19, kBitEpi2 = 20, kBitORead = 21,
  kBitQsDone = 23, kBitUDone = 24
};
__device__ __forceinline__ void wt_bars_init(WtBars& bb) {
  for (int i = 0; i < kRingA; ++i) {
    mbar_init(&bb.full_a[i], 1);
    mbar_init(&bb.empty_a[i], 2 + 8);  // both issuers' commits and one arrival per epilogue warp
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(&bb.full_b[i], 1);
    mbar_init(&bb.empty_b[i], 1);
    mbar_init(&bb.full_c[i], 1);
    mbar_init(&bb.empty_c[i], 1);
    mbar_init(&bb.o_read[i], 8);
  }
  mbar_init(&bb.a_done, 1);
  mbar_init(&bb.pre_done, 1);
  mbar_init(&bb.b_done, 1);
  mbar_init(&bb.o_done, 1);
  mbar_init(&bb.qs_done, 1);
  mbar_init(&bb.u_done, 1);
  mbar_init(&bb.staged, 8);
  mbar_init(&bb.epi1, 8);
  mbar_init(&bb.epi2, 8);
}

// Bounded wait that never diverges: a phase that is already complete costs one try_wait; otherwise
// the thread polls until the phase completes, the budget runs out or another role has given up
// (recorded in *abort), so all threads keep executing the same barriers and none waits for a
// phase that an aborted role will not complete.
__device__ __forceinline__ void role_wait(uint64_t* bar, uint32_t& ph, volatile int* abort) {
  if (!mbar_try_wait(bar, ph)) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, ph)) {
      if (*abort || clock64() - t0 > kWaitBudget) {
        *abort = 1;
        break;
      }
    }
  }
  ph ^= 1;
  tc_fence_after();
}

// Named barrier of the 256 epilogue threads.
__device__ __forceinline__ void e_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// role_wait on the parity bit `bit` of ph.
__device__ __forceinline__ void bit_wait(uint64_t* bar, uint32_t& ph, int bit, volatile int* abort) {
  const uint32_t par = (ph >> bit) & 1u;
  if (!mbar_try_wait(bar, par)) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, par)) {
      if (*abort || clock64() - t0 > kWaitBudget) {
        *abort = 1;
        break;
      }
    }
  }
  ph ^= 1u << bit;
  tc_fence_after();
}

// One arrival per epilogue warp once the warp's tensor-memory accesses (and, with smem, its
// shared-memory writes) are ordered before the products that follow.
__device__ __forceinline__ void warp_handoff(const ChainCtx& cx, bool smem, uint64_t* bar) {
  if (smem) fence_proxy_async_smem();
  tc_fence_before();
  __syncwarp();
  if (cx.lane == 0) mbar_arrive(bar);
}

// Run chunks [gc0, gc1) of one document for value head h from S (epilogue registers, transposed
// layout). Chunks gc >= gc_out write O. kWithU = false runs the transition chain (no U term, no
// output). All threads of the CTA call this; returns false after a failed wait.
template <bool kWithU>
__device__ bool run_wt(const FwdParams& p, ChainCtx& cx, WtBars& bb, uint32_t& ph, volatile int* abort, float* S,
                       int gc0, int gc1, int gc_out, int h, int hk) {
  WtSmem& sm = *reinterpret_cast<WtSmem*>(cx.base);
  const int n = gc1 - gc0;
  if (n <= 0) return true;
  const int Hv = p.d.Hv;
  const int32_t* ctok = ws_ptr<int32_t>(p, p.L.chunk_tok0);
  const int32_t* clen = ws_ptr<int32_t>(p, p.L.chunk_len);
  // the output chunks are the last n - j_out of the run
  const int j_out = !kWithU ? n : (gc_out <= gc0 ? 0 : (gc_out - gc0 < n ? gc_out - gc0 : n));
  const int n_out = n - j_out;

  if (cx.warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (cx.lane == 0) {
      // ring A: K, T_w, gamma, factors of every chunk
      for (int j = 0; j < n; ++j) {
        const int gc = gc0 + j, s = j % kRingA;
        const size_t r = (size_t)gc * Hv + h;
        if (j + kRingA < n) {  // chunk j + 3 into L2 while the ring is full
          const int g3 = gc + kRingA, t3 = ctok[g3];
          tma_prefetch_3d(&p.tm_k, 0, hk, t3);
          tma_prefetch_3d(&p.tm_k, 64, hk, t3);
          bulk_prefetch_l2(p.ws + p.L.tw + ((size_t)g3 * Hv + h) * 8192, 8192);
        }
        if (j >= kRingA) bit_wait(&bb.empty_a[s], ph, kBitEmptyA + (s), abort);
        if (*abort) break;
        mbar_arrive_expect_tx(&bb.full_a[s], 16384 + 8192 + 256 + kFacFloats * 4);
        tma_load_3d(sm.k[s], &p.tm_k, 0, hk, ctok[gc], &bb.full_a[s]);
        tma_load_3d(sm.k[s] + 8192, &p.tm_k, 64, hk, ctok[gc], &bb.full_a[s]);
        bulk_load(sm.tw[s], p.ws + p.L.tw + r * 8192, 8192, &bb.full_a[s]);
        bulk_load(sm.gam[s], p.ws + p.L.gam + r * 256, 256, &bb.full_a[s]);
        bulk_load(sm.fac[s], p.ws + p.L.fac + r * (kFacFloats * 4), kFacFloats * 4, &bb.full_a[s]);
      }
      for (int j = (n > kRingA ? n - kRingA : 0); j < n; ++j)
        bit_wait(&bb.empty_a[j % kRingA], ph, kBitEmptyA + (j % kRingA), abort);
    } else if (cx.lane == 1 && kWithU) {
      // ring B: V, T_u of every chunk
      for (int j = 0; j < n; ++j) {
        const int gc = gc0 + j, s = j & 1;
        const size_t r = (size_t)gc * Hv + h;
        if (j + 2 < n) {
          const int g2 = gc + 2, t2 = ctok[g2];
          tma_prefetch_3d(&p.tm_v, 0, h, t2);
          tma_prefetch_3d(&p.tm_v, 64, h, t2);
          bulk_prefetch_l2(p.ws + p.L.tu + ((size_t)g2 * Hv + h) * 8192, 8192);
        }
        if (j >= 2) bit_wait(&bb.empty_b[s], ph, kBitEmptyB + (s), abort);
        if (*abort) break;
        mbar_arrive_expect_tx(&bb.full_b[s], 16384 + 8192);
        tma_load_3d(sm.v[s], &p.tm_v, 0, h, ctok[gc], &bb.full_b[s]);
        tma_load_3d(sm.v[s] + 8192, &p.tm_v, 64, h, ctok[gc], &bb.full_b[s]);
        bulk_load(sm.tu[s], p.ws + p.L.tu + r * 8192, 8192, &bb.full_b[s]);
      }
      for (int j = (n > 2 ? n - 2 : 0); j < n; ++j) bit_wait(&bb.empty_b[j & 1], ph, kBitEmptyB + (j & 1), abort);
    } else if (cx.lane == 2) {
      // ring C: Q, P'' of the output chunks
      for (int jc = 0; jc < n_out; ++jc) {
        const int gc = gc0 + j_out + jc, s = jc & 1;
        const size_t r = (size_t)gc * Hv + h;
        if (jc + 2 < n_out) {
          const int g2 = gc + 2, t2 = ctok[g2];
          tma_prefetch_3d(&p.tm_q, 0, hk, t2);
          tma_prefetch_3d(&p.tm_q, 64, hk, t2);
          bulk_prefetch_l2(p.p_img + ((size_t)g2 * Hv + h) * 8192, 8192);
        }
        if (jc >= 2) bit_wait(&bb.empty_c[s], ph, kBitEmptyC + (s), abort);
        if (*abort) break;
        mbar_arrive_expect_tx(&bb.full_c[s], 16384 + 8192);
        tma_load_3d(sm.q[s], &p.tm_q, 0, hk, ctok[gc], &bb.full_c[s]);
        tma_load_3d(sm.q[s] + 8192, &p.tm_q, 64, hk, ctok[gc], &bb.full_c[s]);
        bulk_load(sm.pp[s], p.p_img + r * 8192, 8192, &bb.full_c[s]);
      }
      for (int jc = (n_out > 2 ? n_out - 2 : 0); jc < n_out; ++jc)
        bit_wait(&bb.empty_c[jc & 1], ph, kBitEmptyC + (jc & 1), abort);
    }
    return !*abort;
  }
  // MMA issue: an issuing thread waits for the tensor pipe at every product, and shares its
  // sub-partition's issue slots with two epilogue warps, so the products are split over two
  // threads in different sub-partitions: warp 9 issues the two state products, warp 10 the rest.
  const uint32_t tm = cx.tmem;
  constexpr uint32_t id_kt = idesc_bf16(128, 64, 1, 0);   // MN-major A x K-major B: W^T, U^T
  constexpr uint32_t id_sw = idesc_bf16(128, 64, 0, 1);   // tensor-memory A x MN-major B: S^T (-W^T)
  constexpr uint32_t id_tk = idesc_bf16(128, 64, 0, 0);   // tensor-memory A x K-major B: S^T Q^T, V'^T P''^T
  constexpr uint32_t id_d2 = idesc_bf16(128, 128, 0, 1);  // tensor-memory A x MN-major B: V'_s^T K
  // k-step-0 descriptors of slot 0 of every operand (the buffers do not move; slot s of a ring adds
  // s times its size to the start-address field, which never carries out of it)
  const uint64_t d_k = mnmajor_desc(smem_u32(sm.k[0]), 8192, 0);  // slots 16 KB apart
  if (cx.warp == 9) {
    // ------------------------------------------------ issuer of the state products (one lane)
    if (cx.lane == 0) {
      const uint64_t d_wn = mnmajor_desc(smem_u32(sm.wn), 8192, 0);
      for (int j = 0; j < n && !*abort; ++j) {
        const int s = j % kRingA;
        bit_wait(&bb.staged, ph, kBitStaged, abort);  // -W^T(j) and Q(j) are staged
        bit_wait(&bb.epi2, ph, kBitEpi2, abort);      // S^T(j) is staged
        if (kWithU) bit_wait(&bb.u_done, ph, kBitUDone, abort);  // U^T(j) is in D_V
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16_ts(tm + kTtDV, tm + kTtS + 8 * ks, mnmajor_step(d_wn, ks), id_sw, (kWithU || ks > 0) ? 1 : 0);
        umma_commit(&bb.a_done);
        bit_wait(&bb.epi1, ph, kBitEpi1, abort);
        const uint64_t ka = d_k + (uint64_t)(s * (16384 >> 4));
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16_ts(tm + kTtD2, tm + kTtVs + 8 * ks, mnmajor_step(ka, ks), id_d2, ks > 0);
        umma_commit(&bb.b_done);
        umma_commit(&bb.empty_a[s]);
      }
      bit_wait(&bb.epi2, ph, kBitEpi2, abort);  // the epilogue's last state hand-off
    }
    return !*abort;
  }
  if (cx.warp == 10) {
    // ------------------------------------------------ issuer of the other products (one lane):
    // Q S and chunk j + 1's W^T behind the state product D_V, P'' V' and chunk j + 1's U^T behind D_2
    if (cx.lane == 0) {
      const uint64_t d_tw = kmajor_desc(smem_u32(sm.tw[0]), 8192, 0);   // 8 KB
      const uint64_t d_v = mnmajor_desc(smem_u32(sm.v[0]), 8192, 0);    // 16 KB
      const uint64_t d_tu = kmajor_desc(smem_u32(sm.tu[0]), 8192, 0);   // 8 KB
      const uint64_t d_q = kmajor_desc(smem_u32(sm.q[0]), 8192, 0);     // 16 KB
      const uint64_t d_pp = kmajor_desc(smem_u32(sm.pp[0]), 8192, 0);   // 8 KB
      auto prep = [&](int j) {  // W^T of chunk j (the staging of chunk j - 1 has read W^T)
        const int s = j % kRingA;
        bit_wait(&bb.full_a[s], ph, kBitFullA + (s), abort);
        const uint64_t ka = d_k + (uint64_t)(s * (16384 >> 4)), ta = d_tw + (uint64_t)(s * (8192 >> 4));
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tm + kTtW, mnmajor_step(ka, ks), kmajor_step(ta, 8192, ks), id_kt, ks > 0);
        umma_commit(&bb.pre_done);
        umma_commit(&bb.empty_a[s]);
      };
      auto issue_u = [&](int j) {  // U^T of chunk j into D_V (the V' epilogue of chunk j - 1 has read it)
        const int s = j & 1;
        bit_wait(&bb.full_b[s], ph, kBitFullB + (s), abort);
        const uint64_t va = d_v + (uint64_t)(s * (16384 >> 4)), ua = d_tu + (uint64_t)(s * (8192 >> 4));
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_bf16(tm + kTtDV, mnmajor_step(va, ks), kmajor_step(ua, 8192, ks), id_kt, ks > 0);
        umma_commit(&bb.u_done);
        umma_commit(&bb.empty_b[s]);
      };
      prep(0);
      if (kWithU) issue_u(0);
      for (int j = 0; j < n && !*abort; ++j) {
        const bool out = j >= j_out;
        const int so = (j - j_out) & 1;
        bit_wait(&bb.a_done, ph, kBitADone, abort);  // the state product of chunk j has run
        if (out) {
          // Q S (the output of chunk j - 2 has left this buffer)
          if (j - j_out >= 2) bit_wait(&bb.o_read[so], ph, kBitORead + (so), abort);
          bit_wait(&bb.full_c[so], ph, kBitFullC + (so), abort);
          const uint64_t qa = d_q + (uint64_t)(so * (16384 >> 4));
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_bf16_ts(tm + kTtO + 64 * so, tm + kTtS + 8 * ks, kmajor_step(qa, 8192, ks), id_tk, ks > 0);
          umma_commit(&bb.qs_done);
        }
        if (j + 1 < n) prep(j + 1);  // the epilogue stages -W^T(j + 1) while D_2 runs
        bit_wait(&bb.b_done, ph, kBitBDone, abort);  // D_2 has run (V'^T is in place)
        if (out) {
          const uint64_t pa = d_pp + (uint64_t)(so * (8192 >> 4));
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16_ts(tm + kTtO + 64 * so, tm + kTtVp + 8 * ks, kmajor_step(pa, 8192, ks), id_tk, 1);
          umma_commit(&bb.o_done);
          umma_commit(&bb.empty_c[so]);
        }
        if (kWithU && j + 1 < n) issue_u(j + 1);
      }
      // the outputs of the last two chunks have been read (every phase consumed)
      for (int jc = (n_out > 2 ? n_out - 2 : 0); jc < n_out; ++jc)
        bit_wait(&bb.o_read[jc & 1], ph, kBitORead + (jc & 1), abort);
    }
    return !*abort;
  }
  // -------------------------------------------------------------------- epilogue warps 0-7
  const uint32_t lq = (uint32_t)(32 * cx.q4) << 16;
  const int b = 32 * cx.q4 + cx.lane;  // this thread's lane: the value index (the key index of W^T)
  stage_state_t(cx, S);
  tmem_st_wait();
  warp_handoff(cx, false, &bb.epi2);
  // -W^T of chunk j into shared memory (row a = this lane, tokens 32 half ..); for an output chunk,
  // its query rows past the cut zeroed
  auto staging = [&](int j) {
    const int s = j % kRingA;
    bit_wait(&bb.pre_done, ph, kBitPreDone, abort);
    bit_wait(&bb.full_a[s], ph, kBitFullA + (s), abort);
    {
      float w[32];
      tmem_ld32(cx.tmem + lq + kTtW + 32 * cx.half, w);
      tmem_ld_wait();
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int cj = 4 * cx.half + c4;
        const float* x = w + 8 * c4;
        *reinterpret_cast<uint4*>(sm.wn + b * 128 + ((cj ^ (b & 7)) << 4)) =
            make_uint4(pack_bf16x2(-x[0], -x[1]), pack_bf16x2(-x[2], -x[3]), pack_bf16x2(-x[4], -x[5]),
                       pack_bf16x2(-x[6], -x[7]));
      }
    }
    if (j >= j_out) {
      const int so = (j - j_out) & 1;
      bit_wait(&bb.full_c[so], ph, kBitFullC + (so), abort);
      const float* gm = sm.gam[s];
      if (gm[63] < kExactCut) {  // gamma is nonincreasing: zero the query rows past the cut
        for (int e = cx.tid; e < 2 * 64 * 8; e += 256) {
          const int blk = e >> 9, r = (e >> 3) & 63, cj = e & 7;
          if (gm[r] < kExactCut)
            *reinterpret_cast<uint4*>(sm.q[so] + blk * 8192 + r * 128 + (cj << 4)) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    warp_handoff(cx, true, &bb.staged);
  };
  staging(0);
  for (int j = 0; j < n; ++j) {
    const int gc = gc0 + j, s = j % kRingA;
    const bool out = j >= j_out;
    const int so = (j - j_out) & 1;
    const float* fc = sm.fac[s];  // e^{gamma_C - gamma_t} [0, 64), output factors [64, 128), e^{gamma_C}
    const int nn = out ? clen[gc] : 0, tok0 = out ? ctok[gc] : 0;  // (global loads, used by the O stores)
    bit_wait(&bb.a_done, ph, kBitADone, abort);
    {
      // V' of this lane's value index, tokens 32 half ..: V'^T and V'_s^T as bf16 A operands
      float v[32];
      tmem_ld32(cx.tmem + lq + kTtDV + 32 * cx.half, v);
      tmem_ld_wait();
      uint32_t rp[16], rs[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint64_t sc = *reinterpret_cast<const uint64_t*>(fc + 32 * cx.half + 2 * i);
        const uint64_t vs = f2_mul(f2_pack(v[2 * i], v[2 * i + 1]), sc);
        rp[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        rs[i] = pack_bf16x2(f2_lo(vs), f2_hi(vs));
      }
      tmem_st16(cx.tmem + lq + kTtVp + 16 * cx.half, rp);
      tmem_st16(cx.tmem + lq + kTtVs + 16 * cx.half, rs);
      tmem_st_wait();
    }
    warp_handoff(cx, false, &bb.epi1);
    if (j + 1 < n) staging(j + 1);
    bit_wait(&bb.b_done, ph, kBitBDone, abort);
    {
      const float GC = fc[128];
      const uint64_t gc2 = f2_pack(GC, GC);
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float d[32];
        tmem_ld32(cx.tmem + lq + kTtD2 + 64 * cx.half + 32 * hc, d);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; x += 2) {  // e^{gamma_C} S + D_2, two values per instruction
          const uint64_t r = f2_fma(gc2, f2_pack(S[32 * hc + x], S[32 * hc + x + 1]), f2_pack(d[x], d[x + 1]));
          S[32 * hc + x] = f2_lo(r);
          S[32 * hc + x + 1] = f2_hi(r);
        }
      }
      if (out) bit_wait(&bb.qs_done, ph, kBitQsDone, abort);  // Q S(j) has read S^T(j)
      stage_state_t(cx, S);
      tmem_st_wait();
    }
    warp_handoff(cx, false, &bb.epi2);
    if (out) {
      // O of chunk j while chunk j + 1 runs: O^T (lane b, tokens 32 half ..) is turned into rows of
      // O in a 128B-swizzled shared tile (lane pairs swap one value per token pair, so that each
      // 4-byte store holds two neighbouring values of b) and leaves by one TMA store; a partial
      // chunk (the end of a document) is copied row by row so that the next document's rows are not
      // touched
      bit_wait(&bb.o_done, ph, kBitODone, abort);
      float o[32];
      tmem_ld32(cx.tmem + lq + kTtO + 64 * so + 32 * cx.half, o);
      tmem_ld_wait();
      warp_handoff(cx, false, &bb.o_read[so]);
      uint8_t* stg = sm.ostage[so];
      if (cx.tid == 0) bulk_wait_read<1>();  // the store from this tile two chunks ago has read it (only a
                                             // run's last chunk can be partial and skip its store)
      e_sync();
      // the output factors of this thread's 32 tokens, in registers before any store to the tile
      // (the stores could otherwise alias them and serialize the loop)
      uint64_t of[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const ulonglong2 f4 = *reinterpret_cast<const ulonglong2*>(fc + 64 + 32 * cx.half + 4 * q);
        of[2 * q] = f4.x;
        of[2 * q + 1] = f4.y;
      }
      // O times its output factors, two tokens per instruction
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const uint64_t x = f2_mul(f2_pack(o[2 * q], o[2 * q + 1]), of[q]);
        o[2 * q] = f2_lo(x);
        o[2 * q + 1] = f2_hi(x);
      }
      const bool odd = cx.lane & 1;
      const int be = b & ~1;  // the even value index of the pair
      const uint32_t blk = (uint32_t)(be >> 6) * 8192, c = (uint32_t)(be & 63) >> 3, e2 = (uint32_t)(be & 7) * 2;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        // tokens t0 and t0 + 4 (rows four apart keep the two halves of a warp's store on
        // different banks); the even lane stores row t0, the odd lane row t0 + 4
        const int i0 = 8 * (m >> 2) + (m & 3), t0 = 32 * cx.half + i0;
        const float x0 = o[i0], x1 = o[i0 + 4];
        const float got = __shfl_xor_sync(0xffffffffu, odd ? x0 : x1, 1);
        const int t = odd ? t0 + 4 : t0;
        const uint32_t v = odd ? pack_bf16x2(got, x1) : pack_bf16x2(x0, got);
        *reinterpret_cast<uint32_t*>(stg + blk + t * 128 + ((c ^ (t & 7)) << 4) + e2) = v;
      }
      fence_proxy_async_smem();
      e_sync();
      if (nn == kChunk) {
        if (cx.tid == 0) {
          tma_store_3d(&p.tm_o, stg, 0, h, tok0);
          tma_store_3d(&p.tm_o, stg + 8192, 64, h, tok0);
          bulk_commit_group();
        }
      } else {
        for (int e = cx.tid; e < nn * 16; e += 256) {
          const int t = e >> 4, u = e & 15, cj = u & 7;
          reinterpret_cast<uint4*>(p.out + ((size_t)(tok0 + t) * Hv + h) * kDim)[u] =
              *reinterpret_cast<const uint4*>(stg + (u >> 3) * 8192 + t * 128 + ((cj ^ (t & 7)) << 4));
        }
      }
    }
    __syncwarp();
    if (cx.lane == 0) mbar_arrive(&bb.empty_a[s]);  // gamma and the factors of chunk j are read
  }
  if (cx.tid == 0) bulk_wait_all();  // every output store has landed before the tiles are reused
  return !*abort;
}

// ----------------------------------------------------------------- barriers of the record chain
struct WsBars {
  uint64_t full[3], fullq, fullu, empty[3], emptyq, a_done, pre_done, b_done, u_done, epi1, staged, epi2, vfree;
};
struct WsPhase {
  uint32_t full[3], fullq, fullu, empty[3], emptyq, a_done, pre_done, b_done, u_done, epi1, staged, epi2, vfree;
};


// Epilogue hand-off: make this thread's shared-memory writes visible to the async proxy and its
// TMEM reads ordered, meet the other epilogue threads, then one thread arrives on each barrier.
__device__ __forceinline__ void e_handoff(int tid, uint64_t* b1, uint64_t* b2 = nullptr) {
  fence_proxy_async_smem();
  tc_fence_before();
  e_sync();
  if (tid == 0) {
    mbar_arrive(b1);
    if (b2) mbar_arrive(b2);
  }
}

// ============================================================== warp-specialized record chain
//
// The backward's recompute of the forward chain: the same recurrence with compensated bf16
// operands (x = hi + lo for T_w, T_u, W, S and V'_s; K and V are exact in bf16), optionally
// writing the per-chunk records that the gradient kernels read (chunk-start S hi / lo and V'
// hi / lo as 128B-swizzled images). No output. Roles in the chain's CTA:
//   warp 8      TMA producer: K and gamma of chunk j into stage j % 3; T_w hi / lo (one buffer,
//               released by the W product); V and T_u hi / lo (one buffer, released by the U
//               product).
//   warp 9      MMA issuer of the state products, per chunk j: D_V -= W S (M = 64; W S as W hi S hi +
//               W hi S lo + W lo S hi), then D2 = K^T (V'_s hi + V'_s lo) (M = 128).
//   warp 10     MMA issuer of D_V = T_u V (behind chunk j - 1's D2) and chunk j+1's W = T_w K (M = 64).
//   warps 0-7   epilogue: -W hi / lo staging, V' (records, V'_s hi / lo), S = e^{gamma_C} S + D2
//               with its hi / lo staging. A chunk-start state reaches its record by bulk store
//               straight from the staged images.
constexpr int kRecStages = 3;  // K is loaded up to two chunks ahead
struct RecSmem {
  uint8_t k[kRecStages][16384];  // [stage] K rows t, two dk blocks (B MN-major for W, A MN-major for K^T V'_s)
  uint8_t v[16384];       // V rows t, two dv blocks (B MN-major)
  uint8_t tu[2][8192];    // T diag(beta) hi, lo (A K-major, M = 64)
  uint8_t tw[2][8192];    // T diag(beta e^gamma) hi, lo (A K-major, M = 64)
  uint8_t wn[2][16384];   // -W hi, -W lo: two dk blocks of 64 rows each (A K-major, M = 64)
  uint8_t s[2][16384];    // S hi rows dk, two dv blocks (B MN-major)
  uint8_t slo[2][16384];  // S lo
  uint8_t vs[2][8192];    // V'_s = diag(e^{gamma_C - gamma}) V' hi, two dv blocks (B MN-major)
  uint8_t vslo[2][8192];  // V'_s lo
  float gam[kRecStages][64];  // [stage] chunk-local cumulative gate
};
constexpr size_t kSmemBytes = (sizeof(WtSmem) > sizeof(RecSmem) ? sizeof(WtSmem) : sizeof(RecSmem)) + 1024;
static_assert(kSmemBytes <= 232448, "chain shared memory");
__device__ __forceinline__ AffineBufs affine_bufs(RecSmem& sm) {
  return {sm.wn[0], sm.k[0], 16384u, sm.slo[0], 16384u, sm.s[0], reinterpret_cast<float*>(sm.tu[0])};
}

// TMEM columns of the record chain.
constexpr uint32_t kRtW = 0;     // W                          (M = 64, 128 cols)
constexpr uint32_t kRtV = 128;   // D_V = U - W S              (M = 64, 128 cols)
constexpr uint32_t kRtD2 = 256;  // K^T V'_s                   (M = 128, 128 cols)

// This thread's 64 state values (row dk = 32 q4 + lane, dv block `half`) as bf16 hi / lo images.
__device__ __forceinline__ void store_state_comp(RecSmem& sm, const ChainCtx& cx, const float* S) {
  const int r = 32 * cx.q4 + cx.lane;
#pragma unroll
  for (int cj = 0; cj < 8; ++cj) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) split_pair(S[8 * cj + 2 * u], S[8 * cj + 2 * u + 1], hi[u], lo[u]);
    const uint32_t off = r * 128 + ((cj ^ (r & 7)) << 4);
    *reinterpret_cast<uint4*>(sm.s[cx.half] + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(sm.slo[cx.half] + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Run chunks [gc0, gc1) of one document for value head h from S (epilogue registers; its hi / lo
// images are already in sm.s / sm.slo). kWithU = false runs the transition chain (no U term).
// kStore writes the records of the chunks from gc_rec on (the ones before are a warm-up). All
// threads of the CTA call this; returns false after a failed wait.
template <bool kWithU, bool kStore>
__device__ bool run_ws_rec(const FwdParams& p, ChainCtx& cx, WsBars& bb, WsPhase& ph, volatile int* abort,
                           float* S, int gc0, int gc1, int h, int hk, int gc_rec) {
  RecSmem& sm = *reinterpret_cast<RecSmem*>(cx.base);
  const int n = gc1 - gc0;
  if (n <= 0) return true;
  const int Hv = p.d.Hv;
  const int32_t* ctok = ws_ptr<int32_t>(p, p.L.chunk_tok0);
  auto rec = [&](int gc) { return (size_t)gc * Hv + h; };

  if (cx.warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (cx.lane == 0) {
      for (int j = 0; j < n; ++j) {
        const int gc = gc0 + j, st = j % kRecStages, tok0 = ctok[gc];
        if (j >= kRecStages) role_wait(&bb.empty[st], ph.empty[st], abort);
        if (*abort) break;
        mbar_arrive_expect_tx(&bb.full[st], 16384 + 256);
        tma_load_3d(sm.k[st], &p.tm_k, 0, hk, tok0, &bb.full[st]);
        tma_load_3d(sm.k[st] + 8192, &p.tm_k, 64, hk, tok0, &bb.full[st]);
        bulk_load(sm.gam[st], p.ws + p.L.gam + rec(gc) * 256, 256, &bb.full[st]);
        if (j >= 1) role_wait(&bb.emptyq, ph.emptyq, abort);
        if (*abort) break;
        mbar_arrive_expect_tx(&bb.fullq, 16384);
        bulk_load(sm.tw[0], p.ws + p.L.tw + rec(gc) * 8192, 8192, &bb.fullq);
        bulk_load(sm.tw[1], p.tw_lo + rec(gc) * 8192, 8192, &bb.fullq);
        if (kWithU) {
          if (j >= 1) role_wait(&bb.vfree, ph.vfree, abort);
          if (*abort) break;
          mbar_arrive_expect_tx(&bb.fullu, 32768);
          tma_load_3d(sm.v, &p.tm_v, 0, h, tok0, &bb.fullu);
          tma_load_3d(sm.v + 8192, &p.tm_v, 64, h, tok0, &bb.fullu);
          bulk_load(sm.tu[0], p.ws + p.L.tu + rec(gc) * 8192, 8192, &bb.fullu);
          bulk_load(sm.tu[1], p.tu_lo + rec(gc) * 8192, 8192, &bb.fullu);
        }
      }
      // drain: wait for the release of the last uses so that every phase is consumed
      for (int j = (n >= kRecStages ? n - kRecStages : 0); j < n; ++j)
        role_wait(&bb.empty[j % kRecStages], ph.empty[j % kRecStages], abort);
      role_wait(&bb.emptyq, ph.emptyq, abort);
      if (kWithU) role_wait(&bb.vfree, ph.vfree, abort);
    }
    return !*abort;
  }
  // MMA issue in two threads of different sub-partitions (an issuing thread waits for the tensor
  // pipe at every product and shares its sub-partition's issue slots with two epilogue warps):
  // warp 9 issues the state products D_V -= W S and D_2, warp 10 U and chunk j + 1's W.
  const uint32_t tm = cx.tmem;
  constexpr uint32_t i64 = idesc_bf16(64, 128, 0, 1);
  constexpr uint32_t i128 = idesc_bf16(128, 128, 1, 1);
  // k-step-0 descriptors of every operand (the buffers do not move)
  const uint64_t d_kb0 = mnmajor_desc(smem_u32(sm.k[0]), 8192, 0);  // K stages 16 KB apart
  if (cx.warp == 9) {
    // ------------------------------------------------ issuer of the state products (one lane)
    if (cx.lane == 0) {
      const uint64_t d_wn[2] = {kmajor_desc(smem_u32(sm.wn[0]), 8192, 0), kmajor_desc(smem_u32(sm.wn[1]), 8192, 0)};
      const uint64_t d_s = mnmajor_desc(smem_u32(sm.s[0]), 16384, 0);
      const uint64_t d_slo = mnmajor_desc(smem_u32(sm.slo[0]), 16384, 0);
      const uint64_t d_vs[2] = {mnmajor_desc(smem_u32(sm.vs[0]), 8192, 0), mnmajor_desc(smem_u32(sm.vslo[0]), 8192, 0)};
      const uint32_t dv = tm + kRtV;
      for (int j = 0; j < n && !*abort; ++j) {
        const int st = j % kRecStages;
        role_wait(&bb.staged, ph.staged, abort);
        role_wait(&bb.epi2, ph.epi2, abort);
        if (kWithU) role_wait(&bb.u_done, ph.u_done, abort);  // U(j) is in D_V
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          umma_bf16(dv, kmajor_step(d_wn[0], 8192, ks), mnmajor_step(d_s, ks), i64, (kWithU || ks > 0) ? 1 : 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) umma_bf16(dv, kmajor_step(d_wn[0], 8192, ks), mnmajor_step(d_slo, ks), i64, 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) umma_bf16(dv, kmajor_step(d_wn[1], 8192, ks), mnmajor_step(d_s, ks), i64, 1);
        umma_commit(&bb.a_done);
        role_wait(&bb.epi1, ph.epi1, abort);
        const uint64_t ka = d_kb0 + (uint64_t)(st * (16384 >> 4));
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_bf16(tm + kRtD2, mnmajor_step(ka, ks), mnmajor_step(d_vs[0], ks), i128, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_bf16(tm + kRtD2, mnmajor_step(ka, ks), mnmajor_step(d_vs[1], ks), i128, 1);
        umma_commit(&bb.b_done);
        umma_commit(&bb.empty[st]);
      }
      role_wait(&bb.epi2, ph.epi2, abort);  // the epilogue's last state hand-off
    }
    return !*abort;
  }
  if (cx.warp == 10) {
    // ------------------------------------------------ issuer of U and W (one lane)
    if (cx.lane == 0) {
      const uint64_t d_tw[2] = {kmajor_desc(smem_u32(sm.tw[0]), 8192, 0), kmajor_desc(smem_u32(sm.tw[1]), 8192, 0)};
      const uint64_t d_tu[2] = {kmajor_desc(smem_u32(sm.tu[0]), 8192, 0), kmajor_desc(smem_u32(sm.tu[1]), 8192, 0)};
      const uint64_t d_v = mnmajor_desc(smem_u32(sm.v), 8192, 0);
      const uint32_t dv = tm + kRtV;
      auto prep = [&](int j) {  // W(j): the staging of chunk j - 1 has read W (its state product has run)
        role_wait(&bb.full[j % kRecStages], ph.full[j % kRecStages], abort);
        role_wait(&bb.fullq, ph.fullq, abort);
        const uint64_t kb = d_kb0 + (uint64_t)((j % kRecStages) * (16384 >> 4));
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_bf16(tm + kRtW, kmajor_step(d_tw[0], 8192, ks), mnmajor_step(kb, ks), i64, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_bf16(tm + kRtW, kmajor_step(d_tw[1], 8192, ks), mnmajor_step(kb, ks), i64, 1);
        umma_commit(&bb.pre_done);
        umma_commit(&bb.emptyq);
      };
      auto issue_u = [&]() {  // U(j) into D_V: the V' epilogue of chunk j - 1 has read it
        role_wait(&bb.fullu, ph.fullu, abort);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_bf16(dv, kmajor_step(d_tu[0], 8192, ks), mnmajor_step(d_v, ks), i64, ks > 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) umma_bf16(dv, kmajor_step(d_tu[1], 8192, ks), mnmajor_step(d_v, ks), i64, 1);
        umma_commit(&bb.u_done);
        umma_commit(&bb.vfree);
      };
      prep(0);
      if (kWithU) issue_u();
      for (int j = 0; j < n && !*abort; ++j) {
        role_wait(&bb.a_done, ph.a_done, abort);  // the state product of chunk j has run
        if (j + 1 < n) prep(j + 1);
        role_wait(&bb.epi1, ph.epi1, abort);  // V'(j) is read: D_V is free
        if (kWithU && j + 1 < n) {
          role_wait(&bb.b_done, ph.b_done, abort);  // behind D_2 in the tensor pipe
          issue_u();
        } else {
          role_wait(&bb.b_done, ph.b_done, abort);
        }
      }
    }
    return !*abort;
  }
  // -------------------------------------------------------------------- epilogue warps 0-7
  const uint32_t lane_base = (uint32_t)(32 * cx.q4) << 16;
  // M = 64 accumulators, all 32 lanes: rows r0 = 16 q4 + lane / 4 and r0 + 8, column pairs c2 + 8k
  const int c2 = 2 * (cx.lane & 3), r0 = 16 * cx.q4 + (cx.lane >> 2);
  auto store_s_record = [&](int gc) {  // thread 0: the staged chunk-start state to its records
    bulk_store(p.st_img + rec(gc) * 32768, sm.s[0], 32768);
    bulk_store(p.st_lo_img + rec(gc) * 32768, sm.slo[0], 32768);
    bulk_commit_group();
  };
  e_handoff(cx.tid, &bb.epi2);  // S(gc0) is staged
  if (kStore && cx.tid == 0 && gc0 >= gc_rec) store_s_record(gc0);
  auto staging = [&](int j) {
    role_wait(&bb.full[j % kRecStages], ph.full[j % kRecStages], abort);
    role_wait(&bb.pre_done, ph.pre_done, abort);
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      float v[16];
      tmem_ld16x256_x4(cx.tmem + kRtW + lane_base + 64 * cx.half + 32 * hc, v);
      tmem_ld_wait();
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = 32 * hc + 8 * k + c2;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const uint32_t off = cx.half * 8192 + sw128_pair(r0 + 8 * rr, c);
          uint32_t hi, lo;
          split_pair(-v[4 * k + 2 * rr], -v[4 * k + 2 * rr + 1], hi, lo);
          *reinterpret_cast<uint32_t*>(sm.wn[0] + off) = hi;
          *reinterpret_cast<uint32_t*>(sm.wn[1] + off) = lo;
        }
      }
    }
    e_handoff(cx.tid, &bb.staged);
  };
  staging(0);
  for (int j = 0; j < n; ++j) {
    const int gc = gc0 + j, st = j % kRecStages;
    role_wait(&bb.a_done, ph.a_done, abort);
    const float* gm = sm.gam[st];
    const float gC = gm[63];
    if (kStore && cx.tid == 0) bulk_wait_read_all();  // the start-state record has read sm.s / sm.slo
    {
      // V' = D_V: its records (hi / lo) and V'_s = e^{gamma_C - gamma_t} V' (hi / lo) for K^T V'_s
      const float sc[2] = {__expf(gC - gm[r0]), __expf(gC - gm[r0 + 8])};
      const bool recj = kStore && gc >= gc_rec;
      uint8_t* vph = recj ? p.vp_img + rec(gc) * 16384 + cx.half * 8192 : nullptr;
      uint8_t* vpl = recj ? p.vp_lo_img + rec(gc) * 16384 + cx.half * 8192 : nullptr;
      const int qa = cx.lane & 3;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float v[16];
        tmem_ld16x256_x4(cx.tmem + kRtV + lane_base + 64 * cx.half + 32 * hc, v);
        tmem_ld_wait();
        uint32_t rh[2][4], rl[2][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 32 * hc + 8 * k + c2;
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const float x0 = v[4 * k + 2 * rr], x1 = v[4 * k + 2 * rr + 1];
            const uint32_t off = sw128_pair(r0 + 8 * rr, c);
            uint32_t hi, lo;
            split_pair(x0 * sc[rr], x1 * sc[rr], hi, lo);
            *reinterpret_cast<uint32_t*>(sm.vs[cx.half] + off) = hi;
            *reinterpret_cast<uint32_t*>(sm.vslo[cx.half] + off) = lo;
            if (recj) split_pair(x0, x1, rh[rr][k], rl[rr][k]);
          }
        }
        if (recj) {
          // a 4x4 transpose inside each group of four lanes leaves lane qa with the whole 16-byte
          // unit 4 hc + qa of its rows: one 16-byte store per unit instead of four 4-byte ones
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            quad_transpose4(rh[rr], qa);
            quad_transpose4(rl[rr], qa);
            const int r = r0 + 8 * rr, cj = 4 * hc + qa;
            const uint32_t off = r * 128 + ((cj ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(vph + off) = make_uint4(rh[rr][0], rh[rr][1], rh[rr][2], rh[rr][3]);
            *reinterpret_cast<uint4*>(vpl + off) = make_uint4(rl[rr][0], rl[rr][1], rl[rr][2], rl[rr][3]);
          }
        }
      }
    }
    e_handoff(cx.tid, &bb.epi1);
    if (j + 1 < n) staging(j + 1);
    role_wait(&bb.b_done, ph.b_done, abort);
    {
      const float GC = __expf(gC);
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        float v[32];
        tmem_ld16(cx.tmem + kRtD2 + lane_base + 64 * cx.half + 32 * hc, v);
        tmem_ld16(cx.tmem + kRtD2 + lane_base + 64 * cx.half + 32 * hc + 16, v + 16);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; x += 2) {  // two values per instruction
          const uint64_t r = f2_fma(f2_pack(GC, GC), f2_pack(S[32 * hc + x], S[32 * hc + x + 1]), f2_pack(v[x], v[x + 1]));
          S[32 * hc + x] = f2_lo(r);
          S[32 * hc + x + 1] = f2_hi(r);
        }
      }
      store_state_comp(sm, cx, S);
    }
    e_handoff(cx.tid, &bb.epi2, &bb.empty[st]);
    if (kStore && j + 1 < n && gc + 1 >= gc_rec && cx.tid == 0) store_s_record(gc + 1);
  }
  if (cx.tid == 0) bulk_wait_all();  // every record store has landed before the buffers are reused
  return !*abort;
}

__device__ __forceinline__ void publish(int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    st_release(flag, 1);
  }
}

// kRec: the backward's recompute (compensated arithmetic, records in the output pass); otherwise
// the forward. Both warp-specialized, 352 threads.
// The cross-segment walk borrows 192 KB of the chain's shared memory for M and the operand images
// and keeps two bytes per segment after them.
constexpr int kWalkWindow = 4096;
constexpr size_t kWalkFlagsAt = 196608;
static_assert(kWalkFlagsAt + 2 * (kWalkWindow + 64) + 1024 <= kSmemBytes, "walk buffers fit the chain's shared memory");

template <int kMode, bool kRec>
__global__ void __launch_bounds__(kWsThreads, 1) chain_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_align1024(smem_raw);
  WtSmem* wts = reinterpret_cast<WtSmem*>(base);
  RecSmem* rss = reinterpret_cast<RecSmem*>(base);
  __shared__ uint64_t bar_ld, bar_mma;
  __shared__ WsBars wbars;  // record chain
  __shared__ WtBars tbars;  // inference chain
  __shared__ uint32_t tmem_holder;
  __shared__ int s_item, s_ok, s_abort;
  griddep_launch_dependents();
  griddep_wait();  // everything the kernels before this one write
  Header* hd = ws_ptr<Header>(p, p.L.header);
  constexpr bool rec = kRec;
  ChainCtx cx;
  cx.base = base;
  cx.bar_ld = &bar_ld;
  cx.bar_mma = &bar_mma;
  cx.tid = threadIdx.x;
  cx.warp = cx.tid >> 5;
  cx.lane = cx.tid & 31;
  cx.q4 = cx.warp & 3;
  cx.half = cx.warp >> 2;
  cx.ph_ld = 0;
  cx.ph_mma = 0;
  const bool epi = cx.warp < 8;  // threads that hold state rows
  WsPhase ph;
  memset(&ph, 0, sizeof(ph));
  uint32_t tph = 0;  // phase bits of the inference chain's barriers
  const int Hv = p.d.Hv, G = p.d.Hv / p.d.Hk;
  // pass 1: one ticket per (unit, value head), then one per (walk, value head) for the walks that
  // compose a document's segment maps
  const int n_unit_items = (kMode == kModeOut ? 0 : hd->n_p1) * Hv;
  const int n_items = kMode == kModeOut ? hd->n_segs * Hv : n_unit_items + hd->n_walk * Hv;
  if (blockIdx.x >= n_items || get_status(hd) != 0) return;
  const int32_t* si = ws_ptr<int32_t>(p, p.L.seg_info);
  const int32_t* slot = ws_ptr<int32_t>(p, p.L.seg_slot);
  const int32_t* seq_seg0 = ws_ptr<int32_t>(p, p.L.seq_seg0);
  const float* gam_ws = ws_ptr<float>(p, p.L.gam);
  const int32_t* contr = ws_ptr<int32_t>(p, p.L.contr);

  // Pass 1: a unit serves the next segment's start, unless that segment warms up; the transition
  // also serves the reverse chain's publication of this segment's start gradient (record mode). A
  // walk runs for a document whose first segment starts from a known state and that has middle
  // segments. All threads call this (the window evaluation is warp-wide).
  const int32_t* p1 = ws_ptr<int32_t>(p, p.L.p1_list);
  const int32_t* walk_list = ws_ptr<int32_t>(p, p.L.walk_list);
  const int32_t* dch = ws_ptr<int32_t>(p, p.L.seq_chunk0);
  // a ticket's unit (the document's first-segment unit for a walk ticket)
  auto ticket_unit = [&](int item) {
    return item >= n_unit_items ? walk_list[(item - n_unit_items) / Hv] : item / Hv;
  };
  auto rev_needs_m = [&](int s, int part, int seq, int c0, int h) -> bool {
    return kRec && part == 0 && s != seq_seg0[seq] && warm_fwd(gam_ws, contr, Hv, h, c0, dch[seq + 1]) < 0;
  };
  // A unit records its decision per (document, value head) when it draws its ticket: a walk
  // waits for every unit of its document and has nothing to do when none computes M and B.
  int* walk_ctr = ws_ptr<int>(p, p.L.walk_ctr);
  auto p1_skips = [&](int item) -> bool {
    const bool walk = item >= n_unit_items;
    const int unit = ticket_unit(item), h = item % Hv;
    const int s = p1[2 * unit], part = p1[2 * unit + 1];
    const int seq = si[4 * s], c0 = si[4 * s + 1], nch = si[4 * s + 2];
    int* ctr = walk_ctr + 2 * ((size_t)seq * Hv + h);
    if (walk) {
      const int n_units = seq_seg0[seq + 1] - seq_seg0[seq] - 1;  // every split segment but the last
      if (part != 2 || n_units < 2) return true;
      if (cx.tid == 0) {
        const bool ok = wait_count(ctr + 1, n_units, hd, p.flag_budget);
        s_ok = (ok && __ldcg(ctr) > 0) ? 1 : 0;
      }
      __syncthreads();
      const bool skip = s_ok == 0;
      __syncthreads();
      return skip;
    }
    const bool next_warms = warm_back(gam_ws, contr, Hv, h, c0 + nch, dch[seq]) >= 0;
    const bool own_warms = part == 0 && si[4 * s + 3] >= 0 && warm_back(gam_ws, contr, Hv, h, c0, dch[seq]) >= 0;
    if (cx.tid == 0) {
      if (part == 0 && !next_warms && !own_warms) atomicAdd(ctr, 1);  // computes M and B
      __threadfence();
      atomicAdd(ctr + 1, 1);
    }
    return next_warms && !rev_needs_m(s, part, seq, c0, h);
  };
  // Pass 1 claims its tickets before it sets anything up: when every unit it draws is skipped
  // (each boundary warms up), the CTA leaves without touching tensor memory or barriers.
  int first_item = -1;
  if constexpr (kMode == kModeP1) {
    for (;;) {
      if (cx.tid == 0) {
        const int it = (int)atomicAdd(&hd->q_p1, 1u);
        s_item = (get_status(hd) != 0) ? n_items : it;
      }
      __syncthreads();
      const int item = s_item;
      if (item >= n_items) return;
      const bool skip = p1_skips(item);
      __syncthreads();  // every thread has read s_item before the next ticket
      if (!skip) {
        first_item = item;
        break;
      }
    }
  }

  if (cx.tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    if constexpr (kRec) {
      mbar_init(&wbars.full[0], 1);
      mbar_init(&wbars.full[1], 1);
      mbar_init(&wbars.full[2], 1);
      mbar_init(&wbars.fullq, 1);
      mbar_init(&wbars.fullu, 1);
      mbar_init(&wbars.empty[0], 2);
      mbar_init(&wbars.empty[1], 2);
      mbar_init(&wbars.empty[2], 2);
      mbar_init(&wbars.emptyq, 1);
      mbar_init(&wbars.a_done, 1);
      mbar_init(&wbars.pre_done, 1);
      mbar_init(&wbars.b_done, 1);
      mbar_init(&wbars.u_done, 1);
      mbar_init(&wbars.epi1, 1);
      mbar_init(&wbars.staged, 1);
      mbar_init(&wbars.epi2, 1);
      mbar_init(&wbars.vfree, 1);
    } else {
      wt_bars_init(tbars);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (cx.warp == 0) tmem_alloc(&tmem_holder, 512);
  sync_generic_to_async();
  cx.tmem = tmem_holder;

  int* flags_seg = ws_ptr<int>(p, p.L.flags_seg);
  int* flags_fin = ws_ptr<int>(p, p.L.flags_fin);
  int* flags_p1 = ws_ptr<int>(p, p.L.flags_p1);
  int* mzero = ws_ptr<int>(p, p.L.mzero);
  const size_t st_elems = (size_t)kDim * kDim;
  float S[64];
  // the record chain reads S from shared-memory images staged here; the inference chain stages
  // its tensor-memory operand itself at the start of every run
  auto store_s = [&]() {
    if constexpr (rec)
      if (epi) store_state_comp(*rss, cx, S);
  };
  auto ld_state = [&](const float* src, bool cg) {
    if constexpr (rec)
      load_state(cx, src, S, cg);
    else
      load_state_t(cx, src, S, cg);
  };
  auto sv_state = [&](float* dst) {
    if constexpr (rec)
      save_state(cx, dst, S);
    else
      save_state_t(cx, dst, S);
  };
  auto set_zero = [&]() {
    for (int c = 0; c < 64; ++c) S[c] = 0.f;
  };
  auto set_identity = [&]() {
    // row-block layout (record chain): thread row a = 32 q4 + lane; transposed: column b = 32 q4 + lane
    const int r = 32 * cx.q4 + cx.lane;
    for (int c = 0; c < 64; ++c) S[c] = (r == 64 * cx.half + c) ? 1.f : 0.f;
  };
  auto all_zero = [&]() -> bool {
    bool mine = true;
    if (epi)
      for (int x = 0; x < 64; ++x) mine = mine && (S[x] == 0.f);
    return __syncthreads_and(mine) != 0;
  };
  // chain over [g0, g1): outputs from g_out (forward), records from g_out (recompute)
  auto run_fast = [&](int g0, int g1, int g_out, int h, int hk, bool with_u) -> bool {
    if constexpr (rec) {
      if (!with_u) {
        run_ws_rec<false, false>(p, cx, wbars, ph, &s_abort, S, g0, g1, h, hk, g1);
      } else {
        // records from g_out on; the chunks before (a warm-up) run without the record path
        const int gm = g_out < g0 ? g0 : (g_out > g1 ? g1 : g_out);
        if (gm > g0) run_ws_rec<true, false>(p, cx, wbars, ph, &s_abort, S, g0, gm, h, hk, gm);
        if (gm > g0 && g1 > gm) __syncthreads();
        if (g1 > gm && s_abort == 0) run_ws_rec<true, true>(p, cx, wbars, ph, &s_abort, S, gm, g1, h, hk, gm);
      }
    } else {
      if (with_u)
        run_wt<true>(p, cx, tbars, tph, &s_abort, S, g0, g1, g_out, h, hk);
      else
        run_wt<false>(p, cx, tbars, tph, &s_abort, S, g0, g1, g_out, h, hk);
    }
    __syncthreads();
    return s_abort == 0;
  };
  auto affine = [&](const float* Mm, const float* Bm, float* out) -> bool {
    if constexpr (rec)
      return affine_apply<false>(p, cx, affine_bufs(*rss), Mm, Bm, S, out, kRtV);
    else
      return affine_apply<true>(p, cx, affine_bufs(*wts), Mm, Bm, S, out, kTtD2);
  };

  // wait (uniform outcome) for a publication flag
  auto wait_uniform = [&](const int* flag) -> bool {
    if (cx.tid == 0) {
      s_ok = wait_flag(flag, hd, p.flag_budget) ? 1 : 0;
      __threadfence();
    }
    __syncthreads();
    const bool r = s_ok != 0;
    __syncthreads();
    return r;
  };
  // Cross-segment fix-up of one document and value head (pass 1, after the units it reads): the
  // end state of every middle segment whose successor does not warm up and whose own start does
  // not warm up (those publish their own), in segment order: E_s = M_s E_{s-1} + B_s, or E_s = B_s
  // for an exactly zero transition. Each is published as soon as it is written (its flag after
  // the next product is issued), so no output item waits on another output item.
  // E is held transposed (thread: column b = 32 q4 + lane, rows a = 64 half + c) and the product
  // runs as E^T M^T on the tensor cores with compensated bf16 operands; the units stored M's
  // operand images, and they and B arrive by bulk copies while the previous step finishes.
  // Which segment starts warm up, the units' flags and their zero findings are read up front,
  // kWalkWindow segments at a time.
  auto walk_document = [&](int s0, int seq, int h) -> bool {
    float* pub = ws_ptr<float>(p, p.L.pub);
    float* bmat = ws_ptr<float>(p, p.L.bmat);
    const uint8_t* mimg = ws_ptr<uint8_t>(p, p.L.mimg);
    auto at = [&](float* b, int s) { return b + ((size_t)slot[s] * Hv + h) * st_elems; };
    float* bf = reinterpret_cast<float*>(base);  // B fp32 (bulk copy)
    uint8_t* mhi = base + 65536;                 // M hi / lo images (bulk copy, 64 KB)
    uint8_t* mlo = base + 98304;
    uint8_t* ehi = base + 131072;                // E^T hi / lo images, K-major rows b
    uint8_t* warms = base + kWalkFlagsAt;        // warms[s - w0]: segment s starts with a warm-up
    uint8_t* mz = warms + kWalkWindow + 64;      // mz[s - w0]: M_s is exactly zero
    const uint32_t dcol = kRec ? kRtV : kTtD2;
    // B = M^T: MN-major images from the transposed chain's layout, K-major from the record chain's
    const uint32_t id = idesc_bf16(128, 128, 0, kRec ? 0 : 1);
    auto mdesc = [&](const uint8_t* img, int ks) {
      return kRec ? kmajor_step(kmajor_desc(smem_u32(img), 16384, 0), 16384, ks)
                  : mnmajor_step(mnmajor_desc(smem_u32(img), 16384, 0), ks);
    };
    const int s_last = seq_seg0[seq + 1] - 1;  // its end state is the final state
    const int b = 32 * cx.q4 + cx.lane;
    bool have = false;     // E_{s-1} is in S
    bool inflight = false; // bulk copies into bf / mhi are in flight
    int pend = -1;         // segment whose end state is written but not yet flagged
    auto bail = [&]() -> bool {
      if (inflight) wait_all(cx.bar_ld, cx.ph_ld);  // (the copies land before the walk gives up)
      return false;
    };
    auto fetch = [&](int s) {  // M_s images and B_s into shared memory
      if (cx.tid == 0) {
        fence_proxy_async_global();  // (written through the generic proxy by the units)
        mbar_arrive_expect_tx(cx.bar_ld, 131072);
        bulk_load(mhi, mimg + ((size_t)slot[s] * Hv + h) * 65536, 65536, cx.bar_ld);
        bulk_load(bf, at(bmat, s), 65536, cx.bar_ld);
      }
      inflight = true;
    };
    for (int w0 = s0 + 1; w0 < s_last; w0 += kWalkWindow) {
      const int w1 = min(w0 + kWalkWindow, s_last);
      for (int s = w0 + cx.warp; s <= w1; s += kWsThreads / 32) {  // (warp-uniform)
        const bool wv = warm_back(gam_ws, contr, Hv, h, si[4 * s + 1], dch[seq]) >= 0;
        if (cx.lane == 0) warms[s - w0] = wv ? 1 : 0;
      }
      __syncthreads();
      auto computed = [&](int s) { return !warms[s - w0] && !warms[s - w0 + 1]; };
      bool fail = false;
      for (int s = w0 + cx.tid; s < w1; s += kWsThreads) {
        if (!computed(s)) continue;
        if (!wait_flag(&flags_p1[slot[s] * Hv + h], hd, p.flag_budget)) {
          fail = true;
          break;
        }
        mz[s - w0] = __ldcg(&mzero[slot[s] * Hv + h]) ? 1 : 0;
      }
      if (__syncthreads_or(fail)) return bail();
      auto next_m = [&](int from) {  // the next segment whose step runs the product
        while (from < w1 && !(computed(from) && !mz[from - w0])) ++from;
        return from;
      };
      if (next_m(w0) < w1) fetch(next_m(w0));
      for (int s = w0; s < w1; ++s) {
        if (!computed(s)) {
          if (pend >= 0) publish(&flags_seg[pend * Hv + h]);
          pend = -1;
          have = false;
          continue;
        }
        if (mz[s - w0]) {
          if (epi) load_state_t(cx, at(bmat, s), S, true);
        } else {
          if (!have) {  // published by its own unit (a known start or a warm-up)
            if (!wait_uniform(&flags_seg[(s - 1) * Hv + h])) return bail();
            if (epi) load_state_t(cx, at(pub, s - 1), S, true);
          }
          if (epi) {  // E^T hi / lo, K-major (row b, 64 values of a per block)
            uint8_t* eh = ehi + cx.half * 16384;
#pragma unroll
            for (int cj = 0; cj < 8; ++cj) {
              float lo[8];
#pragma unroll
              for (int u = 0; u < 8; ++u)
                lo[u] = S[8 * cj + u] - __bfloat162float(__float2bfloat16_rn(S[8 * cj + u]));
              const uint32_t off = b * 128 + ((cj ^ (b & 7)) << 4);
              *reinterpret_cast<uint4*>(eh + off) =
                  make_uint4(pack_bf16x2(S[8 * cj], S[8 * cj + 1]), pack_bf16x2(S[8 * cj + 2], S[8 * cj + 3]),
                             pack_bf16x2(S[8 * cj + 4], S[8 * cj + 5]), pack_bf16x2(S[8 * cj + 6], S[8 * cj + 7]));
              *reinterpret_cast<uint4*>(eh + 32768 + off) = make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                                                                       pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
            }
          }
          if (!wait_all(cx.bar_ld, cx.ph_ld)) return false;  // M_s and B_s have landed
          cx.ph_ld ^= 1;
          inflight = false;
          sync_generic_to_async();
          if (cx.tid == 0) {
            const uint64_t ah0 = kmajor_desc(smem_u32(ehi), 16384, 0);
            const uint64_t al0 = kmajor_desc(smem_u32(ehi + 32768), 16384, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_bf16(cx.tmem + dcol, kmajor_step(ah0, 16384, ks), mdesc(mhi, ks), id, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_bf16(cx.tmem + dcol, kmajor_step(al0, 16384, ks), mdesc(mhi, ks), id, 1);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_bf16(cx.tmem + dcol, kmajor_step(ah0, 16384, ks), mdesc(mlo, ks), id, 1);
            umma_commit(cx.bar_mma);
          }
          if (pend >= 0 && cx.tid == kWsThreads - 32) {  // (a thread outside the epilogue)
            // the previous end state was stored before the barrier above
            __threadfence();
            st_release(&flags_seg[pend * Hv + h], 1);
          }
          pend = -1;
          if (!wait_all(cx.bar_mma, cx.ph_mma)) return bail();
          cx.ph_mma ^= 1;
          tc_fence_after();
          if (epi) {
            const uint32_t lane_base = (uint32_t)(32 * cx.q4) << 16;
#pragma unroll
            for (int hc = 0; hc < 4; ++hc) {
              float d[16];
              tmem_ld16(cx.tmem + dcol + lane_base + 64 * cx.half + 16 * hc, d);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j) S[16 * hc + j] = d[j] + bf[(64 * cx.half + 16 * hc + j) * kDim + b];
            }
          }
          tc_fence_before();
          __syncthreads();  // bf and the images are consumed
          const int sf = next_m(s + 1);
          if (sf < w1) fetch(sf);
        }
        if (pend >= 0) publish(&flags_seg[pend * Hv + h]);
        if (epi) save_state_t(cx, at(pub, s), S);
        pend = s;
        have = true;
      }
      __syncthreads();  // (the next window's flags overwrite these)
    }
    if (pend >= 0) publish(&flags_seg[pend * Hv + h]);
    return true;
  };

  for (;;) {
    if (first_item < 0 && cx.tid == 0) {
      const int it = (int)atomicAdd(kMode == kModeOut ? &hd->q_chain : &hd->q_p1, 1u);
      s_item = (get_status(hd) != 0) ? n_items : it;
    }
    __syncthreads();
    const int item = first_item >= 0 ? first_item : s_item;
    first_item = -1;
    if (item >= n_items) break;
    const int h = item % Hv, hk = h / G;
    bool ok = true;
    if (kMode == kModeP1) {
      const bool walk = item >= n_unit_items;
      const int unit = ticket_unit(item);
      const int s = p1[2 * unit], part = p1[2 * unit + 1];
      const int seq = si[4 * s], c0 = si[4 * s + 1], nch = si[4 * s + 2];
      const int sl = slot[s];
      if (p1_skips(item)) {
        __syncthreads();  // every thread has read s_item before the next ticket
        continue;
      }
      if (walk) {
        if (!walk_document(s, seq, h)) {
          set_status(hd, kErrTimeout);
          break;
        }
        __syncthreads();
        continue;
      }
      // the next segment needs this segment's end state (it does not warm up)
      const bool need_e = warm_back(gam_ws, contr, Hv, h, c0 + nch, dch[seq]) < 0;
      if (part == 2) {
        // the end state from the document's known start, published directly
        const int x = p.init_idx ? p.init_idx[seq] : -1;
        if (epi && x >= 0 && x < p.d.n_init)
          ld_state(p.initial_state + ((size_t)x * Hv + h) * st_elems, false);
        else
          set_zero();
        store_s();
        sync_generic_to_async();
        if (!run_fast(c0, c0 + nch, c0 + nch, h, hk, true)) break;
        if (epi) sv_state(ws_ptr<float>(p, p.L.pub) + ((size_t)sl * Hv + h) * st_elems);
        publish(&flags_seg[s * Hv + h]);
        __syncthreads();
        continue;
      }
      // a segment whose own start warms up has its end state directly (from zero at the warm-up
      // chunk); otherwise its transition M and its end state B from zero, for the walk
      const int wb = si[4 * s + 3] >= 0 ? warm_back(gam_ws, contr, Hv, h, c0, dch[seq]) : -1;
      const bool direct = need_e && wb >= 0;
      const bool want_b = need_e && !direct;
      const bool want_m = want_b || rev_needs_m(s, part, seq, c0, h);
      if (direct) {
        set_zero();
        store_s();
        sync_generic_to_async();
        if (!run_fast(wb, c0 + nch, c0 + nch, h, hk, true)) break;
        if (epi) sv_state(ws_ptr<float>(p, p.L.pub) + ((size_t)sl * Hv + h) * st_elems);
        publish(&flags_seg[s * Hv + h]);
      }
      float* mdst = ws_ptr<float>(p, p.L.mmat) + ((size_t)sl * Hv + h) * st_elems;
      bool m_zero = false;
      if (want_m) {
        // Transition M = Phi_last ... Phi_first: the chain from I over the segment. An exactly
        // zero M makes the segment's end state its local end state B, and the next segment can
        // start without waiting for this segment's start state.
        set_identity();
        store_s();
        sync_generic_to_async();
        if (!run_fast(c0, c0 + nch, c0 + nch, h, hk, false)) break;
        m_zero = all_zero();
        if (epi) {
          sv_state(mdst);
          store_images(cx, ws_ptr<uint8_t>(p, p.L.mimg) + ((size_t)sl * Hv + h) * 65536, S);
        }
        if (m_zero && cx.tid == 0) mzero[sl * Hv + h] = 1;
      }
      if (want_b) {
        set_zero();
        store_s();
        sync_generic_to_async();
        if (!run_fast(c0, c0 + nch, c0 + nch, h, hk, true)) break;
        if (epi) sv_state(ws_ptr<float>(p, p.L.bmat) + ((size_t)sl * Hv + h) * st_elems);
        publish(&flags_p1[sl * Hv + h]);  // M and B of this segment are written
      }
      __syncthreads();
      continue;
    }

    // ---------------------------------------------------------------- output pass
    const int s = item / Hv;
    const int seq = si[4 * s], c0 = si[4 * s + 1], nch = si[4 * s + 2], dep = si[4 * s + 3];
    const bool last = (s + 1 == seq_seg0[seq + 1]);
    int first_chunk = c0;  // a warm-up may start earlier
    bool have_start = true;
    // exact split: this segment warms up instead of waiting, and the next one needs this item's
    // published end state only when it cannot warm up itself
    const int wb = (p.d.mode == 0 && dep >= 0) ? warm_back(gam_ws, contr, Hv, h, c0, dch[seq]) : -1;
    // (pass 1 has published it already when the document starts from a known state or when this
    // segment warms up)
    const bool pub_next = p.d.mode == 0 && slot[s] >= 0 && wb < 0 && si[4 * seq_seg0[seq] + 3] <= -2 &&
                          warm_back(gam_ws, contr, Hv, h, c0 + nch, dch[seq]) < 0;
    if (pub_next) {  // this item publishes its end state early
      const size_t off = ((size_t)slot[s] * Hv + h) * st_elems;
      prefetch_state_l2(ws_ptr<float>(p, p.L.mmat) + off, cx.tid, blockDim.x);
      prefetch_state_l2(ws_ptr<float>(p, p.L.bmat) + off, cx.tid, blockDim.x);
    }
    if (dep == -1) {
      const int x = p.init_idx ? p.init_idx[seq] : -1;
      if (epi && x >= 0 && x < p.d.n_init)
        ld_state(p.initial_state + ((size_t)x * Hv + h) * st_elems, false);
      else
        set_zero();
    } else if (dep <= -2) {
      const int j = dep_fork_seq(dep);
      if (cx.tid == 0) {
        s_ok = wait_flag(&flags_fin[j * Hv + h], hd, p.flag_budget) ? 1 : 0;
        __threadfence();
      }
      __syncthreads();
      have_start = s_ok != 0;
      if (have_start && epi) ld_state(p.final_state + ((size_t)j * Hv + h) * st_elems, true);
    } else if (p.d.mode == 0) {
      const int dsl = slot[dep];
      if (wb >= 0) {
        // the decay since chunk wb leaves the earlier state below fp32 resolution: warm up from zero
        first_chunk = wb;
        set_zero();
      } else if (__ldcg(&mzero[dsl * Hv + h])) {
        // the previous segment's transition is exactly zero: its end state is its local B
        if (epi) ld_state(ws_ptr<float>(p, p.L.bmat) + ((size_t)dsl * Hv + h) * st_elems, true);
      } else {
        if (cx.tid == 0) {
          s_ok = wait_flag(&flags_seg[dep * Hv + h], hd, p.flag_budget) ? 1 : 0;
          __threadfence();
        }
        __syncthreads();
        have_start = s_ok != 0;
        if (have_start && epi)
          ld_state(ws_ptr<float>(p, p.L.pub) + ((size_t)dsl * Hv + h) * st_elems, true);
      }
    } else {
      // truncation: fewest preceding whole chunks of this document whose summed log-decay is
      // below the threshold; from zero, or from the document's start state if the window reaches it
      const float* gam = ws_ptr<float>(p, p.L.gam);
      const int doc_c0 = ws_ptr<int32_t>(p, p.L.seq_chunk0)[seq];
      int w = c0;
      float acc = 0.f;
      while (w > doc_c0 && acc >= p.trunc_thr) {
        --w;
        acc += gam[((size_t)w * Hv + h) * 64 + 63];
      }
      first_chunk = w;
      set_zero();
      if (w == doc_c0 && acc >= p.trunc_thr) {
        const int s0 = seq_seg0[seq];
        const int d0 = si[4 * s0 + 3];
        if (d0 == -1) {
          const int x = p.init_idx ? p.init_idx[seq] : -1;
          if (epi && x >= 0 && x < p.d.n_init)
            ld_state(p.initial_state + ((size_t)x * Hv + h) * st_elems, false);
        } else {
          const int j = dep_fork_seq(d0);
          if (cx.tid == 0) {
            s_ok = wait_flag(&flags_fin[j * Hv + h], hd, p.flag_budget) ? 1 : 0;
            __threadfence();
          }
          __syncthreads();
          have_start = s_ok != 0;
          if (have_start && epi) ld_state(p.final_state + ((size_t)j * Hv + h) * st_elems, true);
        }
      }
    }
    if (!have_start) break;
    store_s();
    sync_generic_to_async();
    const bool publishes = pub_next && !__ldcg(&mzero[slot[s] * Hv + h]);
    if (publishes && first_chunk < c0) {
      // the publication below needs the state at the segment start: warm up first
      if (!run_fast(first_chunk, c0, c0, h, hk, true)) {
        set_status(hd, kErrTimeout);
        break;
      }
      first_chunk = c0;
    }
    // early publication of this segment's end state (exact split), unless its transition is zero
    if (publishes) {
      const size_t off = ((size_t)slot[s] * Hv + h) * st_elems;
      if (!affine(ws_ptr<float>(p, p.L.mmat) + off, ws_ptr<float>(p, p.L.bmat) + off, ws_ptr<float>(p, p.L.pub) + off)) {
        set_status(hd, kErrTimeout);
        break;
      }
      publish(&flags_seg[s * Hv + h]);
      store_s();  // affine_apply used the staging buffers
      sync_generic_to_async();
    }
    ok = run_fast(first_chunk, c0 + nch, c0, h, hk, true);
    if (!ok) {
      set_status(hd, kErrTimeout);
      break;
    }
    if (last) {
      if (epi) sv_state(p.final_state + ((size_t)seq * Hv + h) * st_elems);
      if (!p.withhold_fin)
        publish(&flags_fin[seq * Hv + h]);
      else
        __syncthreads();
    }
    __syncthreads();
  }
  if (s_abort && cx.tid == 0) set_status(hd, kErrTimeout);
  // drain: make sure no MMA is in flight before releasing tensor memory
  if (cx.tid == 0) {
    umma_commit(&bar_mma);
    mbar_wait(&bar_mma, cx.ph_mma, kWaitBudget);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (cx.warp == 0) tmem_dealloc(cx.tmem, 512);
}

// ================================================================================ output from records
//
// o of one chunk and value head from the recompute's records (the forward of a training step):
// O = diag(scale e^gamma) Q S + P V', with S the chunk-start state and V' = U - W S (bf16 hi images
// written by the record chain) and P = scale (Q K^T o E) (bf16 image from kkt_solve). One CTA of
// 128 threads per (chunk, value head): TMA and bulk loads on one barrier, Q~ formed in place, one
// M = 64 accumulator, O staged over Q~ and written by TMA store (a partial chunk row by row).
struct OutSmem {
  uint8_t q[2][8192];   // Q rows t, two dk blocks -> Q~ in place (A K-major, M = 64); then the O stage
  uint8_t s[2][16384];  // S hi rows dk, two dv blocks (B MN-major)
  uint8_t vp[2][8192];  // V' hi rows t, two dv blocks (B MN-major)
  uint8_t p[8192];      // P rows t (A K-major, M = 64, K = 64)
  float gam[64];
};
constexpr int kOutThreads = 128;
constexpr size_t kOutSmemBytes = sizeof(OutSmem) + 1024;

__global__ void __launch_bounds__(kOutThreads) out_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  OutSmem& sm = *reinterpret_cast<OutSmem*>(smem_align1024(smem_raw));
  __shared__ uint64_t bar_ld, bar_mma;
  __shared__ uint32_t tmem_holder;
  griddep_launch_dependents();
  griddep_wait();  // the records of the chain before it
  Header* hd = ws_ptr<Header>(p, p.L.header);
  const int gc = blockIdx.x, h = blockIdx.y, Hv = p.d.Hv, hk = h / (Hv / p.d.Hk);
  if (gc >= hd->n_chunks || get_status(hd) != 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tok0 = ws_ptr<int32_t>(p, p.L.chunk_tok0)[gc], nn = ws_ptr<int32_t>(p, p.L.chunk_len)[gc];
  const size_t rec = (size_t)gc * Hv + h;
  if (tid == 0) {
    mbar_init(&bar_ld, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&bar_ld, 16384 + 32768 + 16384 + 8192 + 256);
    tma_load_3d(sm.q[0], &p.tm_q, 0, hk, tok0, &bar_ld);
    tma_load_3d(sm.q[1], &p.tm_q, 64, hk, tok0, &bar_ld);
    bulk_load(sm.s[0], p.st_img + rec * 32768, 32768, &bar_ld);
    bulk_load(sm.vp[0], p.vp_img + rec * 16384, 16384, &bar_ld);
    bulk_load(sm.p, p.p_img + rec * 8192, 8192, &bar_ld);
    bulk_load(sm.gam, p.ws + p.L.gam + rec * 256, 256, &bar_ld);
  }
  if (warp == 0) tmem_alloc(&tmem_holder, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_holder;
  bool ok = wait_all(&bar_ld, 0);
  if (ok) {
    // Q~ = diag(scale e^gamma) Q, in place
    for (int e = tid; e < 2 * 64 * 8; e += kOutThreads) {
      const int b = e >> 9, r = (e >> 3) & 63, cj = e & 7;
      const uint32_t off = r * 128 + ((cj ^ (r & 7)) << 4);
      uint4 raw = *reinterpret_cast<const uint4*>(sm.q[b] + off);
      const float sc = __expf(sm.gam[r]) * p.scale;
      __nv_bfloat162* x = reinterpret_cast<__nv_bfloat162*>(&raw);
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 f = __bfloat1622float2(x[u]);
        w[u] = pack_bf16x2(f.x * sc, f.y * sc);
      }
      *reinterpret_cast<uint4*>(sm.q[b] + off) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    sync_generic_to_async();
    if (tid == 0) {
      constexpr uint32_t i64 = idesc_bf16(64, 128, 0, 1);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        umma_bf16(tm, kmajor_step(kmajor_desc(smem_u32(sm.q[0]), 8192, 0), 8192, ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.s[0]), 16384, 0), ks), i64,
                  ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        umma_bf16(tm, kmajor_step(kmajor_desc(smem_u32(sm.p), 8192, 0), 8192, ks),
                  mnmajor_step(mnmajor_desc(smem_u32(sm.vp[0]), 8192, 0), ks), i64, 1);
      umma_commit(&bar_mma);
    }
    ok = wait_all(&bar_mma, 0);
  }
  if (ok) {
    tc_fence_after();
    // M = 64 accumulator, all 32 lanes: rows r0 = 16 warp + lane / 4 and r0 + 8, column pairs
    const int c2 = 2 * (lane & 3), r0 = 16 * warp + (lane >> 2);
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
      float v[16];
      tmem_ld16x256_x4(tm + lane_base + 32 * cb, v);
      tmem_ld_wait();
      uint8_t* blk = sm.q[cb >> 1];  // dv block (the MMA has finished reading Q~)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = 32 * (cb & 1) + 8 * k + c2;
        *reinterpret_cast<uint32_t*>(blk + sw128_pair(r0, c)) = pack_bf16x2(v[4 * k], v[4 * k + 1]);
        *reinterpret_cast<uint32_t*>(blk + sw128_pair(r0 + 8, c)) = pack_bf16x2(v[4 * k + 2], v[4 * k + 3]);
      }
    }
    if (nn == kChunk) {
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tma_store_3d(&p.tm_o, sm.q[0], 0, h, tok0);
        tma_store_3d(&p.tm_o, sm.q[1], 64, h, tok0);
        bulk_commit_group();
        bulk_wait_all();
      }
    } else {
      // the end of a document: only its rows, so that the next document's rows are not touched
      __syncthreads();
      for (int e = tid; e < nn * 16; e += kOutThreads) {
        const int t = e >> 4, u = e & 15, cj = u & 7;
        const uint4 val = *reinterpret_cast<const uint4*>(sm.q[u >> 3] + t * 128 + ((cj ^ (t & 7)) << 4));
        reinterpret_cast<uint4*>(p.out + ((size_t)(tok0 + t) * Hv + h) * kDim)[u] = val;
      }
    }
  } else if (tid == 0) {
    set_status(hd, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tm, 128);
}

// ========================================================================================= launch

int launch_fwd(const FwdParams& p, cudaStream_t stream, cudaEvent_t* ev, bool plan_only) {
  static PerDevice attr_done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kErrCuda;
  if (!attr_done.done(dev)) {
    if (cudaFuncSetAttribute(kkt_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(sizeof(KktSmem) + 1024)) != cudaSuccess)
      return kErrCuda;
    if (cudaFuncSetAttribute(chain_kernel<kModeOut, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(chain_kernel<kModeP1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(chain_kernel<kModeOut, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(chain_kernel<kModeP1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutSmemBytes) !=
            cudaSuccess)
      return kErrCuda;
    attr_done.mark(dev);
  }
  auto mark = [&](int i) {
    if (ev && ev[i]) cudaEventRecord(ev[i], stream);
  };
  mark(0);
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(p, plan_only ? 1 : 0);
  mark(1);
  if (plan_only) {
    for (int i = 2; i < 8; ++i) mark(i);
    mark(16);
    mark(17);
    return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
  }
  mark(2);
  if (p.d.T > 0) {
    dim3 grid((unsigned)p.L.cmax, (unsigned)p.d.Hk);
    launch_early(kkt_solve_kernel, grid, 256, sizeof(KktSmem) + 1024, stream, p);
  }
  mark(3);
  const int64_t items_cap = (int64_t)p.d.num_sms;
  mark(4);
  if (p.d.mode == 0 && p.L.slots > 0 && p.d.T > 0) {
    const int64_t units = 2 * p.L.slots * p.d.Hv;  // units and walks (at most one per unit)
    const int grid = (int)(units < items_cap ? units : items_cap);
    if (p.st_img)
      launch_early(chain_kernel<kModeP1, true>, grid, kWsThreads, kSmemBytes, stream, p);
    else
      launch_early(chain_kernel<kModeP1, false>, grid, kWsThreads, kSmemBytes, stream, p);
  }
  mark(5);
  mark(6);
  {
    const int64_t items = p.L.smax * p.d.Hv;
    const int grid = (int)(items < items_cap ? items : items_cap);
    if (p.st_img)
      launch_early(chain_kernel<kModeOut, true>, grid, kWsThreads, kSmemBytes, stream, p);
    else
      launch_early(chain_kernel<kModeOut, false>, grid, kWsThreads, kSmemBytes, stream, p);
  }
  mark(7);
  // a forward that keeps its records for the backward forms o from them
  mark(16);
  if (p.st_img && p.out && p.d.T > 0)
    launch_early(out_kernel, dim3((unsigned)p.L.cmax, (unsigned)p.d.Hv), kOutThreads, kOutSmemBytes, stream, p);
  mark(17);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace gdn
