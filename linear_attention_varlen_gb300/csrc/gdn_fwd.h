// Kernel parameter block of the forward path and its launcher.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_common.cuh"

namespace gdn {

struct FwdParams {
  CUtensorMap tm_q;  // bf16 [T][Hk][128], box 64 x 1 x 64, 128B swizzle
  CUtensorMap tm_k;  // same shape as q
  CUtensorMap tm_v;  // bf16 [T][Hv][128]
  CUtensorMap tm_o;  // the output, same shape as v (forwards that write o)
  const float* g;
  const float* beta;
  const int32_t* cu;
  const int32_t* init_idx;
  const float* initial_state;
  __nv_bfloat16* out;
  float* final_state;
  uint8_t* ws;
  PlanDims d;
  FwdLayout L;
  float trunc_thr;
  float scale;
  long long flag_budget;  // limit of a wait on another item's publication flag, SM clock cycles
  int withhold_fin;       // test hook: final states are never published to forked documents
  // P = scale (Q K^T o E) per (chunk, value head), E_ij = e^{gamma_i - gamma_j} for j <= i inside
  // the chunk, bf16 smem image [cmax][Hv][8 KB], formed by kkt_solve
  uint8_t* p_img;
  // 1: kkt_solve writes P in the factored form the inference chain uses (row factor scale e^{gamma_i}
  // taken out: P''_ij = (Q K^T)_ij e^{-gamma_j}; see kkt_solve); 0: P itself (the record paths)
  int p_factored;
  // Recording forward only (the backward's recompute, or a forward that keeps its records for the
  // backward; all NULL for a plain forward): per (chunk, value head) records. With `out` set, o is
  // formed from them after the chain.
  uint8_t* st_img;  // S at each chunk start, bf16, 128B-swizzled smem image [cmax][Hv][32 KB]
  uint8_t* vp_img;  // V' = U - W S of each chunk, bf16 smem image [cmax][Hv][16 KB]
  float* t_f32;     // T = (I + A)^{-1}, fp32 [cmax][Hv][64 x 64] in the fz layout
  // Compensated bf16 (x = hi + lo, both bf16) for the backward recompute: the low parts of
  // T diag(beta e^gamma) and T diag(beta) (written by kkt_solve, read by the chain), and of
  // S and V' (written by the chain for the gradient kernels).
  uint8_t* tw_lo;      // [cmax][Hv][8 KB]
  uint8_t* tu_lo;      // [cmax][Hv][8 KB]
  uint8_t* st_lo_img;  // [cmax][Hv][32 KB]
  uint8_t* vp_lo_img;  // [cmax][Hv][16 KB]
};

// events: NULL or cudaEvent_t[2 * 9], recorded around each stage (see gdn_fwd_stage).
// plan_only: the chunk and segment maps only (a backward that reuses a forward's records).
int launch_fwd(const FwdParams& p, cudaStream_t stream, cudaEvent_t* events, bool plan_only = false);

}  // namespace gdn
