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
};

// events: NULL or cudaEvent_t[2 * 8], recorded around each stage (see gdn_fwd_stage).
int launch_fwd(const FwdParams& p, cudaStream_t stream, cudaEvent_t* events);

}  // namespace gdn
