// Backward path: argument block, workspace layout and launcher.
#pragma once
#include <cuda_runtime.h>

#include "gdn_common.cuh"

namespace gdn {

struct BwdArgs {
  const void *q, *k, *v;
  const float *g, *beta;
  const int32_t *cu, *init_idx;
  const float* initial_state;
  const void* dout;
  const float* dfinal;
  void *dq, *dk, *dv;
  float *dg, *dbeta, *dinit;
  void* ws;
  size_t ws_bytes;
  PlanDims d;
  float trunc_thr, scale;
};

struct BwdLayout {
  size_t total;
};

inline BwdLayout bwd_layout(const PlanDims& d) {
  BwdLayout L;
  L.total = fwd_layout(d).total;
  return L;
}

int launch_bwd(const BwdArgs& a, cudaStream_t stream, cudaEvent_t* events);

}  // namespace gdn
