// Backward path: argument block, workspace layout and launcher.
#pragma once
#include <cuda.h>
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
  long long flag_budget;  // limit of a wait on another item's publication flag, SM clock cycles
  int withhold_fin;       // forward of a training step: test hook of gdn_chunk_fwd
};

// Backward workspace: the forward recompute's workspace first, then the per-chunk records.
struct BwdLayout {
  FwdLayout f;
  size_t st_img;    // S at each chunk start, bf16 image [cmax][Hv][32 KB]
  size_t vp_img;    // V' per chunk, bf16 image [cmax][Hv][16 KB]
  size_t t_f32;     // T per chunk, fp32 [cmax][Hv][64 x 64] in the fz layout
  size_t ds_img;    // dL/dS at each chunk end, bf16 image [cmax][Hv][32 KB]
  size_t dvp_img;   // dL/dV' per chunk, bf16 image [cmax][Hv][16 KB]
  size_t tw_lo, tu_lo;    // low parts of the WY factors, bf16 images [cmax][Hv][8 KB]
  size_t st_lo, vp_lo;    // low parts of S and V', bf16 images [cmax][Hv][32 KB / 16 KB]
  size_t fin;       // final states of the recompute, fp32 [N][Hv][128][128]
  size_t ds0;       // dL/dS at each document start, fp32 [N][Hv][128][128]
  size_t flags_ds0; // int32 [N][Hv]
  size_t rpub;      // reverse split: dL/dS at the start of segment s, published at slot[s-1], fp32
  size_t rb;        // reverse split: dL/dS at the start of segment s from a zero end gradient, at slot[s]
  size_t flags_rseg;// int32 [smax][Hv]: rpub of segment s is ready
  size_t hdr2;      // Header of the reverse pass (queue, status mirror)
  size_t total;
};

inline BwdLayout bwd_layout(const PlanDims& d) {
  BwdLayout L;
  L.f = fwd_layout(d);
  size_t o = L.f.total;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t ch = (size_t)L.f.cmax * d.Hv;
  const size_t state = (size_t)kDim * kDim * 4;
  L.st_img = take(ch * 32768);
  L.vp_img = take(ch * 16384);
  L.t_f32 = take(ch * 16384);
  L.ds_img = take(ch * 32768);
  L.dvp_img = take(ch * 16384);
  L.tw_lo = take(ch * 8192);
  L.tu_lo = take(ch * 8192);
  L.st_lo = take(ch * 32768);
  L.vp_lo = take(ch * 16384);
  L.fin = take((size_t)d.N * d.Hv * state);
  L.ds0 = take((size_t)d.N * d.Hv * state);
  L.flags_ds0 = take((size_t)d.N * d.Hv * 4);
  L.rpub = take((size_t)L.f.slots * d.Hv * state);
  L.rb = take((size_t)L.f.slots * d.Hv * state);
  L.flags_rseg = take((size_t)L.f.smax * d.Hv * 4);
  L.hdr2 = take(sizeof(Header));
  L.total = o;
  return L;
}

// reuse: the workspace holds the records of a forward launched with launch_fwd_save on the same
// inputs; only the maps are rebuilt.
int launch_bwd(const BwdArgs& a, bool reuse, cudaStream_t stream, cudaEvent_t* events);
// Forward (o and final states) that leaves its records in a backward workspace for launch_bwd.
int launch_fwd_save(const BwdArgs& a, void* out, float* final_state, cudaStream_t stream, cudaEvent_t* events);

}  // namespace gdn
