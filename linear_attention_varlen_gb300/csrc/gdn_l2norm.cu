// L2 normalisation of q and k per (token, key head), and its backward, for callers that hand the
// library unnormalised queries and keys (GDN_FLAG_L2NORM_QK). The recurrence expects unit-norm q
// and k ("Musings on long-context fine-tuning", section "Triton autotuning in the first backward
// pass": the model normalises q and k before the GDN op, and the separate normalisation backward
// with its length-keyed autotuning was what ran out of memory; here both directions are one plain
// pass each, with no tuning and no allocation).
//
//   forward : y = x r,  r = (x . x + eps)^{-1/2}   (fp32, y rounded once to bf16)
//   backward: dx = r (dy - (y . dy) y)             (y recomputed in fp32 from x)
// One warp per row of 128 elements (4 per lane); q and k rows in one launch.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gdn_common.cuh"
#include "gdn_l2norm.h"

namespace gdn {
namespace {

constexpr int kNormThreads = 256;  // 8 rows per CTA

__device__ __forceinline__ float warp_sum32(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// rows [0, rows) of q then rows [rows, 2 rows) of k
__global__ void __launch_bounds__(kNormThreads) l2norm_fwd_kernel(const __nv_bfloat16* __restrict__ q,
                                                                  const __nv_bfloat16* __restrict__ k,
                                                                  __nv_bfloat16* __restrict__ qn,
                                                                  __nv_bfloat16* __restrict__ kn, int64_t rows) {
  const int64_t row = (int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
  if (row >= 2 * rows) return;
  const int lane = threadIdx.x & 31;
  const bool is_q = row < rows;
  const int64_t r = is_q ? row : row - rows;
  const __nv_bfloat16* src = (is_q ? q : k) + r * kDim + 4 * lane;
  __nv_bfloat16* dst = (is_q ? qn : kn) + r * kDim + 4 * lane;
  const uint2 raw = *reinterpret_cast<const uint2*>(src);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  const float ss = warp_sum32(a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y);
  const float rn = rsqrtf(ss + kL2NormEps);
  __nv_bfloat162 o0 = __floats2bfloat162_rn(a.x * rn, a.y * rn), o1 = __floats2bfloat162_rn(b.x * rn, b.y * rn);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&o0);
  w.y = *reinterpret_cast<uint32_t*>(&o1);
  *reinterpret_cast<uint2*>(dst) = w;
}

// dq, dk hold the gradients with respect to the normalised inputs and are overwritten with those
// with respect to the raw inputs
__global__ void __launch_bounds__(kNormThreads) l2norm_bwd_kernel(const __nv_bfloat16* __restrict__ q,
                                                                  const __nv_bfloat16* __restrict__ k, float* dq,
                                                                  float* dk, int64_t rows) {
  const int64_t row = (int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
  if (row >= 2 * rows) return;
  const int lane = threadIdx.x & 31;
  const bool is_q = row < rows;
  const int64_t r = is_q ? row : row - rows;
  const __nv_bfloat16* src = (is_q ? q : k) + r * kDim + 4 * lane;
  float* g = (is_q ? dq : dk) + r * kDim + 4 * lane;
  const uint2 raw = *reinterpret_cast<const uint2*>(src);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  const float4 dy = *reinterpret_cast<const float4*>(g);
  const float ss = warp_sum32(a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y);
  const float rn = rsqrtf(ss + kL2NormEps);
  const float y0 = a.x * rn, y1 = a.y * rn, y2 = b.x * rn, y3 = b.y * rn;
  const float yd = warp_sum32(y0 * dy.x + y1 * dy.y + y2 * dy.z + y3 * dy.w);
  *reinterpret_cast<float4*>(g) =
      make_float4(rn * (dy.x - yd * y0), rn * (dy.y - yd * y1), rn * (dy.z - yd * y2), rn * (dy.w - yd * y3));
}

}  // namespace

int launch_l2norm_fwd(const void* q, const void* k, void* qn, void* kn, int64_t rows, cudaStream_t stream) {
  if (rows <= 0) return kOk;
  const int64_t blocks = (2 * rows + kNormThreads / 32 - 1) / (kNormThreads / 32);
  l2norm_fwd_kernel<<<(unsigned)blocks, kNormThreads, 0, stream>>>(
      reinterpret_cast<const __nv_bfloat16*>(q), reinterpret_cast<const __nv_bfloat16*>(k),
      reinterpret_cast<__nv_bfloat16*>(qn), reinterpret_cast<__nv_bfloat16*>(kn), rows);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

int launch_l2norm_bwd(const void* q, const void* k, float* dq, float* dk, int64_t rows, cudaStream_t stream) {
  if (rows <= 0) return kOk;
  const int64_t blocks = (2 * rows + kNormThreads / 32 - 1) / (kNormThreads / 32);
  l2norm_bwd_kernel<<<(unsigned)blocks, kNormThreads, 0, stream>>>(reinterpret_cast<const __nv_bfloat16*>(q),
                                                                  reinterpret_cast<const __nv_bfloat16*>(k), dq, dk,
                                                                  rows);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace gdn
