// Input passes that run before (and, for the normalisation, after) the chunked pipeline:
//
// L2 normalisation of q and k per (token, key head), and its backward, for callers that hand the
// library unnormalised queries and keys (GDN_FLAG_L2NORM_QK). The recurrence expects unit-norm q
// and k ("Musings on long-context fine-tuning", section "Triton autotuning in the first backward
// pass": the model normalises q and k before the GDN op, and the separate normalisation backward
// with its length-keyed autotuning was what ran out of memory; here both directions are one plain
// pass each, with no tuning and no allocation).
//   forward : y = x r,  r = (x . x + eps)^{-1/2}   (fp32, y rounded once to bf16)
//   backward: dx = r (dy - (y . dy) y)             (y recomputed in fp32 from x)
// One warp per row of 128 elements (4 per lane); q and k rows in one launch.
//
// fp16 inputs (GDN_FLAG_FP16_INPUTS): the kernels' matrix operands are bf16, so q, k, v and dout
// are rounded once to bf16 copies ("How to Speed Up GDN Kernels for Qwen Models", "Using it, and the
// fine print": bf16 or fp16 inputs); the normalisation reads fp16 directly when both flags are set.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// four consecutive 16-bit values (8 bytes) as fp32
template <bool kF16>
__device__ __forceinline__ float4 load4(const uint16_t* p) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  if constexpr (kF16) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    return make_float4(a.x, a.y, b.x, b.y);
  } else {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
}

// rows [0, rows) of q then rows [rows, 2 rows) of k
template <bool kF16>
__global__ void __launch_bounds__(kNormThreads) l2norm_fwd_kernel(const uint16_t* __restrict__ q,
                                                                  const uint16_t* __restrict__ k,
                                                                  __nv_bfloat16* __restrict__ qn,
                                                                  __nv_bfloat16* __restrict__ kn, int64_t rows) {
  const int64_t row = (int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
  if (row >= 2 * rows) return;
  const int lane = threadIdx.x & 31;
  const bool is_q = row < rows;
  const int64_t r = is_q ? row : row - rows;
  const float4 x = load4<kF16>((is_q ? q : k) + r * kDim + 4 * lane);
  __nv_bfloat16* dst = (is_q ? qn : kn) + r * kDim + 4 * lane;
  const float ss = warp_sum32(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
  const float rn = rsqrtf(ss + kL2NormEps);
  __nv_bfloat162 o0 = __floats2bfloat162_rn(x.x * rn, x.y * rn), o1 = __floats2bfloat162_rn(x.z * rn, x.w * rn);
  uint2 w;
  w.x = *reinterpret_cast<uint32_t*>(&o0);
  w.y = *reinterpret_cast<uint32_t*>(&o1);
  *reinterpret_cast<uint2*>(dst) = w;
}

// dq, dk hold the gradients with respect to the normalised inputs and are overwritten with those
// with respect to the raw inputs
template <bool kF16>
__global__ void __launch_bounds__(kNormThreads) l2norm_bwd_kernel(const uint16_t* __restrict__ q,
                                                                  const uint16_t* __restrict__ k, float* dq, float* dk,
                                                                  int64_t rows) {
  const int64_t row = (int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5);
  if (row >= 2 * rows) return;
  const int lane = threadIdx.x & 31;
  const bool is_q = row < rows;
  const int64_t r = is_q ? row : row - rows;
  const float4 x = load4<kF16>((is_q ? q : k) + r * kDim + 4 * lane);
  float* g = (is_q ? dq : dk) + r * kDim + 4 * lane;
  const float4 dy = *reinterpret_cast<const float4*>(g);
  const float ss = warp_sum32(x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w);
  const float rn = rsqrtf(ss + kL2NormEps);
  const float y0 = x.x * rn, y1 = x.y * rn, y2 = x.z * rn, y3 = x.w * rn;
  const float yd = warp_sum32(y0 * dy.x + y1 * dy.y + y2 * dy.z + y3 * dy.w);
  *reinterpret_cast<float4*>(g) =
      make_float4(rn * (dy.x - yd * y0), rn * (dy.y - yd * y1), rn * (dy.z - yd * y2), rn * (dy.w - yd * y3));
}

// fp16 -> bf16 (round to nearest even), 8 elements per thread; n a multiple of 8
__global__ void __launch_bounds__(256) f16_to_bf16_kernel(const uint16_t* __restrict__ src,
                                                          __nv_bfloat16* __restrict__ dst, int64_t n8) {
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (i >= n8) return;
  const uint4 raw = reinterpret_cast<const uint4*>(src)[i];
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float2 f = __half22float2(h[u]);
    __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
    o[u] = *reinterpret_cast<uint32_t*>(&b);
  }
  reinterpret_cast<uint4*>(dst)[i] = out;
}

}  // namespace

int launch_l2norm_fwd(const void* q, const void* k, void* qn, void* kn, int64_t rows, bool f16, cudaStream_t stream) {
  if (rows <= 0) return kOk;
  const int64_t blocks = (2 * rows + kNormThreads / 32 - 1) / (kNormThreads / 32);
  auto qq = reinterpret_cast<const uint16_t*>(q);
  auto kk = reinterpret_cast<const uint16_t*>(k);
  auto qo = reinterpret_cast<__nv_bfloat16*>(qn);
  auto ko = reinterpret_cast<__nv_bfloat16*>(kn);
  if (f16)
    l2norm_fwd_kernel<true><<<(unsigned)blocks, kNormThreads, 0, stream>>>(qq, kk, qo, ko, rows);
  else
    l2norm_fwd_kernel<false><<<(unsigned)blocks, kNormThreads, 0, stream>>>(qq, kk, qo, ko, rows);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

int launch_l2norm_bwd(const void* q, const void* k, float* dq, float* dk, int64_t rows, bool f16,
                      cudaStream_t stream) {
  if (rows <= 0) return kOk;
  const int64_t blocks = (2 * rows + kNormThreads / 32 - 1) / (kNormThreads / 32);
  auto qq = reinterpret_cast<const uint16_t*>(q);
  auto kk = reinterpret_cast<const uint16_t*>(k);
  if (f16)
    l2norm_bwd_kernel<true><<<(unsigned)blocks, kNormThreads, 0, stream>>>(qq, kk, dq, dk, rows);
  else
    l2norm_bwd_kernel<false><<<(unsigned)blocks, kNormThreads, 0, stream>>>(qq, kk, dq, dk, rows);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

int launch_f16_to_bf16(const void* src, void* dst, int64_t n, cudaStream_t stream) {
  if (n <= 0) return kOk;
  const int64_t n8 = n / 8;  // rows of 128 elements: always a multiple of 8
  f16_to_bf16_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, stream>>>(reinterpret_cast<const uint16_t*>(src),
                                                                       reinterpret_cast<__nv_bfloat16*>(dst), n8);
  return cudaGetLastError() == cudaSuccess ? kOk : kErrCuda;
}

}  // namespace gdn
