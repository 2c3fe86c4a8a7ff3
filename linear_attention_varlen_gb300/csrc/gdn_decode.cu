// Single-token decode step of the gated delta rule over a pool of states (sm_103a).
//
// Serving advances each live sequence by one token at a time: its 128 x 128 state per value head
// is read from a pool, decayed, corrected along the token's key, written back in place, and the
// query reads the updated state ("How to Speed Up GDN Kernels for Qwen Models", FAQ "Does this help
// decode too?": decode is a separate kernel; section "What GDN actually computes": the state is a
// fixed 128 x 128 matrix per head, with no cache that grows). For sequence b, value head h (key
// head hk = h / (H_v / H_k)) and S = pool[state_idx[b], h] (q and k first scaled to unit norm with
// GDN_FLAG_L2NORM_QK, in fp32):
//     S' = e^{g} S,  p = S'^T k,  d = beta (v - p),  S = S' + k d^T,  o = scale * S^T q.
// It is the chunked forward's recurrence for a document of one token that starts from a pool entry
// and whose final state replaces that entry.
//
// Work: one CTA of 256 threads per (sequence, value head). Thread t holds the state rows
// 16 (t / 32) .. +15 at columns 4 (t % 32) .. +3 in registers (a warp reads 512 contiguous bytes per
// row: coalesced), the two reductions over rows (S'^T k and S^T q) go through 4 KB of shared
// memory. The state is read and written once: the step is bound by HBM traffic (128 KB per
// sequence and value head).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_host.h"

namespace gdn {
namespace {

constexpr int kDecThreads = 256;

// one 16-bit input element (bf16, or fp16 with GDN_FLAG_FP16_INPUTS) as fp32
template <bool kF16>
__device__ __forceinline__ float ld16(const uint16_t* p) {
  const uint16_t b = *p;
  if constexpr (kF16)
    return __half2float(__ushort_as_half(b));
  else
    return __bfloat162float(__ushort_as_bfloat16(b));
}

template <bool kF16>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const uint16_t* __restrict__ q,
                                                             const uint16_t* __restrict__ k,
                                                             const uint16_t* __restrict__ v,
                                                             const float* __restrict__ g,
                                                             const float* __restrict__ beta,
                                                             const int32_t* __restrict__ state_idx, float* pool,
                                                             int n_pool, int Hk, int Hv, float scale, int l2norm,
                                                             __nv_bfloat16* __restrict__ out, int32_t* status) {
  const int b = blockIdx.x / Hv, h = blockIdx.x % Hv, hk = h / (Hv / Hk);
  const int t = threadIdx.x, cg = t & 31, rg = t >> 5;  // columns 4 cg .. +3, rows 16 rg .. +15
  __shared__ float s_k[kDim], s_q[kDim], s_red[8][kDim], s_d[kDim];
  const int x = state_idx[b];
  __nv_bfloat16* orow = out + ((size_t)b * Hv + h) * kDim;
  if (x < 0 || x >= n_pool) {  // skipped, reported
    if (t < kDim) orow[t] = __float2bfloat16_rn(0.f);
    if (t == 0 && status) atomicCAS(status, 0, kErrInvalid);
    return;
  }
  if (t < kDim) {
    s_k[t] = ld16<kF16>(k + ((size_t)b * Hk + hk) * kDim + t);
    s_q[t] = ld16<kF16>(q + ((size_t)b * Hk + hk) * kDim + t);
  }
  __syncthreads();
  if (t < 64) {
    // warps 0-1: |q|^2 and |k|^2 (GDN_FLAG_L2NORM_QK) in s_red row 0; the scale
    const float* xv = (t < 32) ? s_q : s_k;
    const int l = t & 31;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) ss += xv[l + 32 * i] * xv[l + 32 * i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (l == 0) s_red[0][t >> 5] = l2norm ? rsqrtf(ss + kL2NormEps) : 1.f;
  }
  __syncthreads();
  if (t < kDim) {
    s_q[t] *= s_red[0][0] * scale;
    s_k[t] *= s_red[0][1];
  }
  const float a = __expf(g[(size_t)b * Hv + h]), bt = beta[(size_t)b * Hv + h];
  float* S = pool + ((size_t)x * Hv + h) * kDim * kDim;
  float4 st[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) st[i] = *reinterpret_cast<const float4*>(S + (size_t)(16 * rg + i) * kDim + 4 * cg);
  __syncthreads();
  // S' = a S and this thread's part of p = S'^T k
  float4 pp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    st[i].x *= a;
    st[i].y *= a;
    st[i].z *= a;
    st[i].w *= a;
    const float kr = s_k[16 * rg + i];
    pp.x += kr * st[i].x;
    pp.y += kr * st[i].y;
    pp.z += kr * st[i].z;
    pp.w += kr * st[i].w;
  }
  *reinterpret_cast<float4*>(&s_red[rg][4 * cg]) = pp;
  __syncthreads();
  if (t < kDim) {
    float p = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) p += s_red[r][t];
    s_d[t] = bt * (ld16<kF16>(v + ((size_t)b * Hv + h) * kDim + t) - p);
  }
  __syncthreads();
  // S = S' + k d^T, written back; this thread's part of o = S^T (scale q)
  const float4 d4 = *reinterpret_cast<const float4*>(&s_d[4 * cg]);
  float4 oo = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = 16 * rg + i;
    const float kr = s_k[r], qr = s_q[r];
    st[i].x += kr * d4.x;
    st[i].y += kr * d4.y;
    st[i].z += kr * d4.z;
    st[i].w += kr * d4.w;
    *reinterpret_cast<float4*>(S + (size_t)r * kDim + 4 * cg) = st[i];
    oo.x += qr * st[i].x;
    oo.y += qr * st[i].y;
    oo.z += qr * st[i].z;
    oo.w += qr * st[i].w;
  }
  *reinterpret_cast<float4*>(&s_red[rg][4 * cg]) = oo;
  __syncthreads();
  if (t < kDim) {
    float o = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) o += s_red[r][t];
    orow[t] = __float2bfloat16_rn(o);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gdn

extern "C" int gdn_decode_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                               int B, int H_k, int H_v, int head_dim, const int32_t* state_idx, float* state_pool,
                               int n_pool, void* out, int32_t* status, const gdn_options* opt, gdn_stream_t stream) {
  if (head_dim != gdn::kDim) return GDN_ERR_UNSUPPORTED;
  if (B < 0 || H_k < 1 || H_v < 1 || H_v % H_k != 0 || n_pool < 0) return GDN_ERR_INVALID_ARG;
  if ((int64_t)B * H_v > (int64_t)INT32_MAX) return GDN_ERR_INVALID_ARG;
  gdn_options o;
  gdn_default_options(&o);
  if (opt) o = *opt;
  if (o.scale != o.scale) return GDN_ERR_INVALID_ARG;
  if (B == 0) return GDN_OK;
  if (!q || !k || !v || !g || !beta || !state_idx || !state_pool || !out || n_pool == 0) return GDN_ERR_INVALID_ARG;
  if (!gdn::aligned16(state_pool)) return GDN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, state_idx, out, status};
  int dev = 0;
  if (gdn::device_of(state_pool, ptrs, (int)(sizeof(ptrs) / sizeof(ptrs[0])), &dev) != gdn::kOk)
    return GDN_ERR_INVALID_ARG;
  gdn::DeviceGuard guard;
  if (!guard.set(dev)) return GDN_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (major != 10 || minor != 3) return GDN_ERR_UNSUPPORTED;
  auto q16 = reinterpret_cast<const uint16_t*>(q);
  auto k16 = reinterpret_cast<const uint16_t*>(k);
  auto v16 = reinterpret_cast<const uint16_t*>(v);
  const int l2 = (o.flags & GDN_FLAG_L2NORM_QK) ? 1 : 0;
  const unsigned grid = (unsigned)(B * H_v);
  if (o.flags & GDN_FLAG_FP16_INPUTS)
    gdn::decode_kernel<true><<<grid, gdn::kDecThreads, 0, (cudaStream_t)stream>>>(
        q16, k16, v16, g, beta, state_idx, state_pool, n_pool, H_k, H_v, o.scale, l2,
        reinterpret_cast<__nv_bfloat16*>(out), status);
  else
    gdn::decode_kernel<false><<<grid, gdn::kDecThreads, 0, (cudaStream_t)stream>>>(
        q16, k16, v16, g, beta, state_idx, state_pool, n_pool, H_k, H_v, o.scale, l2,
        reinterpret_cast<__nv_bfloat16*>(out), status);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
