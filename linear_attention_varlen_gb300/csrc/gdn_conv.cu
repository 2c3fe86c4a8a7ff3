// Width-4 causal depthwise convolution over packed documents, forward and backward (sm_103a).
//
// The short convolution in front of the gated delta rule reads the current input and the three
// before it; documents of a packed batch must not read each other, and a continuation forked from a
// shared prefix P reads P's last three inputs in front of its own, with the gradients through those
// inputs summing back into P ("Musings on long-context fine-tuning", sections "Isolating the
// recurrent layers" and "Backward through P"). Per channel c and document i with tokens x[0 .. n-1]:
//     E = (init[0], init[1], init[2], x[0], ..., x[n-1]),   y[p] = bias[c] + sum_m w[c][m] E[p + m],
//     tail = (E[n], E[n+1], E[n+2]),
// init being zero, a pool entry, or the tail of an earlier document of the call (the same init_idx
// encoding as gdn_chunk_fwd).
//
// Kernels (all bound by memory traffic; two channels per thread, bf16 pairs):
//   conv_check_kernel      cu_seqlens / init_idx validation into the status word
//   conv_tails_kernel      every document's tail, documents in order (forks read earlier tails)
//   conv_fwd_kernel        y over blocks of 32 tokens x 256 channels, a 3-input window in registers
//   conv_bwd_kernel        dx, per-block partial sums of dw and dbias, and each document's gradient at
//                          its three initial inputs (by the block that holds the document's start)
//   conv_reduce_kernel     dw, dbias from the partial sums in block order (deterministic)
//   conv_tails_bwd_kernel  documents in reverse: the tail gradients (given, and those of the forks that
//                          read the tail) into dx of the last inputs, or on into the document's own
//                          start, and the start gradients into the pool entries or the forked document
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_host.h"

namespace gdn {
namespace {

constexpr int kConvTB = 32;       // tokens per block
constexpr int kConvThreads = 128;  // two channels each: 256 channels per block

struct ConvArgs {
  const __nv_bfloat162* x;   // [T][C/2]
  const float* w;            // [C][4]
  const float* bias;         // [C] or null
  const int32_t* cu;
  const int32_t* init_idx;   // [N] or null
  const __nv_bfloat162* conv_init;  // [n_init][3][C/2] or null
  int N, T, C, n_init;
  int32_t* status;           // workspace header
};

struct ConvLayout {
  size_t header, tails, dinit, dtail, part, total;
  int n_tb;
};
inline ConvLayout conv_layout(int N, int T, int C, bool bwd) {
  ConvLayout L{};
  size_t o = 0;
  auto take = [&](size_t b) {
    const size_t at = o;
    o = align_up(o + b, 256);
    return at;
  };
  L.n_tb = (T + kConvTB - 1) / kConvTB;
  L.header = take(256);
  if (bwd) {
    L.tails = take((size_t)N * 3 * C * 2);        // bf16 [N][3][C]: the forward's tails, recomputed
    L.dinit = take((size_t)N * 3 * C * 4);        // fp32 [N][3][C]: gradient at each start (conv part)
    L.dtail = take((size_t)N * 3 * C * 4);        // fp32 [N][3][C]: gradient at each tail (accumulated)
    L.part = take((size_t)L.n_tb * C * 5 * 4);    // fp32 [n_tb][C][5]: dw[4], dbias partial sums
  }
  L.total = o;
  return L;
}

__device__ __forceinline__ bool conv_failed(const int32_t* status) {
  return *reinterpret_cast<const volatile int32_t*>(status) != 0;
}

// The start of document d at channel pair cp: E[0..2] as float2 (zero, pool entry or a fork's tail).
__device__ __forceinline__ void doc_start(const ConvArgs& a, const __nv_bfloat162* tails, int d, int cp,
                                          float2* e) {
  const int s = a.init_idx ? a.init_idx[d] : -1;
  const int C2 = a.C / 2;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    if (s < 0)
      e[k] = make_float2(0.f, 0.f);
    else if (s < a.n_init)
      e[k] = __bfloat1622float2(a.conv_init[((size_t)s * 3 + k) * C2 + cp]);
    else
      e[k] = __bfloat1622float2(tails[((size_t)(s - a.n_init) * 3 + k) * C2 + cp]);
  }
}

// Last index i in [0, N) with cu[i] <= t (a document containing token t; empty ones are passed).
__device__ __forceinline__ int doc_of(const int32_t* cu, int N, int t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(256) conv_check_kernel(ConvArgs a) {
  __shared__ int bad;
  if (threadIdx.x == 0) bad = (a.cu[0] != 0 || a.cu[a.N] != a.T) ? 1 : 0;
  __syncthreads();
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    int b = a.cu[i + 1] < a.cu[i];
    if (a.init_idx) {
      const int s = a.init_idx[i];
      b |= (s < -1) || (s >= a.n_init && s - a.n_init >= i);
    }
    if (b) bad = 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) *a.status = bad ? kErrInvalid : 0;
}

// Documents in order, one thread per channel pair: tail = the last three entries of E.
__global__ void __launch_bounds__(kConvThreads) conv_tails_kernel(ConvArgs a, __nv_bfloat162* tails) {
  if (conv_failed(a.status)) return;
  const int cp = blockIdx.x * kConvThreads + threadIdx.x, C2 = a.C / 2;
  if (cp >= C2) return;
  for (int d = 0; d < a.N; ++d) {
    float2 e[3];
    doc_start(a, tails, d, cp, e);
    const int t0 = a.cu[d], n = a.cu[d + 1] - t0;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int idx = n + k;  // E index of tail entry k
      const __nv_bfloat162 v = idx >= 3 ? a.x[(size_t)(t0 + idx - 3) * C2 + cp] : __floats2bfloat162_rn(e[idx].x, e[idx].y);
      tails[((size_t)d * 3 + k) * C2 + cp] = v;
    }
    __threadfence_block();  // a later fork in this thread reads it back
  }
}

__global__ void __launch_bounds__(kConvThreads) conv_fwd_kernel(ConvArgs a, const __nv_bfloat162* tails,
                                                                __nv_bfloat162* y) {
  if (conv_failed(a.status)) return;
  const int cp = blockIdx.y * kConvThreads + threadIdx.x, C2 = a.C / 2;
  if (cp >= C2) return;
  const int tb0 = blockIdx.x * kConvTB, tb1 = min(tb0 + kConvTB, a.T);
  const float4 w0 = *reinterpret_cast<const float4*>(a.w + (size_t)(2 * cp) * 4);
  const float4 w1 = *reinterpret_cast<const float4*>(a.w + (size_t)(2 * cp + 1) * 4);
  const float b0 = a.bias ? a.bias[2 * cp] : 0.f, b1 = a.bias ? a.bias[2 * cp + 1] : 0.f;
  int d = doc_of(a.cu, a.N, tb0);
  float2 win[3];  // E[p], E[p + 1], E[p + 2] for the current output position p
  bool fresh = true;
  for (int t = tb0; t < tb1; ++t) {
    while (a.cu[d + 1] <= t) {
      ++d;
      fresh = true;
    }
    if (fresh) {
      const int p = t - a.cu[d];
      float2 st[3];
      doc_start(a, tails, d, cp, st);
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int e = p + k;
        win[k] = e < 3 ? st[e] : __bfloat1622float2(a.x[(size_t)(a.cu[d] + e - 3) * C2 + cp]);
      }
      fresh = false;
    }
    const float2 cur = __bfloat1622float2(a.x[(size_t)t * C2 + cp]);
    const float y0 = b0 + w0.x * win[0].x + w0.y * win[1].x + w0.z * win[2].x + w0.w * cur.x;
    const float y1 = b1 + w1.x * win[0].y + w1.y * win[1].y + w1.z * win[2].y + w1.w * cur.y;
    y[(size_t)t * C2 + cp] = __floats2bfloat162_rn(y0, y1);
    win[0] = win[1];
    win[1] = win[2];
    win[2] = cur;
  }
}

__global__ void __launch_bounds__(kConvThreads) conv_bwd_kernel(ConvArgs a, const __nv_bfloat162* tails,
                                                                const __nv_bfloat162* dy, float* dx, float* dinit,
                                                                float* part) {
  if (conv_failed(a.status)) return;
  const int cp = blockIdx.y * kConvThreads + threadIdx.x, C2 = a.C / 2;
  if (cp >= C2) return;
  const int tb0 = blockIdx.x * kConvTB, tb1 = min(tb0 + kConvTB, a.T);
  const float4 w0 = *reinterpret_cast<const float4*>(a.w + (size_t)(2 * cp) * 4);
  const float4 w1 = *reinterpret_cast<const float4*>(a.w + (size_t)(2 * cp + 1) * 4);
  const float wa[4] = {w0.x, w0.y, w0.z, w0.w}, wb[4] = {w1.x, w1.y, w1.z, w1.w};
  float dwa[4] = {0.f, 0.f, 0.f, 0.f}, dwb[4] = {0.f, 0.f, 0.f, 0.f}, dba = 0.f, dbb = 0.f;
  int d = doc_of(a.cu, a.N, tb0);
  for (int t = tb0; t < tb1; ++t) {
    while (a.cu[d + 1] <= t) ++d;
    const int t0 = a.cu[d], t1 = a.cu[d + 1], p = t - t0;
    float2 st[3];
    const bool near_start = p < 3;
    if (near_start) doc_start(a, tails, d, cp, st);
    // as an output: dbias, dw[m] += dy[t] E[p + m]
    const float2 g = __bfloat1622float2(dy[(size_t)t * C2 + cp]);
    dba += g.x;
    dbb += g.y;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = p + m;
      const float2 v = e < 3 ? st[e] : __bfloat1622float2(a.x[(size_t)(t0 + e - 3) * C2 + cp]);
      dwa[m] += g.x * v.x;
      dwb[m] += g.y * v.y;
    }
    // as an input (E index p + 3): read by the outputs p + 3 - m of the same document
    float ga = 0.f, gb = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int to = t + 3 - m;
      if (to < t1) {
        const float2 h = __bfloat1622float2(dy[(size_t)to * C2 + cp]);
        ga += wa[m] * h.x;
        gb += wb[m] * h.y;
      }
    }
    *reinterpret_cast<float2*>(dx + (size_t)t * a.C + 2 * cp) = make_float2(ga, gb);
    // the document's start, E[0..2], read by the outputs 0..2: the block holding its first token
    if (p == 0) {
#pragma unroll
      for (int e = 0; e < 3; ++e) {
        float sa = 0.f, sb = 0.f;
        for (int q = 0; q <= e; ++q) {  // output q reads E[e] with tap e - q
          if (t0 + q < t1) {
            const float2 h = __bfloat1622float2(dy[(size_t)(t0 + q) * C2 + cp]);
            sa += wa[e - q] * h.x;
            sb += wb[e - q] * h.y;
          }
        }
        *reinterpret_cast<float2*>(dinit + ((size_t)d * 3 + e) * a.C + 2 * cp) = make_float2(sa, sb);
      }
    }
  }
  float* pp = part + ((size_t)blockIdx.x * a.C + 2 * cp) * 5;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    pp[m] = dwa[m];
    pp[5 + m] = dwb[m];
  }
  pp[4] = dba;
  pp[9] = dbb;
}

// One warp per channel: lane l sums the partials l, l + 32, ... in order, then a fixed shuffle tree
// (the same order every call: deterministic).
__global__ void __launch_bounds__(256) conv_reduce_kernel(ConvArgs a, const float* part, int n_tb, float* dw,
                                                          float* dbias) {
  if (conv_failed(a.status)) return;
  const int c = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (c >= a.C) return;
  float s[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
  for (int b = lane; b < n_tb; b += 32)
#pragma unroll
    for (int m = 0; m < 5; ++m) s[m] += part[((size_t)b * a.C + c) * 5 + m];
#pragma unroll
  for (int m = 0; m < 5; ++m)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s[m] += __shfl_xor_sync(0xffffffffu, s[m], o);
  if (lane == 0) {
    *reinterpret_cast<float4*>(dw + (size_t)c * 4) = make_float4(s[0], s[1], s[2], s[3]);
    if (dbias) dbias[c] = s[4];
  }
}

// One thread per channel, documents in reverse order.
__global__ void __launch_bounds__(256) conv_tails_bwd_kernel(ConvArgs a, const float* dfinal, const float* dinit_c,
                                                             float* dtail, float* dx, float* dconv_init) {
  if (conv_failed(a.status)) return;
  const int c = blockIdx.x * 256 + threadIdx.x;
  if (c >= a.C) return;
  for (int d = 0; d < a.N; ++d)
    for (int k = 0; k < 3; ++k)
      dtail[((size_t)d * 3 + k) * a.C + c] = dfinal ? dfinal[((size_t)d * 3 + k) * a.C + c] : 0.f;
  if (dconv_init)
    for (int s = 0; s < a.n_init; ++s)
      for (int k = 0; k < 3; ++k) dconv_init[((size_t)s * 3 + k) * a.C + c] = 0.f;
  for (int d = a.N - 1; d >= 0; --d) {
    const int t0 = a.cu[d], n = a.cu[d + 1] - t0;
    float de[3];
#pragma unroll
    for (int e = 0; e < 3; ++e) de[e] = n > 0 ? dinit_c[((size_t)d * 3 + e) * a.C + c] : 0.f;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const float g = dtail[((size_t)d * 3 + k) * a.C + c];
      const int e = n + k;  // tail entry k is E[n + k]
      if (e >= 3)
        dx[(size_t)(t0 + e - 3) * a.C + c] += g;
      else
        de[e] += g;
    }
    const int s = a.init_idx ? a.init_idx[d] : -1;
    if (s >= 0 && s < a.n_init) {
      if (dconv_init)
#pragma unroll
        for (int e = 0; e < 3; ++e) dconv_init[((size_t)s * 3 + e) * a.C + c] += de[e];
    } else if (s >= a.n_init) {
#pragma unroll
      for (int e = 0; e < 3; ++e) dtail[((size_t)(s - a.n_init) * 3 + e) * a.C + c] += de[e];
    }
  }
}

bool aligned(const void* p, uintptr_t b) { return (reinterpret_cast<uintptr_t>(p) % b) == 0; }

int check_common(int N, int T, int C, int n_init, const void* x, const void* w, const int32_t* cu, const void* conv_init,
                 void* workspace) {
  if (N < 1 || T < 0 || C < 8 || C % 8 != 0 || n_init < 0) return GDN_ERR_INVALID_ARG;
  if ((int64_t)T * C > ((int64_t)1 << 40)) return GDN_ERR_INVALID_ARG;
  if (!cu || !w || !workspace || (T > 0 && !x) || (n_init > 0 && !conv_init)) return GDN_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(conv_init, 16) || !aligned(workspace, 256))
    return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

int check_arch_current() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return GDN_ERR_CUDA;
  return (major == 10 && minor == 3) ? GDN_OK : GDN_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace gdn

extern "C" size_t gdn_conv_workspace_size(int N, int T, int C, int backward) {
  if (N < 1 || T < 0 || C < 8 || C % 8 != 0) return 0;
  return gdn::conv_layout(N, T, C, backward != 0).total;
}

extern "C" int gdn_conv_fwd(const void* x, const float* w, const float* bias, const int32_t* cu_seqlens, int N, int T,
                            int C, const int32_t* init_idx, const void* conv_init, int n_init, void* y,
                            void* final_tail, void* workspace, size_t ws_bytes, gdn_stream_t stream) {
  using namespace gdn;
  int rc = check_common(N, T, C, n_init, x, w, cu_seqlens, conv_init, workspace);
  if (rc != GDN_OK) return rc;
  if (!final_tail || (T > 0 && !y) || !aligned(y, 16) || !aligned(final_tail, 16)) return GDN_ERR_INVALID_ARG;
  const ConvLayout L = conv_layout(N, T, C, false);
  if (ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  const void* ptrs[] = {x, w, bias, cu_seqlens, init_idx, conv_init, y, final_tail};
  int dev = 0;
  if (device_of(workspace, ptrs, (int)(sizeof(ptrs) / sizeof(ptrs[0])), &dev) != kOk) return GDN_ERR_INVALID_ARG;
  DeviceGuard guard;
  if (!guard.set(dev)) return GDN_ERR_CUDA;
  if ((rc = check_arch_current()) != GDN_OK) return rc;
  ConvArgs a{reinterpret_cast<const __nv_bfloat162*>(x), w, bias, cu_seqlens, init_idx,
             reinterpret_cast<const __nv_bfloat162*>(conv_init), N, T, C, n_init,
             reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(workspace) + L.header)};
  cudaStream_t s = (cudaStream_t)stream;
  auto* tails = reinterpret_cast<__nv_bfloat162*>(final_tail);
  conv_check_kernel<<<1, 256, 0, s>>>(a);
  const int cb = (C / 2 + kConvThreads - 1) / kConvThreads;
  conv_tails_kernel<<<cb, kConvThreads, 0, s>>>(a, tails);
  if (T > 0) conv_fwd_kernel<<<dim3(L.n_tb, cb), kConvThreads, 0, s>>>(a, tails, reinterpret_cast<__nv_bfloat162*>(y));
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_conv_bwd(const void* x, const float* w, const float* bias, const int32_t* cu_seqlens, int N, int T,
                            int C, const int32_t* init_idx, const void* conv_init, int n_init, const void* dy,
                            const float* dfinal_tail, float* dx, float* dw, float* dbias, float* dconv_init,
                            void* workspace, size_t ws_bytes, gdn_stream_t stream) {
  using namespace gdn;
  int rc = check_common(N, T, C, n_init, x, w, cu_seqlens, conv_init, workspace);
  if (rc != GDN_OK) return rc;
  if (!dw || (T > 0 && (!dy || !dx)) || (n_init > 0 && !dconv_init)) return GDN_ERR_INVALID_ARG;
  if (!aligned(dy, 16) || !aligned(dx, 16) || !aligned(dw, 16) || !aligned(dfinal_tail, 16) ||
      !aligned(dconv_init, 16))
    return GDN_ERR_INVALID_ARG;
  const ConvLayout L = conv_layout(N, T, C, true);
  if (ws_bytes < L.total) return GDN_ERR_WORKSPACE;
  const void* ptrs[] = {x, w, bias, cu_seqlens, init_idx, conv_init, dy, dfinal_tail, dx, dw, dbias, dconv_init};
  int dev = 0;
  if (device_of(workspace, ptrs, (int)(sizeof(ptrs) / sizeof(ptrs[0])), &dev) != kOk) return GDN_ERR_INVALID_ARG;
  DeviceGuard guard;
  if (!guard.set(dev)) return GDN_ERR_CUDA;
  if ((rc = check_arch_current()) != GDN_OK) return rc;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  ConvArgs a{reinterpret_cast<const __nv_bfloat162*>(x), w, bias, cu_seqlens, init_idx,
             reinterpret_cast<const __nv_bfloat162*>(conv_init), N, T, C, n_init,
             reinterpret_cast<int32_t*>(ws + L.header)};
  cudaStream_t s = (cudaStream_t)stream;
  auto* tails = reinterpret_cast<__nv_bfloat162*>(ws + L.tails);
  float* dinit = reinterpret_cast<float*>(ws + L.dinit);
  float* dtail = reinterpret_cast<float*>(ws + L.dtail);
  float* part = reinterpret_cast<float*>(ws + L.part);
  conv_check_kernel<<<1, 256, 0, s>>>(a);
  const int cb = (C / 2 + kConvThreads - 1) / kConvThreads;
  conv_tails_kernel<<<cb, kConvThreads, 0, s>>>(a, tails);
  if (T > 0) {
    conv_bwd_kernel<<<dim3(L.n_tb, cb), kConvThreads, 0, s>>>(a, tails, reinterpret_cast<const __nv_bfloat162*>(dy),
                                                               dx, dinit, part);
  }
  conv_reduce_kernel<<<(C + 7) / 8, 256, 0, s>>>(a, part, L.n_tb, dw, dbias);
  conv_tails_bwd_kernel<<<(C + 255) / 256, 256, 0, s>>>(a, dfinal_tail, dinit, dtail, dx, dconv_init);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
