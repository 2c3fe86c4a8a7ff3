// Forward without a caller-provided workspace.
//
// Some callers cannot allocate device memory: a plain C host program that links this library
// without any device allocator of its own, or a plugin running inside a host framework whose
// memory pool owns all device memory and does not allow outside cudaMalloc calls. For them,
// gdn_chunk_fwd_noalloc runs the same forward kernels as gdn_chunk_fwd with the scratch taken
// from a fixed-size array that lives in this file (static __device__ storage, created when the
// library's module is loaded on a GPU and held until the process exits).
//
// Rules of use:
//  - Problems whose forward workspace exceeds kNoAllocScratchBytes are rejected with
//    GDN_ERR_WORKSPACE before anything is launched.
//  - Every call shares the one array; it keeps the previous call's contents. Nothing in it has
//    to start at zero: the first kernel of the forward rewrites every field the later kernels
//    read (maps, queue counters, flags).
//  - Calls that overlap on the GPU (two streams, two host threads without ordering) race on the
//    array and give undefined results; order them on one stream.
//  - The first call on a device looks up the array's device address (cudaGetSymbolAddress) and
//    caches it per device; make that first call before any stream capture.
//  - Errors found on the GPU (bad cu_seqlens or init_idx, an expired bounded wait) land in the
//    array's status word: gdn_noalloc_status() reads it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_host.h"

namespace {

// 160 MiB: enough for a 32768-token document at 8 value heads (about 129 MiB with 148-152 SMs).
constexpr size_t kNoAllocScratchBytes = size_t(160) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return GDN_ERR_CUDA;
    }
    g_addr[dev] = ptr;
  }
  *out = g_addr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" size_t gdn_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int gdn_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                     const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                                     const int32_t* init_idx, const float* initial_state, int n_init, void* out,
                                     float* final_state, const gdn_options* opt, gdn_stream_t stream) {
  if (head_dim != 128) return GDN_ERR_UNSUPPORTED;
  // records kept for a backward need a workspace that the caller can hand to it
  if (opt && (opt->flags & GDN_FLAG_SAVE_FOR_BWD)) return GDN_ERR_INVALID_ARG;
  // the tensors decide the GPU (the same pointer rules as gdn_chunk_fwd, which checks them again)
  const void* ptrs[] = {out, final_state, q, k, v, g, beta, cu_seqlens, init_idx, initial_state};
  int dev = 0;
  if (gdn::device_of(nullptr, ptrs, (int)(sizeof(ptrs) / sizeof(ptrs[0])), &dev) != gdn::kOk)
    return GDN_ERR_INVALID_ARG;
  gdn::DeviceGuard guard;
  if (!guard.set(dev)) return GDN_ERR_CUDA;
  const size_t need = gdn_fwd_workspace_size(N, T, H_k, H_v, opt);
  if (need == 0) return GDN_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;
  void* ws = nullptr;
  const int rc = scratch_address(&ws);
  if (rc != GDN_OK) return rc;
  return gdn_chunk_fwd(q, k, v, g, beta, cu_seqlens, N, T, H_k, H_v, head_dim, init_idx, initial_state, n_init, out,
                       final_state, ws, kNoAllocScratchBytes, opt, stream);
}

extern "C" int gdn_noalloc_status(int device, gdn_stream_t stream) {
  if (device < 0 || device >= kMaxDevices) return GDN_ERR_INVALID_ARG;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ws = g_addr[device];
  }
  if (!ws) return GDN_ERR_INVALID_ARG;  // no allocation-free call has run on this device
  return gdn_workspace_status(ws, stream);
}
