// Host-side helpers of the C ABI, shared by its translation units: pointer validation and the
// caller's current device.
#pragma once
#include <cuda_runtime.h>

#include <atomic>

namespace gdn {

// Every non-null pointer in ptrs[0..n) must be device memory (cudaMemoryTypeDevice) or managed
// memory; host, pinned-host and unregistered pointers are refused. `anchor` (may be null) decides
// the GPU when given (it must itself be device or managed memory); otherwise the first device
// pointer of the list does, else the first managed one. Every device pointer must live on that
// GPU (managed memory is reachable from all of them). On success *device holds it.
// Returns kOk, kErrInvalid (a refused pointer, pointers on two GPUs, or nothing to decide by).
int device_of(const void* anchor, const void* const* ptrs, int n, int* device);

// Makes a GPU current for the guard's lifetime and gives the caller back its own current device
// afterwards, so that an entry point never changes the calling thread's device.
class DeviceGuard {
 public:
  DeviceGuard() = default;
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
  // false when the switch failed (the caller's device is then unchanged)
  bool set(int device) {
    if (cudaGetDevice(&prev_) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (prev_ == device) return true;
    if (cudaSetDevice(device) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    changed_ = true;
    return true;
  }
  ~DeviceGuard() {
    if (changed_) cudaSetDevice(prev_);
  }

 private:
  int prev_ = 0;
  bool changed_ = false;
};

// Kernel attributes (such as the dynamic shared-memory limit) belong to each GPU's context: a
// launcher sets them the first time it runs on a device. Devices beyond the mask's 64 bits are
// set up on every call.
class PerDevice {
 public:
  bool done(int device) const { return device >= 0 && device < 64 && (mask_.load() >> device & 1ull); }
  void mark(int device) {
    if (device >= 0 && device < 64) mask_.fetch_or(1ull << device);
  }

 private:
  std::atomic<unsigned long long> mask_{0};
};

// A launch that may start while the previous kernel of the stream finishes (programmatic stream
// serialization): the kernel waits for it on the device (griddepcontrol.wait) before it reads or
// writes anything that kernel touches, so only the launch and the CTAs' placement overlap its
// tail. The launch error, if any, is left for cudaGetLastError.
template <typename Params>
inline void launch_early(void (*kernel)(Params), dim3 grid, unsigned threads, size_t smem, cudaStream_t stream,
                         const Params& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace gdn
