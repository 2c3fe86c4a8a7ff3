// C ABI of the GDN library (declared in include/gdn.h): argument checks, workspace sizing,
// tensor-map creation and kernel launches. No allocation, no synchronisation.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_bwd.h"
#include "gdn_common.cuh"
#include "gdn_dev.cuh"
#include "gdn_fwd.h"
#include "gdn_host.h"
#include "gdn_l2norm.h"
#include "tmap.h"

using namespace gdn;

namespace gdn {

int device_of(const void* anchor, const void* const* ptrs, int n, int* device) {
  // 1 = device memory, 2 = managed memory, 0 = refused (host, pinned host, unregistered, error)
  auto kind = [](const void* p, int* dev) -> int {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    *dev = attr.device;
    if (attr.type == cudaMemoryTypeDevice) return 1;
    if (attr.type == cudaMemoryTypeManaged) return 2;
    return 0;
  };
  int chosen = -1, managed = -1;
  if (anchor) {
    int dv = -1;
    if (kind(anchor, &dv) == 0) return kErrInvalid;
    chosen = dv;
  }
  for (int i = 0; i < n; ++i) {
    if (!ptrs[i]) continue;
    int dv = -1;
    const int k = kind(ptrs[i], &dv);
    if (k == 0) return kErrInvalid;
    if (k == 2) {
      if (managed < 0) managed = dv;
      continue;
    }
    if (chosen < 0)
      chosen = dv;
    else if (dv != chosen)
      return kErrInvalid;
  }
  if (chosen < 0) chosen = managed;
  if (chosen < 0) return kErrInvalid;
  *device = chosen;
  return kOk;
}

}  // namespace gdn

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// The kernels use tcgen05 and are compiled for sm_103a (GB300, compute capability 10.3) only.
int check_arch() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kErrCuda;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return kErrCuda;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return kErrCuda;
  return (major == 10 && minor == 3) ? kOk : kErrUnsupported;
}

gdn_options resolve(const gdn_options* opt) {
  gdn_options o;
  gdn_default_options(&o);
  if (opt) o = *opt;
  return o;
}

bool valid_options(const gdn_options& o) {
  return (o.mode == GDN_MODE_EXACT || o.mode == GDN_MODE_TRUNCATE) &&
         (o.flags & ~(GDN_FLAG_SAVE_FOR_BWD | GDN_FLAG_REUSE_FWD | GDN_FLAG_TEST_WITHHOLD_FORK | GDN_FLAG_L2NORM_QK |
                      GDN_FLAG_FP16_INPUTS)) == 0 &&
         o.scale == o.scale && o.flag_wait_us >= 0;
}

// Wait limit of the cross-item waits in SM clock cycles (about 2 cycles per nanosecond at the
// maximum clock; slower clocks make the wait longer, never shorter than asked).
long long flag_budget(const gdn_options& o) {
  return o.flag_wait_us > 0 ? (long long)o.flag_wait_us * 2070LL : kWaitBudget;
}

PlanDims make_dims(int N, int T, int H_k, int H_v, int n_init, const gdn_options& o, int sms) {
  PlanDims d;
  d.N = N;
  d.T = T;
  d.Hk = H_k;
  d.Hv = H_v;
  d.n_init = n_init;
  d.num_sms = sms > 0 ? sms : 1;
  d.seg_override = o.segment_chunks;
  d.mode = o.mode;
  return d;
}

bool sizes_ok(int N, int T, int H_k, int H_v) {
  if (N < 1 || T < 0 || H_k < 1 || H_v < 1 || H_v % H_k != 0) return false;
  if ((int64_t)T * H_v * kDim > ((int64_t)1 << 40)) return false;
  return true;
}

}  // namespace

extern "C" {

void gdn_default_options(gdn_options* opt) {
  if (!opt) return;
  opt->mode = GDN_MODE_EXACT;
  opt->trunc_log_threshold = -10.0f;
  opt->segment_chunks = 0;
  opt->scale = 1.0f;
  opt->flags = 0;
  opt->stage_events = nullptr;
  opt->flag_wait_us = 0;
}

const char* gdn_status_string(int status) {
  switch (status) {
    case GDN_OK:
      return "GDN_OK";
    case GDN_ERR_INVALID_ARG:
      return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED:
      return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_CUDA:
      return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT:
      return "GDN_ERR_TIMEOUT";
    case GDN_ERR_WORKSPACE:
      return "GDN_ERR_WORKSPACE";
    default:
      return "GDN_ERR_UNKNOWN";
  }
}

size_t gdn_fwd_workspace_size(int N, int T, int H_k, int H_v, const gdn_options* opt) {
  if (!sizes_ok(N, T, H_k, H_v)) return 0;
  const gdn_options o = resolve(opt);
  if (!valid_options(o)) return 0;
  if (o.flags & GDN_FLAG_SAVE_FOR_BWD) return gdn_bwd_workspace_size(N, T, H_k, H_v, opt);
  return fwd_layout(make_dims(N, T, H_k, H_v, 0, o, current_sm_count())).total +
         input_copies(T, H_k, H_v, o.flags, false).total;
}

size_t gdn_bwd_workspace_size(int N, int T, int H_k, int H_v, const gdn_options* opt) {
  if (!sizes_ok(N, T, H_k, H_v)) return 0;
  gdn_options o = resolve(opt);
  if (!valid_options(o)) return 0;
  o.mode = GDN_MODE_EXACT;  // the backward is always exact
  return bwd_layout(make_dims(N, T, H_k, H_v, 0, o, current_sm_count())).total +
         input_copies(T, H_k, H_v, o.flags, true).total;
}

int gdn_workspace_status(const void* workspace, gdn_stream_t stream) {
  if (!workspace) return GDN_ERR_INVALID_ARG;
  int dev = 0;
  if (device_of(workspace, nullptr, 0, &dev) != kOk) return GDN_ERR_INVALID_ARG;
  DeviceGuard guard;
  if (!guard.set(dev)) return GDN_ERR_CUDA;
  int32_t st = 0;
  if (cudaMemcpyAsync(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
  return st;
}

}  // extern "C"

namespace {

// Every host-side check of a forward call, in order, up to the launch: sizes, options, null and
// alignment rules, the memory kind and GPU of every pointer, the GPU's architecture and the
// workspace size. On GDN_OK the workspace's GPU is current (through `guard`) and *o holds the
// resolved options.
int prepare_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim, const int32_t* init_idx,
                const float* initial_state, int n_init, void* out, float* final_state, void* workspace,
                size_t ws_bytes, const gdn_options* opt, gdn_options* o, DeviceGuard& guard) {
  if (head_dim != kDim) return GDN_ERR_UNSUPPORTED;
  if (!sizes_ok(N, T, H_k, H_v) || n_init < 0) return GDN_ERR_INVALID_ARG;
  *o = resolve(opt);
  if (!valid_options(*o)) return GDN_ERR_INVALID_ARG;
  if (!cu_seqlens || !final_state || !workspace) return GDN_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
  if (n_init > 0 && !initial_state) return GDN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(final_state, 16) ||
      !aligned(initial_state, 16) || !aligned(workspace, 256))
    return GDN_ERR_INVALID_ARG;
  if (o->flags & GDN_FLAG_REUSE_FWD) return GDN_ERR_INVALID_ARG;  // a backward option
  if ((o->flags & GDN_FLAG_SAVE_FOR_BWD) && o->mode != GDN_MODE_EXACT) return GDN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, g, beta, cu_seqlens, init_idx, initial_state, out, final_state};
  int dev = 0;
  if (device_of(workspace, ptrs, (int)(sizeof(ptrs) / sizeof(ptrs[0])), &dev) != kOk) return GDN_ERR_INVALID_ARG;
  if (!guard.set(dev)) return GDN_ERR_CUDA;
  const int arch = check_arch();
  if (arch != kOk) return arch;
  const PlanDims d = make_dims(N, T, H_k, H_v, n_init, *o, current_sm_count());
  const bool save = (o->flags & GDN_FLAG_SAVE_FOR_BWD) != 0;
  const size_t need = (save ? bwd_layout(d).total : fwd_layout(d).total) + input_copies(T, H_k, H_v, o->flags, save).total;
  if (ws_bytes < need) return GDN_ERR_WORKSPACE;
  return GDN_OK;
}

// Same for a backward call.
int prepare_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim, const int32_t* init_idx,
                const float* initial_state, int n_init, const void* dout, const float* dfinal_state, float* dq,
                float* dk, float* dv, float* dg, float* dbeta, float* dinitial_state, void* workspace,
                size_t ws_bytes, const gdn_options* opt, gdn_options* o, DeviceGuard& guard) {
  if (head_dim != kDim) return GDN_ERR_UNSUPPORTED;
  if (!sizes_ok(N, T, H_k, H_v) || n_init < 0) return GDN_ERR_INVALID_ARG;
  *o = resolve(opt);
  if (!valid_options(*o)) return GDN_ERR_INVALID_ARG;
  if (!cu_seqlens || !workspace) return GDN_ERR_INVALID_ARG;
  if (T > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg || !dbeta))
    return GDN_ERR_INVALID_ARG;
  if (n_init > 0 && (!initial_state || !dinitial_state)) return GDN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dout, 16) || !aligned(dq, 16) ||
      !aligned(dk, 16) || !aligned(dv, 16) || !aligned(initial_state, 16) || !aligned(dfinal_state, 16) ||
      !aligned(dinitial_state, 16) || !aligned(workspace, 256))
    return GDN_ERR_INVALID_ARG;
  if (o->flags & (GDN_FLAG_SAVE_FOR_BWD | GDN_FLAG_TEST_WITHHOLD_FORK)) return GDN_ERR_INVALID_ARG;  // forward options
  const void* ptrs[] = {q,    k,  v,  g,  beta, cu_seqlens, init_idx, initial_state, dout, dfinal_state,
                        dq,   dk, dv, dg, dbeta, dinitial_state};
  int dev = 0;
  if (device_of(workspace, ptrs, (int)(sizeof(ptrs) / sizeof(ptrs[0])), &dev) != kOk) return GDN_ERR_INVALID_ARG;
  if (!guard.set(dev)) return GDN_ERR_CUDA;
  const int arch = check_arch();
  if (arch != kOk) return arch;
  gdn_options oe = *o;
  oe.mode = GDN_MODE_EXACT;
  if (ws_bytes < bwd_layout(make_dims(N, T, H_k, H_v, n_init, oe, current_sm_count())).total +
                     input_copies(T, H_k, H_v, o->flags, true).total)
    return GDN_ERR_WORKSPACE;
  return GDN_OK;
}

// The input copies of GDN_FLAG_L2NORM_QK / GDN_FLAG_FP16_INPUTS at `base`: q and k normalised (from
// bf16 or fp16) or converted, v and dout converted; the pointers are redirected to the copies.
int stage_inputs(const void*& q, const void*& k, const void*& v, const void** dout, uint8_t* base,
                 const InputCopies& c, int flags, int T, int H_k, int H_v, cudaStream_t stream) {
  const bool f16 = (flags & GDN_FLAG_FP16_INPUTS) != 0;
  uint8_t* qn = base + c.q;
  uint8_t* kn = base + c.k;
  const int64_t nqk = (int64_t)T * H_k * kDim, nv = (int64_t)T * H_v * kDim;
  if (flags & GDN_FLAG_L2NORM_QK) {
    if (launch_l2norm_fwd(q, k, qn, kn, (int64_t)T * H_k, f16, stream) != kOk) return GDN_ERR_CUDA;
  } else if (launch_f16_to_bf16(q, qn, nqk, stream) != kOk || launch_f16_to_bf16(k, kn, nqk, stream) != kOk) {
    return GDN_ERR_CUDA;
  }
  q = qn;
  k = kn;
  if (f16) {
    if (launch_f16_to_bf16(v, base + c.v, nv, stream) != kOk) return GDN_ERR_CUDA;
    v = base + c.v;
    if (dout) {
      if (launch_f16_to_bf16(*dout, base + c.dout, nv, stream) != kOk) return GDN_ERR_CUDA;
      *dout = base + c.dout;
    }
  }
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_fwd_check_args(const void* q, const void* k, const void* v, const float* g, const float* beta,
                       const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                       const int32_t* init_idx, const float* initial_state, int n_init, void* out,
                       float* final_state, void* workspace, size_t ws_bytes, const gdn_options* opt) {
  gdn_options o;
  DeviceGuard guard;
  return prepare_fwd(q, k, v, g, beta, cu_seqlens, N, T, H_k, H_v, head_dim, init_idx, initial_state, n_init, out,
                     final_state, workspace, ws_bytes, opt, &o, guard);
}

int gdn_bwd_check_args(const void* q, const void* k, const void* v, const float* g, const float* beta,
                       const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                       const int32_t* init_idx, const float* initial_state, int n_init, const void* dout,
                       const float* dfinal_state, float* dq, float* dk, float* dv, float* dg, float* dbeta,
                       float* dinitial_state, void* workspace, size_t ws_bytes, const gdn_options* opt) {
  gdn_options o;
  DeviceGuard guard;
  return prepare_bwd(q, k, v, g, beta, cu_seqlens, N, T, H_k, H_v, head_dim, init_idx, initial_state, n_init, dout,
                     dfinal_state, dq, dk, dv, dg, dbeta, dinitial_state, workspace, ws_bytes, opt, &o, guard);
}

int gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                  const int32_t* init_idx, const float* initial_state, int n_init, void* out, float* final_state,
                  void* workspace, size_t ws_bytes, const gdn_options* opt, gdn_stream_t stream) {
  gdn_options o;
  DeviceGuard guard;
  const int rc = prepare_fwd(q, k, v, g, beta, cu_seqlens, N, T, H_k, H_v, head_dim, init_idx, initial_state, n_init,
                             out, final_state, workspace, ws_bytes, opt, &o, guard);
  if (rc != GDN_OK) return rc;
  const int sms = current_sm_count();
  cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(o.stage_events);
  if (o.flags & (GDN_FLAG_L2NORM_QK | GDN_FLAG_FP16_INPUTS)) {
    // normalised / converted copies of the inputs after the layout; every later kernel reads them
    const PlanDims d0 = make_dims(N, T, H_k, H_v, n_init, o, sms);
    const bool save = (o.flags & GDN_FLAG_SAVE_FOR_BWD) != 0;
    uint8_t* base = reinterpret_cast<uint8_t*>(workspace) + (save ? bwd_layout(d0).total : fwd_layout(d0).total);
    if (ev && ev[18]) cudaEventRecord(ev[18], (cudaStream_t)stream);
    const int rs = stage_inputs(q, k, v, nullptr, base, input_copies(T, H_k, H_v, o.flags, save), o.flags, T, H_k,
                                H_v, (cudaStream_t)stream);
    if (rs != GDN_OK) return rs;
    if (ev && ev[19]) cudaEventRecord(ev[19], (cudaStream_t)stream);
  } else if (ev) {
    for (int i = 18; i < 20; ++i)
      if (ev[i]) cudaEventRecord(ev[i], (cudaStream_t)stream);
  }
  if (o.flags & GDN_FLAG_SAVE_FOR_BWD) {
    BwdArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.beta = beta;
    a.cu = cu_seqlens;
    a.init_idx = init_idx;
    a.initial_state = initial_state;
    a.ws = workspace;
    a.ws_bytes = ws_bytes;
    a.d = make_dims(N, T, H_k, H_v, n_init, o, sms);
    a.trunc_thr = o.trunc_log_threshold;
    a.scale = o.scale;
    a.flag_budget = flag_budget(o);
    a.withhold_fin = (o.flags & GDN_FLAG_TEST_WITHHOLD_FORK) ? 1 : 0;
    return launch_fwd_save(a, out, final_state, (cudaStream_t)stream, reinterpret_cast<cudaEvent_t*>(o.stage_events));
  }
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.d = make_dims(N, T, H_k, H_v, n_init, o, sms);
  p.L = fwd_layout(p.d);
  if (ws_bytes < p.L.total) return GDN_ERR_WORKSPACE;
  if (T > 0) {
    const uint64_t row_k = (uint64_t)H_k * kDim * 2, row_v = (uint64_t)H_v * kDim * 2;
    if (!make_tmap_bf16_3d(&p.tm_q, q, kDim, H_k, T, kDim * 2, row_k, 64, 1, 64) ||
        !make_tmap_bf16_3d(&p.tm_k, k, kDim, H_k, T, kDim * 2, row_k, 64, 1, 64) ||
        !make_tmap_bf16_3d(&p.tm_v, v, kDim, H_v, T, kDim * 2, row_v, 64, 1, 64) ||
        !make_tmap_bf16_3d(&p.tm_o, out, kDim, H_v, T, kDim * 2, row_v, 64, 1, 64))
      return GDN_ERR_CUDA;
  }
  p.g = g;
  p.beta = beta;
  p.cu = cu_seqlens;
  p.init_idx = init_idx;
  p.initial_state = initial_state;
  p.out = reinterpret_cast<__nv_bfloat16*>(out);
  p.final_state = final_state;
  p.ws = reinterpret_cast<uint8_t*>(workspace);
  p.trunc_thr = o.trunc_log_threshold;
  p.scale = o.scale;
  p.flag_budget = flag_budget(o);
  p.withhold_fin = (o.flags & GDN_FLAG_TEST_WITHHOLD_FORK) ? 1 : 0;
  p.p_img = p.ws + p.L.pimg;
  p.p_factored = 1;
  return launch_fwd(p, (cudaStream_t)stream, reinterpret_cast<cudaEvent_t*>(o.stage_events));
}

int gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const int32_t* cu_seqlens, int N, int T, int H_k, int H_v, int head_dim,
                  const int32_t* init_idx, const float* initial_state, int n_init, const void* dout,
                  const float* dfinal_state, float* dq, float* dk, float* dv, float* dg, float* dbeta,
                  float* dinitial_state, void* workspace, size_t ws_bytes, const gdn_options* opt,
                  gdn_stream_t stream) {
  gdn_options o;
  DeviceGuard guard;
  const int rc = prepare_bwd(q, k, v, g, beta, cu_seqlens, N, T, H_k, H_v, head_dim, init_idx, initial_state, n_init,
                             dout, dfinal_state, dq, dk, dv, dg, dbeta, dinitial_state, workspace, ws_bytes, opt, &o,
                             guard);
  if (rc != GDN_OK) return rc;
  cudaEvent_t* ev = reinterpret_cast<cudaEvent_t*>(o.stage_events);
  gdn_options oe = o;
  oe.mode = GDN_MODE_EXACT;  // the backward recomputes and differentiates the exact forward
  const PlanDims dims = make_dims(N, T, H_k, H_v, n_init, oe, current_sm_count());
  const void* q_raw = q;
  const void* k_raw = k;
  if (o.flags & (GDN_FLAG_L2NORM_QK | GDN_FLAG_FP16_INPUTS)) {
    uint8_t* base = reinterpret_cast<uint8_t*>(workspace) + bwd_layout(dims).total;
    if (ev && ev[18]) cudaEventRecord(ev[18], (cudaStream_t)stream);
    const int rs = stage_inputs(q, k, v, &dout, base, input_copies(T, H_k, H_v, o.flags, true), o.flags, T, H_k,
                                H_v, (cudaStream_t)stream);
    if (rs != GDN_OK) return rs;
    if (ev && ev[19]) cudaEventRecord(ev[19], (cudaStream_t)stream);
  } else if (ev) {
    for (int i = 18; i < 20; ++i)
      if (ev[i]) cudaEventRecord(ev[i], (cudaStream_t)stream);
  }
  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.cu = cu_seqlens;
  a.init_idx = init_idx;
  a.initial_state = initial_state;
  a.dout = dout;
  a.dfinal = dfinal_state;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dg = dg;
  a.dbeta = dbeta;
  a.dinit = dinitial_state;
  a.ws = workspace;
  a.ws_bytes = ws_bytes;
  a.d = dims;
  a.trunc_thr = o.trunc_log_threshold;
  a.scale = o.scale;
  a.flag_budget = flag_budget(o);
  a.withhold_fin = 0;
  const int rb = launch_bwd(a, (o.flags & GDN_FLAG_REUSE_FWD) != 0, (cudaStream_t)stream, ev);
  if (rb != GDN_OK) return rb;
  if (!(o.flags & GDN_FLAG_L2NORM_QK)) {
    if (ev)
      for (int i = 20; i < 22; ++i)
        if (ev[i]) cudaEventRecord(ev[i], (cudaStream_t)stream);
    return GDN_OK;
  }
  // gradients with respect to the unnormalised q and k
  if (ev && ev[20]) cudaEventRecord(ev[20], (cudaStream_t)stream);
  if (launch_l2norm_bwd(q_raw, k_raw, dq, dk, (int64_t)T * H_k, (o.flags & GDN_FLAG_FP16_INPUTS) != 0,
                        (cudaStream_t)stream) != kOk)
    return GDN_ERR_CUDA;
  if (ev && ev[21]) cudaEventRecord(ev[21], (cudaStream_t)stream);
  return GDN_OK;
}

int gdn_plan_host(const int32_t* cu, int N, int T, int H_v, const int32_t* init_idx, int n_init,
                  const gdn_options* opt, int num_sms, int32_t* chunk_seq, int32_t* chunk_tok0, int32_t* chunk_len,
                  int max_chunks_arg, int32_t* seg_info, int max_segs_arg, int32_t* out_counts) {
  if (!cu || N < 1 || T < 0 || H_v < 1 || n_init < 0 || !out_counts) return GDN_ERR_INVALID_ARG;
  const gdn_options o = resolve(opt);
  if (!valid_options(o)) return GDN_ERR_INVALID_ARG;
  if (cu[0] != 0 || cu[N] != T) return GDN_ERR_INVALID_ARG;
  for (int i = 0; i < N; ++i)
    if (plan_check_doc(i, cu, init_idx, n_init) != kOk) return GDN_ERR_INVALID_ARG;
  PlanDims d = make_dims(N, T, 1, H_v, n_init, o, num_sms);
  std::vector<int32_t> seq_chunk0(N + 1), seq_seg0(N + 1);
  int total = 0, longest = 0;
  for (int i = 0; i < N; ++i) {
    seq_chunk0[i] = total;
    const int c = doc_chunks(i, cu);
    total += c;
    if (c > longest) longest = c;
  }
  seq_chunk0[N] = total;
  const int L = plan_seg_len(d, total, longest);
  int segs = 0;
  for (int i = 0; i < N; ++i) {
    seq_seg0[i] = segs;
    segs += doc_segs(doc_chunks(i, cu), L);
  }
  seq_seg0[N] = segs;
  out_counts[0] = total;
  out_counts[1] = segs;
  out_counts[2] = L;
  if (total > max_chunks_arg || segs > max_segs_arg) return GDN_ERR_WORKSPACE;
  for (int c = 0; c < total; ++c) plan_chunk(c, seq_chunk0.data(), N, cu, chunk_seq + c, chunk_tok0 + c, chunk_len + c);
  for (int s = 0; s < segs; ++s)
    plan_segment(s, seq_seg0.data(), seq_chunk0.data(), N, cu, L, init_idx, n_init, seg_info + 4 * s);
  return GDN_OK;
}

}  // extern "C"
