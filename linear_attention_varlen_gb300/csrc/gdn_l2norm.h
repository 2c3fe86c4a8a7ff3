// L2 normalisation of q and k (GDN_FLAG_L2NORM_QK): launchers of the forward prologue and of the
// backward epilogue (gdn_l2norm.cu).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace gdn {

// qn, kn (bf16 [rows][128]) = q, k (bf16 [rows][128]) with every row scaled to unit L2 norm.
int launch_l2norm_fwd(const void* q, const void* k, void* qn, void* kn, int64_t rows, cudaStream_t stream);
// dq, dk (fp32 [rows][128]): from gradients with respect to the normalised rows to gradients with
// respect to the raw rows of q, k, in place.
int launch_l2norm_bwd(const void* q, const void* k, float* dq, float* dk, int64_t rows, cudaStream_t stream);

}  // namespace gdn
