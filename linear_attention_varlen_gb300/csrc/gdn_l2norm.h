// Input passes (gdn_l2norm.cu): the q / k normalisation of GDN_FLAG_L2NORM_QK in both directions,
// and the rounding of fp16 inputs to bf16 (GDN_FLAG_FP16_INPUTS).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace gdn {

// qn, kn (bf16 [rows][128]) = q, k ([rows][128], bf16 or fp16 when f16) with every row scaled to unit
// L2 norm.
int launch_l2norm_fwd(const void* q, const void* k, void* qn, void* kn, int64_t rows, bool f16, cudaStream_t stream);
// dq, dk (fp32 [rows][128]): from gradients with respect to the normalised rows to gradients with
// respect to the raw rows of q, k (bf16 or fp16), in place.
int launch_l2norm_bwd(const void* q, const void* k, float* dq, float* dk, int64_t rows, bool f16,
                      cudaStream_t stream);
// dst (bf16) = src (fp16) rounded to nearest even; n elements, a multiple of 8 (16-byte aligned).
int launch_f16_to_bf16(const void* src, void* dst, int64_t n, cudaStream_t stream);

}  // namespace gdn
