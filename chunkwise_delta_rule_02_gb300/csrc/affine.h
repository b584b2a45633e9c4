// Host side of the batched state affine map (sequence-split composition).
#pragma once

#include <cuda_runtime.h>

namespace gdn {
namespace aff {

// out_i = A_i S_i + B_i for i < count; A [count][dk][dk], S, B, out [count][dk][dv],
// all fp32 row-major on the device; B may be null (treated as zero).  out must not
// overlap A or S.
cudaError_t state_affine(const float *A, const float *S, const float *B, float *out, int count,
                         int dk, int dv, cudaStream_t st);

}  // namespace aff
}  // namespace gdn
