// Host side of the tcgen05 / TMA fast path (bf16, d_k = d_v = 128, C = 64).
#pragma once

#include "common.cuh"

namespace gdn {
namespace fast {

// Whether the fast forward takes this geometry and dtype.
bool supports(const Geo &g, int dtype);

// Device workspace the fast forward needs beyond the common header.
size_t workspace_bytes(const Geo &g);

cudaError_t fwd(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                const __nv_bfloat16 *v, const __nv_bfloat16 *beta, const float *gate,
                const float *h0, __nv_bfloat16 *o, float *hT, void *ws, uint32_t *status,
                cudaStream_t st);

}  // namespace fast
}  // namespace gdn
