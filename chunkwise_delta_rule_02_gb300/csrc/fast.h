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

// Cooperative persistent forward (preparation CTAs + chain CTAs): bf16 with
// d_k = d_v = 128 and C = 64 or 32, or d_k = d_v = 256 and C = 32.
namespace coop {

// Whether this device can run it (cooperative launch, tensor-map encoder).
bool available();

// Whether it takes this geometry and dtype.
bool supports(const Geo &g, int dtype);

// Workspace it needs: control words, packed order, package ring.  sms <= 0 sizes
// for an upper bound on the SM count.
size_t workspace_bytes(const Geo &g, int sms);

cudaError_t fwd(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                const __nv_bfloat16 *v, const __nv_bfloat16 *beta, const float *gate,
                const float *h0, __nv_bfloat16 *o, float *hT, void *ws, size_t ws_bytes,
                uint32_t *status, cudaStream_t st);

}  // namespace coop
}  // namespace gdn
