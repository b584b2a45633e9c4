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

// Extra outputs for the backward (any may be null): every chunk's package into
// keep[slot * stride] (the layout below), the bf16 state entering the chunk into
// sin[slot][dk][dv] and Unew into unew[slot][C][dv], slot = chunk slot * H + head
// with the general kernels' chunk slots (for packed input the Geo's cstart).
struct Emit {
    uint8_t *keep;
    __nv_bfloat16 *sin, *unew;
};

// Byte layout of one package: stride between slots; [-W | Qt] panels of d_k / 64
// at wq + panel * wq_panel (-W rows first, Qt rows at + panel bytes), T at t, P at
// p, the vector (f0[64] = exp(gamma_C - gamma_r) n_r, then exp(gamma_C)) at vec.
// Tiles are bf16 rows of 128 bytes with the 128-byte swizzle (16-byte chunk index
// XOR row % 8).
struct PkLayout {
    uint32_t stride, wq, wq_panel, panel, t, p, vec;
};
PkLayout package_layout(const Geo &g);

// Workspace it needs: control words, packed order, package ring.  sms <= 0 sizes
// for an upper bound on the SM count.
size_t workspace_bytes(const Geo &g, int sms);

// o and hT may be null (not written).
cudaError_t fwd(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                const __nv_bfloat16 *v, const __nv_bfloat16 *beta, const float *gate,
                const float *h0, __nv_bfloat16 *o, float *hT, void *ws, size_t ws_bytes,
                uint32_t *status, cudaStream_t st, const Emit *emit = nullptr);

}  // namespace coop
}  // namespace gdn
