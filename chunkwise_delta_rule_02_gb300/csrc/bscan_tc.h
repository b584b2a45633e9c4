// Host side of the tcgen05 reverse dS scan of the backward (bf16, d_k = d_v = 128,
// C = 64) over the cooperative forward's packages.
#pragma once

#include "common.cuh"
#include "fast.h"

namespace gdn {
namespace bsc {

// Whether it takes this geometry and dtype (a device with the tensor-map encoder).
bool supports(const Geo &g, int dtype);

// Per chunk, from the last chunk of each (sequence, head) to the first, with the
// packages in keep[slot] (layout pk), the raw keys k and dO ([B][H][T][128] bf16,
// packed input [1][H][T][128]):
//   dS_out[slot] = the dS the chunk receives (bf16 [dk][dv]),
//   dUnew[slot] = P^T (scale dO) + diag(f) K dS_out (bf16 [C][dv], rows past the
//   chunk's end zero),
//   dS <- exp(gamma_C) dS + Qt^T (scale dO) - W^T dUnew;
// dS starts at dhT (or 0) and ends in dh0 (if not null).  slot = chunk slot * H +
// head, chunk slots as the general kernels number them (packed: g.cstart).
cudaError_t scan(const Geo &g, const __nv_bfloat16 *k, const __nv_bfloat16 *dO, const float *dhT,
                 float *dh0, const uint8_t *keep, const coop::PkLayout &pk, __nv_bfloat16 *dSo,
                 __nv_bfloat16 *dUn, cudaStream_t st);

}  // namespace bsc
}  // namespace gdn
