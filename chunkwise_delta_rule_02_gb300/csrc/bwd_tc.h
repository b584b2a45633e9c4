// Host side of the tcgen05 per-chunk backward (bf16, d_k = d_v = 128, C = 64).
#pragma once

#include "common.cuh"

namespace gdn {
namespace btc {

// Whether the tcgen05 per-chunk backward takes this geometry and dtype.
bool supports(const Geo &g, int dtype);

// dq, dk, dv, dbeta, dg of every chunk from the raw inputs and the scans' bf16
// outputs: S_in and dS_out [slots][dk][dv], Unew and dUnew [slots][C][dv]
// (slot = chunk slot * H + head; rows past a chunk's end zero).  All token
// arrays [B][H][T][128] bf16, 16-byte aligned.
cudaError_t grads(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                  const __nv_bfloat16 *beta, const float *gate, const __nv_bfloat16 *dO,
                  const __nv_bfloat16 *Sin, const __nv_bfloat16 *dSo, const __nv_bfloat16 *Un,
                  const __nv_bfloat16 *dUn, __nv_bfloat16 *dq, __nv_bfloat16 *dk, __nv_bfloat16 *dv,
                  __nv_bfloat16 *dbeta, float *dg, cudaStream_t st);

}  // namespace btc
}  // namespace gdn
