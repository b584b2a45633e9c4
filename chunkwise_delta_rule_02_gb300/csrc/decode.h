// Launcher of the recurrent decode step (decode.cu).
#pragma once

#include "common.cuh"

namespace gdn {
namespace dec {

struct Args {
    int N, H, dk, dv;          // sequences, heads, head dims (<= kMaxD)
    int l2norm;
    int longhorn;              // step size beta / (1 + beta k^T k) instead of beta
    float scale, eps;
    const float *gate;         // [N][H] log-gate or null (alpha = 1)
    const float *state_in;     // [N][H][dk][dv] or null (zero state)
    float *state_out;          // [N][H][dk][dv]; may equal state_in
};

template <class Tin>
cudaError_t step(const Args &a, const Tin *q, const Tin *k, const Tin *v, const Tin *beta, Tin *o,
                 cudaStream_t st);

}  // namespace dec
}  // namespace gdn
