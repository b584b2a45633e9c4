// Host launchers of the general (fp32 CUDA-core) chunk kernels.
#pragma once

#include "common.cuh"

namespace gdn {
namespace gen {

// Workspace arrays, all float32, indexed by slot = chunk_slot * H + head.
struct Ws {
    float *Kn, *Qn, *W;        // [slots][C][dk]  normalised K, Q; WY factor W
    float *U, *Unew;           // [slots][C][dv]
    float *gam;                // [slots][C]      within-chunk cumulative log-gate
    float *eb;                 // [slots][C]      step size of each token (beta, or Longhorn's)
    float *Sin;                // [slots][dk][dv] state entering the chunk
    float *dSo, *dUn;          // backward: dS leaving the chunk, dUnew
    float *dQ, *dK, *dW;       // backward scratch [slots][C][dk]
    float *P;                  // [slots][C][C]   lower(Q K^T o D), diagonal kept
    float *aux;                // backward [slots][4C + 4]: row sums, <dS_out, S_in>, d gamma / d beta partials
    float *M3;                 // backward [slots][3][C][C]: dP o D, (I + A)^-1, dKK
};

template <class Tin>
cudaError_t fwd(const Geo &g, const Tin *q, const Tin *k, const Tin *v, const Tin *beta,
                const float *gate, const float *h0, Tin *o, float *hT, const Ws &w,
                cudaStream_t st);

template <class Tin>
cudaError_t bwd(const Geo &g, const Tin *q, const Tin *k, const Tin *v, const Tin *beta,
                const float *gate, const float *h0, const Tin *dO, const float *dhT, Tin *dq,
                Tin *dk, Tin *dv, Tin *dbeta, float *dg, float *dh0, const Ws &w,
                cudaStream_t st);

}  // namespace gen
}  // namespace gdn
