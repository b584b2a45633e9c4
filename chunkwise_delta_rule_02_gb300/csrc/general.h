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
    // bf16 copies for the tcgen05 per-chunk backward (null otherwise): when set, the
    // staged scans write these instead of Sin / Unew (forward scan) and dSo / dUn
    // (backward scan), with the rows past a chunk's end as zeros
    __nv_bfloat16 *Sin_b, *dSo_b;   // [slots][dk][dv]
    __nv_bfloat16 *Un_b, *dUn_b;    // [slots][C][dv]
    // when keep is set (bwd_uses_coop), the backward recomputes through the cooperative
    // forward instead: its workspace (coop_ws, coop_bytes), every chunk's package in
    // keep[slot], and the bf16 arrays above; the float arrays are then not used
    uint8_t *keep;
    void *coop_ws;
    size_t coop_bytes;
    // keep, Sin_b and Un_b hold a cooperative forward's output already (the caller's
    // saved buffer): the backward starts at the reverse scan
    bool saved;
};

template <class Tin>
cudaError_t fwd(const Geo &g, const Tin *q, const Tin *k, const Tin *v, const Tin *beta,
                const float *gate, const float *h0, Tin *o, float *hT, const Ws &w,
                cudaStream_t st);

// Whether gdn_chunk_bwd takes the tcgen05 per-chunk backward for this call.
bool bwd_uses_tc(const Geo &g, int dtype, const void *q, const void *k, const void *v, const void *dO);

// Whether that backward gets its states, Unew and the reverse scan's operands from the
// cooperative forward (bf16, d 128, chunk 64, a device that runs it; not with
// GDN_BWD_RECOMPUTE=1, GDN_FORCE_GENERAL=1 or GDN_BWD_STAGED=1): kernels k_coop_fwd,
// k_bscan_pk, k_bwd_tc.
bool bwd_uses_coop(const Geo &g, int dtype);

template <class Tin>
cudaError_t bwd(const Geo &g, const Tin *q, const Tin *k, const Tin *v, const Tin *beta,
                const float *gate, const float *h0, const Tin *dO, const float *dhT, Tin *dq,
                Tin *dk, Tin *dv, Tin *dbeta, float *dg, float *dh0, const Ws &w,
                cudaStream_t st);

}  // namespace gen
}  // namespace gdn
