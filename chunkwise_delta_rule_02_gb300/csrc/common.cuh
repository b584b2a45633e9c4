// Shared host/device definitions of libgdn_gb300: problem geometry, chunk
// indexing, workspace layout, dtype conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kMaxD = 256;       // largest head dim supported (tcgen05 kernels: 128)
constexpr int kMaxC = 64;        // largest chunk

// Geometry of one call, passed by value to every kernel.
struct Geo {
    int B, H, T, dk, dv, C;
    int N;             // sequences: B (fixed length) or num_seqs (packed)
    int NC;            // chunk slots per head (upper bound on chunks)
    int varlen;        // 1: packed, cu/cstart valid
    int l2norm;
    int longhorn;      // step size beta / (1 + beta k^T k) instead of beta
    float scale, eps;
    const int32_t *cu;      // device [N+1] token offsets (packed)
    const int32_t *cstart;  // device [N+1] first chunk slot of each sequence (packed)
    uint32_t *status;       // device status word of the call (see kStatus*)
};

// Chunk slot j -> (batch row b, first token t0 on that row's time axis, rows).
// Returns false for an unused slot (packed input has fewer real chunks than slots).
__device__ __forceinline__ bool chunk_of(const Geo &g, int j, int &b, int &t0, int &len,
                                         int &seq, int &local)
{
    if (!g.varlen) {
        int nc = (g.T + g.C - 1) / g.C;
        b = j / nc;
        local = j - b * nc;
        seq = b;
        t0 = local * g.C;
        len = min(g.C, g.T - t0);
        return b < g.B && len > 0;
    }
    // binary search: last s with cstart[s] <= j
    int lo = 0, hi = g.N;   // cstart[N] = total chunks
    if (j >= g.cstart[g.N]) return false;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (g.cstart[mid] <= j) lo = mid; else hi = mid;
    }
    seq = lo;
    b = 0;
    local = j - g.cstart[lo];
    t0 = g.cu[lo] + local * g.C;
    len = min(g.C, g.cu[lo + 1] - t0);
    return len > 0;
}

// Sequence s -> (batch row, first token, length, first chunk slot, chunk count).
__device__ __forceinline__ void seq_of(const Geo &g, int s, int &b, int &t0, int &L, int &j0,
                                       int &nch)
{
    if (!g.varlen) {
        b = s; t0 = 0; L = g.T;
        nch = (g.T + g.C - 1) / g.C;
        j0 = s * nch;
    } else {
        b = 0; t0 = g.cu[s]; L = g.cu[s + 1] - t0;
        if (L < 0) L = 0;
        j0 = g.cstart[s];
        nch = g.cstart[s + 1] - j0;
    }
}

__device__ __forceinline__ float ld_in(const float *p) { return *p; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Device status word (first word of every workspace).  kStatusPositiveGate: a
// log-gate g > 0 was read (alpha > 1, outside the documented domain: the chunk
// form's decay ratios exp(gamma_r - gamma_i) are then growth factors).
enum : uint32_t { kStatusOk = 0, kStatusTimeout = 1u, kStatusBadOffsets = 2u, kStatusPositiveGate = 4u };

__device__ __forceinline__ void raise_status(uint32_t *status, uint32_t bit)
{
    if (status) atomicOr(status, bit);
}

}  // namespace gdn
