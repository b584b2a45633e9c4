// Batched affine map of states, out_i = A_i S_i + B_i (fp32), the composition
// step of the sequence-split forward: the state leaving a shard of a sequence is
// an affine function of the state entering it (the recurrence is linear in the
// state), and a rank composes the maps of the shards before its own.
#include "affine.h"

namespace gdn {
namespace aff {
namespace {

constexpr int TILE = 64;    // output tile (rows of A / S's columns)
constexpr int KT = 16;      // reduction step

// One CTA per 64 x 64 output tile of one item; 256 threads, each a 4 x 4 block.
__global__ void __launch_bounds__(256) k_state_affine(const float *__restrict__ A,
                                                      const float *__restrict__ S,
                                                      const float *__restrict__ B,
                                                      float *__restrict__ out, int dk, int dv)
{
    __shared__ float sA[KT][TILE + 4];   // A tile, transposed: sA[m][r]
    __shared__ float sS[KT][TILE + 4];   // S tile: sS[m][c]
    const size_t item = blockIdx.z;
    const int r0 = blockIdx.y * TILE, c0 = blockIdx.x * TILE;
    const float *Ai = A + item * (size_t)dk * dk;
    const float *Si = S + item * (size_t)dk * dv;
    const int tr = (threadIdx.x >> 4) * 4, tc = (threadIdx.x & 15) * 4;
    float acc[4][4] = {};
    for (int m0 = 0; m0 < dk; m0 += KT) {
        for (int e = threadIdx.x; e < KT * TILE; e += 256) {
            const int m = e % KT, r = e / KT;          // A read along its rows
            sA[m][r] = (r0 + r < dk && m0 + m < dk) ? Ai[(size_t)(r0 + r) * dk + m0 + m] : 0.f;
            const int mm = e / TILE, c = e % TILE;     // S read along its rows
            sS[mm][c] = (m0 + mm < dk && c0 + c < dv) ? Si[(size_t)(m0 + mm) * dv + c0 + c] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < KT; ++m) {
            float a[4], s[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = sA[m][tr + i]; s[i] = sS[m][tc + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], s[j], acc[i][j]);
        }
        __syncthreads();
    }
    const float *Bi = B ? B + item * (size_t)dk * dv : nullptr;
    float *oi = out + item * (size_t)dk * dv;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + tr + i;
        if (r >= dk) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + tc + j;
            if (c >= dv) continue;
            const size_t idx = (size_t)r * dv + c;
            oi[idx] = acc[i][j] + (Bi ? Bi[idx] : 0.f);
        }
    }
}

}  // namespace

cudaError_t state_affine(const float *A, const float *S, const float *B, float *out, int count,
                         int dk, int dv, cudaStream_t st)
{
    if (count == 0) return cudaSuccess;
    dim3 grid((dv + TILE - 1) / TILE, (dk + TILE - 1) / TILE, count);
    k_state_affine<<<grid, 256, 0, st>>>(A, S, B, out, dk, dv);
    return cudaPeekAtLastError();
}

}  // namespace aff
}  // namespace gdn
