// Device helpers shared by the fused kernels' chunk preparation: bf16 pair
// handling, 2^x, tf32 conversion, a 16x8x8 tf32 tensor-core tile, and the
// 64x64 unit-lower-triangular inverse of the UT transform.
#pragma once

#include <stdint.h>

#include "sm100.cuh"

namespace gdn {
namespace prep {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t scale_pair(uint32_t w, float s)
{
    return sm100::pack_bf16(bf_lo(w) * s, bf_hi(w) * s);
}

// 2^x on the special-function unit (results may flush to 0)
__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// D += A B for one 16x8x8 tile (A row-major 16x8, B 8x8, tf32 in, fp32 accumulate)
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4],
                                                const uint32_t (&b)[2])
{
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc (32 x 32 tile at m0, n0) += A B over k in [0, K), K % 8 == 0, on the tensor
// cores in tf32 (operands rounded to 10-bit mantissas, fp32 accumulation), from fp32
// accessors A(m, k), B(k, n).
template <class FA, class FB>
__device__ __forceinline__ void tile_tf32(float (&acc)[2][4][4], FA A, FB B, int m0, int n0, int K)
{
    const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
    for (int k0 = 0; k0 < K; k0 += 8) {
        uint32_t a[2][4], b[4][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = m0 + 16 * h + gq;
            a[h][0] = tf32(A(m, k0 + t));
            a[h][1] = tf32(A(m + 8, k0 + t));
            a[h][2] = tf32(A(m, k0 + t + 4));
            a[h][3] = tf32(A(m + 8, k0 + t + 4));
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            b[jj][0] = tf32(B(k0 + t, n0 + 8 * jj + gq));
            b[jj][1] = tf32(B(k0 + t + 4, n0 + 8 * jj + gq));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) mma_tf32_16x8x8(acc[h][jj], a[h], b[jj]);
    }
}

// X = (I + A)^-1 for a strictly lower triangular 64 x 64 A (fp32, row stride
// AST floats), called by the 128 threads of one warpgroup (warp q4 = 0..3 in the
// group, lane = lane id).  Diagonal 16 x 16 blocks by substitution (warp w:
// block w, lane c: column c); then block column j (warp j):
//     X_ij = -sum_{m=j}^{i-1} (X_ii A_im) X_mj,
// as 16 x 16 products on the tensor cores (tf32 mma.sync, fp32 accumulate) with
// the product X_ii A_im kept in registers as the A operand of the next one.
// Synchronises the warpgroup (named barrier bar_id) between the two phases and
// at the end; X's strictly upper part is not written.
template <int AST>
__device__ __forceinline__ void solve_unit_lower_64(const float *Af, float *Xf, int lane, int q4,
                                                    int bar_id)
{
    {
        const int base = 16 * q4, c = lane & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int l = 0; l < i; ++l) acc = fmaf(-Af[(base + i) * AST + base + l], x[l], acc);
            x[i] = (i < c) ? 0.f : acc;
        }
        if (lane < 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) Xf[(base + i) * AST + base + c] = x[i];
        }
    }
    sm100::named_bar(bar_id, 128);
    const int g8 = lane >> 2, t4 = lane & 3;
    if (q4 < 3) {
        const int j = q4;
        for (int i = j + 1; i < 4; ++i) {
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int m = j; m < i; ++m) {
                float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float *xa = Xf + (16 * i) * AST + 16 * i + 8 * ks;
                    uint32_t a[4] = {tf32(xa[g8 * AST + t4]), tf32(xa[(g8 + 8) * AST + t4]),
                                     tf32(xa[g8 * AST + t4 + 4]), tf32(xa[(g8 + 8) * AST + t4 + 4])};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float *ab = Af + (16 * i + 8 * ks) * AST + 16 * m + 8 * nt + g8;
                        uint32_t b[2] = {tf32(ab[t4 * AST]), tf32(ab[(t4 + 4) * AST])};
                        mma_tf32_16x8x8(z[nt], a, b);
                    }
                }
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t a[4] = {tf32(z[ks][0]), tf32(z[ks][2]), tf32(z[ks][1]), tf32(z[ks][3])};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float *xb = Xf + (16 * m + 8 * ks) * AST + 16 * j + 8 * nt + g8;
                        uint32_t b[2] = {tf32(xb[(2 * t4) * AST]), tf32(xb[(2 * t4 + 1) * AST])};
                        mma_tf32_16x8x8(acc[nt], a, b);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                float *xo = Xf + (16 * i + g8) * AST + 16 * j + 8 * nt + 2 * t4;
                xo[0] = -acc[nt][0];
                xo[1] = -acc[nt][1];
                xo[8 * AST] = -acc[nt][2];
                xo[8 * AST + 1] = -acc[nt][3];
            }
            __syncwarp();
        }
    }
    sm100::named_bar(bar_id, 128);
}

// The same inverse computed in one buffer, for a 16 NB x 16 NB matrix (NB = 4:
// 64 x 64, NB = 2: 32 x 32).  On entry AX holds the strictly lower
// triangular A below its diagonal (fp32, row stride AST floats; what lies on and
// above the diagonal is ignored).  On return the strictly lower blocks still hold
// A, and X is stored transposed on and above the diagonal:
//     AX[c * AST + r] = X[r][c]   for every r >= c,
// with each diagonal 16 x 16 block rewritten in full as X_ii^T (unit diagonal,
// zeros for the upper part of X_ii).  The off-diagonal blocks X_ij (i > j) go to
// block (j, i); nothing reads or writes A's blocks after the diagonal phase, so
// the column-parallel schedule of solve_unit_lower_64 carries over unchanged.
// Called by the 128 threads of one warpgroup (warps q4 >= NB idle in the diagonal
// phase, warps q4 >= NB - 1 in the off-diagonal one); synchronises it (named
// barrier bar_id) between the phases and at the end.
template <int AST, int NB = 4>
__device__ __forceinline__ void solve_unit_lower_packed(float *AX, int lane, int q4, int bar_id)
{
    static_assert(NB >= 1 && NB <= 4, "16 x 16 blocks, one warp each");
    if (q4 < NB) {
        const int base = 16 * q4, c = lane & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
            for (int l = 0; l < i; ++l) acc = fmaf(-AX[(base + i) * AST + base + l], x[l], acc);
            x[i] = (i < c) ? 0.f : acc;
        }
        __syncwarp();   // every lane has read A_ii before its block is overwritten
        if (lane < 16) {
            if constexpr (AST % 4 == 0) {
                float4 *dst = reinterpret_cast<float4 *>(AX + (base + c) * AST + base);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
            } else {
                static_assert(AST % 2 == 0, "rows must stay 8-byte aligned");
                float2 *dst = reinterpret_cast<float2 *>(AX + (base + c) * AST + base);
#pragma unroll
                for (int q = 0; q < 8; ++q) dst[q] = make_float2(x[2 * q], x[2 * q + 1]);
            }
        }
    }
    sm100::named_bar(bar_id, 128);
    const int g8 = lane >> 2, t4 = lane & 3;
    if (q4 < NB - 1) {
        const int j = q4;
        for (int i = j + 1; i < NB; ++i) {
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int m = j; m < i; ++m) {
                // Z = X_ii A_im
                float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float *xa = AX + (16 * i + 8 * ks) * AST + 16 * i;   // X_ii[r][8ks + k] = xa[k * AST + r]
                    uint32_t a[4] = {tf32(xa[t4 * AST + g8]), tf32(xa[t4 * AST + g8 + 8]),
                                     tf32(xa[(t4 + 4) * AST + g8]), tf32(xa[(t4 + 4) * AST + g8 + 8])};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float *ab = AX + (16 * i + 8 * ks) * AST + 16 * m + 8 * nt + g8;
                        uint32_t b[2] = {tf32(ab[t4 * AST]), tf32(ab[(t4 + 4) * AST])};
                        mma_tf32_16x8x8(z[nt], a, b);
                    }
                }
                // acc += Z X_mj, with Z's accumulator layout reused as the A operand
                // (k order permuted: k = t4 <-> column 2 t4, k = t4 + 4 <-> 2 t4 + 1)
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    uint32_t a[4] = {tf32(z[ks][0]), tf32(z[ks][2]), tf32(z[ks][1]), tf32(z[ks][3])};
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const float2 xb = *reinterpret_cast<const float2 *>(
                            AX + (16 * j + 8 * nt + g8) * AST + 16 * m + 8 * ks + 2 * t4);
                        uint32_t b[2] = {tf32(xb.x), tf32(xb.y)};
                        mma_tf32_16x8x8(acc[nt], a, b);
                    }
                }
            }
            // X_ij = -acc, transposed into block (j, i)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                float *xo = AX + (16 * j + 8 * nt + 2 * t4) * AST + 16 * i + g8;
                xo[0] = -acc[nt][0];
                xo[AST] = -acc[nt][1];
                xo[8] = -acc[nt][2];
                xo[AST + 8] = -acc[nt][3];
            }
            __syncwarp();
        }
    }
    sm100::named_bar(bar_id, 128);
}

template <int AST>
__device__ __forceinline__ void solve_unit_lower_64_packed(float *AX, int lane, int q4, int bar_id)
{
    solve_unit_lower_packed<AST, 4>(AX, lane, q4, bar_id);
}

}  // namespace prep
}  // namespace gdn
