// General chunk kernels: any head dim up to 256, chunk 16/32/64, float32 or
// bfloat16 inputs, gated or not, packed or not.
//
// These kernels carry the fp32 workload (whose 1e-4 tolerance tensor-core
// operands cannot meet), every shape the tcgen05 kernels do not take, and the
// backward.  They follow the chunk form of "Parallelizing Linear Transformers
// with the Delta Rule over Sequence Length" (WY / UT representation, chunk-state
// scan) with the gates of "Gated DeltaNet" folded in as within-chunk cumulative
// log-decays:
//   prep  : per chunk, parallel       normalise q,k; gamma; A; T; W; U; P
//   scan  : per (seq, head, 64-column dv-slice) Unew = U - W S; S <- Gamma_C S + Kt^T Unew
//   out   : per chunk, parallel       O = diag(Gamma) Q S + P Unew
// and the backward (chunk states recomputed by prep + scan, then):
//   bscan : per (seq, head, dv-slice), last chunk first:
//           dUnew = P^T dO + Kt dS;  dS <- Gamma_C dS + (Gamma Q)^T dO - W^T dUnew
//   bbig  : per chunk, parallel       the three products with the d_k x d_v states
//   bchunk: per chunk, parallel       the C x C part: solve adjoint, gate / beta terms
//   bgrad : per chunk, parallel       the C x d part: dq, dk, dv, dg, the norm chain rule.
// (P = lower(Q K^T o D) with the diagonal kept; D_ri = exp(gamma_r - gamma_i).)
//
// Every matrix product is a register-tiled block product (rgemm) -- in the
// kernels with bf16 inputs, a warp-level tensor-core product (mgemm) instead,
// except for the two small products of the solve's adjoint and the output
// kernel: each thread
// owns TM consecutive rows and TN columns spread across the threads, so an
// operand that is contiguous along the output columns is read coalesced (from
// L1) or without bank conflicts (from shared memory).  Operands that would be
// read across rows instead are first staged in shared memory with an odd row
// stride.
//
// For bf16 inputs with power-of-two head dims 32..128 and chunks of 32 or 64
// the staged kernels (k_prep_st, k_scan_st, k_out_st, k_bscan_st, k_bbig_st,
// k_bgrad_st and the staged branch of k_bchunk) replace these: each chunk's operands are
// loaded once with batched 16-byte loads, rounded to bf16 into row-major
// shared-memory tiles with rows padded by 8 elements, and multiplied on the
// tensor cores with ldmatrix fragments and 32 x 32 warp tiles (tile_mma).  The
// fp32 path keeps the kernels above.
#include <type_traits>

#include "common.cuh"
#include "general.h"

#include <stdlib.h>

#include "bscan_tc.h"
#include "bwd_tc.h"
#include "fast.h"
#include "prep_math.cuh"

namespace gdn {
namespace gen {

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// St(m, n, sum_k A(m, k) B(k, n)) for m < M, n < N.  Thread tile: rows
// m0 .. m0 + TM - 1 and columns tn, tn + nt, .., tn + (TN - 1) nt, where nt is
// the number of column tiles.  Accessors are called only inside the bounds.
template <int TM, int TN, class FA, class FB, class FS>
__device__ __forceinline__ void rgemm(int M, int N, int K, FA A, FB B, FS St)
{
    const int mt = (M + TM - 1) / TM, nt = (N + TN - 1) / TN;
    for (int t = threadIdx.x; t < mt * nt; t += blockDim.x) {
        const int m0 = (t / nt) * TM, tn = t - (t / nt) * nt;
        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
        if (m0 + TM <= M && tn + (TN - 1) * nt < N) {
#pragma unroll 2
            for (int k = 0; k < K; ++k) {
                float a[TM], b[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = A(m0 + i, k);
#pragma unroll
                for (int j = 0; j < TN; ++j) b[j] = B(k, tn + j * nt);
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
        } else {
            for (int k = 0; k < K; ++k) {
                float a[TM], b[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = (m0 + i < M) ? A(m0 + i, k) : 0.f;
#pragma unroll
                for (int j = 0; j < TN; ++j) b[j] = (tn + j * nt < N) ? B(k, tn + j * nt) : 0.f;
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j)
                if (m0 + i < M && tn + j * nt < N) St(m0 + i, tn + j * nt, acc[i][j]);
    }
}

// bf16 pair for a tensor-core fragment: lo in the low half
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// brings [p, p + bytes) into L2 ahead of use (p 16-byte aligned, bytes % 16 == 0)
__device__ __forceinline__ void l2_prefetch(const void *p, size_t bytes)
{
    if (bytes > 0)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"((uint32_t)bytes) : "memory");
}

// For e in [0, n): put(e, get(e)), every thread issuing eight loads before it stores any,
// so that their latencies overlap (get reads global memory, put writes shared memory).
template <class FG, class FP>
__device__ __forceinline__ void batched_copy(int n, FG get, FP put)
{
    constexpr int VB = 8;
    for (int base = threadIdx.x; base < n; base += blockDim.x * VB) {
        float x[VB];
#pragma unroll
        for (int u = 0; u < VB; ++u) {
            const int e = base + u * blockDim.x;
            x[u] = e < n ? get(e) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < VB; ++u) {
            const int e = base + u * blockDim.x;
            if (e < n) put(e, x[u]);
        }
    }
}

// D += A B for one 16 x 8 x 16 tile: A row-major, B column-major, bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2])
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// The block product of rgemm on the tensor cores (warp-level mma, bf16 operands
// rounded from the accessors' fp32 values, fp32 accumulation): each warp owns
// 16 x 8 NT output tiles in turn.  Used by the backward when the inputs are bf16,
// where the 2e-2 tolerance leaves room for bf16 operands.
template <int NT, class FA, class FB, class FS>
__device__ __forceinline__ void mgemm(int M, int N, int K, FA A, FB B, FS St)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int mt = (M + 15) / 16, ntl = (N + 8 * NT - 1) / (8 * NT);
    for (int tile = warp; tile < mt * ntl; tile += nw) {
        const int m0 = (tile / ntl) * 16, n0 = (tile - (tile / ntl) * ntl) * 8 * NT;
        float acc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        const bool mn_in = m0 + 16 <= M && n0 + 8 * NT <= N;
        for (int k0 = 0; k0 < K; k0 += 16) {
            uint32_t a[4];
            uint32_t b[NT][2];
            if (mn_in && k0 + 16 <= K) {
                const int ka = k0 + 2 * t;
                a[0] = bf16x2(A(m0 + g, ka), A(m0 + g, ka + 1));
                a[1] = bf16x2(A(m0 + g + 8, ka), A(m0 + g + 8, ka + 1));
                a[2] = bf16x2(A(m0 + g, ka + 8), A(m0 + g, ka + 9));
                a[3] = bf16x2(A(m0 + g + 8, ka + 8), A(m0 + g + 8, ka + 9));
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int n = n0 + 8 * j + g;
                    b[j][0] = bf16x2(B(ka, n), B(ka + 1, n));
                    b[j][1] = bf16x2(B(ka + 8, n), B(ka + 9, n));
                }
            } else {
                auto ga = [&](int m, int k) { return (m < M && k < K) ? A(m, k) : 0.f; };
                auto gb = [&](int k, int n) { return (k < K && n < N) ? B(k, n) : 0.f; };
                const int ka = k0 + 2 * t;
                a[0] = bf16x2(ga(m0 + g, ka), ga(m0 + g, ka + 1));
                a[1] = bf16x2(ga(m0 + g + 8, ka), ga(m0 + g + 8, ka + 1));
                a[2] = bf16x2(ga(m0 + g, ka + 8), ga(m0 + g, ka + 9));
                a[3] = bf16x2(ga(m0 + g + 8, ka + 8), ga(m0 + g + 8, ka + 9));
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int n = n0 + 8 * j + g;
                    b[j][0] = bf16x2(gb(ka, n), gb(ka + 1, n));
                    b[j][1] = bf16x2(gb(ka + 8, n), gb(ka + 9, n));
                }
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) mma_bf16_16816(acc[j], a, b[j]);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int m = m0 + g, n = n0 + 8 * j + 2 * t;
            if (m < M && n < N) St(m, n, acc[j][0]);
            if (m < M && n + 1 < N) St(m, n + 1, acc[j][1]);
            if (m + 8 < M && n < N) St(m + 8, n, acc[j][2]);
            if (m + 8 < M && n + 1 < N) St(m + 8, n + 1, acc[j][3]);
        }
    }
}

// Block product for the backward: tensor cores for bf16 inputs, fp32 otherwise.
template <class Tin, int TM, int TN, class FA, class FB, class FS>
__device__ __forceinline__ void bgemm(int M, int N, int K, FA A, FB B, FS St)
{
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value)
        mgemm<4>(M, N, K, A, B, St);
    else
        rgemm<TM, TN>(M, N, K, A, B, St);
}

// X = (I + A)^-1 diag(d) for the unit lower triangular I + A: A strictly lower in rows
// and columns [0, len) (row stride ld, other entries ignored), d the column scales (or
// null: none).  X is written on and below the diagonal and zero above it, rows and
// columns [0, len).  Blocked by 16: the diagonal blocks Y_b = (I + A_bb)^-1 by
// substitution (a thread per column), then block row b after block row, every block
// left of the diagonal at once, X_bc = -Y_b sum_{k=c..b-1} A_bk X_kc (a thread per
// column, the block's 16 rows in registers), all in fp32.  Every thread of the block
// calls it (barriers inside).
__device__ __noinline__ void unit_lower_solve(const float *A, float *X, const float *d, int len, int ld)
{
    const int nb = (len + 15) >> 4;
    const int tid = threadIdx.x, nt = blockDim.x;
    for (int t = tid; t < nb * 16; t += nt) {
        const int b = t >> 4, c = (b << 4) + (t & 15);
        if (c >= len) continue;
        const int r1 = min(len, (b + 1) << 4);
        for (int r = b << 4; r < r1; ++r) {
            float x;
            if (r < c) {
                x = 0.f;
            } else if (r == c) {
                x = 1.f;
            } else {
                float s = 0.f;
                for (int i = c; i < r; ++i) s = fmaf(A[r * ld + i], X[i * ld + c], s);
                x = -s;
            }
            X[r * ld + c] = x;
        }
    }
    for (int t = tid; t < len * len; t += nt) {
        const int r = t / len, c = t - r * len;
        if ((c >> 4) > (r >> 4)) X[r * ld + c] = 0.f;
    }
    __syncthreads();
    for (int b = 1; b < nb; ++b) {
        const int r0 = b << 4, rows = min(16, len - r0);
        for (int c = tid; c < r0; c += nt) {
            float z[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) z[rr] = 0.f;
            for (int i = c; i < r0; ++i) {
                const float xi = X[i * ld + c];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr)
                    if (rr < rows) z[rr] = fmaf(A[(r0 + rr) * ld + i], xi, z[rr]);
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                if (rr < rows) {
                    float s = 0.f;
#pragma unroll
                    for (int m = 0; m <= rr; ++m) s = fmaf(X[(r0 + rr) * ld + r0 + m], z[m], s);
                    X[(r0 + rr) * ld + c] = -s;
                }
            }
        }
        __syncthreads();
    }
    if (d) {
        for (int t = tid; t < len * len; t += nt) {
            const int r = t / len, c = t - r * len;
            if (c <= r) X[r * ld + c] *= d[c];
        }
    }
}

// ----------------------------------------------------------------------------- prep
template <class Tin>
__global__ void __launch_bounds__(256) k_prep(Geo g, const Tin *__restrict__ q,
                                              const Tin *__restrict__ k,
                                              const Tin *__restrict__ v,
                                              const Tin *__restrict__ beta,
                                              const float *__restrict__ gate, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv, LK = dk + 1, LC = C + 1;
    extern __shared__ float sm[];
    float *sK = sm;                                 // [C][LK] normalised keys
    float *sQ = sK + C * LK;                        // [C][LK] normalised queries, then V [C][dv]
    float *sA = sQ + C * (LK > dv ? LK : dv);       // [C][LC]
    float *sT = sA + C * LC;                        // [C][LC]
    float *sb = sT + C * LC;                        // [C] step sizes (beta, or Longhorn's)
    float *sg = sb + C;                             // [C] gamma
    float *sG = sg + C;                             // [C] exp(gamma)
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;

    for (int r = warp; r < len; r += nw) {
        const Tin *kr = k + (row + r) * dk;
        const Tin *qr = q + (row + r) * dk;
        float sk = 0.f, sq = 0.f;
        for (int c = lane; c < dk; c += 32) {
            float x = ld_in(kr + c), y = ld_in(qr + c);
            sk = fmaf(x, x, sk);
            sq = fmaf(y, y, sq);
        }
        sk = warp_sum(sk);
        sq = warp_sum(sq);
        float rk = g.l2norm ? rsqrtf(sk + g.eps) : 1.f;
        float rq = g.l2norm ? rsqrtf(sq + g.eps) : 1.f;
        if (lane == 0) {
            // the token's step size: beta, or Longhorn's beta / (1 + beta k^T k) with
            // k^T k = |k|^2 rk^2 of the key the update uses
            float bt = ld_in(beta + row + r);
            if (g.longhorn) bt = bt / fmaf(bt, sk * rk * rk, 1.f);
            sb[r] = bt;
            w.eb[slot * C + r] = bt;
        }
        for (int c = lane; c < dk; c += 32) {
            float x = ld_in(kr + c) * rk, y = ld_in(qr + c) * rq;
            sK[r * LK + c] = x;
            sQ[r * LK + c] = y;
            w.Kn[slot * C * dk + r * dk + c] = x;
            w.Qn[slot * C * dk + r * dk + c] = y;
        }
    }
    if (warp == 0) {
        // within-chunk cumulative log-gate, two rows per lane (C <= 64)
        float x0 = (gate && lane < len) ? gate[row + lane] : 0.f;
        float x1 = (gate && lane + 32 < len) ? gate[row + lane + 32] : 0.f;
        if (__any_sync(0xffffffffu, x0 > 0.f || x1 > 0.f) && lane == 0)
            raise_status(g.status, kStatusPositiveGate);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (lane >= o) { x0 += y0; x1 += y1; }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        if (lane < len) {
            sg[lane] = x0;
            sG[lane] = expf(x0);
            w.gam[slot * C + lane] = x0;
        }
        if (lane + 32 < len) {
            sg[lane + 32] = x1;
            sG[lane + 32] = expf(x1);
            w.gam[slot * C + lane + 32] = x1;
        }
    }
    __syncthreads();
    // A = strict_lower(diag(beta) (K K^T o D)),  P = lower(Q K^T o D)
    bgemm<Tin, 4, 4>(len, len, dk, [&](int m, int kk) { return sK[m * LK + kk]; },
                [&](int kk, int n) { return sK[n * LK + kk]; },
                [&](int m, int n, float s) {
                    sA[m * LC + n] = (n < m) ? sb[m] * s * expf(sg[m] - sg[n]) : 0.f;
                });
    float *Pg = w.P + slot * C * C;
    bgemm<Tin, 4, 4>(len, len, dk, [&](int m, int kk) { return sQ[m * LK + kk]; },
                [&](int kk, int n) { return sK[n * LK + kk]; },
                [&](int m, int n, float s) { Pg[m * C + n] = (n <= m) ? s * expf(sg[m] - sg[n]) : 0.f; });
    __syncthreads();
    // T = (I + A)^-1 diag(beta)
    bool solved = false;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        if (C == 64) {
            // blocked solve (16 x 16 diagonal blocks by substitution, the rest on the
            // tensor cores in tf32) over the full 64 x 64, so A is zero outside the chunk
            for (int idx = threadIdx.x; idx < 64 * 64; idx += blockDim.x) {
                const int r = idx >> 6, c = idx & 63;
                if (r >= len || c >= len) sA[r * 65 + c] = 0.f;
            }
            __syncthreads();
            if (warp < 4) prep::solve_unit_lower_64<65>(sA, sT, lane, warp, 1);
            __syncthreads();
            for (int idx = threadIdx.x; idx < 64 * 64; idx += blockDim.x) {
                const int r = idx >> 6, c = idx & 63;
                sT[r * 65 + c] = (c <= r && c < len) ? sT[r * 65 + c] * sb[c] : 0.f;
            }
            solved = true;
        }
    }
    if (!solved) unit_lower_solve(sA, sT, sb, len, LC);
    for (int idx = threadIdx.x; idx < len * dv; idx += blockDim.x) {
        int r = idx / dv, c = idx - r * dv;
        sQ[r * dv + c] = ld_in(v + (row + r) * dv + c);
    }
    __syncthreads();
    // W = T diag(Gamma) K,  U = T V
    bgemm<Tin, 4, 8>(len, dk, len, [&](int m, int i) { return sT[m * LC + i]; },
                [&](int i, int n) { return sG[i] * sK[i * LK + n]; },
                [&](int m, int n, float s) { w.W[slot * C * dk + m * dk + n] = s; });
    bgemm<Tin, 4, 8>(len, dv, len, [&](int m, int i) { return sT[m * LC + i]; },
                [&](int i, int n) { return sQ[i * dv + n]; },
                [&](int m, int n, float s) { w.U[slot * C * dv + m * dv + n] = s; });
}

// ----------------------------------------------------------------------------- scan
template <class Tin>
__global__ void __launch_bounds__(256) k_scan(Geo g, const float *__restrict__ h0,
                                              float *__restrict__ hT, Ws w, int BV)
{
    const int s = blockIdx.x, h = blockIdx.y, n0 = blockIdx.z * BV;
    const int nb = min(BV, g.dv - n0);
    const int C = g.C, dk = g.dk, dv = g.dv;
    int b, t0, L, j0, nch;
    seq_of(g, s, b, t0, L, j0, nch);
    extern __shared__ float sm[];
    const int LK = dk + 1;
    float *sS = sm;               // [dk][BV]
    float *sU = sS + dk * BV;     // [C][BV]
    float *sE = sU + C * BV;      // [C] exp(gamma_C - gamma_r)
    float *sW = sE + C;           // [C][LK] W of the chunk
    float *sK = sW + C * LK;      // [C][LK] K of the chunk
    const size_t sidx = ((size_t)s * g.H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
        int kk = idx / nb, n = idx - kk * nb;
        sS[kk * BV + n] = h0 ? h0[sidx + (size_t)kk * dv + n0 + n] : 0.f;
    }
    // W and K of a chunk are copied into shared memory first (all loads of a thread in
    // flight together), the next chunk's rows prefetched into L2 meanwhile
    auto stage_rows = [&](const float *src, float *dst, int len) {
        constexpr int VB = 8;
        for (int base = threadIdx.x; base < len * dk; base += blockDim.x * VB) {
            float x[VB];
#pragma unroll
            for (int u = 0; u < VB; ++u) {
                const int e = base + u * blockDim.x;
                x[u] = e < len * dk ? src[e] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < VB; ++u) {
                const int e = base + u * blockDim.x;
                if (e < len * dk) {
                    const int r = e / dk;
                    dst[r * LK + e - r * dk] = x[u];
                }
            }
        }
    };
    __syncthreads();
    for (int c = 0; c < nch; ++c) {
        const int len = min(C, L - c * C);
        const size_t slot = (size_t)(j0 + c) * g.H + h;
        if (threadIdx.x == 0 && c + 1 < nch) {
            const size_t sl = slot + g.H;
            l2_prefetch(w.W + sl * C * dk, sizeof(float) * C * dk);
            l2_prefetch(w.Kn + sl * C * dk, sizeof(float) * C * dk);
            l2_prefetch(w.U + sl * C * dv, sizeof(float) * C * dv);
        }
        const float *gam = w.gam + slot * C;
        const float gC = gam[len - 1];
        for (int r = threadIdx.x; r < len; r += blockDim.x) sE[r] = expf(gC - gam[r]);
        for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
            int kk = idx / nb, n = idx - kk * nb;
            w.Sin[slot * dk * dv + (size_t)kk * dv + n0 + n] = sS[kk * BV + n];
        }
        stage_rows(w.W + slot * C * dk, sW, len);
        stage_rows(w.Kn + slot * C * dk, sK, len);
        batched_copy(len * nb, [&](int idx) {
            const int r = idx / nb;
            return w.U[slot * C * dv + (size_t)r * dv + n0 + idx - r * nb];
        }, [&](int idx, float val) {
            const int r = idx / nb;
            sU[r * BV + idx - r * nb] = val;
        });
        __syncthreads();
        float *Un = w.Unew + slot * C * dv;
        bgemm<Tin, 4, 4>(len, nb, dk, [&](int r, int kk) { return sW[r * LK + kk]; },
                    [&](int kk, int n) { return sS[kk * BV + n]; },
                    [&](int r, int n, float acc) {
                        float u = sU[r * BV + n] - acc;
                        sU[r * BV + n] = u;
                        Un[r * dv + n0 + n] = u;
                    });
        __syncthreads();
        const float GC = expf(gC);
        bgemm<Tin, 8, 4>(dk, nb, len, [&](int kk, int r) { return sE[r] * sK[r * LK + kk]; },
                    [&](int r, int n) { return sU[r * BV + n]; },
                    [&](int kk, int n, float acc) { sS[kk * BV + n] = fmaf(GC, sS[kk * BV + n], acc); });
        __syncthreads();
    }
    if (hT) {
        for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
            int kk = idx / nb, n = idx - kk * nb;
            hT[sidx + (size_t)kk * dv + n0 + n] = sS[kk * BV + n];
        }
    }
}

// ----------------------------------------------------------------------------- output
template <class Tout>
__global__ void __launch_bounds__(256) k_out(Geo g, Tout *__restrict__ o, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv;
    extern __shared__ float sm[];
    // the operands in shared memory: A = [diag(Gamma) Q | P] rows, B = [S_in ; Unew]
    // one 64-column slice of d_v at a time
    const int KA = dk + len, LA = dk + C + 1, BV = 64, LB = BV + 1;
    float *sG = sm;            // [C] exp(gamma)
    float *sA = sG + C;        // [C][LA]
    float *sB = sA + C * LA;   // [dk + C][LB]
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *gam = w.gam + slot * C;
    const float *Qn = w.Qn + slot * C * dk;
    const float *Sin = w.Sin + slot * dk * dv;
    const float *Un = w.Unew + slot * C * dv;
    const float *Pg = w.P + slot * C * C;
    for (int r = threadIdx.x; r < len; r += blockDim.x) sG[r] = expf(gam[r]);
    __syncthreads();
    batched_copy(len * KA, [&](int idx) {
        const int r = idx / KA, x = idx - r * KA;
        return x < dk ? sG[r] * Qn[r * dk + x] : Pg[r * C + (x - dk)];
    }, [&](int idx, float val) {
        const int r = idx / KA;
        sA[r * LA + idx - r * KA] = val;
    });
    const float sc = g.scale;
    for (int n0 = 0; n0 < dv; n0 += BV) {
        const int nb = min(BV, dv - n0);
        __syncthreads();
        batched_copy(KA * nb, [&](int idx) {
            const int x = idx / nb, n = idx - x * nb;
            return x < dk ? Sin[(size_t)x * dv + n0 + n] : Un[(x - dk) * dv + n0 + n];
        }, [&](int idx, float val) {
            const int x = idx / nb;
            sB[x * LB + idx - x * nb] = val;
        });
        __syncthreads();
        rgemm<4, 8>(len, nb, KA, [&](int r, int x) { return sA[r * LA + x]; },
                    [&](int x, int n) { return sB[x * LB + n]; },
                    [&](int r, int n, float acc) { st_out(o + (row + r) * dv + n0 + n, sc * acc); });
    }
}

// ----------------------------------------------------------------------------- backward scan
template <class Tin>
__global__ void __launch_bounds__(256) k_bscan(Geo g, const Tin *__restrict__ dO,
                                               const float *__restrict__ dhT,
                                               float *__restrict__ dh0, Ws w, int BV)
{
    const int s = blockIdx.x, h = blockIdx.y, n0 = blockIdx.z * BV;
    const int nb = min(BV, g.dv - n0);
    const int C = g.C, dk = g.dk, dv = g.dv;
    int b, t0, L, j0, nch;
    seq_of(g, s, b, t0, L, j0, nch);
    extern __shared__ float sm[];
    float *sdS = sm;               // [dk][BV]
    float *sdU = sdS + dk * BV;    // [C][BV]
    float *sdO = sdU + C * BV;     // [C][BV]  scale * dO
    float *sE = sdO + C * BV;      // [C]
    float *sG = sE + C;            // [C]
    const size_t sidx = ((size_t)s * g.H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
        int kk = idx / nb, n = idx - kk * nb;
        sdS[kk * BV + n] = dhT ? dhT[sidx + (size_t)kk * dv + n0 + n] : 0.f;
    }
    __syncthreads();
    for (int c = nch - 1; c >= 0; --c) {
        const int len = min(C, L - c * C);
        const size_t slot = (size_t)(j0 + c) * g.H + h;
        const size_t row = ((size_t)b * g.H + h) * g.T + t0 + (size_t)c * C;
        const float *gam = w.gam + slot * C;
        const float gC = gam[len - 1];
        const float *Qn = w.Qn + slot * C * dk;
        const float *Kn = w.Kn + slot * C * dk;
        const float *W = w.W + slot * C * dk;
        const float *Pg = w.P + slot * C * C;
        for (int r = threadIdx.x; r < len; r += blockDim.x) {
            sE[r] = expf(gC - gam[r]);
            sG[r] = expf(gam[r]);
        }
        for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
            int kk = idx / nb, n = idx - kk * nb;
            w.dSo[slot * dk * dv + (size_t)kk * dv + n0 + n] = sdS[kk * BV + n];
        }
        for (int idx = threadIdx.x; idx < len * nb; idx += blockDim.x) {
            int r = idx / nb, n = idx - r * nb;
            sdO[r * BV + n] = g.scale * ld_in(dO + (row + r) * dv + n0 + n);
        }
        __syncthreads();
        // dUnew(i, n) = sum_r P(r, i) dO(r, n) + exp(gC - gam_i) sum_kk K(i, kk) dS(kk, n)
        float *dUg = w.dUn + slot * C * dv;
        bgemm<Tin, 4, 4>(len, nb, len + dk,
                    [&](int i, int x) { return x < len ? Pg[x * C + i] : sE[i] * Kn[i * dk + (x - len)]; },
                    [&](int x, int n) { return x < len ? sdO[x * BV + n] : sdS[(x - len) * BV + n]; },
                    [&](int i, int n, float u) {
                        sdU[i * BV + n] = u;
                        dUg[i * dv + n0 + n] = u;
                    });
        __syncthreads();
        // dS <- Gamma_C dS + (Gamma Q)^T dO - W^T dUnew
        const float GC = expf(gC);
        bgemm<Tin, 8, 4>(dk, nb, 2 * len,
                    [&](int kk, int x) { return x < len ? sG[x] * Qn[x * dk + kk] : -W[(x - len) * dk + kk]; },
                    [&](int x, int n) { return x < len ? sdO[x * BV + n] : sdU[(x - len) * BV + n]; },
                    [&](int kk, int n, float acc) { sdS[kk * BV + n] = fmaf(GC, sdS[kk * BV + n], acc); });
        __syncthreads();
    }
    if (dh0) {
        for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
            int kk = idx / nb, n = idx - kk * nb;
            dh0[sidx + (size_t)kk * dv + n0 + n] = sdS[kk * BV + n];
        }
    }
}

// ----------------------------------------------------------------------------- staged scans (bf16)
// The two sequential scans for bf16 inputs with d_k, d_v <= 128: one CTA per
// (sequence, head) walks the chunks in order.  Each chunk's operands are first
// copied into shared memory in their natural row-major layout (16-byte loads issued
// in batches, rounded to bf16 once, rows padded by 8 elements so that 8 consecutive
// rows fall in different bank groups), and the warp-level tensor-core products take
// their fragments with ldmatrix (transposing on load where the reduction runs down
// the rows).

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const __nv_bfloat16 *p, bool trans)
{
    // the "memory" clobber: the statement reads shared memory through an address held
    // in a register, so the compiler must not move shared-memory stores across it
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    if (trans)
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a) : "memory");
    else
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a) : "memory");
}

// acc (the warp's 32 x 32 tile at m0, n0: two 16-row halves of four 16 x 8
// accumulators) += A B over k in [0, K), K % 16 == 0.  A(m, k) is stored at
// A[m * lda + k] (AT false) or A[k * lda + m] (AT true); B(k, n) at B[n * ldb + k]
// (BT false) or B[k * ldb + n] (BT true).  lda, ldb % 8 == 0; m0, n0 % 32 == 0.
template <bool AT, bool BT>
__device__ __forceinline__ void tile_mma(float (&acc)[2][4][4], const __nv_bfloat16 *A, int lda,
                                         const __nv_bfloat16 *B, int ldb, int m0, int n0, int K)
{
    const int lane = threadIdx.x & 31, mi = lane >> 3, r = lane & 7;
    for (int k0 = 0; k0 < K; k0 += 16) {
        uint32_t a[2][4], b[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int mh = m0 + 16 * h;
            if (AT) ldsm4(a[h], A + (k0 + (mi >> 1) * 8 + r) * lda + mh + (mi & 1) * 8, true);
            else ldsm4(a[h], A + (mh + (mi & 1) * 8 + r) * lda + k0 + (mi >> 1) * 8, false);
        }
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
            const int nt = 2 * jp + (mi >> 1);
            if (BT) ldsm4(b[jp], B + (k0 + (mi & 1) * 8 + r) * ldb + n0 + 8 * nt, true);
            else ldsm4(b[jp], B + (n0 + 8 * nt + r) * ldb + k0 + (mi & 1) * 8, false);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t bb[2] = {b[j >> 1][2 * (j & 1)], b[j >> 1][2 * (j & 1) + 1]};
                mma_bf16_16816(acc[h][j], a[h], bb);
            }
    }
}

using prep::tile_tf32;

// Runs Body(m0, n0, acc) for every 32 x 32 tile of an M x N product (M, N % 32 == 0),
// the tiles dealt round-robin to the warps, with acc zeroed; then St(m, n, v0, v1)
// for each pair of adjacent results (n even).  ntl_log2 = log2(N / 32).
template <class Body, class FS>
__device__ __forceinline__ void tiles(int M, int ntl_log2, Body body, FS St)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int ntiles = (M / 32) << ntl_log2;
    for (int tile = warp; tile < ntiles; tile += nw) {
        const int m0 = (tile >> ntl_log2) * 32, n0 = (tile & ((1 << ntl_log2) - 1)) * 32;
        float acc[2][4][4];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[h][j][0] = acc[h][j][1] = acc[h][j][2] = acc[h][j][3] = 0.f;
        body(m0, n0, acc);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + 8 * j + 2 * t;
                St(m0 + 16 * h + g, n, acc[h][j][0], acc[h][j][1]);
                St(m0 + 16 * h + g + 8, n, acc[h][j][2], acc[h][j][3]);
            }
    }
}

__device__ __forceinline__ int ilog2(int x) { return 31 - __clz(x); }

// floats of padding after k_bchunk's last C x C buffer so that its last two buffers
// can hold two staged bf16 tiles of C rows of max(dk, dv) + 8 elements
__host__ __device__ __forceinline__ int bchunk_pad(int C, int dk, int dv)
{
    const int need = C * ((dk > dv ? dk : dv) + 8), have = 2 * C * (C + 1);
    return need > have ? ((need - have + 3) & ~3) : 0;
}

__host__ __device__ __forceinline__ bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// head dims of 32, 64 or 128 and chunks of 32 or 64: every tile is a whole number of
// 32 x 32 warp tiles and every index split is a shift
__host__ __device__ __forceinline__ bool staged_ok(const Geo &g)
{
    return pow2(g.dk) && pow2(g.dv) && g.dk >= 32 && g.dv >= 32 && g.dk <= 128 && g.dv <= 128 && g.C >= 32;
}

// Copies the rows x cols fp32 row-major block at src (cols % 4 == 0, src 16-byte
// aligned) through registers: every thread first issues its 16-byte loads for a batch,
// then hands each group of four to put(r, c, v).  Rows at or past `live` read as zero.
template <class FP>
__device__ __forceinline__ void stage_f32(const float *__restrict__ src, int rows, int cols, int live, FP put)
{
    constexpr int VB = 8;
    const int lc4 = ilog2(cols) - 2, n4 = (rows * cols) >> 2;   // cols: a power of two >= 4
    for (int base = threadIdx.x; base < n4; base += blockDim.x * VB) {
        float4 v[VB];
#pragma unroll
        for (int u = 0; u < VB; ++u) {
            const int e = base + u * blockDim.x;
            v[u] = (e < n4 && (e >> lc4) < live) ? __ldg(reinterpret_cast<const float4 *>(src) + e)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < VB; ++u) {
            const int e = base + u * blockDim.x;
            if (e < n4) put(e >> lc4, (e & ((1 << lc4) - 1)) << 2, v[u]);
        }
    }
}

// four values, scaled, as bf16 at dst (8-byte aligned)
__device__ __forceinline__ void put_bf4(__nv_bfloat16 *dst, float4 v, float s)
{
    *reinterpret_cast<uint2 *>(dst) = make_uint2(bf16x2(s * v.x, s * v.y), bf16x2(s * v.z, s * v.w));
}

__device__ __forceinline__ void put_bf2(__nv_bfloat16 *dst, float lo, float hi)
{
    *reinterpret_cast<uint32_t *>(dst) = bf16x2(lo, hi);
}

// The same copy split in two, for a block of at most NB x blockDim.x pieces of 16 bytes:
// reg_load issues every load into registers, reg_put hands them to put(r, c, v), so
// that the loads of several blocks are in flight together.
template <int NB>
__device__ __forceinline__ void reg_load(float4 (&v)[NB], const float *__restrict__ src, int rows, int cols, int live)
{
    const int lc4 = ilog2(cols) - 2, n4 = (rows * cols) >> 2;
#pragma unroll
    for (int u = 0; u < NB; ++u) {
        const int e = threadIdx.x + u * blockDim.x;
        v[u] = (e < n4 && (e >> lc4) < live) ? __ldg(reinterpret_cast<const float4 *>(src) + e)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
// rows x cols bf16 row-major (cols a power of two >= 8), eight elements per piece
template <int NB>
__device__ __forceinline__ void reg_load_bf(uint4 (&v)[NB], const __nv_bfloat16 *__restrict__ src, int rows, int cols,
                                            int live)
{
    const int lc8 = ilog2(cols) - 3, n8 = (rows * cols) >> 3;
#pragma unroll
    for (int u = 0; u < NB; ++u) {
        const int e = threadIdx.x + u * blockDim.x;
        v[u] = (e < n8 && (e >> lc8) < live) ? __ldg(reinterpret_cast<const uint4 *>(src) + e)
                                             : make_uint4(0u, 0u, 0u, 0u);
    }
}
template <int NB, class FP>
__device__ __forceinline__ void reg_put_bf(const uint4 (&v)[NB], int rows, int cols, FP put)
{
    const int lc8 = ilog2(cols) - 3, n8 = (rows * cols) >> 3;
#pragma unroll
    for (int u = 0; u < NB; ++u) {
        const int e = threadIdx.x + u * blockDim.x;
        if (e < n8) put(e >> lc8, (e & ((1 << lc8) - 1)) << 3, v[u]);
    }
}
template <int NB, class FP>
__device__ __forceinline__ void reg_put(const float4 (&v)[NB], int rows, int cols, FP put)
{
    const int lc4 = ilog2(cols) - 2, n4 = (rows * cols) >> 2;
#pragma unroll
    for (int u = 0; u < NB; ++u) {
        const int e = threadIdx.x + u * blockDim.x;
        if (e < n4) put(e >> lc4, (e & ((1 << lc4) - 1)) << 2, v[u]);
    }
}


// row strides (elements) of the staged tiles
__host__ __device__ __forceinline__ int spad(int cols) { return cols + 8; }

// forward recompute: S_in of every chunk, and Unew = U - W S_in, S <- Gamma_C S + K~^T Unew
__global__ void __launch_bounds__(512) k_scan_st(Geo g, const float *__restrict__ h0,
                                                 float *__restrict__ hT, Ws w)
{
    const int s = blockIdx.x, h = blockIdx.y;
    const int C = g.C, dk = g.dk, dv = g.dv;
    const int LS = dv + 8, LK = spad(dk), LV = spad(dv), ldv = ilog2(dv);
    int b, t0, L, j0, nch;
    seq_of(g, s, b, t0, L, j0, nch);
    extern __shared__ float sm[];
    float *sS = sm;                                          // [dk][LS] fp32 state
    float *sE = sS + dk * LS;                                // [C] exp(gamma_C - gamma_r)
    float *sU = sE + 64;                                     // [C][dv] U
    __nv_bfloat16 *Wt = reinterpret_cast<__nv_bfloat16 *>(sU + C * dv);   // W [C][LK]
    __nv_bfloat16 *Sb = Wt + C * LK;                         // S [dk][LV]
    __nv_bfloat16 *EK = Sb + dk * LV;                        // diag(E) K [C][LK]
    __nv_bfloat16 *Ub = EK + C * LK;                         // Unew [C][LV]
    const size_t sidx = ((size_t)s * g.H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < dk * dv / 2; idx += blockDim.x) {
        const int kk = (2 * idx) >> ldv, n = (2 * idx) & (dv - 1);
        const float v0 = h0 ? h0[sidx + 2 * idx] : 0.f, v1 = h0 ? h0[sidx + 2 * idx + 1] : 0.f;
        *reinterpret_cast<float2 *>(sS + kk * LS + n) = make_float2(v0, v1);
        put_bf2(Sb + kk * LV + n, v0, v1);
    }
    __syncthreads();
    // chunk c's W, K, U rows and log-gates: into L2 two chunks ahead; at the top of the
    // chunk, every load of its operands is issued at once into registers, then the
    // registers go to shared memory once the previous chunk's state has been written out
    auto prefetch = [&](int c) {
        if (threadIdx.x == 0 && c >= 0 && c < nch) {
            const size_t sl = (size_t)(j0 + c) * g.H + h;
            l2_prefetch(w.W + sl * C * dk, sizeof(float) * C * dk);
            l2_prefetch(w.Kn + sl * C * dk, sizeof(float) * C * dk);
            l2_prefetch(w.U + sl * C * dv, sizeof(float) * C * dv);
            l2_prefetch(w.gam + sl * C, sizeof(float) * C);
        }
    };
    constexpr int NB = 4;   // C * d / 4 <= 4 * 512 pieces
    float4 rW[NB], rK[NB], rU[NB];
    float rg = 0.f, rgC = 0.f;   // gam[threadIdx.x] and gam[len - 1] of the chunk
    auto issue = [&](int c) {
        const int ln = min(C, L - c * C);
        const size_t sl = (size_t)(j0 + c) * g.H + h;
        reg_load(rW, w.W + sl * C * dk, C, dk, ln);
        reg_load(rK, w.Kn + sl * C * dk, C, dk, ln);
        reg_load(rU, w.U + sl * C * dv, C, dv, ln);
        rg = (int)threadIdx.x < ln ? __ldg(w.gam + sl * C + threadIdx.x) : 0.f;
        rgC = __ldg(w.gam + sl * C + ln - 1);
    };
    prefetch(0);
    prefetch(1);
    for (int c = 0; c < nch; ++c) {
        issue(c);
        const int len = min(C, L - c * C);
        const size_t slot = (size_t)(j0 + c) * g.H + h;
        const float gC = rgC;
        float *Un = w.Unew + slot * C * dv;
        float *Sin = w.Sin + slot * dk * dv;
        __nv_bfloat16 *Unb = w.Un_b ? w.Un_b + slot * C * dv : nullptr;
        if ((int)threadIdx.x < C) sE[threadIdx.x] = (int)threadIdx.x < len ? expf(gC - rg) : 0.f;
        if (w.Sin_b) {
            __nv_bfloat16 *Sb16 = w.Sin_b + slot * dk * dv;
            for (int idx = threadIdx.x; idx < dk * dv / 4; idx += blockDim.x) {
                const int kk = (4 * idx) >> ldv, n = (4 * idx) & (dv - 1);
                put_bf4(Sb16 + 4 * idx, *reinterpret_cast<const float4 *>(sS + kk * LS + n), 1.f);
            }
        } else {
            for (int idx = threadIdx.x; idx < dk * dv / 4; idx += blockDim.x) {
                const int kk = (4 * idx) >> ldv, n = (4 * idx) & (dv - 1);
                reinterpret_cast<float4 *>(Sin)[idx] = *reinterpret_cast<const float4 *>(sS + kk * LS + n);
            }
        }
        __syncthreads();
        reg_put(rW, C, dk, [&](int r, int kk, float4 v) { put_bf4(Wt + r * LK + kk, v, 1.f); });
        reg_put(rK, C, dk, [&](int r, int kk, float4 v) { put_bf4(EK + r * LK + kk, v, sE[r]); });
        reg_put(rU, C, dv, [&](int r, int n, float4 v) { *reinterpret_cast<float4 *>(sU + r * dv + n) = v; });
        __syncthreads();
        prefetch(c + 2);
        // Unew[r][n] = U[r][n] - sum_kk W[r][kk] S[kk][n]
        tiles(C, ldv - 5, [&](int m0, int n0, float (&acc)[2][4][4]) { tile_mma<false, true>(acc, Wt, LK, Sb, LV, m0, n0, dk); },
              [&](int r, int n, float a0, float a1) {
                  const bool live = r < len;
                  const float u0 = live ? sU[r * dv + n] - a0 : 0.f, u1 = live ? sU[r * dv + n + 1] - a1 : 0.f;
                  if (Unb) put_bf2(Unb + r * dv + n, u0, u1);
                  else if (live) *reinterpret_cast<float2 *>(Un + r * dv + n) = make_float2(u0, u1);
                  put_bf2(Ub + r * LV + n, u0, u1);
              });
        __syncthreads();
        // S[kk][n] <- Gamma_C S[kk][n] + sum_r E_r K[r][kk] Unew[r][n]
        const float GC = expf(gC);
        tiles(dk, ldv - 5, [&](int m0, int n0, float (&acc)[2][4][4]) { tile_mma<true, true>(acc, EK, LK, Ub, LV, m0, n0, C); },
              [&](int kk, int n, float a0, float a1) {
                  float2 *sp = reinterpret_cast<float2 *>(sS + kk * LS + n);
                  const float2 o = *sp;
                  const float v0 = fmaf(GC, o.x, a0), v1 = fmaf(GC, o.y, a1);
                  *sp = make_float2(v0, v1);
                  put_bf2(Sb + kk * LV + n, v0, v1);
              });
        __syncthreads();
    }
    if (hT)
        for (int idx = threadIdx.x; idx < dk * dv; idx += blockDim.x) {
            const int kk = idx >> ldv, n = idx & (dv - 1);
            hT[sidx + idx] = sS[kk * LS + n];
        }
}

// backward scan: dS_out of every chunk, and
//   dUnew = P^T dO + K~ dS,   dS <- Gamma_C dS + (Gamma Q)^T dO - W^T dUnew
__global__ void __launch_bounds__(512) k_bscan_st(Geo g, const __nv_bfloat16 *__restrict__ dO,
                                                  const float *__restrict__ dhT,
                                                  float *__restrict__ dh0, Ws w)
{
    const int s = blockIdx.x, h = blockIdx.y;
    const int C = g.C, dk = g.dk, dv = g.dv;
    const int LS = dv + 8, LC = spad(C), LK = spad(dk), LV = spad(dv), ldv = ilog2(dv);
    int b, t0, L, j0, nch;
    seq_of(g, s, b, t0, L, j0, nch);
    extern __shared__ float sm[];
    float *sdS = sm;                                         // [dk][LS] fp32
    float *sE = sdS + dk * LS;                               // [C] exp(gamma_C - gamma_r)
    float *sG = sE + 64;                                     // [C] exp(gamma_r)
    __nv_bfloat16 *Ps = reinterpret_cast<__nv_bfloat16 *>(sG + 64);   // P [C][LC]
    __nv_bfloat16 *EK = Ps + C * LC;                         // diag(E) K [C][LK]
    __nv_bfloat16 *GQ = EK + C * LK;                         // diag(G) Q [C][LK]
    __nv_bfloat16 *Wn = GQ + C * LK;                         // -W [C][LK]
    __nv_bfloat16 *dOb = Wn + C * LK;                        // scale dO [C][LV]
    __nv_bfloat16 *dUb = dOb + C * LV;                       // dUnew [C][LV]
    __nv_bfloat16 *dSb = dUb + C * LV;                       // dS [dk][LV]
    const size_t sidx = ((size_t)s * g.H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < dk * dv / 2; idx += blockDim.x) {
        const int kk = (2 * idx) >> ldv, n = (2 * idx) & (dv - 1);
        const float v0 = dhT ? dhT[sidx + 2 * idx] : 0.f, v1 = dhT ? dhT[sidx + 2 * idx + 1] : 0.f;
        *reinterpret_cast<float2 *>(sdS + kk * LS + n) = make_float2(v0, v1);
        put_bf2(dSb + kk * LV + n, v0, v1);
    }
    __syncthreads();
    // chunk c's P, K, Q, W, dO rows and log-gates: into L2 two chunks ahead; at the top
    // of the chunk, every load of its operands is issued at once into registers, then the
    // registers go to shared memory once the previous chunk's dS has been written out
    auto prefetch = [&](int c) {
        if (threadIdx.x == 0 && c >= 0 && c < nch) {
            const size_t sl = (size_t)(j0 + c) * g.H + h;
            const int ln = min(C, L - c * C);
            l2_prefetch(w.P + sl * C * C, sizeof(float) * C * C);
            l2_prefetch(w.Kn + sl * C * dk, sizeof(float) * C * dk);
            l2_prefetch(w.Qn + sl * C * dk, sizeof(float) * C * dk);
            l2_prefetch(w.W + sl * C * dk, sizeof(float) * C * dk);
            l2_prefetch(w.gam + sl * C, sizeof(float) * C);
            l2_prefetch(dO + (((size_t)b * g.H + h) * g.T + t0 + (size_t)c * C) * dv, sizeof(__nv_bfloat16) * ln * dv);
        }
    };
    constexpr int NB = 4, NBP = 2;   // C * d / 4 <= 4 * 512 and C * C / 4, C * d / 8 <= 2 * 512 pieces
    float4 rP[NBP], rK[NB], rQ[NB], rW[NB];
    uint4 rO[NBP];
    float rg = 0.f, rgC = 0.f;   // gam[threadIdx.x] and gam[len - 1] of the chunk
    const int n8 = (C * dv) >> 3, lc8 = ldv - 3;
    auto issue = [&](int c) {
        const int ln = min(C, L - c * C);
        const size_t sl = (size_t)(j0 + c) * g.H + h;
        const size_t rw = ((size_t)b * g.H + h) * g.T + t0 + (size_t)c * C;
        reg_load(rP, w.P + sl * C * C, C, C, ln);
        reg_load(rK, w.Kn + sl * C * dk, C, dk, ln);
        reg_load(rQ, w.Qn + sl * C * dk, C, dk, ln);
        reg_load(rW, w.W + sl * C * dk, C, dk, ln);
#pragma unroll
        for (int u = 0; u < NBP; ++u) {
            const int e = threadIdx.x + u * blockDim.x;
            rO[u] = (e < n8 && (e >> lc8) < ln) ? __ldg(reinterpret_cast<const uint4 *>(dO + rw * dv) + e)
                                                : make_uint4(0u, 0u, 0u, 0u);
        }
        rg = (int)threadIdx.x < ln ? __ldg(w.gam + sl * C + threadIdx.x) : 0.f;
        rgC = __ldg(w.gam + sl * C + ln - 1);
    };
    prefetch(nch - 1);
    prefetch(nch - 2);
    for (int c = nch - 1; c >= 0; --c) {
        issue(c);
        const int len = min(C, L - c * C);
        const size_t slot = (size_t)(j0 + c) * g.H + h;
        const float gC = rgC;
        float *dUg = w.dUn + slot * C * dv;
        float *dSo = w.dSo + slot * dk * dv;
        __nv_bfloat16 *dUb16 = w.dUn_b ? w.dUn_b + slot * C * dv : nullptr;
        if ((int)threadIdx.x < C) {
            const bool live = (int)threadIdx.x < len;
            sE[threadIdx.x] = live ? expf(gC - rg) : 0.f;
            sG[threadIdx.x] = live ? expf(rg) : 0.f;
        }
        if (w.dSo_b) {
            __nv_bfloat16 *dS16 = w.dSo_b + slot * dk * dv;
            for (int idx = threadIdx.x; idx < dk * dv / 4; idx += blockDim.x) {
                const int kk = (4 * idx) >> ldv, n = (4 * idx) & (dv - 1);
                put_bf4(dS16 + 4 * idx, *reinterpret_cast<const float4 *>(sdS + kk * LS + n), 1.f);
            }
        } else {
            for (int idx = threadIdx.x; idx < dk * dv / 4; idx += blockDim.x) {
                const int kk = (4 * idx) >> ldv, n = (4 * idx) & (dv - 1);
                reinterpret_cast<float4 *>(dSo)[idx] = *reinterpret_cast<const float4 *>(sdS + kk * LS + n);
            }
        }
        __syncthreads();
        // P's columns i >= len are not written by the preparation; they only reach rows
        // i >= len of dUnew, which are dropped below
        reg_put(rP, C, C, [&](int x, int i, float4 v) { put_bf4(Ps + x * LC + i, v, 1.f); });
        reg_put(rK, C, dk, [&](int r, int kk, float4 v) { put_bf4(EK + r * LK + kk, v, sE[r]); });
        reg_put(rQ, C, dk, [&](int r, int kk, float4 v) { put_bf4(GQ + r * LK + kk, v, sG[r]); });
        reg_put(rW, C, dk, [&](int r, int kk, float4 v) { put_bf4(Wn + r * LK + kk, v, -1.f); });
#pragma unroll
        for (int u = 0; u < NBP; ++u) {
            // scale dO, 8 bf16 per piece
            const int e = threadIdx.x + u * blockDim.x;
            if (e >= n8) continue;
            const int r = e >> lc8, n = (e & ((1 << lc8) - 1)) << 3;
            const uint32_t wv[4] = {rO[u].x, rO[u].y, rO[u].z, rO[u].w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                o[q] = bf16x2(g.scale * __uint_as_float(wv[q] << 16), g.scale * __uint_as_float(wv[q] & 0xFFFF0000u));
            *reinterpret_cast<uint4 *>(dOb + r * LV + n) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncthreads();
        prefetch(c - 2);
        // dUnew[i][n] = sum_x P[x][i] dO[x][n] + E_i sum_kk K[i][kk] dS[kk][n]
        tiles(C, ldv - 5,
              [&](int m0, int n0, float (&acc)[2][4][4]) {
                  tile_mma<true, true>(acc, Ps, LC, dOb, LV, m0, n0, C);
                  tile_mma<false, true>(acc, EK, LK, dSb, LV, m0, n0, dk);
              },
              [&](int i, int n, float u0, float u1) {
                  const bool live = i < len;
                  if (dUb16) put_bf2(dUb16 + i * dv + n, live ? u0 : 0.f, live ? u1 : 0.f);
                  else if (live) *reinterpret_cast<float2 *>(dUg + i * dv + n) = make_float2(u0, u1);
                  put_bf2(dUb + i * LV + n, live ? u0 : 0.f, live ? u1 : 0.f);
              });
        __syncthreads();
        // dS[kk][n] <- Gamma_C dS[kk][n] + sum_x G_x Q[x][kk] dO[x][n] - sum_x W[x][kk] dUnew[x][n]
        const float GC = expf(gC);
        tiles(dk, ldv - 5,
              [&](int m0, int n0, float (&acc)[2][4][4]) {
                  tile_mma<true, true>(acc, GQ, LK, dOb, LV, m0, n0, C);
                  tile_mma<true, true>(acc, Wn, LK, dUb, LV, m0, n0, C);
              },
              [&](int kk, int n, float a0, float a1) {
                  float2 *sp = reinterpret_cast<float2 *>(sdS + kk * LS + n);
                  const float2 o = *sp;
                  const float v0 = fmaf(GC, o.x, a0), v1 = fmaf(GC, o.y, a1);
                  *sp = make_float2(v0, v1);
                  put_bf2(dSb + kk * LV + n, v0, v1);
              });
        __syncthreads();
    }
    if (dh0)
        for (int idx = threadIdx.x; idx < dk * dv; idx += blockDim.x) {
            const int kk = idx >> ldv, n = idx & (dv - 1);
            dh0[sidx + idx] = sdS[kk * LS + n];
        }
}

// backward scan over the cooperative forward's packages (bf16 tiles in the 128-byte
// swizzle: -W, Qt = diag(exp(gamma) m) Q, P, the vector f0 = exp(gamma_C - gamma) n and
// exp(gamma_C)) and the raw keys, instead of the recompute's fp32 arrays:
//   dUnew = P^T dO + diag(f0) K dS,   dS <- exp(gamma_C) dS + Qt^T dO - W^T dUnew
// (diag(f0) K = diag(exp(gamma_C - gamma)) K~ and Qt = diag(exp(gamma)) Q~ of k_bscan_st).
// Writes dS_out and dUnew as bf16 (the tcgen05 per-chunk backward's inputs).
__global__ void __launch_bounds__(512) k_bscan_pk(Geo g, const __nv_bfloat16 *__restrict__ kin,
                                                  const __nv_bfloat16 *__restrict__ dO,
                                                  const float *__restrict__ dhT, float *__restrict__ dh0,
                                                  const uint8_t *__restrict__ keep, coop::PkLayout pk, Ws w)
{
    const int s = blockIdx.x, h = blockIdx.y;
    const int C = g.C, dk = g.dk, dv = g.dv;
    const int LS = dv + 8, LC = spad(C), LK = spad(dk), LV = spad(dv), ldv = ilog2(dv);
    int b, t0, L, j0, nch;
    seq_of(g, s, b, t0, L, j0, nch);
    extern __shared__ float sm[];
    float *sdS = sm;                                         // [dk][LS] fp32
    float *sF = sdS + dk * LS;                               // [C] f0
    __nv_bfloat16 *Ps = reinterpret_cast<__nv_bfloat16 *>(sF + 128);   // P [C][LC]
    __nv_bfloat16 *EK = Ps + C * LC;                         // diag(f0) K [C][LK]
    __nv_bfloat16 *GQ = EK + C * LK;                         // Qt [C][LK]
    __nv_bfloat16 *Wn = GQ + C * LK;                         // -W [C][LK]
    __nv_bfloat16 *dOb = Wn + C * LK;                        // scale dO [C][LV]
    __nv_bfloat16 *dUb = dOb + C * LV;                       // dUnew [C][LV]
    __nv_bfloat16 *dSb = dUb + C * LV;                       // dS [dk][LV]
    const size_t sidx = ((size_t)s * g.H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < dk * dv / 2; idx += blockDim.x) {
        const int kk = (2 * idx) >> ldv, n = (2 * idx) & (dv - 1);
        const float v0 = dhT ? dhT[sidx + 2 * idx] : 0.f, v1 = dhT ? dhT[sidx + 2 * idx + 1] : 0.f;
        *reinterpret_cast<float2 *>(sdS + kk * LS + n) = make_float2(v0, v1);
        put_bf2(dSb + kk * LV + n, v0, v1);
    }
    __syncthreads();
    const uint8_t *pkg0 = keep + (size_t)h * pk.stride;   // + chunk slot * H * stride
    auto pkg = [&](int c) { return pkg0 + (size_t)(j0 + c) * g.H * pk.stride; };
    // chunk c's package, keys and dO into L2 two chunks ahead; at the top of the chunk
    // every load of its operands is issued at once into registers
    auto prefetch = [&](int c) {
        if (threadIdx.x == 0 && c >= 0 && c < nch) {
            const int ln = min(C, L - c * C);
            const size_t rw = ((size_t)b * g.H + h) * g.T + t0 + (size_t)c * C;
            l2_prefetch(pkg(c), pk.stride);
            l2_prefetch(kin + rw * dk, sizeof(__nv_bfloat16) * ln * dk);
            l2_prefetch(dO + rw * dv, sizeof(__nv_bfloat16) * ln * dv);
        }
    };
    // swizzled tile pieces: row r of a 64-column panel holds 16-byte chunks c ^ (r % 8)
    auto swz = [](int r, int c8) { return (uint32_t)(r * 128 + (((c8 ^ (r & 7)) & 7) << 4)); };
    constexpr int NB = 2;   // C * d / 8 <= 2 * 512 pieces of 16 bytes; C * C / 8 <= 512
    uint4 rP, rK[NB], rQ[NB], rW[NB], rO[NB];
    float rf = 0.f, rgC = 0.f;
    const int nkp = (C * dk) >> 3, lk8 = ilog2(dk) - 3;   // pieces of a C x dk tile, per row
    auto issue = [&](int c) {
        const int ln = min(C, L - c * C);
        const size_t rw = ((size_t)b * g.H + h) * g.T + t0 + (size_t)c * C;
        const uint8_t *pg = pkg(c);
        {
            const int e = threadIdx.x;   // P: C rows x 8 pieces
            rP = (e < C * 8) ? __ldg(reinterpret_cast<const uint4 *>(pg + pk.p + swz(e >> 3, e & 7)))
                             : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < NB; ++u) {
            const int e = threadIdx.x + u * blockDim.x;
            const int r = e >> lk8, c16 = e & ((1 << lk8) - 1), q = c16 >> 3;
            const uint8_t *tile = pg + pk.wq + q * pk.wq_panel + swz(r, c16 & 7);
            const bool in = e < nkp;
            rW[u] = in ? __ldg(reinterpret_cast<const uint4 *>(tile)) : make_uint4(0u, 0u, 0u, 0u);
            rQ[u] = in ? __ldg(reinterpret_cast<const uint4 *>(tile + pk.panel)) : make_uint4(0u, 0u, 0u, 0u);
        }
        reg_load_bf(rK, kin + rw * dk, C, dk, ln);
        reg_load_bf(rO, dO + rw * dv, C, dv, ln);
        const float *vec = reinterpret_cast<const float *>(pg + pk.vec);
        rf = (int)threadIdx.x < C ? __ldg(vec + threadIdx.x) : 0.f;
        rgC = __ldg(vec + 64);
    };
    prefetch(nch - 1);
    prefetch(nch - 2);
    for (int c = nch - 1; c >= 0; --c) {
        issue(c);
        const int len = min(C, L - c * C);
        const size_t slot = (size_t)(j0 + c) * g.H + h;
        __nv_bfloat16 *dUb16 = w.dUn_b + slot * C * dv;
        if ((int)threadIdx.x < C) sF[threadIdx.x] = rf;
        {
            __nv_bfloat16 *dS16 = w.dSo_b + slot * dk * dv;
            for (int idx = threadIdx.x; idx < dk * dv / 4; idx += blockDim.x) {
                const int kk = (4 * idx) >> ldv, n = (4 * idx) & (dv - 1);
                put_bf4(dS16 + 4 * idx, *reinterpret_cast<const float4 *>(sdS + kk * LS + n), 1.f);
            }
        }
        __syncthreads();
        {
            const int e = threadIdx.x;
            if (e < C * 8) *reinterpret_cast<uint4 *>(Ps + (e >> 3) * LC + ((e & 7) << 3)) = rP;
        }
        reg_put_bf(rW, C, dk, [&](int r, int kk, uint4 v) { *reinterpret_cast<uint4 *>(Wn + r * LK + kk) = v; });
        reg_put_bf(rQ, C, dk, [&](int r, int kk, uint4 v) { *reinterpret_cast<uint4 *>(GQ + r * LK + kk) = v; });
        reg_put_bf(rK, C, dk, [&](int r, int kk, uint4 v) {
            const float f = sF[r];
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                o[q] = bf16x2(f * __uint_as_float(wv[q] << 16), f * __uint_as_float(wv[q] & 0xFFFF0000u));
            *reinterpret_cast<uint4 *>(EK + r * LK + kk) = make_uint4(o[0], o[1], o[2], o[3]);
        });
        reg_put_bf(rO, C, dv, [&](int r, int n, uint4 v) {
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                o[q] = bf16x2(g.scale * __uint_as_float(wv[q] << 16), g.scale * __uint_as_float(wv[q] & 0xFFFF0000u));
            *reinterpret_cast<uint4 *>(dOb + r * LV + n) = make_uint4(o[0], o[1], o[2], o[3]);
        });
        __syncthreads();
        prefetch(c - 2);
        // dUnew[i][n] = sum_x P[x][i] dO[x][n] + sum_kk (f0 K)[i][kk] dS[kk][n]
        tiles(C, ldv - 5,
              [&](int m0, int n0, float (&acc)[2][4][4]) {
                  tile_mma<true, true>(acc, Ps, LC, dOb, LV, m0, n0, C);
                  tile_mma<false, true>(acc, EK, LK, dSb, LV, m0, n0, dk);
              },
              [&](int i, int n, float u0, float u1) {
                  const bool live = i < len;
                  put_bf2(dUb16 + i * dv + n, live ? u0 : 0.f, live ? u1 : 0.f);
                  put_bf2(dUb + i * LV + n, live ? u0 : 0.f, live ? u1 : 0.f);
              });
        __syncthreads();
        // dS[kk][n] <- exp(gamma_C) dS[kk][n] + sum_x Qt[x][kk] dO[x][n] - sum_x W[x][kk] dUnew[x][n]
        const float GC = rgC;
        tiles(dk, ldv - 5,
              [&](int m0, int n0, float (&acc)[2][4][4]) {
                  tile_mma<true, true>(acc, GQ, LK, dOb, LV, m0, n0, C);
                  tile_mma<true, true>(acc, Wn, LK, dUb, LV, m0, n0, C);
              },
              [&](int kk, int n, float a0, float a1) {
                  float2 *sp = reinterpret_cast<float2 *>(sdS + kk * LS + n);
                  const float2 o = *sp;
                  const float v0 = fmaf(GC, o.x, a0), v1 = fmaf(GC, o.y, a1);
                  *sp = make_float2(v0, v1);
                  put_bf2(dSb + kk * LV + n, v0, v1);
              });
        __syncthreads();
    }
    if (dh0)
        for (int idx = threadIdx.x; idx < dk * dv; idx += blockDim.x) {
            const int kk = idx >> ldv, n = idx & (dv - 1);
            dh0[sidx + idx] = sdS[kk * LS + n];
        }
}

// ----------------------------------------------------------------------------- backward: state products
// Per chunk: Y = scale dO S_in^T (dQ = diag(Gamma) Y), dW = -dUnew S_in^T and
// Kt = Unew dS_out^T (dK = diag(exp(gamma_C - gamma)) Kt); plus the row sums
// <Q_r, Y_r>, <Kt_r, K_r> and <dS_out, S_in> that the gate gradient needs.
template <class Tin>
__global__ void __launch_bounds__(512) k_bbig(Geo g, const Tin *__restrict__ dO, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv, LK = dk + 1;
    extern __shared__ float sm[];
    float *sT = sm;                 // [<= 128][LK] d_v columns of a state, transposed
    float *sE = sT + (dv < 128 ? dv : 128) * LK;   // [C]
    float *sG = sE + C;             // [C]
    float *sqt = sG + C;            // [C] <Q_r, Y_r>
    float *set = sqt + C;           // [C] <Kt_r, K_r>
    float *sred = set + C;          // [1] <dS_out, S_in>
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *gam = w.gam + slot * C;
    const float *Sin = w.Sin + slot * dk * dv;
    const float *dSo = w.dSo + slot * dk * dv;
    const float *Un = w.Unew + slot * C * dv;
    const float *dUn = w.dUn + slot * C * dv;
    const float *Qn = w.Qn + slot * C * dk;
    const float *Kn = w.Kn + slot * C * dk;
    float *dQ = w.dQ + slot * C * dk;
    float *dK = w.dK + slot * C * dk;
    float *dW = w.dW + slot * C * dk;
    const float gC = gam[len - 1], sc = g.scale;
    const int lane = threadIdx.x & 31;
    for (int r = threadIdx.x; r < C; r += blockDim.x) {
        sE[r] = r < len ? expf(gC - gam[r]) : 0.f;
        sG[r] = r < len ? expf(gam[r]) : 0.f;
        sqt[r] = 0.f;
        set[r] = 0.f;
    }
    if (threadIdx.x == 0) sred[0] = 0.f;
    __syncthreads();
    {
        float p = 0.f;
        for (int idx = threadIdx.x; idx < dk * dv; idx += blockDim.x) p = fmaf(dSo[idx], Sin[idx], p);
        p = warp_sum(p);
        if (lane == 0) atomicAdd(sred, p);
    }
    // the states are staged transposed, at most 128 of their d_v columns at a time
    const int NB = dv < 128 ? dv : 128;
    for (int nb0 = 0; nb0 < dv; nb0 += NB) {
        const int nbn = min(NB, dv - nb0);
        const bool first = nb0 == 0;
        __syncthreads();
        for (int idx = threadIdx.x; idx < dk * nbn; idx += blockDim.x) {
            int kk = idx / nbn, n = idx - kk * nbn;
            sT[n * LK + kk] = Sin[(size_t)kk * dv + nb0 + n];
        }
        __syncthreads();
        bgemm<Tin, 4, 8>(len, dk, nbn, [&](int r, int n) { return sc * ld_in(dO + (row + r) * dv + nb0 + n); },
                         [&](int n, int kk) { return sT[n * LK + kk]; },
                         [&](int r, int kk, float y) {
                             dQ[r * dk + kk] = (first ? 0.f : dQ[r * dk + kk]) + sG[r] * y;
                             atomicAdd(&sqt[r], Qn[r * dk + kk] * y);
                         });
        bgemm<Tin, 4, 8>(len, dk, nbn, [&](int r, int n) { return -dUn[r * dv + nb0 + n]; },
                         [&](int n, int kk) { return sT[n * LK + kk]; },
                         [&](int r, int kk, float s) { dW[r * dk + kk] = (first ? 0.f : dW[r * dk + kk]) + s; });
    }
    for (int nb0 = 0; nb0 < dv; nb0 += NB) {
        const int nbn = min(NB, dv - nb0);
        const bool first = nb0 == 0;
        __syncthreads();
        for (int idx = threadIdx.x; idx < dk * nbn; idx += blockDim.x) {
            int kk = idx / nbn, n = idx - kk * nbn;
            sT[n * LK + kk] = dSo[(size_t)kk * dv + nb0 + n];
        }
        __syncthreads();
        bgemm<Tin, 4, 8>(len, dk, nbn, [&](int r, int n) { return Un[r * dv + nb0 + n]; },
                         [&](int n, int kk) { return sT[n * LK + kk]; },
                         [&](int r, int kk, float s) {
                             dK[r * dk + kk] = (first ? 0.f : dK[r * dk + kk]) + sE[r] * s;
                             atomicAdd(&set[r], s * Kn[r * dk + kk]);
                         });
    }
    __syncthreads();
    float *aux = w.aux + slot * (4 * C + 4);
    for (int r = threadIdx.x; r < len; r += blockDim.x) {
        aux[r] = sqt[r];
        aux[C + r] = set[r];
    }
    if (threadIdx.x == 0) aux[2 * C] = sred[0];
}

// The same three state products for bf16 inputs on the staged layout (the shapes of
// staged_ok): dO, dUnew, Unew and both states rounded to bf16 into row-major tiles,
// Q and K kept in fp32 for the row sums, <dS_out, S_in> accumulated in fp32 while
// the states are loaded.  512 threads; the 3 (C / 32)(d_k / 32) warp tiles of the
// three products are dealt round-robin to the warps.
__global__ void __launch_bounds__(512) k_bbig_st(Geo g, const __nv_bfloat16 *__restrict__ dO, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv;
    const int LV = spad(dv), LQ = dk + 4, ldv = ilog2(dv), ldk = ilog2(dk);
    extern __shared__ float sm[];
    float *sE = sm;                 // [C] exp(gamma_C - gamma_r)
    float *sG = sE + 64;            // [C] exp(gamma_r)
    float *sqt = sG + 64;           // [C] <Q_r, Y_r>
    float *set = sqt + 64;          // [C] <Kt_r, K_r>
    float *sred = set + 64;         // [4] <dS_out, S_in>
    float *Qs = sred + 4;           // [C][LQ] fp32
    float *Ks = Qs + C * LQ;        // [C][LQ] fp32
    __nv_bfloat16 *dOs = reinterpret_cast<__nv_bfloat16 *>(Ks + C * LQ);   // scale dO [C][LV]
    __nv_bfloat16 *dUs = dOs + C * LV;                       // dUnew [C][LV]
    __nv_bfloat16 *Us = dUs + C * LV;                        // Unew [C][LV]
    __nv_bfloat16 *Ss = Us + C * LV;                         // S_in [dk][LV]
    __nv_bfloat16 *dSs = Ss + dk * LV;                       // dS_out [dk][LV]
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *gam = w.gam + slot * C;
    const float gC = gam[len - 1], sc = g.scale;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) {
        // every row this CTA reads, into L2 before the staging loads below
        l2_prefetch(w.Qn + slot * C * dk, sizeof(float) * C * dk);
        l2_prefetch(w.Kn + slot * C * dk, sizeof(float) * C * dk);
        l2_prefetch(w.dUn + slot * C * dv, sizeof(float) * C * dv);
        l2_prefetch(w.Unew + slot * C * dv, sizeof(float) * C * dv);
        l2_prefetch(w.Sin + slot * dk * dv, sizeof(float) * dk * dv);
        l2_prefetch(w.dSo + slot * dk * dv, sizeof(float) * dk * dv);
        l2_prefetch(dO + row * dv, sizeof(__nv_bfloat16) * len * dv);
    }
    for (int r = threadIdx.x; r < C; r += blockDim.x) {
        sE[r] = r < len ? expf(gC - gam[r]) : 0.f;
        sG[r] = r < len ? expf(gam[r]) : 0.f;
        sqt[r] = 0.f;
        set[r] = 0.f;
    }
    if (threadIdx.x == 0) sred[0] = 0.f;
    {
        // the four row blocks in one batch of loads (512 threads: C d / 4 <= 4 x 512 pieces)
        float4 rq[4], rk[4], rdu[4], ru[4];
        reg_load(rq, w.Qn + slot * C * dk, C, dk, len);
        reg_load(rk, w.Kn + slot * C * dk, C, dk, len);
        reg_load(rdu, w.dUn + slot * C * dv, C, dv, len);
        reg_load(ru, w.Unew + slot * C * dv, C, dv, len);
        reg_put(rq, C, dk, [&](int r, int kk, float4 v) { *reinterpret_cast<float4 *>(Qs + r * LQ + kk) = v; });
        reg_put(rk, C, dk, [&](int r, int kk, float4 v) { *reinterpret_cast<float4 *>(Ks + r * LQ + kk) = v; });
        reg_put(rdu, C, dv, [&](int r, int n, float4 v) { put_bf4(dUs + r * LV + n, v, 1.f); });
        reg_put(ru, C, dv, [&](int r, int n, float4 v) { put_bf4(Us + r * LV + n, v, 1.f); });
    }
    {
        // both states, and <dS_out, S_in> in fp32 on the way
        const float4 *S4 = reinterpret_cast<const float4 *>(w.Sin + slot * dk * dv);
        const float4 *D4 = reinterpret_cast<const float4 *>(w.dSo + slot * dk * dv);
        const int n4 = (dk * dv) >> 2, lc4 = ldv - 2;
        float p = 0.f;
        for (int base = threadIdx.x; base < n4; base += blockDim.x * 4) {
            float4 a[4], d[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = base + u * blockDim.x;
                a[u] = e < n4 ? __ldg(S4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                d[u] = e < n4 ? __ldg(D4 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = base + u * blockDim.x;
                if (e >= n4) continue;
                p = fmaf(a[u].x, d[u].x, fmaf(a[u].y, d[u].y, fmaf(a[u].z, d[u].z, fmaf(a[u].w, d[u].w, p))));
                const int kk = e >> lc4, n = (e & ((1 << lc4) - 1)) << 2;
                put_bf4(Ss + kk * LV + n, a[u], 1.f);
                put_bf4(dSs + kk * LV + n, d[u], 1.f);
            }
        }
        p = warp_sum(p);
        __syncthreads();   // sred cleared
        if (lane == 0) atomicAdd(sred, p);
    }
    {
        // scale dO, 8 bf16 per 16-byte load
        const int n8 = (C * dv) >> 3, lc8 = ldv - 3;
        for (int base = threadIdx.x; base < n8; base += blockDim.x * 2) {
            uint4 v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int e = base + u * blockDim.x;
                v[u] = (e < n8 && (e >> lc8) < len) ? __ldg(reinterpret_cast<const uint4 *>(dO + row * dv) + e)
                                                    : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int e = base + u * blockDim.x;
                if (e >= n8) continue;
                const int r = e >> lc8, n = (e & ((1 << lc8) - 1)) << 3;
                const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    o[q] = bf16x2(sc * __uint_as_float(wv[q] << 16), sc * __uint_as_float(wv[q] & 0xFFFF0000u));
                *reinterpret_cast<uint4 *>(dOs + r * LV + n) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
    __syncthreads();
    float *dQ = w.dQ + slot * C * dk;
    float *dK = w.dK + slot * C * dk;
    float *dW = w.dW + slot * C * dk;
    const int gq = lane >> 2, t = lane & 3;
    const int ltn = ldk - 5, per = (C / 32) << ltn;   // warp tiles per product
    for (int tile = warp; tile < 3 * per; tile += nw) {
        const int prod = tile / per, tl = tile - prod * per;
        const int m0 = (tl >> ltn) * 32, n0 = (tl & ((1 << ltn) - 1)) * 32;
        float acc[2][4][4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[hh][jj][0] = acc[hh][jj][1] = acc[hh][jj][2] = acc[hh][jj][3] = 0.f;
        // Y = dO S_in^T, Z = dUnew S_in^T, X = Unew dS_out^T (rows r, columns kk, sum over n)
        const __nv_bfloat16 *A = prod == 0 ? dOs : (prod == 1 ? dUs : Us);
        const __nv_bfloat16 *B = prod == 2 ? dSs : Ss;
        tile_mma<false, false>(acc, A, LV, B, LV, m0, n0, dv);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int r = m0 + 16 * hh + gq + 8 * half;
                const bool live = r < len;
                float rs = 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int kk = n0 + 8 * jj + 2 * t;
                    const float v0 = acc[hh][jj][2 * half], v1 = acc[hh][jj][2 * half + 1];
                    if (prod == 0) {
                        if (live) *reinterpret_cast<float2 *>(dQ + r * dk + kk) = make_float2(sG[r] * v0, sG[r] * v1);
                        rs = fmaf(Qs[r * LQ + kk], v0, fmaf(Qs[r * LQ + kk + 1], v1, rs));
                    } else if (prod == 1) {
                        if (live) *reinterpret_cast<float2 *>(dW + r * dk + kk) = make_float2(-v0, -v1);
                    } else {
                        if (live) *reinterpret_cast<float2 *>(dK + r * dk + kk) = make_float2(sE[r] * v0, sE[r] * v1);
                        rs = fmaf(Ks[r * LQ + kk], v0, fmaf(Ks[r * LQ + kk + 1], v1, rs));
                    }
                }
                if (prod != 1) {
                    rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                    rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                    if (t == 0 && live) atomicAdd(prod == 0 ? &sqt[r] : &set[r], rs);
                }
            }
    }
    __syncthreads();
    float *aux = w.aux + slot * (4 * C + 4);
    for (int r = threadIdx.x; r < len; r += blockDim.x) {
        aux[r] = sqt[r];
        aux[C + r] = set[r];
    }
    if (threadIdx.x == 0) aux[2 * C] = sred[0];
}

// ----------------------------------------------------------------------------- backward per chunk
// Two kernels per chunk.  k_bchunk: K K^T, dP, the solve (I + A)^-1 and its
// adjoint, dT, and the gate / beta terms that need the C x C matrices; it hands
// dP o D, (I + A)^-1 and dKK to k_bgrad through the workspace, together with its
// partial d gamma and d beta.  k_bgrad: the C x d products into dq, dk, dv, the
// gate's reverse cumsum and the normalisation chain rule.  The split keeps each
// kernel's shared memory small enough for two (k_bchunk, bf16) or three (k_bgrad)
// 256-thread CTAs per SM.
template <class Tin>
__global__ void __launch_bounds__(256, 2) k_bchunk(Geo g, const Tin *__restrict__ v,
                                                const Tin *__restrict__ dO, Ws w)
{
    constexpr bool kStage = !std::is_same<Tin, __nv_bfloat16>::value;   // fp32: stage row operands
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv, LC = C + 1;
    const int LS = (dk > dv ? dk : dv) + 1;
    extern __shared__ float sm[];
    float *sKK = sm;                // K K^T
    float *sdP = sKK + C * LC;      // lower(dO Unew^T)
    float *sDP = sdP + C * LC;      // dP o D, later X = Linv^T dT diag(beta)
    float *sdT = sDP + C * LC;      // dT
    float *sLi = sdT + C * LC;      // (I + A)^-1
    float *sY = sLi + C * LC;       // A, then dA, then dKK
    // bf16 path: before the solve, sLi, sY and a pad hold two staged operand tiles
    __nv_bfloat16 *Ta = reinterpret_cast<__nv_bfloat16 *>(sLi);
    const int LT = spad(dk > dv ? dk : dv);
    __nv_bfloat16 *Tb = Ta + C * LT;
    float *sb = sY + C * LC + bchunk_pad(C, dk, dv);   // step sizes
    float *sg = sb + C;             // gamma
    float *sG = sg + C;             // exp(gamma)
    float *sdg = sG + C;            // d gamma (partial)
    float *sdb = sdg + C;           // d beta (partial)
    float *sS = sdb + C;            // fp32 only: [C][LS] staged rows (K, Unew, V)
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *Kn = w.Kn + slot * C * dk;
    const float *Un = w.Unew + slot * C * dv;
    const float *dUn = w.dUn + slot * C * dv;
    const float *Pg = w.P + slot * C * C;
    float *aux = w.aux + slot * (4 * C + 4);
    float *M3 = w.M3 + slot * 3 * C * C;   // dP o D | (I + A)^-1 | dKK
    const float *dW = w.dW + slot * C * dk;
    const float *gam = w.gam + slot * C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const float sc = g.scale;

    for (int r = threadIdx.x; r < len; r += blockDim.x) {
        sb[r] = w.eb[slot * C + r];
        sg[r] = gam[r];
        sG[r] = expf(gam[r]);
        sdg[r] = sG[r] * aux[r];      // q-term of d gamma
        sdb[r] = 0.f;
    }
    if (kStage) {
        for (int idx = threadIdx.x; idx < len * dk; idx += blockDim.x) {
            int r = idx / dk, c = idx - r * dk;
            sS[r * LS + c] = Kn[idx];
        }
    }
    __syncthreads();
    auto Dm = [&](int r, int i) { return i <= r ? expf(sg[r] - sg[i]) : 0.f; };
    auto Kt = [&](int kk, int i) { return kStage ? sS[i * LS + kk] : Kn[i * dk + kk]; };
    bool staged = false;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        staged = staged_ok(g) && (((uintptr_t)dO | (uintptr_t)v) & 15u) == 0;
        if (staged && threadIdx.x == 0) {
            // every row this CTA reads, into L2 before the staging loads below
            l2_prefetch(Kn, sizeof(float) * C * dk);
            l2_prefetch(dW, sizeof(float) * C * dk);
            l2_prefetch(Un, sizeof(float) * C * dv);
            l2_prefetch(dUn, sizeof(float) * C * dv);
            l2_prefetch(Pg, sizeof(float) * C * C);
            l2_prefetch(dO + row * dv, sizeof(__nv_bfloat16) * len * dv);
            l2_prefetch(v + row * dv, sizeof(__nv_bfloat16) * len * dv);
        }
        if (staged) {
            // the four C x C products on staged bf16 tiles, two tiles at a time
            const int ltc = ilog2(C) - 5, nt = 1 << (2 * ltc);   // warp tiles per C x C product
            auto each = [&](int nprod, auto prod) {
                for (int tile = warp; tile < nprod * nt; tile += nw) {
                    const int p = tile >> (2 * ltc), tl = tile & (nt - 1);
                    const int m0 = (tl >> ltc) * 32, n0 = (tl & ((1 << ltc) - 1)) * 32;
                    float acc[2][4][4];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) acc[hh][jj][0] = acc[hh][jj][1] = acc[hh][jj][2] = acc[hh][jj][3] = 0.f;
                    prod(p, m0, n0, acc);
                }
            };
            // element (r, i) of accumulator [hh][jj][e] in the tile at (m0, n0)
            auto at = [&](int m0, int n0, int hh, int jj, int e, int &r, int &i) {
                r = m0 + 16 * hh + (lane >> 2) + 8 * (e >> 1);
                i = n0 + 8 * jj + 2 * (lane & 3) + (e & 1);
            };
            // K K^T and dT = dW (diag(Gamma) K)^T
            const int LKt = spad(dk), LVt = spad(dv);
            {
                // K and dW in one batch of loads (C d / 4 <= 8 x 256 pieces)
                float4 ra[8], rb[8];
                reg_load(ra, Kn, C, dk, len);
                reg_load(rb, dW, C, dk, len);
                reg_put(ra, C, dk, [&](int r, int kk, float4 x) { put_bf4(Ta + r * LKt + kk, x, 1.f); });
                reg_put(rb, C, dk, [&](int r, int kk, float4 x) { put_bf4(Tb + r * LKt + kk, x, 1.f); });
            }
            __syncthreads();
            each(2, [&](int p, int m0, int n0, float (&acc)[2][4][4]) {
                tile_mma<false, false>(acc, p ? Tb : Ta, LKt, Ta, LKt, m0, n0, dk);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            int r, i;
                            at(m0, n0, hh, jj, e, r, i);
                            if (p == 0) sKK[r * LC + i] = acc[hh][jj][e];
                            else sdT[r * LC + i] = i < len ? sG[i] * acc[hh][jj][e] : 0.f;
                        }
            });
            __syncthreads();
            // dP = lower(scale dO Unew^T); scale dO and Unew in one batch of loads
            // (C d / 8 <= 4 x 256 and C d / 4 <= 8 x 256 pieces)
            {
                uint4 ro[4];
                float4 ru[8];
                reg_load_bf(ro, dO + row * dv, C, dv, len);
                reg_load(ru, Un, C, dv, len);
                reg_put_bf(ro, C, dv, [&](int r, int n, uint4 x) {
                    const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
                    uint32_t o[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        o[q] = bf16x2(sc * __uint_as_float(wv[q] << 16), sc * __uint_as_float(wv[q] & 0xFFFF0000u));
                    *reinterpret_cast<uint4 *>(Ta + r * LVt + n) = make_uint4(o[0], o[1], o[2], o[3]);
                });
                reg_put(ru, C, dv, [&](int r, int n, float4 x) { put_bf4(Tb + r * LVt + n, x, 1.f); });
            }
            __syncthreads();
            each(1, [&](int, int m0, int n0, float (&acc)[2][4][4]) {
                tile_mma<false, false>(acc, Ta, LVt, Tb, LVt, m0, n0, dv);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            int r, i;
                            at(m0, n0, hh, jj, e, r, i);
                            const bool keep = i <= r && r < len;
                            sdP[r * LC + i] = keep ? acc[hh][jj][e] : 0.f;
                            sDP[r * LC + i] = keep ? acc[hh][jj][e] * expf(sg[r] - sg[i]) : 0.f;
                        }
            });
            __syncthreads();
            // dT += dUnew V^T
            {
                // dUnew and V in one batch of loads
                float4 ru[8];
                uint4 rv[4];
                reg_load(ru, dUn, C, dv, len);
                reg_load_bf(rv, v + row * dv, C, dv, len);
                reg_put(ru, C, dv, [&](int r, int n, float4 x) { put_bf4(Ta + r * LVt + n, x, 1.f); });
                reg_put_bf(rv, C, dv, [&](int r, int n, uint4 x) { *reinterpret_cast<uint4 *>(Tb + r * LVt + n) = x; });
            }
            __syncthreads();
            each(1, [&](int, int m0, int n0, float (&acc)[2][4][4]) {
                tile_mma<false, false>(acc, Ta, LVt, Tb, LVt, m0, n0, dv);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            int r, i;
                            at(m0, n0, hh, jj, e, r, i);
                            if (i < len) sdT[r * LC + i] += acc[hh][jj][e];
                        }
            });
            __syncthreads();
        }
    }
    if (!staged) {
    // K K^T and the first half of dT = dW (diag(Gamma) K)^T + dUnew V^T
    bgemm<Tin, 4, 4>(len, len, dk, [&](int r, int kk) { return Kn[r * dk + kk]; }, Kt,
                     [&](int r, int i, float s) { sKK[r * LC + i] = s; });
    bgemm<Tin, 4, 4>(len, len, dk, [&](int r, int kk) { return dW[r * dk + kk]; },
                     [&](int kk, int i) { return sG[i] * Kt(kk, i); },
                     [&](int r, int i, float s) { sdT[r * LC + i] = s; });
    __syncthreads();
    if (kStage) {
        for (int idx = threadIdx.x; idx < len * dv; idx += blockDim.x) {
            int r = idx / dv, c = idx - r * dv;
            sS[r * LS + c] = Un[idx];
        }
        __syncthreads();
    }
    // dP = lower(scale dO Unew^T)
    bgemm<Tin, 4, 4>(len, len, dv, [&](int r, int n) { return sc * ld_in(dO + (row + r) * dv + n); },
                     [&](int n, int i) { return kStage ? sS[i * LS + n] : Un[i * dv + n]; },
                     [&](int r, int i, float s) {
                         sdP[r * LC + i] = (i <= r) ? s : 0.f;
                         sDP[r * LC + i] = (i <= r) ? s * expf(sg[r] - sg[i]) : 0.f;
                     });
    }
    for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
        int r = idx / len, i = idx - r * len;
        sY[r * LC + i] = (i < r) ? sb[r] * sKK[r * LC + i] * expf(sg[r] - sg[i]) : 0.f;
    }
    __syncthreads();
    bool solved = false;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        if (C == 64) {
            // blocked solve over the full 64 x 64 (A zero outside the chunk), as in k_prep
            for (int idx = threadIdx.x; idx < 64 * 64; idx += blockDim.x) {
                const int r = idx >> 6, c = idx & 63;
                if (r >= len || c >= len) sY[r * 65 + c] = 0.f;
            }
            __syncthreads();
            if (warp < 4) prep::solve_unit_lower_64<65>(sY, sLi, lane, warp, 1);
            __syncthreads();
            for (int idx = threadIdx.x; idx < 64 * 64; idx += blockDim.x) {
                const int r = idx >> 6, c = idx & 63;
                if (c > r) sLi[r * 65 + c] = 0.f;
            }
            solved = true;
        }
    }
    if (!solved) unit_lower_solve(sY, sLi, nullptr, len, LC);
    if (kStage) {
        for (int idx = threadIdx.x; idx < len * dv; idx += blockDim.x) {
            int r = idx / dv, c = idx - r * dv;
            sS[r * LS + c] = ld_in(v + (row + r) * dv + c);
        }
    }
    for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
        int r = idx / len, i = idx - r * len;
        M3[r * C + i] = sDP[r * LC + i];
    }
    __syncthreads();
    // dT += dUnew V^T (the staged path did it before the solve)
    if (!staged)
        bgemm<Tin, 4, 4>(len, len, dv, [&](int r, int n) { return dUn[r * dv + n]; },
                         [&](int n, int i) { return kStage ? sS[i * LS + n] : ld_in(v + (row + i) * dv + n); },
                         [&](int r, int i, float s) { sdT[r * LC + i] += s; });
    __syncthreads();
    if (staged && solved) {
        // the same tail on the full 64 x 64 (everything outside the chunk is zero):
        // d beta through T, X = Linv^T (dT diag(beta)) and dA = strict_lower(-X Linv^T)
        // on the tensor cores in tf32, then one elementwise pass for the gate and beta
        // sums and dKK
        for (int i = threadIdx.x; i < len; i += blockDim.x) {
            float a = 0.f;
            for (int r = i; r < len; ++r) a = fmaf(sLi[r * LC + i], sdT[r * LC + i], a);
            sdb[i] += a;
        }
        auto tiles64 = [&](auto A, auto B, auto St) {
            // four 32 x 32 tiles, warps 0..3
            if (warp < 4) {
                const int m0 = (warp >> 1) * 32, n0 = (warp & 1) * 32;
                float acc[2][4][4];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) acc[hh][jj][0] = acc[hh][jj][1] = acc[hh][jj][2] = acc[hh][jj][3] = 0.f;
                tile_tf32(acc, A, B, m0, n0, 64);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            St(m0 + 16 * hh + (lane >> 2) + 8 * (e >> 1), n0 + 8 * jj + 2 * (lane & 3) + (e & 1),
                               acc[hh][jj][e]);
            }
        };
        tiles64([&](int a, int r) { return sLi[r * LC + a]; },
                [&](int r, int bb) { return bb < len ? sdT[r * LC + bb] * sb[bb] : 0.f; },
                [&](int a, int bb, float x) { sDP[a * LC + bb] = x; });
        __syncthreads();
        tiles64([&](int a, int c) { return sDP[a * LC + c]; }, [&](int c, int bb) { return sLi[bb * LC + c]; },
                [&](int a, int bb, float x) { sY[a * LC + bb] = (bb < a) ? -x : 0.f; });
        __syncthreads();
        // F = dA o KK o D (beta sums) into sDP, E = beta_r F + dP o P (gate sums) into sdT,
        // and sY <- dKK = dA o beta_r o D
        for (int idx = threadIdx.x; idx < len * 64; idx += blockDim.x) {
            const int r = idx >> 6, i = idx & 63;
            float f = 0.f, e = 0.f, y = 0.f;
            if (i < len) {
                const float d = i <= r ? expf(sg[r] - sg[i]) : 0.f, dA = sY[r * LC + i];
                f = dA * sKK[r * LC + i] * d;
                e = fmaf(sb[r], f, i <= r ? sdP[r * LC + i] * Pg[r * C + i] : 0.f);
                y = dA * sb[r] * d;
            }
            sDP[r * LC + i] = f;
            sdT[r * LC + i] = e;
            sY[r * LC + i] = y;
        }
        __syncthreads();
        for (int r = warp; r < len; r += nw) {
            float db = 0.f, rs = 0.f;
            for (int i = lane; i < len; i += 32) {
                db += sDP[r * LC + i];
                rs += sdT[r * LC + i];
            }
            db = warp_sum(db);
            rs = warp_sum(rs);
            if (lane == 0) {
                sdb[r] += db;
                sdg[r] += rs;
            }
        }
        for (int i = warp; i < len; i += nw) {
            float cs = 0.f;
            for (int r = lane; r < len; r += 32) cs += sdT[r * LC + i];
            cs = warp_sum(cs);
            if (lane == 0) atomicAdd(&sdg[i], -cs);
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
            int r = idx / len, i = idx - r * len;
            M3[C * C + r * C + i] = sLi[r * LC + i];
            M3[2 * C * C + r * C + i] = sY[r * LC + i];
        }
        for (int r = threadIdx.x; r < len; r += blockDim.x) {
            aux[2 * C + 4 + r] = sdg[r];
            aux[3 * C + 4 + r] = sdb[r];
        }
        return;
    }
    // d beta through T = Linv diag(beta)
    for (int i = threadIdx.x; i < len; i += blockDim.x) {
        float a = 0.f;
        for (int r = i; r < len; ++r) a = fmaf(sLi[r * LC + i], sdT[r * LC + i], a);
        sdb[i] += a;
    }
    // X = Linv^T (dT diag(beta))
    rgemm<4, 4>(len, len, len, [&](int a, int r) { return sLi[r * LC + a]; },
                [&](int r, int bb) { return sdT[r * LC + bb] * sb[bb]; },
                [&](int a, int bb, float s) { sDP[a * LC + bb] = s; });
    __syncthreads();
    // dA = strict_lower(-X Linv^T)
    rgemm<4, 4>(len, len, len, [&](int a, int c) { return sDP[a * LC + c]; },
                [&](int c, int bb) { return sLi[bb * LC + c]; },
                [&](int a, int bb, float s) { sY[a * LC + bb] = (bb < a) ? -s : 0.f; });
    __syncthreads();
    // d beta from A, E = dD o D, d gamma row / column sums;  then Y <- dKK = dA o beta_r o D
    for (int r = warp; r < len; r += nw) {
        float db = 0.f, rs = 0.f;
        for (int i = lane; i < len; i += 32) {
            const float dA = sY[r * LC + i], Dri = Dm(r, i);
            db = fmaf(dA * sKK[r * LC + i], Dri, db);
            rs += dA * sb[r] * sKK[r * LC + i] * Dri + (i <= r ? sdP[r * LC + i] * Pg[r * C + i] : 0.f);
        }
        db = warp_sum(db);
        rs = warp_sum(rs);
        if (lane == 0) {
            sdb[r] += db;
            sdg[r] += rs;
        }
    }
    for (int i = warp; i < len; i += nw) {
        float cs = 0.f;
        for (int r = lane; r < len; r += 32)
            cs += sY[r * LC + i] * sb[r] * sKK[r * LC + i] * Dm(r, i) +
                  (i <= r ? sdP[r * LC + i] * Pg[r * C + i] : 0.f);
        cs = warp_sum(cs);
        if (lane == 0) atomicAdd(&sdg[i], -cs);
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
        int r = idx / len, i = idx - r * len;
        M3[C * C + r * C + i] = sLi[r * LC + i];
        M3[2 * C * C + r * C + i] = sY[r * LC + i] * sb[r] * Dm(r, i);
    }
    for (int r = threadIdx.x; r < len; r += blockDim.x) {
        aux[2 * C + 4 + r] = sdg[r];
        aux[3 * C + 4 + r] = sdb[r];
    }
}

template <class Tin>
__global__ void __launch_bounds__(256, 3) k_bgrad(Geo g, const Tin *__restrict__ q,
                                               const Tin *__restrict__ k,
                                               Tin *__restrict__ dq, Tin *__restrict__ dkout,
                                               Tin *__restrict__ dvout,
                                               Tin *__restrict__ dbeta,
                                               float *__restrict__ dg, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv, LC = C + 1;
    extern __shared__ float sm[];
    float *sDP = sm;                // dP o D
    float *sLi = sDP + C * LC;      // (I + A)^-1
    float *sY = sLi + C * LC;       // dKK
    float *sb = sY + C * LC;        // step sizes
    float *sG = sb + C;             // exp(gamma)
    float *sdg = sG + C;            // d gamma
    float *sdb = sdg + C;           // d beta
    float *se = sdb + C;            // e_r (K~ gate term)
    float *sk2 = se + C;            // <dGK_r, K_r>
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *Qn = w.Qn + slot * C * dk;
    const float *Kn = w.Kn + slot * C * dk;
    const float *dUn = w.dUn + slot * C * dv;
    const float *aux = w.aux + slot * (4 * C + 4);
    const float *M3 = w.M3 + slot * 3 * C * C;
    float *dQ = w.dQ + slot * C * dk;
    float *dK = w.dK + slot * C * dk;
    const float *dW = w.dW + slot * C * dk;
    const float *gam = w.gam + slot * C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const float gC = gam[len - 1];

    for (int r = threadIdx.x; r < len; r += blockDim.x) {
        sb[r] = w.eb[slot * C + r];
        sG[r] = expf(gam[r]);
        se[r] = expf(gC - gam[r]) * aux[C + r];
        sdg[r] = aux[2 * C + 4 + r];
        sdb[r] = aux[3 * C + 4 + r];
        sk2[r] = 0.f;
    }
    for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
        int r = idx / len, i = idx - r * len;
        sDP[r * LC + i] = M3[r * C + i];
        sLi[r * LC + i] = M3[C * C + r * C + i];
        sY[r * LC + i] = M3[2 * C * C + r * C + i];
    }
    __syncthreads();
    // dQ += (dP o D) K;  dK += (dP o D)^T Q
    bgemm<Tin, 4, 8>(len, dk, len, [&](int r, int i) { return sDP[r * LC + i]; },
                     [&](int i, int kk) { return Kn[i * dk + kk]; },
                     [&](int r, int kk, float s) { dQ[r * dk + kk] += s; });
    bgemm<Tin, 4, 8>(len, dk, len, [&](int r, int i) { return sDP[i * LC + r]; },
                     [&](int i, int kk) { return Qn[i * dk + kk]; },
                     [&](int r, int kk, float s) { dK[r * dk + kk] += s; });
    __syncthreads();
    // dGK = T^T dW (T = Linv diag(beta)); dK += Gamma dGK; d gamma += Gamma <dGK, K>;  dV = T^T dUnew
    bgemm<Tin, 4, 8>(len, dk, len, [&](int r, int i) { return sLi[i * LC + r]; },
                     [&](int i, int kk) { return dW[i * dk + kk]; },
                     [&](int r, int kk, float s) {
                         const float a = sb[r] * s;
                         dK[r * dk + kk] += sG[r] * a;
                         atomicAdd(&sk2[r], a * Kn[r * dk + kk]);
                     });
    bgemm<Tin, 4, 8>(len, dv, len, [&](int r, int i) { return sLi[i * LC + r]; },
                     [&](int i, int n) { return dUn[i * dv + n]; },
                     [&](int r, int n, float s) { st_out(dvout + (row + r) * dv + n, sb[r] * s); });
    __syncthreads();
    // dK += (dKK + dKK^T) K
    bgemm<Tin, 4, 8>(len, dk, len, [&](int r, int i) { return sY[r * LC + i] + sY[i * LC + r]; },
                     [&](int i, int kk) { return Kn[i * dk + kk]; },
                     [&](int r, int kk, float s) { dK[r * dk + kk] += s; });
    __syncthreads();
    if (threadIdx.x == 0) {
        float es = 0.f;
        for (int r = 0; r < len; ++r) {
            sdg[r] += sG[r] * sk2[r] - se[r];
            es += se[r];
        }
        sdg[len - 1] += es + expf(gC) * aux[2 * C];
        // d g = reverse cumulative sum of d gamma within the chunk
        float acc = 0.f;
        for (int r = len - 1; r >= 0; --r) {
            acc += sdg[r];
            if (dg) dg[row + r] = acc;
        }
    }
    // the normalisation chain rule for dq, dk
    for (int r = warp; r < len; r += nw) {
        const Tin *qr = q + (row + r) * dk;
        const Tin *kr = k + (row + r) * dk;
        float sq = 0.f, sk = 0.f, pq = 0.f, pk = 0.f;
        for (int kk = lane; kk < dk; kk += 32) {
            float x = ld_in(qr + kk), y = ld_in(kr + kk);
            sq = fmaf(x, x, sq);
            sk = fmaf(y, y, sk);
            pq = fmaf(Qn[r * dk + kk], dQ[r * dk + kk], pq);
            pk = fmaf(Kn[r * dk + kk], dK[r * dk + kk], pk);
        }
        sq = warp_sum(sq); sk = warp_sum(sk); pq = warp_sum(pq); pk = warp_sum(pk);
        float rq = g.l2norm ? rsqrtf(sq + g.eps) : 1.f;
        float rk = g.l2norm ? rsqrtf(sk + g.eps) : 1.f;
        // sdb holds d/d(step size).  Longhorn's step e = b / (1 + b kap), kap = k^T k:
        // de/db = (1 - e kap)^2 and de/dkap = -e^2, with d kap / dk = 2 k
        float db = sdb[r], dkap = 0.f;
        if (g.longhorn) {
            const float kap = sk * rk * rk, e = sb[r], f = fmaf(-e, kap, 1.f);
            dkap = -db * e * e;
            db *= f * f;
            pk = fmaf(2.f * dkap, kap, pk);
        }
        for (int kk = lane; kk < dk; kk += 32) {
            float a = dQ[r * dk + kk], c = fmaf(2.f * dkap, Kn[r * dk + kk], dK[r * dk + kk]);
            if (g.l2norm) {
                a = rq * (a - Qn[r * dk + kk] * pq);
                c = rk * (c - Kn[r * dk + kk] * pk);
            }
            st_out(dq + (row + r) * dk + kk, a);
            st_out(dkout + (row + r) * dk + kk, c);
        }
        if (lane == 0) st_out(dbeta + row + r, db);
    }
}

// k_bgrad for bf16 inputs on the staged layout (the shapes of staged_ok): K, Q, dW,
// dUnew and the three C x C matrices from k_bchunk rounded to bf16 into row-major
// tiles (entries past the chunk masked to zero), the products on ldmatrix fragments.
// Warp w owns one 32 x 32 tile of dQ and dK (and of dV) and chains the products
// through its registers; the normalisation chain rule then runs per row as in k_bgrad.
__global__ void __launch_bounds__(256, 2) k_bgrad_st(Geo g, const __nv_bfloat16 *__restrict__ q,
                                                    const __nv_bfloat16 *__restrict__ k,
                                                    __nv_bfloat16 *__restrict__ dq,
                                                    __nv_bfloat16 *__restrict__ dkout,
                                                    __nv_bfloat16 *__restrict__ dvout,
                                                    __nv_bfloat16 *__restrict__ dbeta,
                                                    float *__restrict__ dg, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv;
    const int LK = spad(dk), LV = spad(dv), LC = spad(C);
    extern __shared__ float sm[];
    float *sb = sm;                 // [C] step sizes
    float *sG = sb + 64;            // [C] exp(gamma)
    float *sdg = sG + 64;           // [C] d gamma
    float *sdb = sdg + 64;          // [C] d beta
    float *se = sdb + 64;           // [C] e_r (K~ gate term)
    float *sk2 = se + 64;           // [C] <dGK_r, K_r>
    __nv_bfloat16 *Kb = reinterpret_cast<__nv_bfloat16 *>(sk2 + 64);   // K [C][LK]
    __nv_bfloat16 *Qb = Kb + C * LK;                         // Q [C][LK]
    __nv_bfloat16 *dWb = Qb + C * LK;                        // dW [C][LK]
    __nv_bfloat16 *dUb = dWb + C * LK;                       // dUnew [C][LV] (first the fp32 dKK)
    const int dub = C * LV > 2 * C * C ? C * LV : 2 * C * C; // elements: room for either
    __nv_bfloat16 *DPb = dUb + dub;                          // dP o D [C][LC]
    __nv_bfloat16 *Lib = DPb + C * LC;                       // (I + A)^-1 [C][LC]
    __nv_bfloat16 *YYb = Lib + C * LC;                       // dKK + dKK^T [C][LC]
    float *Yf = reinterpret_cast<float *>(dUb);              // dKK fp32 [C][C], before dUnew is staged
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *Qn = w.Qn + slot * C * dk;
    const float *Kn = w.Kn + slot * C * dk;
    const float *aux = w.aux + slot * (4 * C + 4);
    const float *M3 = w.M3 + slot * 3 * C * C;
    float *dQ = w.dQ + slot * C * dk;
    float *dK = w.dK + slot * C * dk;
    const float *gam = w.gam + slot * C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) {
        // every workspace row this CTA reads, into L2 before the staging loads below
        l2_prefetch(Kn, sizeof(float) * C * dk);
        l2_prefetch(Qn, sizeof(float) * C * dk);
        l2_prefetch(w.dW + slot * C * dk, sizeof(float) * C * dk);
        l2_prefetch(M3, sizeof(float) * 3 * C * C);
        l2_prefetch(w.dUn + slot * C * dv, sizeof(float) * C * dv);
        l2_prefetch(dQ, sizeof(float) * C * dk);
        l2_prefetch(dK, sizeof(float) * C * dk);
    }
    const float gC = gam[len - 1];
    const int lC = ilog2(C);

    for (int r = threadIdx.x; r < C; r += blockDim.x) {
        const bool live = r < len;
        sb[r] = live ? w.eb[slot * C + r] : 0.f;
        sG[r] = live ? expf(gam[r]) : 0.f;
        se[r] = live ? expf(gC - gam[r]) * aux[C + r] : 0.f;
        sdg[r] = live ? aux[2 * C + 4 + r] : 0.f;
        sdb[r] = live ? aux[3 * C + 4 + r] : 0.f;
        sk2[r] = 0.f;
    }
    // the C x C matrices, entries with r or i past the chunk set to zero
    auto mask4 = [&](int i, float4 v) {
        return make_float4(i < len ? v.x : 0.f, i + 1 < len ? v.y : 0.f, i + 2 < len ? v.z : 0.f, i + 3 < len ? v.w : 0.f);
    };
    {
        // K and Q in one batch of loads, then dW with the three C x C matrices
        // (C d / 4 <= 8 x 256 and C C / 4 <= 4 x 256 pieces)
        float4 ra[8], rb[8];
        reg_load(ra, Kn, C, dk, len);
        reg_load(rb, Qn, C, dk, len);
        reg_put(ra, C, dk, [&](int r, int kk, float4 v) { put_bf4(Kb + r * LK + kk, v, 1.f); });
        reg_put(rb, C, dk, [&](int r, int kk, float4 v) { put_bf4(Qb + r * LK + kk, v, 1.f); });
        float4 rc[8], r0[4], r1[4], r2[4];
        reg_load(rc, w.dW + slot * C * dk, C, dk, len);
        reg_load(r0, M3, C, C, len);
        reg_load(r1, M3 + C * C, C, C, len);
        reg_load(r2, M3 + 2 * C * C, C, C, len);
        reg_put(rc, C, dk, [&](int r, int kk, float4 v) { put_bf4(dWb + r * LK + kk, v, 1.f); });
        reg_put(r0, C, C, [&](int r, int i, float4 v) { put_bf4(DPb + r * LC + i, mask4(i, v), 1.f); });
        reg_put(r1, C, C, [&](int r, int i, float4 v) { put_bf4(Lib + r * LC + i, mask4(i, v), 1.f); });
        reg_put(r2, C, C, [&](int r, int i, float4 v) { *reinterpret_cast<float4 *>(Yf + r * C + i) = mask4(i, v); });
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < C * C / 2; idx += blockDim.x) {
        const int r = (2 * idx) >> lC, i = (2 * idx) & (C - 1);
        put_bf2(YYb + r * LC + i, Yf[r * C + i] + Yf[i * C + r], Yf[r * C + i + 1] + Yf[(i + 1) * C + r]);
    }
    __syncthreads();
    stage_f32(w.dUn + slot * C * dv, C, dv, len, [&](int r, int n, float4 v) { put_bf4(dUb + r * LV + n, v, 1.f); });
    __syncthreads();

    const int gq = lane >> 2, t = lane & 3;
    auto zero = [&](float (&a)[2][4][4]) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) a[hh][jj][0] = a[hh][jj][1] = a[hh][jj][2] = a[hh][jj][3] = 0.f;
    };
    // (row, column) of element e (0..3) of accumulator [hh][jj] in the tile at (m0, n0)
    auto rc = [&](int m0, int n0, int hh, int jj, int e, int &r, int &c) {
        r = m0 + 16 * hh + gq + 8 * (e >> 1);
        c = n0 + 8 * jj + 2 * t + (e & 1);
    };
    const int ltk = ilog2(dk) - 5, ntk = (C / 32) << ltk;
    if (warp < ntk) {
        const int m0 = (warp >> ltk) * 32, n0 = (warp & ((1 << ltk) - 1)) * 32;
        float acc[2][4][4];
        // dQ += (dP o D) K
        zero(acc);
        tile_mma<false, true>(acc, DPb, LC, Kb, LK, m0, n0, C);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int r, c;
                    rc(m0, n0, hh, jj, e, r, c);
                    if (r < len) {
                        float2 *p = reinterpret_cast<float2 *>(dQ + r * dk + c);
                        const float2 o = *p;
                        *p = make_float2(o.x + acc[hh][jj][e], o.y + acc[hh][jj][e + 1]);
                    }
                }
        // dGK = T^T dW (T = Linv diag(beta)): d gamma gets G_r <beta_r dGK_r, K_r>, and
        // dK starts from G_r beta_r dGK
        zero(acc);
        tile_mma<true, true>(acc, Lib, LC, dWb, LK, m0, n0, C);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int r = m0 + 16 * hh + gq + 8 * half;
                float rs = 0.f;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int c = n0 + 8 * jj + 2 * t;
                    float &a0 = acc[hh][jj][2 * half], &a1 = acc[hh][jj][2 * half + 1];
                    a0 *= sb[r];
                    a1 *= sb[r];
                    const uint32_t kw = *reinterpret_cast<const uint32_t *>(Kb + r * LK + c);
                    rs = fmaf(a0, __uint_as_float(kw << 16), fmaf(a1, __uint_as_float(kw & 0xFFFF0000u), rs));
                    a0 *= sG[r];
                    a1 *= sG[r];
                }
                rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                if (t == 0 && r < len) atomicAdd(&sk2[r], rs);
            }
        // dK += (dP o D)^T Q + (dKK + dKK^T) K, on top of G beta dGK
        tile_mma<true, true>(acc, DPb, LC, Qb, LK, m0, n0, C);
        tile_mma<false, true>(acc, YYb, LC, Kb, LK, m0, n0, C);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int r, c;
                    rc(m0, n0, hh, jj, e, r, c);
                    if (r < len) {
                        float2 *p = reinterpret_cast<float2 *>(dK + r * dk + c);
                        const float2 o = *p;
                        *p = make_float2(o.x + acc[hh][jj][e], o.y + acc[hh][jj][e + 1]);
                    }
                }
    }
    const int ltv = ilog2(dv) - 5, ntv = (C / 32) << ltv;
    for (int tile = warp; tile < ntv; tile += nw) {
        // dV = T^T dUnew
        const int m0 = (tile >> ltv) * 32, n0 = (tile & ((1 << ltv) - 1)) * 32;
        float acc[2][4][4];
        zero(acc);
        tile_mma<true, true>(acc, Lib, LC, dUb, LV, m0, n0, C);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r, c;
                    rc(m0, n0, hh, jj, e, r, c);
                    if (r < len) st_out(dvout + (row + r) * dv + c, sb[r] * acc[hh][jj][e]);
                }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float es = 0.f;
        for (int r = 0; r < len; ++r) {
            sdg[r] += sG[r] * sk2[r] - se[r];
            es += se[r];
        }
        sdg[len - 1] += es + expf(gC) * aux[2 * C];
        // d g = reverse cumulative sum of d gamma within the chunk
        float acc = 0.f;
        for (int r = len - 1; r >= 0; --r) {
            acc += sdg[r];
            if (dg) dg[row + r] = acc;
        }
    }
    // the normalisation chain rule for dq, dk: two rows per warp at a time, every
    // load of a row issued before any of it is used (d_k <= 128: at most 4 per lane)
    const int ne = dk >> 5;
    for (int r0 = 2 * warp; r0 < len; r0 += 2 * nw) {
        float xq[2][4], xk[2][4], Qv[2][4], Kv[2][4], a[2][4], c[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int r = r0 + rr;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kk = lane + 32 * e;
                const bool on = r < len && e < ne;
                xq[rr][e] = on ? ld_in(q + (row + r) * dk + kk) : 0.f;
                xk[rr][e] = on ? ld_in(k + (row + r) * dk + kk) : 0.f;
                Qv[rr][e] = on ? Qn[r * dk + kk] : 0.f;
                Kv[rr][e] = on ? Kn[r * dk + kk] : 0.f;
                a[rr][e] = on ? dQ[r * dk + kk] : 0.f;
                c[rr][e] = on ? dK[r * dk + kk] : 0.f;
            }
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int r = r0 + rr;
            if (r >= len) break;
            float sq = 0.f, sk = 0.f, pq = 0.f, pk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sq = fmaf(xq[rr][e], xq[rr][e], sq);
                sk = fmaf(xk[rr][e], xk[rr][e], sk);
                pq = fmaf(Qv[rr][e], a[rr][e], pq);
                pk = fmaf(Kv[rr][e], c[rr][e], pk);
            }
            sq = warp_sum(sq); sk = warp_sum(sk); pq = warp_sum(pq); pk = warp_sum(pk);
            const float rq = g.l2norm ? rsqrtf(sq + g.eps) : 1.f;
            const float rk = g.l2norm ? rsqrtf(sk + g.eps) : 1.f;
            // sdb holds d/d(step size).  Longhorn's step e = b / (1 + b kap), kap = k^T k:
            // de/db = (1 - e kap)^2 and de/dkap = -e^2, with d kap / dk = 2 k
            float db = sdb[r], dkap = 0.f;
            if (g.longhorn) {
                const float kap = sk * rk * rk, ee = sb[r], f = fmaf(-ee, kap, 1.f);
                dkap = -db * ee * ee;
                db *= f * f;
                pk = fmaf(2.f * dkap, kap, pk);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (e >= ne) break;
                const int kk = lane + 32 * e;
                float av = a[rr][e], cv = fmaf(2.f * dkap, Kv[rr][e], c[rr][e]);
                if (g.l2norm) {
                    av = rq * (av - Qv[rr][e] * pq);
                    cv = rk * (cv - Kv[rr][e] * pk);
                }
                st_out(dq + (row + r) * dk + kk, av);
                st_out(dkout + (row + r) * dk + kk, cv);
            }
            if (lane == 0) st_out(dbeta + row + r, db);
        }
    }
}

// k_prep for bf16 inputs on the staged layout (the shapes of staged_ok, 16-byte
// aligned v): the normalised K and Q rounded to bf16 into row-major tiles as the norms
// are taken, V copied as it is, and the four products (A, P, W, U) on ldmatrix
// fragments; T and T diag(Gamma) are staged the same way after the solve.
__global__ void __launch_bounds__(256) k_prep_st(Geo g, const __nv_bfloat16 *__restrict__ q,
                                                 const __nv_bfloat16 *__restrict__ k,
                                                 const __nv_bfloat16 *__restrict__ v,
                                                 const __nv_bfloat16 *__restrict__ beta,
                                                 const float *__restrict__ gate, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv, LC = C + 1;
    const int LK = spad(dk), LV = spad(dv), LT = spad(C);
    extern __shared__ float sm[];
    float *sA = sm;                                 // [C][LC] A, for the solve
    float *sT = sA + C * LC;                        // [C][LC] (I + A)^-1, or T
    float *sb = sT + C * LC;                        // [C] step sizes (beta, or Longhorn's)
    float *sg = sb + 64;                            // [C] gamma
    float *sG = sg + 64;                            // [C] exp(gamma)
    __nv_bfloat16 *Kb = reinterpret_cast<__nv_bfloat16 *>(sG + 64);   // normalised K [C][LK]
    __nv_bfloat16 *Qb = Kb + C * LK;                // normalised Q [C][LK]
    __nv_bfloat16 *Vb = Qb + C * LK;                // V [C][LV]
    __nv_bfloat16 *Tb = Vb + C * LV;                // T [C][LT]
    __nv_bfloat16 *TGb = Tb + C * LT;               // T diag(Gamma) [C][LT]
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) {
        // the chunk's q, k, v rows into L2 before the per-row loads below
        l2_prefetch(q + row * dk, sizeof(__nv_bfloat16) * len * dk);
        l2_prefetch(k + row * dk, sizeof(__nv_bfloat16) * len * dk);
        l2_prefetch(v + row * dv, sizeof(__nv_bfloat16) * len * dv);
    }

    for (int r = warp; r < C; r += nw) {
        if (r >= len) {
            for (int c = lane; c < dk; c += 32) {
                Kb[r * LK + c] = __float2bfloat16_rn(0.f);
                Qb[r * LK + c] = __float2bfloat16_rn(0.f);
            }
            if (lane == 0) sb[r] = 0.f;
            continue;
        }
        const __nv_bfloat16 *kr = k + (row + r) * dk;
        const __nv_bfloat16 *qr = q + (row + r) * dk;
        float sk = 0.f, sq = 0.f;
        for (int c = lane; c < dk; c += 32) {
            float x = ld_in(kr + c), y = ld_in(qr + c);
            sk = fmaf(x, x, sk);
            sq = fmaf(y, y, sq);
        }
        sk = warp_sum(sk);
        sq = warp_sum(sq);
        float rk = g.l2norm ? rsqrtf(sk + g.eps) : 1.f;
        float rq = g.l2norm ? rsqrtf(sq + g.eps) : 1.f;
        if (lane == 0) {
            // the token's step size: beta, or Longhorn's beta / (1 + beta k^T k) with
            // k^T k = |k|^2 rk^2 of the key the update uses
            float bt = ld_in(beta + row + r);
            if (g.longhorn) bt = bt / fmaf(bt, sk * rk * rk, 1.f);
            sb[r] = bt;
            w.eb[slot * C + r] = bt;
        }
        for (int c = lane; c < dk; c += 32) {
            float x = ld_in(kr + c) * rk, y = ld_in(qr + c) * rq;
            Kb[r * LK + c] = __float2bfloat16_rn(x);
            Qb[r * LK + c] = __float2bfloat16_rn(y);
            w.Kn[slot * C * dk + r * dk + c] = x;
            w.Qn[slot * C * dk + r * dk + c] = y;
        }
    }
    if (warp == 0) {
        // within-chunk cumulative log-gate, two rows per lane (C <= 64)
        float x0 = (gate && lane < len) ? gate[row + lane] : 0.f;
        float x1 = (gate && lane + 32 < len) ? gate[row + lane + 32] : 0.f;
        if (__any_sync(0xffffffffu, x0 > 0.f || x1 > 0.f) && lane == 0)
            raise_status(g.status, kStatusPositiveGate);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float y0 = __shfl_up_sync(0xffffffffu, x0, o), y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (lane >= o) { x0 += y0; x1 += y1; }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        sg[lane] = x0;
        sG[lane] = lane < len ? expf(x0) : 0.f;
        sg[lane + 32] = x1;
        sG[lane + 32] = lane + 32 < len ? expf(x1) : 0.f;
        if (lane < len) w.gam[slot * C + lane] = x0;
        if (lane + 32 < len) w.gam[slot * C + lane + 32] = x1;
    }
    {
        // V, 8 bf16 per 16-byte load (rows past the chunk zero)
        const int n8 = (C * dv) >> 3, lc8 = ilog2(dv) - 3;
        for (int e = threadIdx.x; e < n8; e += blockDim.x) {
            const int r = e >> lc8, n = (e & ((1 << lc8) - 1)) << 3;
            *reinterpret_cast<uint4 *>(Vb + r * LV + n) =
                r < len ? __ldg(reinterpret_cast<const uint4 *>(v + row * dv) + e) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    __syncthreads();
    const int ltc = ilog2(C) - 5, nt = 1 << (2 * ltc);   // warp tiles of a C x C product
    auto at = [&](int m0, int n0, int hh, int jj, int e, int &r, int &c) {
        r = m0 + 16 * hh + (lane >> 2) + 8 * (e >> 1);
        c = n0 + 8 * jj + 2 * (lane & 3) + (e & 1);
    };
    auto zero = [&](float (&a)[2][4][4]) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) a[hh][jj][0] = a[hh][jj][1] = a[hh][jj][2] = a[hh][jj][3] = 0.f;
    };
    // A = strict_lower(diag(beta) (K K^T o D)),  P = lower(Q K^T o D)
    float *Pg = w.P + slot * C * C;
    for (int tile = warp; tile < 2 * nt; tile += nw) {
        const int p = tile >> (2 * ltc), tl = tile & (nt - 1);
        const int m0 = (tl >> ltc) * 32, n0 = (tl & ((1 << ltc) - 1)) * 32;
        float acc[2][4][4];
        zero(acc);
        tile_mma<false, false>(acc, p ? Qb : Kb, LK, Kb, LK, m0, n0, dk);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int r, i;
                    at(m0, n0, hh, jj, e, r, i);
                    const bool live = r < len && i < len;
                    if (p == 0) sA[r * LC + i] = (live && i < r) ? sb[r] * acc[hh][jj][e] * expf(sg[r] - sg[i]) : 0.f;
                    else Pg[r * C + i] = (live && i <= r) ? acc[hh][jj][e] * expf(sg[r] - sg[i]) : 0.f;
                }
    }
    __syncthreads();
    // T = (I + A)^-1 diag(beta)
    if (C == 64) {
        if (warp < 4) prep::solve_unit_lower_64<65>(sA, sT, lane, warp, 1);
        __syncthreads();
        for (int idx = threadIdx.x; idx < C * C; idx += blockDim.x) {
            const int r = idx >> 6, i = idx & 63;
            const float t = (i <= r && r < len) ? sT[r * LC + i] * sb[i] : 0.f;
            Tb[r * LT + i] = __float2bfloat16_rn(t);
            TGb[r * LT + i] = __float2bfloat16_rn(t * sG[i]);
        }
    } else {
        unit_lower_solve(sA, sT, sb, len, LC);
        __syncthreads();
        for (int idx = threadIdx.x; idx < C * C; idx += blockDim.x) {
            const int r = idx >> (ltc + 5), i = idx & (C - 1);
            const float t = (i <= r && r < len) ? sT[r * LC + i] : 0.f;
            Tb[r * LT + i] = __float2bfloat16_rn(t);
            TGb[r * LT + i] = __float2bfloat16_rn(t * sG[i]);
        }
    }
    __syncthreads();
    // W = T diag(Gamma) K,  U = T V
    const int ltk = ilog2(dk) - 5, ltv = ilog2(dv) - 5;
    const int ntw = (C / 32) << ltk, ntu = (C / 32) << ltv;
    for (int tile = warp; tile < ntw + ntu; tile += nw) {
        const bool isw = tile < ntw;
        const int tl = isw ? tile : tile - ntw, lt = isw ? ltk : ltv, D = isw ? dk : dv;
        const int m0 = (tl >> lt) * 32, n0 = (tl & ((1 << lt) - 1)) * 32;
        float acc[2][4][4];
        zero(acc);
        if (isw) tile_mma<false, true>(acc, TGb, LT, Kb, LK, m0, n0, C);
        else tile_mma<false, true>(acc, Tb, LT, Vb, LV, m0, n0, C);
        float *dst = (isw ? w.W + slot * C * dk : w.U + slot * C * dv);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    int r, c;
                    at(m0, n0, hh, jj, e, r, c);
                    if (r < len) *reinterpret_cast<float2 *>(dst + r * D + c) = make_float2(acc[hh][jj][e], acc[hh][jj][e + 1]);
                }
    }
}

// k_out for bf16 inputs on the staged layout (the shapes of staged_ok):
// O = diag(Gamma) Q S_in + P Unew from bf16 tiles (Q and P row-major, S_in and Unew
// read down their rows with ldmatrix.trans), one 32 x 32 output tile per warp.
__global__ void __launch_bounds__(256) k_out_st(Geo g, __nv_bfloat16 *__restrict__ o, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv;
    const int LK = spad(dk), LV = spad(dv), LC = spad(C);
    extern __shared__ float sm[];
    float *sG = sm;                                                       // [C] exp(gamma)
    __nv_bfloat16 *Qb = reinterpret_cast<__nv_bfloat16 *>(sG + 64);       // diag(Gamma) Q [C][LK]
    __nv_bfloat16 *Sb = Qb + C * LK;                                      // S_in [dk][LV]
    __nv_bfloat16 *Pb = Sb + dk * LV;                                     // P [C][LC]
    __nv_bfloat16 *Ub = Pb + C * LC;                                      // Unew [C][LV]
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *gam = w.gam + slot * C;
    for (int r = threadIdx.x; r < C; r += blockDim.x) sG[r] = r < len ? expf(gam[r]) : 0.f;
    __syncthreads();
    stage_f32(w.Qn + slot * C * dk, C, dk, len, [&](int r, int kk, float4 x) { put_bf4(Qb + r * LK + kk, x, sG[r]); });
    stage_f32(w.Sin + slot * dk * dv, dk, dv, dk, [&](int kk, int n, float4 x) { put_bf4(Sb + kk * LV + n, x, 1.f); });
    // P's entries outside the chunk are zero (written so by k_prep_st)
    stage_f32(w.P + slot * C * C, C, C, len, [&](int r, int i, float4 x) { put_bf4(Pb + r * LC + i, x, 1.f); });
    stage_f32(w.Unew + slot * C * dv, C, dv, len, [&](int r, int n, float4 x) { put_bf4(Ub + r * LV + n, x, 1.f); });
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int ltv = ilog2(dv) - 5, nt = (C / 32) << ltv;
    const float sc = g.scale;
    for (int tile = warp; tile < nt; tile += nw) {
        const int m0 = (tile >> ltv) * 32, n0 = (tile & ((1 << ltv) - 1)) * 32;
        float acc[2][4][4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[hh][jj][0] = acc[hh][jj][1] = acc[hh][jj][2] = acc[hh][jj][3] = 0.f;
        tile_mma<false, true>(acc, Qb, LK, Sb, LV, m0, n0, dk);
        tile_mma<false, true>(acc, Pb, LC, Ub, LV, m0, n0, C);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = m0 + 16 * hh + (lane >> 2) + 8 * (e >> 1), n = n0 + 8 * jj + 2 * (lane & 3) + (e & 1);
                    if (r < len) st_out(o + (row + r) * dv + n, sc * acc[hh][jj][e]);
                }
    }
}

// ----------------------------------------------------------------------------- host launchers
static size_t smem_prep(const Geo &g)
{
    const size_t LK = g.dk + 1, LC = g.C + 1;
    return sizeof(float) * (g.C * LK + g.C * (LK > (size_t)g.dv ? LK : g.dv) + 2 * g.C * LC + 3 * g.C);
}
static size_t smem_scan(const Geo &g, int BV)
{
    return sizeof(float) * (g.dk * BV + g.C * BV + g.C + 2 * (size_t)g.C * (g.dk + 1));
}
static size_t smem_out(const Geo &g)
{
    return sizeof(float) * (g.C + (size_t)g.C * (g.dk + g.C + 1) + (size_t)(g.dk + g.C) * 65);
}
static size_t smem_bscan(const Geo &g, int BV) { return sizeof(float) * (g.dk * BV + 2 * g.C * BV + 2 * g.C); }
static size_t smem_bbig(const Geo &g)
{
    return sizeof(float) * ((g.dv < 128 ? g.dv : 128) * (g.dk + 1) + 4 * g.C + 4);
}
template <class Tin>
static size_t smem_bchunk(const Geo &g)
{
    const size_t LC = g.C + 1, LS = (g.dk > g.dv ? g.dk : g.dv) + 1;
    const size_t stage = std::is_same<Tin, __nv_bfloat16>::value ? 0 : g.C * LS;
    return sizeof(float) * (6 * g.C * LC + bchunk_pad(g.C, g.dk, g.dv) + 5 * g.C + stage);
}
static size_t smem_bgrad(const Geo &g) { return sizeof(float) * (3 * (size_t)g.C * (g.C + 1) + 6 * g.C); }

static int slice_width(const Geo &g) { return g.dv < 64 ? g.dv : 64; }

static size_t smem_scan_st(const Geo &g)
{
    const size_t LS = g.dv + 8, LK = spad(g.dk), LV = spad(g.dv);
    return sizeof(float) * ((size_t)g.dk * LS + 64 + (size_t)g.C * g.dv) +
           2 * (2 * g.C * LK + (size_t)(g.dk + g.C) * LV);
}
static size_t smem_bbig_st(const Geo &g)
{
    const size_t LV = spad(g.dv), LQ = g.dk + 4;
    return sizeof(float) * (4 * 64 + 4 + 2 * (size_t)g.C * LQ) + 2 * (3 * g.C + 2 * (size_t)g.dk) * LV;
}
static size_t smem_bgrad_st(const Geo &g)
{
    const size_t LK = spad(g.dk), LV = spad(g.dv), LC = spad(g.C);
    const size_t dub = (size_t)g.C * LV * 2 > (size_t)g.C * g.C * 4 ? (size_t)g.C * LV * 2 : (size_t)g.C * g.C * 4;
    return sizeof(float) * 6 * 64 + 2 * (3 * (size_t)g.C * LK + 3 * (size_t)g.C * LC) + dub;
}
static size_t smem_prep_st(const Geo &g)
{
    const size_t LC = g.C + 1, LK = spad(g.dk), LV = spad(g.dv), LT = spad(g.C);
    return sizeof(float) * (2 * g.C * LC + 3 * 64) + 2 * (size_t)g.C * (2 * LK + LV + 2 * LT);
}
static size_t smem_out_st(const Geo &g)
{
    const size_t LK = spad(g.dk), LV = spad(g.dv), LC = spad(g.C);
    return sizeof(float) * 64 + 2 * ((size_t)g.C * LK + (size_t)g.dk * LV + (size_t)g.C * LC + (size_t)g.C * LV);
}
static size_t smem_bscan_st(const Geo &g)
{
    const size_t LS = g.dv + 8, LC = spad(g.C), LK = spad(g.dk), LV = spad(g.dv);
    return sizeof(float) * ((size_t)g.dk * LS + 128) +
           2 * (g.C * LC + 3 * g.C * LK + (size_t)(2 * g.C + g.dk) * LV);
}
template <class Tin>
static bool use_staged(const Geo &g, const void *dO = nullptr)
{
    return std::is_same<Tin, __nv_bfloat16>::value && staged_ok(g) && ((uintptr_t)dO & 15u) == 0;
}

template <class K>
static cudaError_t set_smem(K kernel, size_t bytes)
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <class Tin>
static cudaError_t forward_states(const Geo &g, const Tin *q, const Tin *k, const Tin *v,
                                  const Tin *beta, const float *gate, const float *h0, float *hT,
                                  const Ws &w, cudaStream_t st)
{
    cudaError_t e;
    bool prepped = false;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        if (use_staged<Tin>(g, v)) {
            if ((e = set_smem(k_prep_st, smem_prep_st(g))) != cudaSuccess) return e;
            if (g.NC > 0) k_prep_st<<<dim3(g.NC, g.H), 256, smem_prep_st(g), st>>>(g, q, k, v, beta, gate, w);
            prepped = true;
        }
    }
    if (!prepped) {
        if ((e = set_smem(k_prep<Tin>, smem_prep(g))) != cudaSuccess) return e;
        if (g.NC > 0) k_prep<Tin><<<dim3(g.NC, g.H), 256, smem_prep(g), st>>>(g, q, k, v, beta, gate, w);
    }
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
    if (use_staged<Tin>(g)) {
        if ((e = set_smem(k_scan_st, smem_scan_st(g))) != cudaSuccess) return e;
        if (g.N > 0) k_scan_st<<<dim3(g.N, g.H), 512, smem_scan_st(g), st>>>(g, h0, hT, w);
        return cudaPeekAtLastError();
    }
    const int BV = slice_width(g);
    if ((e = set_smem(k_scan<Tin>, smem_scan(g, BV))) != cudaSuccess) return e;
    if (g.N > 0)
        k_scan<Tin><<<dim3(g.N, g.H, (g.dv + BV - 1) / BV), 256, smem_scan(g, BV), st>>>(g, h0, hT, w, BV);
    return cudaPeekAtLastError();
}

template <class Tin>
cudaError_t fwd(const Geo &g, const Tin *q, const Tin *k, const Tin *v, const Tin *beta,
                const float *gate, const float *h0, Tin *o, float *hT, const Ws &w,
                cudaStream_t st)
{
    cudaError_t e = forward_states(g, q, k, v, beta, gate, h0, hT, w, st);
    if (e != cudaSuccess) return e;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        if (use_staged<Tin>(g, v)) {
            if ((e = set_smem(k_out_st, smem_out_st(g))) != cudaSuccess) return e;
            if (g.NC > 0) k_out_st<<<dim3(g.NC, g.H), 256, smem_out_st(g), st>>>(g, o, w);
            return cudaPeekAtLastError();
        }
    }
    if ((e = set_smem(k_out<Tin>, smem_out(g))) != cudaSuccess) return e;
    if (g.NC > 0) k_out<Tin><<<dim3(g.NC, g.H), 256, smem_out(g), st>>>(g, o, w);
    return cudaPeekAtLastError();
}

// GDN_BWD_STAGED=1 keeps the staged warp-level per-chunk kernels for shapes the
// tcgen05 per-chunk backward takes (used by the tests to compare the two).
static bool force_staged_bwd()
{
    const char *e = getenv("GDN_BWD_STAGED");
    return e && e[0] && e[0] != '0';
}

bool bwd_uses_tc(const Geo &g, int dtype, const void *q, const void *k, const void *v, const void *dO)
{
    return dtype == DN_BF16 && staged_ok(g) && btc::supports(g, dtype) && !force_staged_bwd() &&
           ((((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)dO) & 15u) == 0);
}

// GDN_BSCAN_STAGED=1 keeps the warp-level reverse scan over the packages (k_bscan_pk)
// where the tcgen05 one would run (used by the tests to compare the two).
static bool staged_bscan()
{
    const char *e = getenv("GDN_BSCAN_STAGED");
    return e && e[0] && e[0] != '0';
}

bool bwd_uses_coop(const Geo &g, int dtype)
{
    for (const char *name : {"GDN_BWD_RECOMPUTE", "GDN_FORCE_GENERAL"}) {
        const char *e = getenv(name);
        if (e && e[0] && e[0] != '0') return false;
    }
    const void *aligned = (const void *)(uintptr_t)256;
    return bwd_uses_tc(g, dtype, aligned, aligned, aligned, aligned) && g.C == 64 && g.dk == 128 &&
           g.dv == 128 && coop::available() && coop::supports(g, dtype);
}

template <class Tin>
cudaError_t bwd(const Geo &g, const Tin *q, const Tin *k, const Tin *v, const Tin *beta,
                const float *gate, const float *h0, const Tin *dO, const float *dhT, Tin *dq,
                Tin *dk, Tin *dv, Tin *dbeta, float *dg, float *dh0, const Ws &w,
                cudaStream_t st)
{
    cudaError_t e;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        if (w.keep && bwd_uses_tc(g, DN_BF16, q, k, v, dO)) {
            // the cooperative forward writes every chunk's package, S_in and Unew; the
            // reverse scan reads the packages; then the tcgen05 per-chunk gradients
            const coop::Emit em{w.keep, w.Sin_b, w.Un_b};
            if (!w.saved && (e = coop::fwd(g, q, k, v, beta, gate, h0, nullptr, nullptr, w.coop_ws,
                                           w.coop_bytes, g.status, st, &em)) != cudaSuccess)
                return e;
            if (bsc::supports(g, DN_BF16) && !staged_bscan()) {
                // the reverse scan on tcgen05, dS resident in TMEM
                if ((e = bsc::scan(g, k, dO, dhT, dh0, w.keep, coop::package_layout(g), w.dSo_b, w.dUn_b,
                                   st)) != cudaSuccess)
                    return e;
            } else {
                if ((e = set_smem(k_bscan_pk, smem_bscan_st(g))) != cudaSuccess) return e;
                if (g.N > 0)
                    k_bscan_pk<<<dim3(g.N, g.H), 512, smem_bscan_st(g), st>>>(g, k, dO, dhT, dh0, w.keep,
                                                                              coop::package_layout(g), w);
                if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
            }
            return btc::grads(g, q, k, v, beta, gate, dO, w.Sin_b, w.dSo_b, w.Un_b, w.dUn_b, dq, dk, dv,
                              dbeta, dg, st);
        }
        if (bwd_uses_tc(g, DN_BF16, q, k, v, dO)) {
            // recompute and the two staged scans, writing bf16 states and Unew / dUnew
            // (over the fp32 arrays they replace), then the tcgen05 per-chunk gradients
            Ws w2 = w;
            w2.Sin_b = reinterpret_cast<__nv_bfloat16 *>(w.Sin);
            w2.dSo_b = reinterpret_cast<__nv_bfloat16 *>(w.dSo);
            w2.Un_b = reinterpret_cast<__nv_bfloat16 *>(w.Unew);
            w2.dUn_b = reinterpret_cast<__nv_bfloat16 *>(w.dUn);
            if ((e = forward_states(g, q, k, v, beta, gate, h0, nullptr, w2, st)) != cudaSuccess) return e;
            if ((e = set_smem(k_bscan_st, smem_bscan_st(g))) != cudaSuccess) return e;
            if (g.N > 0) k_bscan_st<<<dim3(g.N, g.H), 512, smem_bscan_st(g), st>>>(g, dO, dhT, dh0, w2);
            if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
            return btc::grads(g, q, k, v, beta, gate, dO, w2.Sin_b, w2.dSo_b, w2.Un_b, w2.dUn_b, dq, dk, dv,
                              dbeta, dg, st);
        }
    }
    e = forward_states(g, q, k, v, beta, gate, h0, nullptr, w, st);
    if (e != cudaSuccess) return e;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        if (use_staged<Tin>(g, dO)) {
            if ((e = set_smem(k_bscan_st, smem_bscan_st(g))) != cudaSuccess) return e;
            if (g.N > 0) k_bscan_st<<<dim3(g.N, g.H), 512, smem_bscan_st(g), st>>>(g, dO, dhT, dh0, w);
        }
    }
    if (!use_staged<Tin>(g, dO)) {
        const int BV = slice_width(g);
        if ((e = set_smem(k_bscan<Tin>, smem_bscan(g, BV))) != cudaSuccess) return e;
        if (g.N > 0)
            k_bscan<Tin><<<dim3(g.N, g.H, (g.dv + BV - 1) / BV), 256, smem_bscan(g, BV), st>>>(
                g, dO, dhT, dh0, w, BV);
    }
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        if (use_staged<Tin>(g, dO)) {
            if ((e = set_smem(k_bbig_st, smem_bbig_st(g))) != cudaSuccess) return e;
            if (g.NC > 0) k_bbig_st<<<dim3(g.NC, g.H), 512, smem_bbig_st(g), st>>>(g, dO, w);
        }
    }
    if (!use_staged<Tin>(g, dO)) {
        if ((e = set_smem(k_bbig<Tin>, smem_bbig(g))) != cudaSuccess) return e;
        if (g.NC > 0) k_bbig<Tin><<<dim3(g.NC, g.H), 512, smem_bbig(g), st>>>(g, dO, w);
    }
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
    if ((e = set_smem(k_bchunk<Tin>, smem_bchunk<Tin>(g))) != cudaSuccess) return e;
    if (g.NC > 0) k_bchunk<Tin><<<dim3(g.NC, g.H), 256, smem_bchunk<Tin>(g), st>>>(g, v, dO, w);
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
    if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        if (use_staged<Tin>(g, dO)) {
            if ((e = set_smem(k_bgrad_st, smem_bgrad_st(g))) != cudaSuccess) return e;
            if (g.NC > 0)
                k_bgrad_st<<<dim3(g.NC, g.H), 256, smem_bgrad_st(g), st>>>(g, q, k, dq, dk, dv, dbeta, dg, w);
            return cudaPeekAtLastError();
        }
    }
    if ((e = set_smem(k_bgrad<Tin>, smem_bgrad(g))) != cudaSuccess) return e;
    if (g.NC > 0)
        k_bgrad<Tin><<<dim3(g.NC, g.H), 256, smem_bgrad(g), st>>>(g, q, k, dq, dk, dv, dbeta, dg, w);
    return cudaPeekAtLastError();
}

template cudaError_t fwd<float>(const Geo &, const float *, const float *, const float *,
                                const float *, const float *, const float *, float *, float *,
                                const Ws &, cudaStream_t);
template cudaError_t fwd<__nv_bfloat16>(const Geo &, const __nv_bfloat16 *, const __nv_bfloat16 *,
                                        const __nv_bfloat16 *, const __nv_bfloat16 *, const float *,
                                        const float *, __nv_bfloat16 *, float *, const Ws &,
                                        cudaStream_t);
template cudaError_t bwd<float>(const Geo &, const float *, const float *, const float *,
                                const float *, const float *, const float *, const float *,
                                const float *, float *, float *, float *, float *, float *,
                                float *, const Ws &, cudaStream_t);
template cudaError_t bwd<__nv_bfloat16>(const Geo &, const __nv_bfloat16 *, const __nv_bfloat16 *,
                                        const __nv_bfloat16 *, const __nv_bfloat16 *, const float *,
                                        const float *, const __nv_bfloat16 *, const float *,
                                        __nv_bfloat16 *, __nv_bfloat16 *, __nv_bfloat16 *,
                                        __nv_bfloat16 *, float *, float *, const Ws &,
                                        cudaStream_t);

}  // namespace gen
}  // namespace gdn
