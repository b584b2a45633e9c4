// General chunk kernels: fp32 arithmetic on the CUDA cores, any head dim up to
// 128, chunk 16/32/64, float32 or bfloat16 inputs, gated or not, packed or not.
//
// These kernels carry the fp32 workload (whose 1e-4 tolerance tensor-core
// operands cannot meet) and every shape the tcgen05 fast path does not take.
// They follow the chunk form of "Parallelizing Linear Transformers with the
// Delta Rule over Sequence Length" (WY / UT representation, chunk-state scan)
// with the gates of "Gated DeltaNet" folded in as within-chunk cumulative
// log-decays:
//   prep  : per chunk, parallel       normalise q,k; gamma; A; T; W; U
//   scan  : per (seq, head, dv-slice) Unew = U - W S; S <- Gamma_C S + Kt^T Unew
//   out   : per chunk, parallel       O = diag(Gamma) Q S + lower(QK^T o D) Unew
// and the backward (chunk states recomputed by prep+scan, then):
//   bscan : per (seq, head, dv-slice), last chunk first:
//           dUnew = lower(..)^T dO + Kt dS;  dS <- Gamma_C dS + (Gamma Q)^T dO - W^T dUnew
//   bchunk: per chunk, parallel       every input gradient of the chunk.
#include "common.cuh"
#include "general.h"

namespace gdn {
namespace gen {

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Block-cooperative small GEMM: out(m, n) = sum_k A(m, k) B(k, n), handed to St.
template <class FA, class FB, class FS>
__device__ __forceinline__ void bgemm(int M, int N, int K, FA A, FB B, FS St)
{
    for (int idx = threadIdx.x; idx < M * N; idx += blockDim.x) {
        int m = idx / N, n = idx - m * N;
        float s = 0.f;
        for (int k = 0; k < K; ++k) s = fmaf(A(m, k), B(k, n), s);
        St(m, n, s);
    }
}

// Column-parallel forward substitution: X = (I + A)^-1 diag(d), A strictly lower
// (len x len, row stride C).  Thread j solves column j on its own.
__device__ __forceinline__ void unit_lower_solve(const float *A, float *X, const float *d,
                                                 int len, int C)
{
    for (int jc = threadIdx.x; jc < len; jc += blockDim.x) {
        for (int r = 0; r < len; ++r) {
            float x;
            if (r < jc) {
                x = 0.f;
            } else if (r == jc) {
                x = d ? d[jc] : 1.f;
            } else {
                float s = 0.f;
                for (int i = jc; i < r; ++i) s = fmaf(A[r * C + i], X[i * C + jc], s);
                x = -s;
            }
            X[r * C + jc] = x;
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
    const int C = g.C, dk = g.dk, dv = g.dv;
    extern __shared__ float sm[];
    float *sK = sm;               // [C][dk] normalised keys
    float *sA = sK + C * dk;      // [C][C]
    float *sT = sA + C * C;       // [C][C]
    float *sb = sT + C * C;       // [C] beta
    float *sg = sb + C;           // [C] gamma
    float *sG = sg + C;           // [C] exp(gamma)
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
        for (int c = lane; c < dk; c += 32) {
            float x = ld_in(kr + c) * rk;
            sK[r * dk + c] = x;
            w.Kn[slot * C * dk + r * dk + c] = x;
            w.Qn[slot * C * dk + r * dk + c] = ld_in(qr + c) * rq;
        }
    }
    if (threadIdx.x == 0) {
        float acc = 0.f;
        for (int r = 0; r < len; ++r) {
            acc += gate ? gate[row + r] : 0.f;
            sg[r] = acc;
            sG[r] = expf(acc);
            sb[r] = ld_in(beta + row + r);
            w.gam[slot * C + r] = acc;
        }
    }
    __syncthreads();
    // A = strict_lower(diag(beta) (K K^T o D))
    bgemm(len, len, dk, [&](int m, int kk) { return sK[m * dk + kk]; },
          [&](int kk, int n) { return sK[n * dk + kk]; },
          [&](int m, int n, float s) {
              sA[m * C + n] = (n < m) ? sb[m] * s * expf(sg[m] - sg[n]) : 0.f;
          });
    __syncthreads();
    unit_lower_solve(sA, sT, sb, len, C);   // T = (I + A)^-1 diag(beta)
    __syncthreads();
    for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
        int r = idx / len, c = idx - r * len;
        w.Tm[slot * C * C + r * C + c] = sT[r * C + c];
    }
    // W = T diag(Gamma) K,  U = T V
    bgemm(len, dk, len, [&](int m, int i) { return sT[m * C + i]; },
          [&](int i, int n) { return sG[i] * sK[i * dk + n]; },
          [&](int m, int n, float s) { w.W[slot * C * dk + m * dk + n] = s; });
    bgemm(len, dv, len, [&](int m, int i) { return sT[m * C + i]; },
          [&](int i, int n) { return ld_in(v + (row + i) * dv + n); },
          [&](int m, int n, float s) { w.U[slot * C * dv + m * dv + n] = s; });
}

// ----------------------------------------------------------------------------- scan
__global__ void __launch_bounds__(256) k_scan(Geo g, const float *__restrict__ h0,
                                              float *__restrict__ hT, Ws w, int BV)
{
    const int s = blockIdx.x, h = blockIdx.y, n0 = blockIdx.z * BV;
    const int nb = min(BV, g.dv - n0);
    const int C = g.C, dk = g.dk, dv = g.dv;
    int b, t0, L, j0, nch;
    seq_of(g, s, b, t0, L, j0, nch);
    extern __shared__ float sm[];
    float *sS = sm;               // [dk][BV]
    float *sU = sS + dk * BV;     // [C][BV]
    float *sE = sU + C * BV;      // [C] exp(gamma_C - gamma_r)
    const size_t sidx = ((size_t)s * g.H + h) * dk * dv;
    for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
        int kk = idx / nb, n = idx - kk * nb;
        sS[kk * BV + n] = h0 ? h0[sidx + (size_t)kk * dv + n0 + n] : 0.f;
    }
    __syncthreads();
    for (int c = 0; c < nch; ++c) {
        const int len = min(C, L - c * C);
        const size_t slot = (size_t)(j0 + c) * g.H + h;
        const float *gam = w.gam + slot * C;
        const float gC = gam[len - 1];
        for (int r = threadIdx.x; r < len; r += blockDim.x) sE[r] = expf(gC - gam[r]);
        for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
            int kk = idx / nb, n = idx - kk * nb;
            w.Sin[slot * dk * dv + (size_t)kk * dv + n0 + n] = sS[kk * BV + n];
        }
        const float *W = w.W + slot * C * dk;
        const float *U = w.U + slot * C * dv;
        float *Un = w.Unew + slot * C * dv;
        bgemm(len, nb, dk, [&](int r, int kk) { return W[r * dk + kk]; },
              [&](int kk, int n) { return sS[kk * BV + n]; },
              [&](int r, int n, float acc) {
                  float u = U[r * dv + n0 + n] - acc;
                  sU[r * BV + n] = u;
                  Un[r * dv + n0 + n] = u;
              });
        __syncthreads();
        const float *Kn = w.Kn + slot * C * dk;
        const float GC = expf(gC);
        bgemm(dk, nb, len, [&](int kk, int r) { return sE[r] * Kn[r * dk + kk]; },
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
    float *sP = sm;            // [C][C]
    float *sG = sP + C * C;    // [C]
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *gam = w.gam + slot * C;
    const float *Qn = w.Qn + slot * C * dk;
    const float *Kn = w.Kn + slot * C * dk;
    const float *Sin = w.Sin + slot * dk * dv;
    const float *Un = w.Unew + slot * C * dv;
    for (int r = threadIdx.x; r < len; r += blockDim.x) sG[r] = expf(gam[r]);
    bgemm(len, len, dk, [&](int r, int kk) { return Qn[r * dk + kk]; },
          [&](int kk, int i) { return Kn[i * dk + kk]; },
          [&](int r, int i, float s) { sP[r * C + i] = (i <= r) ? s * expf(gam[r] - gam[i]) : 0.f; });
    __syncthreads();
    for (int idx = threadIdx.x; idx < len * dv; idx += blockDim.x) {
        int r = idx / dv, n = idx - r * dv;
        float a = 0.f, bsum = 0.f;
        for (int kk = 0; kk < dk; ++kk) a = fmaf(Qn[r * dk + kk], Sin[(size_t)kk * dv + n], a);
        for (int i = 0; i <= r; ++i) bsum = fmaf(sP[r * C + i], Un[i * dv + n], bsum);
        st_out(o + (row + r) * dv + n, g.scale * fmaf(sG[r], a, bsum));
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
    float *sP = sdO + C * BV;      // [C][C]
    float *sE = sP + C * C;        // [C]
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
        bgemm(len, len, dk, [&](int r, int kk) { return Qn[r * dk + kk]; },
              [&](int kk, int i) { return Kn[i * dk + kk]; },
              [&](int r, int i, float v) { sP[r * C + i] = (i <= r) ? v * expf(gam[r] - gam[i]) : 0.f; });
        __syncthreads();
        // dUnew(i, n) = sum_r P(r, i) dO(r, n) + sum_kk exp(gC - gam_i) K(i, kk) dS(kk, n)
        float *dUg = w.dUn + slot * C * dv;
        for (int idx = threadIdx.x; idx < len * nb; idx += blockDim.x) {
            int i = idx / nb, n = idx - i * nb;
            float a = 0.f, e = 0.f;
            for (int r = i; r < len; ++r) a = fmaf(sP[r * C + i], sdO[r * BV + n], a);
            for (int kk = 0; kk < dk; ++kk) e = fmaf(Kn[i * dk + kk], sdS[kk * BV + n], e);
            float u = fmaf(sE[i], e, a);
            sdU[i * BV + n] = u;
            dUg[i * dv + n0 + n] = u;
        }
        __syncthreads();
        // dS <- Gamma_C dS + (Gamma Q)^T dO - W^T dUnew
        const float GC = expf(gC);
        for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
            int kk = idx / nb, n = idx - kk * nb;
            float acc = GC * sdS[kk * BV + n];
            for (int r = 0; r < len; ++r) {
                acc = fmaf(sG[r] * Qn[r * dk + kk], sdO[r * BV + n], acc);
                acc = fmaf(-W[r * dk + kk], sdU[r * BV + n], acc);
            }
            sdS[kk * BV + n] = acc;
        }
        __syncthreads();
    }
    if (dh0) {
        for (int idx = threadIdx.x; idx < dk * nb; idx += blockDim.x) {
            int kk = idx / nb, n = idx - kk * nb;
            dh0[sidx + (size_t)kk * dv + n0 + n] = sdS[kk * BV + n];
        }
    }
}

// ----------------------------------------------------------------------------- backward per chunk
template <class Tin>
__global__ void __launch_bounds__(256) k_bchunk(Geo g, const Tin *__restrict__ q,
                                                const Tin *__restrict__ k,
                                                const Tin *__restrict__ v,
                                                const Tin *__restrict__ beta,
                                                const Tin *__restrict__ dO,
                                                Tin *__restrict__ dq, Tin *__restrict__ dkout,
                                                Tin *__restrict__ dvout,
                                                Tin *__restrict__ dbeta,
                                                float *__restrict__ dg, Ws w)
{
    const int j = blockIdx.x, h = blockIdx.y;
    int b, t0, len, seq, local;
    if (!chunk_of(g, j, b, t0, len, seq, local)) return;
    const int C = g.C, dk = g.dk, dv = g.dv;
    extern __shared__ float sm[];
    float *sD = sm;                 // D_ri = exp(gam_r - gam_i), i <= r
    float *sKK = sD + C * C;        // K K^T
    float *sQK = sKK + C * C;       // Q K^T
    float *sLi = sQK + C * C;       // (I + A)^-1
    float *sdP = sLi + C * C;       // lower(dO Unew^T)
    float *sdT = sdP + C * C;       // dT
    float *sX = sdT + C * C;        // A, later Linv^T dT diag(beta)
    float *sY = sX + C * C;         // dA, then dKK
    float *sb = sY + C * C;         // beta
    float *sg = sb + C;             // gamma
    float *sG = sg + C;             // exp(gamma)
    float *sE = sG + C;             // exp(gamma_C - gamma)
    float *sdg = sE + C;            // d gamma
    float *sdb = sdg + C;           // d beta
    float *se = sdb + C;            // e_r (K~ gate term)
    float *sred = se + C;           // [1] <dS_out, S_in>
    const size_t row = ((size_t)b * g.H + h) * g.T + t0;
    const size_t slot = (size_t)j * g.H + h;
    const float *Qn = w.Qn + slot * C * dk;
    const float *Kn = w.Kn + slot * C * dk;
    const float *Sin = w.Sin + slot * dk * dv;
    const float *dSo = w.dSo + slot * dk * dv;
    const float *Un = w.Unew + slot * C * dv;
    const float *dUn = w.dUn + slot * C * dv;
    float *dQ = w.dQ + slot * C * dk;
    float *dK = w.dK + slot * C * dk;
    float *dW = w.dW + slot * C * dk;
    const float *gam = w.gam + slot * C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const float gC = gam[len - 1];
    const float sc = g.scale;

    for (int r = threadIdx.x; r < len; r += blockDim.x) {
        sb[r] = ld_in(beta + row + r);
        sg[r] = gam[r];
        sG[r] = expf(gam[r]);
        sE[r] = expf(gC - gam[r]);
        sdg[r] = 0.f;
        sdb[r] = 0.f;
    }
    if (threadIdx.x == 0) sred[0] = 0.f;
    __syncthreads();
    for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
        int r = idx / len, i = idx - r * len;
        sD[r * C + i] = (i <= r) ? expf(sg[r] - sg[i]) : 0.f;
    }
    bgemm(len, len, dk, [&](int r, int kk) { return Kn[r * dk + kk]; },
          [&](int kk, int i) { return Kn[i * dk + kk]; },
          [&](int r, int i, float s) { sKK[r * C + i] = s; });
    bgemm(len, len, dk, [&](int r, int kk) { return Qn[r * dk + kk]; },
          [&](int kk, int i) { return Kn[i * dk + kk]; },
          [&](int r, int i, float s) { sQK[r * C + i] = s; });
    bgemm(len, len, dv, [&](int r, int n) { return sc * ld_in(dO + (row + r) * dv + n); },
          [&](int n, int i) { return Un[i * dv + n]; },
          [&](int r, int i, float s) { sdP[r * C + i] = (i <= r) ? s : 0.f; });
    __syncthreads();
    for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
        int r = idx / len, i = idx - r * len;
        sX[r * C + i] = (i < r) ? sb[r] * sKK[r * C + i] * sD[r * C + i] : 0.f;
    }
    __syncthreads();
    unit_lower_solve(sX, sLi, nullptr, len, C);
    // Rows of dQ / dK / dW: one warp per row; also the q-term of d gamma and e_r.
    for (int r = warp; r < len; r += nw) {
        float qterm = 0.f, eterm = 0.f;
        for (int kk = lane; kk < dk; kk += 32) {
            float y = 0.f, kt = 0.f, wv = 0.f;
            for (int n = 0; n < dv; ++n) {
                float sin_kn = Sin[(size_t)kk * dv + n];
                y = fmaf(sc * ld_in(dO + (row + r) * dv + n), sin_kn, y);
                kt = fmaf(Un[r * dv + n], dSo[(size_t)kk * dv + n], kt);
                wv = fmaf(-dUn[r * dv + n], sin_kn, wv);
            }
            float a = 0.f, c2 = 0.f;
            for (int i = 0; i <= r; ++i) a = fmaf(sdP[r * C + i] * sD[r * C + i], Kn[i * dk + kk], a);
            for (int i = r; i < len; ++i) c2 = fmaf(sdP[i * C + r] * sD[i * C + r], Qn[i * dk + kk], c2);
            dQ[r * dk + kk] = fmaf(sG[r], y, a);
            dK[r * dk + kk] = fmaf(sE[r], kt, c2);
            dW[r * dk + kk] = wv;
            qterm = fmaf(Qn[r * dk + kk], y, qterm);
            eterm = fmaf(kt, Kn[r * dk + kk], eterm);
        }
        qterm = warp_sum(qterm);
        eterm = warp_sum(eterm);
        if (lane == 0) {
            sdg[r] += sG[r] * qterm;
            se[r] = sE[r] * eterm;
        }
    }
    // <dS_out, S_in>
    {
        float p = 0.f;
        for (int idx = threadIdx.x; idx < dk * dv; idx += blockDim.x) p = fmaf(dSo[idx], Sin[idx], p);
        p = warp_sum(p);
        if (lane == 0) atomicAdd(sred, p);
    }
    __syncthreads();
    // dT = dW (diag(Gamma) K)^T + dUnew V^T
    bgemm(len, len, dk + dv,
          [&](int r, int x) { return x < dk ? dW[r * dk + x] : dUn[r * dv + (x - dk)]; },
          [&](int x, int i) {
              return x < dk ? sG[i] * Kn[i * dk + x] : ld_in(v + (row + i) * dv + (x - dk));
          },
          [&](int r, int i, float s) { sdT[r * C + i] = s; });
    __syncthreads();
    // dGK = T^T dW (T = Linv diag(beta)); dK += Gamma dGK; d gamma += Gamma <dGK, K>
    for (int r = warp; r < len; r += nw) {
        float s2 = 0.f;
        for (int kk = lane; kk < dk; kk += 32) {
            float a = 0.f;
            for (int i = r; i < len; ++i) a = fmaf(sLi[i * C + r], dW[i * dk + kk], a);
            a *= sb[r];
            dK[r * dk + kk] += sG[r] * a;
            s2 = fmaf(a, Kn[r * dk + kk], s2);
        }
        s2 = warp_sum(s2);
        if (lane == 0) sdg[r] += sG[r] * s2;
        // dV = T^T dUnew
        for (int n = lane; n < dv; n += 32) {
            float a = 0.f;
            for (int i = r; i < len; ++i) a = fmaf(sLi[i * C + r], dUn[i * dv + n], a);
            st_out(dvout + (row + r) * dv + n, sb[r] * a);
        }
    }
    // d beta (through T = Linv diag(beta)) and X = Linv^T (dT diag(beta))
    for (int i = threadIdx.x; i < len; i += blockDim.x) {
        float a = 0.f;
        for (int r = i; r < len; ++r) a = fmaf(sLi[r * C + i], sdT[r * C + i], a);
        sdb[i] += a;
    }
    bgemm(len, len, len, [&](int a, int r) { return sLi[r * C + a]; },
          [&](int r, int bb) { return sdT[r * C + bb] * sb[bb]; },
          [&](int a, int bb, float s) { sX[a * C + bb] = s; });
    __syncthreads();
    // dA = strict_lower(-X Linv^T)
    bgemm(len, len, len, [&](int a, int c) { return sX[a * C + c]; },
          [&](int c, int bb) { return sLi[bb * C + c]; },
          [&](int a, int bb, float s) { sY[a * C + bb] = (bb < a) ? -s : 0.f; });
    __syncthreads();
    // d beta from A, E = dD o D, d gamma row/col sums;  Y <- dKK = dA o beta_r o D
    for (int r = warp; r < len; r += nw) {
        float db = 0.f, rs = 0.f;
        for (int i = lane; i < len; i += 32) {
            float dA = sY[r * C + i];
            float Dri = sD[r * C + i];
            db = fmaf(dA * sKK[r * C + i], Dri, db);
            float E = (dA * sb[r] * sKK[r * C + i] + (i <= r ? sdP[r * C + i] * sQK[r * C + i] : 0.f)) * Dri;
            rs += E;
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
        for (int r = lane; r < len; r += 32) {
            float Dri = sD[r * C + i];
            float E = (sY[r * C + i] * sb[r] * sKK[r * C + i] + (i <= r ? sdP[r * C + i] * sQK[r * C + i] : 0.f)) * Dri;
            cs += E;
        }
        cs = warp_sum(cs);
        if (lane == 0) sdg[i] -= cs;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < len * len; idx += blockDim.x) {
        int r = idx / len, i = idx - r * len;
        sY[r * C + i] = sY[r * C + i] * sb[r] * sD[r * C + i];
    }
    __syncthreads();
    // dK += dKK K + dKK^T K;  then the normalisation chain rule for dq, dk
    for (int r = warp; r < len; r += nw) {
        for (int kk = lane; kk < dk; kk += 32) {
            float a = 0.f;
            for (int i = 0; i < len; ++i)
                a = fmaf(sY[r * C + i] + sY[i * C + r], Kn[i * dk + kk], a);
            dK[r * dk + kk] += a;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float es = 0.f;
        for (int r = 0; r < len; ++r) {
            sdg[r] -= se[r];
            es += se[r];
        }
        sdg[len - 1] += es + expf(gC) * sred[0];
        // d g = reverse cumulative sum of d gamma within the chunk
        float acc = 0.f;
        for (int r = len - 1; r >= 0; --r) {
            acc += sdg[r];
            if (dg) dg[row + r] = acc;
        }
    }
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
        for (int kk = lane; kk < dk; kk += 32) {
            float a = dQ[r * dk + kk], c = dK[r * dk + kk];
            if (g.l2norm) {
                a = rq * (a - Qn[r * dk + kk] * pq);
                c = rk * (c - Kn[r * dk + kk] * pk);
            }
            st_out(dq + (row + r) * dk + kk, a);
            st_out(dkout + (row + r) * dk + kk, c);
        }
        if (lane == 0) st_out(dbeta + row + r, sdb[r]);
    }
}

// ----------------------------------------------------------------------------- host launchers
static size_t smem_prep(const Geo &g) { return sizeof(float) * (g.C * g.dk + 2 * g.C * g.C + 3 * g.C); }
static size_t smem_scan(const Geo &g, int BV) { return sizeof(float) * (g.dk * BV + g.C * BV + g.C); }
static size_t smem_out(const Geo &g) { return sizeof(float) * (g.C * g.C + g.C); }
static size_t smem_bscan(const Geo &g, int BV)
{
    return sizeof(float) * (g.dk * BV + 2 * g.C * BV + g.C * g.C + 2 * g.C);
}
static size_t smem_bchunk(const Geo &g) { return sizeof(float) * (8 * g.C * g.C + 7 * g.C + 1); }

static int slice_width(const Geo &g) { return g.dv < 32 ? g.dv : 32; }

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
    if ((e = set_smem(k_prep<Tin>, smem_prep(g))) != cudaSuccess) return e;
    if (g.NC > 0) k_prep<Tin><<<dim3(g.NC, g.H), 256, smem_prep(g), st>>>(g, q, k, v, beta, gate, w);
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
    const int BV = slice_width(g);
    if ((e = set_smem(k_scan, smem_scan(g, BV))) != cudaSuccess) return e;
    if (g.N > 0)
        k_scan<<<dim3(g.N, g.H, (g.dv + BV - 1) / BV), 256, smem_scan(g, BV), st>>>(g, h0, hT, w, BV);
    return cudaPeekAtLastError();
}

template <class Tin>
cudaError_t fwd(const Geo &g, const Tin *q, const Tin *k, const Tin *v, const Tin *beta,
                const float *gate, const float *h0, Tin *o, float *hT, const Ws &w,
                cudaStream_t st)
{
    cudaError_t e = forward_states(g, q, k, v, beta, gate, h0, hT, w, st);
    if (e != cudaSuccess) return e;
    if ((e = set_smem(k_out<Tin>, smem_out(g))) != cudaSuccess) return e;
    if (g.NC > 0) k_out<Tin><<<dim3(g.NC, g.H), 256, smem_out(g), st>>>(g, o, w);
    return cudaPeekAtLastError();
}

template <class Tin>
cudaError_t bwd(const Geo &g, const Tin *q, const Tin *k, const Tin *v, const Tin *beta,
                const float *gate, const float *h0, const Tin *dO, const float *dhT, Tin *dq,
                Tin *dk, Tin *dv, Tin *dbeta, float *dg, float *dh0, const Ws &w,
                cudaStream_t st)
{
    cudaError_t e = forward_states(g, q, k, v, beta, gate, h0, nullptr, w, st);
    if (e != cudaSuccess) return e;
    const int BV = slice_width(g);
    if ((e = set_smem(k_bscan<Tin>, smem_bscan(g, BV))) != cudaSuccess) return e;
    if (g.N > 0)
        k_bscan<Tin><<<dim3(g.N, g.H, (g.dv + BV - 1) / BV), 256, smem_bscan(g, BV), st>>>(
            g, dO, dhT, dh0, w, BV);
    if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
    if ((e = set_smem(k_bchunk<Tin>, smem_bchunk(g))) != cudaSuccess) return e;
    if (g.NC > 0)
        k_bchunk<Tin><<<dim3(g.NC, g.H), 256, smem_bchunk(g), st>>>(g, q, k, v, beta, dO, dq, dk,
                                                                     dv, dbeta, dg, w);
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
