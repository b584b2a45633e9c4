// Recurrent decode step of the (gated) delta rule: one new token per sequence,
// the state updated in place or into a second buffer.
//
// Per (sequence, head), with the state S stored d_k x d_v (key index outer) and
// the token's normalised q, k:
//     S' = alpha (I - beta k k^T) S + beta k v^T,   o = scale S'^T q
// ("Gated DeltaNet", Table 1, row Gated DeltaNet; alpha = 1 is DeltaNet; with
// Longhorn's step size beta / (1 + beta k^T k) in place of beta, row Longhorn).
// Each column n of S evolves on its own:
//     r_n = sum_i S[i][n] k_i,   u_n = beta (v_n - alpha r_n),
//     S'[i][n] = alpha S[i][n] + k_i u_n,
//     o_n = scale (alpha sum_i S[i][n] q_i + u_n (k . q)),
// so one pass reads the state once, keeps it in registers, and writes it once
// (16-byte accesses, one CTA per (sequence, head), when d_v % 4 == 0 and
// d_k, d_v <= 128; else
// 4-byte accesses, one CTA per 32-column slice):
// the step moves the compulsory 2 d_k d_v fp32 state bytes per head and is
// bound by HBM bandwidth.
#include "common.cuh"
#include "decode.h"

namespace gdn {
namespace dec {

namespace {

constexpr int kCols = 32;            // d_v columns per CTA (one warp's width)
constexpr int kGroups = 8;           // row groups: 256 threads
constexpr int kRows = kMaxD / kGroups;   // rows per thread, 4-byte kernel
constexpr int kGroups4 = 16;             // row groups of the 16-byte kernel: 512 threads

// the step size: beta, or Longhorn's beta / (1 + beta k^T k) ("Gated DeltaNet",
// Table 1, row Longhorn), kk = k^T k of the key the update uses
__device__ __forceinline__ float step_size(const Args &a, float b, float kk)
{
    return a.longhorn ? b / fmaf(b, kk, 1.f) : b;
}

template <class Tin>
__global__ void __launch_bounds__(kCols * kGroups) k_decode(Args a, const Tin *__restrict__ q,
                                                          const Tin *__restrict__ k,
                                                          const Tin *__restrict__ v,
                                                          const Tin *__restrict__ beta,
                                                          Tin *__restrict__ o)
{
    const int nsl = (a.dv + kCols - 1) / kCols;
    const int seq = blockIdx.x / nsl, sl = blockIdx.x - seq * nsl, h = blockIdx.y;
    const int col = threadIdx.x & 31, rg = threadIdx.x >> 5;
    const int n = sl * kCols + col;
    const size_t item = (size_t)seq * a.H + h;
    __shared__ float sk[kMaxD], sq[kMaxD];
    __shared__ float sr[kGroups][kCols], sp[kGroups][kCols];
    __shared__ float su[kCols];
    __shared__ float sscal[3];   // k . q, alpha, k . k

    for (int i = threadIdx.x; i < a.dk; i += blockDim.x) {
        sk[i] = ld_in(k + item * a.dk + i);
        sq[i] = ld_in(q + item * a.dk + i);
    }
    __syncthreads();
    if (rg == 0) {
        float kk = 0.f, qq = 0.f;
        for (int i = col; i < a.dk; i += 32) {
            kk = fmaf(sk[i], sk[i], kk);
            qq = fmaf(sq[i], sq[i], qq);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, o2);
            qq += __shfl_xor_sync(0xffffffffu, qq, o2);
        }
        const float rk = a.l2norm ? rsqrtf(kk + a.eps) : 1.f;
        const float rq = a.l2norm ? rsqrtf(qq + a.eps) : 1.f;
        float kq = 0.f;
        for (int i = col; i < a.dk; i += 32) {
            sk[i] *= rk;
            sq[i] *= rq;
            kq = fmaf(sk[i], sq[i], kq);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o2);
        if (col == 0) {
            sscal[0] = kq;
            sscal[1] = a.gate ? expf(a.gate[item]) : 1.f;
            sscal[2] = kk * rk * rk;
        }
    }
    __syncthreads();
    const float alpha = sscal[1];
    // this thread's rows rg, rg + 8, ... of column n: read once, kept in registers
    float s[kRows];
    float r = 0.f, p = 0.f;
    const float *Sin = a.state_in ? a.state_in + item * a.dk * a.dv : nullptr;
    float *Sout = a.state_out + item * a.dk * a.dv;
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
        const int i = rg + kGroups * j;
        s[j] = (n < a.dv && i < a.dk && Sin) ? Sin[(size_t)i * a.dv + n] : 0.f;
        if (i < a.dk) {
            r = fmaf(s[j], sk[i], r);
            p = fmaf(s[j], sq[i], p);
        }
    }
    sr[rg][col] = r;
    sp[rg][col] = p;
    __syncthreads();
    if (rg == 0) {
        float rt = 0.f, pt = 0.f;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
            rt += sr[g][col];
            pt += sp[g][col];
        }
        float u = 0.f;
        if (n < a.dv) {
            const float b = step_size(a, ld_in(beta + item), sscal[2]);
            u = b * (ld_in(v + item * a.dv + n) - alpha * rt);
            st_out(o + item * a.dv + n, a.scale * fmaf(alpha, pt, u * sscal[0]));
        }
        su[col] = u;
    }
    __syncthreads();
    if (n < a.dv) {
        const float u = su[col];
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
            const int i = rg + kGroups * j;
            if (i < a.dk) Sout[(size_t)i * a.dv + n] = fmaf(alpha, s[j], sk[i] * u);
        }
    }
}

// The same step with 16-byte state accesses: one CTA per (sequence, head), lane
// l of every warp owns columns 4l .. 4l + 3, so a warp moves one 512-byte state
// row per instruction (needs d_v % 4 == 0 and 16-byte aligned states).  NG warps
// take interleaved rows (128 / NG rows per thread): 16 warps keep two CTAs and
// 32 warps per SM, with all their state loads in flight.
template <class Tin, int NG>
__global__ void __launch_bounds__(32 * NG) k_decode4(Args a, const Tin *__restrict__ q,
                                                 const Tin *__restrict__ k,
                                                 const Tin *__restrict__ v,
                                                 const Tin *__restrict__ beta,
                                                 Tin *__restrict__ o)
{
    const int seq = blockIdx.x, h = blockIdx.y;
    const int lane = threadIdx.x & 31, rg = threadIdx.x >> 5;
    const int n4 = 4 * lane;
    const bool live = n4 < a.dv;
    const size_t item = (size_t)seq * a.H + h;
    __shared__ float sk[kMaxD], sq[kMaxD];
    __shared__ float4 sr[NG][32], sp[NG][32];
    __shared__ float4 su[32];
    __shared__ float sscal[3];

    // the state's loads go out first: they do not depend on the token, and their
    // latency then covers the normalisation of q and k below
    const float4 *Sin = a.state_in ? reinterpret_cast<const float4 *>(a.state_in + item * a.dk * a.dv) : nullptr;
    float4 *Sout = reinterpret_cast<float4 *>(a.state_out + item * a.dk * a.dv);
    const int dv4 = a.dv >> 2;
    constexpr int NR = 128 / NG;   // rows per thread (d_k <= 128)
    float4 s[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int i = rg + NG * j;
        s[j] = (live && i < a.dk && Sin) ? Sin[(size_t)i * dv4 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // so do this thread's v and beta (thread c < d_v owns column c below)
    const float vc = (int)threadIdx.x < a.dv ? ld_in(v + item * a.dv + threadIdx.x) : 0.f;
    const float braw = ld_in(beta + item);

    for (int i = threadIdx.x; i < a.dk; i += blockDim.x) {
        sk[i] = ld_in(k + item * a.dk + i);
        sq[i] = ld_in(q + item * a.dk + i);
    }
    __syncthreads();
    if (rg == 0) {
        float kk = 0.f, qq = 0.f;
        for (int i = lane; i < a.dk; i += 32) {
            kk = fmaf(sk[i], sk[i], kk);
            qq = fmaf(sq[i], sq[i], qq);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, o2);
            qq += __shfl_xor_sync(0xffffffffu, qq, o2);
        }
        const float rk = a.l2norm ? rsqrtf(kk + a.eps) : 1.f;
        const float rq = a.l2norm ? rsqrtf(qq + a.eps) : 1.f;
        float kq = 0.f;
        for (int i = lane; i < a.dk; i += 32) {
            sk[i] *= rk;
            sq[i] *= rq;
            kq = fmaf(sk[i], sq[i], kq);
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o2);
        if (lane == 0) {
            sscal[0] = kq;
            sscal[1] = a.gate ? expf(a.gate[item]) : 1.f;
            sscal[2] = kk * rk * rk;
        }
    }
    __syncthreads();
    const float alpha = sscal[1];
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int i = rg + NG * j;
        if (i < a.dk) {
            const float ki = sk[i], qi = sq[i];
            r.x = fmaf(s[j].x, ki, r.x); r.y = fmaf(s[j].y, ki, r.y);
            r.z = fmaf(s[j].z, ki, r.z); r.w = fmaf(s[j].w, ki, r.w);
            p.x = fmaf(s[j].x, qi, p.x); p.y = fmaf(s[j].y, qi, p.y);
            p.z = fmaf(s[j].z, qi, p.z); p.w = fmaf(s[j].w, qi, p.w);
        }
    }
    sr[rg][lane] = r;
    sp[rg][lane] = p;
    __syncthreads();
    if (threadIdx.x < a.dv) {
        // column c = threadIdx.x: component c & 3 of lane c >> 2
        const int c = threadIdx.x, L = c >> 2, e = c & 3;
        float rt = 0.f, pt = 0.f;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            rt += reinterpret_cast<const float *>(&sr[g][L])[e];
            pt += reinterpret_cast<const float *>(&sp[g][L])[e];
        }
        const float b = step_size(a, braw, sscal[2]);
        const float u = b * (vc - alpha * rt);
        st_out(o + item * a.dv + c, a.scale * fmaf(alpha, pt, u * sscal[0]));
        reinterpret_cast<float *>(&su[L])[e] = u;
    }
    __syncthreads();
    if (live) {
        const float4 u = su[lane];
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int i = rg + NG * j;
            if (i < a.dk) {
                const float ki = sk[i];
                Sout[(size_t)i * dv4 + lane] = make_float4(fmaf(alpha, s[j].x, ki * u.x), fmaf(alpha, s[j].y, ki * u.y),
                                                           fmaf(alpha, s[j].z, ki * u.z), fmaf(alpha, s[j].w, ki * u.w));
            }
        }
    }
}

}  // namespace

template <class Tin>
cudaError_t step(const Args &a, const Tin *q, const Tin *k, const Tin *v, const Tin *beta, Tin *o,
                 cudaStream_t st)
{
    if (a.N == 0) return cudaSuccess;
    const bool aligned = ((uintptr_t)a.state_out & 15u) == 0 && ((uintptr_t)a.state_in & 15u) == 0;
    if (a.dv % 4 == 0 && a.dv <= 128 && a.dk <= 128 && aligned) {
        if (a.N > 0x7fffffff || a.H > 65535) return cudaErrorInvalidValue;
        k_decode4<Tin, kGroups4><<<dim3((unsigned)a.N, a.H), 32 * kGroups4, 0, st>>>(a, q, k, v, beta, o);
        return cudaPeekAtLastError();
    }
    const int nsl = (a.dv + kCols - 1) / kCols;
    const long long blocks = (long long)a.N * nsl;
    if (blocks > 0x7fffffffLL || a.H > 65535) return cudaErrorInvalidValue;
    k_decode<Tin><<<dim3((unsigned)blocks, a.H), kCols * kGroups, 0, st>>>(a, q, k, v, beta, o);
    return cudaPeekAtLastError();
}

template cudaError_t step<float>(const Args &, const float *, const float *, const float *,
                                 const float *, float *, cudaStream_t);
template cudaError_t step<__nv_bfloat16>(const Args &, const __nv_bfloat16 *, const __nv_bfloat16 *,
                                         const __nv_bfloat16 *, const __nv_bfloat16 *, __nv_bfloat16 *,
                                         cudaStream_t);

}  // namespace dec
}  // namespace gdn
