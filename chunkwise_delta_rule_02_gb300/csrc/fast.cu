// Fused tcgen05 / TMA forward of the (gated) delta rule for bf16 inputs with
// d_k = d_v = 128 and chunk C = 64, on one GB300 SM per (sequence, head).
//
// Chunk form ("Parallelizing Linear Transformers with the Delta Rule over
// Sequence Length": WY representation via the UT transform, chunkwise-parallel
// form; "Gated DeltaNet": gates folded in as within-chunk cumulative log-decays
// gamma, D_ri = exp(gamma_r - gamma_i)).  With raw q, k rows and their
// normalisation factors m_r, n_r (q_hat = m q, k_hat = n k):
//   A   = strict_lower(diag(beta) (K_hat K_hat^T o D)),  T = (I + A)^-1 diag(beta)
//   W   = T diag(exp(gamma) n) K,   U = T V,   Unew = U - W S
//   S'  = exp(gamma_C) S + K^T diag(exp(gamma_C - gamma) n) Unew
//   O   = diag(exp(gamma) m) Q S + P Unew,  P_ri = m_r n_i (q_r . k_i) D_ri (i <= r)
//
// Everything is computed transposed so every tcgen05.mma has M = 128 (the state
// S^T lives in TMEM with lane = value column, column = key row):
//   G   : TMEM[GW]  = [K; Q] K^T              (SS, 128 x 64 x 128)
//   W^T : TMEM[GW]  = K^T T'^T                 (SS, A MN-major; T' = T diag(exp(gamma) n))
//   U^T : TMEM[X]   = V^T T^T                  (SS, A MN-major)
//   1   : TMEM[X]  += S^T (-W^T)               (TS tf32: A = the fp32 state in TMEM)
//   3   : TMEM[O]   = S_snap^T Qt^T            (TS bf16, Qt = diag(exp(gamma) m) Q)
//   4   : TMEM[O]  += Unew^T P^T               (TS bf16)
//   2   : TMEM[S]  += U2^T K                   (TS bf16, B MN-major; U2 = diag(f) Unew)
// with the state's own decay exp(gamma_C) applied in place in TMEM between 1
// and 2 by the warpgroup that also takes the bf16 snapshot for 3.
//
// Warp roles (512 threads): warp 0 issues TMA loads, warp 1 owns TMEM and one
// of its lanes issues every MMA (an event-driven scheduler that keeps the
// sequential chain 1 -> 2 -> 1 ahead of everything else); warpgroup 1 turns the
// Unew accumulator into the bf16 operands U1 / U2; warpgroup 2 does the chunk
// preparation (gates, norms, Gram masks, triangular solve, W); warpgroup 3 owns
// the state (initial state, decay + snapshot, final state) and the output.
// Every wait is bounded; a wait that runs out sets the status word and the
// block winds down (waiting, bounded, for its own copies and MMAs) before
// releasing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "fast.h"
#include "sm100.cuh"

namespace gdn {
namespace fast {
using namespace sm100;

namespace {

constexpr int C = 64;
constexpr int D = 128;
constexpr int NTHREADS = 512;
constexpr long long WAIT_BUDGET = 4000000000LL;   // clock cycles (about 2 s)

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_KQ = 0;          // 2 stages x 32 KB: per 64-column half: K rows | Q rows
constexpr uint32_t OFF_V = 65536;       // 2 stages x 16 KB: V, two 64-column halves
constexpr uint32_t OFF_WF = 98304;      // 32 KB  -W as tf32 operand [token][dk], 4 atoms of 32 dk
constexpr uint32_t OFF_TB = 131072;     // 8 KB   T  bf16 [r][i]
constexpr uint32_t OFF_TPB = 139264;    // 8 KB   T' bf16 [r][i]
constexpr uint32_t OFF_PB = 147456;     // 2 x 8 KB P bf16 [r][i]
constexpr uint32_t OFF_OST = 163840;    // 16 KB  output staging [64][128] bf16
constexpr uint32_t AST = 65;            // row stride (floats) of the solve matrices
constexpr uint32_t OFF_AF = 180224;     // A fp32 [64][65]
constexpr uint32_t OFF_XF = OFF_AF + 64 * AST * 4;  // X = (I + A)^-1 fp32 [64][65]
constexpr uint32_t OFF_Y = OFF_XF + 64 * AST * 4;   // 3 blocks 16 x 17 fp32
constexpr uint32_t OFF_VEC = OFF_Y + 3 * 16 * 17 * 4;  // beta, gamma, nk, nq (64 floats each)
constexpr uint32_t OFF_RING = OFF_VEC + 4 * 64 * 4;    // 2 ring slots
constexpr uint32_t OFF_BAR = OFF_RING + 2 * 320;
constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
constexpr uint32_t SMEM_USED = OFF_MISC + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for the manual 1024-byte alignment

struct Ring {           // per-chunk scalars handed from the prep warpgroup to the others
    float f[64];        // exp(gamma_C - gamma_r) n_r (0 past the end of the chunk)
    float gammaC;       // exp(gamma_C)
    int len;            // rows of this chunk
    long long row0;     // first token row (flattened [B*H*T] index)
    int pad[12];
};
static_assert(sizeof(Ring) <= 320, "ring slot");

// TMEM column map (512 columns allocated)
constexpr uint32_t TM_S = 0;       // 128: S^T fp32 (lane = dv, column = dk)
constexpr uint32_t TM_SNAP = 128;  // 64 : S^T bf16 pairs
constexpr uint32_t TM_X = 192;     // 64 : Unew^T accumulator (lane = dv, column = token)
constexpr uint32_t TM_U1 = 256;    // 2 x 32: Unew^T bf16 pairs
constexpr uint32_t TM_U2 = 320;    // 2 x 32: (f o Unew)^T bf16 pairs
constexpr uint32_t TM_GW = 384;    // 64 : [K;Q]K^T, then W^T
constexpr uint32_t TM_O = 448;     // 64 : O^T

// mbarrier slots
enum {
    B_FULL = 0, B_EMPTY = 2, B_G = 4, B_W = 5, B_X = 6, B_O = 7, B_F = 9, B_TREADY = 10,
    B_WREADY = 11, B_GWFREE = 12, B_XFREE = 13, B_U2READY = 14, B_SNAP = 15, B_OFREE = 16,
    B_RINGFREE = 17, B_RINGREADY = 19, B_SINIT = 21, B_ABORTED = 22, NBAR = 23
};

constexpr uint32_t ID_F16_N64 = idesc(1, 128, 64, false, false);
constexpr uint32_t ID_F16_N64_AMN = idesc(1, 128, 64, true, false);
constexpr uint32_t ID_F16_N128_BMN = idesc(1, 128, 128, false, true);
constexpr uint32_t ID_TF32_N64 = idesc(2, 128, 64, false, false);

struct Params {
    const __nv_bfloat16 *beta;
    const float *gate;
    const float *h0;
    __nv_bfloat16 *o;
    float *hT;
    uint32_t *status;
    const int32_t *cu;       // packed offsets or null
    const int32_t *order;    // packed: sequences longest first (or null)
    int H, T, N;
    float scale, eps;
    int l2norm;
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t scale_pair(uint32_t w, float s)
{
    return pack_bf16(bf_lo(w) * s, bf_hi(w) * s);
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 1)
k_fast_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    uint64_t *bar = (uint64_t *)(sm + OFF_BAR);
    volatile int *abort_flag = (volatile int *)(sm + OFF_MISC);
    uint32_t *tmem_slot = (uint32_t *)(sm + OFF_MISC + 8);
    float *s_beta = (float *)(sm + OFF_VEC);
    float *s_gam = s_beta + 64;
    float *s_nk = s_gam + 64;
    float *s_nq = s_nk + 64;
    Ring *ring = (Ring *)(sm + OFF_RING);
    float *Af = (float *)(sm + OFF_AF);
    float *Xf = (float *)(sm + OFF_XF);
    float *Yf = (float *)(sm + OFF_Y);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- work item: (sequence, head); packed input runs the longest sequences first
    const int h = blockIdx.x % p.H;
    const int rank = blockIdx.x / p.H;
    int seq, t0, L;
    long long rowbase;
    if (p.cu) {
        seq = p.order ? p.order[rank] : rank;
        t0 = p.cu[seq];
        int t1 = p.cu[seq + 1];
        if (t0 < 0 || t1 < t0 || t1 > p.T) t0 = t1 = 0;   // malformed offsets: empty (flagged elsewhere)
        L = t1 - t0;
        rowbase = (long long)h * p.T + t0;
    } else {
        seq = rank;
        t0 = 0;
        L = p.T;
        rowbase = ((long long)seq * p.H + h) * p.T;
    }
    const int nch = (L + C - 1) / C;
    const size_t sidx = ((size_t)seq * p.H + h) * D * D;

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == B_TREADY || i == B_WREADY || i == B_GWFREE || i == B_XFREE || i == B_U2READY ||
                i == B_SNAP || i == B_OFREE || i == B_RINGREADY || i == B_RINGREADY + 1 || i == B_SINIT)
                cnt = 4;
            if (i == B_RINGFREE || i == B_RINGFREE + 1) cnt = 8;
            mbar_init(&bar[i], cnt);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&]() {
        if (!*abort_flag) {
            *abort_flag = 1;
            raise_status(p.status, kStatusTimeout);
        }
    };
    auto wait = [&](int b, uint32_t k) -> bool {
        if (mbar_wait(&bar[b], k & 1u, WAIT_BUDGET, abort_flag)) return true;
        fail();
        return false;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int n = 0; n < nch && !*abort_flag; ++n) {
                const int s = n & 1;
                if (n >= 2 && !wait(B_EMPTY + s, (uint32_t)((n >> 1) - 1))) break;
                const int row = (int)(rowbase + (long long)n * C);
                uint8_t *kq = sm + OFF_KQ + s * 32768;
                uint8_t *vv = sm + OFF_V + s * 16384;
                mbar_expect_tx(&bar[B_FULL + s], 49152);
                tma_load_2d(kq, &tm_k, &bar[B_FULL + s], 0, row);
                tma_load_2d(kq + 16384, &tm_k, &bar[B_FULL + s], 64, row);
                tma_load_2d(kq + 8192, &tm_q, &bar[B_FULL + s], 0, row);
                tma_load_2d(kq + 24576, &tm_q, &bar[B_FULL + s], 64, row);
                tma_load_2d(vv, &tm_v, &bar[B_FULL + s], 0, row);
                tma_load_2d(vv + 8192, &tm_v, &bar[B_FULL + s], 64, row);
                issued = n + 1;
            }
            if (*abort_flag) {
                // let copies still in flight land before the block's shared memory goes away
                for (int n = (issued > 2 ? issued - 2 : 0); n < issued; ++n)
                    mbar_wait(&bar[B_FULL + (n & 1)], (uint32_t)(n >> 1) & 1u, WAIT_BUDGET, nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && nch > 0) {
            int nG = 0, nW = 0, n1 = 0, n2 = 0, n3 = 0, n4 = 0;
            long long t_last = clock64();
            auto poll = [&](int b, uint32_t k) { return mbar_try_wait(&bar[b], k & 1u); };
            while (n4 < nch) {
                if (*abort_flag) break;
                bool did = false;
                if (n1 < nch && n1 == n2 && nW > n1 && n3 >= n1 && n4 + 1 >= n1 &&
                    (n1 > 0 || poll(B_SINIT, 0)) && poll(B_WREADY, (uint32_t)n1)) {
                    // 1: X += S^T (-W^T)   tf32, A = fp32 state in TMEM
                    tc_fence_after();
                    for (int j = 0; j < 16; ++j) {
                        uint64_t bd = sdesc(sb + OFF_WF + (j >> 2) * 8192 + (j & 3) * 32, 16, 1024);
                        mma_tf32_ts(tmem + TM_X, tmem + TM_S + 8 * j, bd, ID_TF32_N64, 1);
                    }
                    mma_commit(&bar[B_X]);
                    ++n1;
                    did = true;
                } else if (n2 < n1 && n3 > n2 && poll(B_U2READY, (uint32_t)n2) &&
                           poll(B_SNAP, (uint32_t)n2)) {
                    // 2: S^T += U2^T K      B = K tile, MN-major (dk contiguous)
                    tc_fence_after();
                    const uint32_t kq = sb + OFF_KQ + (n2 & 1) * 32768;
                    for (int j = 0; j < 4; ++j) {
                        uint64_t bd = sdesc(kq + j * 2048, 16384, 1024);
                        mma_bf16_ts(tmem + TM_S, tmem + TM_U2 + (n2 & 1) * 32 + 8 * j, bd,
                                    ID_F16_N128_BMN, 1);
                    }
                    mma_commit(&bar[B_EMPTY + (n2 & 1)]);
                    ++n2;
                    if (n2 == nch) mma_commit(&bar[B_F]);
                    did = true;
                } else if (n3 < n1 && n3 == n4 && poll(B_SNAP, (uint32_t)n3) &&
                           (n3 == 0 || poll(B_OFREE, (uint32_t)(n3 - 1)))) {
                    // 3: O^T = S_snap^T Qt^T
                    tc_fence_after();
                    const uint32_t kq = sb + OFF_KQ + (n3 & 1) * 32768;
                    for (int j = 0; j < 8; ++j) {
                        uint64_t bd = sdesc(kq + (j >> 2) * 16384 + 8192 + (j & 3) * 32, 16, 1024);
                        mma_bf16_ts(tmem + TM_O, tmem + TM_SNAP + 8 * j, bd, ID_F16_N64, j > 0);
                    }
                    ++n3;
                    did = true;
                } else if (n4 < n3 && n4 < n2) {
                    // 4: O^T += Unew^T P^T
                    for (int j = 0; j < 4; ++j) {
                        uint64_t bd = sdesc(sb + OFF_PB + (n4 & 1) * 8192 + j * 32, 16, 1024);
                        mma_bf16_ts(tmem + TM_O, tmem + TM_U1 + (n4 & 1) * 32 + 8 * j, bd,
                                    ID_F16_N64, 1);
                    }
                    mma_commit(&bar[B_O + (n4 & 1)]);
                    ++n4;
                    did = true;
                } else if (nG < nch && nG <= n1 + 1 && poll(B_FULL + (nG & 1), (uint32_t)(nG >> 1)) &&
                           (nG == 0 || poll(B_GWFREE, (uint32_t)(nG - 1)))) {
                    // G: [K;Q] K^T
                    tc_fence_after();
                    const uint32_t kq = sb + OFF_KQ + (nG & 1) * 32768;
                    for (int j = 0; j < 8; ++j) {
                        uint32_t a = kq + (j >> 2) * 16384 + (j & 3) * 32;
                        mma_bf16_ss(tmem + TM_GW, sdesc(a, 16, 1024), sdesc(a, 16, 1024), ID_F16_N64,
                                    j > 0);
                    }
                    mma_commit(&bar[B_G]);
                    ++nG;
                    did = true;
                } else if (nW < nG && (nW == 0 || poll(B_XFREE, (uint32_t)(nW - 1))) &&
                           poll(B_TREADY, (uint32_t)nW)) {
                    // W^T = K^T T'^T  and  U^T = V^T T^T
                    tc_fence_after();
                    const uint32_t kq = sb + OFF_KQ + (nW & 1) * 32768;
                    const uint32_t vv = sb + OFF_V + (nW & 1) * 16384;
                    for (int j = 0; j < 4; ++j) {
                        mma_bf16_ss(tmem + TM_GW, sdesc(kq + j * 2048, 16384, 1024),
                                    sdesc(sb + OFF_TPB + j * 32, 16, 1024), ID_F16_N64_AMN, j > 0);
                    }
                    for (int j = 0; j < 4; ++j) {
                        mma_bf16_ss(tmem + TM_X, sdesc(vv + j * 2048, 8192, 1024),
                                    sdesc(sb + OFF_TB + j * 32, 16, 1024), ID_F16_N64_AMN, j > 0);
                    }
                    mma_commit(&bar[B_W]);
                    ++nW;
                    did = true;
                }
                if (did) {
                    t_last = clock64();
                } else if (clock64() - t_last > WAIT_BUDGET) {
                    fail();
                    break;
                }
            }
            // every MMA issued must be complete before TMEM is released
            mma_commit(&bar[B_ABORTED]);
            mbar_wait(&bar[B_ABORTED], 0, WAIT_BUDGET, nullptr);
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ WG1: Unew -> U1, U2
        const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
        for (int n = 0; n < nch; ++n) {
            if (!wait(B_X, (uint32_t)n)) break;
            tc_fence_after();
            uint32_t x[64];
            tmem_ld32(tmem + lrow + TM_X, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
            tmem_ld32(tmem + lrow + TM_X + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_XFREE]);
            if (!wait(B_RINGREADY + (n & 1), (uint32_t)(n >> 1))) break;
            const Ring &rg = ring[n & 1];
            uint32_t u1[32], u2[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                float a = __uint_as_float(x[2 * c]), b = __uint_as_float(x[2 * c + 1]);
                u1[c] = pack_bf16(a, b);
                u2[c] = pack_bf16(a * rg.f[2 * c], b * rg.f[2 * c + 1]);
            }
            tmem_st32(tmem + lrow + TM_U1 + (n & 1) * 32, u1);
            tmem_st32(tmem + lrow + TM_U2 + (n & 1) * 32, u2);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar[B_U2READY]);
                mbar_arrive(&bar[B_RINGFREE + (n & 1)]);
            }
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ WG2: chunk preparation
        const int t = tid - 256;          // 0..127
        const int q4 = warp & 3;          // TMEM lane quarter
        const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
        for (int n = 0; n < nch; ++n) {
            const int s = n & 1;
            const int len = min(C, L - n * C);
            const long long row0 = rowbase + (long long)n * C;
            uint8_t *kq = sm + OFF_KQ + s * 32768;
            if (n >= 2) wait(B_RINGFREE + s, (uint32_t)((n >> 1) - 1));
            wait(B_FULL + s, (uint32_t)(n >> 1));
            // gates and beta; inclusive scan of g within the chunk (one warp, two rows per lane)
            if (warp == 8) {
                float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
                if (lane < len) {
                    b0 = __bfloat162float(p.beta[row0 + lane]);
                    g0 = p.gate ? p.gate[row0 + lane] : 0.f;
                }
                if (lane + 32 < len) {
                    b1 = __bfloat162float(p.beta[row0 + lane + 32]);
                    g1 = p.gate ? p.gate[row0 + lane + 32] : 0.f;
                }
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    float a0 = __shfl_up_sync(0xffffffffu, g0, o);
                    float a1 = __shfl_up_sync(0xffffffffu, g1, o);
                    if (lane >= o) { g0 += a0; g1 += a1; }
                }
                g1 += __shfl_sync(0xffffffffu, g0, 31);
                s_beta[lane] = b0;
                s_beta[lane + 32] = b1;
                s_gam[lane] = g0;
                s_gam[lane + 32] = g1;
            }
            // L2 norms of the raw k and q rows (two threads per row, one 64-column half each)
            {
                const int r = t >> 1, hh = t & 1;
                float sk = 0.f, sq = 0.f;
                const uint8_t *kr = kq + hh * 16384 + r * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int jj = (j + r) & 7;
                    uint4 a = *(const uint4 *)(kr + jj * 16);
                    uint4 b = *(const uint4 *)(kr + 8192 + jj * 16);
                    uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float x0 = bf_lo(wa[e]), x1 = bf_hi(wa[e]);
                        float y0 = bf_lo(wb[e]), y1 = bf_hi(wb[e]);
                        sk = fmaf(x0, x0, fmaf(x1, x1, sk));
                        sq = fmaf(y0, y0, fmaf(y1, y1, sq));
                    }
                }
                sk += __shfl_xor_sync(0xffffffffu, sk, 1);
                sq += __shfl_xor_sync(0xffffffffu, sq, 1);
                if (hh == 0) {
                    const bool ok = r < len;
                    s_nk[r] = ok ? (p.l2norm ? rsqrtf(sk + p.eps) : 1.f) : 0.f;
                    s_nq[r] = ok ? (p.l2norm ? rsqrtf(sq + p.eps) : 1.f) : 0.f;
                }
            }
            named_bar(2, 128);
            // per-chunk scalars for the other warpgroups
            const float gC = s_gam[len - 1];
            if (t < 64) {
                ring[s].f[t] = (t < len) ? __expf(gC - s_gam[t]) * s_nk[t] : 0.f;
                if (t == 0) {
                    ring[s].gammaC = __expf(gC);
                    ring[s].len = len;
                    ring[s].row0 = row0;
                }
            }
            named_bar(2, 128);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_RINGREADY + s]);
            // Gram / QK^T from TMEM -> A (fp32) and P (bf16)
            wait(B_G, (uint32_t)n);
            tc_fence_after();
            if (q4 >= 2 && n >= 2) wait(B_O + s, (uint32_t)((n >> 1) - 1));
            {
                uint32_t v[64];
                tmem_ld32(tmem + lrow + TM_GW, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(tmem + lrow + TM_GW + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tmem_ld_wait();
                if (q4 < 2) {
                    const int r = q4 * 32 + lane;
                    const float br = s_beta[r] * s_nk[r], gr = s_gam[r];
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        float a = 0.f;
                        if (i < r) a = br * s_nk[i] * __uint_as_float(v[i]) * __expf(gr - s_gam[i]);
                        Af[r * AST + i] = a;
                    }
                } else {
                    const int r = (q4 - 2) * 32 + lane;
                    const float mr = s_nq[r], gr = s_gam[r];
                    uint8_t *prow = sm + OFF_PB + s * 8192;
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i0 = c8 * 8 + 2 * e, i1 = i0 + 1;
                            float a0 = (i0 <= r) ? mr * s_nk[i0] * __uint_as_float(v[i0]) * __expf(gr - s_gam[i0]) : 0.f;
                            float a1 = (i1 <= r) ? mr * s_nk[i1] * __uint_as_float(v[i1]) * __expf(gr - s_gam[i1]) : 0.f;
                            w[e] = pack_bf16(a0, a1);
                        }
                        *(uint4 *)(prow + sw128(r, c8 * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            // Qt = diag(exp(gamma) m) Q, in place in the stage buffer (MMA G has read Q)
            {
                const int r = t >> 1, hh = t & 1;
                const float f = (r < len) ? __expf(s_gam[r]) * s_nq[r] : 0.f;
                uint8_t *qr = kq + hh * 16384 + 8192 + r * 128;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint4 a = *(uint4 *)(qr + j * 16);
                    a.x = scale_pair(a.x, f); a.y = scale_pair(a.y, f);
                    a.z = scale_pair(a.z, f); a.w = scale_pair(a.w, f);
                    *(uint4 *)(qr + j * 16) = a;
                }
            }
            tc_fence_before();
            named_bar(2, 128);
            // X = (I + A)^-1 by 16 x 16 blocks: diagonal blocks by substitution ...
            if (t < 64) {
                const int bb = t >> 4, c = t & 15, base = 16 * bb;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float acc = (i == c) ? 1.f : 0.f;
#pragma unroll
                    for (int l = 0; l < i; ++l) acc = fmaf(-Af[(base + i) * AST + base + l], x[l], acc);
                    x[i] = (i < c) ? 0.f : acc;
                    Xf[(base + i) * AST + base + c] = x[i];
                }
            }
            named_bar(2, 128);
            // ... then block sub-diagonals: X_ij = -X_ii sum_{m=j}^{i-1} A_im X_mj
            for (int lvl = 1; lvl <= 3; ++lvl) {
                const int nblk = 4 - lvl;
                for (int idx = t; idx < nblk * 256; idx += 128) {
                    const int j = idx >> 8, e = idx & 255, rr = e >> 4, cc = e & 15, i = j + lvl;
                    float acc = 0.f;
                    for (int m = j; m < i; ++m) {
                        const float *arow = Af + (16 * i + rr) * AST + 16 * m;
                        const float *xcol = Xf + (16 * m) * AST + 16 * j + cc;
#pragma unroll
                        for (int k = 0; k < 16; ++k) acc = fmaf(arow[k], xcol[k * AST], acc);
                    }
                    Yf[j * 272 + rr * 17 + cc] = acc;
                }
                named_bar(2, 128);
                for (int idx = t; idx < nblk * 256; idx += 128) {
                    const int j = idx >> 8, e = idx & 255, rr = e >> 4, cc = e & 15, i = j + lvl;
                    const float *xrow = Xf + (16 * i + rr) * AST + 16 * i;
                    float acc = 0.f;
#pragma unroll
                    for (int k = 0; k < 16; ++k) acc = fmaf(xrow[k], Yf[j * 272 + k * 17 + cc], acc);
                    Xf[(16 * i + rr) * AST + 16 * j + cc] = -acc;
                }
                named_bar(2, 128);
            }
            // T = X diag(beta) and T' = T diag(exp(gamma) n) as bf16 operands [r][i]
            {
                const int r = t >> 1, hh = t & 1;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint32_t wt[4], wp[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = hh * 32 + c8 * 8 + 2 * e, i1 = i0 + 1;
                        float x0 = (i0 <= r) ? Xf[r * AST + i0] * s_beta[i0] : 0.f;
                        float x1 = (i1 <= r) ? Xf[r * AST + i1] * s_beta[i1] : 0.f;
                        wt[e] = pack_bf16(x0, x1);
                        wp[e] = pack_bf16(x0 * __expf(s_gam[i0]) * s_nk[i0], x1 * __expf(s_gam[i1]) * s_nk[i1]);
                    }
                    const uint32_t off = sw128(r, (hh * 4 + c8) * 16);
                    *(uint4 *)(sm + OFF_TB + off) = make_uint4(wt[0], wt[1], wt[2], wt[3]);
                    *(uint4 *)(sm + OFF_TPB + off) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_TREADY]);
            // W^T from TMEM -> -W as the tf32 operand of MMA 1
            wait(B_W, (uint32_t)n);
            tc_fence_after();
            {
                uint32_t v[64];
                tmem_ld32(tmem + lrow + TM_GW, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(tmem + lrow + TM_GW + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[B_GWFREE]);
                if (n >= 1) wait(B_X, (uint32_t)(n - 1));
                const int dk = q4 * 32 + lane;
                uint8_t *wf = sm + OFF_WF + (dk >> 5) * 8192;
#pragma unroll
                for (int r = 0; r < 64; ++r)
                    *(float *)(wf + sw128(r, (dk & 31) * 4)) = -__uint_as_float(v[r]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_WREADY]);
            if (bar_any(2, 128, *abort_flag != 0)) break;
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ WG3: state and output
        const int t = tid - 384;
        const int dv = (warp & 3) * 32 + lane;
        const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
        // initial state: S^T[dv][dk] = h0[dk][dv]
        for (int k0 = 0; k0 < D; k0 += 32) {
            uint32_t r[32];
#pragma unroll
            for (int k = 0; k < 32; ++k)
                r[k] = __float_as_uint(p.h0 ? p.h0[sidx + (size_t)(k0 + k) * D + dv] : 0.f);
            tmem_st32(tmem + lrow + TM_S + k0, r);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[B_SINIT]);
        bool ok = true;
        for (int n = 0; n < nch; ++n) {
            const int s = n & 1;
            // decay + snapshot: S_snap = bf16(S); S <- exp(gamma_C) S
            wait(B_X, (uint32_t)n);
            tc_fence_after();
            wait(B_RINGREADY + s, (uint32_t)(n >> 1));
            const float GC = ring[s].gammaC;
            const int len = ring[s].len;
            const long long row0 = ring[s].row0;
            for (int k0 = 0; k0 < D; k0 += 32) {
                uint32_t r[32], hbuf[16];
                tmem_ld32(tmem + lrow + TM_S + k0, r);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    hbuf[c] = pack_bf16(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]));
#pragma unroll
                for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * GC);
                tmem_st16(tmem + lrow + TM_SNAP + k0 / 2, hbuf);
                tmem_st32(tmem + lrow + TM_S + k0, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_SNAP]);
            // output of chunk n
            wait(B_O + s, (uint32_t)(n >> 1));
            tc_fence_after();
            uint32_t ov[64];
            tmem_ld32(tmem + lrow + TM_O, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
            tmem_ld32(tmem + lrow + TM_O + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_OFREE]);
            __nv_bfloat16 *ost = (__nv_bfloat16 *)(sm + OFF_OST);
#pragma unroll
            for (int r = 0; r < 64; ++r) ost[r * D + dv] = __float2bfloat16_rn(p.scale * __uint_as_float(ov[r]));
            named_bar(3, 128);
            for (int c = t; c < 64 * 16; c += 128) {
                const int r = c >> 4, c16 = c & 15;
                if (r < len)
                    *(uint4 *)((uint8_t *)(p.o + (row0 + r) * D) + c16 * 16) =
                        *(const uint4 *)(sm + OFF_OST + r * 256 + c16 * 16);
            }
            named_bar(3, 128);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_RINGFREE + s]);
            if (bar_any(3, 128, *abort_flag != 0)) { ok = false; break; }
        }
        // final state
        if (ok && p.hT) {
            if (nch == 0 || wait(B_F, 0)) {
                tc_fence_after();
                for (int k0 = 0; k0 < D; k0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lrow + TM_S + k0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) p.hT[sidx + (size_t)(k0 + k) * D + dv] = __uint_as_float(r[k]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Packed input: sequences ordered by length, longest first (ties by index).
__global__ void k_order(const int32_t *cu, int N, int32_t *order)
{
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= N) return;
    const int Ls = cu[s + 1] - cu[s];
    int rank = 0;
    for (int o = 0; o < N; ++o) {
        const int Lo = cu[o + 1] - cu[o];
        rank += (Lo > Ls) || (Lo == Ls && o < s);
    }
    order[rank] = s;
}

// ----------------------------------------------------------------------------- host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    return fn;
}

bool make_map(CUtensorMap *m, const void *base, long long rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t gstr[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), gdim, gstr, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool supports(const Geo &g, int dtype)
{
    return dtype == DN_BF16 && g.dk == D && g.dv == D && g.C == C &&
           (long long)g.B * g.H * (long long)g.T < (1LL << 31) && encode_fn() != nullptr;
}

size_t workspace_bytes(const Geo &g) { return g.varlen ? sizeof(int32_t) * (size_t)(g.N + 1) : 0; }

cudaError_t fwd(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                const __nv_bfloat16 *v, const __nv_bfloat16 *beta, const float *gate,
                const float *h0, __nv_bfloat16 *o, float *hT, void *ws, uint32_t *status,
                cudaStream_t st)
{
    const long long rows = (long long)g.B * g.H * g.T;
    const int items = g.N * g.H;
    if (items == 0) return cudaSuccess;
    Params p;
    p.beta = beta; p.gate = gate; p.h0 = h0; p.o = o; p.hT = hT; p.status = status;
    p.cu = g.varlen ? g.cu : nullptr;
    p.order = nullptr;
    p.H = g.H; p.T = g.T; p.N = g.N; p.scale = g.scale; p.eps = g.eps; p.l2norm = g.l2norm;
    if (g.varlen) {
        int32_t *order = (int32_t *)ws;
        k_order<<<(g.N + 127) / 128, 128, 0, st>>>(g.cu, g.N, order);
        cudaError_t e = cudaPeekAtLastError();
        if (e != cudaSuccess) return e;
        p.order = order;
    }
    CUtensorMap mq, mk, mv;
    const long long maprows = rows > 0 ? rows : 1;
    if (!make_map(&mq, q, maprows) || !make_map(&mk, k, maprows) || !make_map(&mv, v, maprows))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_fast_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    k_fast_fwd<<<items, NTHREADS, SMEM_BYTES, st>>>(mq, mk, mv, p);
    return cudaPeekAtLastError();
}

}  // namespace fast
}  // namespace gdn
