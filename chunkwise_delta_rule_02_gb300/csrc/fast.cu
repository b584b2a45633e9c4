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
// The state is kept in TMEM as S_hat = S / G with a pending scale G (the
// product of the chunk decays exp(gamma_C) since the last renormalisation), so
// the decay costs nothing on the sequential chain: the factors G enter W, Qt
// and the U2 operand instead, and S_hat is rescaled in place only when G would
// fall below 2^-30 (or a single chunk decays further than that).
//
// Everything is computed transposed so every tcgen05.mma has M = 128 (S_hat^T
// lives in TMEM with lane = value column, column = key row):
//   G   : TMEM[GW]  = [K; Q] K^T              (SS, 128 x 64 x 128)
//   W^T : TMEM[GW]  = K^T T'^T                 (SS, A MN-major; T' = T diag(exp(gamma) n))
//   U^T : TMEM[X]   = V^T T^T                  (SS, A MN-major)
//   1   : TMEM[X]  += S_hat^T (-G W^T)         (TS tf32: A = the fp32 state in TMEM)
//   3   : TMEM[O]   = S_snap^T Qt^T            (TS bf16, Qt = diag(exp(gamma) m G) Q)
//   4   : TMEM[O]  += Unew^T P^T               (TS bf16)
//   2   : TMEM[S]  += U2^T K                   (TS bf16, B MN-major; U2 = diag(f) Unew)
//
// Warp roles (512 threads): warp 0 issues TMA loads and fetches beta / g;
// warp 1 owns TMEM and one of its lanes issues every MMA (an event-driven
// scheduler that keeps the sequential chain 1 -> 2 -> 1 ahead of everything
// else); warpgroup 1 turns the Unew accumulator into the bf16 operands U1 / U2;
// warpgroup 2 does the chunk preparation (gates, norms, Gram masks, triangular
// solve, W); warpgroup 3 owns the state (initial state, bf16 snapshot,
// renormalisation, final state) and the output.  Every wait is bounded; a wait
// that runs out sets the status word and the block winds down (waiting, bounded,
// for its own copies and MMAs) before releasing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "fast.h"
#include "prep_math.cuh"
#include "sm100.cuh"

// Optional event timeline of block 0 (compiled only with -DGDN_TRACE).
#ifdef GDN_TRACE
__device__ unsigned long long g_gdn_trace[256][24];
#define TR(n, e)                                                                 \
    do {                                                                         \
        if (blockIdx.x == 0 && (n) < 256) {                                      \
            unsigned long long t_;                                               \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));               \
            g_gdn_trace[(n)][(e)] = t_;                                          \
        }                                                                        \
    } while (0)
#else
#define TR(n, e) \
    do {         \
    } while (0)
#endif

namespace gdn {
namespace fast {
using namespace sm100;
using namespace prep;

namespace {

constexpr int C = 64;
constexpr int D = 128;
constexpr int NTHREADS = 512;
constexpr long long WAIT_BUDGET = 4000000000LL;   // clock cycles (about 2 s)
constexpr float RENORM_BELOW = 9.313225746154785e-10f;  // 2^-30

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_KQ = 0;          // 2 stages x 32 KB: per 64-column half: K rows | Q rows
constexpr uint32_t OFF_V = 65536;       // 2 stages x 16 KB: V, two 64-column halves
constexpr uint32_t OFF_WF = 98304;      // 32 KB  -G W as tf32 operand [token][dk], 4 atoms of 32 dk
constexpr uint32_t OFF_TB = 131072;     // 8 KB   T  bf16 [r][i]
constexpr uint32_t OFF_TPB = 139264;    // 8 KB   T' bf16 [r][i]
constexpr uint32_t OFF_PB = 147456;     // 2 x 8 KB P bf16 [r][i]
constexpr uint32_t OFF_OST = 163840;    // 16 KB  output staging [64][128] bf16
constexpr uint32_t AST = 68;            // row stride (floats) of the solve matrices
constexpr uint32_t OFF_AF = 180224;     // A fp32 [64][68]
constexpr uint32_t OFF_XF = OFF_AF + 64 * AST * 4;  // X = (I + A)^-1 fp32 [64][68]
constexpr uint32_t OFF_BG = OFF_XF + 64 * AST * 4;  // 2 stages x (beta[64], g[64]) fp32
constexpr uint32_t OFF_VEC = OFF_BG + 2 * 128 * 4;  // per-chunk vectors, 9 x 64 floats
constexpr uint32_t OFF_RING = OFF_VEC + 9 * 64 * 4; // 2 ring slots
constexpr uint32_t OFF_BAR = OFF_RING + 2 * 320;
constexpr uint32_t OFF_MISC = OFF_BAR + 32 * 8;
constexpr uint32_t SMEM_USED = OFF_MISC + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for the manual 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory");

struct Ring {           // per-chunk scalars handed from the prep warpgroup to the others
    float f[64];        // U2 row scale: exp(gamma_C - gamma_r) n_r / G_next (0 past the chunk)
    float rscale;       // renormalising chunk: S_hat <- rscale S_hat before MMA 2
    float gnext;        // pending scale after the chunk
    int renorm;         // 1 if this chunk renormalises
    int len;            // rows of this chunk
    long long row0;     // first token row (flattened [B*H*T] index)
    int pad[10];
};
static_assert(sizeof(Ring) <= 320, "ring slot");

// TMEM column map (512 columns allocated)
constexpr uint32_t TM_S = 0;       // 128: S_hat^T fp32 (lane = dv, column = dk)
constexpr uint32_t TM_SNAP = 128;  // 64 : S_hat^T bf16 pairs
constexpr uint32_t TM_X = 192;     // 64 : Unew^T accumulator (lane = dv, column = token)
constexpr uint32_t TM_U1 = 256;    // 2 x 32: Unew^T bf16 pairs
constexpr uint32_t TM_U2 = 320;    // 2 x 32: (f o Unew)^T bf16 pairs
constexpr uint32_t TM_GW = 384;    // 64 : [K;Q]K^T, then W^T
constexpr uint32_t TM_O = 448;     // 64 : O^T

// mbarrier slots
enum {
    B_FULL = 0, B_EMPTY = 2, B_G = 4, B_W = 5, B_X = 6, B_O = 7, B_F = 9, B_TREADY = 10,
    B_WREADY = 11, B_GWFREE = 12, B_XFREE = 13, B_U2READY = 14, B_SNAP = 15, B_OFREE = 16,
    B_RINGFREE = 17, B_RINGREADY = 19, B_SINIT = 21, B_ABORTED = 22, B_S = 23, B_SFIX = 24,
    NBAR = 25
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
    int longhorn;           // step size beta / (1 + beta k^T k) instead of beta
};

// shared-memory descriptor advanced by a byte offset (start address field, >> 4)
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

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
    int *s_safe = (int *)(sm + OFF_MISC + 16);
    float *s_beta = (float *)(sm + OFF_VEC);   // beta_r (0 past the chunk)
    float *s_gl = s_beta + 64;                  // gamma_r * log2(e)
    float *s_nk = s_gl + 64;                    // key norm factors n_r
    float *s_nq = s_nk + 64;                    // query norm factors m_r
    float *s_tc = s_nq + 64;                    // beta_i exp(gamma_i) n_i   (columns of T')
    float *s_qs = s_tc + 64;                    // exp(gamma_r) m_r G        (rows of Qt)
    float *s_ra = s_qs + 64;                    // beta_r n_r exp(gamma_r)   (rows of A, factored)
    float *s_cb = s_ra + 64;                    // n_i exp(-gamma_i)         (columns of A and P, factored)
    float *s_kk = s_cb + 64;                    // k_hat_r^T k_hat_r         (Longhorn's step size)
    Ring *ring = (Ring *)(sm + OFF_RING);
    float *Af = (float *)(sm + OFF_AF);
    float *Xf = (float *)(sm + OFF_XF);

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
                i == B_SNAP || i == B_OFREE || i == B_RINGREADY || i == B_RINGREADY + 1 ||
                i == B_SINIT || i == B_SFIX)
                cnt = 4;
            if (i == B_RINGFREE || i == B_RINGFREE + 1) cnt = 8;
            if (i == B_FULL || i == B_FULL + 1) cnt = 2;
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
        int issued = 0;
        for (int n = 0; n < nch; ++n) {
            const int s = n & 1;
            bool ok = true;
            if (n >= 2) {
                if (lane == 0) ok = wait(B_EMPTY + s, (uint32_t)((n >> 1) - 1));
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            }
            // leave together: the warp's later shuffles and __syncwarp need every lane
            if (__shfl_sync(0xffffffffu, (!ok || *abort_flag) ? 1 : 0, 0)) break;
            const long long row = rowbase + (long long)n * C;
            const int len = min(C, L - n * C);
            if (lane == 0) {
                uint8_t *kq = sm + OFF_KQ + s * 32768;
                uint8_t *vv = sm + OFF_V + s * 16384;
                mbar_expect_tx(&bar[B_FULL + s], 49152);
                TR(n, 0);
                tma_load_2d(kq, &tm_k, &bar[B_FULL + s], 0, (int)row);
                tma_load_2d(kq + 16384, &tm_k, &bar[B_FULL + s], 64, (int)row);
                tma_load_2d(kq + 8192, &tm_q, &bar[B_FULL + s], 0, (int)row);
                tma_load_2d(kq + 24576, &tm_q, &bar[B_FULL + s], 64, (int)row);
                tma_load_2d(vv, &tm_v, &bar[B_FULL + s], 0, (int)row);
                tma_load_2d(vv + 8192, &tm_v, &bar[B_FULL + s], 64, (int)row);
            }
            // beta and g of the chunk's rows (zero past its end)
            float *bg = (float *)(sm + OFF_BG) + s * 128;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = lane + 32 * hh;
                bg[r] = r < len ? __bfloat162float(p.beta[row + r]) : 0.f;
                bg[64 + r] = (r < len && p.gate) ? p.gate[row + r] : 0.f;
            }
            if (__any_sync(0xffffffffu, bg[64 + lane] > 0.f || bg[96 + lane] > 0.f) && lane == 0)
                raise_status(p.status, kStatusPositiveGate);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_FULL + s]);
            issued = n + 1;
        }
        if (lane == 0 && *abort_flag) {
            // let copies still in flight land before the block's shared memory goes away
            for (int n = (issued > 2 ? issued - 2 : 0); n < issued; ++n)
                mbar_wait(&bar[B_FULL + (n & 1)], (uint32_t)(n >> 1) & 1u, WAIT_BUDGET, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && nch > 0) {
            // descriptor bases; every operand offset below is a compile-time constant
            const uint64_t dKQ0 = sdesc(sb + OFF_KQ, 16, 1024), dKQ1 = sdesc(sb + OFF_KQ + 32768, 16, 1024);
            const uint64_t dKm0 = sdesc(sb + OFF_KQ, 16384, 1024), dKm1 = sdesc(sb + OFF_KQ + 32768, 16384, 1024);
            const uint64_t dVm0 = sdesc(sb + OFF_V, 8192, 1024), dVm1 = sdesc(sb + OFF_V + 16384, 8192, 1024);
            const uint64_t dTB = sdesc(sb + OFF_TB, 16, 1024), dTPB = sdesc(sb + OFF_TPB, 16, 1024);
            const uint64_t dPB0 = sdesc(sb + OFF_PB, 16, 1024), dPB1 = sdesc(sb + OFF_PB + 8192, 16, 1024);
            const uint64_t dWF = sdesc(sb + OFF_WF, 16, 1024);
            // A fixed order per chunk n, each step blocking (suspending) on what it needs:
            //   1(n); 3(n); G(n+1); 2(n); 4(n); W/U(n+1)
            // G(n+1) only needs TMA data and the W^T of chunk n read out, which come before
            // 1(n) is possible, so nothing off the chain holds the chain 1(n) -> 2(n) -> 1(n+1).
            auto issue_G = [&](int m) {
                tc_fence_after();
                const uint64_t dq = (m & 1) ? dKQ1 : dKQ0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint64_t d = dadd(dq, (j >> 2) * 16384 + (j & 3) * 32);
                    mma_bf16_ss(tmem + TM_GW, d, d, ID_F16_N64, j > 0);
                }
                mma_commit(&bar[B_G]);
                TR(m, 7);
            };
            auto issue_WU = [&](int m) {
                tc_fence_after();
                const uint64_t dk = (m & 1) ? dKm1 : dKm0;
                const uint64_t dv = (m & 1) ? dVm1 : dVm0;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_bf16_ss(tmem + TM_GW, dadd(dk, j * 2048), dadd(dTPB, j * 32), ID_F16_N64_AMN, j > 0);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_bf16_ss(tmem + TM_X, dadd(dv, j * 2048), dadd(dTB, j * 32), ID_F16_N64_AMN, j > 0);
                mma_commit(&bar[B_W]);
                TR(m, 8);
            };
            bool ok = wait(B_FULL, 0);
            if (ok) issue_G(0);
            ok = ok && wait(B_TREADY, 0);
            if (ok) issue_WU(0);
            ok = ok && wait(B_SINIT, 0);
            for (int n = 0; n < nch && ok; ++n) {
                // 1: X += S_hat^T (-G W^T)   tf32, A = fp32 state in TMEM
                if (!(ok = wait(B_WREADY, (uint32_t)n))) break;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    mma_tf32_ts(tmem + TM_X, tmem + TM_S + 8 * j, dadd(dWF, (j >> 2) * 8192 + (j & 3) * 32),
                                ID_TF32_N64, 1);
                mma_commit(&bar[B_X]);
                TR(n, 9);
                // 3: O^T = S_snap^T Qt^T
                if (!(ok = wait(B_SNAP, (uint32_t)n))) break;
                if (n >= 1 && !(ok = wait(B_OFREE, (uint32_t)(n - 1)))) break;
                tc_fence_after();
                {
                    const uint64_t dq = (n & 1) ? dKQ1 : dKQ0;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        mma_bf16_ts(tmem + TM_O, tmem + TM_SNAP + 8 * j,
                                    dadd(dq, (j >> 2) * 16384 + 8192 + (j & 3) * 32), ID_F16_N64, j > 0);
                }
                TR(n, 10);
                // G of the next chunk
                if (n + 1 < nch) {
                    if (!(ok = wait(B_FULL + ((n + 1) & 1), (uint32_t)((n + 1) >> 1)))) break;
                    if (!(ok = wait(B_GWFREE, (uint32_t)n))) break;
                    issue_G(n + 1);
                }
                // 2: S_hat^T += U2^T K      B = K tile, MN-major (dk contiguous)
                if (!(ok = wait(B_U2READY, (uint32_t)n))) break;
                if (!(ok = wait(B_SFIX, (uint32_t)n))) break;
                tc_fence_after();
                {
                    const uint64_t dk = (n & 1) ? dKm1 : dKm0;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_bf16_ts(tmem + TM_S, tmem + TM_U2 + (n & 1) * 32 + 8 * j, dadd(dk, j * 2048),
                                    ID_F16_N128_BMN, 1);
                }
                mma_commit(&bar[B_S]);
                mma_commit(&bar[B_EMPTY + (n & 1)]);
                if (n + 1 == nch) mma_commit(&bar[B_F]);
                TR(n, 11);
                // 4: O^T += Unew^T P^T
                {
                    const uint64_t dp = (n & 1) ? dPB1 : dPB0;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_bf16_ts(tmem + TM_O, tmem + TM_U1 + (n & 1) * 32 + 8 * j, dadd(dp, j * 32),
                                    ID_F16_N64, 1);
                }
                mma_commit(&bar[B_O + (n & 1)]);
                TR(n, 12);
                // W^T and U^T of the next chunk (X is free once Unew(n) has been read out)
                if (n + 1 < nch) {
                    if (!(ok = wait(B_TREADY, (uint32_t)(n + 1)))) break;
                    if (!(ok = wait(B_XFREE, (uint32_t)n))) break;
                    issue_WU(n + 1);
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
            // warp-uniform decisions only: tcgen05.ld / st below are warp-collective
            if (!__all_sync(0xffffffffu, wait(B_X, (uint32_t)n))) break;
            if (warp == 4 && lane == 0) TR(n, 13);
            tc_fence_after();
            uint32_t x[64];
            tmem_ld32(tmem + lrow + TM_X, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
            tmem_ld32(tmem + lrow + TM_X + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_XFREE]);
            if (!__all_sync(0xffffffffu, wait(B_RINGREADY + (n & 1), (uint32_t)(n >> 1)))) break;
            const float4 *f4 = reinterpret_cast<const float4 *>(ring[n & 1].f);
            uint32_t u1[32], u2[32];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float4 f = f4[c];
                const float a = __uint_as_float(x[4 * c]), b = __uint_as_float(x[4 * c + 1]);
                const float cc = __uint_as_float(x[4 * c + 2]), d = __uint_as_float(x[4 * c + 3]);
                u1[2 * c] = pack_bf16(a, b);
                u1[2 * c + 1] = pack_bf16(cc, d);
                u2[2 * c] = pack_bf16(a * f.x, b * f.y);
                u2[2 * c + 1] = pack_bf16(cc * f.z, d * f.w);
            }
            tmem_st32(tmem + lrow + TM_U1 + (n & 1) * 32, u1);
            tmem_st32(tmem + lrow + TM_U2 + (n & 1) * 32, u2);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (warp == 4) TR(n, 14);
                mbar_arrive(&bar[B_U2READY]);
                mbar_arrive(&bar[B_RINGFREE + (n & 1)]);
            }
        }
    } else if (warp >= 8 && warp < 12) {
        // ------------------------------------------------------------ WG2: chunk preparation
        const int t = tid - 256;          // 0..127
        const int q4 = warp & 3;          // TMEM lane quarter / warp index in the group
        const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
        float Gpend = 1.f;                // pending scale of the state entering the chunk
        for (int n = 0; n < nch; ++n) {
            const int s = n & 1;
            const int len = min(C, L - n * C);
            const long long row0 = rowbase + (long long)n * C;
            uint8_t *kq = sm + OFF_KQ + s * 32768;
            if (n >= 2) wait(B_RINGFREE + s, (uint32_t)((n >> 1) - 1));
            wait(B_FULL + s, (uint32_t)(n >> 1));
            if (t == 0) TR(n, 1);
            // gates: inclusive scan of g within the chunk, in log2 units (one warp, two rows per lane)
            if (warp == 8) {
                const float *bg = (const float *)(sm + OFF_BG) + s * 128;
                float g0 = bg[64 + lane], g1 = bg[96 + lane];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    float a0 = __shfl_up_sync(0xffffffffu, g0, o);
                    float a1 = __shfl_up_sync(0xffffffffu, g1, o);
                    if (lane >= o) { g0 += a0; g1 += a1; }
                }
                g1 += __shfl_sync(0xffffffffu, g0, 31);
                g0 *= 1.4426950408889634f;
                g1 *= 1.4426950408889634f;
                s_gl[lane] = g0;
                s_gl[lane + 32] = g1;
                s_beta[lane] = bg[lane];
                s_beta[lane + 32] = bg[32 + lane];
                // factored exponentials exp(gamma_r) exp(-gamma_i) are safe when |gamma| stays small
                float mx = fmaxf(fabsf(g0), fabsf(g1));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (lane == 0) *s_safe = mx < 100.f;
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
                    const float nk = ok ? (p.l2norm ? rsqrtf(sk + p.eps) : 1.f) : 0.f;
                    s_nk[r] = nk;
                    s_nq[r] = ok ? (p.l2norm ? rsqrtf(sq + p.eps) : 1.f) : 0.f;
                    s_kk[r] = sk * nk * nk;
                }
            }
            named_bar(2, 128);
            // pending-scale bookkeeping (every thread keeps the same copy) and per-row vectors
            const float glC = s_gl[len - 1];
            const float GammaC = ex2f(glC);
            const float Gn = Gpend;
            float Gnext = Gn * GammaC;
            const bool renorm = Gnext < RENORM_BELOW;
            const float fdiv = renorm ? 1.f : 1.f / Gnext;
            if (renorm) Gnext = 1.f;
            Gpend = Gnext;
            const bool safe = *s_safe != 0;
            if (t < 64) {
                const float gl = s_gl[t];
                const float e = ex2f(gl);
                // the step size: beta, or Longhorn's beta / (1 + beta k^T k)
                float bt = s_beta[t];
                if (p.longhorn) {
                    bt = bt / fmaf(bt, s_kk[t], 1.f);
                    s_beta[t] = bt;
                }
                s_tc[t] = bt * e * s_nk[t];
                s_qs[t] = e * s_nq[t] * Gn;
                s_ra[t] = bt * s_nk[t] * e;
                s_cb[t] = safe ? s_nk[t] * ex2f(-gl) : 0.f;
                ring[s].f[t] = ex2f(glC - gl) * s_nk[t] * fdiv;
                if (t == 0) {
                    ring[s].rscale = Gn * GammaC;
                    ring[s].gnext = Gnext;
                    ring[s].renorm = renorm ? 1 : 0;
                    ring[s].len = len;
                    ring[s].row0 = row0;
                }
            }
            named_bar(2, 128);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_RINGREADY + s]);
            if (t == 0) TR(n, 2);
            // Gram / QK^T from TMEM -> A (fp32) and P (bf16)
            wait(B_G, (uint32_t)n);
            if (t == 0) TR(n, 3);
            tc_fence_after();
            if (q4 >= 2 && n >= 2) wait(B_O + s, (uint32_t)((n >> 1) - 1));
            {
                uint32_t v[64];
                tmem_ld32(tmem + lrow + TM_GW, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
                tmem_ld32(tmem + lrow + TM_GW + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
                tmem_ld_wait();
                if (q4 < 2) {
                    const int r = q4 * 32 + lane;
                    float4 *arow = reinterpret_cast<float4 *>(Af + r * AST);
                    if (safe) {
                        const float ra = s_ra[r];
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            float a[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 4 * c + e;
                                a[e] = (i < r) ? ra * s_cb[i] * __uint_as_float(v[i]) : 0.f;
                            }
                            arow[c] = make_float4(a[0], a[1], a[2], a[3]);
                        }
                    } else {
                        const float br = s_beta[r] * s_nk[r], gr = s_gl[r];
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            float a[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = 4 * c + e;
                                a[e] = (i < r) ? br * s_nk[i] * __uint_as_float(v[i]) * ex2f(gr - s_gl[i]) : 0.f;
                            }
                            arow[c] = make_float4(a[0], a[1], a[2], a[3]);
                        }
                    }
                } else {
                    const int r = (q4 - 2) * 32 + lane;
                    uint8_t *prow = sm + OFF_PB + s * 8192;
                    const float mr = s_nq[r], gr = s_gl[r];
                    const float rp = mr * ex2f(gr);
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i0 = c8 * 8 + 2 * e, i1 = i0 + 1;
                            float a0, a1;
                            if (safe) {
                                a0 = (i0 <= r) ? rp * s_cb[i0] * __uint_as_float(v[i0]) : 0.f;
                                a1 = (i1 <= r) ? rp * s_cb[i1] * __uint_as_float(v[i1]) : 0.f;
                            } else {
                                a0 = (i0 <= r) ? mr * s_nk[i0] * __uint_as_float(v[i0]) * ex2f(gr - s_gl[i0]) : 0.f;
                                a1 = (i1 <= r) ? mr * s_nk[i1] * __uint_as_float(v[i1]) * ex2f(gr - s_gl[i1]) : 0.f;
                            }
                            w[e] = pack_bf16(a0, a1);
                        }
                        *(uint4 *)(prow + sw128(r, c8 * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            if (t == 0) TR(n, 20);
            // Qt = diag(exp(gamma) m G) Q, in place in the stage buffer (MMA G has read Q)
            {
                const int r = t >> 1, hh = t & 1;
                const float f = s_qs[r];
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
            // X = (I + A)^-1 (16 x 16 blocks; tensor-core off-diagonal products)
            solve_unit_lower_64<AST>(Af, Xf, lane, q4, 2);
            if (t == 0) TR(n, 19);
            // T = X diag(beta) and T' = X diag(beta exp(gamma) n) as bf16 operands [r][i]
            {
                const int r = t >> 1, hh = t & 1;
                const float4 *xr = reinterpret_cast<const float4 *>(Xf + r * AST + hh * 32);
                const float4 *b4 = reinterpret_cast<const float4 *>(s_beta + hh * 32);
                const float4 *c4 = reinterpret_cast<const float4 *>(s_tc + hh * 32);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint32_t wt[4], wp[4];
#pragma unroll
                    for (int e2 = 0; e2 < 2; ++e2) {
                        const int q = c8 * 2 + e2;
                        float4 x = xr[q];
                        const int i0 = hh * 32 + 4 * q;
                        if (i0 > r) x.x = 0.f;
                        if (i0 + 1 > r) x.y = 0.f;
                        if (i0 + 2 > r) x.z = 0.f;
                        if (i0 + 3 > r) x.w = 0.f;
                        const float4 bb = b4[q], cc = c4[q];
                        wt[2 * e2] = pack_bf16(x.x * bb.x, x.y * bb.y);
                        wt[2 * e2 + 1] = pack_bf16(x.z * bb.z, x.w * bb.w);
                        wp[2 * e2] = pack_bf16(x.x * cc.x, x.y * cc.y);
                        wp[2 * e2 + 1] = pack_bf16(x.z * cc.z, x.w * cc.w);
                    }
                    const uint32_t off = sw128(r, (hh * 4 + c8) * 16);
                    *(uint4 *)(sm + OFF_TB + off) = make_uint4(wt[0], wt[1], wt[2], wt[3]);
                    *(uint4 *)(sm + OFF_TPB + off) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_TREADY]);
            if (t == 0) TR(n, 4);
            // W^T from TMEM -> -G W as the tf32 operand of MMA 1
            wait(B_W, (uint32_t)n);
            if (t == 0) TR(n, 5);
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
                const float ng = -Gn;
#pragma unroll
                for (int r = 0; r < 64; ++r)
                    *(float *)(wf + sw128(r, (dk & 31) * 4)) = ng * __uint_as_float(v[r]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_WREADY]);
            if (t == 0) TR(n, 6);
            if (bar_any(2, 128, *abort_flag != 0)) break;
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ WG3: state and output
        const int t = tid - 384;
        const int dv = (warp & 3) * 32 + lane;
        const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
        // initial state: S^T[dv][dk] = h0[dk][dv] (pending scale 1)
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
        // output epilogue of chunk m: O^T from TMEM -> o rows (staged through shared memory)
        auto output = [&](int m) {
            const int s = m & 1;
            wait(B_O + s, (uint32_t)(m >> 1));
            if (t == 0) TR(m, 17);
            tc_fence_after();
            uint32_t ov[64];
            tmem_ld32(tmem + lrow + TM_O, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
            tmem_ld32(tmem + lrow + TM_O + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_OFREE]);
            const int len = ring[s].len;
            const long long row0 = ring[s].row0;
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
            if (t == 0) TR(m, 18);
        };
        bool ok = true;
        for (int n = 0; n < nch; ++n) {
            const int s = n & 1;
            // bf16 snapshot of S_hat_n (after MMA 2 of the previous chunk)
            if (n >= 1) wait(B_S, (uint32_t)(n - 1));
            if (t == 0) TR(n, 15);
            tc_fence_after();
            for (int k0 = 0; k0 < D; k0 += 32) {
                uint32_t r[32], hbuf[16];
                tmem_ld32(tmem + lrow + TM_S + k0, r);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    hbuf[c] = pack_bf16(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1]));
                tmem_st16(tmem + lrow + TM_SNAP + k0 / 2, hbuf);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_SNAP]);
            if (t == 0) TR(n, 16);
            // renormalising chunk: S_hat <- (G exp(gamma_C)) S_hat once MMA 1 has read it
            wait(B_RINGREADY + s, (uint32_t)(n >> 1));
            if (ring[s].renorm) {
                const float rs = ring[s].rscale;
                wait(B_X, (uint32_t)n);
                tc_fence_after();
                for (int k0 = 0; k0 < D; k0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lrow + TM_S + k0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * rs);
                    tmem_st32(tmem + lrow + TM_S + k0, r);
                }
                tmem_st_wait();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_SFIX]);
            if (n >= 1) output(n - 1);
            if (bar_any(3, 128, *abort_flag != 0)) { ok = false; break; }
        }
        if (ok && nch > 0) output(nch - 1);
        // final state h_T = G S_hat
        if (ok && !*abort_flag && p.hT) {
            const float Gf = nch > 0 ? ring[(nch - 1) & 1].gnext : 1.f;
            if (nch == 0 || wait(B_F, 0)) {
                tc_fence_after();
                for (int k0 = 0; k0 < D; k0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lrow + TM_S + k0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        p.hT[sidx + (size_t)(k0 + k) * D + dv] = Gf * __uint_as_float(r[k]);
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
#ifdef GDN_TRACE
extern "C" int gdn_trace_fetch(unsigned long long *host, size_t count)
{
    return cudaMemcpyFromSymbol(host, g_gdn_trace, count * sizeof(unsigned long long)) == cudaSuccess ? 0 : 1;
}
#endif

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
    p.longhorn = g.longhorn;
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
