// Per-chunk gradients of the (gated) delta rule on the tcgen05 tensor cores, for
// bf16 inputs with d_k = d_v = 128 and chunk C = 64.  It replaces the three staged
// per-chunk backward kernels of the general path: given the state entering each
// chunk and the adjoint leaving it (S_in, dS_out, with Unew and dUnew, all bf16 from
// the two scans), one persistent CTA per SM takes chunks in turn and computes
// dq, dk, dv, dbeta and dg of the chunk, recomputing from the raw q, k, v, beta, g
// everything else it needs (norms, gates, the UT transform).
//
// (Reverse-mode derivative of the chunk form: "Parallelizing Linear Transformers
// with the Delta Rule over Sequence Length", WY / UT representation, with the chunk
// states recomputed in the backward, reply Q2; "Gated DeltaNet", gates as
// within-chunk cumulative log-decays.)  Per chunk, with rows r, i < len, raw q, k,
// normalised K^ = diag(n) K, Q^ = diag(m) Q, Gamma = exp(gamma), E = exp(gamma_C -
// gamma), D_ri = exp(gamma_r - gamma_i), b the step size:
//   Y = dO S_in^T, Z = dUnew S_in^T (dW = -Z), X = Unew dS_out^T, dP = s lower(dO Unew^T)
//   A = strict_lower(diag(b) K^K^T o D), Linv = (I + A)^-1, T = Linv diag(b)
//   dT = dW (diag(Gamma) K^)^T + dUnew V^T, X2 = Linv^T dT diag(b), dA = strict_lower(-X2 Linv^T)
//   dQ^ = s diag(Gamma) Y + (dP o D) K^
//   dK^ = diag(Gamma) T^T dW + (dP o D)^T Q^ + (dKK + dKK^T) K^ + diag(E) X,  dKK = dA o b_r o D
//   dV  = T^T dUnew,  d beta through T and A,  d gamma from Gamma, E, D, Gamma_C
// then the normalisation's chain rule.
//
// Every product is one tcgen05.mma chain with M = 128: operands whose rows are the
// chunk's 64 tokens are stacked two to a tile ([dO; dUnew], [U; dO], [K; Q]) or
// used with their upper 64 rows as don't-care rows whose results are never read;
// the state products keep M = 128 as the state's rows.  The C x C inverse and its
// adjoint (two 64 x 64 x 64 products) stay on warp-level tf32 tiles, as the
// triangular solve does everywhere in this library.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "bwd_tc.h"
#include "prep_math.cuh"
#include "sm100.cuh"

// Optional event timeline of CTA 0's first tasks (compiled only with -DGDN_TRACE).
#ifdef GDN_TRACE
__device__ unsigned long long g_btc_trace[16][24];
#define BTR(n, e)                                                                \
    do {                                                                         \
        if (blockIdx.x == 0 && threadIdx.x == 0 && (n) < 16) {                   \
            unsigned long long t_;                                               \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));               \
            g_btc_trace[(n)][(e)] = t_;                                          \
        }                                                                        \
    } while (0)
extern "C" int gdn_btc_trace_fetch(unsigned long long *host, size_t count)
{
    return cudaMemcpyFromSymbol(host, g_btc_trace, count * sizeof(unsigned long long)) == cudaSuccess ? 0 : 1;
}
#else
#define BTR(n, e) \
    do {          \
    } while (0)
#endif

namespace gdn {
namespace btc {
using namespace sm100;
using namespace prep;

namespace {

constexpr int C = 64;
constexpr int D = 128;
constexpr int NTHREADS = 512;
constexpr int NCOMPUTE = NTHREADS - 32;    // warps 0..14 compute; warp 15 issues the copies
constexpr int NCWARPS = NCOMPUTE / 32;
constexpr long long BUDGET = 4000000000LL;   // clock cycles (about 2 s) for any one wait

// shared memory (bytes from a 1024-aligned base).  Tiles are bf16 with the 128-byte
// swizzle, stored as 64-column halves of 128-byte rows.
constexpr uint32_t SM_KQ = 0;          // half h at h * 16384: K rows (8 KB) | Q rows (8 KB)
constexpr uint32_t SM_UOD = 32768;     // half h at h * 24576: Unew | dO | dUnew (8 KB each)
constexpr uint32_t SM_V = 81920;       // half h at h * 8192
constexpr uint32_t SM_S = 98304;       // S_in [dk][dv], half h at h * 16384
constexpr uint32_t SM_DS = 131072;     // dS_out [dk][dv]
constexpr uint32_t SM_VEC = 163840;    // 24 vectors of 64 floats
constexpr uint32_t SM_RED = SM_VEC + 24 * 256;   // 2048 floats of partial row sums
constexpr uint32_t SM_BAR = SM_RED + 8192;
constexpr uint32_t SM_XTRA = SM_BAR + 1024;   // two fp32 C x C buffers of their own
constexpr int AST = 66;                    // row stride (floats) of the fp32 C x C buffers: rows
                                           // 8-byte aligned, a column touches 16 banks
constexpr uint32_t FBYTES = 64 * AST * 4;  // one fp32 C x C buffer
constexpr uint32_t SM_OUT = SM_XTRA + 17408;   // dq, dk tiles (bf16, 16 KB each) for the tensor stores
constexpr uint32_t SM_END = SM_OUT + 32768;
constexpr uint32_t SMEM_BYTES = SM_END + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
constexpr uint32_t UOD_HALF = 24576;

// reuse once the first products have completed (S_in, dS_out, Unew, dO free)
constexpr uint32_t F_AX = SM_S;                // fp32 [64][AST]: A, then the packed inverse
constexpr uint32_t F_KD = SM_S + FBYTES;       // K^K^T o D (strict lower), then dKK
constexpr uint32_t F_G = SM_S + 2 * FBYTES;    // P, then dP o P, then E
static_assert(SM_S + 3 * FBYTES <= SM_VEC, "fp32 buffers over S_in, dS_out");
constexpr uint32_t F_TMP = SM_XTRA;            // Linv o dT, then the dv tile
static_assert(FBYTES <= 17408 && SM_XTRA % 1024 == 0, "dv tile over the Linv o dT buffer");
constexpr uint32_t T_DQ = SM_OUT, T_DK = SM_OUT + 16384, T_DV = SM_XTRA;   // [64 rows][128] bf16, two 8 KB halves
constexpr uint32_t T_Z = SM_UOD;           // Z rows (over Unew): half h at h * UOD_HALF
constexpr uint32_t T_DP = SM_UOD + 8192;   // (dP o D) n_i [r][i] (over dO, half 0)
constexpr uint32_t T_DP2 = SM_UOD + UOD_HALF + 8192;   // (dP o D) m_r [r][i] (over dO, half 1)
// once the dUnew V^T product has completed (V free)
constexpr uint32_t T_LI = SM_V;            // Linv [r][i]
constexpr uint32_t T_ADJ = SM_V + 8192;    // dT diag(b) [r][c], then X2 [a][c], then (dKK + dKK^T) n_r [i][r]
// row-sum scratch (floats): [0, 512) the dq and dk epilogues' partials, [512, 1024) the
// F / E pass's, whose first 16 also hold the <dS_out, S_in> partials early in a task,
// [1024, 1280) <Q^_r, Y_r> (dq epilogue), [1280, 1536) <K^_r, X_r> (last epilogue)
constexpr int RED_FE = 512;
constexpr int RED_SDS = 512;
constexpr int RED_QT = 1024;
constexpr int RED_SE = 1280;

// vectors (each 64 floats)
enum {
    V_BETA = 0, V_GAM, V_G, V_GI, V_E, V_N, V_M, V_KAP, V_B, V_GN, V_QT, V_SE, V_DB, V_DG, V_K2,
    V_CS, NV
};
static_assert(NV <= 24, "vectors");

// TMEM columns
constexpr uint32_t TM_A = 0;      // Gram [K;Q][K;Q]^T -> dT parts (Z K^T | dUnew V^T) -> dQ2 -> dK accumulator
constexpr uint32_t TM_YZ = 128;   // [Y; Z] -> T^T dW accumulator
constexpr uint32_t TM_X = 256;    // X (lanes 0..63) until the end
constexpr uint32_t TM_DP = 384;   // dO Unew^T (64 columns) -> T^T dUnew accumulator (128)
constexpr uint32_t TM_ADJ = 384;  // X2 (64 columns), dA' = X2 Linv^T (64 columns), after dO Unew^T is read

enum { B_TMA = 0, B_M1, B_M4, B_M5, B_X2, B_DA, B_M6, B_KQFREE, B_SDSFREE, B_DRAIN, NBAR };

constexpr uint32_t ID_128_128 = idesc(1, 128, 128, false, false);
constexpr uint32_t ID_128_64 = idesc(1, 128, 64, false, false);
constexpr uint32_t ID_128_128_BMN = idesc(1, 128, 128, false, true);
constexpr uint32_t ID_128_128_ABMN = idesc(1, 128, 128, true, true);
constexpr uint32_t ID_128_64_ABMN = idesc(1, 128, 64, true, true);

struct Params {
    Geo g;
    const __nv_bfloat16 *beta;
    const float *gate;
    __nv_bfloat16 *dq, *dk, *dv, *dbeta;
    float *dg;
    int ntasks;
};

__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// 32 consecutive bf16 of row `row` of a [rows][128] tile stored as two halves
// `hstride` bytes apart, starting at column c0 (a multiple of 32), as floats
__device__ __forceinline__ void row32(const uint8_t *tile, uint32_t hstride, int row, int c0, float (&x)[32])
{
    const uint8_t *half = tile + (c0 >> 6) * hstride;
    const int cb = (c0 & 63) * 2;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 w = *reinterpret_cast<const uint4 *>(half + sw128(row, cb + 16 * q));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[8 * q + 2 * e] = bf_lo(u[e]);
            x[8 * q + 2 * e + 1] = bf_hi(u[e]);
        }
    }
}

// writes 32 floats as bf16 into row `row`, columns [c0, c0 + 32) of a 64-column half tile
__device__ __forceinline__ void put_row32(uint8_t *half, int row, int c0, const float (&x)[32])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16(x[8 * q + 2 * e], x[8 * q + 2 * e + 1]);
        *reinterpret_cast<uint4 *>(half + sw128(row, c0 * 2 + 16 * q)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__device__ __forceinline__ void tld32(uint32_t taddr, float (&x)[32])
{
    tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
}

__device__ __forceinline__ void tld16(uint32_t taddr, float (&x)[16])
{
    tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(&x[0]));
}

// writes 16 floats as bf16 into row `row`, columns [c0, c0 + 16) of a 64-column half tile
__device__ __forceinline__ void put_row16(uint8_t *half, int row, int c0, const float (&x)[16])
{
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16(x[8 * q + 2 * e], x[8 * q + 2 * e + 1]);
        *reinterpret_cast<uint4 *>(half + sw128(row, c0 * 2 + 16 * q)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// N consecutive floats of an fp32 C x C buffer row (rows only 8-byte aligned) into registers
template <int N>
__device__ __forceinline__ void rowN(const float *v, float (&x)[N])
{
#pragma unroll
    for (int q = 0; q < N / 2; ++q) {
        const float2 t = reinterpret_cast<const float2 *>(v)[q];
        x[2 * q] = t.x; x[2 * q + 1] = t.y;
    }
}

__device__ __forceinline__ float warp_sum32(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace

// ================================================================================= kernel
__global__ void __launch_bounds__(NTHREADS, 1)
k_bwd_tc(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
         const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_ds,
         const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_du,
         const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
         const __grid_constant__ CUtensorMap tm_dv, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    uint64_t *bar = (uint64_t *)(sm + SM_BAR);
    uint32_t *tmem_slot = (uint32_t *)(sm + SM_BAR + NBAR * 8);
    volatile int *s_abort = (volatile int *)(sm + SM_BAR + NBAR * 8 + 4);
    volatile int *s_safe = (volatile int *)(sm + SM_BAR + NBAR * 8 + 8);
    float *vec = (float *)(sm + SM_VEC);
    float *red = (float *)(sm + SM_RED);   // partial row sums
    auto V = [&](int i) { return vec + 64 * i; };
    float *fAX = (float *)(sm + F_AX), *fKD = (float *)(sm + F_KD), *fG = (float *)(sm + F_G),
          *fTMP = (float *)(sm + F_TMP);
    const Geo &g = p.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, cg = warp >> 2;              // TMEM lane quarter, column group
    const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
    const float sc = g.scale;

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(&bar[i], i == B_KQFREE ? 8 : 1);
        fence_barrier_init();
        *s_abort = 0;
        prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_s); prefetch_tmap(&tm_ds); prefetch_tmap(&tm_u); prefetch_tmap(&tm_du);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // base descriptors (the shared-memory base with each stride pair); an operand's descriptor
    // is its base plus the operand's byte offset (>> 4), a constant at every MMA below
    const uint64_t dKM = sdesc(sb, 16, 1024), dM16 = sdesc(sb, 16384, 1024), dM8 = sdesc(sb, 8192, 1024),
                   dMU = sdesc(sb, UOD_HALF, 1024);

    // a bounded wait; a timeout is recorded and ends the CTA's work at the next task boundary
    auto wait = [&](int b, uint32_t phase) -> bool {
        if (mbar_wait(&bar[b], phase & 1u, BUDGET, nullptr)) return true;
        *s_abort = 1;
        raise_status(g.status, kStatusTimeout);
        return false;
    };
    auto task_of = [&](int t, int &j, int &h, int &b, int &t0, int &len) -> bool {
        j = t / g.H;
        h = t - j * g.H;
        int seq, local;
        return chunk_of(g, j, b, t0, len, seq, local);
    };
    // the next task of this CTA at or after t that holds a chunk (ntasks if none)
    auto next_valid = [&](int t) {
        int j, h, b, t0, len;
        while (t < p.ntasks && !task_of(t, j, h, b, t0, len)) t += gridDim.x;
        return t;
    };
    auto coords = [&](int t, long long &row, int &slot) {
        int j, h, b, t0, len;
        task_of(t, j, h, b, t0, len);
        row = ((long long)b * g.H + h) * g.T + t0;
        slot = j * g.H + h;
    };
    // (thread 0) copies of task t's tiles: everything but K, Q first (those tiles are
    // free as soon as a task's last products have completed), K, Q when the task's last
    // epilogue has read them; one phase of B_TMA per task
    // the states (opens the task's phase of B_TMA with all its bytes)
    auto issue_sds = [&](int t) {
        long long row;
        int slot;
        coords(t, row, slot);
        mbar_expect_tx(&bar[B_TMA], 163840);
        for (int hh = 0; hh < 2; ++hh) {
            const int x = 64 * hh;
            tma_load_2d(sm + SM_S + hh * 16384, &tm_s, &bar[B_TMA], x, slot * D);
            tma_load_2d(sm + SM_S + hh * 16384 + 8192, &tm_s, &bar[B_TMA], x, slot * D + 64);
            tma_load_2d(sm + SM_DS + hh * 16384, &tm_ds, &bar[B_TMA], x, slot * D);
            tma_load_2d(sm + SM_DS + hh * 16384 + 8192, &tm_ds, &bar[B_TMA], x, slot * D + 64);
        }
    };
    // Unew, dO, dUnew, V
    auto issue_uodv = [&](int t) {
        long long row;
        int slot;
        coords(t, row, slot);
        for (int hh = 0; hh < 2; ++hh) {
            const int x = 64 * hh;
            tma_load_2d(sm + SM_UOD + hh * UOD_HALF, &tm_u, &bar[B_TMA], x, slot * C);
            tma_load_2d(sm + SM_UOD + hh * UOD_HALF + 8192, &tm_do, &bar[B_TMA], x, (int)row);
            tma_load_2d(sm + SM_UOD + hh * UOD_HALF + 16384, &tm_du, &bar[B_TMA], x, slot * C);
            tma_load_2d(sm + SM_V + hh * 8192, &tm_v, &bar[B_TMA], x, (int)row);
        }
    };
    auto issue_kq = [&](int t) {
        long long row;
        int slot;
        coords(t, row, slot);
        for (int hh = 0; hh < 2; ++hh) {
            tma_load_2d(sm + SM_KQ + hh * 16384, &tm_k, &bar[B_TMA], 64 * hh, (int)row);
            tma_load_2d(sm + SM_KQ + hh * 16384 + 8192, &tm_q, &bar[B_TMA], 64 * hh, (int)row);
        }
    };
    auto prefetch_l2 = [&](int t) {
        long long row;
        int slot;
        coords(t, row, slot);
        const int rn = (int)row;
        for (int hh = 0; hh < 2; ++hh) {
            const int x = 64 * hh;
            tma_prefetch_2d(&tm_k, x, rn); tma_prefetch_2d(&tm_q, x, rn);
            tma_prefetch_2d(&tm_v, x, rn); tma_prefetch_2d(&tm_do, x, rn);
            tma_prefetch_2d(&tm_u, x, slot * C); tma_prefetch_2d(&tm_du, x, slot * C);
            tma_prefetch_2d(&tm_s, x, slot * D); tma_prefetch_2d(&tm_s, x, slot * D + 64);
            tma_prefetch_2d(&tm_ds, x, slot * D); tma_prefetch_2d(&tm_ds, x, slot * D + 64);
        }
    };
    // Warp 15 (one lane) issues every copy and takes no part in the compute barriers: a
    // thread can stall on issuing copies while earlier ones are in flight.  A task's
    // copies go out in three parts, each as soon as the previous task no longer needs
    // the space (mbarriers): the states once its F / E pass has read the fp32 buffers
    // over them, then Unew, dO, dUnew and V once its last products have completed, then
    // K and Q once its last epilogue has read its K rows.  Thread 0 issues the MMAs.
    // A staged output tile (rows of the chunk, two 64-column halves) to global memory:
    // the tensor store by thread 0 for a whole chunk, else the chunk's rows by the compute
    // threads with plain 16-byte stores, consecutive threads along a row.
    auto store_tile = [&](const CUtensorMap *map, uint32_t tile, __nv_bfloat16 *out, long long row, int len) {
        if (len == C) {
            if (tid == 0) {
                tma_store_2d(map, sm + tile, 0, (int)row);
                tma_store_2d(map, sm + tile + 8192, 64, (int)row);
                bulk_commit();
            }
        } else {
            for (int e = tid; e < len * 16; e += NCOMPUTE) {
                const int r = e >> 4, c16 = e & 15, hh = c16 >> 3;
                const uint4 v = *reinterpret_cast<const uint4 *>(sm + tile + hh * 8192 + sw128(r, (c16 & 7) * 16));
                reinterpret_cast<uint4 *>(out + (row + r) * D)[c16] = v;
            }
        }
    };
    bool mma_issued = false;
    uint32_t it = 0;   // tasks run by this CTA (barrier phases)
    if (warp == NCWARPS) {
        if (lane == 0) {
            uint32_t n = 0;   // tasks whose copies have been issued (one B_TMA phase each)
            int tt = next_valid(blockIdx.x);
            while (tt < p.ntasks) {
                if (n > 0 && !mbar_wait(&bar[B_SDSFREE], (n - 1) & 1u, BUDGET, s_abort)) break;
                issue_sds(tt);
                bool ok = n == 0 || mbar_wait(&bar[B_M6], (n - 1) & 1u, BUDGET, s_abort);
                issue_uodv(tt);   // issued either way, so that the phase the first part opened completes
                ok = ok && (n == 0 || mbar_wait(&bar[B_KQFREE], (n - 1) & 1u, BUDGET, s_abort));
                issue_kq(tt);
                ++n;
                const int tn = next_valid(tt + gridDim.x);
                // the task after into L2 once this task's copies have landed (its compute starts)
                ok = ok && mbar_wait(&bar[B_TMA], (n - 1) & 1u, BUDGET, s_abort);
                if (ok && tn < p.ntasks) prefetch_l2(tn);
                if (!ok) break;
                tt = tn;
            }
            // every copy issued has landed before the block exits
            if (n > 0) mbar_wait(&bar[B_TMA], (n - 1) & 1u, BUDGET, nullptr);
        }
    } else {
    int t = next_valid(blockIdx.x);
    while (t < p.ntasks) {
        int j, h, b, t0, len;
        task_of(t, j, h, b, t0, len);
        const long long row = ((long long)b * g.H + h) * g.T + t0;   // first token of the chunk
        const int tnext = next_valid(t + gridDim.x);
        BTR(it, 0);
        // beta, g of the chunk; gamma by a warp scan, in log2 units
        if (warp == 0) {
            float g0 = 0.f, g1 = 0.f;
            const float b0 = lane < len ? __bfloat162float(p.beta[row + lane]) : 0.f;
            const float b1 = lane + 32 < len ? __bfloat162float(p.beta[row + lane + 32]) : 0.f;
            if (p.gate) {
                g0 = lane < len ? p.gate[row + lane] : 0.f;
                g1 = lane + 32 < len ? p.gate[row + lane + 32] : 0.f;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float a0 = __shfl_up_sync(0xffffffffu, g0, o), a1 = __shfl_up_sync(0xffffffffu, g1, o);
                if (lane >= o) { g0 += a0; g1 += a1; }
            }
            g1 += __shfl_sync(0xffffffffu, g0, 31);
            g0 *= 1.4426950408889634f;   // exp(gamma) = 2^g
            g1 *= 1.4426950408889634f;
            V(V_BETA)[lane] = b0;
            V(V_BETA)[lane + 32] = b1;
            V(V_GAM)[lane] = g0;
            V(V_GAM)[lane + 32] = g1;
            // exp(gamma_r - gamma_i) factored as exp(gamma_r) exp(-gamma_i) while both stay in range
            float mx = fmaxf(fabsf(g0), fabsf(g1));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) *s_safe = mx < 100.f;
        }
        wait(B_TMA, it);
        // the previous task's tensor stores have read their staged tiles (long since)
        if (tid == 0) bulk_wait_read();
        if (len < C) {
            // rows past the chunk's end are zero in every token tile
            for (int e = tid; e < (C - len) * 6 * 2 * 8; e += NCOMPUTE) {
                const int r = len + e / 96, rest = e % 96, tile = rest / 16, piece = rest % 16;
                const int hh = piece >> 3, c16 = piece & 7;
                uint32_t base;
                switch (tile) {
                case 0: base = SM_KQ + hh * 16384; break;
                case 1: base = SM_KQ + hh * 16384 + 8192; break;
                case 2: base = SM_UOD + hh * UOD_HALF; break;
                case 3: base = SM_UOD + hh * UOD_HALF + 8192; break;
                case 4: base = SM_UOD + hh * UOD_HALF + 16384; break;
                default: base = SM_V + hh * 8192; break;
                }
                *reinterpret_cast<uint4 *>(sm + base + r * 128 + c16 * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_async_smem();
        }
        named_bar(3, NCOMPUTE);
        if (*s_abort) break;
        BTR(it, 1);
        const float gC = V(V_GAM)[len - 1];
        if (tid == 0) {
            // ---------------------------------------------------------- first products
            mma_issued = true;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t hk = (k & 3) * 32;
                const uint32_t h16 = (k >> 2) * 16384, h24 = (k >> 2) * UOD_HALF;
                const uint64_t dKQ = dadd(dKM, SM_KQ + h16 + hk);
                mma_bf16_ss(tmem + TM_A, dKQ, dKQ, ID_128_128, k > 0);                       // [K;Q][K;Q]^T
                const uint64_t dOdU = dadd(dKM, SM_UOD + h24 + 8192 + hk);
                mma_bf16_ss(tmem + TM_YZ, dOdU, dadd(dKM, SM_S + h16 + hk), ID_128_128, k > 0);   // [dO;dU] S^T
                const uint64_t dUdO = dadd(dKM, SM_UOD + h24 + hk);
                mma_bf16_ss(tmem + TM_X, dUdO, dadd(dKM, SM_DS + h16 + hk), ID_128_128, k > 0);   // [U;dO] dS^T
                mma_bf16_ss(tmem + TM_DP, dOdU, dadd(dKM, SM_UOD + h24 + hk), ID_128_64, k > 0);  // [dO;dU] U^T
            }
            mma_commit(&bar[B_M1]);
        }
        if (tid < 64) {
            const float gm = V(V_GAM)[tid];
            V(V_G)[tid] = tid < len ? ex2f(gm) : 0.f;
            V(V_GI)[tid] = *s_safe ? ex2f(-gm) : 0.f;
            V(V_E)[tid] = tid < len ? ex2f(gC - gm) : 0.f;
            V(V_DG)[tid] = 0.f;
        }
        {
            // <dS_out, S_in> from the bf16 tiles (read before the fp32 buffers overlay them):
            // two rows per warp step, 16-byte pieces over the lanes
            float acc = 0.f;
            const int hh = (lane >> 3) & 1, c16 = lane & 7;
            for (int kk = 2 * warp + (lane >> 4); kk < D; kk += 2 * NCWARPS) {
                const uint32_t off = hh * 16384 + sw128(kk, c16 * 16);
                const uint4 a = *reinterpret_cast<const uint4 *>(sm + SM_S + off);
                const uint4 d = *reinterpret_cast<const uint4 *>(sm + SM_DS + off);
                const uint32_t au[4] = {a.x, a.y, a.z, a.w}, du[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc = fmaf(bf_lo(au[e]), bf_lo(du[e]), fmaf(bf_hi(au[e]), bf_hi(du[e]), acc));
            }
            acc = warp_sum32(acc);
            if (lane == 0) red[RED_SDS + warp] = acc;
        }
        wait(B_M1, it);
        tc_fence_after();
        BTR(it, 2);
        // ------------------------------------------------------------------ norms
        if (warp < 4) {
            float v[32];
            tld32(tmem + lrow + TM_A + 32 * q4, v);
            tmem_ld_wait();
            float dg = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) dg = (i == lane) ? v[i] : dg;
            const int r = (q4 & 1) * 32 + lane;
            const float nrm = r < len ? (g.l2norm ? rsqrtf(dg + g.eps) : 1.f) : 0.f;
            if (q4 < 2) {
                // the key row's norm, k^T k after it, the step size, Gamma n
                const float kap = dg * nrm * nrm;
                float bt = V(V_BETA)[r];
                if (g.longhorn) bt = bt / fmaf(bt, kap, 1.f);
                V(V_N)[r] = nrm;
                V(V_KAP)[r] = kap;
                V(V_B)[r] = bt;
                V(V_GN)[r] = V(V_G)[r] * nrm;
            } else {
                V(V_M)[r] = nrm;
            }
        }
        named_bar(3, NCOMPUTE);
        float sds = 0.f;   // <dS_out, S_in>
        for (int w = 0; w < NCWARPS; ++w) sds += red[RED_SDS + w];
        BTR(it, 3);
        // ------------------------------------------------------------------ first epilogues
        const float *gam = V(V_GAM);
        const bool safe = *s_safe != 0;
        // D_ri = exp(gamma_r - gamma_i) for i <= r: exp(gamma_r) exp(-gamma_i) while both stay
        // in range.  (Each loop below computes into registers and stores after the loop, so
        // that its reads of the vectors need not wait for stores through other pointers.)
        auto Dri = [&](int r, int i) { return safe ? V(V_G)[r] * V(V_GI)[i] : ex2f(gam[r] - gam[i]); };
        if (q4 < 2) {
            const int r = q4 * 32 + lane;   // chunk row (lanes 0..63)
            if (cg < 2) {
                // K^K^T o D (strict lower) and A = diag(b) (K^K^T o D), columns [32 cg, 32 cg + 32)
                float v[32];
                tld32(tmem + lrow + TM_A + 32 * cg, v);
                tmem_ld_wait();
                const float nr = V(V_N)[r], br = V(V_B)[r];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int i = 32 * cg + e;
                    v[e] = (i < r && r < len) ? nr * V(V_N)[i] * v[e] * Dri(r, i) : 0.f;
                }
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int i = 32 * cg + e;
                    *reinterpret_cast<float2 *>(fKD + r * AST + i) = make_float2(v[e], v[e + 1]);
                    *reinterpret_cast<float2 *>(fAX + r * AST + i) = make_float2(br * v[e], br * v[e + 1]);
                }
            }
        } else {
            const int r = (q4 - 2) * 32 + lane;   // lanes 64..127: Q rows of the Gram, Z rows
            if (cg < 2) {
                // P = lower(Q^ K^T o D), diagonal kept
                float v[32];
                tld32(tmem + lrow + TM_A + 32 * cg, v);
                tmem_ld_wait();
                const float mr = V(V_M)[r];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int i = 32 * cg + e;
                    v[e] = (i <= r && r < len) ? mr * V(V_N)[i] * v[e] * Dri(r, i) : 0.f;
                }
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    *reinterpret_cast<float2 *>(fG + r * AST + 32 * cg + e) = make_float2(v[e], v[e + 1]);
            } else if (warp < NCWARPS) {
                // Z = dUnew S_in^T into the Z tile (bf16 rows): warps 10 and 14 one 64-column
                // half each of lanes 64..95, warp 11 both halves of lanes 96..127
                float v[32];
                for (int hh = (q4 == 3 ? 0 : cg - 2); hh <= (q4 == 3 ? 1 : cg - 2); ++hh) {
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        tld32(tmem + lrow + TM_YZ + 64 * hh + 32 * part, v);
                        tmem_ld_wait();
                        put_row32(sm + T_Z + hh * UOD_HALF, r, 32 * part, v);
                    }
                }
            }
        }
        fence_async_smem();
        tc_fence_before();
        named_bar(3, NCOMPUTE);
        if (tid == 0) {
            // ---------------------------------------------------------- dT parts: Z K^T | dUnew V^T
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t hk = (k & 3) * 32, h24 = (k >> 2) * UOD_HALF;
                mma_bf16_ss(tmem + TM_A, dadd(dKM, T_Z + h24 + hk),
                            dadd(dKM, SM_KQ + (k >> 2) * 16384 + hk), ID_128_64, k > 0);
                mma_bf16_ss(tmem + TM_A + 64, dadd(dKM, SM_UOD + h24 + 16384 + hk),
                            dadd(dKM, SM_V + (k >> 2) * 8192 + hk), ID_128_64, k > 0);
            }
            mma_commit(&bar[B_M4]);
        }
        BTR(it, 4);
        // ------------------------------------------------------------------ dP; the inverse
        if (q4 < 2 && cg < 2) {
            const int r = q4 * 32 + lane;
            float v[32], dp1[32], dp2[32];
            tld32(tmem + lrow + TM_DP + 32 * cg, v);
            tmem_ld_wait();
            const float mr = V(V_M)[r];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int i = 32 * cg + e;
                const bool keep = i <= r && r < len;
                const float dp = keep ? sc * v[e] : 0.f;
                const float dpd = keep ? dp * Dri(r, i) : 0.f;
                v[e] = dp;
                dp1[e] = dpd * V(V_N)[i];
                dp2[e] = dpd * mr;
            }
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                // dP o P over P's row
                float2 *pp = reinterpret_cast<float2 *>(fG + r * AST + 32 * cg + e);
                const float2 pv = *pp;
                *pp = make_float2(pv.x * v[e], pv.y * v[e + 1]);
            }
            put_row32(sm + T_DP, r, 32 * cg, dp1);
            put_row32(sm + T_DP2, r, 32 * cg, dp2);
        } else if (q4 >= 2 && cg < 2) {
            // (I + A)^-1 by the four warps 2, 3, 6, 7 (named barrier 1)
            solve_unit_lower_64_packed<AST>(fAX, lane, (q4 - 2) + 2 * cg, 1);
        }
        fence_async_smem();
        named_bar(3, NCOMPUTE);
        wait(B_M4, it);
        tc_fence_after();
        BTR(it, 5);
        // ------------------------------------------------------------------ dT (and Linv's tile)
        if (q4 < 2 && cg < 2) {
            // dT = dUnew V^T - diag-scaled Z K^T; its bf16 tile dT diag(b) [r][c] for the
            // adjoint, Linv o dT for d b
            const int r = q4 * 32 + lane;
            float wv[32], uv[32], tb[32];
            tld32(tmem + lrow + TM_A + 32 * cg, wv);
            tld32(tmem + lrow + TM_A + 64 + 32 * cg, uv);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int i = 32 * cg + e;
                const float dt = (r < len && i < len) ? uv[e] - V(V_GN)[i] * wv[e] : 0.f;
                tb[e] = dt * V(V_B)[i];
                wv[e] = i <= r ? fAX[i * AST + r] * dt : 0.f;   // Linv[r][i] dT[r][i]
            }
#pragma unroll
            for (int e = 0; e < 32; e += 2)
                *reinterpret_cast<float2 *>(fTMP + r * AST + 32 * cg + e) = make_float2(wv[e], wv[e + 1]);
            put_row32(sm + T_ADJ, r, 32 * cg, tb);
        } else if (q4 >= 2 && cg < 2) {
            // Linv [r][i] (r >= i) into its bf16 tile; Linv[r][i] = AX[i][r]
            const int r = (q4 - 2) * 32 + lane;
            float x[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int i = 32 * cg + e;
                x[e] = (i <= r && r < len) ? fAX[i * AST + r] : 0.f;
            }
            put_row32(sm + T_LI, r, 32 * cg, x);
        }
        fence_async_smem();
        tc_fence_before();
        named_bar(3, NCOMPUTE);
        if (tid == 0) {
            // ---------------------------------------------------------- dQ2 = (dP o D) diag(n) K,
            // X2 = Linv^T (dT diag b)
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tmem + TM_A, dadd(dKM, T_DP + k * 32),
                            dadd(dM16, SM_KQ + k * 2048), ID_128_128_BMN, k > 0);
            mma_commit(&bar[B_M5]);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tmem + TM_ADJ, dadd(dM8, T_LI + k * 2048),
                            dadd(dM8, T_ADJ + k * 2048), ID_128_64_ABMN, k > 0);
            mma_commit(&bar[B_X2]);
        }
        BTR(it, 6);
        for (int i = warp; i < C; i += NCWARPS) {
            // d b through T = Linv diag(b): column sums of Linv o dT
            float a = fTMP[lane * AST + i] + fTMP[(lane + 32) * AST + i];
            a = warp_sum32(a);
            if (lane == 0) V(V_DB)[i] = a;
        }
        wait(B_X2, it);
        tc_fence_after();
        if (q4 < 2) {
            // X2 rows (bf16) over dT's tile, the A operand of dA' = X2 Linv^T
            const int a = q4 * 32 + lane;
            float x[16];
            tld16(tmem + lrow + TM_ADJ + 16 * cg, x);
            tmem_ld_wait();
            put_row16(sm + T_ADJ, a, 16 * cg, x);
        }
        fence_async_smem();
        tc_fence_before();
        named_bar(3, NCOMPUTE);
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tmem + TM_ADJ + 64, dadd(dKM, T_ADJ + k * 32),
                            dadd(dKM, T_LI + k * 32), ID_128_64, k > 0);
            mma_commit(&bar[B_DA]);
        }
        BTR(it, 7);
        // ------------------------------------------------------------------ dq (while dA' runs)
        wait(B_M5, it);
        tc_fence_after();
        if (q4 < 2) {
            const int r = q4 * 32 + lane;
            float y[32], q2[32], qx[32];
            tld32(tmem + lrow + TM_YZ + 32 * cg, y);
            tld32(tmem + lrow + TM_A + 32 * cg, q2);
            row32(sm + SM_KQ + 8192, 16384, r, 32 * cg, qx);
            tmem_ld_wait();
            const float sg = sc * V(V_G)[r], mr = V(V_M)[r];
            float pq = 0.f, qy = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                qy = fmaf(qx[e], y[e], qy);     // <Q_r, Y_r> (raw Q) for d gamma
                y[e] = fmaf(sg, y[e], q2[e]);   // dQ^
                pq = fmaf(qx[e] * mr, y[e], pq);
            }
            red[RED_QT + cg * 64 + r] = qy;
            red[cg * 64 + r] = pq;
            named_bar(2, 256);
            pq = red[r] + red[64 + r] + red[128 + r] + red[192 + r];
            // dq row r, columns [32 cg, 32 cg + 32), into its staged tile
            if (g.l2norm) {
#pragma unroll
                for (int e = 0; e < 32; ++e) y[e] = mr * (y[e] - qx[e] * mr * pq);
            }
            put_row32(sm + T_DQ + (cg >> 1) * 8192, r, 32 * (cg & 1), y);
            fence_async_smem();
        }
        wait(B_DA, it);
        tc_fence_after();
        BTR(it, 8);
        // F = dA o K^K^T o D (d b, row sums), E = b_r F + dP o P (d gamma, row minus column
        // sums), dKK = dA o b_r o D; dA = strict_lower(-X2 Linv^T) read from the tensor memory
        if (q4 < 2) {
            const int a = q4 * 32 + lane;
            float x[16];
            tld16(tmem + lrow + TM_ADJ + 64 + 16 * cg, x);
            tmem_ld_wait();
            const float ba = V(V_B)[a];
            float kdI[16], gI[16];
            rowN(fKD + a * AST + 16 * cg, kdI);
            rowN(fG + a * AST + 16 * cg, gI);
            float db = 0.f, rs = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int bb = 16 * cg + e;
                const bool lower = bb < a && a < len;
                const float dA = lower ? -x[e] : 0.f;
                const float f = dA * kdI[e];
                const float ev = fmaf(ba, f, gI[e]);
                db += f;
                rs += ev;
                gI[e] = ev;
                // masked, not multiplied by zero: above the diagonal exp(gamma_a - gamma_b)
                // overflows once the gates leave the factored range
                kdI[e] = lower ? dA * ba * Dri(a, bb) : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                *reinterpret_cast<float2 *>(fG + a * AST + 16 * cg + e) = make_float2(gI[e], gI[e + 1]);
                *reinterpret_cast<float2 *>(fKD + a * AST + 16 * cg + e) = make_float2(kdI[e], kdI[e + 1]);
            }
            // a region of their own: the dq epilogue's partials may still be being read
            red[RED_FE + cg * 64 + a] = db;
            red[RED_FE + 256 + cg * 64 + a] = rs;
        }
        tc_fence_before();
        named_bar(3, NCOMPUTE);
        store_tile(&tm_dq, T_DQ, p.dq, row, len);
        if (tid < 64) {
            const float *rf = red + RED_FE;
            V(V_DB)[tid] += rf[tid] + rf[64 + tid] + rf[128 + tid] + rf[192 + tid];
            V(V_DG)[tid] += rf[256 + tid] + rf[320 + tid] + rf[384 + tid] + rf[448 + tid];
        }
        for (int i = warp; i < C; i += NCWARPS) {
            float cs = fG[lane * AST + i] + fG[(lane + 32) * AST + i];
            cs = warp_sum32(cs);
            if (lane == 0) V(V_CS)[i] = cs;
        }
        // (dKK + dKK^T) n_r [i][r] into its bf16 tile (rows i), over X2's
        if (warp >= 8 && warp < 12) {
            const int i = (warp - 8) * 16 + (lane >> 1), c0 = (lane & 1) * 32;
            float x[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int r = c0 + e;
                x[e] = (fKD[i * AST + r] + fKD[r * AST + i]) * V(V_N)[r];
            }
            put_row32(sm + T_ADJ, i, c0, x);
        }
        fence_async_smem();
        tc_fence_before();
        named_bar(3, NCOMPUTE);
        BTR(it, 9);
        if (tid < 64) V(V_DG)[tid] -= V(V_CS)[tid];
        if (tid == 0) mbar_arrive(&bar[B_SDSFREE]);   // the fp32 buffers over the states are no longer read
        if (tid == 0) {
            // ---------------------------------------------------------- dK, T^T dW, T^T dUnew
            tc_fence_after();
            const uint64_t dK = dadd(dM16, SM_KQ), dQ = dadd(dM16, SM_KQ + 8192);
            const uint64_t dP2 = dadd(dM8, T_DP2), dLI = dadd(dM8, T_LI);
            const uint64_t dZ = dadd(dMU, T_Z), dU = dadd(dMU, SM_UOD + 16384);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tmem + TM_A, dadd(dP2, k * 2048), dadd(dQ, k * 2048), ID_128_128_ABMN, k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tmem + TM_A, dadd(dKM, T_ADJ + k * 32), dadd(dK, k * 2048), ID_128_128_BMN, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tmem + TM_YZ, dadd(dLI, k * 2048), dadd(dZ, k * 2048), ID_128_128_ABMN, k > 0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ss(tmem + TM_DP, dadd(dLI, k * 2048), dadd(dU, k * 2048), ID_128_128_ABMN, k > 0);
            mma_commit(&bar[B_M6]);
        }
        wait(B_M6, it);
        tc_fence_after();
        BTR(it, 10);
        // ------------------------------------------------------------------ dk, dv, d beta, dg
        if (q4 < 2) {
            const int i = q4 * 32 + lane;
            float gz[32], ka[32], xv[32], kx[32];
            tld32(tmem + lrow + TM_YZ + 32 * cg, gz);
            tld32(tmem + lrow + TM_A + 32 * cg, ka);
            tld32(tmem + lrow + TM_X + 32 * cg, xv);
            row32(sm + SM_KQ, 16384, i, 32 * cg, kx);
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_KQFREE]);   // this task's K rows have been read
            tmem_ld_wait();
            BTR(it, 13);
            const float bi = V(V_B)[i], gi = V(V_G)[i], ei = V(V_E)[i], ni = V(V_N)[i];
            float k2 = 0.f, pk = 0.f, kxs = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) kxs = fmaf(kx[e], xv[e], kxs);   // <K_r, X_r> (raw K) for d gamma
            red[RED_SE + cg * 64 + i] = kxs;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float kh = kx[e] * ni;            // K^
                const float dgk = -bi * gz[e];          // b_i (Linv^T dW)_i, dW = -Z
                k2 = fmaf(dgk, kh, k2);
                ka[e] = fmaf(gi, dgk, fmaf(ei, xv[e], ka[e]));   // dK^
                pk = fmaf(kh, ka[e], pk);
            }
            red[cg * 64 + i] = k2;
            red[256 + cg * 64 + i] = pk;
            float dvv[32];
            tld32(tmem + lrow + TM_DP + 32 * cg, dvv);
            tmem_ld_wait();
            BTR(it, 14);
            named_bar(2, 256);
            BTR(it, 15);
            k2 = red[i] + red[64 + i] + red[128 + i] + red[192 + i];
            pk = red[256 + i] + red[320 + i] + red[384 + i] + red[448 + i];
            if (cg == 0) V(V_K2)[i] = k2;
            // Longhorn's step e = b / (1 + b kap): de/db = (1 - e kap)^2, de/dkap = -e^2, dkap/dk = 2 k^
            float dkap = 0.f;
            if (g.longhorn) {
                const float kap = V(V_KAP)[i], db = V(V_DB)[i];
                dkap = -db * bi * bi;
                pk = fmaf(2.f * dkap, kap, pk);
            }
            // dk and dv rows i, columns [32 cg, 32 cg + 32), into their staged tiles
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                float c = fmaf(2.f * dkap, kx[e] * ni, ka[e]);
                if (g.l2norm) c = ni * (c - kx[e] * ni * pk);
                ka[e] = c;
                dvv[e] *= bi;
            }
            put_row32(sm + T_DK + (cg >> 1) * 8192, i, 32 * (cg & 1), ka);
            put_row32(sm + T_DV + (cg >> 1) * 8192, i, 32 * (cg & 1), dvv);
            fence_async_smem();
        }
        tc_fence_before();
        named_bar(3, NCOMPUTE);
        BTR(it, 11);
        store_tile(&tm_dk, T_DK, p.dk, row, len);
        store_tile(&tm_dv, T_DV, p.dv, row, len);
        if (warp == 0) {
            // d gamma, its reverse cumulative sum within the chunk (dg), and d beta
            const int r0 = lane, r1 = lane + 32;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = lane + 32 * hh;
                const float *qt = red + RED_QT, *se = red + RED_SE;
                V(V_QT)[r] = sc * V(V_G)[r] * V(V_M)[r] * (qt[r] + qt[64 + r] + qt[128 + r] + qt[192 + r]);
                V(V_SE)[r] = V(V_E)[r] * V(V_N)[r] * (se[r] + se[64 + r] + se[128 + r] + se[192 + r]);
            }
            __syncwarp();
            auto dgam = [&](int r) {
                return r < len ? V(V_QT)[r] + V(V_DG)[r] + V(V_G)[r] * V(V_K2)[r] - V(V_SE)[r] : 0.f;
            };
            float s0 = dgam(r0), s1 = dgam(r1);
            float se = (r0 < len ? V(V_SE)[r0] : 0.f) + (r1 < len ? V(V_SE)[r1] : 0.f);
            se = warp_sum32(se);
            const float extra = se + ex2f(gC) * sds;
            if (r0 == len - 1) s0 += extra;
            if (r1 == len - 1) s1 += extra;
            // reverse inclusive scan over 64 rows: rows 32..63 first, then their total onto 0..31
            float t1 = s1, t0 = s0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float a1 = __shfl_down_sync(0xffffffffu, t1, o), a0 = __shfl_down_sync(0xffffffffu, t0, o);
                if (lane + o < 32) { t1 += a1; t0 += a0; }
            }
            t0 += __shfl_sync(0xffffffffu, t1, 0);
            if (p.dg) {
                if (r0 < len) p.dg[row + r0] = t0;
                if (r1 < len) p.dg[row + r1] = t1;
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = lane + 32 * hh;
                if (r >= len) continue;
                float db = V(V_DB)[r];
                if (g.longhorn) {
                    const float ee = V(V_B)[r], f = fmaf(-ee, V(V_KAP)[r], 1.f);
                    db *= f * f;
                }
                p.dbeta[row + r] = __float2bfloat16_rn(db);
            }
        }
        named_bar(3, NCOMPUTE);   // the vectors are rewritten by the next task
        BTR(it, 12);
        ++it;
        t = tnext;
        if (*s_abort) break;
    }
    }   // compute warps
    // drain: nothing of this CTA may still be in flight when it exits (the producer waited
    // for its copies above)
    if (tid == 0) {
        bulk_wait_all();   // the tensor stores of the last task
        if (mma_issued) {
            mma_commit(&bar[B_DRAIN]);
            mbar_wait(&bar[B_DRAIN], 0, BUDGET, nullptr);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ================================================================================= host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    return fn;
}

// a [rows][128] bf16 array read in 64 x 64 boxes with the 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, long long rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)(rows > 0 ? rows : 1)};
    cuuint64_t gstr[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), gdim, gstr, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool supports(const Geo &g, int dtype)
{
    return dtype == DN_BF16 && g.dk == D && g.dv == D && g.C == C && encode_fn() != nullptr;
}

cudaError_t grads(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                  const __nv_bfloat16 *beta, const float *gate, const __nv_bfloat16 *dO,
                  const __nv_bfloat16 *Sin, const __nv_bfloat16 *dSo, const __nv_bfloat16 *Un,
                  const __nv_bfloat16 *dUn, __nv_bfloat16 *dq, __nv_bfloat16 *dk, __nv_bfloat16 *dv,
                  __nv_bfloat16 *dbeta, float *dg, cudaStream_t st)
{
    const int ntasks = g.NC * g.H;
    if (ntasks == 0 || g.T == 0) return cudaSuccess;
    const long long rows = (long long)g.B * g.H * g.T;
    const long long slots = (long long)g.NC * g.H;
    CUtensorMap mq, mk, mv, mo, ms, mds, mu, mdu, mgq, mgk, mgv;
    if (!make_map(&mq, q, rows) || !make_map(&mk, k, rows) || !make_map(&mv, v, rows) ||
        !make_map(&mo, dO, rows) || !make_map(&ms, Sin, slots * D) || !make_map(&mds, dSo, slots * D) ||
        !make_map(&mu, Un, slots * C) || !make_map(&mdu, dUn, slots * C) || !make_map(&mgq, dq, rows) ||
        !make_map(&mgk, dk, rows) || !make_map(&mgv, dv, rows))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k_bwd_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES)) !=
        cudaSuccess)
        return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    Params p;
    p.g = g; p.beta = beta; p.gate = gate; p.dq = dq; p.dk = dk; p.dv = dv; p.dbeta = dbeta; p.dg = dg;
    p.ntasks = ntasks;
    const int grid = ntasks < sms ? ntasks : sms;
    k_bwd_tc<<<grid, NTHREADS, SMEM_BYTES, st>>>(mq, mk, mv, mo, ms, mds, mu, mdu, mgq, mgk, mgv, p);
    return cudaPeekAtLastError();
}

}  // namespace btc
}  // namespace gdn
