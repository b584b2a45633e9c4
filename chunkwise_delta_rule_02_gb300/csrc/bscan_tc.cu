// Reverse dS scan of the backward on tcgen05 (bf16, d_k = d_v = 128, C = 64).
//
// Per (sequence, head) item, from its last chunk to its first, with dS resident in
// TMEM as dS^T (lane = d_v column, column = d_k) under a pending scale G (dS = G dS^,
// renormalised when G < 2^-30), and every operand tile in the 128-byte swizzle:
//   dS_out          = G dS^                                  (bf16 snapshot: operand and output)
//   [A1 | A2]       = (dO^T P | dS_out^T K^T)                (12 MMAs, N = 64)
//   dUnew^T         = scale A1 + A2 diag(f)                  (epilogue; output)
//   dS^            += (scale dO / G')^T Qt + (dUnew / G')^T (-W),  G' = G exp(gamma_C)   (8 MMAs, N = 128)
// (the chunk-form gradients of "Parallelizing Linear Transformers with the Delta
// Rule over Sequence Length", with the gates of "Gated DeltaNet" as within-chunk
// cumulative log-decays: dUnew = P^T dO + K~ dS, dS <- Gamma_C dS + (Gamma Q)^T dO -
// W^T dUnew, K~ = diag(f) K, f = exp(gamma_C - gamma) n.)  The packages -- [-W | Qt]
// panels, P and the vector (f, exp(gamma_C)) -- are the cooperative forward's, copied
// from the workspace as they are; K and dO come by TMA.  One CTA per item (a CTA takes
// items b, b + grid, ...); every wait is bounded and reports a timeout through the
// status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>

#include "bscan_tc.h"
#include "sm100.cuh"

namespace gdn {
namespace bsc {
using namespace sm100;

namespace {

constexpr int C = 64;
constexpr int D = 128;
constexpr int NTHREADS = 512;
constexpr long long BUDGET = 4000000000LL;              // clock cycles (about 2 s)
constexpr float RENORM_BELOW = 9.313225746154785e-10f;   // 2^-30

constexpr uint32_t PANEL = C * 128;          // one 64-column panel of a chunk's rows
constexpr uint32_t WQ = 4 * PANEL;           // [-W | Qt] panels (2 x [C rows -W | C rows Qt])
constexpr uint32_t WQP = 2 * PANEL;          // one [-W | Qt] panel
constexpr uint32_t VEC_BYTES = 272;          // f[64], exp(gamma_C), padding
// one chunk's copies in shared memory: [-W | Qt] panels, P, the vector
constexpr uint32_t PK_P = WQ;
constexpr uint32_t PK_VEC = PK_P + PANEL;
constexpr uint32_t PKS = (PK_VEC + VEC_BYTES + 1023u) & ~1023u;
constexpr uint32_t TILE = 2 * PANEL;         // a C x 128 bf16 tile (K, dO)

constexpr uint32_t SM_PK = 0;                          // 2 package copies
constexpr uint32_t SM_K = SM_PK + 2 * PKS;             // 2 K tiles [token][d_k]
constexpr uint32_t SM_DO = SM_K + 2 * TILE;            // 2 dO tiles [token][d_v]
constexpr uint32_t SM_DOS = SM_DO + 2 * TILE;          // scale dO / G', same layout
constexpr uint32_t SM_SB = SM_DOS + TILE;              // dS_out^T bf16 [d_v][d_k] (2 panels of 128 rows)
constexpr uint32_t SM_US = SM_SB + 32768;              // (dUnew / G')^T bf16 [d_v][token]
constexpr uint32_t SM_BAR = SM_US + 16384;
constexpr uint32_t SM_END = SM_BAR + 32 * 8 + 64;
constexpr uint32_t SMEM_BYTES = SM_END + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

constexpr uint32_t TM_S = 0;      // dS^T fp32, 128 columns
constexpr uint32_t TM_A = 128;    // [A1 (64) | A2 (64)] for two chunks

enum { B_FULL = 0, B_EMPTY = 2, B_SNAP = 4, B_A = 5, B_DOSC = 7, B_U2 = 8, B_S = 9, B_ABORTED = 10, NBAR = 11 };

constexpr uint32_t ID_A1 = idesc(1, 128, C, true, true);      // dO^T P
constexpr uint32_t ID_A2 = idesc(1, 128, C, false, false);    // dS_out^T K^T
constexpr uint32_t ID_U1 = idesc(1, 128, 128, true, true);    // (scale dO / G')^T Qt
constexpr uint32_t ID_U2 = idesc(1, 128, 128, false, true);   // (dUnew / G')^T (-W)

struct Params {
    const float *dhT;
    float *dh0;
    const uint8_t *keep;
    uint32_t pk_stride, pk_wq, pk_p, pk_vec;
    __nv_bfloat16 *dSo, *dUn;
    const int32_t *cu, *cstart;
    uint32_t *status;
    int H, T, N, items, nchs;
    float scale;
};

__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

struct Item {
    int seq, h, L, nch, j0;
    long long rowbase;
};

__device__ __forceinline__ Item item_of(const Params &p, int it)
{
    Item r;
    r.h = it % p.H;
    r.seq = it / p.H;
    if (p.cu) {
        int t0 = p.cu[r.seq], t1 = p.cu[r.seq + 1];
        if (t0 < 0 || t1 < t0 || t1 > p.T) t0 = t1 = 0;   // malformed offsets: empty (flagged elsewhere)
        r.L = t1 - t0;
        r.rowbase = (long long)r.h * p.T + t0;
        r.j0 = p.cstart[r.seq];
    } else {
        r.L = p.T;
        r.rowbase = ((long long)r.seq * p.H + r.h) * p.T;
        r.j0 = r.seq * p.nchs;
    }
    r.nch = (r.L + C - 1) / C;
    return r;
}

// The chunks of a CTA's items b, b + grid, ..., each item from its last chunk to its first.
struct RStream {
    int it, c;
    Item cur;
    bool valid;
    __device__ void start(const Params &p)
    {
        it = (int)blockIdx.x - (int)gridDim.x;
        advance_item(p);
    }
    __device__ void advance_item(const Params &p)
    {
        while (true) {
            it += gridDim.x;
            if (it >= p.items) { valid = false; return; }
            cur = item_of(p, it);
            if (cur.nch > 0) break;
        }
        c = cur.nch - 1;
        valid = true;
    }
    __device__ void next(const Params &p)
    {
        if (--c < 0) advance_item(p);
    }
    __device__ bool first() const { return c == cur.nch - 1; }   // the first one processed
    __device__ bool last() const { return c == 0; }
    __device__ int len() const { return min(C, cur.L - c * C); }
    __device__ int row0() const { return (int)(cur.rowbase + (long long)c * C); }
    __device__ size_t slot(const Params &p) const { return (size_t)(cur.j0 + c) * p.H + cur.h; }
    __device__ size_t sidx(const Params &p) const { return ((size_t)cur.seq * p.H + cur.h) * D * D; }
};

__device__ __forceinline__ int stream_length(const Params &p)
{
    int J = 0;
    for (int it = blockIdx.x; it < p.items; it += gridDim.x) J += item_of(p, it).nch;
    return J;
}

}  // namespace

__global__ void __launch_bounds__(NTHREADS, 1)
k_bscan_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_do, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    uint64_t *bar = (uint64_t *)(sm + SM_BAR);
    volatile int *abort_flag = (volatile int *)(sm + SM_BAR + 32 * 8);
    uint32_t *tmem_slot = (uint32_t *)(sm + SM_BAR + 32 * 8 + 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr unsigned FULL = 0xffffffffu;

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == B_SNAP || i == B_U2) cnt = 8;   // warps 4-11
            if (i == B_DOSC) cnt = 4;                // warps 12-15
            mbar_init(&bar[i], cnt);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_do);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int J = stream_length(p);

    auto fail = [&]() {
        if (!*abort_flag) {
            *abort_flag = 1;
            raise_status(p.status, kStatusTimeout);
        }
    };
    auto wait = [&](int b, uint32_t k) -> bool {
        if (mbar_wait(&bar[b], k & 1u, BUDGET, abort_flag)) return true;
        fail();
        return false;
    };

    if (warp == 0) {
        // ---------------------------------------------------------------- copies in
        if (lane == 0) {
            RStream st, ahead;
            st.start(p);
            ahead.start(p);
            for (int a = 0; a < 2 && ahead.valid; ++a) ahead.next(p);
            int issued = 0;
            for (int j = 0; j < J && st.valid; ++j, st.next(p)) {
                const int s = j & 1;
                if (ahead.valid) {
                    // K and dO of chunk j + 2 into L2
                    const int ra = ahead.row0();
                    tma_prefetch_2d(&tm_k, 0, ra);
                    tma_prefetch_2d(&tm_k, 64, ra);
                    tma_prefetch_2d(&tm_do, 0, ra);
                    tma_prefetch_2d(&tm_do, 64, ra);
                    ahead.next(p);
                }
                if (j >= 2 && !wait(B_EMPTY + s, (uint32_t)((j >> 1) - 1))) break;
                const uint8_t *src = p.keep + st.slot(p) * p.pk_stride;
                uint8_t *pk = sm + SM_PK + s * PKS;
                const int row = st.row0();
                mbar_expect_tx(&bar[B_FULL + s], WQ + PANEL + VEC_BYTES + 2 * TILE);
                bulk_load(pk, src + p.pk_wq, WQ, &bar[B_FULL + s]);
                bulk_load(pk + PK_P, src + p.pk_p, PANEL, &bar[B_FULL + s]);
                bulk_load(pk + PK_VEC, src + p.pk_vec, VEC_BYTES, &bar[B_FULL + s]);
                tma_load_2d(sm + SM_K + s * TILE, &tm_k, &bar[B_FULL + s], 0, row);
                tma_load_2d(sm + SM_K + s * TILE + PANEL, &tm_k, &bar[B_FULL + s], 64, row);
                tma_load_2d(sm + SM_DO + s * TILE, &tm_do, &bar[B_FULL + s], 0, row);
                tma_load_2d(sm + SM_DO + s * TILE + PANEL, &tm_do, &bar[B_FULL + s], 64, row);
                issued = j + 1;
            }
            // the last copies issued into each buffer have landed before shared memory goes away
            for (int jj = (issued > 2 ? issued - 2 : 0); jj < issued; ++jj)
                mbar_wait(&bar[B_FULL + (jj & 1)], (uint32_t)(jj >> 1) & 1u, BUDGET, nullptr);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && J > 0) {
            const uint64_t dSB = sdesc(sb + SM_SB, 16, 1024);
            const uint64_t dUS = sdesc(sb + SM_US, 16, 1024);
            const uint64_t dDOS = sdesc(sb + SM_DOS, PANEL, 1024);
            const uint64_t dPK0 = sdesc(sb + SM_PK, WQP, 1024);       // -W rows, MN-major (N = d_k)
            const uint64_t dP0 = sdesc(sb + SM_PK + PK_P, PANEL, 1024);
            const uint64_t dK0 = sdesc(sb + SM_K, 16, 1024);          // K rows, K-major
            const uint64_t dDO0 = sdesc(sb + SM_DO, PANEL, 1024);     // dO^T, MN-major (M = d_v)
            auto a1 = [&](int j) -> bool {
                // A1 = dO^T P into the first half of chunk j's accumulator pair
                const int s = j & 1;
                if (!wait(B_FULL + s, (uint32_t)(j >> 1))) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    mma_bf16_ss(tmem + TM_A + s * 128, dadd(dadd(dDO0, s * TILE), k * 2048),
                                dadd(dadd(dP0, s * PKS), k * 2048), ID_A1, k > 0);
                return true;
            };
            bool ok = a1(0);
            for (int j = 0; j < J && ok; ++j) {
                const int s = j & 1;
                // A2 = dS_out^T K^T once the snapshot is in shared memory
                if (!(ok = wait(B_SNAP, (uint32_t)j))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16_ss(tmem + TM_A + s * 128 + C, dadd(dSB, (k >> 2) * 16384 + (k & 3) * 32),
                                dadd(dadd(dK0, s * TILE), (k >> 2) * PANEL + (k & 3) * 32), ID_A2, k > 0);
                mma_commit(&bar[B_A + s]);
                // dS^ += (scale dO / G')^T Qt
                if (!(ok = wait(B_DOSC, (uint32_t)j))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    mma_bf16_ss(tmem + TM_S, dadd(dDOS, k * 2048), dadd(dadd(dPK0, s * PKS), PANEL + k * 2048),
                                ID_U1, 1);
                // dS^ += (dUnew / G')^T (-W) once the epilogue has written it
                if (!(ok = wait(B_U2, (uint32_t)j))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    mma_bf16_ss(tmem + TM_S, dadd(dUS, k * 32), dadd(dadd(dPK0, s * PKS), k * 2048), ID_U2, 1);
                mma_commit(&bar[B_S]);
                mma_commit(&bar[B_EMPTY + s]);
                if (j + 1 < J) ok = a1(j + 1);
            }
            mma_commit(&bar[B_ABORTED]);
            mbar_wait(&bar[B_ABORTED], 0, BUDGET, nullptr);
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------- dS snapshot and the dUnew epilogue
        // warpgroup `half`: d_k columns [64 half, 64 half + 64) of the snapshot, tokens
        // [32 half, 32 half + 32) of the epilogue; TMEM lane = d_v column
        const int half = (warp >> 2) - 1;
        const int dv = (warp & 3) * 32 + lane;
        const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
        // items without chunks: dh0 = dhT
        if (p.dh0) {
            for (int it = blockIdx.x; it < p.items; it += gridDim.x) {
                const Item I = item_of(p, it);
                if (I.nch == 0) {
                    const size_t sidx = ((size_t)I.seq * p.H + I.h) * D * D;
                    for (int kk = 64 * half; kk < 64 * half + 64; ++kk)
                        p.dh0[sidx + (size_t)kk * D + dv] = p.dhT ? p.dhT[sidx + (size_t)kk * D + dv] : 0.f;
                }
            }
        }
        RStream st;
        st.start(p);
        float G = 1.f;
        for (int j = 0; j < J && st.valid; ++j) {
            const int s = j & 1;
            const size_t slot = st.slot(p), sidx = st.sidx(p);
            if (st.first()) {
                // dS^T = dhT^T of the item, scale 1
                G = 1.f;
                for (int k0 = 64 * half; k0 < 64 * half + 64; k0 += 32) {
                    uint32_t r[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        r[k] = __float_as_uint(p.dhT ? p.dhT[sidx + (size_t)(k0 + k) * D + dv] : 0.f);
                    tmem_st32(tmem + lrow + TM_S + k0, r);
                }
                tmem_st_wait();
            } else if (!__all_sync(FULL, wait(B_S, (uint32_t)(j - 1)))) {
                break;
            }
            if (!__all_sync(FULL, wait(B_FULL + s, (uint32_t)(j >> 1)))) break;
            tc_fence_after();
            const float *vec = (const float *)(sm + SM_PK + s * PKS + PK_VEC);
            const float Gn = G, Gnext = Gn * vec[64];
            const bool renorm = Gnext < RENORM_BELOW;
            const float fdiv = renorm ? 1.f : 1.f / Gnext;
            G = renorm ? 1.f : Gnext;
            {
                // dS_out = Gn dS^: bf16 operand (this warpgroup's panel) and output [d_k][d_v];
                // a tiny Gnext also rescales dS^
                uint32_t r[64];
                tmem_ld32(tmem + lrow + TM_S + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                tmem_ld32(tmem + lrow + TM_S + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                tmem_ld_wait();
                uint8_t *sbp = sm + SM_SB + half * 16384;
                uint16_t *out = reinterpret_cast<uint16_t *>(p.dSo) + slot * D * D + dv;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16(Gn * __uint_as_float(r[c8 * 8 + 2 * e]), Gn * __uint_as_float(r[c8 * 8 + 2 * e + 1]));
                    *(uint4 *)(sbp + sw128(dv, c8 * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                    const int k0 = 64 * half + c8 * 8;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        out[(size_t)(k0 + 2 * e) * D] = (uint16_t)(w[e] & 0xFFFFu);
                        out[(size_t)(k0 + 2 * e + 1) * D] = (uint16_t)(w[e] >> 16);
                    }
                }
                if (renorm) {
#pragma unroll
                    for (int e = 0; e < 64; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * Gnext);
                    tmem_st32(tmem + lrow + TM_S + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                    tmem_st32(tmem + lrow + TM_S + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                    tmem_st_wait();
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_SNAP]);
            // dUnew = scale A1 + A2 diag(f): output (rows past the chunk's end zero) and
            // (dUnew / G')^T for the state update
            if (!__all_sync(FULL, wait(B_A + s, (uint32_t)(j >> 1)))) break;
            tc_fence_after();
            {
                uint32_t x1[32], x2[32];
                tmem_ld32(tmem + lrow + TM_A + s * 128 + 32 * half, x1);
                tmem_ld32(tmem + lrow + TM_A + s * 128 + C + 32 * half, x2);
                tmem_ld_wait();
                const int len = st.len();
                const float *f = vec + 32 * half;
                uint16_t *du = reinterpret_cast<uint16_t *>(p.dUn) + (slot * C + 32 * half) * D + dv;
                uint8_t *us = sm + SM_US;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint32_t wo[4], ws[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = c8 * 8 + 2 * e;
                        const bool l0 = 32 * half + i0 < len, l1 = 32 * half + i0 + 1 < len;
                        const float u0 = l0 ? fmaf(p.scale, __uint_as_float(x1[i0]), f[i0] * __uint_as_float(x2[i0])) : 0.f;
                        const float u1 = l1 ? fmaf(p.scale, __uint_as_float(x1[i0 + 1]), f[i0 + 1] * __uint_as_float(x2[i0 + 1])) : 0.f;
                        wo[e] = pack_bf16(u0, u1);
                        ws[e] = pack_bf16(u0 * fdiv, u1 * fdiv);
                        du[(size_t)i0 * D] = (uint16_t)(wo[e] & 0xFFFFu);
                        du[(size_t)(i0 + 1) * D] = (uint16_t)(wo[e] >> 16);
                    }
                    *(uint4 *)(us + sw128(dv, (4 * half + c8) * 16)) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_U2]);
            if (st.last()) {
                // dh0 = G dS^ once the item's first chunk has been folded in
                if (!__all_sync(FULL, wait(B_S, (uint32_t)j))) break;
                tc_fence_after();
                if (p.dh0 && !*abort_flag) {
                    for (int k0 = 64 * half; k0 < 64 * half + 64; k0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lrow + TM_S + k0, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k) p.dh0[sidx + (size_t)(k0 + k) * D + dv] = G * __uint_as_float(r[k]);
                    }
                }
            }
            st.next(p);
            if (__any_sync(FULL, *abort_flag != 0)) break;
        }
    } else if (warp >= 12) {
        // ------------------------------------------------- scale dO / G' (operand of the update)
        const int t = tid - 384;
        RStream st;
        st.start(p);
        float G = 1.f;
        for (int j = 0; j < J && st.valid; ++j, st.next(p)) {
            const int s = j & 1;
            if (st.first()) G = 1.f;
            if (!__all_sync(FULL, wait(B_FULL + s, (uint32_t)(j >> 1)))) break;
            const float *vec = (const float *)(sm + SM_PK + s * PKS + PK_VEC);
            const float Gnext = G * vec[64];
            const bool renorm = Gnext < RENORM_BELOW;
            const float fs = renorm ? p.scale : p.scale / Gnext;
            G = renorm ? 1.f : Gnext;
            // the previous chunk's update has read the buffer
            if (j >= 1 && !__all_sync(FULL, wait(B_S, (uint32_t)(j - 1)))) break;
            const uint8_t *src = sm + SM_DO + s * TILE;
            uint8_t *dst = sm + SM_DOS;
#pragma unroll
            for (int u = 0; u < (int)(TILE / 16) / 128; ++u) {
                const uint32_t off = (uint32_t)(u * 128 + t) * 16;
                const uint4 a = *(const uint4 *)(src + off);
                const uint32_t wv[4] = {a.x, a.y, a.z, a.w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    o[q] = pack_bf16(fs * __uint_as_float(wv[q] << 16), fs * __uint_as_float(wv[q] & 0xFFFF0000u));
                *(uint4 *)(dst + off) = make_uint4(o[0], o[1], o[2], o[3]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_DOSC]);
            if (__any_sync(FULL, *abort_flag != 0)) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================================================= host
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

// bf16 [rows][128], boxes of 64 columns x 64 rows, 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, long long rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t gstr[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)C};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), gdim, gstr, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

bool supports(const Geo &g, int dtype)
{
    return dtype == DN_BF16 && g.dk == D && g.dv == D && g.C == C &&
           (long long)g.B * g.H * (long long)g.T < (1LL << 31) && encode_fn() != nullptr;
}

cudaError_t scan(const Geo &g, const __nv_bfloat16 *k, const __nv_bfloat16 *dO, const float *dhT,
                 float *dh0, const uint8_t *keep, const coop::PkLayout &pk, __nv_bfloat16 *dSo,
                 __nv_bfloat16 *dUn, cudaStream_t st)
{
    const int items = g.N * g.H;
    if (items == 0) return cudaSuccess;
    if (g.varlen && !g.cstart) return cudaErrorInvalidValue;
    const int sms = num_sms();
    if (sms < 1) return cudaErrorNotSupported;
    Params p;
    p.dhT = dhT; p.dh0 = dh0; p.keep = keep;
    p.pk_stride = pk.stride; p.pk_wq = pk.wq; p.pk_p = pk.p; p.pk_vec = pk.vec;
    p.dSo = dSo; p.dUn = dUn;
    p.cu = g.varlen ? g.cu : nullptr;
    p.cstart = g.varlen ? g.cstart : nullptr;
    p.status = g.status;
    p.H = g.H; p.T = g.T; p.N = g.N; p.items = items; p.nchs = (g.T + C - 1) / C;
    p.scale = g.scale;
    const long long rows = (long long)g.B * g.H * g.T;
    CUtensorMap mk, mdo;
    const long long maprows = rows > 0 ? rows : 1;
    if (!make_map(&mk, k, maprows) || !make_map(&mdo, dO, maprows)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_bscan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int grid = items < sms ? items : sms;
    k_bscan_tc<<<grid, NTHREADS, SMEM_BYTES, st>>>(mk, mdo, p);
    return cudaPeekAtLastError();
}

}  // namespace bsc
}  // namespace gdn
