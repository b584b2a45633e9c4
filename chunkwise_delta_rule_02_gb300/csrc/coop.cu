// Cooperative persistent forward of the (gated) delta rule for bf16 inputs with
// d_k = d_v, one launch whose CTAs take one of two roles.  Instances: chunk C = 64
// with d = 128, and C = 32 with d = 128 or 256 (at d = 256 and C = 64 one chunk's
// operand tiles do not fit a CTA's shared memory).
//
//   preparation CTAs (four independent pipelines each): for a chunk, compute
//     everything that does not depend on the state -- norms, gates, the Gram and
//     Q K^T masks, the UT transform T = (I + A)^-1 diag(beta), T' = T diag(exp(gamma) n),
//     -W = -T' K, Qt = diag(exp(gamma) m) Q, P = lower(Q K^T o D) with the norms --
//     and publish them as one package into an L2-resident ring slot of the chain
//     CTAs that own the chunk;
//   chain CTAs (one per SM, persistent over their (sequence, head) items; at
//     d_v = 256 two of them per item, each owning 128 of its d_v columns and
//     reading the same packages): keep the state in TMEM and run, per chunk, only
//       U^T            = V^T T^T                       (tcgen05 MMAs, K = C)
//       [Unew^T | O^T] += S^T [-W | Qt]^T              (shared-memory operands, N = 2C, K = d_k)
//       S_hat^T        += (f o Unew)^T K               (N = d_k, K = C)
//       O^T            += Unew^T P^T                   (N = C, K = C)
//     with bf16 copies of S (the A operand above), Unew and f o Unew written to
//     shared memory by the warpgroups that read the accumulators.
//
// (Chunk form: "Parallelizing Linear Transformers with the Delta Rule over
// Sequence Length", WY / UT representation and the chunk-state scan;
// "Gated DeltaNet", gates folded in as within-chunk cumulative log-decays.)
//
// The launch is cooperative, so every CTA is resident and the producer /
// consumer flags in the workspace cannot deadlock on scheduling.  Tasks are
// handed out in order (chunk index major), a preparation pipeline waits for its
// ring slot to be consumed (RING slots per ring), and a chain CTA waits for its
// next package; every such wait, like every mbarrier wait, is bounded and
// reports a timeout through the status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>

#include "fast.h"
#include "prep_math.cuh"
#include "sm100.cuh"

// Optional event timeline of chain CTA 0 and of the preparation of its chunks
// (compiled only with -DGDN_TRACE).
#ifdef GDN_TRACE
__device__ unsigned long long g_coop_trace[256][32];
#define CTR(n, e)                                                                \
    do {                                                                         \
        if ((n) < 256) {                                                         \
            unsigned long long t_;                                               \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));               \
            g_coop_trace[(n)][(e)] = t_;                                         \
        }                                                                        \
    } while (0)
#else
#define CTR(n, e) \
    do {          \
    } while (0)
#endif

namespace gdn {
namespace coop {
using namespace sm100;
using namespace prep;

namespace {

constexpr int NTHREADS = 512;
constexpr int PIPES = 4;   // preparation pipelines per CTA (four warps each)
// control block, in 32-bit words: line 0 holds the task counter [0] and Jmax [1];
// then one 128-byte line per chain CTA for its consumed count and one per ring
// (chain group) for its RING ready flags, so that pollers and the task counter do
// not share lines; the last line holds the launch-wide abort word (set by the
// first CTA whose bounded wait runs out, polled by every cross-CTA wait so that
// the launch winds down)
constexpr int CTL_LINE = 32;
__host__ __device__ constexpr size_t ctl_words(int nc, int ng) { return (size_t)CTL_LINE * (2 + (size_t)nc + (size_t)ng); }
__device__ __forceinline__ uint32_t *consumed_word(uint32_t *ctl, int c) { return ctl + CTL_LINE * (1 + c); }
__device__ __forceinline__ uint32_t *ready_words(uint32_t *ctl, int nc, int grp) { return ctl + CTL_LINE * (1 + nc + grp); }
__device__ __forceinline__ uint32_t *abort_word(uint32_t *ctl, int nc, int ng) { return ctl + CTL_LINE * (1 + nc + ng); }
constexpr long long BUDGET = 4000000000LL;                 // clock cycles (about 2 s)
// With the test hook GDN_DEBUG_WITHHOLD_TASK set, the cross-CTA flag waits give up
// after this many cycles (about 1 ms) instead of BUDGET.
constexpr long long HOOK_FLAG_BUDGET = 2000000LL;
constexpr float RENORM_BELOW = 9.313225746154785e-10f;      // 2^-30

__host__ __device__ constexpr uint32_t round1k(uint32_t x) { return (x + 1023u) & ~1023u; }
__host__ __device__ constexpr uint32_t umax(uint32_t a, uint32_t b) { return a > b ? a : b; }

// Layout of one instance: chunk C_, head dims d_k = d_v = DK_.  Every bf16 operand
// tile is stored in 64-column panels of 128-byte rows with the 128-byte swizzle; a
// row of C elements (C = 32) fills the first half of its 128 bytes.
template <int C_, int DK_>
struct Cfg {
    static constexpr int C = C_;
    static constexpr int DK = DK_;
    static constexpr int DV = DK_;
    static constexpr int NV = DV / 128;        // chain CTAs per (sequence, head)
    static constexpr int NQ = DK / 64;         // 64-column panels of a d_k-wide tile
    static constexpr int KW = C / 32;          // warps over a chunk's rows
    static constexpr uint32_t PANEL = (uint32_t)C * 128;   // one panel of a chunk's rows
    // package ring depth: about 450 KB per ring (deeper rings spill packages from
    // L2 to HBM: 10 slots of the C = 64 package added 78 MB of DRAM traffic per launch)
    static constexpr int RING = C == 64 ? 9 : (DK == 128 ? 18 : 20);
    // the backward's outputs (packages, S_in, Unew) are compiled into the instance the
    // tcgen05 backward takes only
    static constexpr bool EMIT = C == 64 && DK == 128;

    // package (ring slot in global memory and its copy in a chain CTA's shared memory)
    static constexpr uint32_t WQ_PANEL = 2 * PANEL;        // per panel [-W rows | Qt rows]
    static constexpr uint32_t PK_WQ = 0;
    static constexpr uint32_t PK_T = NQ * WQ_PANEL;        // T bf16 [r][i]
    static constexpr uint32_t PK_P = PK_T + PANEL;         // P bf16 [r][i]
    static constexpr uint32_t PK_VEC = PK_P + PANEL;       // f0[64] = exp(gamma_C - gamma_r) n_r, then exp(gamma_C)
    static constexpr uint32_t VEC_BYTES = 272;
    static constexpr uint32_t PK_BYTES = PK_VEC + VEC_BYTES;
    static constexpr uint32_t PK_STRIDE = round1k(PK_BYTES);

    // chain CTA shared memory
    static constexpr uint32_t KTILE = NQ * PANEL;
    static constexpr uint32_t CH_K = 0;                          // 2 K tiles [token][d_k]
    static constexpr uint32_t CH_V = 2 * KTILE;                  // V tile [token][128 d_v]
    static constexpr uint32_t CH_PK = CH_V + 2 * PANEL;          // 2 package slots
    static constexpr uint32_t CH_SB = CH_PK + 2 * PK_STRIDE;     // S^T bf16 [dv][dk], NQ panels of 128 rows
    static constexpr uint32_t CH_U1 = CH_SB + NQ * 16384;        // Unew^T bf16 [dv][token] (16 KB)
    static constexpr uint32_t CH_U2 = CH_U1 + 16384;             // (f o Unew)^T bf16 (16 KB)
    static constexpr uint32_t CH_BAR = CH_U2 + 16384;
    static constexpr uint32_t CH_END = CH_BAR + 32 * 8 + 64;

    // preparation pipeline shared memory
    static constexpr uint32_t AST = C == 64 ? 72 : 40;           // row stride (floats) of the solve buffer
    static constexpr uint32_t PP_TL = 0;        // per panel [K rows | Q rows]; K becomes -W, Q becomes Qt
                                                //   and then T (panel 0) | P (panel 1)
    static constexpr uint32_t PP_AX = NQ * WQ_PANEL;             // fp32 [C][AST]: A below the diagonal, X^T on
                                                                 //   and above it; then T' (bf16)
    // The M = 128 products read 128 A rows where C = 32 fills fewer: T' K reads
    // 16 KB from PP_AX, the Gram 8 KB past the last [K | Q] panel.  Both windows
    // end before the vectors and barriers and hold only the solve buffer, which
    // nothing writes while those products run; their result rows are never read.
    static constexpr uint32_t PP_VEC = PP_AX + umax((uint32_t)C * AST * 4, 16384);   // vectors, 12 x 64 floats
    static constexpr uint32_t PP_BAR = PP_VEC + 12 * 256;        // barriers + task word
    static constexpr uint32_t PP_STRIDE = round1k(PP_BAR + 64);
    static constexpr uint32_t SMEM_USED = umax(CH_END, PIPES * PP_STRIDE);
    static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;

    // chain TMEM columns: S_hat^T fp32 (lane = dv, column = dk), then per chunk
    // parity [X (C) | O (C)]
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_XO = DK;
    static constexpr uint32_t XO_STRIDE = 2 * C;

    static constexpr uint32_t ID_U = idesc(1, 128, C, true, false);         // V^T T^T
    static constexpr uint32_t ID_XO = idesc(1, 128, 2 * C, false, false);   // S^T [-W | Qt]^T; [K;Q][K;Q]^T
    static constexpr uint32_t ID_S = idesc(1, 128, DK, false, true);        // (f o Unew)^T K
    static constexpr uint32_t ID_O = idesc(1, 128, C, false, false);        // Unew^T P^T
    static constexpr uint32_t ID_TK = idesc(1, 128, 128, false, true);      // T' K, 128 columns of d_k

    static_assert(C == 32 || C == 64, "chunk");
    static_assert(DK == 128 || DK == 256, "head dim");
    static_assert(RING <= CTL_LINE, "ready flags of one ring fit one line");
    static_assert(PP_STRIDE % 1024 == 0 && PP_AX % 1024 == 0 && PK_STRIDE % 1024 == 0, "swizzled operands need 1 KB alignment");
    static_assert((uint32_t)C * 128 <= (uint32_t)C * AST * 4, "T' fits the solve buffer");
    static_assert(TM_XO + 2 * XO_STRIDE <= 512, "TMEM columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

using Cfg64 = Cfg<64, 128>;
using Cfg32 = Cfg<32, 128>;
using Cfg32w = Cfg<32, 256>;

// chain barriers
enum {
    B_KFULL = 0, B_KEMPTY = 2, B_VFULL = 4, B_VEMPTY = 5, B_PFULL = 6, B_PEMPTY = 8, B_X = 10,
    B_S = 12, B_O = 13, B_U2READY = 15, B_SNAP = 16, B_OFREE = 17, B_ABORTED = 19, NBAR_CH = 20
};
// preparation barriers (per pipeline)
enum { P_FULL = 0, P_G = 1, P_W = 2, P_DONE = 3, NBAR_PP = 4 };

struct Params {
    const __nv_bfloat16 *beta;
    const float *gate;
    const float *h0;
    __nv_bfloat16 *o;
    float *hT;
    uint32_t *status;
    const int32_t *cu;       // packed offsets or null
    const int32_t *order;    // packed: sequences longest first (or null)
    uint32_t *ctl;           // control block (ctl_words(Nc, Ng) words, see CTL_LINE)
    uint8_t *ring;           // Ng x RING package slots
    int H, T, N, items, Nc, Ng, Jmax_fixed;   // Ng = Nc / NV chain groups, one ring each
    float scale, eps;
    int l2norm;
    int longhorn;           // step size beta / (1 + beta k^T k) instead of beta
    int withhold;           // test hook: this task's package is never published (-1: none)
    long long flag_budget;  // cycles a cross-CTA flag wait may take before it gives up
    // for the backward (null otherwise): every package also into keep[slot], the bf16
    // state entering each chunk into sin_out[slot][dk][dv] and Unew into
    // unew_out[slot][C][dv], slot = chunk slot * H + head (chunk slots of a sequence
    // from cstart, packed input, or nchs per sequence)
    uint8_t *keep;
    __nv_bfloat16 *sin_out, *unew_out;
    const int32_t *cstart;
    int nchs;
};

// workspace slot of chunk n of (sequence seq, head h), as the general kernels number them
__device__ __forceinline__ size_t slot_of(const Params &p, int seq, int h, int n)
{
    const int j0 = p.cstart ? p.cstart[seq] : seq * p.nchs;
    return (size_t)(j0 + n) * p.H + h;
}

__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

struct Item {
    int seq, h, L, nch;
    long long rowbase;
};

template <int C>
__device__ __forceinline__ Item item_of(const Params &p, int it)
{
    Item r;
    r.h = it % p.H;
    const int rank = it / p.H;
    if (p.cu) {
        r.seq = p.order ? p.order[rank] : rank;
        int t0 = p.cu[r.seq], t1 = p.cu[r.seq + 1];
        if (t0 < 0 || t1 < t0 || t1 > p.T) t0 = t1 = 0;   // malformed offsets: empty (flagged elsewhere)
        r.L = t1 - t0;
        r.rowbase = (long long)r.h * p.T + t0;
    } else {
        r.seq = rank;
        r.L = p.T;
        r.rowbase = ((long long)r.seq * p.H + r.h) * p.T;
    }
    r.nch = (r.L + C - 1) / C;
    return r;
}

// Walks the chunk stream of chain group g: its items g, g + Ng, ... (empty ones
// skipped), each chunk in order.
template <int C>
struct Stream {
    int it, n;
    Item cur;
    bool valid;
    __device__ void start(const Params &p, int g)
    {
        it = g - p.Ng;
        advance_item(p);
    }
    __device__ void advance_item(const Params &p)
    {
        while (true) {
            it += p.Ng;
            if (it >= p.items) { valid = false; return; }
            cur = item_of<C>(p, it);
            if (cur.nch > 0) break;
        }
        n = 0;
        valid = true;
    }
    __device__ void next(const Params &p)
    {
        if (++n >= cur.nch) advance_item(p);
    }
    __device__ bool first() const { return n == 0; }
    __device__ bool last() const { return n == cur.nch - 1; }
    __device__ int len() const { return min(C, cur.L - n * C); }
    __device__ long long row0() const { return cur.rowbase + (long long)n * C; }
};

template <int C>
__device__ __forceinline__ int stream_length(const Params &p, int g)
{
    int J = 0;
    for (int it = g; it < p.items; it += p.Ng) J += item_of<C>(p, it).nch;
    return J;
}

// r[0, 32 N) <- 32 N consecutive TMEM columns of this warp's lanes
template <int N32>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t *r)
{
#pragma unroll
    for (int i = 0; i < N32; ++i) tmem_ld32(taddr + 32 * i, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * i));
}

}  // namespace

// ================================================================================= chain role
template <class L>
__device__ __forceinline__ void chain_cta(const Params &p, const CUtensorMap *tm_k,
                                          const CUtensorMap *tm_v, uint8_t *sm, int c)
{
    constexpr int C = L::C, DK = L::DK, DV = L::DV, NQ = L::NQ;
    constexpr uint32_t PANEL = L::PANEL;
    const uint32_t sb = smem_u32(sm);
    uint64_t *bar = (uint64_t *)(sm + L::CH_BAR);
    volatile int *abort_flag = (volatile int *)(sm + L::CH_BAR + 32 * 8);
    uint32_t *tmem_slot = (uint32_t *)(sm + L::CH_BAR + 32 * 8 + 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = c / L::NV, hv = c % L::NV;   // chain group (ring) and d_v half
    uint32_t *consumed = consumed_word(p.ctl, c);
    uint32_t *ready = ready_words(p.ctl, p.Nc, grp);
    volatile uint32_t *gabort = abort_word(p.ctl, p.Nc, p.Ng);
    const uint8_t *ring = p.ring + (size_t)grp * L::RING * L::PK_STRIDE;

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < NBAR_CH; ++i) {
            uint32_t cnt = 1;
            if (i == B_U2READY || i == B_SNAP) cnt = 8;
            if (i == B_OFREE || i == B_OFREE + 1) cnt = 4;
            mbar_init(&bar[i], cnt);
        }
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(tm_k);
        prefetch_tmap(tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int J = stream_length<C>(p, grp);

    auto fail = [&]() {
        if (!*abort_flag) {
            *abort_flag = 1;
            raise_status(p.status, kStatusTimeout);
            atomicExch((uint32_t *)gabort, 1u);
        }
    };
    auto wait = [&](int b, uint32_t k) -> bool {
        if (mbar_wait(&bar[b], k & 1u, BUDGET, abort_flag)) return true;
        fail();
        return false;
    };

    if (warp == 0) {
        // ---------------------------------------------------------------- K / V tiles (TMA)
        if (lane == 0) {
            Stream<C> st;
            st.start(p, grp);
            int jk = -1, jv = -1;   // last chunk whose K / V copy was issued
            for (int j = 0; j < J && st.valid; ++j, st.next(p)) {
                const int s = j & 1;
                const int row = (int)st.row0();
                if (j >= 2 && !wait(B_KEMPTY + s, (uint32_t)((j >> 1) - 1))) break;
                mbar_expect_tx(&bar[B_KFULL + s], L::KTILE);
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    tma_load_2d(sm + L::CH_K + s * L::KTILE + q * PANEL, tm_k, &bar[B_KFULL + s], 64 * q, row);
                jk = j;
                if (j >= 1 && !wait(B_VEMPTY, (uint32_t)(j - 1))) break;
                mbar_expect_tx(&bar[B_VFULL], 2 * PANEL);
                tma_load_2d(sm + L::CH_V, tm_v, &bar[B_VFULL], 128 * hv, row);
                tma_load_2d(sm + L::CH_V + PANEL, tm_v, &bar[B_VFULL], 128 * hv + 64, row);
                jv = j;
            }
            // the last copies issued into each buffer have landed before shared memory
            // goes away (on the normal path they have long since been consumed and
            // these waits return at once; after an abort nothing else waits for them)
            for (int jj = (jk > 0 ? jk - 1 : 0); jj <= jk; ++jj)
                mbar_wait(&bar[B_KFULL + (jj & 1)], (uint32_t)(jj >> 1) & 1u, BUDGET, nullptr);
            if (jv >= 0) mbar_wait(&bar[B_VFULL], (uint32_t)jv & 1u, BUDGET, nullptr);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------------- packages (bulk copies)
        if (lane == 0) {
            // two copies in flight: chunk j's copy is issued before chunk j - 1's has been
            // waited for, and the producer's flag of chunk j is polled while that copy lands
            int issued = 0, landed = 0;
            bool ok = true;
            for (int j = 0; j < J && ok; ++j) {
                const int s = j & 1, slot = j % L::RING;
                // wait for the producer's flag
                const long long t0 = clock64();
                unsigned ns = 32;
                while (ld_acquire_gpu(&ready[slot]) != (uint32_t)(j + 1)) {
                    if (*abort_flag || *gabort || clock64() - t0 > p.flag_budget) { ok = false; break; }
                    __nanosleep(ns);
                    ns = ns < 256 ? 2 * ns : ns;
                }
                if (!ok) { fail(); break; }
                fence_async_global();
                if (c == 0) CTR(j, 0);
                if (j >= 2 && !(ok = wait(B_PEMPTY + s, (uint32_t)((j >> 1) - 1)))) break;
                mbar_expect_tx(&bar[B_PFULL + s], L::PK_BYTES);
                bulk_load(sm + L::CH_PK + s * L::PK_STRIDE, ring + (size_t)slot * L::PK_STRIDE, L::PK_BYTES,
                          &bar[B_PFULL + s]);
                issued = j + 1;
                if (c == 0) CTR(j, 1);
                // chunk j - 1's copy has landed: its ring slot may be refilled
                if (j >= 1) {
                    if (!(ok = wait(B_PFULL + ((j - 1) & 1), (uint32_t)((j - 1) >> 1)))) break;
                    landed = j;
                    st_release_gpu(consumed, (uint32_t)landed);
                }
            }
            if (ok && issued == J && J > 0 && (ok = wait(B_PFULL + ((J - 1) & 1), (uint32_t)((J - 1) >> 1)))) {
                landed = J;
                st_release_gpu(consumed, (uint32_t)landed);
            }
            // on a failure, let the copies in flight land before shared memory goes away
            for (int n = landed; n < issued; ++n)
                mbar_wait(&bar[B_PFULL + (n & 1)], (uint32_t)(n >> 1) & 1u, BUDGET, nullptr);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && J > 0) {
            const uint64_t dSB = sdesc(sb + L::CH_SB, 16, 1024);
            const uint64_t dU1 = sdesc(sb + L::CH_U1, 16, 1024), dU2 = sdesc(sb + L::CH_U2, 16, 1024);
            const uint64_t dK0 = sdesc(sb + L::CH_K, PANEL, 1024), dK1 = sdesc(sb + L::CH_K + L::KTILE, PANEL, 1024);
            const uint64_t dV = sdesc(sb + L::CH_V, PANEL, 1024);
            const uint64_t dPK0 = sdesc(sb + L::CH_PK, 16, 1024), dPK1 = sdesc(sb + L::CH_PK + L::PK_STRIDE, 16, 1024);
            auto issue_U = [&](int m) {
                // U^T = V^T T^T into X[m & 1]
                tc_fence_after();
                const uint64_t dpk = (m & 1) ? dPK1 : dPK0;
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    mma_bf16_ss(tmem + L::TM_XO + (m & 1) * L::XO_STRIDE, dadd(dV, k * 2048),
                                dadd(dpk, L::PK_T + k * 32), L::ID_U, k > 0);
                mma_commit(&bar[B_VEMPTY]);
            };
            bool ok = wait(B_VFULL, 0) && wait(B_PFULL, 0);
            if (ok) issue_U(0);
            for (int j = 0; j < J && ok; ++j) {
                const int s = j & 1;
                const uint64_t dpk = s ? dPK1 : dPK0;
                // [Unew^T | O^T] += S^T [-W | Qt]^T
                if (!(ok = wait(B_PFULL + s, (uint32_t)(j >> 1)))) break;
                if (!(ok = wait(B_SNAP, (uint32_t)j))) break;
                if (!(ok = wait(B_OFREE + s, (uint32_t)(j >> 1)))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4 * NQ; ++k)
                    mma_bf16_ss(tmem + L::TM_XO + s * L::XO_STRIDE, dadd(dSB, (k >> 2) * 16384 + (k & 3) * 32),
                                dadd(dpk, L::PK_WQ + (k >> 2) * L::WQ_PANEL + (k & 3) * 32), L::ID_XO, 1);
                mma_commit(&bar[B_X + s]);
                if (c == 0) CTR(j, 2);
                // S_hat^T += U2^T K ; O^T += U1^T P^T
                if (!(ok = wait(B_U2READY, (uint32_t)j))) break;
                if (c == 0) CTR(j, 3);
                if (!(ok = wait(B_KFULL + s, (uint32_t)(j >> 1)))) break;
                tc_fence_after();
                {
                    const uint64_t dk = s ? dK1 : dK0;
#pragma unroll
                    for (int k = 0; k < C / 16; ++k)
                        mma_bf16_ss(tmem + L::TM_S, dadd(dU2, k * 32), dadd(dk, k * 2048), L::ID_S, 1);
                }
                mma_commit(&bar[B_S]);
                mma_commit(&bar[B_KEMPTY + s]);
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    mma_bf16_ss(tmem + L::TM_XO + s * L::XO_STRIDE + C, dadd(dU1, k * 32),
                                dadd(dpk, L::PK_P + k * 32), L::ID_O, 1);
                mma_commit(&bar[B_O + s]);
                mma_commit(&bar[B_PEMPTY + s]);
                if (c == 0) CTR(j, 4);
                // U of the next chunk
                if (j + 1 < J) {
                    if (!(ok = wait(B_VFULL, (uint32_t)(j + 1)))) break;
                    if (!(ok = wait(B_PFULL + ((j + 1) & 1), (uint32_t)((j + 1) >> 1)))) break;
                    issue_U(j + 1);
                    if (c == 0) CTR(j, 5);
                }
            }
            mma_commit(&bar[B_ABORTED]);
            mbar_wait(&bar[B_ABORTED], 0, BUDGET, nullptr);
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------- state and Unew, split in halves over two warpgroups
        // warpgroup `half` owns S columns (d_k) [DK/2 half, DK/2 half + DK/2) and chunk
        // tokens [C/2 half, C/2 half + C/2); per chunk: state snapshot for the next
        // MMA, then Unew -> U1, U2 once X is in TMEM; h0 in and h_T out at item ends
        constexpr int KH = DK / 2, CH = C / 2;
        const int half = (warp >> 2) - 1;
        const int dvl = (warp & 3) * 32 + lane;   // TMEM lane: d_v column within this CTA's 128
        const int dvg = 128 * hv + dvl;           // d_v column of the item
        const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
        const int tid_trace = 128 + 128 * half;
        // items without chunks pass their initial state straight through
        if (p.hT) {
            for (int it = grp; it < p.items; it += p.Ng) {
                const Item I = item_of<C>(p, it);
                if (I.nch == 0) {
                    const size_t sidx = ((size_t)I.seq * p.H + I.h) * DK * DV;
                    for (int k = KH * half; k < KH * half + KH; ++k)
                        p.hT[sidx + (size_t)k * DV + dvg] = p.h0 ? p.h0[sidx + (size_t)k * DV + dvg] : 0.f;
                }
            }
        }
        Stream<C> st;
        st.start(p, grp);
        float Gpend = 1.f;
        for (int j = 0; j < J && st.valid; ++j) {
            const int s = j & 1;
            const size_t sidx = ((size_t)st.cur.seq * p.H + st.cur.h) * DK * DV;
            if (st.first()) {
                // S^T[dv][dk] = h0[dk][dv] into TMEM, pending scale 1
                Gpend = 1.f;
                for (int k0 = KH * half; k0 < KH * half + KH; k0 += 32) {
                    uint32_t r[32];
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        r[k] = __float_as_uint(p.h0 ? p.h0[sidx + (size_t)(k0 + k) * DV + dvg] : 0.f);
                    tmem_st32(tmem + lrow + L::TM_S + k0, r);
                }
                tmem_st_wait();
            } else {
                wait(B_S, (uint32_t)(j - 1));
            }
            wait(B_PFULL + s, (uint32_t)(j >> 1));
            tc_fence_after();
            const float *vec = (const float *)(sm + L::CH_PK + s * L::PK_STRIDE + L::PK_VEC);
            const float GC = vec[64];
            if (c == 0 && tid == tid_trace) CTR(j, 8);
            const float Gn = Gpend;
            const float Gnext = Gn * GC;
            const bool renorm = Gnext < RENORM_BELOW;
            // bf16 snapshot of the true state S = G S_hat (A operand of the next MMA);
            // a renormalising chunk also rescales S_hat in TMEM to exp(gamma_C) S
#pragma unroll 1
            for (int pp = 0; pp < KH / 64; ++pp) {
                const int panel = half * (KH / 64) + pp;
                uint8_t *sbp = sm + L::CH_SB + panel * 16384;
                uint32_t r[64];
                tmem_ld_cols<2>(tmem + lrow + L::TM_S + 64 * panel, r);
                tmem_ld_wait();
                uint16_t *sin = (L::EMIT && p.sin_out) ? reinterpret_cast<uint16_t *>(p.sin_out) +
                                                slot_of(p, st.cur.seq, st.cur.h, st.n) * DK * DV + dvg
                                          : nullptr;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16(Gn * __uint_as_float(r[c8 * 8 + 2 * e]), Gn * __uint_as_float(r[c8 * 8 + 2 * e + 1]));
                    *(uint4 *)(sbp + sw128(dvl, c8 * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                    if (L::EMIT && sin) {
                        // S_in[dk][dv]: w[e] holds rows k0 + 2e, k0 + 2e + 1 of this thread's d_v
                        // column; with the neighbouring lane's word, the even lane stores row
                        // k0 + 2e and the odd lane row k0 + 2e + 1, two d_v columns each
                        const int k0 = 64 * panel + c8 * 8;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t nb = __shfl_xor_sync(0xffffffffu, w[e], 1);
                            const bool odd = lane & 1;
                            const uint32_t pr = odd ? __byte_perm(nb, w[e], 0x7632u) : __byte_perm(w[e], nb, 0x5410u);
                            *reinterpret_cast<uint32_t *>(sin + (size_t)(k0 + 2 * e + (odd ? 1 : 0)) * DV - (odd ? 1 : 0)) = pr;
                        }
                    }
                }
                if (renorm) {
#pragma unroll
                    for (int e = 0; e < 64; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * Gnext);
                    tmem_st32(tmem + lrow + L::TM_S + 64 * panel, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                    tmem_st32(tmem + lrow + L::TM_S + 64 * panel + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                    tmem_st_wait();
                }
            }
            Gpend = renorm ? 1.f : Gnext;
            const float fdiv = renorm ? 1.f : 1.f / Gnext;
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_SNAP]);
            if (c == 0 && tid == tid_trace) CTR(j, 9);
            // Unew (this warpgroup's C/2 tokens) -> U1 = Unew^T, U2 = (f o Unew)^T / G, bf16
            if (!__all_sync(0xffffffffu, wait(B_X + s, (uint32_t)(j >> 1)))) break;
            if (c == 0 && tid == tid_trace) CTR(j, 6);
            tc_fence_after();
            {
                uint32_t x[CH];
                if constexpr (CH == 32) tmem_ld32(tmem + lrow + L::TM_XO + s * L::XO_STRIDE + CH * half, x);
                else tmem_ld16(tmem + lrow + L::TM_XO + s * L::XO_STRIDE + CH * half, x);
                tmem_ld_wait();
                uint8_t *u1 = sm + L::CH_U1, *u2 = sm + L::CH_U2;
                const float *f0 = vec + CH * half;
#pragma unroll
                for (int c8 = 0; c8 < CH / 8; ++c8) {
                    uint32_t w1[4], w2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = c8 * 8 + 2 * e;
                        const float a = __uint_as_float(x[i0]), b = __uint_as_float(x[i0 + 1]);
                        w1[e] = pack_bf16(a, b);
                        w2[e] = pack_bf16(a * f0[i0] * fdiv, b * f0[i0 + 1] * fdiv);
                    }
                    const uint32_t off = sw128(dvl, ((CH / 8) * half + c8) * 16);
                    *(uint4 *)(u1 + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                    *(uint4 *)(u2 + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
                }
                if (L::EMIT && p.unew_out) {
                    // Unew[token][dv] (rows past the chunk's end are zeros here already): token
                    // pairs of this thread's d_v column, exchanged with the neighbouring lane so
                    // that each lane stores one token row of two d_v columns
                    uint16_t *un = reinterpret_cast<uint16_t *>(p.unew_out) +
                                   (slot_of(p, st.cur.seq, st.cur.h, st.n) * C + CH * half) * DV + dvg;
                    const bool odd = lane & 1;
#pragma unroll
                    for (int i = 0; i < CH; i += 2) {
                        const uint32_t wv = pack_bf16(__uint_as_float(x[i]), __uint_as_float(x[i + 1]));
                        const uint32_t nb = __shfl_xor_sync(0xffffffffu, wv, 1);
                        const uint32_t pr = odd ? __byte_perm(nb, wv, 0x7632u) : __byte_perm(wv, nb, 0x5410u);
                        *reinterpret_cast<uint32_t *>(un + (size_t)(i + (odd ? 1 : 0)) * DV - (odd ? 1 : 0)) = pr;
                    }
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_U2READY]);
            if (c == 0 && tid == tid_trace) CTR(j, 7);
            if (st.last()) {
                // h_T = G S_hat once the chunk's state update has landed
                wait(B_S, (uint32_t)j);
                tc_fence_after();
                if (p.hT && !*abort_flag) {
                    for (int k0 = KH * half; k0 < KH * half + KH; k0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(tmem + lrow + L::TM_S + k0, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            p.hT[sidx + (size_t)(k0 + k) * DV + dvg] = Gpend * __uint_as_float(r[k]);
                    }
                }
            }
            st.next(p);
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
    } else if (warp >= 12) {
        // ---------------------------------------------------------------- output
        const int dvl = (warp & 3) * 32 + lane;
        const int dvg = 128 * hv + dvl;
        const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16;
        {
            uint32_t z[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) z[k] = 0u;
            for (int s = 0; s < 2; ++s)
#pragma unroll
                for (int cc = 0; cc < C; cc += 32) tmem_st32(tmem + lrow + L::TM_XO + s * L::XO_STRIDE + C + cc, z);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar[B_OFREE]);
                mbar_arrive(&bar[B_OFREE + 1]);
            }
        }
        Stream<C> st;
        st.start(p, grp);
        for (int j = 0; j < J && st.valid; ++j, st.next(p)) {
            const int s = j & 1;
            if (!__all_sync(0xffffffffu, wait(B_O + s, (uint32_t)(j >> 1)))) break;
            if (c == 0 && tid == 384) CTR(j, 10);
            tc_fence_after();
            uint32_t ov[C];
            tmem_ld_cols<C / 32>(tmem + lrow + L::TM_XO + s * L::XO_STRIDE + C, ov);
            tmem_ld_wait();
            uint32_t z[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) z[k] = 0u;
#pragma unroll
            for (int cc = 0; cc < C; cc += 32) tmem_st32(tmem + lrow + L::TM_XO + s * L::XO_STRIDE + C + cc, z);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[B_OFREE + s]);
            const int len = st.len();
            if (p.o) {
                __nv_bfloat16 *orow = p.o + st.row0() * DV + dvg;
#pragma unroll
                for (int r = 0; r < C; ++r)
                    if (r < len) orow[(size_t)r * DV] = __float2bfloat16_rn(p.scale * __uint_as_float(ov[r]));
            }
            if (c == 0 && tid == 384) CTR(j, 11);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================================================= preparation role
// Four independent pipelines (warps 4p .. 4p + 3) take chunk tasks from a global
// counter.  One task, for chunk n of item (seq, head):
//   TMA K, Q -> [K;Q][K;Q]^T on the tensor cores (Gram rows, Q K^T rows, both
//   norms on the diagonal) -> gates, scale vectors -> Qt in place, published at
//   once -> A (warps [0, C/32)) while P is built (warps [C/32, C/16)) -> (I + A)^-1
//   in place -> T, T' -> -(T' K) on the tensor cores, 128 columns of d_k at a
//   time -> -W over K -> publish, ready flag.
template <class L>
__device__ __forceinline__ void prep_cta(const Params &p, const CUtensorMap *tm_q,
                                         const CUtensorMap *tm_k, uint8_t *sm)
{
    constexpr int C = L::C, DK = L::DK, NQ = L::NQ, KW = L::KW, AST = (int)L::AST;
    constexpr uint32_t PANEL = L::PANEL, WQP = L::WQ_PANEL;
    constexpr int TPUB = 32 * KW;   // the thread that publishes (first thread of the P warps)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    if (tid == 0) s_abort = 0;
    if (warp == 0) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    const int pipe = warp >> 2;
    uint8_t *base = sm + pipe * L::PP_STRIDE;
    uint64_t *bar = (uint64_t *)(base + L::PP_BAR);
    if ((warp & 3) == 0 && lane == 0) {
        for (int i = 0; i < NBAR_PP; ++i) mbar_init(&bar[i], 1);
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int *abort_flag = &s_abort;

    const int t = tid & 127;   // thread within the pipeline
    const int q4 = warp & 3;   // warp within the pipeline = its TMEM lane quarter
    const int bar_id = 1 + pipe;            // the pipeline's four warps
    const int bar_hi = 1 + PIPES + pipe;    // its P warps
    const uint32_t lrow = (uint32_t)(q4 * 32) << 16;
    const uint32_t tg = tmem + pipe * 128;  // [K;Q][K;Q]^T (2C columns), later T' K (128)
    const uint32_t sbase = smem_u32(base);
    volatile int *task_word = (volatile int *)(base + L::PP_BAR + NBAR_PP * 8);
    float *vb = (float *)(base + L::PP_VEC);
    float *s_beta = vb, *s_gl = vb + 64, *s_nk = vb + 128, *s_nq = vb + 192, *s_tc = vb + 256;
    float *s_qs = vb + 320, *s_ra = vb + 384, *s_cb = vb + 448, *s_f0 = vb + 512, *s_g = vb + 576;
    int *s_safe = (int *)(vb + 640);
    float *s_kk = vb + 704;             // k_hat_r^T k_hat_r (Longhorn's step size)
    float *AX = (float *)(base + L::PP_AX);
    uint8_t *tl = base + L::PP_TL;
    const int Jmax = p.cu ? (int)p.ctl[1] : p.Jmax_fixed;
    const long long ntasks = (long long)p.Ng * Jmax;
    volatile uint32_t *gabort = abort_word(p.ctl, p.Nc, p.Ng);
    auto fail = [&]() {
        if (!*abort_flag) {
            *abort_flag = 1;
            raise_status(p.status, kStatusTimeout);
            atomicExch((uint32_t *)gabort, 1u);
        }
    };
    auto wait = [&](int b, uint32_t k) -> bool {
        if (mbar_wait(&bar[b], k & 1u, BUDGET, abort_flag)) return true;
        fail();
        return false;
    };
    // chunk j of chain group g: item and chunk within it (false if the stream is shorter)
    auto locate = [&](int g, int j, Item &I, int &n) -> bool {
        n = j;
        for (int it = g; it < p.items; it += p.Ng) {
            I = item_of<C>(p, it);
            if (n < I.nch) return true;
            n -= I.nch;
        }
        return false;
    };
    uint32_t k_task = 0;   // tasks this pipeline has run (barrier phases)
    uint32_t k_w = 0;      // T' K products this pipeline has waited for (P_W phases)
    uint32_t tma_phase = 0;   // (t == 0) barrier phase of the K, Q copy last issued
    bool tma_pending = false, mma_issued = false;
    uint32_t *pend_ready = nullptr;     // (t == TPUB) flag of a package still being written
    uint32_t pend_val = 0;
    while (true) {
        if (t == TPUB && pend_ready) {
            // the previous package has landed: raise its ready flag (while thread 0 fetches a task)
            bulk_wait_all();
            fence_async_global();
            __threadfence();
            st_release_gpu(pend_ready, pend_val);
            pend_ready = nullptr;
        }
        if (t == 0) {
            const int tk = (int)atomicAdd(&p.ctl[0], 1u);
            // one decision for the whole pipeline
            *task_word = (*abort_flag || *gabort) ? 0x7fffffff : tk;
        }
        named_bar(bar_id, 128);
        const int task = *task_word;
        named_bar(bar_id, 128);
        if (task >= ntasks) break;
        const int grp = task % p.Ng, j = task / p.Ng;
        Item I;
        int n;
        if (!locate(grp, j, I, n)) continue;
        if (task == p.withhold) continue;   // test hook: the chain CTAs' wait for it must run out
        if (grp == 0 && t == 0) CTR(j, 12);
        const int len = min(C, I.L - n * C);
        const long long row0 = I.rowbase + (long long)n * C;
        const int slot = j % L::RING;
        uint32_t *ready = ready_words(p.ctl, p.Nc, grp) + slot;
        uint8_t *dst = p.ring + ((size_t)grp * L::RING + slot) * L::PK_STRIDE;
        uint8_t *kdst = (L::EMIT && p.keep) ? p.keep + slot_of(p, I.seq, I.h, n) * L::PK_STRIDE : nullptr;
        if (t == 0) {
            // the ring slot must have been copied out by every chain CTA of the group
            const long long t0 = clock64();
            unsigned ns = 64;
            for (int hv = 0; hv < L::NV && !*abort_flag; ++hv) {
                uint32_t *consumed = consumed_word(p.ctl, grp * L::NV + hv);
                while ((int)ld_acquire_gpu(consumed) < j - L::RING + 1) {
                    if (*gabort || clock64() - t0 > p.flag_budget) { fail(); break; }
                    __nanosleep(ns);
                    ns = ns < 256 ? 2 * ns : ns;   // a freed slot is seen within ~0.3 us
                }
            }
            if (!*abort_flag) {
                mbar_expect_tx(&bar[P_FULL], NQ * WQP);
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    tma_load_2d(tl + q * WQP, tm_k, &bar[P_FULL], 64 * q, (int)row0);
                    tma_load_2d(tl + q * WQP + PANEL, tm_q, &bar[P_FULL], 64 * q, (int)row0);
                }
                tma_pending = true;
                tma_phase = k_task;
                if (grp == 0) CTR(j, 13);
            }
        }
        if (q4 == 0) {
            // beta and g (zero past the chunk), gates scanned in log2 units
            float gv[KW];
            bool pos = false;
#pragma unroll
            for (int e = 0; e < KW; ++e) {
                const int i = lane + 32 * e;
                s_beta[i] = i < len ? __bfloat162float(p.beta[row0 + i]) : 0.f;
                gv[e] = (p.gate && i < len) ? p.gate[row0 + i] : 0.f;
                pos = pos || gv[e] > 0.f;
            }
            if (p.gate && __any_sync(0xffffffffu, pos) && lane == 0) raise_status(p.status, kStatusPositiveGate);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                for (int e = 0; e < KW; ++e) {
                    const float a = __shfl_up_sync(0xffffffffu, gv[e], o);
                    if (lane >= o) gv[e] += a;
                }
            }
            float carry = 0.f, mx = 0.f;
#pragma unroll
            for (int e = 0; e < KW; ++e) {
                gv[e] += carry;
                carry = __shfl_sync(0xffffffffu, gv[e], 31);
                gv[e] *= 1.4426950408889634f;
                s_gl[lane + 32 * e] = gv[e];
                mx = fmaxf(mx, fabsf(gv[e]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) *s_safe = mx < 100.f;
        }
        if (wait(P_FULL, k_task) && t == 0) tma_pending = false;
        if (grp == 0 && t == 0) CTR(j, 14);
        if (t == 0) {
            // [K;Q][K;Q]^T: Gram rows, Q K^T rows and both norms on the diagonals
            // (C = 32: A rows 64..127 are the next panel's, their results unread)
            mma_issued = true;
            tc_fence_after();
            const uint64_t d = sdesc(sbase + L::PP_TL, 16, 1024);
#pragma unroll
            for (int k = 0; k < 4 * NQ; ++k) {
                const uint64_t dk = dadd(d, (k >> 2) * WQP + (k & 3) * 32);
                mma_bf16_ss(tg, dk, dk, L::ID_XO, k > 0);
            }
            mma_commit(&bar[P_G]);
        }
        wait(P_G, k_task);
        tc_fence_after();
        if (grp == 0 && t == 0) CTR(j, 15);
        if (q4 < 2 * KW) {
            // diagonal element of this lane's row: column 32 q4 + lane
            uint32_t v[32];
            tmem_ld32(tg + lrow + 32 * q4, v);
            tmem_ld_wait();
            float dg = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) dg = (i == lane) ? __uint_as_float(v[i]) : dg;
            const int r = (q4 % KW) * 32 + lane;
            const float nrm = r < len ? (p.l2norm ? rsqrtf(dg + p.eps) : 1.f) : 0.f;
            if (q4 < KW) {
                s_nk[r] = nrm;
                s_kk[r] = dg * nrm * nrm;
            } else {
                s_nq[r] = nrm;
            }
        }
        named_bar(bar_id, 128);
        const bool safe = *s_safe != 0;
        const float glC = s_gl[len - 1];
        if (t < C) {
            const float gl = s_gl[t];
            const float e = ex2f(gl);
            // the step size: beta, or Longhorn's beta / (1 + beta k^T k)
            float bt = s_beta[t];
            if (p.longhorn) {
                bt = bt / fmaf(bt, s_kk[t], 1.f);
                s_beta[t] = bt;
            }
            s_tc[t] = bt * e * s_nk[t];
            s_qs[t] = e * s_nq[t];
            s_ra[t] = bt * s_nk[t] * e;
            s_cb[t] = safe ? s_nk[t] * ex2f(-gl) : 0.f;
            s_f0[t] = ex2f(glC - gl) * s_nk[t];
            if (t == 0) s_g[0] = ex2f(glC);
        }
        named_bar(bar_id, 128);
        if (grp == 0 && t == 0) CTR(j, 19);
        {
            // Qt = diag(exp(gamma) m) Q in place: 16-byte pieces, a warp covers 4 whole rows
#pragma unroll
            for (int u = 0; u < NQ * C / 16; ++u) {
                const int idx = u * 128 + t;
                const int hh = idx / (C * 8), r = (idx >> 3) % C;
                uint4 *qp = (uint4 *)(tl + hh * WQP + PANEL + r * 128 + (idx & 7) * 16);
                const float f = s_qs[r];
                uint4 a = *qp;
                a.x = scale_pair(a.x, f); a.y = scale_pair(a.y, f);
                a.z = scale_pair(a.z, f); a.w = scale_pair(a.w, f);
                *qp = a;
            }
        }
        fence_async_smem();
        named_bar(bar_id, 128);
        if (grp == 0 && t == 0) CTR(j, 22);
        if (q4 < KW) {
            // A = strict_lower(diag(beta n) (K K^T o D) diag(n)), full rows (zeros on and above the diagonal)
            const int r = q4 * 32 + lane;
            uint32_t v[C];
            tmem_ld_cols<C / 32>(tg + lrow, v);
            tmem_ld_wait();
            float4 *arow = reinterpret_cast<float4 *>(AX + r * AST);
            if (safe) {
                // exp(gamma_r - gamma_i) factored as exp(gamma_r) * exp(-gamma_i)
                const float ra = s_ra[r];
                const float4 *cb4 = reinterpret_cast<const float4 *>(s_cb);
#pragma unroll
                for (int c4 = 0; c4 < C / 4; ++c4) {
                    const float4 cb = cb4[c4];
                    const int i = 4 * c4;
                    arow[c4] = make_float4(i < r ? ra * cb.x * __uint_as_float(v[i]) : 0.f,
                                           i + 1 < r ? ra * cb.y * __uint_as_float(v[i + 1]) : 0.f,
                                           i + 2 < r ? ra * cb.z * __uint_as_float(v[i + 2]) : 0.f,
                                           i + 3 < r ? ra * cb.w * __uint_as_float(v[i + 3]) : 0.f);
                }
            } else {
                const float br = s_beta[r] * s_nk[r], gr = s_gl[r];
                for (int c4 = 0; c4 < C / 4; ++c4) {
                    float a[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 4 * c4 + e;
                        a[e] = (i < r) ? br * s_nk[i] * __uint_as_float(v[i]) * ex2f(gr - s_gl[i]) : 0.f;
                    }
                    arow[c4] = make_float4(a[0], a[1], a[2], a[3]);
                }
            }
            if (grp == 0 && t == 0) CTR(j, 25);
        } else if (q4 < 2 * KW) {
            // publish Qt now; once the copy has read it, its space takes T and P
            if (t == TPUB && !*abort_flag) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    bulk_store(dst + L::PK_WQ + q * WQP + PANEL, tl + q * WQP + PANEL, PANEL);
                    if (kdst) bulk_store(kdst + L::PK_WQ + q * WQP + PANEL, tl + q * WQP + PANEL, PANEL);
                }
                bulk_commit();
                bulk_wait_read();
            }
            named_bar(bar_hi, 32 * KW);
            if (grp == 0 && t == TPUB) CTR(j, 26);
            // P = lower(m_r n_i (q_r . k_i) D_ri), bf16 [r][i], into panel 1's Qt rows
            uint8_t *pt = tl + WQP + PANEL;
            const int r = (q4 - KW) * 32 + lane;
            uint32_t v[C];
            tmem_ld_cols<C / 32>(tg + lrow, v);
            tmem_ld_wait();
            const float mr = s_nq[r], gr = s_gl[r];
            if (safe) {
                const float rp = mr * ex2f(gr);
                const float4 *cb4 = reinterpret_cast<const float4 *>(s_cb);
#pragma unroll
                for (int c8 = 0; c8 < C / 8; ++c8) {
                    const float4 ca = cb4[2 * c8], cc = cb4[2 * c8 + 1];
                    const float cbv[8] = {ca.x, ca.y, ca.z, ca.w, cc.x, cc.y, cc.z, cc.w};
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = c8 * 8 + 2 * e;
                        const float a0 = (i0 <= r) ? rp * cbv[2 * e] * __uint_as_float(v[i0]) : 0.f;
                        const float a1 = (i0 + 1 <= r) ? rp * cbv[2 * e + 1] * __uint_as_float(v[i0 + 1]) : 0.f;
                        w[e] = pack_bf16(a0, a1);
                    }
                    *(uint4 *)(pt + sw128(r, c8 * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            } else {
                for (int c8 = 0; c8 < C / 8; ++c8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = c8 * 8 + 2 * e, i1 = i0 + 1;
                        const float a0 = (i0 <= r) ? mr * s_nk[i0] * __uint_as_float(v[i0]) * ex2f(gr - s_gl[i0]) : 0.f;
                        const float a1 = (i1 <= r) ? mr * s_nk[i1] * __uint_as_float(v[i1]) * ex2f(gr - s_gl[i1]) : 0.f;
                        w[e] = pack_bf16(a0, a1);
                    }
                    *(uint4 *)(pt + sw128(r, c8 * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            if (grp == 0 && t == TPUB) CTR(j, 28);
        }
        tc_fence_before();   // G's last reads precede the MMA that reuses its columns
        named_bar(bar_id, 128);
        if (grp == 0 && t == 0) CTR(j, 20);
        solve_unit_lower_packed<AST, C / 16>(AX, lane, q4, bar_id);
        if (grp == 0 && t == 0) CTR(j, 16);
        {
            // T = X diag(beta) (package, into panel 0's Qt rows) and T' = X diag(beta exp(gamma) n)
            // (operand of the next MMA, over the solve buffer); X[r][i] = AX[i][r] for i <= r.
            // Thread t: row t % C, columns [CW (t / C), CW (t / C) + CW).
            constexpr int CW = C * C / 128;
            const int r = t % C, hh = t / C;
            float x[CW];
#pragma unroll
            for (int e = 0; e < CW; ++e) {
                const int i = CW * hh + e;
                x[e] = (i <= r) ? AX[i * AST + r] : 0.f;
            }
            named_bar(bar_id, 128);   // all of X has been read before T' overwrites it
#pragma unroll
            for (int c8 = 0; c8 < CW / 8; ++c8) {
                uint32_t wt[4], wp[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i0 = CW * hh + 8 * c8 + 2 * e;
                    const float x0 = x[8 * c8 + 2 * e], x1 = x[8 * c8 + 2 * e + 1];
                    wt[e] = pack_bf16(x0 * s_beta[i0], x1 * s_beta[i0 + 1]);
                    wp[e] = pack_bf16(x0 * s_tc[i0], x1 * s_tc[i0 + 1]);
                }
                const uint32_t off = sw128(r, (hh * (CW / 8) + c8) * 16);
                *(uint4 *)(tl + PANEL + off) = make_uint4(wt[0], wt[1], wt[2], wt[3]);
                *(uint4 *)(base + L::PP_AX + off) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
            }
            if (grp == 0 && t == 0) CTR(j, 29);
        }
        fence_async_smem();
        named_bar(bar_id, 128);
        if (grp == 0 && t == 0) CTR(j, 21);
#pragma unroll 1
        for (int hn = 0; hn < DK / 128; ++hn) {
            if (t == 0) {
                // (T' K)[r][dk], 128 columns of d_k from panel 2 hn on, with r on TMEM
                // lanes 0..C-1 (A rows C..127 are don't-care)
                tc_fence_after();
                const uint64_t da = sdesc(sbase + L::PP_AX, 16, 1024);
                const uint64_t db = sdesc(sbase + L::PP_TL + 2 * hn * WQP, WQP, 1024);
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    mma_bf16_ss(tg, dadd(da, k * 32), dadd(db, k * 2048), L::ID_TK, k > 0);
                mma_commit(&bar[P_W]);
                if (grp == 0) CTR(j, 24);
            }
            if (hn == 0 && t == TPUB && !*abort_flag) {
                bulk_store(dst + L::PK_T, tl + PANEL, PANEL);
                bulk_store(dst + L::PK_P, tl + WQP + PANEL, PANEL);
                bulk_store(dst + L::PK_VEC, s_f0, L::VEC_BYTES);   // f0[64], exp(gamma_C)
                if (kdst) {
                    bulk_store(kdst + L::PK_T, tl + PANEL, PANEL);
                    bulk_store(kdst + L::PK_P, tl + WQP + PANEL, PANEL);
                    bulk_store(kdst + L::PK_VEC, s_f0, L::VEC_BYTES);
                }
                bulk_commit();
            }
            wait(P_W, k_w++);
            tc_fence_after();
            if (grp == 0 && t == 0) CTR(j, 17);
            if (q4 < KW) {
                // -W rows over the K rows: token r, 128 columns
                const int r = q4 * 32 + lane;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[64];
                    tmem_ld_cols<2>(tg + lrow + 64 * h, v);
                    tmem_ld_wait();
                    uint8_t *wrow = tl + (2 * hn + h) * WQP;
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16(-__uint_as_float(v[8 * c8 + 2 * e]), -__uint_as_float(v[8 * c8 + 2 * e + 1]));
                        *(uint4 *)(wrow + sw128(r, c8 * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            tc_fence_before();   // the columns' last reads precede the next product into them
            if (hn + 1 < DK / 128) named_bar(bar_id, 128);
        }
        fence_async_smem();
        named_bar(bar_id, 128);
        if (grp == 0 && t == 0) CTR(j, 23);
        if (t == TPUB) {
            // publish -W; the ready flag goes up at the top of the pipeline's next
            // task, once every copy of the package has landed
            if (!*abort_flag) {
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    bulk_store(dst + L::PK_WQ + q * WQP, tl + q * WQP, PANEL);
                    if (kdst) bulk_store(kdst + L::PK_WQ + q * WQP, tl + q * WQP, PANEL);
                }
                bulk_commit();
                pend_ready = ready;
                pend_val = (uint32_t)(j + 1);
                if (grp == 0) CTR(j, 18);
            }
            bulk_wait_read();   // the buffers may be refilled
        }
        ++k_task;
        named_bar(bar_id, 128);
    }
    if (t == TPUB) {
        bulk_wait_all();
        if (pend_ready && !*abort_flag) {
            fence_async_global();
            __threadfence();
            st_release_gpu(pend_ready, pend_val);
        }
    }
    if (t == 0) {
        // nothing of this pipeline may still be in flight when the block exits
        if (tma_pending) mbar_wait(&bar[P_FULL], tma_phase & 1u, BUDGET, nullptr);
        if (mma_issued) {
            mma_commit(&bar[P_DONE]);
            mbar_wait(&bar[P_DONE], 0, BUDGET, nullptr);
        }
        bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ================================================================================= kernel
template <class L>
__global__ void __launch_bounds__(NTHREADS, 1)
k_coop_fwd(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    if ((int)blockIdx.x < p.Nc) chain_cta<L>(p, &tm_k, &tm_v, sm, blockIdx.x);
    else prep_cta<L>(p, &tm_q, &tm_k, sm);
}

// Packed input: longest-first order of the sequences and the longest chunk stream of
// any chain group (written to ctl[1]).  One block.
template <int C>
__global__ void k_plan(const int32_t *cu, int N, int T, int H, int Ng, int32_t *order, uint32_t *ctl)
{
    __shared__ int s_max;
    if (threadIdx.x == 0) s_max = 0;
    __syncthreads();
    for (int s = threadIdx.x; s < N; s += blockDim.x) {
        int a = cu[s], b = cu[s + 1];
        if (a < 0 || b < a || b > T) a = b = 0;
        const int Ls = b - a;
        int rank = 0;
        if (N <= 4096) {
            for (int o = 0; o < N; ++o) {
                int a2 = cu[o], b2 = cu[o + 1];
                if (a2 < 0 || b2 < a2 || b2 > T) a2 = b2 = 0;
                const int Lo = b2 - a2;
                rank += (Lo > Ls) || (Lo == Ls && o < s);
            }
        } else {
            rank = s;
        }
        order[rank] = s;
    }
    __syncthreads();
    const int items = N * H;
    for (int g = threadIdx.x; g < Ng; g += blockDim.x) {
        int Jc = 0;
        for (int it = g; it < items; it += Ng) {
            const int sq = order[it / H];
            int a = cu[sq], b = cu[sq + 1];
            if (a < 0 || b < a || b > T) a = b = 0;
            Jc += (b - a + C - 1) / C;
        }
        atomicMax(&s_max, Jc);
    }
    __syncthreads();
    if (threadIdx.x == 0) ctl[1] = (uint32_t)s_max;
}

// ================================================================================= host
#ifdef GDN_TRACE
extern "C" int gdn_coop_trace_fetch(unsigned long long *host, size_t count)
{
    return cudaMemcpyFromSymbol(host, g_coop_trace, count * sizeof(unsigned long long)) == cudaSuccess ? 0 : 1;
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

// bf16 [rows][width] row-major, boxes of 64 columns x box_rows rows, 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, long long rows, int width, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)width, (cuuint64_t)rows};
    cuuint64_t gstr[1] = {(cuuint64_t)width * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
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

// Split of the SMs: chain CTAs (about 27 / 64 of them, at most NV per item, a
// multiple of NV), the rest prepare.
template <class L>
int chain_ctas(const Geo &g, int sms)
{
    const int items = g.N * g.H;
    int nc = (sms * 27 + 32) / 64;   // 64 of 152
    if (nc > items * L::NV) nc = items * L::NV;
    nc -= nc % L::NV;
    if (nc < L::NV) nc = L::NV;
    return nc;
}

template <class L>
size_t workspace_bytes_t(const Geo &g, int sms)
{
    if (sms <= 0) sms = 160;   // sizing without a device: an upper bound
    const int nc = chain_ctas<L>(g, sms), ng = nc / L::NV;
    const size_t ctl = ctl_words(nc, ng) * sizeof(uint32_t);
    const size_t order = g.varlen ? sizeof(int32_t) * (size_t)(g.N + 1) : 0;
    auto al = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
    return al(ctl) + al(order) + (size_t)ng * L::RING * L::PK_STRIDE;
}

template <class L>
cudaError_t fwd_t(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                  const __nv_bfloat16 *v, const __nv_bfloat16 *beta, const float *gate,
                  const float *h0, __nv_bfloat16 *o, float *hT, void *ws, size_t ws_bytes,
                  uint32_t *status, cudaStream_t st, const Emit *emit)
{
    const int sms = num_sms();
    if (sms < 2) return cudaErrorNotSupported;
    if (ws_bytes < workspace_bytes_t<L>(g, sms)) return cudaErrorInvalidValue;
    const int items = g.N * g.H;
    if (items == 0) return cudaSuccess;
    const int nc = chain_ctas<L>(g, sms), ng = nc / L::NV;
    if (nc >= sms) return cudaErrorNotSupported;
    auto al = [](size_t x) { return (x + 1023) & ~(size_t)1023; };
    uint8_t *w = (uint8_t *)ws;
    const size_t ctl_bytes = ctl_words(nc, ng) * sizeof(uint32_t);
    Params p;
    p.beta = beta; p.gate = gate; p.h0 = h0; p.o = o; p.hT = hT; p.status = status;
    p.cu = g.varlen ? g.cu : nullptr;
    p.ctl = (uint32_t *)w;
    p.order = g.varlen ? (const int32_t *)(w + al(ctl_bytes)) : nullptr;
    p.ring = w + al(ctl_bytes) + (g.varlen ? al(sizeof(int32_t) * (size_t)(g.N + 1)) : 0);
    p.H = g.H; p.T = g.T; p.N = g.N; p.items = items; p.Nc = nc; p.Ng = ng;
    p.Jmax_fixed = g.varlen ? 0 : ((items + ng - 1) / ng) * ((g.T + L::C - 1) / L::C);
    p.scale = g.scale; p.eps = g.eps; p.l2norm = g.l2norm; p.longhorn = g.longhorn;
    p.keep = emit ? emit->keep : nullptr;
    p.sin_out = emit ? emit->sin : nullptr;
    p.unew_out = emit ? emit->unew : nullptr;
    p.cstart = g.varlen ? g.cstart : nullptr;
    p.nchs = (g.T + L::C - 1) / L::C;
    if (emit && ((g.varlen && !g.cstart) || !L::EMIT)) return cudaErrorInvalidValue;
    // Test hook (failure detection): GDN_DEBUG_WITHHOLD_TASK=n makes the preparation
    // CTAs skip task n (chunk n / Ng of chain group n % Ng), so that group's bounded
    // wait for the package runs out; every cross-CTA flag wait then gives up after
    // about 1 ms, the launch winds down and the status word reports the timeout.
    p.withhold = -1;
    p.flag_budget = BUDGET;
    if (const char *e = getenv("GDN_DEBUG_WITHHOLD_TASK")) {
        if (e[0]) {
            p.withhold = atoi(e);
            p.flag_budget = HOOK_FLAG_BUDGET;
        }
    }
    cudaError_t e = cudaMemsetAsync(p.ctl, 0, ctl_bytes, st);
    if (e != cudaSuccess) return e;
    if (g.varlen) {
        k_plan<L::C><<<1, 1024, 0, st>>>(g.cu, g.N, g.T, g.H, ng, (int32_t *)p.order, p.ctl);
        if ((e = cudaPeekAtLastError()) != cudaSuccess) return e;
    }
    const long long rows = (long long)g.B * g.H * g.T;
    CUtensorMap mq, mk, mv;
    const long long maprows = rows > 0 ? rows : 1;
    if (!make_map(&mq, q, maprows, L::DK, L::C) || !make_map(&mk, k, maprows, L::DK, L::C) ||
        !make_map(&mv, v, maprows, L::DV, L::C))
        return cudaErrorInvalidValue;
    if ((e = cudaFuncSetAttribute(k_coop_fwd<L>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)L::SMEM_BYTES)) != cudaSuccess)
        return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_coop_fwd<L>, NTHREADS, L::SMEM_BYTES)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    void *args[] = {(void *)&mq, (void *)&mk, (void *)&mv, (void *)&p};
    e = cudaLaunchCooperativeKernel((const void *)k_coop_fwd<L>, dim3(sms), dim3(NTHREADS), args,
                                    L::SMEM_BYTES, st);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

// 0: (C 64, d 128), 1: (C 32, d 128), 2: (C 32, d 256), -1: none
int instance(const Geo &g)
{
    if (g.dk != g.dv) return -1;
    if (g.dk == 128 && g.C == 64) return 0;
    if (g.dk == 128 && g.C == 32) return 1;
    if (g.dk == 256 && g.C == 32) return 2;
    return -1;
}

}  // namespace

bool supports(const Geo &g, int dtype)
{
    return dtype == DN_BF16 && instance(g) >= 0 && (long long)g.B * g.H * (long long)g.T < (1LL << 31) &&
           encode_fn() != nullptr;
}

size_t workspace_bytes(const Geo &g, int sms)
{
    switch (instance(g)) {
    case 0: return workspace_bytes_t<Cfg64>(g, sms);
    case 1: return workspace_bytes_t<Cfg32>(g, sms);
    case 2: return workspace_bytes_t<Cfg32w>(g, sms);
    }
    return 0;
}

bool available()
{
    static int ok = -1;
    if (ok < 0) {
        int dev = 0, coop = 0;
        ok = cudaGetDevice(&dev) == cudaSuccess &&
             cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
             encode_fn() != nullptr && num_sms() >= 2;
    }
    return ok == 1;
}

cudaError_t fwd(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                const __nv_bfloat16 *v, const __nv_bfloat16 *beta, const float *gate,
                const float *h0, __nv_bfloat16 *o, float *hT, void *ws, size_t ws_bytes,
                uint32_t *status, cudaStream_t st, const Emit *emit)
{
    switch (instance(g)) {
    case 0: return fwd_t<Cfg64>(g, q, k, v, beta, gate, h0, o, hT, ws, ws_bytes, status, st, emit);
    case 1: return fwd_t<Cfg32>(g, q, k, v, beta, gate, h0, o, hT, ws, ws_bytes, status, st, emit);
    case 2: return fwd_t<Cfg32w>(g, q, k, v, beta, gate, h0, o, hT, ws, ws_bytes, status, st, emit);
    }
    return cudaErrorInvalidValue;
}

PkLayout package_layout(const Geo &g)
{
    PkLayout r{};
    auto fill = [&](auto cfg) {
        using L = decltype(cfg);
        r.stride = L::PK_STRIDE; r.wq = L::PK_WQ; r.wq_panel = L::WQ_PANEL; r.panel = L::PANEL;
        r.t = L::PK_T; r.p = L::PK_P; r.vec = L::PK_VEC;
    };
    switch (instance(g)) {
    case 0: fill(Cfg64{}); break;
    case 1: fill(Cfg32{}); break;
    case 2: fill(Cfg32w{}); break;
    }
    return r;
}

}  // namespace coop
}  // namespace gdn
