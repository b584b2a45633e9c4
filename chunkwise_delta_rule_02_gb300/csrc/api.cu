// C ABI of libgdn_gb300.so: argument validation, workspace layout, dispatch
// between the tcgen05 fast path and the general fp32 path, host-buffer entry
// point and the device status word.
#include <stdlib.h>
#include <string.h>

#include <cuda.h>

#include <mutex>

#include "affine.h"
#include "common.cuh"
#include "decode.h"
#include "fast.h"
#include "general.h"

namespace gdn {
namespace {

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool is_aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Validates the shape; on success fills the geometry (without device pointers).
dn_status check_shape(const dn_shape *s, Geo *g)
{
    if (!s) return DN_ERR_INVALID_ARG;
    if (s->B < 1 || s->H < 1 || s->T < 0 || s->dk < 1 || s->dv < 1) return DN_ERR_INVALID_ARG;
    if (s->dtype != DN_F32 && s->dtype != DN_BF16) return DN_ERR_INVALID_ARG;
    if (s->chunk != 16 && s->chunk != 32 && s->chunk != 64) return DN_ERR_UNSUPPORTED;
    if (s->dk > kMaxD || s->dv > kMaxD) return DN_ERR_UNSUPPORTED;
    if (!(s->eps >= 0.f) || !(s->scale == s->scale)) return DN_ERR_INVALID_ARG;
    if (s->beta_mode != DN_BETA_DELTA && s->beta_mode != DN_BETA_LONGHORN) return DN_ERR_INVALID_ARG;
    if (s->cu_seqlens) {
        if (s->B != 1 || s->num_seqs < 0) return DN_ERR_INVALID_ARG;
        if ((uintptr_t)s->cu_seqlens & 3u) return DN_ERR_INVALID_ARG;
    }
    // keep every element index inside 63 bits comfortably
    double elems = (double)s->B * s->H * (double)(s->T + 1) * (s->dk > s->dv ? s->dk : s->dv);
    if (elems > 4.0e15) return DN_ERR_INVALID_ARG;
    Geo x;
    memset(&x, 0, sizeof(x));
    x.B = s->B; x.H = s->H; x.T = s->T; x.dk = s->dk; x.dv = s->dv; x.C = s->chunk;
    x.varlen = s->cu_seqlens != nullptr;
    x.N = x.varlen ? s->num_seqs : s->B;
    x.NC = x.varlen ? (s->T + x.C - 1) / x.C + x.N : x.B * ((s->T + x.C - 1) / x.C);
    x.l2norm = s->qk_l2norm != 0;
    x.longhorn = s->beta_mode == DN_BETA_LONGHORN;
    x.scale = s->scale;
    x.eps = s->eps;
    x.cu = s->cu_seqlens;
    *g = x;
    return DN_OK;
}

// SM count of the current device (0 when there is no device, e.g. when sizing on a
// build machine; the workspace is then sized for an upper bound).
int device_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

struct Layout {
    size_t status, cstart, fast;
    size_t Kn, Qn, W, U, Unew, gam, eb, Sin, dSo, dUn, dQ, dK, dW, P, aux, M3;
    size_t coop, coop_bytes, keep, Sin_b, Un_b, dSo_b, dUn_b;   // backward through the cooperative forward
    size_t total;
};

// Which forward kernel a call takes.
enum class Fwd { General, Coop, PerItem };

// kind: the fused forward the call takes (its scratch follows the header); the
// cooperative kernel's package ring lives in the workspace.
Layout make_layout(const Geo &g, const dn_shape *s, int for_backward, Fwd kind)
{
    Layout L;
    memset(&L, 0, sizeof(L));
    size_t off = 0;
    L.status = off; off += 256;
    L.cstart = off; off += align256(sizeof(int32_t) * (size_t)(g.N + 1));
    if (kind != Fwd::General && !for_backward) {
        const size_t a = kind == Fwd::Coop ? coop::workspace_bytes(g, device_sms()) : fast::workspace_bytes(g);
        L.fast = off; off += align256(a);
        L.total = off;
        return L;
    }
    const size_t slots = (size_t)g.NC * g.H, C = g.C, dk = g.dk, dv = g.dv;
    auto take = [&](size_t nfloat) { size_t o = off; off += align256(nfloat * sizeof(float)); return o; };
    if (for_backward && gen::bwd_uses_coop(g, s->dtype)) {
        // the cooperative forward's ring, every chunk's package, and the bf16 states,
        // Unew, dS_out, dUnew of the tcgen05 per-chunk backward (for_backward = 2: the
        // caller's saved buffer holds the packages, states and Unew)
        auto takeb = [&](size_t bytes) { size_t o = off; off += align256(bytes); return o; };
        if (for_backward == 2) {
            L.dSo_b = takeb(slots * dk * dv * 2);
            L.dUn_b = takeb(slots * C * dv * 2);
            L.total = off;
            return L;
        }
        L.coop_bytes = coop::workspace_bytes(g, device_sms());
        L.coop = takeb(L.coop_bytes);
        L.keep = takeb(slots * coop::package_layout(g).stride);
        L.Sin_b = takeb(slots * dk * dv * 2);
        L.dSo_b = takeb(slots * dk * dv * 2);
        L.Un_b = takeb(slots * C * dv * 2);
        L.dUn_b = takeb(slots * C * dv * 2);
        L.total = off;
        return L;
    }
    L.Kn = take(slots * C * dk);
    L.Qn = take(slots * C * dk);
    L.W = take(slots * C * dk);
    L.U = take(slots * C * dv);
    L.Unew = take(slots * C * dv);
    L.gam = take(slots * C);
    L.eb = take(slots * C);
    L.Sin = take(slots * dk * dv);
    L.P = take(slots * C * C);
    if (for_backward) {
        L.aux = take(slots * (4 * C + 4));
        L.M3 = take(slots * 3 * C * C);
        L.dSo = take(slots * dk * dv);
        L.dUn = take(slots * C * dv);
        L.dQ = take(slots * C * dk);
        L.dK = take(slots * C * dk);
        L.dW = take(slots * C * dk);
    }
    (void)s;
    L.total = off;
    return L;
}

gen::Ws general_ws(const Layout &L, char *base)
{
    gen::Ws w;
    memset(&w, 0, sizeof(w));
    auto F = [&](size_t o) { return o ? (float *)(base + o) : (float *)nullptr; };
    w.Kn = F(L.Kn); w.Qn = F(L.Qn); w.W = F(L.W); w.U = F(L.U); w.Unew = F(L.Unew);
    w.gam = F(L.gam); w.eb = F(L.eb); w.Sin = F(L.Sin); w.dSo = F(L.dSo); w.dUn = F(L.dUn);
    w.dQ = F(L.dQ); w.dK = F(L.dK); w.dW = F(L.dW);
    w.P = F(L.P); w.aux = F(L.aux); w.M3 = F(L.M3);
    if (L.dSo_b) {
        auto B = [&](size_t o) { return (__nv_bfloat16 *)(base + o); };
        w.dSo_b = B(L.dSo_b); w.dUn_b = B(L.dUn_b);
    }
    if (L.keep) {
        auto B = [&](size_t o) { return (__nv_bfloat16 *)(base + o); };
        w.keep = (uint8_t *)(base + L.keep);
        w.coop_ws = base + L.coop;
        w.coop_bytes = L.coop_bytes;
        w.Sin_b = B(L.Sin_b); w.dSo_b = B(L.dSo_b); w.Un_b = B(L.Un_b); w.dUn_b = B(L.dUn_b);
    }
    return w;
}

// The saved buffer of gdn_chunk_fwd_save / gdn_chunk_bwd_saved: every chunk's
// package, then S_in and Unew in bf16 (offsets into the buffer; total 0 when the
// shape has no such path).
struct Saved {
    size_t keep, sin, unew, total;
};

Saved saved_layout(const Geo &g, int dtype)
{
    Saved r{0, 0, 0, 0};
    if (!gen::bwd_uses_coop(g, dtype)) return r;
    const size_t slots = (size_t)g.NC * g.H;
    size_t off = 0;
    r.keep = off; off += align256(slots * coop::package_layout(g).stride);
    r.sin = off; off += align256(slots * g.dk * g.dv * 2);
    r.unew = off; off += align256(slots * g.C * g.dv * 2);
    r.total = off;
    return r;
}

// First chunk slot of every packed sequence; flags malformed offsets (which are
// then treated as empty sequences) in the status word.
__global__ void k_cstart(const int32_t *cu, int N, int T, int C, int32_t *cstart, uint32_t *status)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    bool ok = cu[0] == 0 && cu[N] == T;
    for (int s = 0; s < N && ok; ++s) ok = cu[s + 1] >= cu[s];
    int acc = 0;
    cstart[0] = 0;
    for (int s = 0; s < N; ++s) {
        int L = ok ? cu[s + 1] - cu[s] : 0;
        acc += (L + C - 1) / C;
        cstart[s + 1] = acc;
    }
    if (!ok) raise_status(status, kStatusBadOffsets);
}

// GDN_FORCE_GENERAL=1 in the environment routes every call to the general fp32
// kernels (used by the tests to compare the two kernel families).
bool force_general()
{
    const char *e = getenv("GDN_FORCE_GENERAL");
    return e && e[0] && e[0] != '0';
}

// The cooperative forward is used where the device supports it, unless
// GDN_FUSED_PER_ITEM=1 asks for the one-CTA-per-(sequence, head) fused kernel.
bool use_coop()
{
    const char *e = getenv("GDN_FUSED_PER_ITEM");
    if (e && e[0] && e[0] != '0') return false;
    return coop::available();
}

// The forward a call takes: the cooperative kernel (bf16, d_k = d_v = 128 with
// C = 64 or 32, d_k = d_v = 256 with C = 32) where the device runs it and
// allow_coop holds, else the one-CTA-per-item fused kernel (bf16, d 128, C 64),
// else the general kernels.  honour_env = false ignores GDN_FORCE_GENERAL (the
// allocation-free entry point serves the fused-kernel shapes whatever the
// environment says).
Fwd fwd_kind(const dn_shape *s, const Geo &g, int for_backward, bool allow_coop, bool honour_env = true)
{
    if (for_backward || (honour_env && force_general())) return Fwd::General;
    if (allow_coop && use_coop() && coop::supports(g, s->dtype)) return Fwd::Coop;
    if (fast::supports(g, s->dtype)) return Fwd::PerItem;
    return Fwd::General;
}

dn_status begin_call(const dn_shape *s, Geo &g, int for_backward, void *ws, size_t ws_bytes,
                     cudaStream_t st, Layout &L, Fwd &kind, bool allow_coop, bool honour_env = true,
                     bool clear_status = true)
{
    kind = fwd_kind(s, g, for_backward, allow_coop, honour_env);
    L = make_layout(g, s, for_backward, kind);
    if (!ws || !is_aligned16(ws)) return DN_ERR_WORKSPACE;
    if (ws_bytes < L.total) return DN_ERR_WORKSPACE;
    char *base = (char *)ws;
    g.status = (uint32_t *)(base + L.status);
    if (clear_status && cudaMemsetAsync(base + L.status, 0, sizeof(uint32_t), st) != cudaSuccess)
        return DN_ERR_CUDA;
    if (g.varlen) {
        g.cstart = (const int32_t *)(base + L.cstart);
        k_cstart<<<1, 32, 0, st>>>(g.cu, g.N, g.T, g.C, (int32_t *)(base + L.cstart),
                                   (uint32_t *)(base + L.status));
        if (cudaPeekAtLastError() != cudaSuccess) return DN_ERR_CUDA;
    }
    return DN_OK;
}

dn_status fwd_impl(const dn_shape *s, const void *q, const void *k, const void *v,
                   const void *beta, const float *gate, const float *h0, void *o, float *hT,
                   void *ws, size_t ws_bytes, void *stream, bool allow_coop = true,
                   bool honour_env = true, const coop::Emit *emit = nullptr, bool clear_status = true)
{
    Geo g;
    dn_status rc = check_shape(s, &g);
    if (rc != DN_OK) return rc;
    const bool any = g.T > 0;
    if (any && (!q || !k || !v || !beta || !o)) return DN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, beta, gate, h0, o, hT};
    for (const void *p : ptrs)
        if (p && !is_aligned16(p)) return DN_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    Layout L;
    Fwd kind;
    if (emit && fwd_kind(s, g, 0, allow_coop, honour_env) != Fwd::Coop) return DN_ERR_UNSUPPORTED;
    if ((rc = begin_call(s, g, 0, ws, ws_bytes, st, L, kind, allow_coop, honour_env, clear_status)) != DN_OK)
        return rc;
    char *base = (char *)ws;
    cudaError_t e;
    if (kind == Fwd::Coop) {
        e = coop::fwd(g, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                      (const __nv_bfloat16 *)v, (const __nv_bfloat16 *)beta, gate, h0,
                      (__nv_bfloat16 *)o, hT, base + L.fast, ws_bytes - L.fast,
                      (uint32_t *)(base + L.status), st, emit);
    } else if (kind == Fwd::PerItem) {
        e = fast::fwd(g, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                      (const __nv_bfloat16 *)v, (const __nv_bfloat16 *)beta, gate, h0,
                      (__nv_bfloat16 *)o, hT, base + L.fast, (uint32_t *)(base + L.status), st);
    } else {
        gen::Ws w = general_ws(L, base);
        if (s->dtype == DN_F32)
            e = gen::fwd<float>(g, (const float *)q, (const float *)k, (const float *)v,
                                (const float *)beta, gate, h0, (float *)o, hT, w, st);
        else
            e = gen::fwd<__nv_bfloat16>(g, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                                        (const __nv_bfloat16 *)v, (const __nv_bfloat16 *)beta,
                                        gate, h0, (__nv_bfloat16 *)o, hT, w, st);
    }
    return e == cudaSuccess ? DN_OK : DN_ERR_CUDA;
}

// Synchronises `st`, then reads the status word at device address `word_dev`,
// clears it if it is set, and maps its bits to a status code (a timeout first,
// then malformed packed offsets, then a log-gate outside its domain).
dn_status read_status_word(void *word_dev, cudaStream_t st)
{
    if (cudaStreamSynchronize(st) != cudaSuccess) return DN_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, word_dev, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DN_ERR_CUDA;
    if (word == 0) return DN_OK;
    if (cudaMemset(word_dev, 0, sizeof(word)) != cudaSuccess) return DN_ERR_CUDA;
    if (word & kStatusTimeout) return DN_ERR_TIMEOUT;
    if (word & kStatusBadOffsets) return DN_ERR_INVALID_ARG;
    return DN_ERR_DOMAIN;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

size_t dn_workspace_size(const dn_shape *shape, int for_backward)
{
    Geo g;
    if (check_shape(shape, &g) != DN_OK) return 0;
    if (for_backward == 2 && !gen::bwd_uses_coop(g, shape->dtype)) return 0;
    return make_layout(g, shape, for_backward, fwd_kind(shape, g, for_backward, true)).total;
}

int dn_uses_fast_path(const dn_shape *shape, int for_backward)
{
    Geo g;
    if (check_shape(shape, &g) != DN_OK) return -1;
    return fwd_kind(shape, g, for_backward, true) != Fwd::General ? 1 : 0;
}

int dn_plan(const dn_shape *shape, int for_backward, int *kernels)
{
    Geo g;
    if (check_shape(shape, &g) != DN_OK) return -1;
    const int offsets = g.varlen ? 1 : 0;   // k_cstart
    int path, n;
    if (for_backward == 2) {
        // gdn_chunk_bwd_saved: k_bscan_pk, k_bwd_tc (+ k_cstart)
        if (!gen::bwd_uses_coop(g, shape->dtype)) return -1;
        path = DN_PATH_GENERAL;
        n = 2 + offsets;
    } else if (for_backward) {
        path = DN_PATH_GENERAL;
        // k_coop_fwd (+ k_plan), k_bscan_pk, k_bwd_tc; or k_prep, k_scan, k_bscan, then
        // k_bwd_tc (tcgen05) or k_bbig, k_bchunk, k_bgrad (the entry point requires the
        // 16-byte pointer alignment the tcgen05 kernel needs)
        const void *aligned = (const void *)(uintptr_t)256;
        if (gen::bwd_uses_coop(g, shape->dtype))
            n = 3 + 2 * offsets;
        else
            n = (gen::bwd_uses_tc(g, shape->dtype, aligned, aligned, aligned, aligned) ? 4 : 6) + offsets;
    } else if (fwd_kind(shape, g, 0, true) == Fwd::General) {
        path = DN_PATH_GENERAL;
        n = 3 + offsets;                    // k_prep, k_scan, k_out
    } else if (fwd_kind(shape, g, 0, true) == Fwd::Coop) {
        path = DN_PATH_COOP;
        n = 1 + 2 * offsets;                // k_coop_fwd (+ k_cstart, k_plan)
    } else {
        path = DN_PATH_FUSED;
        n = 1 + 2 * offsets;                // k_fast_fwd (+ k_cstart, k_order)
    }
    if (kernels) *kernels = n;
    return path;
}

dn_status dn_chunk_fwd(const dn_shape *shape, const void *q, const void *k, const void *v,
                       const void *beta, const float *h0, void *o, float *hT, void *ws,
                       size_t ws_bytes, void *stream)
{
    return fwd_impl(shape, q, k, v, beta, nullptr, h0, o, hT, ws, ws_bytes, stream);
}

dn_status gdn_chunk_fwd(const dn_shape *shape, const void *q, const void *k, const void *v,
                        const void *beta, const float *g, const float *h0, void *o, float *hT,
                        void *ws, size_t ws_bytes, void *stream)
{
    return fwd_impl(shape, q, k, v, beta, g, h0, o, hT, ws, ws_bytes, stream);
}

}  // extern "C"

namespace gdn {
namespace {
// gdn_chunk_bwd (saved == NULL) and gdn_chunk_bwd_saved
dn_status bwd_impl(const dn_shape *shape, const void *q, const void *k, const void *v,
                   const void *beta, const float *gate, const float *h0, const void *dO,
                   const float *dhT, void *dq, void *dk, void *dv, void *dbeta, float *dg,
                   float *dh0, void *ws, size_t ws_bytes, void *stream, void *saved,
                   size_t saved_bytes)
{
    Geo g;
    dn_status rc = check_shape(shape, &g);
    if (rc != DN_OK) return rc;
    if (dg && !gate) return DN_ERR_INVALID_ARG;
    if (g.T > 0 && (!q || !k || !v || !beta || !dO || !dq || !dk || !dv || !dbeta))
        return DN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, beta, gate, h0, dO, dhT, dq, dk, dv, dbeta, dg, dh0, saved};
    for (const void *p : ptrs)
        if (p && !is_aligned16(p)) return DN_ERR_INVALID_ARG;
    Saved sv{0, 0, 0, 0};
    if (saved) {
        sv = saved_layout(g, shape->dtype);
        if (sv.total == 0) return DN_ERR_UNSUPPORTED;
        if (saved_bytes < sv.total) return DN_ERR_INVALID_ARG;
    }
    cudaStream_t st = (cudaStream_t)stream;
    Layout L;
    Fwd kind;
    if ((rc = begin_call(shape, g, saved ? 2 : 1, ws, ws_bytes, st, L, kind, false)) != DN_OK) return rc;
    gen::Ws w = general_ws(L, (char *)ws);
    if (saved) {
        char *sb = (char *)saved;
        w.keep = (uint8_t *)(sb + sv.keep);
        w.Sin_b = (__nv_bfloat16 *)(sb + sv.sin);
        w.Un_b = (__nv_bfloat16 *)(sb + sv.unew);
        w.saved = true;
    }
    cudaError_t e;
    if (shape->dtype == DN_F32)
        e = gen::bwd<float>(g, (const float *)q, (const float *)k, (const float *)v,
                            (const float *)beta, gate, h0, (const float *)dO, dhT, (float *)dq,
                            (float *)dk, (float *)dv, (float *)dbeta, dg, dh0, w, st);
    else
        e = gen::bwd<__nv_bfloat16>(
            g, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
            (const __nv_bfloat16 *)beta, gate, h0, (const __nv_bfloat16 *)dO, dhT,
            (__nv_bfloat16 *)dq, (__nv_bfloat16 *)dk, (__nv_bfloat16 *)dv,
            (__nv_bfloat16 *)dbeta, dg, dh0, w, st);
    return e == cudaSuccess ? DN_OK : DN_ERR_CUDA;
}
}  // namespace
}  // namespace gdn

extern "C" {

dn_status gdn_chunk_bwd(const dn_shape *shape, const void *q, const void *k, const void *v,
                        const void *beta, const float *gate, const float *h0, const void *dO,
                        const float *dhT, void *dq, void *dk, void *dv, void *dbeta, float *dg,
                        float *dh0, void *ws, size_t ws_bytes, void *stream)
{
    return bwd_impl(shape, q, k, v, beta, gate, h0, dO, dhT, dq, dk, dv, dbeta, dg, dh0, ws, ws_bytes,
                    stream, nullptr, 0);
}

size_t dn_saved_size(const dn_shape *shape)
{
    Geo g;
    if (check_shape(shape, &g) != DN_OK) return 0;
    if (fwd_kind(shape, g, 0, true) != Fwd::Coop) return 0;
    return saved_layout(g, shape->dtype).total;
}

dn_status gdn_chunk_fwd_save(const dn_shape *shape, const void *q, const void *k, const void *v,
                             const void *beta, const float *g, const float *h0, void *o, float *hT,
                             void *saved, size_t saved_bytes, void *ws, size_t ws_bytes, void *stream)
{
    Geo geo;
    dn_status rc = check_shape(shape, &geo);
    if (rc != DN_OK) return rc;
    const Saved sv = saved_layout(geo, shape->dtype);
    if (sv.total == 0 || fwd_kind(shape, geo, 0, true) != Fwd::Coop) return DN_ERR_UNSUPPORTED;
    if (!saved || !is_aligned16(saved) || saved_bytes < sv.total) return DN_ERR_INVALID_ARG;
    char *sb = (char *)saved;
    const coop::Emit em{(uint8_t *)(sb + sv.keep), (__nv_bfloat16 *)(sb + sv.sin),
                        (__nv_bfloat16 *)(sb + sv.unew)};
    return fwd_impl(shape, q, k, v, beta, g, h0, o, hT, ws, ws_bytes, stream, true, true, &em);
}

dn_status gdn_chunk_bwd_saved(const dn_shape *shape, const void *q, const void *k, const void *v,
                              const void *beta, const float *gate, const void *dO, const float *dhT,
                              const void *saved, size_t saved_bytes, void *dq, void *dk, void *dv,
                              void *dbeta, float *dg, float *dh0, void *ws, size_t ws_bytes,
                              void *stream)
{
    if (!saved) return DN_ERR_INVALID_ARG;
    return bwd_impl(shape, q, k, v, beta, gate, nullptr, dO, dhT, dq, dk, dv, dbeta, dg, dh0, ws, ws_bytes,
                    stream, const_cast<void *>(saved), saved_bytes);
}

dn_status gdn_decode_step(const dn_shape *shape, const void *q, const void *k, const void *v,
                          const void *beta, const float *g, const float *state_in, float *state_out,
                          void *o, void *stream)
{
    Geo gg;
    dn_status rc = check_shape(shape, &gg);
    if (rc != DN_OK) return rc;
    if (shape->cu_seqlens || shape->T != 1) return DN_ERR_INVALID_ARG;
    if (!q || !k || !v || !beta || !state_out || !o) return DN_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, beta, g, state_in, state_out, o};
    for (const void *p : ptrs)
        if (p && ((uintptr_t)p & 3u)) return DN_ERR_INVALID_ARG;
    dec::Args a;
    a.N = shape->B; a.H = shape->H; a.dk = shape->dk; a.dv = shape->dv;
    a.l2norm = shape->qk_l2norm != 0; a.scale = shape->scale; a.eps = shape->eps;
    a.longhorn = shape->beta_mode == DN_BETA_LONGHORN;
    a.gate = g; a.state_in = state_in; a.state_out = state_out;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (shape->dtype == DN_F32)
        e = dec::step<float>(a, (const float *)q, (const float *)k, (const float *)v,
                             (const float *)beta, (float *)o, st);
    else
        e = dec::step<__nv_bfloat16>(a, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                                     (const __nv_bfloat16 *)v, (const __nv_bfloat16 *)beta,
                                     (__nv_bfloat16 *)o, st);
    return e == cudaSuccess ? DN_OK : DN_ERR_CUDA;
}

dn_status dn_state_affine(const float *A, const float *S, const float *B, float *out, int count,
                          int dk, int dv, void *stream)
{
    if (count < 0 || dk < 1 || dv < 1 || dk > kMaxD || dv > kMaxD) return DN_ERR_INVALID_ARG;
    if (count == 0) return DN_OK;
    if (count > 65535) return DN_ERR_UNSUPPORTED;
    if (!A || !S || !out) return DN_ERR_INVALID_ARG;
    const void *ptrs[] = {A, S, B, out};
    for (const void *p : ptrs)
        if (p && ((uintptr_t)p & 3u)) return DN_ERR_INVALID_ARG;
    // out may not overlap A or S (other CTAs still read them while it is written)
    const uintptr_t o0 = (uintptr_t)out, o1 = o0 + (size_t)count * dk * dv * sizeof(float);
    const uintptr_t a0 = (uintptr_t)A, a1 = a0 + (size_t)count * dk * dk * sizeof(float);
    const uintptr_t s0 = (uintptr_t)S, s1 = s0 + (size_t)count * dk * dv * sizeof(float);
    if ((o0 < a1 && a0 < o1) || (o0 < s1 && s0 < o1)) return DN_ERR_INVALID_ARG;
    return aff::state_affine(A, S, B, out, count, dk, dv, (cudaStream_t)stream) == cudaSuccess ? DN_OK
                                                                                             : DN_ERR_CUDA;
}

size_t dn_host_arena_size(const dn_shape *s, int gated, int with_h0)
{
    Geo g;
    if (check_shape(s, &g) != DN_OK) return 0;
    const size_t es = s->dtype == DN_BF16 ? 2 : 4;
    const size_t tok = (size_t)g.B * g.H * g.T;
    const size_t st = (size_t)g.N * g.H * g.dk * g.dv * sizeof(float);
    size_t n = 0;
    n += align256(tok * g.dk * es) * 2;           // q, k
    n += align256(tok * g.dv * es) * 2;           // v, o
    n += align256(tok * es);                      // beta
    if (gated) n += align256(tok * sizeof(float));
    if (with_h0) n += align256(st);
    n += align256(st);                            // hT
    n += 2 * align256(st);                        // the state between time segments (two, in turn)
    return n;
}

// ---------------------------------------------------------------------------
// The host entry point's pipeline.  Fixed-length input of at least 32 chunks is cut
// along time into segments of whole chunks; the copies of segment i + 1 into the
// arena overlap segment i's forward, and segment i's output goes back to the host
// while later segments compute.  Each segment is a forward over [B][H][Ts] with the
// state handed on through the arena, so the host link (the call's bound: about 0.2 TB/s
// either way, the two directions concurrently) is busy throughout instead of in turns.
// At most four segments: with eight, the strided copies of the two directions (rows of
// 256 KB for T = 8192, d = 128) no longer overlapped on a GB300 (measured).
namespace {
CUcontext current_context();

constexpr int kMaxSegments = 4;
constexpr int kMinSegmentChunks = 16;
constexpr int kMaxPipeDevices = 64;

struct HostPipe {
    CUcontext ctx;
    cudaStream_t in, out;                 // copies to the arena, copies back
    cudaEvent_t fork, join;
    cudaEvent_t landed[kMaxSegments];     // segment i's inputs are in the arena
    cudaEvent_t done[kMaxSegments];       // segment i's forward has completed
};
std::mutex g_pipe_mu;
HostPipe g_pipe[kMaxPipeDevices];

// Segments of the time axis for the pipelined host path (1: no pipeline).
int host_segments(const Geo &g)
{
    if (g.varlen || g.T <= 0) return 1;
    const int nch = (g.T + g.C - 1) / g.C;
    int n = nch / kMinSegmentChunks;
    return n < 1 ? 1 : (n > kMaxSegments ? kMaxSegments : n);
}

// Head groups for the pipelined host path with packed input (1: none).  Packed tensors
// are [H][T] rows, so a group of heads is one contiguous block of each, and heads are
// independent: each group is a forward over its heads, its copies overlapping the
// others' compute.  (Packed input cannot be cut along time here: its sequence bounds are
// on the device.)  A group's beta rows must start 16-byte aligned in the arena.
int host_head_groups(const Geo &g)
{
    if (!g.varlen || g.T <= 0 || (g.T + g.C - 1) / g.C < 2 * kMinSegmentChunks) return 1;
    for (int G = kMaxSegments; G >= 2; --G)
        if (g.H % G == 0 && ((size_t)g.T * (g.H / G)) % 8 == 0) return G;
    return 1;
}

// The device's streams and events for the pipeline, made on first use in each context.
// Called with g_pipe_mu held.
HostPipe *host_pipe()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxPipeDevices) return nullptr;
    HostPipe &hp = g_pipe[dev];
    const CUcontext ctx = current_context();
    if (hp.in && hp.ctx == ctx) return &hp;
    HostPipe fresh{};
    bool ok = cudaStreamCreateWithFlags(&fresh.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&fresh.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&fresh.fork, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&fresh.join, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kMaxSegments; ++i)
        ok = cudaEventCreateWithFlags(&fresh.landed[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&fresh.done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return nullptr;
    fresh.ctx = ctx;
    hp = fresh;
    return &hp;
}

// [rows][width] bytes out of (or into) rows of `pitch` bytes, as one 2D copy.
bool copy2d(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width, size_t rows,
            cudaMemcpyKind kind, cudaStream_t st)
{
    if (width == 0 || rows == 0) return true;
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, st) == cudaSuccess;
}

}  // namespace

dn_status gdn_chunk_fwd_host(const dn_shape *s, const void *q, const void *k, const void *v,
                             const void *beta, const float *gate, const float *h0, void *o,
                             float *hT, void *arena, size_t arena_bytes, void *ws,
                             size_t ws_bytes, void *stream)
{
    Geo g;
    dn_status rc = check_shape(s, &g);
    if (rc != DN_OK) return rc;
    if (!arena || !is_aligned16(arena)) return DN_ERR_INVALID_ARG;
    if (arena_bytes < dn_host_arena_size(s, gate != nullptr, h0 != nullptr)) return DN_ERR_INVALID_ARG;
    if (g.T > 0 && (!q || !k || !v || !beta || !o)) return DN_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t es = s->dtype == DN_BF16 ? 2 : 4;
    const size_t tok = (size_t)g.B * g.H * g.T;
    const size_t sbytes = (size_t)g.N * g.H * g.dk * g.dv * sizeof(float);
    char *p = (char *)arena;
    auto carve = [&](size_t bytes) { char *r = p; p += align256(bytes); return r; };
    char *dq = carve(tok * g.dk * es), *dk = carve(tok * g.dk * es);
    char *dvv = carve(tok * g.dv * es), *dout = carve(tok * g.dv * es);
    char *db = carve(tok * es);
    char *dgate = gate ? carve(tok * sizeof(float)) : nullptr;
    char *dh0 = h0 ? carve(sbytes) : nullptr;
    char *dhT = carve(sbytes);
    char *dst2[2] = {carve(sbytes), carve(sbytes)};   // the state between segments, in turn
    const int nseg = host_segments(g);
    if (nseg > 1) {
        // segments of lch whole chunks: inputs of segment i land in its part of the arena
        // (contiguous [B][H][Ts] rows, one strided copy per tensor), then its forward runs on
        // `stream` from the state segment i - 1 left, then its output goes back
        std::lock_guard<std::mutex> lock(g_pipe_mu);
        HostPipe *hp = host_pipe();
        if (!hp) return DN_ERR_CUDA;
        const int nch = (g.T + g.C - 1) / g.C;
        const int lch = (nch + nseg - 1) / nseg;
        const size_t tseg = (size_t)lch * g.C;
        const int S = (int)(((size_t)g.T + tseg - 1) / tseg);
        const size_t BH = (size_t)g.B * g.H, T = (size_t)g.T;
        const size_t kb = (size_t)g.dk * es, vb = (size_t)g.dv * es, gb = sizeof(float);
        const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
        if (cudaEventRecord(hp->fork, st) != cudaSuccess || cudaStreamWaitEvent(hp->in, hp->fork, 0) != cudaSuccess ||
            cudaStreamWaitEvent(hp->out, hp->fork, 0) != cudaSuccess)
            return DN_ERR_CUDA;
        if (dh0 && cudaMemcpyAsync(dh0, h0, sbytes, H2D, hp->in) != cudaSuccess) return DN_ERR_CUDA;
        for (int i = 0; i < S; ++i) {
            const size_t t0 = (size_t)i * tseg, ts = T - t0 < tseg ? T - t0 : tseg;
            const size_t off = BH * t0;   // tokens of the earlier segments in each arena tensor
            const bool ok =
                copy2d(dq + off * kb, ts * kb, (const char *)q + t0 * kb, T * kb, ts * kb, BH, H2D, hp->in) &&
                copy2d(dk + off * kb, ts * kb, (const char *)k + t0 * kb, T * kb, ts * kb, BH, H2D, hp->in) &&
                copy2d(dvv + off * vb, ts * vb, (const char *)v + t0 * vb, T * vb, ts * vb, BH, H2D, hp->in) &&
                copy2d(db + off * es, ts * es, (const char *)beta + t0 * es, T * es, ts * es, BH, H2D, hp->in) &&
                (!dgate ||
                 copy2d(dgate + off * gb, ts * gb, (const char *)gate + t0 * gb, T * gb, ts * gb, BH, H2D, hp->in));
            if (!ok || cudaEventRecord(hp->landed[i], hp->in) != cudaSuccess ||
                cudaStreamWaitEvent(st, hp->landed[i], 0) != cudaSuccess)
                return DN_ERR_CUDA;
            dn_shape seg = *s;
            seg.T = (int32_t)ts;
            const float *h0i = i == 0 ? (const float *)dh0 : (const float *)dst2[(i - 1) & 1];
            float *hTi = i == S - 1 ? (hT ? (float *)dhT : nullptr) : (float *)dst2[i & 1];
            // the status word is cleared by the first segment only, so that it keeps what any
            // segment flags
            rc = fwd_impl(&seg, dq + off * kb, dk + off * kb, dvv + off * vb, db + off * es,
                          dgate ? (const float *)(dgate + off * gb) : nullptr, h0i, dout + off * vb, hTi, ws,
                          ws_bytes, stream, true, true, nullptr, i == 0);
            if (rc != DN_OK) return rc;
            if (cudaEventRecord(hp->done[i], st) != cudaSuccess || cudaStreamWaitEvent(hp->out, hp->done[i], 0) != cudaSuccess)
                return DN_ERR_CUDA;
            if (!copy2d((char *)o + t0 * vb, T * vb, dout + off * vb, ts * vb, ts * vb, BH, D2H, hp->out))
                return DN_ERR_CUDA;
        }
        if (hT && cudaMemcpyAsync(hT, dhT, sbytes, D2H, hp->out) != cudaSuccess) return DN_ERR_CUDA;
        if (cudaEventRecord(hp->join, hp->out) != cudaSuccess || cudaStreamWaitEvent(st, hp->join, 0) != cudaSuccess)
            return DN_ERR_CUDA;
        return DN_OK;
    }
    const int ngrp = host_head_groups(g);
    if (ngrp > 1) {
        // packed input: group i is heads [i Hg, (i + 1) Hg), contiguous in every [H][T] tensor;
        // its states are [N][Hg][dk][dv] in the arena, strided [N][H][dk][dv] on the host
        std::lock_guard<std::mutex> lock(g_pipe_mu);
        HostPipe *hp = host_pipe();
        if (!hp) return DN_ERR_CUDA;
        const int Hg = g.H / ngrp;
        const size_t per = (size_t)Hg * g.T;   // token rows of a group
        const size_t kb = (size_t)g.dk * es, vb = (size_t)g.dv * es, gb = sizeof(float);
        const size_t srow = (size_t)g.dk * g.dv * sizeof(float);   // one (sequence, head) state
        const size_t sgrp = (size_t)g.N * Hg * srow;
        const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
        if (cudaEventRecord(hp->fork, st) != cudaSuccess || cudaStreamWaitEvent(hp->in, hp->fork, 0) != cudaSuccess ||
            cudaStreamWaitEvent(hp->out, hp->fork, 0) != cudaSuccess)
            return DN_ERR_CUDA;
        for (int i = 0; i < ngrp; ++i) {
            const size_t t0 = per * i;
            const bool ok =
                cudaMemcpyAsync(dq + t0 * kb, (const char *)q + t0 * kb, per * kb, H2D, hp->in) == cudaSuccess &&
                cudaMemcpyAsync(dk + t0 * kb, (const char *)k + t0 * kb, per * kb, H2D, hp->in) == cudaSuccess &&
                cudaMemcpyAsync(dvv + t0 * vb, (const char *)v + t0 * vb, per * vb, H2D, hp->in) == cudaSuccess &&
                cudaMemcpyAsync(db + t0 * es, (const char *)beta + t0 * es, per * es, H2D, hp->in) == cudaSuccess &&
                (!dgate || cudaMemcpyAsync(dgate + t0 * gb, (const char *)gate + t0 * gb, per * gb, H2D, hp->in) ==
                               cudaSuccess) &&
                (!dh0 || copy2d(dh0 + i * sgrp, Hg * srow, (const char *)h0 + (size_t)i * Hg * srow, (size_t)g.H * srow,
                                Hg * srow, (size_t)g.N, H2D, hp->in));
            if (!ok || cudaEventRecord(hp->landed[i], hp->in) != cudaSuccess ||
                cudaStreamWaitEvent(st, hp->landed[i], 0) != cudaSuccess)
                return DN_ERR_CUDA;
            dn_shape sub = *s;
            sub.H = Hg;
            // the status word is cleared by the first group only
            rc = fwd_impl(&sub, dq + t0 * kb, dk + t0 * kb, dvv + t0 * vb, db + t0 * es,
                          dgate ? (const float *)(dgate + t0 * gb) : nullptr, dh0 ? (const float *)(dh0 + i * sgrp) : nullptr,
                          dout + t0 * vb, hT ? (float *)(dhT + i * sgrp) : nullptr, ws, ws_bytes, stream, true, true,
                          nullptr, i == 0);
            if (rc != DN_OK) return rc;
            if (cudaEventRecord(hp->done[i], st) != cudaSuccess || cudaStreamWaitEvent(hp->out, hp->done[i], 0) != cudaSuccess)
                return DN_ERR_CUDA;
            if (cudaMemcpyAsync((char *)o + t0 * vb, dout + t0 * vb, per * vb, D2H, hp->out) != cudaSuccess ||
                (hT && !copy2d((char *)hT + (size_t)i * Hg * srow, (size_t)g.H * srow, dhT + i * sgrp, Hg * srow,
                               Hg * srow, (size_t)g.N, D2H, hp->out)))
                return DN_ERR_CUDA;
        }
        if (cudaEventRecord(hp->join, hp->out) != cudaSuccess || cudaStreamWaitEvent(st, hp->join, 0) != cudaSuccess)
            return DN_ERR_CUDA;
        return DN_OK;
    }
    struct { void *dst; const void *src; size_t n; } cp[] = {
        {dq, q, tok * g.dk * es}, {dk, k, tok * g.dk * es}, {dvv, v, tok * g.dv * es},
        {db, beta, tok * es}, {dgate, gate, tok * sizeof(float)}, {dh0, h0, sbytes}};
    for (auto &c : cp) {
        if (!c.dst || !c.src || c.n == 0) continue;
        if (cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return DN_ERR_CUDA;
    }
    rc = fwd_impl(s, dq, dk, dvv, db, (const float *)dgate, (const float *)dh0, dout,
                  (float *)dhT, ws, ws_bytes, stream);
    if (rc != DN_OK) return rc;
    if (o && tok && cudaMemcpyAsync(o, dout, tok * g.dv * es, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return DN_ERR_CUDA;
    if (hT && sbytes && cudaMemcpyAsync(hT, dhT, sbytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return DN_ERR_CUDA;
    return DN_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free forward.  The scratch it needs (the status word and, for
// packed input, the per-sequence chunk starts and longest-first order) lives in
// this file-scope array instead of a caller-provided workspace.  Every GPU that
// loads the library holds the array until the process exits.
constexpr size_t kNoAllocScratchBytes = 256 * 1024;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct NoAllocEntry {
    CUcontext ctx;   // context the address belongs to
    void *ptr;       // device address of g_noalloc_scratch in it
};
NoAllocEntry g_noalloc[kMaxDevices];

// The calling thread's current CUDA context (null if none), through the driver
// entry point the runtime hands out, so that the library links only cudart.
CUcontext current_context()
{
    typedef CUresult (*GetCurrent)(CUcontext *);
    static GetCurrent fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (GetCurrent)p;
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// Device address of the array on the current device.  It is looked up with
// cudaGetSymbolAddress, with that device current, on the first call on each
// device, and again whenever the device's context has changed since (after
// cudaDeviceReset the module is loaded anew and the array can move).  Returns
// null on failure.
void *noalloc_scratch()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoAllocEntry &e = g_noalloc[dev];
    if (!e.ptr || !ctx || e.ctx != ctx) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        e.ptr = ptr;
        e.ctx = current_context();   // current now, if it was not before the lookup
    }
    return e.ptr;
}
}  // namespace

dn_status gdn_chunk_fwd_noalloc(const dn_shape *shape, const void *q, const void *k, const void *v,
                                const void *beta, const float *g, const float *h0, void *o,
                                float *hT, void *stream)
{
    Geo geo;
    dn_status rc = check_shape(shape, &geo);
    if (rc != DN_OK) return rc;
    if (fwd_kind(shape, geo, 0, false, false) != Fwd::PerItem) return DN_ERR_UNSUPPORTED;
    if (make_layout(geo, shape, 0, Fwd::PerItem).total > kNoAllocScratchBytes) return DN_ERR_WORKSPACE;
    void *ws = noalloc_scratch();
    if (!ws) return DN_ERR_CUDA;
    // the one-CTA-per-item fused kernel: its scratch fits the static array
    return fwd_impl(shape, q, k, v, beta, g, h0, o, hT, ws, kNoAllocScratchBytes, stream, false, false);
}

dn_status dn_noalloc_status(void *stream)
{
    void *ws = noalloc_scratch();
    if (!ws) return DN_ERR_CUDA;
    // the status word is the first word of the static array (the workspace layout's header)
    return read_status_word(ws, (cudaStream_t)stream);
}

dn_status dn_device_status(void *ws, void *stream)
{
    if (!ws) return DN_ERR_WORKSPACE;
    return read_status_word(ws, (cudaStream_t)stream);
}

const char *dn_status_str(dn_status s)
{
    switch (s) {
    case DN_OK: return "ok";
    case DN_ERR_INVALID_ARG: return "invalid argument";
    case DN_ERR_UNSUPPORTED: return "unsupported shape or option";
    case DN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DN_ERR_CUDA: return "CUDA error";
    case DN_ERR_TIMEOUT: return "a bounded device wait ran out";
    case DN_ERR_DOMAIN: return "an input value outside its documented domain (log-gate g > 0)";
    }
    return "unknown status";
}

}  // extern "C"
