/*
 * gdn.h — C ABI of libgdn_gb300.so: chunkwise-parallel DeltaNet and Gated
 * DeltaNet on one NVIDIA GB300 (sm_103a).
 *
 * The operation (per sequence and head, state S stored d_k x d_v, key index
 * outer):
 *     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 * — "Gated DeltaNet: Improving Mamba2 with Delta Rule", rebuttal Table 1,
 * rows "DeltaNet" (alpha_t = 1) and "Gated DeltaNet" (there written with the
 * d_v x d_k transpose, S_t = S_{t-1}(alpha_t(I - beta_t k_t k_t^T)) +
 * beta_t v_t k_t^T).  alpha_t = exp(g_t) for a per-token, per-head log-gate g.
 * q and k are L2-normalised per token inside the kernels when
 * shape->qk_l2norm is set: x / sqrt(sum x^2 + eps).
 *
 * The kernels evaluate it chunk by chunk ("Parallelizing Linear Transformers
 * with the Delta Rule over Sequence Length": WY representation of the
 * Householder-like products, chunkwise parallel form; GDN page: the same
 * algorithm extended with gating).  Per chunk of C tokens, with gamma the
 * within-chunk cumulative log-gate and D_ri = exp(gamma_r - gamma_i):
 *     T = (I + strict_lower(diag(beta)(K K^T o D)))^-1 diag(beta)
 *     W = T diag(exp gamma) K,  U = T V,  Unew = U - W S
 *     O = diag(exp gamma) Q S + lower(Q K^T o D) Unew
 *     S <- exp(gamma_C) S + (diag(exp(gamma_C - gamma)) K)^T Unew
 *
 * Layouts.  Token arrays are [B][H][T][d] row-major (time axis of one batch
 * row and head contiguous); beta, g are [B][H][T]; states are
 * [N][H][dk][dv] float32 where N = B, or the number of packed sequences.
 * Packed variable-length input: B == 1, T = total tokens,
 * shape->cu_seqlens = device int32 offsets [num_seqs + 1] (first 0, last T,
 * non-decreasing); chunks never cross a sequence boundary.
 *
 * Dtypes.  shape->dtype fixes q, k, v, beta, o (forward) and dO, dq, dk, dv,
 * dbeta (backward): DN_F32 (float) or DN_BF16 (bfloat16).  g, h0, hT, dhT,
 * dg, dh0 are always float32.  Arithmetic is float32 (bf16 tensor-core
 * operands with float32 accumulation on the bf16 fast path).
 *
 * Ownership.  The caller owns every buffer and the stream; the library
 * allocates nothing, keeps no state between calls and never synchronises
 * the stream (except dn_device_status, which says so).  All device pointers
 * must be 16-byte aligned.  Calls are asynchronous on `stream`
 * (a cudaStream_t; NULL = legacy default stream).
 *
 * Errors.  Every entry point returns a dn_status and never aborts or throws.
 * Argument errors are found on the host before anything is launched.  Launch
 * errors return DN_ERR_CUDA.  Every device-side wait in the kernels is
 * bounded; a wait that runs out records DN_ERR_TIMEOUT in the workspace's
 * status word, which dn_device_status reads back.  The same word records what
 * only the device can see in the inputs: malformed packed offsets
 * (DN_ERR_INVALID_ARG) and a log-gate g > 0 (DN_ERR_DOMAIN).  Each call clears
 * the word when it starts, so it describes the most recent call on it.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DN_OK = 0,
    DN_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad sizes or offsets */
    DN_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. dk > 256)     */
    DN_ERR_WORKSPACE = 3,     /* ws == NULL or ws_bytes < dn_workspace_size     */
    DN_ERR_CUDA = 4,          /* a CUDA call or kernel launch failed            */
    DN_ERR_TIMEOUT = 5,       /* a bounded device wait ran out (see above)      */
    DN_ERR_DOMAIN = 6         /* an input outside its domain: log-gate g > 0    */
} dn_status;

typedef enum { DN_F32 = 0, DN_BF16 = 1 } dn_dtype;

typedef struct {
    int32_t B, H, T;              /* batch rows, heads, tokens per row (packed: B = 1) */
    int32_t dk, dv;               /* head dims, 1..256 (tcgen05 kernels: 128)           */
    int32_t chunk;                /* C: 16, 32 or 64 (64 is the tuned size)             */
    int32_t dtype;                /* dn_dtype                                           */
    const int32_t *cu_seqlens;    /* device, [num_seqs + 1], or NULL for fixed length   */
    int32_t num_seqs;             /* packed sequences (ignored when cu_seqlens == NULL) */
    int32_t qk_l2norm;            /* 1: normalise q and k per token inside the kernels  */
    float scale;                  /* o = scale * S^T q                                  */
    float eps;                    /* normalisation epsilon (1e-6 is the default)        */
    int32_t beta_mode;            /* dn_beta_mode: how beta becomes the step size       */
} dn_shape;

/* The step size each token's update uses ("Gated DeltaNet" rebuttal, Table 1):
 *   DN_BETA_DELTA     beta_t as given (rows "DeltaNet" / "Gated DeltaNet");
 *   DN_BETA_LONGHORN  beta_t / (1 + beta_t k_t^T k_t), k_t the key the update
 *                     uses (after the normalisation when qk_l2norm = 1): row
 *                     "Longhorn" with its scalar beta.  The update is then the
 *                     minimiser of |S - alpha_t S_{t-1}|^2 + beta_t |S k_t - v_t|^2;
 *                     gradients (gdn_chunk_bwd) are with respect to the raw beta
 *                     and k through this map.
 * Any other value: DN_ERR_INVALID_ARG. */
typedef enum { DN_BETA_DELTA = 0, DN_BETA_LONGHORN = 1 } dn_beta_mode;

/* Bytes of device workspace the calls below need for `shape` (0 on bad
 * arguments).  for_backward = 1 sizes it for gdn_chunk_bwd, 2 for
 * gdn_chunk_bwd_saved (0 where the shape has no saved path). */
size_t dn_workspace_size(const dn_shape *shape, int for_backward);

/* DeltaNet forward (alpha = 1; Table 1 row "DeltaNet").
 *   q, k [B,H,T,dk], v [B,H,T,dv], beta [B,H,T]   (dtype)
 *   h0   [N,H,dk,dv] float32 initial state, NULL = zero
 *   o    [B,H,T,dv] (dtype) output
 *   hT   [N,H,dk,dv] float32 final state, NULL = not written
 *   ws   device workspace of ws_bytes >= dn_workspace_size(shape, 0)      */
dn_status dn_chunk_fwd(const dn_shape *shape, const void *q, const void *k, const void *v,
                       const void *beta, const float *h0, void *o, float *hT, void *ws,
                       size_t ws_bytes, void *stream);

/* Gated DeltaNet forward (Table 1 row "Gated DeltaNet"): as dn_chunk_fwd plus
 *   g [B,H,T] float32 log-gate, alpha = exp(g); g must be <= 0 (alpha <= 1).
 *   g == NULL is the same as g = 0 (alpha = 1).
 * A gate alpha in (0, 1] is a decay; the chunk form relies on it, through the
 * ratios exp(gamma_r - gamma_i) <= 1 inside a chunk and the state's pending
 * decay factor.  A value g > 0 is not rejected (the device would have to read g
 * before the launch) but flagged: the kernels set the status word and
 * dn_device_status returns DN_ERR_DOMAIN.  The result is still computed; it
 * follows the recurrence only while exp(sum of g over a chunk) and the growth
 * of the state stay inside float32 range.                                      */
dn_status gdn_chunk_fwd(const dn_shape *shape, const void *q, const void *k, const void *v,
                        const void *beta, const float *g, const float *h0, void *o,
                        float *hT, void *ws, size_t ws_bytes, void *stream);

/* Gated DeltaNet backward: gradients of L = <o, dO> + <hT, dhT>.
 * Recomputes the chunk states from q, k, v, beta, g, h0 (chunk states are
 * recomputed in the backward rather than kept — DeltaNet page, reply Q2).  For
 * bf16 with dk = dv = 128 and chunk 64 the recompute is a run of the cooperative
 * forward that also leaves every chunk's prepared operands and its state in the
 * workspace (dn_workspace_size(shape, 1) counts them: about 145 KB per chunk and
 * head); GDN_BWD_RECOMPUTE=1 or GDN_FORCE_GENERAL=1 recompute with the general
 * kernels instead.  A bounded wait that runs out in that run is reported like the
 * forward's (DN_ERR_TIMEOUT from dn_device_status).
 *   dO  [B,H,T,dv] (dtype), dhT [N,H,dk,dv] float32 or NULL (= 0)
 *   dq, dk [B,H,T,dk], dv [B,H,T,dv], dbeta [B,H,T]   (dtype), with respect to
 *   the raw q and k given (chained through the normalisation)
 *   dg  [B,H,T] float32 or NULL (not written; must be NULL when g is NULL)
 *   dh0 [N,H,dk,dv] float32 or NULL (not written)
 *   ws  >= dn_workspace_size(shape, 1) bytes                                   */
dn_status gdn_chunk_bwd(const dn_shape *shape, const void *q, const void *k, const void *v,
                        const void *beta, const float *g, const float *h0, const void *dO,
                        const float *dhT, void *dq, void *dk, void *dv, void *dbeta,
                        float *dg, float *dh0, void *ws, size_t ws_bytes, void *stream);

/* Training step without the backward's recompute (bf16, dk = dv = 128, chunk 64,
 * a device that runs the cooperative forward; DN_ERR_UNSUPPORTED otherwise, and
 * dn_saved_size returns 0).  gdn_chunk_fwd_save is gdn_chunk_fwd that also fills
 * `saved` (device, 16-byte aligned, >= dn_saved_size(shape) bytes: about 97 KB per
 * chunk of 64 tokens and head) with every chunk's prepared operands, the state
 * entering it and Unew, in bf16.  gdn_chunk_bwd_saved is gdn_chunk_bwd starting
 * from that buffer: no recompute, h0 not needed (it is inside the saved states);
 * the other arguments must be those of the forward call that filled it (the
 * library does not check).  Workspaces: dn_workspace_size(shape, 0) and
 * dn_workspace_size(shape, 2).  This keeps what the pages recompute (DeltaNet
 * page, reply Q2): it trades the saved buffer's memory for one forward pass. */
size_t dn_saved_size(const dn_shape *shape);
dn_status gdn_chunk_fwd_save(const dn_shape *shape, const void *q, const void *k, const void *v,
                             const void *beta, const float *g, const float *h0, void *o, float *hT,
                             void *saved, size_t saved_bytes, void *ws, size_t ws_bytes,
                             void *stream);
dn_status gdn_chunk_bwd_saved(const dn_shape *shape, const void *q, const void *k, const void *v,
                              const void *beta, const float *g, const void *dO, const float *dhT,
                              const void *saved, size_t saved_bytes, void *dq, void *dk, void *dv,
                              void *dbeta, float *dg, float *dh0, void *ws, size_t ws_bytes,
                              void *stream);

/* Recurrent decode step (one new token per sequence; the recurrence itself, as
 * in Table 1 of the Gated DeltaNet page, row "Gated DeltaNet", and the
 * Gated DeltaNet page's reply on decoding with a fixed-size state):
 *   S' = alpha (I - beta k k^T) S + beta k v^T,   o = scale S'^T q,
 * q, k normalised in the kernel when shape->qk_l2norm.  Shape: B = number of
 * sequences, H heads, T must be 1, dk, dv <= 256, cu_seqlens NULL; chunk is
 * ignored (any accepted value).  Layouts (dtype = shape->dtype unless noted):
 *   q, k [B,H,dk], v [B,H,dv], beta [B,H]; g [B,H] float32 log-gate or NULL
 *   (alpha = 1); state_in [B,H,dk,dv] float32 or NULL (zero state);
 *   state_out [B,H,dk,dv] float32, may be the same buffer as state_in (the
 *   update is then in place); o [B,H,dv].
 * Needs no workspace, allocates nothing, does not synchronise.  Errors:
 * DN_ERR_INVALID_ARG for a bad shape, T != 1, packed input, a missing buffer or
 * a pointer that is not 4-byte aligned; DN_ERR_UNSUPPORTED for head dims above
 * 256; DN_ERR_CUDA if the launch fails. */
dn_status gdn_decode_step(const dn_shape *shape, const void *q, const void *k, const void *v,
                          const void *beta, const float *g, const float *state_in,
                          float *state_out, void *o, void *stream);

/* Batched affine map of states: out_i = A_i S_i + B_i for i < count, fp32.
 * The recurrence is linear in the state ("Gated DeltaNet" rebuttal, Table 1,
 * row "Gated DeltaNet": S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + ...),
 * so the state leaving a span of tokens is A S + B, with A the product of the
 * span's transitions (the final state of a forward call with v = 0 and
 * h0 = I) and B the span's own final state from a zero state (a forward call
 * with h0 = NULL).  Composing these maps over consecutive spans in order gives
 * every span its entering state: the exchange step of a forward split along the
 * sequence (each GPU, or each pass, owning a span).
 *   A   [count][dk][dk], S, B, out [count][dk][dv], all device float32,
 *       row-major, 4-byte aligned; B may be NULL (zero); out must not overlap A
 *       or S (DN_ERR_INVALID_ARG), it may be B.
 * count <= 65535 (DN_ERR_UNSUPPORTED above), dk, dv in 1..256.  Asynchronous
 * on `stream`; allocates nothing.                                               */
dn_status dn_state_affine(const float *A, const float *S, const float *B, float *out, int count,
                          int dk, int dv, void *stream);

/* Bytes of the device staging arena gdn_chunk_fwd_host needs (0 on bad args):
 * the inputs, o, h0 and hT, and two more states for the time segments.      */
size_t dn_host_arena_size(const dn_shape *shape, int gated, int with_h0);

/* Gated DeltaNet forward on HOST buffers: copies q, k, v, beta, g, h0 (host,
 * pinned for asynchronous copies) into `arena` (device, >= dn_host_arena_size
 * bytes), runs the forward on `stream`, and copies o and hT back into the
 * host buffers.  Returns once the work is enqueued: synchronise `stream`
 * before reading o / hT.  g, h0, hT may be NULL as in gdn_chunk_fwd; for
 * packed input shape->cu_seqlens must still be a DEVICE pointer.
 * Fixed-length input of at least 32 chunks runs as up to 4 time segments of
 * whole chunks, so that the copies over the host link overlap the compute:
 *  - segment i's inputs go into the arena on a stream of the library's own;
 *  - segment i's forward runs on `stream` from the state segment i - 1 left
 *    (fp32, in the arena);
 *  - segment i's o goes back on a second stream of the library's own.
 * `stream` waits for those streams (events) before the call's work on it
 * ends, so that completing `stream` means o and hT are on the host.
 * Consequences:
 *  - The results equal one forward over the whole sequence up to the fp32
 *    rounding of the state between segments.
 *  - The device status word (dn_device_status) keeps what any segment flags.
 *  - The library's streams and events for this are made on the first such
 *    call in each context; make that call before any stream capture.
 *  - Calls from several host threads are enqueued one at a time.
 * Packed input of at least 32 chunks runs instead as up to 4 groups of heads
 * (H divisible by their number), each group's rows of every [H][T] tensor one
 * contiguous copy and its states copied from and into their [N][H] places;
 * heads are independent, so the results equal one forward's.  Other packed
 * input runs as one forward between the copies.                            */
dn_status gdn_chunk_fwd_host(const dn_shape *shape, const void *q, const void *k,
                             const void *v, const void *beta, const float *g,
                             const float *h0, void *o, float *hT, void *arena,
                             size_t arena_bytes, void *ws, size_t ws_bytes, void *stream);

/* Gated DeltaNet forward that allocates nothing and takes no workspace.
 * (The pages have no counterpart: this is a deployment variant.)  It is for
 * callers that cannot allocate device memory or hand the library a scratch
 * buffer: operator / plugin interfaces whose call signature carries no
 * workspace argument, and code running inside a host framework that owns all
 * device memory or forbids allocation on its hot path.
 * It runs the fused forward with one CTA per (sequence, head) -- the
 * cooperative forward gdn_chunk_fwd prefers needs a multi-megabyte package
 * ring in its workspace -- with that kernel's scratch (the device status word
 * and, for packed input, per-sequence chunk offsets and a longest-first order)
 * in a 256 KiB array of static device memory that every GPU loading the
 * library keeps until the process exits.  Limits:
 * the fast-path shapes only (dtype DN_BF16, dk = dv = 128, chunk 64;
 * otherwise DN_ERR_UNSUPPORTED), and at most about 32,000 packed sequences
 * (larger returns DN_ERR_WORKSPACE).  The first call on each device looks up
 * the array's device address with that device current; make that first call
 * before any stream capture.  The address is looked up again when the
 * device's context has changed (for example after cudaDeviceReset).  All calls
 * share the one array, so calls whose work overlaps on the GPU race on it:
 * serialise them (one stream, or events).  GDN_FORCE_GENERAL does not apply
 * here.  Arguments, layouts and host-side errors are those of gdn_chunk_fwd;
 * what the device finds (a bounded wait that ran out, malformed packed offsets,
 * a log-gate g > 0) goes to the array's status word, read by
 * dn_noalloc_status. */
dn_status gdn_chunk_fwd_noalloc(const dn_shape *shape, const void *q, const void *k,
                                const void *v, const void *beta, const float *g,
                                const float *h0, void *o, float *hT, void *stream);

/* Synchronises `stream`, then reads and clears the status word in `ws` that
 * the last call using `ws` wrote: DN_OK, DN_ERR_TIMEOUT (a bounded device wait
 * ran out; the outputs are not valid), DN_ERR_INVALID_ARG (malformed packed
 * offsets; those sequences were treated as empty) or DN_ERR_DOMAIN (a log-gate
 * g > 0 was read), in that order of precedence. */
dn_status dn_device_status(void *ws, void *stream);

/* The same for gdn_chunk_fwd_noalloc, whose status word lies in the library's
 * static scratch array on the current device rather than in a workspace:
 * synchronises `stream`, then reads, clears and maps that word as
 * dn_device_status does.  Allocates nothing.  As the array is shared, the word
 * describes the most recent gdn_chunk_fwd_noalloc call on this device; read it
 * before the next one starts.  Returns DN_ERR_CUDA if the array's address
 * cannot be looked up. */
dn_status dn_noalloc_status(void *stream);

/* Static description of a status code. */
const char *dn_status_str(dn_status s);

/* Which kernel family `shape` runs on: 1 = tcgen05/TMA fast path, 0 = the
 * general fp32 path, -1 = invalid shape.  for_backward as above. */
int dn_uses_fast_path(const dn_shape *shape, int for_backward);

/* Which kernels one call with `shape` runs, for launch accounting and CUDA
 * graph planning.  Returns DN_PATH_GENERAL (fp32 CUDA-core kernels),
 * DN_PATH_FUSED (one fused tcgen05 CTA per (sequence, head)) or DN_PATH_COOP
 * (the cooperative persistent tcgen05 kernel), or -1 for an invalid shape.  If
 * `kernels` is not null it receives the number of the library's own kernels the
 * call launches (memsets of the workspace are not counted).  for_backward as
 * above (2: gdn_chunk_bwd_saved, -1 where it is not available); the
 * gdn_chunk_fwd_noalloc entry point never takes DN_PATH_COOP. */
enum { DN_PATH_GENERAL = 0, DN_PATH_FUSED = 1, DN_PATH_COOP = 2 };
int dn_plan(const dn_shape *shape, int for_backward, int *kernels);

#ifdef __cplusplus
}
#endif
#endif /* GDN_GB300_H */
