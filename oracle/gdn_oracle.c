/*
 * Oracle for the (gated) delta rule: plain fp64, token by token, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or calls
 * this file; only the tests, the package's smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header or constant with the CUDA
 * kernels under chunkwise_delta_rule_02_gb300/csrc.
 *
 * What it computes (per sequence s and head h, independently):
 *
 *   Gated DeltaNet, "Gated DeltaNet: Improving Mamba2 with Delta Rule",
 *   rebuttal Table 1, row "Gated DeltaNet":
 *       S_t = S_{t-1} (alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T
 *   with S a d_v x d_k matrix.  DeltaNet is the same row with alpha_t = 1
 *   (Table 1, row "DeltaNet").  This file stores the transpose, a d_k x d_v
 *   matrix M = S^T, row-major (key index outer), so the step reads
 *       M_t = alpha_t (I - beta_t k_t k_t^T) M_{t-1} + beta_t k_t v_t^T
 *   and is evaluated in its rank-1 form
 *       r_t = M_{t-1}^T k_t,  u_t = beta_t (v_t - alpha_t r_t),
 *       M_t = alpha_t M_{t-1} + k_t u_t^T,
 *   which is the same expression with the product multiplied out.
 *   The read-out is o_t = scale * M_t^T q_t (o_t = q_t S_t in the row-vector
 *   convention), i.e. the output uses the state after the token's own write.
 *   alpha_t = exp(g_t), g_t being the per-token, per-head log-gate.
 *
 *   q and k are L2-normalised per token before use when qk_l2norm != 0:
 *       x_hat = x / sqrt(sum(x^2) + eps).
 *
 *   Longhorn's step size (longhorn != 0; same rebuttal, Table 1, row
 *   "Longhorn", scalar beta): the step uses
 *       eps_t = beta_t / (1 + beta_t k_hat_t^T k_hat_t)
 *   in place of beta_t, k_hat_t being the key the step uses (after the
 *   normalisation, when it is on).  With alpha_t = exp(g_t) the step is then
 *   the minimiser of ||S - alpha_t S_{t-1}||_F^2 + beta_t ||S k_t - v_t||^2.
 *
 * Backward: back-propagation through time over the same loop, written by hand
 * (each line is the derivative of one forward line), with forward checkpoints
 * every CKPT tokens and the states of a segment recomputed before it is walked
 * backwards.  Gradients are with respect to the raw q and k (chained through the
 * normalisation), v, beta, the log-gate g and the initial state.
 *
 * Layout of every token-indexed array: [NB][H][Ttot][d] row-major (the time
 * axis of batch row b and head h is contiguous).  Fixed-length input: NB = B
 * sequences, each of length Ttot, offs == NULL.  Packed variable-length input:
 * NB = 1, offs[0..n_seqs] are the token offsets of the sequences on the time
 * axis.  States: [n_seqs][H][dk][dv].
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define CKPT 64

typedef struct {
    int n_seqs, NB, H, Ttot, dk, dv;
    const long long *offs;
    const double *q, *k, *v, *beta, *g, *h0;
    int qk_l2norm, longhorn;
    double scale, eps;
    /* forward outputs */
    double *o, *hT;
    /* backward inputs / outputs */
    const double *dout, *dhT;
    double *dq, *dk_out, *dv_out, *dbeta, *dg, *dh0;
    int nthreads;
    int status;
} job_t;

typedef struct {
    job_t *job;
    int tid;
    int backward;
} worker_arg_t;

/* token range and base offsets of work item (sequence s, head h) */
static void item_range(const job_t *J, int s, int h, long long *t0, long long *t1,
                       long long *row)
{
    if (J->offs) {
        *t0 = J->offs[s];
        *t1 = J->offs[s + 1];
        *row = (long long)h * J->Ttot;           /* batch row 0 */
    } else {
        *t0 = 0;
        *t1 = J->Ttot;
        *row = ((long long)s * J->H + h) * J->Ttot;
    }
}

/* the step size the update uses: beta, or Longhorn's beta / (1 + beta k^T k) */
static double step_size(const job_t *J, double beta, const double *kh)
{
    if (!J->longhorn) return beta;
    double kk = 0.0;
    for (int i = 0; i < J->dk; ++i) kk += kh[i] * kh[i];
    return beta / (1.0 + beta * kk);
}

static void l2norm(const double *x, int d, double eps, double *xh, double *rho_out)
{
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += x[i] * x[i];
    double rho = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < d; ++i) xh[i] = x[i] * rho;
    if (rho_out) *rho_out = rho;
}

/* one recurrence step: M <- alpha M + k u^T with u = beta (v - alpha M^T k);
 * writes r = M_prev^T k and u when the caller wants them */
static void step(double *M, const double *kh, const double *v, double beta,
                 double alpha, int dk, int dv, double *r, double *u)
{
    for (int j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += M[(size_t)i * dv + j] * kh[i];
        r[j] = acc;
    }
    for (int j = 0; j < dv; ++j) u[j] = beta * (v[j] - alpha * r[j]);
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j)
            M[(size_t)i * dv + j] = alpha * M[(size_t)i * dv + j] + kh[i] * u[j];
}

static void fwd_item(job_t *J, int s, int h, double *M, double *kh, double *qh,
                     double *r, double *u)
{
    const int dk = J->dk, dv = J->dv;
    long long t0, t1, row;
    item_range(J, s, h, &t0, &t1, &row);
    size_t sidx = ((size_t)s * J->H + h) * (size_t)dk * dv;
    if (J->h0) memcpy(M, J->h0 + sidx, sizeof(double) * dk * dv);
    else memset(M, 0, sizeof(double) * dk * dv);
    for (long long t = t0; t < t1; ++t) {
        const double *kt = J->k + (row + t) * dk;
        const double *qt = J->q + (row + t) * dk;
        const double *vt = J->v + (row + t) * dv;
        if (J->qk_l2norm) {
            l2norm(kt, dk, J->eps, kh, NULL);
            l2norm(qt, dk, J->eps, qh, NULL);
        } else {
            memcpy(kh, kt, sizeof(double) * dk);
            memcpy(qh, qt, sizeof(double) * dk);
        }
        double alpha = J->g ? exp(J->g[row + t]) : 1.0;
        step(M, kh, vt, step_size(J, J->beta[row + t], kh), alpha, dk, dv, r, u);
        double *ot = J->o + (row + t) * dv;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += M[(size_t)i * dv + j] * qh[i];
            ot[j] = J->scale * acc;
        }
    }
    if (J->hT) memcpy(J->hT + sidx, M, sizeof(double) * dk * dv);
}

/* Backward through time for one (sequence, head). */
static int bwd_item(job_t *J, int s, int h)
{
    const int dk = J->dk, dv = J->dv;
    const size_t SZ = (size_t)dk * dv;
    long long t0, t1, row;
    item_range(J, s, h, &t0, &t1, &row);
    long long L = t1 - t0;
    size_t sidx = ((size_t)s * J->H + h) * SZ;
    long long nseg = (L + CKPT - 1) / CKPT;

    double *ck = (double *)malloc(sizeof(double) * SZ * (size_t)(nseg + 1));
    double *seg = (double *)malloc(sizeof(double) * SZ * (CKPT + 1));
    double *dS = (double *)malloc(sizeof(double) * SZ);
    double *kh = (double *)malloc(sizeof(double) * dk);
    double *qh = (double *)malloc(sizeof(double) * dk);
    double *dkh = (double *)malloc(sizeof(double) * dk);
    double *dqh = (double *)malloc(sizeof(double) * dk);
    double *r = (double *)malloc(sizeof(double) * dv);
    double *u = (double *)malloc(sizeof(double) * dv);
    double *du = (double *)malloc(sizeof(double) * dv);
    double *dr = (double *)malloc(sizeof(double) * dv);
    if (!ck || !seg || !dS || !kh || !qh || !dkh || !dqh || !r || !u || !du || !dr) {
        free(ck); free(seg); free(dS); free(kh); free(qh); free(dkh); free(dqh);
        free(r); free(u); free(du); free(dr);
        return 1;
    }

    /* forward pass keeping a checkpoint at the start of every segment */
    double *M = ck;
    if (J->h0) memcpy(M, J->h0 + sidx, sizeof(double) * SZ);
    else memset(M, 0, sizeof(double) * SZ);
    for (long long sg = 0; sg < nseg; ++sg) {
        double *next = ck + (size_t)(sg + 1) * SZ;
        memcpy(next, ck + (size_t)sg * SZ, sizeof(double) * SZ);
        long long ta = t0 + sg * CKPT, tb = ta + CKPT < t1 ? ta + CKPT : t1;
        for (long long t = ta; t < tb; ++t) {
            const double *kt = J->k + (row + t) * dk;
            if (J->qk_l2norm) l2norm(kt, dk, J->eps, kh, NULL);
            else memcpy(kh, kt, sizeof(double) * dk);
            double alpha = J->g ? exp(J->g[row + t]) : 1.0;
            step(next, kh, J->v + (row + t) * dv, step_size(J, J->beta[row + t], kh), alpha, dk,
                 dv, r, u);
        }
    }

    if (J->dhT) memcpy(dS, J->dhT + sidx, sizeof(double) * SZ);
    else memset(dS, 0, sizeof(double) * SZ);

    for (long long sg = nseg - 1; sg >= 0; --sg) {
        long long ta = t0 + sg * CKPT, tb = ta + CKPT < t1 ? ta + CKPT : t1;
        /* states seg[0] = state before token ta, seg[i] = state after token ta+i-1 */
        memcpy(seg, ck + (size_t)sg * SZ, sizeof(double) * SZ);
        for (long long t = ta; t < tb; ++t) {
            double *dst = seg + (size_t)(t - ta + 1) * SZ;
            memcpy(dst, dst - SZ, sizeof(double) * SZ);
            const double *kt = J->k + (row + t) * dk;
            if (J->qk_l2norm) l2norm(kt, dk, J->eps, kh, NULL);
            else memcpy(kh, kt, sizeof(double) * dk);
            double alpha = J->g ? exp(J->g[row + t]) : 1.0;
            step(dst, kh, J->v + (row + t) * dv, step_size(J, J->beta[row + t], kh), alpha, dk,
                 dv, r, u);
        }
        for (long long t = tb - 1; t >= ta; --t) {
            const double *Sprev = seg + (size_t)(t - ta) * SZ;
            const double *Scur = Sprev + SZ;
            const double *kt = J->k + (row + t) * dk;
            const double *qt = J->q + (row + t) * dk;
            const double *vt = J->v + (row + t) * dv;
            const double *dot = J->dout + (row + t) * dv;
            double rho_k = 1.0, rho_q = 1.0;
            if (J->qk_l2norm) {
                l2norm(kt, dk, J->eps, kh, &rho_k);
                l2norm(qt, dk, J->eps, qh, &rho_q);
            } else {
                memcpy(kh, kt, sizeof(double) * dk);
                memcpy(qh, qt, sizeof(double) * dk);
            }
            double beta = step_size(J, J->beta[row + t], kh);
            double alpha = J->g ? exp(J->g[row + t]) : 1.0;
            /* recompute r and u of this token from the state before it */
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += Sprev[(size_t)i * dv + j] * kh[i];
                r[j] = acc;
                u[j] = beta * (vt[j] - alpha * r[j]);
            }
            /* o_t = scale * S_t^T q_hat */
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) {
                    dS[(size_t)i * dv + j] += J->scale * qh[i] * dot[j];
                    acc += Scur[(size_t)i * dv + j] * dot[j];
                }
                dqh[i] = J->scale * acc;
            }
            /* S_t = alpha S_{t-1} + k_hat u^T */
            double dalpha = 0.0;
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) {
                    dalpha += dS[(size_t)i * dv + j] * Sprev[(size_t)i * dv + j];
                    acc += dS[(size_t)i * dv + j] * u[j];
                }
                dkh[i] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += dS[(size_t)i * dv + j] * kh[i];
                du[j] = acc;
            }
            /* u = beta (v - alpha r) */
            double dbeta = 0.0, dr_alpha = 0.0;
            for (int j = 0; j < dv; ++j) {
                dbeta += du[j] * (vt[j] - alpha * r[j]);
                dr_alpha += du[j] * r[j];
                dr[j] = -alpha * beta * du[j];
            }
            dalpha -= beta * dr_alpha;
            /* r = S_{t-1}^T k_hat, and the direct path alpha S_{t-1} */
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) {
                    acc += Sprev[(size_t)i * dv + j] * dr[j];
                    dS[(size_t)i * dv + j] = alpha * dS[(size_t)i * dv + j] + kh[i] * dr[j];
                }
                dkh[i] += acc;
            }
            double *dvt = J->dv_out + (row + t) * dv;
            for (int j = 0; j < dv; ++j) dvt[j] = beta * du[j];
            if (J->longhorn) {
                /* beta = b / (1 + b kk), kk = k_hat^T k_hat: d/db = 1 / (1 + b kk)^2,
                 * d/dkk = -b^2 / (1 + b kk)^2, and d kk / d k_hat = 2 k_hat */
                double b = J->beta[row + t], kk = 0.0;
                for (int i = 0; i < dk; ++i) kk += kh[i] * kh[i];
                double den = 1.0 + b * kk;
                double dkk = -dbeta * b * b / (den * den);
                for (int i = 0; i < dk; ++i) dkh[i] += 2.0 * dkk * kh[i];
                dbeta /= den * den;
            }
            J->dbeta[row + t] = dbeta;
            if (J->dg) J->dg[row + t] = J->g ? alpha * dalpha : 0.0;
            /* through the normalisation x_hat = x * rho, rho = (|x|^2+eps)^-1/2 */
            double *dkt = J->dk_out + (row + t) * dk;
            double *dqt = J->dq + (row + t) * dk;
            if (J->qk_l2norm) {
                double pk = 0.0, pq = 0.0;
                for (int i = 0; i < dk; ++i) { pk += kh[i] * dkh[i]; pq += qh[i] * dqh[i]; }
                for (int i = 0; i < dk; ++i) {
                    dkt[i] = rho_k * (dkh[i] - kh[i] * pk);
                    dqt[i] = rho_q * (dqh[i] - qh[i] * pq);
                }
            } else {
                memcpy(dkt, dkh, sizeof(double) * dk);
                memcpy(dqt, dqh, sizeof(double) * dk);
            }
        }
    }
    if (J->dh0) memcpy(J->dh0 + sidx, dS, sizeof(double) * SZ);

    free(ck); free(seg); free(dS); free(kh); free(qh); free(dkh); free(dqh);
    free(r); free(u); free(du); free(dr);
    return 0;
}

static void *worker(void *p)
{
    worker_arg_t *a = (worker_arg_t *)p;
    job_t *J = a->job;
    const int n_items = J->n_seqs * J->H;
    double *M = NULL, *kh = NULL, *qh = NULL, *r = NULL, *u = NULL;
    if (!a->backward) {
        M = (double *)malloc(sizeof(double) * (size_t)J->dk * J->dv);
        kh = (double *)malloc(sizeof(double) * J->dk);
        qh = (double *)malloc(sizeof(double) * J->dk);
        r = (double *)malloc(sizeof(double) * J->dv);
        u = (double *)malloc(sizeof(double) * J->dv);
        if (!M || !kh || !qh || !r || !u) {
            J->status = 1;
            free(M); free(kh); free(qh); free(r); free(u);
            return NULL;
        }
    }
    for (int it = a->tid; it < n_items; it += J->nthreads) {
        int s = it / J->H, h = it % J->H;
        if (a->backward) {
            if (bwd_item(J, s, h)) J->status = 1;
        } else {
            fwd_item(J, s, h, M, kh, qh, r, u);
        }
    }
    free(M); free(kh); free(qh); free(r); free(u);
    return NULL;
}

static int run(job_t *J, int backward)
{
    int nt = J->nthreads < 1 ? 1 : J->nthreads;
    int n_items = J->n_seqs * J->H;
    if (nt > n_items) nt = n_items < 1 ? 1 : n_items;
    J->nthreads = nt;
    J->status = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    worker_arg_t *args = (worker_arg_t *)malloc(sizeof(worker_arg_t) * nt);
    if (!th || !args) { free(th); free(args); return 1; }
    int started = 0;
    for (int i = 0; i < nt; ++i) {
        args[i].job = J; args[i].tid = i; args[i].backward = backward;
        if (i == 0) continue;
        if (pthread_create(&th[i], NULL, worker, &args[i]) != 0) break;
        ++started;
    }
    /* thread 0's share runs here; items of threads that failed to start run too */
    for (int i = 0; i < nt; ++i)
        if (i == 0 || i > started) worker(&args[i]);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    free(th); free(args);
    return J->status;
}

static int check_dims(int n_seqs, int NB, int H, int Ttot, int dk, int dv, const long long *offs)
{
    if (n_seqs < 0 || NB < 0 || H < 1 || Ttot < 0 || dk < 1 || dv < 1) return 1;
    if (offs) {
        if (NB != 1 || offs[0] != 0 || offs[n_seqs] != Ttot) return 1;
        for (int i = 0; i < n_seqs; ++i) if (offs[i + 1] < offs[i]) return 1;
    } else if (NB != n_seqs) {
        return 1;
    }
    return 0;
}

int gdn_oracle_fwd(int n_seqs, int NB, int H, int Ttot, int dk, int dv,
                   const long long *offs, const double *q, const double *k,
                   const double *v, const double *beta, const double *g,
                   const double *h0, int qk_l2norm, double scale, double eps,
                   int longhorn, double *o, double *hT, int nthreads)
{
    if (check_dims(n_seqs, NB, H, Ttot, dk, dv, offs)) return 2;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.n_seqs = n_seqs; J.NB = NB; J.H = H; J.Ttot = Ttot; J.dk = dk; J.dv = dv;
    J.offs = offs; J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0;
    J.qk_l2norm = qk_l2norm; J.scale = scale; J.eps = eps; J.longhorn = longhorn;
    J.o = o; J.hT = hT; J.nthreads = nthreads;
    return run(&J, 0);
}

int gdn_oracle_bwd(int n_seqs, int NB, int H, int Ttot, int dk, int dv,
                   const long long *offs, const double *q, const double *k,
                   const double *v, const double *beta, const double *g,
                   const double *h0, int qk_l2norm, double scale, double eps,
                   int longhorn, const double *dout, const double *dhT, double *dq, double *dk_out,
                   double *dv_out, double *dbeta, double *dg, double *dh0, int nthreads)
{
    if (check_dims(n_seqs, NB, H, Ttot, dk, dv, offs)) return 2;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.n_seqs = n_seqs; J.NB = NB; J.H = H; J.Ttot = Ttot; J.dk = dk; J.dv = dv;
    J.offs = offs; J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0;
    J.qk_l2norm = qk_l2norm; J.scale = scale; J.eps = eps; J.longhorn = longhorn;
    J.dout = dout; J.dhT = dhT; J.dq = dq; J.dk_out = dk_out; J.dv_out = dv_out;
    J.dbeta = dbeta; J.dg = dg; J.dh0 = dh0; J.nthreads = nthreads;
    return run(&J, 1);
}
