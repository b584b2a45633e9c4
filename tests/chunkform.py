"""Chunk form of the (gated) delta rule in fp64 numpy — test helper only.

This is the derivation the CUDA kernels implement, written as plainly as
possible so the tests can check it against the token-by-token oracle.  It is
not the oracle (the oracle is the recurrence in ``oracle/``) and the library
does not import it.

Forward (per sequence and head; rows r = 1..c of one chunk; S the d_k x d_v
state entering the chunk; gamma the within-chunk cumulative sum of the
log-gate g; Gamma = exp(gamma); D_ri = exp(gamma_r - gamma_i) for i <= r):

    A    = strict_lower( diag(beta) (K K^T o D) )
    T    = (I + A)^-1 diag(beta)                    (UT transform)
    W    = T diag(Gamma) K,   U = T V               (WY factors)
    Unew = U - W S
    O    = scale * ( diag(Gamma) Q S + lower(Q K^T o D) Unew )   (diagonal kept)
    S'   = Gamma_c S + (diag(exp(gamma_c - gamma)) K)^T Unew

With g = 0 these are the DeltaNet chunk equations (T, W = TK, U = TV, the
scan S <- S + K^T (U - W S), O = QS + tril(QK^T)(U - WS)).  The derivation:
u_r = beta_r (v_r - alpha_r S_{r-1}^T k_r) and S_r = alpha_r S_{r-1} + k_r u_r^T
unroll to S_r = Gamma_r S + sum_{i<=r} D_ri k_i u_i^T, hence
(I + A) Unew = diag(beta)(V - diag(Gamma) K S).

Backward: reverse-mode derivative of the lines above, chunk by chunk, with the
entering states recomputed by a forward pass (the backward of the DeltaNet page
recomputes chunk states rather than storing them).
"""
from __future__ import annotations

import numpy as np


def l2n(x, eps):
    rho = 1.0 / np.sqrt((x * x).sum(-1, keepdims=True) + eps)
    return x * rho, rho


def _chunk_consts(K, b, gg):
    c = K.shape[0]
    gam = np.cumsum(gg) if gg is not None else np.zeros(c)
    Gam = np.exp(gam)
    low = np.tril(np.ones((c, c)))
    D = np.exp(gam[:, None] - gam[None, :]) * low
    KK = K @ K.T
    A = np.tril(b[:, None] * KK * D, -1)
    Linv = np.linalg.inv(np.eye(c) + A)
    Tm = Linv * b[None, :]
    eC = np.exp(gam[-1] - gam)
    return gam, Gam, D, KK, A, Linv, Tm, eC


def fwd_seq(q, k, v, beta, g, h0, C, scale=1.0, l2norm=True, eps=1e-6):
    """One (sequence, head): q,k [L,dk], v [L,dv], beta,g [L], h0 [dk,dv] or None."""
    L, dk = k.shape
    dv = v.shape[1]
    if l2norm:
        q, _ = l2n(q, eps)
        k, _ = l2n(k, eps)
    S = np.zeros((dk, dv)) if h0 is None else h0.copy()
    O = np.zeros((L, dv))
    for c0 in range(0, L, C):
        c1 = min(L, c0 + C)
        Q, K, V, b = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1]
        gg = None if g is None else g[c0:c1]
        gam, Gam, D, KK, A, Linv, Tm, eC = _chunk_consts(K, b, gg)
        W = Tm @ (Gam[:, None] * K)
        U = Tm @ V
        Unew = U - W @ S
        M = np.tril(Q @ K.T * D)
        O[c0:c1] = scale * (Gam[:, None] * (Q @ S) + M @ Unew)
        S = Gam[-1] * S + (eC[:, None] * K).T @ Unew
    return O, S


def fwd_seq_substituted(q, k, v, beta, g, h0, C, scale=1.0, l2norm=True, eps=1e-6):
    """fwd_seq with the state substituted into the next chunk's Unew:

        Unew_{j+1} = U_{j+1} - Gamma_c(j) W_{j+1} S_j + N_{j+1} Unew_j,
        N_{j+1}    = -W_{j+1} (diag(exp(gamma_c - gamma)) K)_j^T,

    which follows from S_{j+1} = Gamma_c(j) S_j + K~_j^T Unew_j.  Unew then depends
    on the previous chunk's Unew through one C x C product, and on a state one chunk
    older, so a kernel can keep the state update off its critical cycle.  The output
    takes the older state the same way, with R_{j+1} = Qt_{j+1} K~_j^T
    (Qt = diag(Gamma) Q):

        O_{j+1} = scale * (Gamma_c(j) Qt_{j+1} S_j + R_{j+1} Unew_j + M_{j+1} Unew_{j+1}).

    The first chunk of a sequence uses Unew_0 = U_0 - W_0 S_0 and O_0 as in fwd_seq."""
    L, dk = k.shape
    dv = v.shape[1]
    if l2norm:
        q, _ = l2n(q, eps)
        k, _ = l2n(k, eps)
    S = np.zeros((dk, dv)) if h0 is None else h0.copy()   # S_j, the state entering chunk j
    O = np.zeros((L, dv))
    prev = None   # (Gamma_c, K~, Unew, S) of chunk j - 1
    for c0 in range(0, L, C):
        c1 = min(L, c0 + C)
        Q, K, V, b = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1]
        gg = None if g is None else g[c0:c1]
        gam, Gam, D, KK, A, Linv, Tm, eC = _chunk_consts(K, b, gg)
        W = Tm @ (Gam[:, None] * K)
        U = Tm @ V
        if prev is None:
            Unew = U - W @ S
        else:
            GC_p, Kt_p, Unew_p, S_p = prev
            N = -W @ Kt_p.T
            Unew = U - GC_p * (W @ S_p) + N @ Unew_p
        M = np.tril(Q @ K.T * D)
        Qt = Gam[:, None] * Q
        if prev is None:
            O[c0:c1] = scale * (Qt @ S + M @ Unew)
        else:
            R = Qt @ Kt_p.T
            O[c0:c1] = scale * (GC_p * (Qt @ S_p) + R @ Unew_p + M @ Unew)
        Kt = eC[:, None] * K
        prev = (Gam[-1], Kt, Unew, S)
        S = Gam[-1] * S + Kt.T @ Unew
    return O, S


def bwd_seq(q, k, v, beta, g, h0, dO, dST, C, scale=1.0, l2norm=True, eps=1e-6):
    """Reverse-mode gradients of (O, S_final) for one (sequence, head)."""
    L, dk = k.shape
    dv = v.shape[1]
    qr, kr = q, k
    if l2norm:
        q, rq = l2n(q, eps)
        k, rk = l2n(k, eps)
    # forward recompute of the states entering each chunk
    starts = list(range(0, L, C))
    S = np.zeros((dk, dv)) if h0 is None else h0.copy()
    S_in = []
    for c0 in starts:
        c1 = min(L, c0 + C)
        K, V, b = k[c0:c1], v[c0:c1], beta[c0:c1]
        gg = None if g is None else g[c0:c1]
        gam, Gam, D, KK, A, Linv, Tm, eC = _chunk_consts(K, b, gg)
        S_in.append(S)
        Unew = Tm @ V - Tm @ (Gam[:, None] * K) @ S
        S = Gam[-1] * S + (eC[:, None] * K).T @ Unew
    dq = np.zeros_like(q)
    dk_ = np.zeros_like(k)
    dv_ = np.zeros_like(v)
    dbeta = np.zeros_like(beta)
    dgam_all = np.zeros(L)
    dS = np.zeros((dk, dv)) if dST is None else dST.copy()
    for ci in range(len(starts) - 1, -1, -1):
        c0 = starts[ci]
        c1 = min(L, c0 + C)
        Q, K, V, b = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1]
        gg = None if g is None else g[c0:c1]
        gam, Gam, D, KK, A, Linv, Tm, eC = _chunk_consts(K, b, gg)
        Sin = S_in[ci]
        GK = Gam[:, None] * K
        W = Tm @ GK
        Unew = Tm @ V - W @ Sin
        QK = Q @ K.T
        M = np.tril(QK * D)
        dOc = scale * dO[c0:c1]
        dSo = dS
        dUnew = M.T @ dOc + (eC[:, None] * K) @ dSo
        dS = Gam[-1] * dSo + (Gam[:, None] * Q).T @ dOc - W.T @ dUnew
        dP = np.tril(dOc @ Unew.T)
        dQ = Gam[:, None] * (dOc @ Sin.T) + (dP * D) @ K
        dK = (dP * D).T @ Q
        dKt = Unew @ dSo.T
        dK += eC[:, None] * dKt
        dW = -dUnew @ Sin.T
        dT = dW @ GK.T + dUnew @ V.T
        dGK = Tm.T @ dW
        dK += Gam[:, None] * dGK
        dV = Tm.T @ dUnew
        dLinv = dT * b[None, :]
        db = np.einsum("ri,ri->i", Linv, dT)
        dL = -Linv.T @ dLinv @ Linv.T
        dA = np.tril(dL, -1)
        db += (dA * KK * D).sum(1)
        dKK = dA * b[:, None] * D
        dK += dKK @ K + dKK.T @ K
        dD = dA * b[:, None] * KK + dP * QK
        E = dD * D
        dgam = E.sum(1) - E.sum(0)
        dgam += Gam * (dOc * (Q @ Sin)).sum(1)
        dgam += Gam * (dGK * K).sum(1)
        e = (dKt * K).sum(1) * eC
        dgam -= e
        dgam[-1] += e.sum() + Gam[-1] * (dSo * Sin).sum()
        dq[c0:c1] = dQ
        dk_[c0:c1] = dK
        dv_[c0:c1] = dV
        dbeta[c0:c1] = db
        dgam_all[c0:c1] = dgam
    dg = None
    if g is not None:
        dg = np.zeros(L)
        for c0 in starts:
            c1 = min(L, c0 + C)
            dg[c0:c1] = np.cumsum(dgam_all[c0:c1][::-1])[::-1]
    if l2norm:
        dq = rq * (dq - q * (q * dq).sum(-1, keepdims=True))
        dk_ = rk * (dk_ - k * (k * dk_).sum(-1, keepdims=True))
    return dict(dq=dq, dk=dk_, dv=dv_, dbeta=dbeta, dg=dg, dh0=dS)
