"""Pins for the fp64 oracle: each test checks it against something other than
itself — explicit matrix products, the WY form, closed forms, the one-step
gradient-descent reading of the online-learning table, state passing,
finite differences, and the chunk-form derivation the kernels use.

Sources:
  [GDN-T1]  "Gated DeltaNet: Improving Mamba2 with Delta Rule", rebuttal
            Table 1 (online-learning objectives and updates for LA, Mamba2,
            Longhorn, DeltaNet, Gated DeltaNet) and its caption (DeltaNet as
            one explicit gradient step).
  [DN-W2]   "Parallelizing Linear Transformers with the Delta Rule over
            Sequence Length", reply W2 (products of Householder-like
            matrices, WY representation) and reply W3 (the delta rule removes
            the old value stored under a key and writes the new one).
  [GDN-SP]  same GDN page, reply on length extrapolation (state passing).
"""
import numpy as np
import pytest

import oracle
import chunkform

RNG = np.random.default_rng


def _rand_inputs(rng, NB, H, T, dk, dv, gated=True, h0=True):
    q = rng.standard_normal((NB, H, T, dk))
    k = rng.standard_normal((NB, H, T, dk))
    v = rng.standard_normal((NB, H, T, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((NB, H, T))))
    g = -np.log1p(np.exp(rng.standard_normal((NB, H, T)))) / 4.0 if gated else None
    S0 = rng.standard_normal((NB, H, dk, dv)) * 0.3 if h0 else None
    return q, k, v, beta, g, S0


# ---------------------------------------------------------------- [GDN-T1], [DN-W2]
@pytest.mark.parametrize("seed,T,dk,dv,gated", [(0, 1, 3, 2, False), (1, 4, 4, 3, False),
                                                (2, 6, 4, 4, True), (3, 5, 2, 3, True)])
def test_explicit_householder_products(seed, T, dk, dv, gated):
    """S_T built from explicit d_k x d_k transition matrices alpha_t (I - beta_t k_t k_t^T)
    (the Table-1 update, pages' S transposed) equals the oracle's state and read-out."""
    rng = RNG(seed)
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 1, T, dk, dv, gated)
    o, hT = oracle.fwd(q, k, v, beta, g, S0, qk_l2norm=False)
    S = S0[0, 0].copy()
    for t in range(T):
        kt, vt, qt = k[0, 0, t], v[0, 0, t], q[0, 0, t]
        a = np.exp(g[0, 0, t]) if gated else 1.0
        Tr = a * (np.eye(dk) - beta[0, 0, t] * np.outer(kt, kt))
        S = Tr @ S + beta[0, 0, t] * np.outer(kt, vt)
        np.testing.assert_allclose(o[0, 0, t], S.T @ qt, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(hT[0, 0], S, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed,T,d", [(4, 3, 3), (5, 6, 4), (6, 2, 4)])
def test_wy_representation(seed, T, d):
    """prod_t (I - beta_t k_t k_t^T) = I - sum_i k_i w_i^T with w_t = beta_t (k_t - sum_{i<t}
    w_i (k_i . k_t)) (the WY form of a product of Householder-like factors, [DN-W2]); the
    oracle with v = 0 maps h0 to that product times h0, and with h0 = 0 its state is
    sum_i k_i u_i^T with u_t = beta_t (v_t - sum_{i<t} u_i (k_i . k_t))."""
    rng = RNG(seed)
    q, k, v, beta, _, S0 = _rand_inputs(rng, 1, 1, T, d, d, gated=False)
    K, b = k[0, 0], beta[0, 0]
    P = np.eye(d)
    for t in range(T):
        P = (np.eye(d) - b[t] * np.outer(K[t], K[t])) @ P
    w = []
    for t in range(T):
        w.append(b[t] * (K[t] - sum(wi * (K[i] @ K[t]) for i, wi in enumerate(w))))
    P_wy = np.eye(d) - sum(np.outer(K[i], w[i]) for i in range(T))
    np.testing.assert_allclose(P, P_wy, rtol=1e-12, atol=1e-12)
    _, hT = oracle.fwd(q, k, np.zeros_like(v), beta, None, S0, qk_l2norm=False)
    np.testing.assert_allclose(hT[0, 0], P_wy @ S0[0, 0], rtol=1e-12, atol=1e-12)
    u = []
    for t in range(T):
        u.append(b[t] * (v[0, 0, t] - sum(ui * (K[i] @ K[t]) for i, ui in enumerate(u))))
    _, hT = oracle.fwd(q, k, v, beta, None, None, qk_l2norm=False)
    np.testing.assert_allclose(hT[0, 0], sum(np.outer(K[i], u[i]) for i in range(T)),
                               rtol=1e-12, atol=1e-12)


def test_l2_normalisation_matches_numpy():
    """In-kernel normalisation x / sqrt(|x|^2 + eps): the oracle with it on equals the oracle
    with it off on inputs normalised by numpy.linalg.norm."""
    rng = RNG(7)
    q, k, v, beta, g, S0 = _rand_inputs(rng, 2, 2, 17, 8, 5)
    eps = 1e-6
    qn = q / np.sqrt(np.linalg.norm(q, axis=-1, keepdims=True) ** 2 + eps)
    kn = k / np.sqrt(np.linalg.norm(k, axis=-1, keepdims=True) ** 2 + eps)
    o1, h1 = oracle.fwd(q, k, v, beta, g, S0, qk_l2norm=True, eps=eps)
    o2, h2 = oracle.fwd(qn, kn, v, beta, g, S0, qk_l2norm=False)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h1, h2, rtol=1e-12, atol=1e-13)


def test_alpha_one_reduces_gated_to_plain():
    """[GDN-T1]: Gated DeltaNet with alpha = exp(0) = 1 is DeltaNet, bit for bit."""
    rng = RNG(8)
    q, k, v, beta, _, S0 = _rand_inputs(rng, 2, 3, 33, 6, 7, gated=False)
    o1, h1 = oracle.fwd(q, k, v, beta, np.zeros_like(beta), S0)
    o2, h2 = oracle.fwd(q, k, v, beta, None, S0)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


def test_beta_zero_keeps_or_decays_state():
    """beta = 0: no write, no erase.  Plain: S_T = S_0 and o_t = q_hat_t^T S_0.  Gated:
    S_t = exp(sum_{s<=t} g_s) S_0, a pure decay."""
    rng = RNG(9)
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 2, 40, 5, 4)
    z = np.zeros_like(beta)
    o, hT = oracle.fwd(q, k, v, z, None, S0)
    np.testing.assert_array_equal(hT, S0)
    qn = q / np.sqrt((q * q).sum(-1, keepdims=True) + oracle.EPS)
    np.testing.assert_allclose(o, np.einsum("bhtk,bhkv->bhtv", qn, S0), rtol=1e-12, atol=1e-14)
    o, hT = oracle.fwd(q, k, v, z, g, S0)
    cum = np.cumsum(g, axis=-1)
    np.testing.assert_allclose(hT, np.exp(cum[..., -1])[..., None, None] * S0, rtol=1e-12)
    np.testing.assert_allclose(o, np.exp(cum)[..., None] * np.einsum("bhtk,bhkv->bhtv", qn, S0),
                               rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("m", [1, 5, 16])
def test_exact_retrieval_orthonormal_keys(m):
    """beta = 1, alpha = 1, zero start, orthonormal keys: reading with key k_i returns v_i
    exactly (the associative-memory reading of the delta rule, [DN-W3])."""
    d, dv = 16, 9
    rng = RNG(10 + m)
    Kq, _ = np.linalg.qr(rng.standard_normal((d, d)))
    keys = Kq[:, :m].T[None, None]
    vals = rng.standard_normal((1, 1, m, dv))
    ones = np.ones((1, 1, m))
    _, hT = oracle.fwd(keys, keys, vals, ones, None, None, qk_l2norm=True, eps=0.0)
    np.testing.assert_allclose(np.einsum("tk,kv->tv", keys[0, 0], hT[0, 0]), vals[0, 0],
                               rtol=0, atol=1e-12)


def test_overwrite_same_key():
    """Writing the same unit key twice with beta = 1 leaves only the second value
    ("subtract the old value, write the new one", [DN-W3])."""
    rng = RNG(11)
    kvec = rng.standard_normal(6)
    kvec /= np.linalg.norm(kvec)
    keys = np.stack([kvec, kvec])[None, None]
    vals = rng.standard_normal((1, 1, 2, 4))
    _, hT = oracle.fwd(keys, keys, vals, np.ones((1, 1, 2)), None, None, qk_l2norm=False)
    np.testing.assert_allclose(hT[0, 0], np.outer(kvec, vals[0, 0, 1]), atol=1e-13)


def _fd_grad(f, X, h=1e-6):
    G = np.zeros_like(X)
    for idx in np.ndindex(X.shape):
        Xp = X.copy(); Xp[idx] += h
        Xm = X.copy(); Xm[idx] -= h
        G[idx] = (f(Xp) - f(Xm)) / (2 * h)
    return G


def test_one_step_gradient_descent_identity():
    """[GDN-T1] caption: a DeltaNet step is one explicit gradient step of size beta on
    1/2 |S k - v|^2 (pages' d_v x d_k S) taken at S_{t-1}; the gradient here is a central
    finite difference of that objective, not a formula."""
    rng = RNG(12)
    dk, dv = 4, 3
    Sp = rng.standard_normal((dv, dk))               # pages' orientation
    kv = rng.standard_normal(dk); kv /= np.linalg.norm(kv)
    vv = rng.standard_normal(dv)
    b = 0.37
    grad = _fd_grad(lambda S: 0.5 * np.sum((S @ kv - vv) ** 2), Sp)
    expected = Sp - b * grad
    _, hT = oracle.fwd(np.zeros((1, 1, 1, dk)), kv[None, None, None], vv[None, None, None],
                       np.array([[[b]]]), None, Sp.T[None, None].copy(), qk_l2norm=False)
    np.testing.assert_allclose(hT[0, 0].T, expected, rtol=1e-8, atol=1e-9)


def test_gated_update_minimises_table_objective():
    """[GDN-T1] row Gated DeltaNet: the update is the minimiser of
    L(S) = |S - a S_{t-1}|_F^2 - 2 <S k, b (v - a S_{t-1} k)>; its finite-difference gradient
    vanishes at the oracle's S_t and is nonzero away from it."""
    rng = RNG(13)
    dk, dv = 4, 5
    Sp = rng.standard_normal((dv, dk))
    kv = rng.standard_normal(dk)
    vv = rng.standard_normal(dv)
    a, b = 0.8, 0.6

    def L(S):
        return np.sum((S - a * Sp) ** 2) - 2 * (S @ kv) @ (b * (vv - a * Sp @ kv))

    _, hT = oracle.fwd(np.zeros((1, 1, 1, dk)), kv[None, None, None], vv[None, None, None],
                       np.array([[[b]]]), np.array([[[np.log(a)]]]), Sp.T[None, None].copy(),
                       qk_l2norm=False)
    St = hT[0, 0].T
    assert np.abs(_fd_grad(L, St)).max() < 1e-7
    assert np.abs(_fd_grad(L, St + 0.01)).max() > 1e-3


def test_scalar_closed_form():
    """d_k = d_v = 1: s_t = a_t (1 - b_t k_t^2) s_{t-1} + b_t k_t v_t and o_t = q_t s_t."""
    rng = RNG(14)
    T = 25
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 1, T, 1, 1)
    o, hT = oracle.fwd(q, k, v, beta, g, S0, qk_l2norm=False)
    s = S0[0, 0, 0, 0]
    for t in range(T):
        a = np.exp(g[0, 0, t]); kt = k[0, 0, t, 0]; bt = beta[0, 0, t]
        s = a * (1 - bt * kt * kt) * s + bt * kt * v[0, 0, t, 0]
        assert abs(o[0, 0, t, 0] - q[0, 0, t, 0] * s) <= 1e-12 * (1 + abs(s))
    assert abs(hT[0, 0, 0, 0] - s) <= 1e-12 * (1 + abs(s))


def test_output_uses_state_after_own_write():
    """o_t = q_t S_t (spec reading): from a zero state a single token already reads
    back beta (q_hat . k_hat) v."""
    rng = RNG(15)
    q, k, v, beta, _, _ = _rand_inputs(rng, 1, 1, 1, 8, 3, gated=False, h0=False)
    o, _ = oracle.fwd(q, k, v, beta, None, None, scale=0.5)
    qn = q / np.sqrt((q * q).sum() + oracle.EPS)
    kn = k / np.sqrt((k * k).sum() + oracle.EPS)
    np.testing.assert_allclose(o[0, 0, 0], 0.5 * beta[0, 0, 0] * float(qn[0, 0, 0] @ kn[0, 0, 0]) * v[0, 0, 0],
                               rtol=1e-13)


def test_single_step_from_a_state_is_the_matrix_update():
    """The decode step: from a non-zero state, one token gives S' = alpha (I - beta k k^T) S
    + beta k v^T with the normalised key, and o = scale S'^T q_hat ([GDN] Table 1 row
    Gated DeltaNet, written out as matrices)."""
    rng = RNG(26)
    q, k, v, beta, g, S0 = _rand_inputs(rng, 2, 3, 1, 7, 5)
    o, hT = oracle.fwd(q, k, v, beta, g, S0, scale=0.7)
    for b in range(2):
        for h in range(3):
            kn = k[b, h, 0] / np.sqrt((k[b, h, 0] ** 2).sum() + oracle.EPS)
            qn = q[b, h, 0] / np.sqrt((q[b, h, 0] ** 2).sum() + oracle.EPS)
            a, bt = np.exp(g[b, h, 0]), beta[b, h, 0]
            Sp = a * (np.eye(7) - bt * np.outer(kn, kn)) @ S0[b, h] + bt * np.outer(kn, v[b, h, 0])
            np.testing.assert_allclose(hT[b, h], Sp, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(o[b, h, 0], 0.7 * Sp.T @ qn, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- [GDN-SP], packing
def test_state_passing_split_equals_whole():
    rng = RNG(16)
    q, k, v, beta, g, S0 = _rand_inputs(rng, 2, 2, 90, 6, 5)
    o, hT = oracle.fwd(q, k, v, beta, g, S0)
    o1, h1 = oracle.fwd(q[:, :, :37], k[:, :, :37], v[:, :, :37], beta[:, :, :37], g[:, :, :37], S0)
    o2, h2 = oracle.fwd(q[:, :, 37:], k[:, :, 37:], v[:, :, 37:], beta[:, :, 37:], g[:, :, 37:], h1)
    np.testing.assert_allclose(np.concatenate([o1, o2], 2), o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h2, hT, rtol=1e-12, atol=1e-13)


def test_packed_varlen_equals_separate():
    rng = RNG(17)
    lens = [5, 64, 1, 70, 0, 33]
    cu = np.cumsum([0] + lens)
    Tt = int(cu[-1])
    q, k, v, beta, g, _ = _rand_inputs(rng, 1, 3, Tt, 6, 4)
    S0 = rng.standard_normal((len(lens), 3, 6, 4))
    o, hT = oracle.fwd(q, k, v, beta, g, S0, cu_seqlens=cu)
    for i, L in enumerate(lens):
        a, b = cu[i], cu[i + 1]
        oi, hi = oracle.fwd(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], beta[:, :, a:b],
                            g[:, :, a:b], S0[i:i + 1])
        np.testing.assert_allclose(o[:, :, a:b], oi, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(hT[i:i + 1], hi, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- chunk form (kernels' algebra)
@pytest.mark.parametrize("C", [1, 2, 3, 7, 64])
def test_chunk_form_equals_recurrence(C):
    """The chunk equations the kernels use (UT transform, WY factors, state scan, output)
    reproduce the token recurrence for every chunk size, ragged tail included; C = 1 is
    the recurrence itself."""
    rng = RNG(20 + C)
    L, dk, dv = 150, 8, 6
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 1, L, dk, dv)
    for gg in (g, None):
        o, hT = oracle.fwd(q, k, v, beta, gg, S0, scale=0.7)
        O, S = chunkform.fwd_seq(q[0, 0], k[0, 0], v[0, 0], beta[0, 0],
                                 None if gg is None else gg[0, 0], S0[0, 0], C, scale=0.7)
        np.testing.assert_allclose(O, o[0, 0], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(S, hT[0, 0], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("C", [1, 5, 16, 64])
def test_substituted_chain_equals_recurrence(C):
    """The chain with the state substituted into the next chunk's Unew and output (one
    C x C product on the critical cycle, the state one chunk behind) reproduces the
    token recurrence: gated and not, with an initial state, ragged tail included."""
    rng = RNG(40 + C)
    L, dk, dv = 150, 8, 6
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 1, L, dk, dv)
    for gg in (g, None):
        o, hT = oracle.fwd(q, k, v, beta, gg, S0, scale=0.7)
        O, S = chunkform.fwd_seq_substituted(q[0, 0], k[0, 0], v[0, 0], beta[0, 0],
                                             None if gg is None else gg[0, 0], S0[0, 0], C, scale=0.7)
        np.testing.assert_allclose(O, o[0, 0], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(S, hT[0, 0], rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("C", [1, 5, 64])
def test_chunk_backward_equals_bptt(C):
    rng = RNG(30 + C)
    L, dk, dv = 100, 7, 5
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 1, L, dk, dv)
    dO = rng.standard_normal((1, 1, L, dv))
    dST = rng.standard_normal((1, 1, dk, dv))
    ref = oracle.bwd(q, k, v, beta, g, S0, dO, dST, scale=0.9)
    got = chunkform.bwd_seq(q[0, 0], k[0, 0], v[0, 0], beta[0, 0], g[0, 0], S0[0, 0], dO[0, 0],
                            dST[0, 0], C, scale=0.9)
    for name in ("dq", "dk", "dv", "dbeta", "dg", "dh0"):
        np.testing.assert_allclose(got[name], ref[name][0, 0], rtol=1e-9, atol=1e-11,
                                   err_msg=name)


# ---------------------------------------------------------------- gradients vs finite differences
def _loss(q, k, v, beta, g, S0, dO, dST, **kw):
    o, hT = oracle.fwd(q, k, v, beta, g, S0, **kw)
    return float((o * dO).sum() + (hT * dST).sum())


@pytest.mark.parametrize("gated", [True, False])
def test_bptt_matches_finite_differences_full(gated):
    """Every gradient, every coordinate, central differences in fp64 on a tiny case."""
    rng = RNG(40)
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 1, 9, 3, 2, gated=gated)
    dO = rng.standard_normal((1, 1, 9, 2))
    dST = rng.standard_normal((1, 1, 3, 2))
    kw = dict(scale=1.3)
    grads = oracle.bwd(q, k, v, beta, g, S0, dO, dST, **kw)
    args = dict(q=q, k=k, v=v, beta=beta, g=g, S0=S0)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "S0": "dh0"}
    for name, gname in names.items():
        if args[name] is None:
            continue

        def f(X, name=name):
            a = dict(args); a[name] = X
            return _loss(a["q"], a["k"], a["v"], a["beta"], a["g"], a["S0"], dO, dST, **kw)
        fd = _fd_grad(f, args[name])
        np.testing.assert_allclose(grads[gname], fd, rtol=1e-6, atol=1e-8, err_msg=gname)


def test_bptt_matches_finite_differences_slice():
    """The B1 H1 T128 d16 slice: sampled coordinates of every input and random directions,
    central differences (h = 1e-6), relative agreement <= 1e-6."""
    rng = RNG(41)
    T, d = 128, 16
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 1, T, d, d)
    g = g / 4.0
    dO = rng.standard_normal((1, 1, T, d))
    dST = rng.standard_normal((1, 1, d, d)) * 0.01
    grads = oracle.bwd(q, k, v, beta, g, S0, dO, dST, nthreads=1)
    args = dict(q=q, k=k, v=v, beta=beta, g=g, S0=S0)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "S0": "dh0"}
    h = 1e-6
    for name, gname in names.items():
        X = args[name]
        G = grads[gname]
        idxs = [tuple(int(rng.integers(0, s)) for s in X.shape) for _ in range(12)]
        for idx in idxs:
            Xp = X.copy(); Xp[idx] += h
            Xm = X.copy(); Xm[idx] -= h
            ap = dict(args); ap[name] = Xp
            am = dict(args); am[name] = Xm
            fd = (_loss(**ap, dO=dO, dST=dST, nthreads=1) - _loss(**am, dO=dO, dST=dST, nthreads=1)) / (2 * h)
            assert abs(fd - G[idx]) <= 1e-6 * max(1.0, abs(fd)) + 1e-7, (name, idx, fd, G[idx])
        dirn = rng.standard_normal(X.shape)
        ap = dict(args); ap[name] = X + h * dirn
        am = dict(args); am[name] = X - h * dirn
        fd = (_loss(**ap, dO=dO, dST=dST, nthreads=1) - _loss(**am, dO=dO, dST=dST, nthreads=1)) / (2 * h)
        an = float((G * dirn).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, fd, an)


def test_packed_varlen_backward_equals_separate():
    rng = RNG(42)
    lens = [3, 70, 0, 41]
    cu = np.cumsum([0] + lens)
    Tt = int(cu[-1])
    q, k, v, beta, g, _ = _rand_inputs(rng, 1, 2, Tt, 5, 4)
    S0 = rng.standard_normal((len(lens), 2, 5, 4))
    dO = rng.standard_normal((1, 2, Tt, 4))
    dST = rng.standard_normal((len(lens), 2, 5, 4))
    full = oracle.bwd(q, k, v, beta, g, S0, dO, dST, cu_seqlens=cu)
    for i in range(len(lens)):
        a, b = cu[i], cu[i + 1]
        part = oracle.bwd(q[:, :, a:b], k[:, :, a:b], v[:, :, a:b], beta[:, :, a:b], g[:, :, a:b],
                          S0[i:i + 1], dO[:, :, a:b], dST[i:i + 1])
        for n in ("dq", "dk", "dv", "dbeta", "dg"):
            np.testing.assert_allclose(full[n][:, :, a:b], part[n], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(full["dh0"][i:i + 1], part["dh0"], rtol=1e-12, atol=1e-14)


def test_threads_do_not_change_results():
    rng = RNG(43)
    q, k, v, beta, g, S0 = _rand_inputs(rng, 3, 5, 50, 4, 4)
    o1, h1 = oracle.fwd(q, k, v, beta, g, S0, nthreads=1)
    o2, h2 = oracle.fwd(q, k, v, beta, g, S0, nthreads=7)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


# ---------------------------------------------------------------- [GDN-T1] row Longhorn
@pytest.mark.parametrize("l2norm,gated", [(False, False), (False, True), (True, True)])
def test_longhorn_steps_solve_the_regression_objective(l2norm, gated):
    """[GDN-T1] row Longhorn: each step is the minimiser of
    |S - a S_{t-1}|_F^2 + b |S k - v|^2 (a = 1 without the gate), i.e. the solution of the
    normal equations S (I + b k k^T) = a S_{t-1} + b v k^T, solved here by numpy's dense
    solver token after token (no closed form for the step size)."""
    rng = RNG(50)
    T, dk, dv = 7, 5, 4
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 2, T, dk, dv, gated=gated)
    beta = beta * 3.0                       # step sizes where b |k|^2 is far from 0
    o, hT = oracle.fwd(q, k, v, beta, g, S0, scale=0.8, qk_l2norm=l2norm, longhorn=True)
    for h in range(2):
        S = S0[0, h].T                      # pages' d_v x d_k orientation
        for t in range(T):
            kt, qt = k[0, h, t], q[0, h, t]
            if l2norm:
                kt = kt / np.sqrt((kt ** 2).sum() + oracle.EPS)
                qt = qt / np.sqrt((qt ** 2).sum() + oracle.EPS)
            a = np.exp(g[0, h, t]) if gated else 1.0
            b = beta[0, h, t]
            lhs = np.eye(dk) + b * np.outer(kt, kt)          # symmetric
            S = np.linalg.solve(lhs, (a * S + b * np.outer(v[0, h, t], kt)).T).T
            np.testing.assert_allclose(o[0, h, t], 0.8 * S @ qt, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(hT[0, h], S.T, rtol=1e-11, atol=1e-12)


def test_longhorn_update_is_stationary_point_of_objective():
    """The finite-difference gradient of |S - a S_{t-1}|^2 + b |S k - v|^2 vanishes at the
    oracle's Longhorn state, and not at the plain delta-rule state for the same inputs."""
    rng = RNG(51)
    dk, dv = 4, 3
    Sp = rng.standard_normal((dv, dk))
    kv = rng.standard_normal(dk) * 1.5
    vv = rng.standard_normal(dv)
    a, b = 0.7, 0.9

    def L(S):
        return np.sum((S - a * Sp) ** 2) + b * np.sum((S @ kv - vv) ** 2)

    args = (np.zeros((1, 1, 1, dk)), kv[None, None, None], vv[None, None, None],
            np.array([[[b]]]), np.array([[[np.log(a)]]]), Sp.T[None, None].copy())
    _, hl = oracle.fwd(*args, qk_l2norm=False, longhorn=True)
    _, hd = oracle.fwd(*args, qk_l2norm=False)
    assert np.abs(_fd_grad(L, hl[0, 0].T)).max() < 1e-7
    assert np.abs(_fd_grad(L, hd[0, 0].T)).max() > 1e-2


def test_longhorn_small_step_limit_and_retrieval():
    """As b -> 0 the Longhorn step size b / (1 + b|k|^2) = b - b^2 |k|^2 + ..., so the step
    agrees with the delta rule to first order in b; as b -> inf the stored value is read back exactly under the
    written key (S_t k = v), which the delta rule does only for |k| = 1."""
    rng = RNG(52)
    dk, dv = 6, 3
    q, k, v, _, _, S0 = _rand_inputs(rng, 1, 1, 1, dk, dv, gated=False)
    k = k * 2.0
    diff = []
    for b in (1e-4, 1e-3):
        beta = np.full((1, 1, 1), b)
        _, hl = oracle.fwd(q, k, v, beta, None, S0, qk_l2norm=False, longhorn=True)
        _, hd = oracle.fwd(q, k, v, beta, None, S0, qk_l2norm=False)
        diff.append(np.abs(hl - hd).max())
    # the two steps differ at second order in b: ten times b, a hundred times the gap
    assert 0 < diff[0] < 1e-6 and abs(diff[1] / diff[0] / 100 - 1) < 0.05
    _, hl = oracle.fwd(q, k, v, np.full((1, 1, 1), 1e12), None, S0, qk_l2norm=False, longhorn=True)
    np.testing.assert_allclose(hl[0, 0].T @ k[0, 0, 0], v[0, 0, 0], rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("gated,l2norm", [(True, False), (False, False), (True, True)])
def test_longhorn_bptt_matches_finite_differences(gated, l2norm):
    """Every gradient of the Longhorn loop, every coordinate, central differences in fp64:
    the step size's dependence on beta and on the key is part of what is checked."""
    rng = RNG(53)
    q, k, v, beta, g, S0 = _rand_inputs(rng, 1, 1, 8, 3, 2, gated=gated)
    beta = beta * 2.0
    dO = rng.standard_normal((1, 1, 8, 2))
    dST = rng.standard_normal((1, 1, 3, 2))
    kw = dict(scale=1.1, qk_l2norm=l2norm, longhorn=True)
    grads = oracle.bwd(q, k, v, beta, g, S0, dO, dST, **kw)
    args = dict(q=q, k=k, v=v, beta=beta, g=g, S0=S0)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "S0": "dh0"}
    for name, gname in names.items():
        if args[name] is None:
            continue

        def f(X, name=name):
            a = dict(args); a[name] = X
            return _loss(a["q"], a["k"], a["v"], a["beta"], a["g"], a["S0"], dO, dST, **kw)
        fd = _fd_grad(f, args[name])
        np.testing.assert_allclose(grads[gname], fd, rtol=1e-6, atol=1e-8, err_msg=gname)
