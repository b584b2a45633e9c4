"""fp64 CPU oracle for the (gated) delta rule — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The library
(``chunkwise_delta_rule_02_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, token by token); this
module only compiles it with gcc and marshals numpy arrays through ctypes.

What it follows:
  * forward — "Gated DeltaNet: Improving Mamba2 with Delta Rule", rebuttal
    Table 1, rows "DeltaNet" (alpha = 1) and "Gated DeltaNet":
    S_t = S_{t-1}(alpha_t (I - beta_t k_t k_t^T)) + beta_t v_t k_t^T, stored
    transposed (d_k x d_v), read out as o_t = scale * q_t S_t;
    with ``longhorn=True`` the step size is Longhorn's
    beta_t / (1 + beta_t k_t^T k_t) in place of beta_t (same Table 1, row
    "Longhorn", with its scalar beta);
  * backward — back-propagation through time of that loop, written by hand;
    the DeltaNet page ("Parallelizing Linear Transformers with the Delta Rule
    over Sequence Length", reply Q2 on chunk states) fixes only that the
    backward recomputes states, which the checkpointed segments here also do.

Every function is pinned by ``tests/test_oracle_pins.py`` against facts the
pages and the mathematics fix (explicit Householder products, the WY form,
exact retrieval, the one-step gradient-descent reading of Table 1, closed
forms, state passing, finite differences).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

EPS = 1e-6  # the normalisation's epsilon: x / sqrt(sum(x^2) + EPS)


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``liboracle.so`` (portable C, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.gdn_oracle_fwd.restype = I
            lib.gdn_oracle_fwd.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, I, D, D, I, P, P, I]
            lib.gdn_oracle_bwd.restype = I
            lib.gdn_oracle_bwd.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, I, D, D, I,
                                           P, P, P, P, P, P, P, P, I]
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    return None if x is None else x.ctypes.data


def _threads(nthreads):
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    return int(nthreads)


def _dims(q, v, cu_seqlens):
    NB, H, Ttot, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        return NB, NB, H, Ttot, dk, dv, None
    offs = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    if NB != 1:
        raise ValueError("packed variable-length input must have batch dimension 1")
    return len(offs) - 1, NB, H, Ttot, dk, dv, offs


def fwd(q, k, v, beta, g=None, h0=None, cu_seqlens=None, scale=1.0,
        qk_l2norm=True, eps=EPS, nthreads=None, longhorn=False):
    """Token-by-token forward (``longhorn``: Longhorn's step size).  Arrays: q,k [NB,H,T,dk], v [NB,H,T,dv],
    beta,g [NB,H,T], h0 [N,H,dk,dv] (N = NB, or the number of packed sequences).
    Returns (o [NB,H,T,dv], hT [N,H,dk,dv]) in float64."""
    q, k, v, beta, g, h0 = map(_f64, (q, k, v, beta, g, h0))
    n_seqs, NB, H, Ttot, dk, dv, offs = _dims(q, v, cu_seqlens)
    o = np.zeros((NB, H, Ttot, dv), np.float64)
    hT = np.zeros((n_seqs, H, dk, dv), np.float64)
    rc = _load().gdn_oracle_fwd(n_seqs, NB, H, Ttot, dk, dv, _ptr(offs), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), int(bool(qk_l2norm)),
                                float(scale), float(eps), int(bool(longhorn)), _ptr(o), _ptr(hT),
                                _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle forward failed with code %d" % rc)
    return o, hT


def bwd(q, k, v, beta, g=None, h0=None, do=None, dhT=None, cu_seqlens=None, scale=1.0,
        qk_l2norm=True, eps=EPS, nthreads=None, longhorn=False):
    """Back-propagation through time of :func:`fwd` for the loss
    sum(o * do) + sum(hT * dhT).  Returns dict with dq, dk, dv, dbeta, dg (None when
    g is None) and dh0, all float64."""
    q, k, v, beta, g, h0, do, dhT = map(_f64, (q, k, v, beta, g, h0, do, dhT))
    n_seqs, NB, H, Ttot, dk, dv, offs = _dims(q, v, cu_seqlens)
    if do is None:
        do = np.zeros((NB, H, Ttot, dv), np.float64)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dbeta=np.zeros_like(beta),
               dg=np.zeros_like(beta) if g is not None else None,
               dh0=np.zeros((n_seqs, H, dk, dv), np.float64))
    rc = _load().gdn_oracle_bwd(n_seqs, NB, H, Ttot, dk, dv, _ptr(offs), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(beta), _ptr(g), _ptr(h0), int(bool(qk_l2norm)),
                                float(scale), float(eps), int(bool(longhorn)), _ptr(do), _ptr(dhT),
                                _ptr(out["dq"]),
                                _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dbeta"]),
                                _ptr(out["dg"]), _ptr(out["dh0"]), _threads(nthreads))
    if rc != 0:
        raise RuntimeError("oracle backward failed with code %d" % rc)
    return out
