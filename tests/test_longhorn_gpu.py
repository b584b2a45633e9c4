"""GPU parity of Longhorn's step size (DN_BETA_LONGHORN): every token's update uses
beta / (1 + beta k^T k) in place of beta ("Gated DeltaNet" rebuttal, Table 1, row
Longhorn, scalar beta).  The CUDA path, through the C ABI, against the fp64
oracle run with the same option: the general kernels (fp32 and bf16), both tcgen05
forwards, the backward (gradients with respect to the raw beta and k) and the
decode step; with and without the normalisation, where k^T k is far from 1."""
import os

import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL, f64, rel, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GRADS = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gen(B, H, T, d, dtype, gated=True, with_h0=True, seed=0, backward=False, l2=True, lengths=None):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("lh", B, H, T, d, dtype, gated, with_h0, seed, backward=backward,
                           varlen_total=1 if lengths else 0, varlen_n=1 if lengths else 0)
    x = workloads.generate(w, lengths=lengths) if lengths else workloads.generate(w)
    if not l2:
        # unnormalised keys with k^T k of order 1-3: the step size then differs from
        # beta / (1 + beta) token by token
        f = 1.3 / np.sqrt(d)
        x["q"] = (x["q"].float() * f).to(x["q"].dtype)
        x["k"] = (x["k"].float() * f).to(x["k"].dtype)
    return x


def _cu(x):
    return None if x["cu_seqlens"] is None else x["cu_seqlens"].numpy().astype(np.int64)


def _oracle_fwd(x, l2=True, scale=1.0):
    return oracle.fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["beta"]), f64(x["g"]), f64(x["h0"]),
                      cu_seqlens=_cu(x), scale=scale, qk_l2norm=l2, longhorn=True)


def _oracle_bwd(x, l2=True):
    return oracle.bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["beta"]), f64(x["g"]), f64(x["h0"]),
                      f64(x["do"]), f64(x["dhT"]), cu_seqlens=_cu(x), qk_l2norm=l2, longhorn=True)


def _fwd(x, path, l2=True, chunk=64, scale=1.0):
    """Forward through the C ABI on the chosen kernel family."""
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    d = to_dev(x, DEV)
    env = {"GDN_FORCE_GENERAL": "1" if path == "general" else "0",
           "GDN_FUSED_PER_ITEM": "1" if path == "fused" else "0"}
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        shape = gdn.make_shape(d["q"], d["v"], chunk, d["cu_seqlens"], scale, l2, longhorn=True)
        want = {"general": binding.DN_PATH_GENERAL, "fused": binding.DN_PATH_FUSED,
                "coop": binding.DN_PATH_COOP}[path]
        assert binding.dn_plan(shape)[0] == want
        ws = binding.alloc_workspace(shape, False, DEV)
        o = torch.full_like(d["v"], float("nan"))
        N = x["q"].shape[0] if x["cu_seqlens"] is None else x["cu_seqlens"].numel() - 1
        hT = torch.full((N, x["q"].shape[1], x["q"].shape[-1], x["v"].shape[-1]), float("nan"),
                        device=DEV)
        if d["g"] is None:
            gdn.dn_chunk_fwd(shape, d["q"], d["k"], d["v"], d["beta"], d["h0"], o, hT, ws)
        else:
            gdn.gdn_chunk_fwd(shape, d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], o, hT, ws)
        torch.cuda.synchronize()
        assert gdn.dn_device_status(ws) == 0
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v
    return o.float().cpu().numpy(), hT.cpu().numpy()


def _check(name, got, ref, tol):
    e = rel(got, ref)
    assert e <= tol, "%s: relative error %.3e > %.1e" % (name, e, tol)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,d,chunk", [(1, 16, 64), (65, 64, 64), (200, 48, 32), (130, 256, 64)])
@pytest.mark.parametrize("l2", [True, False])
def test_longhorn_forward_general(dtype, T, d, chunk, l2):
    x = _gen(2, 2, T, d, dtype, gated=T % 2 == 0, seed=300 + T + d, l2=l2)
    o, hT = _fwd(x, "general", l2=l2, chunk=chunk, scale=0.9)
    ro, rh = _oracle_fwd(x, l2=l2, scale=0.9)
    _check("o", o, ro, TOL[dtype])
    _check("hT", hT, rh, TOL[dtype])


@pytest.mark.parametrize("path", ["coop", "fused"])
@pytest.mark.parametrize("T,gated,l2", [(64, True, True), (65, False, True), (200, True, False),
                                        (1000, True, True)])
def test_longhorn_forward_tcgen05(path, T, gated, l2):
    x = _gen(1, 2, T, 128, "bf16", gated=gated, seed=400 + T, l2=l2)
    o, hT = _fwd(x, path, l2=l2)
    ro, rh = _oracle_fwd(x, l2=l2)
    _check("o", o, ro, TOL["bf16"])
    _check("hT", hT, rh, TOL["bf16"])


@pytest.mark.parametrize("path", ["coop", "fused", "general"])
def test_longhorn_forward_varlen(path):
    x = _gen(1, 3, 0, 128, "bf16", seed=41, lengths=[1, 130, 64, 0, 257])
    o, hT = _fwd(x, path)
    ro, rh = _oracle_fwd(x)
    _check("o", o, ro, TOL["bf16"])
    _check("hT", hT, rh, TOL["bf16"])


def test_longhorn_is_not_the_delta_rule():
    """The option reaches the kernels: the same inputs without it give a different
    output, which matches the oracle's plain delta rule instead."""
    import chunkwise_delta_rule_02_gb300 as gdn
    x = _gen(1, 2, 130, 128, "bf16", seed=43)
    d = to_dev(x, DEV)
    o_lh, _ = _fwd(x, "coop")
    o_dn, _ = gdn.forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    o_dn = o_dn.float().cpu().numpy()
    ro, _ = oracle.fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["beta"]), f64(x["g"]), f64(x["h0"]))
    assert rel(o_dn, ro) <= TOL["bf16"]
    assert rel(o_lh, o_dn) > 10 * TOL["bf16"]


def _bwd(x, l2=True, chunk=64):
    import chunkwise_delta_rule_02_gb300 as gdn
    d = to_dev(x, DEV)
    out = gdn.backward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["do"], d["dhT"],
                       cu_seqlens=d["cu_seqlens"], chunk=chunk, qk_l2norm=l2, longhorn=True)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.float().cpu().numpy()) for k, v in out.items()}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,d,gated,l2", [(1, 16, True, True), (65, 64, True, False),
                                          (130, 128, False, True), (97, 128, True, False)])
def test_longhorn_backward(dtype, T, d, gated, l2):
    x = _gen(2, 2, T, d, dtype, gated=gated, seed=500 + T + d, backward=True, l2=l2)
    got = _bwd(x, l2=l2)
    ref = _oracle_bwd(x, l2=l2)
    for n in GRADS:
        if ref[n] is None:
            continue
        _check(n, got[n], ref[n], TOL[dtype])


def test_longhorn_backward_varlen():
    x = _gen(1, 2, 0, 128, "bf16", seed=51, backward=True, lengths=[70, 1, 0, 190])
    got = _bwd(x)
    ref = _oracle_bwd(x)
    for n in GRADS:
        _check(n, got[n], ref[n], TOL["bf16"])


@pytest.mark.parametrize("l2,lengths", [(True, None), (False, [70, 1, 0, 190])])
def test_longhorn_saved_path(l2, lengths):
    """Longhorn's step size through the training path: forward(save=True) keeps the
    chunk operands the cooperative forward prepared with it, backward(saved=...) starts
    at the reverse scan over them.  The gradients equal the recompute path's (dg up to
    the order of its atomic row sums) and match the oracle."""
    import chunkwise_delta_rule_02_gb300 as gdn
    x = _gen(2, 2, 333, 128, "bf16", seed=71, backward=True, l2=l2) if lengths is None else \
        _gen(1, 2, 0, 128, "bf16", seed=72, backward=True, l2=l2, lengths=lengths)
    d = to_dev(x, DEV)
    kw = dict(cu_seqlens=d["cu_seqlens"], qk_l2norm=l2, longhorn=True)
    if not gdn.saved_supported(d["q"], d["v"], cu_seqlens=d["cu_seqlens"]):
        pytest.skip("no saved path on this device")
    o1, h1, saved = gdn.forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], save=True, **kw)
    o2, h2 = gdn.forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], **kw)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    a = gdn.backward(d["q"], d["k"], d["v"], d["beta"], d["g"], None, d["do"], d["dhT"], saved=saved, **kw)
    b = gdn.backward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["do"], d["dhT"], **kw)
    torch.cuda.synchronize()
    for n in GRADS:
        if n == "dg":
            assert (a[n] - b[n]).abs().max() <= 1e-6 * b[n].abs().max()
        else:
            assert torch.equal(a[n], b[n]), n
    ref = _oracle_bwd(x, l2=l2)
    for n in GRADS:
        _check(n, a[n].float().cpu().numpy(), ref[n], TOL["bf16"])


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 64), ("bf16", 96, 30)])
@pytest.mark.parametrize("l2", [True, False])
def test_longhorn_decode_steps(dtype, dk, dv, l2):
    """Chained decode steps with the option against the oracle's token loop."""
    import chunkwise_delta_rule_02_gb300 as gdn
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    gen = torch.Generator().manual_seed(61 + dk + dv)
    N, H, T = 2, 3, 12
    f = 1.0 if l2 else 1.3 / np.sqrt(dk)
    q = (torch.randn(N, H, T, dk, generator=gen) * f).to(tdt)
    k = (torch.randn(N, H, T, dk, generator=gen) * f).to(tdt)
    v = torch.randn(N, H, T, dv, generator=gen).to(tdt)
    beta = (torch.rand(N, H, T, generator=gen) * 2.0).to(tdt)
    g = -torch.rand(N, H, T, generator=gen) * 0.3
    S0 = torch.randn(N, H, dk, dv, generator=gen) * 0.2
    ro, rh = oracle.fwd(f64(q), f64(k), f64(v), f64(beta), f64(g), f64(S0), scale=0.7,
                        qk_l2norm=l2, longhorn=True)
    state = S0.to(DEV)
    outs = []
    for t in range(T):
        args = [x[:, :, t].contiguous().to(DEV) for x in (q, k, v, beta, g)]
        o, state = gdn.decode_step(*args, state=state, out_state=state, scale=0.7, qk_l2norm=l2,
                                   longhorn=True)
        outs.append(o.float())
    torch.cuda.synchronize()
    o = torch.stack(outs, 2).cpu().numpy()
    _check("o", o, ro, TOL[dtype])
    _check("state", state.cpu().numpy(), rh, TOL[dtype])
