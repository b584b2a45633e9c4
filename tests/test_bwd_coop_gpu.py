"""The backward's recompute through the cooperative forward (bf16, d_k = d_v = 128,
chunk 64): one run of the forward kernel that also writes every chunk's prepared
operands, S_in and Unew; the reverse dS scan over those operands (k_bscan_pk); the
tcgen05 per-chunk gradients.  Against the fp64 oracle, and against the general
kernels' recompute of the same gradients (GDN_BWD_RECOMPUTE=1): chunk states are
recomputed in the backward (DeltaNet page, reply Q2), and both recomputes must give
the oracle's gradients."""
import os

import numpy as np
import pytest
import torch

from parity_util import TOL, oracle_bwd, rel, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
GRADS = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gen(B, H, T, seed, lengths=None, gated=True, with_h0=True):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("bwc", B, H, T, 128, "bf16", gated, with_h0, seed, backward=True,
                           varlen_total=1 if lengths else 0, varlen_n=1 if lengths else 0)
    return workloads.generate(w, lengths=lengths) if lengths else workloads.generate(w)


def _bwd(x, env=None):
    import chunkwise_delta_rule_02_gb300 as gdn
    env = env or {}
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        d = to_dev(x, DEV)
        out = gdn.backward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["do"], d["dhT"],
                           cu_seqlens=d["cu_seqlens"])
        torch.cuda.synchronize()
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v
    return {k: (None if v is None else v.float().cpu().numpy()) for k, v in out.items()}


def _plan(x, env):
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    old = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    try:
        d = to_dev(x, DEV)
        return binding.dn_plan(gdn.make_shape(d["q"], d["v"], 64, d["cu_seqlens"]), True)
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


def _coop_here(x):
    from chunkwise_delta_rule_02_gb300 import binding
    return _plan(x, {})[1] == 3


def test_plan_takes_the_cooperative_recompute():
    """Three kernels (k_coop_fwd, k_bscan_pk, k_bwd_tc); the general recompute has four
    (k_prep_st, k_scan_st, k_bscan_st, k_bwd_tc)."""
    from chunkwise_delta_rule_02_gb300 import binding
    x = _gen(1, 2, 128, seed=1)
    if not _coop_here(x):
        pytest.skip("the cooperative kernel is not available on this device")
    assert _plan(x, {}) == (binding.DN_PATH_GENERAL, 3)
    assert _plan(x, {"GDN_BWD_RECOMPUTE": "1"}) == (binding.DN_PATH_GENERAL, 4)
    assert _plan(x, {"GDN_FORCE_GENERAL": "1"}) == (binding.DN_PATH_GENERAL, 4)
    xv = _gen(1, 2, 0, seed=2, lengths=[5, 130])
    assert _plan(xv, {}) == (binding.DN_PATH_GENERAL, 5)   # + k_cstart, k_plan


@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 777])
@pytest.mark.parametrize("gated,h0", [(True, True), (False, False)])
def test_small_and_ragged(T, gated, h0):
    x = _gen(2, 2, T, seed=900 + T, gated=gated, with_h0=h0)
    got = _bwd(x)
    ref = oracle_bwd(x)
    for n in GRADS:
        if ref[n] is None:
            assert got[n] is None
            continue
        assert np.isfinite(got[n]).all(), n
        assert rel(got[n], ref[n]) <= TOL["bf16"], (n, rel(got[n], ref[n]))


def test_packed_sequences():
    """Chunk slots of packed sequences (empty, one-token and ragged ones among them):
    the forward writes each chunk's operands where the reverse scan and the per-chunk
    gradients look for them."""
    x = _gen(1, 3, 0, seed=31, lengths=[5, 64, 0, 130, 1, 63, 300])
    got = _bwd(x)
    ref = oracle_bwd(x)
    for n in GRADS:
        assert rel(got[n], ref[n]) <= TOL["bf16"], (n, rel(got[n], ref[n]))


def test_matches_the_general_recompute():
    """More (sequence, head) items than chain CTAs, against the general kernels'
    recompute on the same inputs (both are bf16 pipelines with fp32 accumulation)."""
    x = _gen(8, 16, 200, seed=32)
    a = _bwd(x)
    b = _bwd(x, {"GDN_BWD_RECOMPUTE": "1"})
    for n in GRADS:
        assert rel(a[n], b[n]) <= 1e-2, (n, rel(a[n], b[n]))
    sel = [(0, 0), (7, 15)]
    for (bi, h), r in zip(sel, oracle_bwd(x, sel=sel)):
        for n in GRADS:
            assert rel(a[n][bi:bi + 1, h:h + 1], r[n]) <= TOL["bf16"], (n, bi, h)


def test_timeout_in_the_recompute_is_reported():
    """A withheld package (the test hook of the cooperative kernel) makes the
    recompute's bounded wait run out: gdn_chunk_bwd still returns, the status word
    says DN_ERR_TIMEOUT, and the next call is correct."""
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    x = _gen(1, 2, 24 * 64, seed=33)
    if not _coop_here(x):
        pytest.skip("the cooperative kernel is not available on this device")
    d = to_dev(x, DEV)
    shape = gdn.make_shape(d["q"], d["v"])
    ws = binding.alloc_workspace(shape, True, DEV)
    outs = [torch.empty_like(d[n]) for n in ("q", "k", "v", "beta")] + [torch.empty_like(d["g"]),
                                                                      torch.empty_like(d["h0"])]
    args = (shape, d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["do"], d["dhT"], *outs, ws)
    os.environ["GDN_DEBUG_WITHHOLD_TASK"] = "5"
    try:
        binding.gdn_chunk_bwd(*args)
        assert binding.dn_device_status(ws) == binding.DN_ERR_TIMEOUT
    finally:
        del os.environ["GDN_DEBUG_WITHHOLD_TASK"]
    binding.gdn_chunk_bwd(*args)
    assert binding.dn_device_status(ws) == binding.DN_OK
    got = dict(zip(("dq", "dk", "dv", "dbeta", "dg", "dh0"), (t.float().cpu().numpy() for t in outs)))
    ref = oracle_bwd(x)
    for n in GRADS:
        assert rel(got[n], ref[n]) <= TOL["bf16"], n


# ----------------------------------------------------------------------------- the saved path
def _saved_case(x):
    import chunkwise_delta_rule_02_gb300 as gdn
    d = to_dev(x, DEV)
    if not gdn.saved_supported(d["q"], d["v"], cu_seqlens=d["cu_seqlens"]):
        pytest.skip("no saved path on this device")
    return d


@pytest.mark.parametrize("lengths", [None, [5, 64, 0, 130, 1, 63, 300]])
def test_saved_path_equals_the_recompute(lengths):
    """gdn_chunk_fwd_save writes what the backward's recompute writes (the same kernel on
    the same inputs), so its o, h_T and the gradients of gdn_chunk_bwd_saved equal
    gdn_chunk_fwd's and gdn_chunk_bwd's bit for bit (dg up to the order of its atomic
    row sums); and they match the oracle."""
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    x = _gen(2, 3, 333, seed=34) if lengths is None else _gen(1, 3, 0, seed=35, lengths=lengths)
    d = _saved_case(x)
    kw = dict(cu_seqlens=d["cu_seqlens"])
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
    ref = oracle_bwd(x)
    for n in GRADS:
        assert rel(a[n].float().cpu().numpy(), ref[n]) <= TOL["bf16"], n
    shape = gdn.make_shape(d["q"], d["v"], 64, d["cu_seqlens"])
    assert binding.dn_plan(shape, 2) == (binding.DN_PATH_GENERAL, 2 + (1 if lengths else 0))
    assert binding.dn_workspace_size(shape, 2) < binding.dn_workspace_size(shape, 1)


def test_saved_path_ungated_without_initial_state():
    """DeltaNet (no gate) from a zero initial state through the saved path: dg is absent;
    the other gradients (dh0 with respect to the zero state among them) equal the
    recompute path's and match the oracle."""
    import chunkwise_delta_rule_02_gb300 as gdn
    x = _gen(2, 2, 200, seed=38, gated=False, with_h0=False)
    d = _saved_case(x)
    o, hT, saved = gdn.forward(d["q"], d["k"], d["v"], d["beta"], None, None, save=True)
    a = gdn.backward(d["q"], d["k"], d["v"], d["beta"], None, None, d["do"], d["dhT"], saved=saved)
    b = gdn.backward(d["q"], d["k"], d["v"], d["beta"], None, None, d["do"], d["dhT"])
    torch.cuda.synchronize()
    assert a["dg"] is None
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        assert torch.equal(a[n], b[n]), n
    ref = oracle_bwd(x)
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        if ref[n] is not None:
            assert rel(a[n].float().cpu().numpy(), ref[n]) <= TOL["bf16"], n


def test_saved_path_refuses_other_shapes():
    """d 64: no saved path (dn_saved_size 0, DN_ERR_UNSUPPORTED)."""
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding, workloads
    w = workloads.Workload("ns", 1, 2, 64, 64, "bf16", True, True, 1, backward=True)
    d = to_dev(workloads.generate(w), DEV)
    assert not gdn.saved_supported(d["q"], d["v"])
    with pytest.raises(gdn.GdnError) as err:
        gdn.forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], save=True)
    assert err.value.status == binding.DN_ERR_UNSUPPORTED


# ----------------------------------------------------------------------------- the tcgen05 reverse scan
def test_tc_reverse_scan_matches_the_warp_level_scan():
    """k_bscan_tc (dS in TMEM) against k_bscan_pk (GDN_BSCAN_STAGED=1) on the same
    packages, with more (sequence, head) items than SMs (a CTA takes several, each
    from its last chunk to its first), and against the oracle on sampled items."""
    x = _gen(8, 20, 300, seed=36)
    a = _bwd(x)
    b = _bwd(x, {"GDN_BSCAN_STAGED": "1"})
    for n in GRADS:
        assert rel(a[n], b[n]) <= 1e-2, (n, rel(a[n], b[n]))
    sel = [(0, 0), (5, 13), (7, 19)]
    for (bi, h), r in zip(sel, oracle_bwd(x, sel=sel)):
        for n in GRADS:
            assert rel(a[n][bi:bi + 1, h:h + 1], r[n]) <= TOL["bf16"], (n, bi, h)


def test_tc_reverse_scan_strong_decay():
    """Chunk decays near exp(-130): the reverse scan's pending scale renormalises the
    TMEM state within a sequence."""
    x = _gen(1, 2, 700, seed=37)
    x["g"] = x["g"] * 40.0
    x["beta"] = torch.ones_like(x["beta"])
    got = _bwd(x)
    ref = oracle_bwd(x)
    for n in GRADS:
        assert np.isfinite(got[n]).all(), n
        assert rel(got[n], ref[n]) <= TOL["bf16"], (n, rel(got[n], ref[n]))
