"""GPU parity: the CUDA path, called through the C ABI, against the fp64 oracle on
the same seeded inputs.  Tolerance: relative Frobenius error per tensor, 1e-4 for
float32 inputs and 2e-2 for bfloat16 inputs, on o, the final state and every
gradient.  bf16 inputs reach the oracle as their rounded values upcast to fp64,
so the error measured is the kernels', not the input quantisation's."""
import numpy as np
import pytest
import torch

from parity_util import TOL, f64, oracle_bwd, oracle_fwd, rel, to_dev

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gdn():
    import chunkwise_delta_rule_02_gb300 as gdn
    return gdn


def _w(name):
    from chunkwise_delta_rule_02_gb300 import workloads
    return workloads.WORKLOADS[name]


def _gen(name, **kw):
    from chunkwise_delta_rule_02_gb300 import workloads
    return workloads.generate(_w(name), **kw)


def _run_fwd(x, **kw):
    d = to_dev(x, DEV)
    o, hT = _gdn().forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"],
                           cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), hT.cpu().numpy()


def _assert_close(name, got, ref, tol):
    e = rel(got, ref)
    assert e <= tol, "%s: relative error %.3e > %.1e" % (name, e, tol)
    return e


# ----------------------------------------------------------------------------- small sweeps
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
@pytest.mark.parametrize("d", [16, 64, 128])
def test_forward_small(dtype, T, d):
    base = "gdn_fwd_bf16_b4h16t8192d128_h0"
    from chunkwise_delta_rule_02_gb300 import workloads
    w = _w(base)
    w = workloads.Workload(w.name, 2, 2, T, d, dtype, gated=(T + d) % 2 == 0,
                           with_h0=(T % 3 != 0), seed=100 + T + d)
    x = workloads.generate(w)
    o, hT = _run_fwd(x)
    ro, rh = oracle_fwd(x)
    _assert_close("o", o, ro, TOL[dtype])
    _assert_close("hT", hT, rh, TOL[dtype])


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward_chunk_sizes_and_options(chunk, dtype):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("opt", 1, 3, 150, 48, dtype, True, True, seed=7 + chunk)
    x = workloads.generate(w)
    # rectangular heads: dv != dk
    x["v"] = x["v"][..., :40].contiguous()
    x["h0"] = x["h0"][..., :40].contiguous()
    for scale, l2 in ((1.0, True), (0.125, True), (1.0, False)):
        xx = dict(x)
        if not l2:   # keep magnitudes sane without the normalisation
            xx["q"] = (x["q"].float() / 7.0).to(x["q"].dtype)
            xx["k"] = (x["k"].float() / 7.0).to(x["k"].dtype)
        o, hT = _run_fwd(xx, chunk=chunk, scale=scale, qk_l2norm=l2)
        import oracle
        ro, rh = oracle.fwd(f64(xx["q"]), f64(xx["k"]), f64(xx["v"]), f64(xx["beta"]), f64(xx["g"]),
                            f64(xx["h0"]), scale=scale, qk_l2norm=l2)
        _assert_close("o", o, ro, TOL[dtype])
        _assert_close("hT", hT, rh, TOL[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_forward_varlen_small(dtype):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("vl", 1, 3, 0, 64, dtype, True, True, seed=11, varlen_total=1, varlen_n=1)
    x = workloads.generate(w, lengths=[5, 64, 0, 1, 130, 65, 200, 63])
    o, hT = _run_fwd(x)
    ro, rh = oracle_fwd(x)
    _assert_close("o", o, ro, TOL[dtype])
    _assert_close("hT", hT, rh, TOL[dtype])


def test_empty_sequence_passes_state_through():
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("empty", 2, 2, 0, 32, "f32", True, True, seed=3)
    x = workloads.generate(w)
    o, hT = _run_fwd(x)
    assert o.size == 0
    np.testing.assert_array_equal(hT, x["h0"].numpy())


def test_beta_zero_is_pure_decay():
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("b0", 1, 2, 130, 64, "f32", True, True, seed=4)
    x = workloads.generate(w)
    x["beta"] = torch.zeros_like(x["beta"])
    _, hT = _run_fwd(x)
    decay = torch.exp(x["g"].double().sum(-1)).numpy()[..., None, None]
    np.testing.assert_allclose(hT, decay * x["h0"].double().numpy(), rtol=1e-5, atol=1e-7)


def test_state_passing_across_calls():
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("sp", 2, 2, 300, 64, "f32", True, True, seed=5)
    x = workloads.generate(w)
    o, hT = _run_fwd(x)
    a = {k: (v[:, :, :130].contiguous() if k in ("q", "k", "v", "beta", "g") else v) for k, v in x.items()}
    o1, h1 = _run_fwd(a)
    b = {k: (v[:, :, 130:].contiguous() if k in ("q", "k", "v", "beta", "g") else v) for k, v in x.items()}
    b["h0"] = torch.from_numpy(h1)
    o2, h2 = _run_fwd(b)
    assert rel(np.concatenate([o1, o2], 2), o) <= 1e-5
    assert rel(h2, hT) <= 1e-5


def test_bad_offsets_are_reported_on_device():
    gdn = _gdn()
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("bad", 1, 2, 0, 32, "f32", True, False, seed=6, varlen_total=1, varlen_n=1)
    x = workloads.generate(w, lengths=[10, 5, 5])
    d = to_dev(x, DEV)
    d["cu_seqlens"] = torch.tensor([0, 10, 5, 20], dtype=torch.int32, device=DEV)  # not monotone
    shape = gdn.make_shape(d["q"], d["v"], cu_seqlens=d["cu_seqlens"])
    ws = gdn.binding.alloc_workspace(shape, False, DEV)
    o = torch.zeros_like(d["v"])
    hT = torch.zeros((3, 2, 32, 32), device=DEV)
    gdn.gdn_chunk_fwd(shape, d["q"], d["k"], d["v"], d["beta"], d["g"], None, o, hT, ws)
    assert gdn.dn_device_status(ws) == gdn.binding.DN_ERR_INVALID_ARG
    assert gdn.dn_device_status(ws) == gdn.binding.DN_OK   # reading clears it


# ----------------------------------------------------------------------------- full-size workloads
def test_dn_fwd_f32_b1h2t256d64():
    x = _gen("dn_fwd_f32_b1h2t256d64")
    o, hT = _run_fwd(x)
    ro, rh = oracle_fwd(x)
    _assert_close("o", o, ro, 1e-4)
    _assert_close("hT", hT, rh, 1e-4)


@pytest.mark.parametrize("name,sel", [
    ("dn_fwd_bf16_b8h16t2048d128", [(0, 0), (3, 7), (7, 15), (5, 2)]),
    ("gdn_fwd_bf16_b4h16t8192d128_h0", [(0, 0), (1, 9), (3, 15), (2, 4)]),
    ("gdn_fwd_bf16_b4h16t8192d128_c32_h0", [(0, 0), (2, 11), (3, 15)]),
    ("gdn_fwd_bf16_b4h8t8192d256_c32_h0", [(0, 0), (1, 5), (3, 7)]),
])
def test_full_size_forward_sampled(name, sel):
    """Full-size launch (the benchmark's configuration); the oracle recomputes sampled
    (batch, head) items, each over its whole sequence."""
    x = _gen(name)
    o, hT = _run_fwd(x, chunk=_w(name).chunk)
    refs = oracle_fwd(x, sel=sel)
    for (b, h), (ro, rh) in zip(sel, refs):
        _assert_close("o[%d,%d]" % (b, h), o[b:b + 1, h:h + 1], ro, TOL["bf16"])
        _assert_close("hT[%d,%d]" % (b, h), hT[b:b + 1, h:h + 1], rh, TOL["bf16"])
    assert np.isfinite(o).all() and np.isfinite(hT).all()


def test_full_size_varlen_sampled():
    import oracle
    x = _gen("gdn_fwd_bf16_varlen_h32_n8_t65536")
    o, hT = _run_fwd(x)
    cu = x["cu_seqlens"].tolist()
    for s, h in [(0, 0), (3, 17), (7, 31)]:
        a, b = cu[s], cu[s + 1]
        sl = lambda t: t[:, h:h + 1, a:b]
        ro, rh = oracle.fwd(f64(sl(x["q"])), f64(sl(x["k"])), f64(sl(x["v"])), f64(sl(x["beta"])),
                            f64(sl(x["g"])), None)
        _assert_close("o[s%d,h%d]" % (s, h), o[:, h:h + 1, a:b], ro, TOL["bf16"])
        _assert_close("hT[s%d,h%d]" % (s, h), hT[s:s + 1, h:h + 1], rh, TOL["bf16"])
    assert np.isfinite(o).all()


# ----------------------------------------------------------------------------- backward
def _run_bwd(x, **kw):
    d = to_dev(x, DEV)
    out = _gdn().backward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], d["do"], d["dhT"],
                          cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return {k: (None if v is None else v.float().cpu().numpy()) for k, v in out.items()}


GRADS = ("dq", "dk", "dv", "dbeta", "dg", "dh0")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,d", [(1, 16), (65, 64), (130, 128), (64, 32)])
def test_backward_small(dtype, T, d):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("bw", 2, 2, T, d, dtype, True, True, seed=200 + T + d, backward=True)
    x = workloads.generate(w)
    got = _run_bwd(x)
    ref = oracle_bwd(x)
    for n in GRADS:
        _assert_close(n, got[n], ref[n], TOL[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,dk,dv,chunk", [(130, 256, 256, 64), (97, 256, 192, 32), (64, 160, 256, 16)])
def test_head_dim_256_forward_and_backward(dtype, T, dk, dv, chunk):
    """Head dims up to 256 (the Gated DeltaNet head size) on the general kernels,
    including d_k != d_v, ragged chunks and the smaller chunk sizes."""
    from chunkwise_delta_rule_02_gb300 import workloads
    import oracle as orc
    w = workloads.Workload("d256", 1, 2, T, dk, dtype, True, True, seed=T + dk + dv, chunk=chunk,
                           backward=True)
    x = workloads.generate(w)
    if dv != dk:   # the generator draws square heads: cut v, h0, do, dhT to d_v columns
        for key in ("v", "do"):
            x[key] = x[key][..., :dv].contiguous()
        for key in ("h0", "dhT"):
            x[key] = x[key][..., :dv].contiguous()
    o, hT = _run_fwd(x, chunk=chunk)
    ro, rh = oracle_fwd(x)
    _assert_close("o", o, ro, TOL[dtype])
    _assert_close("hT", hT, rh, TOL[dtype])
    got = _run_bwd(x, chunk=chunk)
    ref = oracle_bwd(x)
    for n in GRADS:
        _assert_close(n, got[n], ref[n], TOL[dtype])


@pytest.mark.parametrize("T,dk,dv,chunk", [(130, 64, 128, 32), (97, 128, 64, 64), (70, 32, 32, 32),
                                          (64, 128, 32, 64), (33, 64, 64, 32)])
def test_staged_bf16_shapes_forward_and_backward(T, dk, dv, chunk):
    """The staged bf16 kernels (power-of-two head dims 32-128, chunks of 32 or 64):
    d_k != d_v both ways, chunk 32 (column solve) and 64 (blocked solve), ragged tails."""
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("stg", 2, 2, T, max(dk, dv), "bf16", True, True, seed=3 * T + dk + dv,
                           chunk=chunk, backward=True)
    x = workloads.generate(w)
    for key in ("q", "k"):
        x[key] = x[key][..., :dk].contiguous()
    for key in ("v", "do"):
        x[key] = x[key][..., :dv].contiguous()
    for key in ("h0", "dhT"):
        x[key] = x[key][:, :, :dk, :dv].contiguous()
    o, hT = _run_fwd(x, chunk=chunk)
    ro, rh = oracle_fwd(x)
    _assert_close("o", o, ro, TOL["bf16"])
    _assert_close("hT", hT, rh, TOL["bf16"])
    got = _run_bwd(x, chunk=chunk)
    ref = oracle_bwd(x)
    for n in GRADS:
        _assert_close(n, got[n], ref[n], TOL["bf16"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_varlen_small(dtype):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("bwv", 1, 2, 0, 32, dtype, True, True, seed=21, varlen_total=1,
                           varlen_n=1, backward=True)
    x = workloads.generate(w, lengths=[70, 0, 1, 64, 129])
    got = _run_bwd(x)
    ref = oracle_bwd(x)
    for n in GRADS:
        _assert_close(n, got[n], ref[n], TOL[dtype])


def test_backward_ungated():
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("bwu", 1, 2, 100, 32, "f32", False, False, seed=22, backward=True)
    x = workloads.generate(w)
    got = _run_bwd(x)
    ref = oracle_bwd(x)
    assert got["dg"] is None
    for n in ("dq", "dk", "dv", "dbeta", "dh0"):
        _assert_close(n, got[n], ref[n], 1e-4)


def test_backward_finite_difference_slice():
    """The B1 H1 T128 d16 slice: the GPU gradients (fp32 inputs) against central finite
    differences of the fp64 oracle's loss <o, dO> + <hT, dhT>, along random directions."""
    import oracle
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("fd", 1, 1, 128, 16, "f32", True, True, seed=4, backward=True)
    x = workloads.generate(w)
    got = _run_bwd(x)
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "h0": "dh0"}
    args = {n: f64(x[n]) for n in names}
    dO, dST = f64(x["do"]), f64(x["dhT"])

    def loss(a):
        o, hT = oracle.fwd(a["q"], a["k"], a["v"], a["beta"], a["g"], a["h0"], nthreads=1)
        return float((o * dO).sum() + (hT * dST).sum())

    rng = np.random.default_rng(0)
    h = 1e-6
    for n, gname in names.items():
        for _ in range(3):
            dirn = rng.standard_normal(args[n].shape)
            ap = dict(args); ap[n] = args[n] + h * dirn
            am = dict(args); am[n] = args[n] - h * dirn
            fd = (loss(ap) - loss(am)) / (2 * h)
            an = float((got[gname].astype(np.float64) * dirn).sum())
            assert abs(fd - an) <= 1e-4 * max(1.0, abs(fd)), (n, fd, an)


def test_full_size_backward_sampled():
    name = "gdn_fwdbwd_bf16_b8h16t4096d128"
    x = _gen(name)
    o, hT = _run_fwd(x)
    got = _run_bwd(x)
    sel = [(0, 0), (4, 9), (7, 15)]
    frefs = oracle_fwd(x, sel=sel)
    brefs = oracle_bwd(x, sel=sel)
    for (b, h), (ro, rh), rg in zip(sel, frefs, brefs):
        _assert_close("o", o[b:b + 1, h:h + 1], ro, TOL["bf16"])
        _assert_close("hT", hT[b:b + 1, h:h + 1], rh, TOL["bf16"])
        for n in GRADS:
            _assert_close("%s[%d,%d]" % (n, b, h), got[n][b:b + 1, h:h + 1], rg[n], TOL["bf16"])
    for n in GRADS:
        assert np.isfinite(got[n]).all(), n
