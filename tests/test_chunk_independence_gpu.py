"""Chunk independence of the general kernels, bit for bit.

The chunk form computes chunk j from its own inputs and the state entering it
(the state passing of the Gated DeltaNet page's reply on length extrapolation).
So, on kernels that keep the state in fp32 and do every product in a fixed order:

  * the first chunk of a call over two chunks equals a call over that chunk alone,
    and the second chunk equals a call over it alone started from the first call's
    final state — to the last bit;
  * backward: the last chunk's gradients equal those of a call over it alone from the
    same entering state, and the first chunk's equal those of a call over it alone
    given the second call's dh0 as its dhT.

A hazard that lets one chunk's data reach another chunk's arithmetic (a missing
barrier, an aliased staging buffer, a staging index past its tile, operands of the
next chunk overwriting this chunk's in shared memory) breaks these equalities at
once, at a size where relative-error parity could still pass.  The staged bf16
scans, the staged per-chunk kernels and the fp32 kernels are covered (the general
path; the cooperative forward keeps a pending decay factor across chunks, so its
rounding depends on where a call starts)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(dtype, d, C, seed):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("ind", 2, 2, 2 * C, d, dtype, True, True, seed, chunk=C, backward=True)
    x = workloads.generate(w)
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _half(x, a, b):
    return {n: x[n][:, :, a:b].contiguous() for n in ("q", "k", "v", "beta", "g", "do")}


def _same(a, b, what, order_free=False):
    """Bit for bit; order_free: the tensor comes out of sums whose order is not fixed
    (shared-memory atomic adds of the gate gradient's row sums), so it may differ in
    its last bits between any two calls: equal to 1e-6 of its largest entry."""
    a = a.float().cpu().numpy()
    b = b.float().cpu().numpy()
    if order_free:
        assert np.abs(a - b).max() <= 1e-6 * np.abs(b).max(), "%s differs: max |diff| %.3e" % (
            what, np.abs(a - b).max())
    else:
        assert np.array_equal(a, b), "%s differs: max |diff| %.3e" % (what, np.abs(a - b).max())


@pytest.mark.parametrize("dtype,d,C", [("bf16", 128, 64), ("bf16", 64, 32), ("f32", 64, 64)])
def test_chunks_do_not_reach_each_other(dtype, d, C, monkeypatch):
    import chunkwise_delta_rule_02_gb300 as gdn
    monkeypatch.setenv("GDN_FORCE_GENERAL", "1")   # the general kernels (forward and the backward's recompute)
    x = _inputs(dtype, d, C, seed=71 + d + C)
    f, s = _half(x, 0, C), _half(x, C, 2 * C)
    kw = dict(chunk=C)
    # forward
    o, hT = gdn.forward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], **kw)
    o1, h1 = gdn.forward(f["q"], f["k"], f["v"], f["beta"], f["g"], x["h0"], **kw)
    o2, h2 = gdn.forward(s["q"], s["k"], s["v"], s["beta"], s["g"], h1, **kw)
    _same(o[:, :, :C], o1, "o, first chunk")
    _same(o[:, :, C:], o2, "o, second chunk")
    _same(hT, h2, "final state")
    # backward
    g = gdn.backward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["h0"], x["do"], x["dhT"], **kw)
    g2 = gdn.backward(s["q"], s["k"], s["v"], s["beta"], s["g"], h1, s["do"], x["dhT"], **kw)
    g1 = gdn.backward(f["q"], f["k"], f["v"], f["beta"], f["g"], x["h0"], f["do"], g2["dh0"], **kw)
    for n in ("dq", "dk", "dv", "dbeta", "dg"):
        _same(g[n][:, :, C:], g2[n], n + ", last chunk", order_free=(n == "dg"))
        _same(g[n][:, :, :C], g1[n], n + ", first chunk", order_free=(n == "dg"))
    _same(g["dh0"], g1["dh0"], "dh0")
