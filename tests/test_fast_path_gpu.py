"""GPU parity of the tcgen05 / TMA fused forwards against the fp64 oracle, on small
and ragged cases, plus agreement with the general kernels on the same inputs: the
cooperative kernel's three instances (bf16, d_k = d_v = 128 with chunk 64 or 32,
d_k = d_v = 256 with chunk 32) and the one-CTA-per-item kernel (d 128, chunk 64)."""
import os

import numpy as np
import pytest
import torch

from parity_util import TOL, oracle_fwd, rel, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _wl(**kw):
    from chunkwise_delta_rule_02_gb300 import workloads
    base = dict(name="fast", B=1, H=2, T=128, d=128, dtype="bf16", gated=True, with_h0=True, seed=5)
    base.update(kw)
    return workloads.Workload(**base)


def _run(x, force_general=False, kernel="coop", chunk=64):
    """Forward through the C ABI on the general kernels, the cooperative kernel
    (kernel="coop", the default path) or the one-CTA-per-item fused kernel."""
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    d = to_dev(x, DEV)
    old = {k: os.environ.get(k) for k in ("GDN_FORCE_GENERAL", "GDN_FUSED_PER_ITEM")}
    os.environ["GDN_FORCE_GENERAL"] = "1" if force_general else "0"
    os.environ["GDN_FUSED_PER_ITEM"] = "1" if kernel == "fused" else "0"
    try:
        shape = gdn.make_shape(d["q"], d["v"], chunk, cu_seqlens=d["cu_seqlens"])
        assert gdn.dn_uses_fast_path(shape) == (0 if force_general else 1)
        want = binding.DN_PATH_GENERAL if force_general else (
            binding.DN_PATH_FUSED if kernel == "fused" else binding.DN_PATH_COOP)
        assert binding.dn_plan(shape)[0] == want
        ws = gdn.binding.alloc_workspace(shape, False, DEV)
        o = torch.empty_like(d["v"])
        N = x["cu_seqlens"].numel() - 1 if x["cu_seqlens"] is not None else x["q"].shape[0]
        hT = torch.empty((N, x["q"].shape[1], x["q"].shape[-1], x["v"].shape[-1]), device=DEV)
        if d["g"] is None:
            gdn.dn_chunk_fwd(shape, d["q"], d["k"], d["v"], d["beta"], d["h0"], o, hT, ws)
        else:
            gdn.gdn_chunk_fwd(shape, d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], o, hT, ws)
        assert gdn.dn_device_status(ws) == 0
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v
    return o.float().cpu().numpy(), hT.cpu().numpy()


@pytest.mark.parametrize("kernel", ["coop", "fused"])
@pytest.mark.parametrize("T", [64, 1, 65, 200, 1000])
@pytest.mark.parametrize("gated,h0", [(True, True), (False, False)])
def test_fast_forward_small(T, gated, h0, kernel):
    from chunkwise_delta_rule_02_gb300 import workloads
    x = workloads.generate(_wl(T=T, gated=gated, with_h0=h0, seed=T))
    o, hT = _run(x, kernel=kernel)
    ro, rh = oracle_fwd(x)
    assert np.isfinite(o).all() and np.isfinite(hT).all()
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


@pytest.mark.parametrize("kernel", ["coop", "fused"])
def test_fast_forward_varlen_ragged(kernel):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = _wl(B=1, H=3, T=0, with_h0=True, varlen_total=1, varlen_n=1, seed=9)
    x = workloads.generate(w, lengths=[5, 64, 0, 130, 300, 1, 63])
    o, hT = _run(x, kernel=kernel)
    ro, rh = oracle_fwd(x)
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


def test_fast_matches_general():
    from chunkwise_delta_rule_02_gb300 import workloads
    x = workloads.generate(_wl(B=2, H=4, T=700, seed=77))
    o1, h1 = _run(x)
    o2, h2 = _run(x, force_general=True)
    assert rel(o1, o2) <= 1e-2 and rel(h1, h2) <= 1e-2


def test_fast_strong_decay_and_unit_beta():
    """Gates near the bottom of fp32's exp range inside one chunk and beta = 1."""
    from chunkwise_delta_rule_02_gb300 import workloads
    x = workloads.generate(_wl(T=256, seed=3))
    x["g"] = x["g"] * 40.0            # mean about -2 per token: chunk decays ~exp(-130)
    x["beta"] = torch.ones_like(x["beta"])
    ro, rh = oracle_fwd(x)
    for kernel in ("coop", "fused"):
        o, hT = _run(x, kernel=kernel)
        assert np.isfinite(o).all() and np.isfinite(hT).all()
        assert rel(o, ro) <= TOL["bf16"], (kernel, rel(o, ro))
        assert rel(hT, rh) <= TOL["bf16"], (kernel, rel(hT, rh))


# ----------------------------------------------------------------------------- chunk 32, head dim 256
# The cooperative kernel's other instances: (chunk, d) = (32, 128) and (32, 256); at
# d = 256 two chain CTAs share each (sequence, head), 128 d_v columns each.
INSTANCES = [(32, 128), (32, 256)]


@pytest.mark.parametrize("C,d", INSTANCES)
@pytest.mark.parametrize("T", [1, 31, 32, 33, 200, 1000])
@pytest.mark.parametrize("gated,h0", [(True, True), (False, False)])
def test_coop_instances_small(C, d, T, gated, h0):
    from chunkwise_delta_rule_02_gb300 import workloads
    x = workloads.generate(_wl(T=T, d=d, gated=gated, with_h0=h0, seed=T + d + C, chunk=C))
    o, hT = _run(x, chunk=C)
    ro, rh = oracle_fwd(x)
    assert np.isfinite(o).all() and np.isfinite(hT).all()
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


@pytest.mark.parametrize("C,d", INSTANCES)
def test_coop_instances_varlen_ragged(C, d):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = _wl(B=1, H=3, T=0, d=d, with_h0=True, varlen_total=1, varlen_n=1, seed=19 + d, chunk=C)
    x = workloads.generate(w, lengths=[5, 32, 0, 33, 130, 300, 1, 31])
    o, hT = _run(x, chunk=C)
    ro, rh = oracle_fwd(x)
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


@pytest.mark.parametrize("C,d", INSTANCES)
def test_coop_instances_match_general(C, d):
    """More (sequence, head) items than chain groups (each group walks several items,
    state reloaded from h0 at each), against the general kernels on the same inputs."""
    from chunkwise_delta_rule_02_gb300 import workloads
    x = workloads.generate(_wl(B=8, H=16 if d == 128 else 12, T=100, d=d, seed=78 + d, chunk=C))
    o1, h1 = _run(x, chunk=C)
    o2, h2 = _run(x, force_general=True, chunk=C)
    assert rel(o1, o2) <= 1e-2 and rel(h1, h2) <= 1e-2
    sel = [(0, 0), (7, 11)]
    for (b, h), (ro, rh) in zip(sel, oracle_fwd(x, sel=sel)):
        assert rel(o1[b:b + 1, h:h + 1], ro) <= TOL["bf16"]
        assert rel(h1[b:b + 1, h:h + 1], rh) <= TOL["bf16"]


@pytest.mark.parametrize("C,d", INSTANCES)
def test_coop_instances_strong_decay_and_unit_beta(C, d):
    from chunkwise_delta_rule_02_gb300 import workloads
    x = workloads.generate(_wl(T=256, d=d, seed=4, chunk=C))
    x["g"] = x["g"] * 40.0            # chunk decays ~exp(-65): the renormalised state scale
    x["beta"] = torch.ones_like(x["beta"])
    ro, rh = oracle_fwd(x)
    o, hT = _run(x, chunk=C)
    assert np.isfinite(o).all() and np.isfinite(hT).all()
    assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
    assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


def test_chunk_64_head_dim_256_stays_on_the_general_kernels():
    """One chunk's operand tiles at d 256 and chunk 64 do not fit a CTA's shared memory."""
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding, workloads
    d = to_dev(workloads.generate(_wl(T=64, d=256, seed=1)), DEV)
    assert binding.dn_plan(gdn.make_shape(d["q"], d["v"], 64))[0] == binding.DN_PATH_GENERAL
    assert binding.dn_plan(gdn.make_shape(d["q"], d["v"], 32))[0] == binding.DN_PATH_COOP
