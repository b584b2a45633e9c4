"""Device-side status reports through the C ABI.

A log-gate g > 0 (alpha > 1) lies outside the domain the header documents
(g <= 0: the gate is a decay, "Gated DeltaNet" rebuttal Table 1, row "Gated
DeltaNet", alpha_t in (0, 1)).  Every forward kernel family flags it in the
status word (DN_ERR_DOMAIN) and still computes the recurrence while the growth
stays in float32 range; the backward's recompute flags it too.  The Python
helpers read the word and raise.
"""
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


def _inputs(dtype, d, T, seed, positive=True, backward=False):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("pos", 2, 2, T, d, dtype, True, True, seed, backward=backward)
    x = workloads.generate(w)
    if positive:
        # the mirror image of the workload's gate distribution: +softplus(N(0,1))/16
        x["g"] = x["g"].abs()
    return x


# path -> (environment, dtype, head dim)
PATHS = {
    "coop": ({}, "bf16", 128),
    "fused": ({"GDN_FUSED_PER_ITEM": "1"}, "bf16", 128),
    "general_bf16": ({"GDN_FORCE_GENERAL": "1"}, "bf16", 128),
    "general_f32": ({}, "f32", 64),
}


@pytest.mark.parametrize("path", list(PATHS))
def test_positive_gate_is_flagged_and_computed(path, monkeypatch):
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    env, dtype, d = PATHS[path]
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    x = _inputs(dtype, d, T=130, seed=41)
    dd = to_dev(x, DEV)
    shape = binding.make_shape(dd["q"], dd["v"])
    ws = binding.alloc_workspace(shape, False, DEV)
    o = torch.empty_like(dd["v"])
    hT = torch.empty((2, 2, d, d), device=DEV)
    binding.gdn_chunk_fwd(shape, dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"], o, hT, ws)
    assert binding.dn_device_status(ws) == binding.DN_ERR_DOMAIN
    assert binding.dn_device_status(ws) == binding.DN_OK          # reading clears it
    ro, rh = oracle_fwd(x)
    assert rel(o.float().cpu().numpy(), ro) <= TOL[dtype]
    assert rel(hT.cpu().numpy(), rh) <= TOL[dtype]
    # the same inputs with the gate in its domain are not flagged
    dd["g"] = -dd["g"]
    binding.gdn_chunk_fwd(shape, dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"], o, hT, ws)
    assert binding.dn_device_status(ws) == binding.DN_OK
    # the helper reads the word and raises
    dd["g"] = -dd["g"]
    with pytest.raises(gdn.GdnError) as err:
        gdn.forward(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"])
    assert err.value.status == binding.DN_ERR_DOMAIN


def test_positive_gate_is_flagged_by_the_backward():
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    x = _inputs("bf16", 64, T=70, seed=42, backward=True)
    dd = to_dev(x, DEV)
    with pytest.raises(gdn.GdnError) as err:
        gdn.backward(dd["q"], dd["k"], dd["v"], dd["beta"], dd["g"], dd["h0"], dd["do"], dd["dhT"])
    assert err.value.status == binding.DN_ERR_DOMAIN
    # the same inputs with the gate in its domain pass the check
    out = gdn.backward(dd["q"], dd["k"], dd["v"], dd["beta"], -dd["g"], dd["h0"], dd["do"], dd["dhT"])
    assert np.isfinite(out["dq"].float().cpu().numpy()).all()
