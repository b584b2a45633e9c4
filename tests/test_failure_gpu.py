"""Failure detection in the cooperative forward, exercised without any GPU fault.

Every wait across CTAs in k_coop_fwd is bounded.  The test hook
GDN_DEBUG_WITHHOLD_TASK=n makes the preparation CTAs skip task n, so the chain
CTA that owns it waits for a package nobody publishes; with the hook set such
waits give up after about a millisecond.  The chain CTA then records the timeout
in the workspace's status word and raises the launch-wide abort word, every CTA
drains its copies and tensor-core work and leaves, and dn_device_status returns
DN_ERR_TIMEOUT.  The context stays usable: the next call without the hook is
correct.
"""
import time

import pytest
import torch

from parity_util import TOL, oracle_fwd, rel, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _case(T=24 * 64, seed=61):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("fail", 1, 2, T, 128, "bf16", True, True, seed)
    return workloads.generate(w)


def _call(d, shape, ws):
    from chunkwise_delta_rule_02_gb300 import binding
    o = torch.zeros_like(d["v"])
    hT = torch.zeros((1, 2, 128, 128), device=DEV)
    binding.gdn_chunk_fwd(shape, d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], o, hT, ws)
    return o, hT


# tasks are numbered chunk-major over the chain CTAs (two chain CTAs here, one per head):
# 5 is chunk 2 of chain CTA 1, whose later packages then also wait for a ring slot that
# is never consumed; 46 is the last chunk (23) of chain CTA 0
@pytest.mark.parametrize("task", [5, 46])
def test_withheld_package_times_out_and_the_context_stays_usable(task, monkeypatch):
    from chunkwise_delta_rule_02_gb300 import binding
    x = _case()
    d = to_dev(x, DEV)
    shape = binding.make_shape(d["q"], d["v"])
    if binding.dn_plan(shape)[0] != binding.DN_PATH_COOP:
        pytest.skip("the cooperative kernel is not available on this device")
    ws = binding.alloc_workspace(shape, False, DEV)
    monkeypatch.setenv("GDN_DEBUG_WITHHOLD_TASK", str(task))
    t0 = time.perf_counter()
    _call(d, shape, ws)
    assert binding.dn_device_status(ws) == binding.DN_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 10.0      # the launch wound down, nothing waited out 2 s budgets
    assert binding.dn_device_status(ws) == binding.DN_OK
    monkeypatch.delenv("GDN_DEBUG_WITHHOLD_TASK")
    o, hT = _call(d, shape, ws)
    assert binding.dn_device_status(ws) == binding.DN_OK
    ro, rh = oracle_fwd(x)
    assert rel(o.float().cpu().numpy(), ro) <= TOL["bf16"]
    assert rel(hT.cpu().numpy(), rh) <= TOL["bf16"]


def test_helper_raises_on_a_timeout(monkeypatch):
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding
    d = to_dev(_case(T=8 * 64, seed=62), DEV)
    if binding.dn_plan(binding.make_shape(d["q"], d["v"]))[0] != binding.DN_PATH_COOP:
        pytest.skip("the cooperative kernel is not available on this device")
    monkeypatch.setenv("GDN_DEBUG_WITHHOLD_TASK", "0")
    with pytest.raises(gdn.GdnError) as err:
        gdn.forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    assert err.value.status == binding.DN_ERR_TIMEOUT
