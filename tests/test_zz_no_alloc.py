"""The allocation-free forward, gdn_chunk_fwd_noalloc, against gdn_chunk_fwd.

gdn_chunk_fwd_noalloc serves callers that cannot allocate device memory or pass
a workspace (operator interfaces without a scratch argument, frameworks that own
all device memory).  Its scratch lives in a static device array inside the
library.  This file is named to be collected last, so that a run stopping at the
first failure has run every other test first; it also passes on its own in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity_util import TOL, rel, to_dev

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(lengths=None, T=300, seed=31):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("na", 2 if lengths is None else 1, 3, T, 128, "bf16", True, True, seed,
                           varlen_total=1 if lengths else 0, varlen_n=1 if lengths else 0)
    return to_dev(workloads.generate(w, lengths=lengths), DEV)


def _reference(d):
    import chunkwise_delta_rule_02_gb300 as gdn
    o, hT = gdn.forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), hT.cpu().numpy()


def _noalloc(d):
    """Two calls in a row through the C ABI, each into fresh output buffers."""
    from chunkwise_delta_rule_02_gb300 import binding
    lib = binding.lib()
    shape = binding.make_shape(d["q"], d["v"], cu_seqlens=d["cu_seqlens"])
    N = shape.num_seqs if d["cu_seqlens"] is not None else d["q"].shape[0]
    outs = []
    for _ in range(2):
        o = torch.full_like(d["v"], float("nan"))
        hT = torch.full((N, d["q"].shape[1], 128, 128), float("nan"), device=DEV)
        rc = lib.gdn_chunk_fwd_noalloc(ctypes.byref(shape), d["q"].data_ptr(), d["k"].data_ptr(),
                                       d["v"].data_ptr(), d["beta"].data_ptr(), d["g"].data_ptr(),
                                       d["h0"].data_ptr(), o.data_ptr(), hT.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
        assert rc == binding.DN_OK, binding.status_str(rc)
        torch.cuda.synchronize()
        outs.append((o.float().cpu().numpy(), hT.cpu().numpy()))
    return outs


@pytest.mark.parametrize("lengths", [None, [5, 64, 0, 130, 300, 1, 63]])
def test_noalloc_matches_workspace_entry_point(lengths):
    d = _inputs(lengths)
    ro, rh = _reference(d)
    for o, hT in _noalloc(d):
        assert np.isfinite(o).all() and np.isfinite(hT).all()
        assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
        assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


def _noalloc_call(lib, shape, d, o, hT, g=None):
    return lib.gdn_chunk_fwd_noalloc(ctypes.byref(shape), d["q"].data_ptr(), d["k"].data_ptr(),
                                     d["v"].data_ptr(), d["beta"].data_ptr(),
                                     None if g is None else g.data_ptr(), None, o.data_ptr(),
                                     hT.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_status_word_is_readable():
    """What the device finds during an allocation-free call (here malformed packed
    offsets, then a log-gate above zero) reaches the caller through
    dn_noalloc_status, which needs no workspace pointer; reading clears it."""
    from chunkwise_delta_rule_02_gb300 import binding
    lib = binding.lib()
    d = _inputs([10, 5, 5], seed=32)
    o = torch.zeros_like(d["v"])
    hT = torch.zeros((3, d["q"].shape[1], 128, 128), device=DEV)
    bad = torch.tensor([0, 10, 5, 20], dtype=torch.int32, device=DEV)   # not monotone
    shape = binding.make_shape(d["q"], d["v"], cu_seqlens=bad)
    assert _noalloc_call(lib, shape, d, o, hT, d["g"]) == binding.DN_OK
    assert binding.dn_noalloc_status() == binding.DN_ERR_INVALID_ARG
    assert binding.dn_noalloc_status() == binding.DN_OK
    shape = binding.make_shape(d["q"], d["v"], cu_seqlens=d["cu_seqlens"])
    assert _noalloc_call(lib, shape, d, o, hT, d["g"].abs()) == binding.DN_OK
    assert binding.dn_noalloc_status() == binding.DN_ERR_DOMAIN
    assert _noalloc_call(lib, shape, d, o, hT, d["g"]) == binding.DN_OK
    assert binding.dn_noalloc_status() == binding.DN_OK


def test_noalloc_ignores_the_general_path_override(monkeypatch):
    """GDN_FORCE_GENERAL sends the workspace entry points to the general kernels;
    the allocation-free one has no workspace for them and keeps the fused kernel."""
    monkeypatch.setenv("GDN_FORCE_GENERAL", "1")
    d = _inputs(None, seed=33)
    ro, rh = _reference(d)
    for o, hT in _noalloc(d):
        assert rel(o, ro) <= TOL["bf16"], rel(o, ro)
        assert rel(hT, rh) <= TOL["bf16"], rel(hT, rh)


def test_noalloc_rejects_what_it_cannot_serve():
    from chunkwise_delta_rule_02_gb300 import binding
    lib = binding.lib()
    d = _inputs()
    # shapes outside the fused kernel (fp32 / other head dims) would need a workspace
    q32 = d["q"].float()
    shape = binding.make_shape(q32, d["v"].float())
    rc = lib.gdn_chunk_fwd_noalloc(ctypes.byref(shape), q32.data_ptr(), q32.data_ptr(), q32.data_ptr(),
                                   q32.data_ptr(), None, None, q32.data_ptr(), None, None)
    assert rc == binding.DN_ERR_UNSUPPORTED
    # more packed sequences than the static scratch holds
    cu = torch.zeros(100001, dtype=torch.int32, device=DEV)
    shape = binding.make_shape(d["q"][:1], d["v"][:1], cu_seqlens=cu)
    rc = lib.gdn_chunk_fwd_noalloc(ctypes.byref(shape), d["q"].data_ptr(), d["k"].data_ptr(),
                                   d["v"].data_ptr(), d["beta"].data_ptr(), None, None,
                                   d["v"].data_ptr(), None, None)
    assert rc == binding.DN_ERR_WORKSPACE
