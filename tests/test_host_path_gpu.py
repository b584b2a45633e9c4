"""gdn_chunk_fwd_host: the forward on host (pinned) buffers, against the oracle and
against gdn_chunk_fwd on the same inputs, with and without gate, initial and
final state, on the tcgen05 kernels (bf16, d = 128) and the general kernels
(fp32), as one forward and as time segments whose copies overlap the compute."""
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


def _host_forward(x, want_hT=True):
    """Run gdn_chunk_fwd_host on pinned copies of x; returns (o, hT) as numpy."""
    from chunkwise_delta_rule_02_gb300 import binding
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) and k in ("q", "k", "v", "beta", "g", "h0")
               else v) for k, v in x.items()}
    shape = binding.make_shape(pin["q"], pin["v"])
    B, H, T, d = x["q"].shape
    o = torch.full(tuple(x["v"].shape), float("nan"), dtype=x["v"].dtype).pin_memory()
    hT = torch.full((B, H, d, x["v"].shape[-1]), float("nan")).pin_memory() if want_hT else None
    arena = torch.empty(binding.dn_host_arena_size(shape, pin["g"] is not None, pin["h0"] is not None),
                        dtype=torch.uint8, device=DEV)
    ws = binding.alloc_workspace(shape, False, DEV)
    stream = torch.cuda.current_stream()
    binding.gdn_chunk_fwd_host(shape, pin["q"], pin["k"], pin["v"], pin["beta"], pin["g"], pin["h0"], o,
                               hT, arena, ws, stream)
    stream.synchronize()
    assert binding.dn_device_status(ws) == binding.DN_OK
    return o.float().numpy(), (hT.numpy() if hT is not None else None)


def _device_forward(x):
    import chunkwise_delta_rule_02_gb300 as gdn
    d = to_dev(x, DEV)
    o, hT = gdn.forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"])
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), hT.cpu().numpy()


def _inputs(B, H, T, d, dtype, gated, with_h0, seed):
    from chunkwise_delta_rule_02_gb300 import workloads
    w = workloads.Workload("host", B, H, T, d, dtype, gated, with_h0, seed)
    return workloads.generate(w)


# Fixed-length input of at least 32 chunks runs as time segments whose copies overlap the
# compute (up to 4 segments of >= 16 chunks, the state handed on between them); shorter
# input runs as one forward.
@pytest.mark.parametrize("B,H,T,d,dtype,gated,with_h0", [
    (2, 3, 4133, 128, "bf16", True, True),     # ragged last chunk; 4 segments, the last ragged
    (1, 2, 2048, 128, "bf16", False, False),   # DeltaNet, zero initial state; 2 segments
    (2, 2, 300, 128, "bf16", True, True),      # one forward
    (1, 2, 2100, 64, "f32", True, True),       # general fp32 kernels; 2 segments
    (1, 2, 8229, 128, "bf16", True, True),     # 4 segments of 33 chunks, the last 1893 tokens
    (1, 1, 4100, 64, "f32", True, False),      # fp32, 4 segments, zero initial state
])
def test_host_forward_matches_oracle_and_device_path(B, H, T, d, dtype, gated, with_h0):
    x = _inputs(B, H, T, d, dtype, gated, with_h0, seed=T + d)
    ho, hh = _host_forward(x)
    do, dh = _device_forward(x)
    assert np.isfinite(ho).all() and np.isfinite(hh).all()
    assert rel(ho, do) <= TOL[dtype] and rel(hh, dh) <= TOL[dtype]
    sel = [(0, 0), (B - 1, H - 1)]
    for (b, h), (ro, rh) in zip(sel, oracle_fwd(x, sel=sel)):
        assert rel(ho[b, h], ro[0, 0]) <= TOL[dtype], rel(ho[b, h], ro[0, 0])
        assert rel(hh[b, h], rh[0, 0]) <= TOL[dtype], rel(hh[b, h], rh[0, 0])


def test_host_forward_without_final_state():
    x = _inputs(1, 2, 2048, 128, "bf16", True, True, seed=5)
    ho, _ = _host_forward(x, want_hT=False)
    do, _ = _device_forward(x)
    assert rel(ho, do) <= TOL["bf16"]


def test_host_forward_reuses_its_arena():
    """Two segmented calls in a row on the same arena and stream, the second on other
    inputs: the second call's copies into the arena wait for the first call's work."""
    xa = _inputs(1, 2, 4096, 128, "bf16", True, True, seed=11)
    xb = _inputs(1, 2, 4096, 128, "bf16", True, True, seed=12)
    from chunkwise_delta_rule_02_gb300 import binding
    pins = [{k: (v.pin_memory() if isinstance(v, torch.Tensor) and k in ("q", "k", "v", "beta", "g", "h0")
                 else v) for k, v in x.items()} for x in (xa, xb)]
    shape = binding.make_shape(pins[0]["q"], pins[0]["v"])
    arena = torch.empty(binding.dn_host_arena_size(shape, True, True), dtype=torch.uint8, device=DEV)
    ws = binding.alloc_workspace(shape, False, DEV)
    outs = []
    stream = torch.cuda.current_stream()
    for pin in pins:
        o = torch.full(tuple(pin["v"].shape), float("nan"), dtype=pin["v"].dtype).pin_memory()
        hT = torch.full((1, 2, 128, 128), float("nan")).pin_memory()
        binding.gdn_chunk_fwd_host(shape, pin["q"], pin["k"], pin["v"], pin["beta"], pin["g"], pin["h0"], o,
                                   hT, arena, ws, stream)
        outs.append((o, hT))
    stream.synchronize()
    for x, (o, hT) in zip((xa, xb), outs):
        do, dh = _device_forward(x)
        assert rel(o.float().numpy(), do) <= TOL["bf16"] and rel(hT.numpy(), dh) <= TOL["bf16"]


def test_segments_keep_a_timeout_flagged_by_an_earlier_segment(monkeypatch):
    """The status word is cleared by the first segment only.  With T = 8229 the call runs
    as segments of 33, 33, 33 and 30 chunks; with two heads the cooperative kernel numbers
    its tasks 2 x chunk + head, so the test hook's task 62 (chunk 31 of head 0) is withheld
    in the first three segments and does not exist in the last, which completes cleanly:
    the call still reports the timeout, and the next call is correct."""
    from chunkwise_delta_rule_02_gb300 import binding
    x = _inputs(1, 2, 8229, 128, "bf16", True, True, seed=13)
    pin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) and k in ("q", "k", "v", "beta", "g", "h0")
               else v) for k, v in x.items()}
    shape = binding.make_shape(pin["q"], pin["v"])
    if binding.dn_plan(shape)[0] != binding.DN_PATH_COOP:
        pytest.skip("the cooperative kernel is not available on this device")
    arena = torch.empty(binding.dn_host_arena_size(shape, True, True), dtype=torch.uint8, device=DEV)
    ws = binding.alloc_workspace(shape, False, DEV)
    o = torch.empty(tuple(x["v"].shape), dtype=x["v"].dtype).pin_memory()
    hT = torch.empty((1, 2, 128, 128)).pin_memory()
    stream = torch.cuda.current_stream()
    monkeypatch.setenv("GDN_DEBUG_WITHHOLD_TASK", "62")
    binding.gdn_chunk_fwd_host(shape, pin["q"], pin["k"], pin["v"], pin["beta"], pin["g"], pin["h0"], o, hT,
                               arena, ws, stream)
    stream.synchronize()
    assert binding.dn_device_status(ws) == binding.DN_ERR_TIMEOUT
    monkeypatch.delenv("GDN_DEBUG_WITHHOLD_TASK")
    binding.gdn_chunk_fwd_host(shape, pin["q"], pin["k"], pin["v"], pin["beta"], pin["g"], pin["h0"], o, hT,
                               arena, ws, stream)
    stream.synchronize()
    assert binding.dn_device_status(ws) == binding.DN_OK
    do, dh = _device_forward(x)
    assert rel(o.float().numpy(), do) <= TOL["bf16"] and rel(hT.numpy(), dh) <= TOL["bf16"]


@pytest.mark.parametrize("H,lengths", [(4, [1000, 64, 0, 3000, 5, 1123]), (6, [2048, 2048])])
def test_host_forward_packed_runs_as_head_groups(H, lengths):
    """Packed input of >= 32 chunks runs as groups of heads whose copies overlap the
    compute (H 4: four groups of one head; H 6: three groups of two), the states copied
    per group from and into their [N][H] places; against the device path and the oracle,
    with an empty and a one-token sequence among them."""
    import chunkwise_delta_rule_02_gb300 as gdn
    from chunkwise_delta_rule_02_gb300 import binding, workloads
    w = workloads.Workload("hostv", 1, H, 0, 128, "bf16", True, True, 21, varlen_total=1, varlen_n=1)
    x = workloads.generate(w, lengths=lengths)
    pin = {k: x[k].pin_memory() for k in ("q", "k", "v", "beta", "g", "h0")}
    cu = x["cu_seqlens"].to(DEV)
    shape = binding.make_shape(pin["q"], pin["v"], 64, cu)
    N = len(lengths)
    o = torch.full(tuple(x["v"].shape), float("nan"), dtype=x["v"].dtype).pin_memory()
    hT = torch.full((N, H, 128, 128), float("nan")).pin_memory()
    arena = torch.empty(binding.dn_host_arena_size(shape, True, True), dtype=torch.uint8, device=DEV)
    ws = binding.alloc_workspace(shape, False, DEV)
    stream = torch.cuda.current_stream()
    binding.gdn_chunk_fwd_host(shape, pin["q"], pin["k"], pin["v"], pin["beta"], pin["g"], pin["h0"], o, hT,
                               arena, ws, stream)
    stream.synchronize()
    assert binding.dn_device_status(ws) == binding.DN_OK
    d = to_dev(x, DEV)
    od, hd = gdn.forward(d["q"], d["k"], d["v"], d["beta"], d["g"], d["h0"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    ho, hh = o.float().numpy(), hT.numpy()
    assert np.isfinite(ho).all() and np.isfinite(hh).all()
    assert rel(ho, od.float().cpu().numpy()) <= TOL["bf16"] and rel(hh, hd.cpu().numpy()) <= TOL["bf16"]
    ro, rh = oracle_fwd(x)
    assert rel(ho, ro) <= TOL["bf16"] and rel(hh, rh) <= TOL["bf16"]
