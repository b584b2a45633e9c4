"""GPU parity of the recurrent decode step (gdn_decode_step, through the C ABI)
against the fp64 oracle: one step from a given state, a run of steps chained
through the state (in place and into a second buffer), and agreement with the
chunked forward when a prefix is prefilled and the next token decoded."""
import ctypes

import numpy as np
import pytest
import torch

from parity_util import TOL, f64, rel

import oracle

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _seq(N, H, T, dk, dv, dtype, gated, seed):
    """Inputs of T tokens, [N,H,T,d]; the initial state ~ N(0, 0.02^2)."""
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(N, H, T, dk, generator=gen)
    k = torch.randn(N, H, T, dk, generator=gen)
    v = torch.randn(N, H, T, dv, generator=gen)
    beta = torch.sigmoid(torch.randn(N, H, T, generator=gen))
    g = -torch.nn.functional.softplus(torch.randn(N, H, T, generator=gen)) / 16 if gated else None
    S0 = 0.02 * torch.randn(N, H, dk, dv, generator=gen)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v, beta = (t.to(tdt) for t in (q, k, v, beta))
    return q, k, v, beta, g, S0


def _oracle(q, k, v, beta, g, S0, scale=1.0):
    return oracle.fwd(f64(q), f64(k), f64(v), f64(beta), f64(g), f64(S0), scale=scale)


@pytest.mark.parametrize("N,H,dk,dv,dtype,gated,zero_state", [
    (4, 3, 128, 128, "bf16", True, False),
    (2, 2, 64, 64, "f32", False, False),
    (3, 2, 64, 96, "f32", True, False),      # d_v not a multiple of the 32-column slice
    (2, 4, 128, 128, "bf16", True, True),    # no initial state
    (1, 1, 16, 20, "f32", True, False),
    (2, 2, 32, 30, "f32", True, False),      # d_v % 4 != 0: the 4-byte-access kernel
    (2, 2, 256, 256, "bf16", True, False),   # head dim 256: the 4-byte-access kernel
])
def test_one_step_matches_oracle(N, H, dk, dv, dtype, gated, zero_state):
    import chunkwise_delta_rule_02_gb300 as gdn
    q, k, v, beta, g, S0 = _seq(N, H, 1, dk, dv, dtype, gated, seed=dk + dv + N)
    if zero_state:
        S0 = torch.zeros_like(S0)
    ro, rh = _oracle(q, k, v, beta, g, S0, scale=0.8)
    dq, dk_, dvv, db = (t[:, :, 0].contiguous().to(DEV) for t in (q, k, v, beta))
    dg = g[:, :, 0].contiguous().to(DEV) if gated else None
    st = None if zero_state else S0.to(DEV)
    o, S1 = gdn.decode_step(dq, dk_, dvv, db, dg, st, scale=0.8)
    torch.cuda.synchronize()
    assert rel(o.float().cpu().numpy(), ro[:, :, 0]) <= TOL[dtype]
    assert rel(S1.cpu().numpy(), rh) <= TOL[dtype]


@pytest.mark.parametrize("dtype,in_place", [("bf16", True), ("bf16", False), ("f32", True)])
def test_chained_steps_match_oracle(dtype, in_place):
    import chunkwise_delta_rule_02_gb300 as gdn
    N, H, T, d = 2, 3, 24, 128 if dtype == "bf16" else 64
    q, k, v, beta, g, S0 = _seq(N, H, T, d, d, dtype, True, seed=7)
    ro, rh = _oracle(q, k, v, beta, g, S0)
    state = S0.to(DEV)
    other = torch.empty_like(state)
    outs = []
    for t in range(T):
        args = [x[:, :, t].contiguous().to(DEV) for x in (q, k, v, beta, g)]
        dst = state if in_place else other
        o, new = gdn.decode_step(*args, state=state, out_state=dst)
        outs.append(o.float())
        if not in_place:
            state, other = new, state
    torch.cuda.synchronize()
    o = torch.stack(outs, 2).cpu().numpy()
    assert rel(o, ro) <= TOL[dtype], rel(o, ro)
    assert rel(state.cpu().numpy(), rh) <= TOL[dtype]


def test_prefill_then_decode_equals_longer_forward():
    """Chunked forward over T tokens, then one decode step from its final state, gives
    the output and state of the chunked forward over T + 1 tokens."""
    import chunkwise_delta_rule_02_gb300 as gdn
    N, H, T, d = 2, 4, 200, 128
    q, k, v, beta, g, S0 = _seq(N, H, T + 1, d, d, "bf16", True, seed=9)
    dev = [x.to(DEV) for x in (q, k, v, beta, g, S0)]
    qd, kd, vd, bd, gd, hd = dev
    o_all, h_all = gdn.forward(qd, kd, vd, bd, gd, hd)
    o_pre, h_pre = gdn.forward(qd[:, :, :T].contiguous(), kd[:, :, :T].contiguous(), vd[:, :, :T].contiguous(),
                               bd[:, :, :T].contiguous(), gd[:, :, :T].contiguous(), hd)
    o1, h1 = gdn.decode_step(qd[:, :, T].contiguous(), kd[:, :, T].contiguous(), vd[:, :, T].contiguous(),
                             bd[:, :, T].contiguous(), gd[:, :, T].contiguous(), state=h_pre)
    torch.cuda.synchronize()
    assert rel(o1.float().cpu().numpy(), o_all[:, :, T].float().cpu().numpy()) <= TOL["bf16"]
    assert rel(h1.cpu().numpy(), h_all.cpu().numpy()) <= TOL["bf16"]


def test_decode_rejects_what_it_cannot_serve():
    from chunkwise_delta_rule_02_gb300 import binding
    lib = binding.lib()
    x = torch.zeros(2, 2, 1, 64, device=DEV)
    st = torch.zeros(2, 2, 64, 64, device=DEV)
    bad_T = binding.make_shape(torch.zeros(2, 2, 3, 64, device=DEV), torch.zeros(2, 2, 3, 64, device=DEV))
    rc = lib.gdn_decode_step(ctypes.byref(bad_T), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                             None, st.data_ptr(), st.data_ptr(), x.data_ptr(), None)
    assert rc == binding.DN_ERR_INVALID_ARG
    ok = binding.make_shape(x, x)
    rc = lib.gdn_decode_step(ctypes.byref(ok), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                             None, None, None, x.data_ptr(), None)
    assert rc == binding.DN_ERR_INVALID_ARG   # no output state
