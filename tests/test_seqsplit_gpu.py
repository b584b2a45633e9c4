"""The sequence-split forward on one GPU: the per-shard forwards and the composition
(dn_state_affine) run in the library's kernels; the exchange, which several GPUs
would do with one all_gather, is a list in one process (the shards run one after
another, none waits on another).  Checked against the fp64 oracle on the whole
sequence at the kernels' tolerance, and dn_state_affine against a plain PyTorch
product."""
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


@pytest.mark.parametrize("count,dk,dv", [(5, 128, 128), (3, 128, 96), (2, 200, 256), (7, 16, 24)])
def test_state_affine_matches_torch(count, dk, dv):
    from chunkwise_delta_rule_02_gb300 import binding
    gen = torch.Generator().manual_seed(count + dk)
    A = torch.randn(count, dk, dk, generator=gen) / dk ** 0.5
    S = torch.randn(count, dk, dv, generator=gen)
    B = torch.randn(count, dk, dv, generator=gen)
    want = (A.double() @ S.double() + B.double()).numpy()
    Ad, Sd, Bd = A.to(DEV), S.to(DEV), B.to(DEV)
    out = torch.empty_like(Sd)
    binding.dn_state_affine(Ad, Sd, Bd, out)
    assert rel(out.cpu().numpy(), want) <= 1e-6
    binding.dn_state_affine(Ad, Sd, None, out)
    assert rel(out.cpu().numpy(), (A.double() @ S.double()).numpy()) <= 1e-6
    binding.dn_state_affine(Ad, Sd, Bd, Bd)          # out may be B
    torch.cuda.synchronize()
    assert rel(Bd.cpu().numpy(), want) <= 1e-6


@pytest.mark.parametrize("dtype,d,world,T", [("bf16", 128, 3, 700), ("bf16", 128, 2, 64),
                                              ("f32", 64, 4, 300)])
def test_split_forward_on_one_gpu(dtype, d, world, T):
    from chunkwise_delta_rule_02_gb300 import seqsplit, workloads
    w = workloads.Workload("split", 2, 2, T, d, dtype, True, True, 51)
    x = workloads.generate(w)
    dd = to_dev(x, DEV)
    ops = seqsplit.LibraryOps()
    bounds = seqsplit.shard_bounds(T, world, 64)
    sh = lambda r: [dd[n][:, :, bounds[r][0]:bounds[r][1]].contiguous() for n in ("q", "k", "v", "beta", "g")]
    maps = []
    for r in range(world):
        if r == 0:
            _, hT0 = ops.forward(*sh(0), dd["h0"])
            maps.append((torch.zeros(2, 2, d, d, device=DEV), hT0))
        else:
            maps.append(seqsplit.shard_map(*sh(r), ops))
    outs = []
    for r in range(world):
        o, hT = seqsplit.forward_seqsplit(*sh(r), dd["h0"] if r == 0 else None, r, world,
                                          lambda A, Bm: maps, ops)
        outs.append(o)
    torch.cuda.synchronize()
    ro, rh = oracle_fwd(x)
    assert rel(torch.cat(outs, 2).float().cpu().numpy(), ro) <= TOL[dtype]
    assert rel(hT.cpu().numpy(), rh) <= TOL[dtype]
