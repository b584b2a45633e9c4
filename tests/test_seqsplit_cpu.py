"""The forward split along the sequence (chunkwise_delta_rule_02_gb300.seqsplit) on
the CPU: its host logic — shard bounds, the affine maps of the shards, their
composition and the one all-gather — with the fp64 oracle standing in for the
per-shard forward.  The split result must equal the oracle run on the whole
sequence (state passing: the Gated DeltaNet page's reply on length extrapolation;
linearity of the recurrence in the state, rebuttal Table 1).

The two-rank case runs as two processes over gloo; more shards run in one process
with the exchange replaced by a list."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))


class OracleOps:
    """The split's per-shard operations done by the oracle (fp64, CPU tensors)."""

    def forward(self, q, k, v, beta, g, h0):
        import oracle
        f = lambda t: None if t is None else t.double().numpy()
        o, hT = oracle.fwd(f(q), f(k), f(v), f(beta), f(g), f(h0))
        return torch.from_numpy(o), torch.from_numpy(hT)

    def affine(self, A, S, B):
        return A @ S + B


def _problem(B=1, H=2, T=200, d=16, seed=3, dv=None):
    gen = torch.Generator().manual_seed(seed)
    dv = dv or d
    q = torch.randn(B, H, T, d, generator=gen, dtype=torch.float64)
    k = torch.randn(B, H, T, d, generator=gen, dtype=torch.float64)
    v = torch.randn(B, H, T, dv, generator=gen, dtype=torch.float64)
    beta = torch.sigmoid(torch.randn(B, H, T, generator=gen, dtype=torch.float64))
    g = -torch.nn.functional.softplus(torch.randn(B, H, T, generator=gen, dtype=torch.float64)) / 16
    h0 = 0.02 * torch.randn(B, H, d, dv, generator=gen, dtype=torch.float64)
    return q, k, v, beta, g, h0


def _shard(t, a, b):
    return t[:, :, a:b].contiguous()


def _split_in_process(world, T=200, chunk=16, dv=None):
    """Every shard's step 1 first, then the exchange as a list, then step 3/4."""
    from chunkwise_delta_rule_02_gb300 import seqsplit
    q, k, v, beta, g, h0 = _problem(T=T, dv=dv)
    bounds = seqsplit.shard_bounds(T, world, chunk)
    ops = OracleOps()
    maps = []
    for r, (a, b) in enumerate(bounds):
        sh = [_shard(t, a, b) for t in (q, k, v, beta, g)]
        if r == 0:
            _, hT0 = ops.forward(*sh, h0)
            maps.append((torch.zeros(1, 2, q.shape[-1], q.shape[-1], dtype=torch.float64), hT0))
        else:
            maps.append(seqsplit.shard_map(*sh, ops))
    outs = []
    for r, (a, b) in enumerate(bounds):
        sh = [_shard(t, a, b) for t in (q, k, v, beta, g)]
        o, hT = seqsplit.forward_seqsplit(*sh, h0 if r == 0 else None, r, world,
                                          lambda A, Bm: maps, ops)
        outs.append(o)
    ro, rh = ops.forward(q, k, v, beta, g, h0)
    return torch.cat(outs, 2), hT, ro, rh


def test_shard_bounds_are_contiguous_and_chunk_aligned():
    from chunkwise_delta_rule_02_gb300 import seqsplit
    for T, world, C in ((200, 2, 64), (8192, 8, 64), (65, 4, 64), (0, 3, 64), (1000, 3, 16)):
        b = seqsplit.shard_bounds(T, world, C)
        assert len(b) == world and b[0][0] == 0 and b[-1][1] == T
        for (a0, a1), (c0, c1) in zip(b, b[1:]):
            assert a1 == c0
        for a0, a1 in b[:-1]:
            assert a0 % C == 0 and a1 % C == 0 or a1 == T
        sizes = [a1 - a0 for a0, a1 in b]
        assert max(sizes) - min(sizes) <= C


@pytest.mark.parametrize("world", [1, 2, 3, 5, 16])
def test_split_equals_the_whole_sequence(world):
    """Any number of shards (16 shards of a 200-token sequence in chunks of 16 leaves
    some shards empty) gives the oracle's outputs and final state on the whole."""
    o, hT, ro, rh = _split_in_process(world)
    assert np.abs(o.numpy() - ro.numpy()).max() <= 1e-10 * max(1.0, np.abs(ro.numpy()).max())
    assert np.abs(hT.numpy() - rh.numpy()).max() <= 1e-10 * max(1.0, np.abs(rh.numpy()).max())


def test_split_with_dk_different_from_dv():
    o, hT, ro, rh = _split_in_process(3, T=150, dv=24)
    assert np.allclose(o.numpy(), ro.numpy(), rtol=0, atol=1e-10)
    assert np.allclose(hT.numpy(), rh.numpy(), rtol=0, atol=1e-10)


def test_shard_map_is_the_affine_map_of_the_shard():
    """S_out = A S_in + B for an arbitrary entering state, with A, B from two calls."""
    from chunkwise_delta_rule_02_gb300 import seqsplit
    q, k, v, beta, g, _ = _problem(T=90)
    ops = OracleOps()
    A, Bm = seqsplit.shard_map(q, k, v, beta, g, ops)
    S = torch.randn(1, 2, 16, 16, dtype=torch.float64, generator=torch.Generator().manual_seed(9))
    _, want = ops.forward(q, k, v, beta, g, S)
    assert np.allclose((A @ S + Bm).numpy(), want.numpy(), rtol=0, atol=1e-12)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q_out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path[:0] = [ROOT, HERE]
    import torch.distributed as dist
    from chunkwise_delta_rule_02_gb300 import seqsplit
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v, beta, g, h0 = _problem(T=200)
    a, b = seqsplit.shard_bounds(200, world, 64)[rank]
    sh = [_shard(t, a, b) for t in (q, k, v, beta, g)]
    o, hT = seqsplit.forward_seqsplit(*sh, h0 if rank == 0 else None, rank, world,
                                      seqsplit.torch_all_gather(), OracleOps())
    q_out.put((rank, o.numpy(), hT.numpy()))
    dist.destroy_process_group()


def test_two_ranks_over_gloo():
    """Two processes, one shard each, one all_gather: rank outputs concatenated and the
    final state (on both ranks) equal the oracle on the whole sequence."""
    ctx = mp.get_context("spawn")
    qo = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, qo)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((qo.get(timeout=180) for _ in procs), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ro, rh = OracleOps().forward(*_problem(T=200))
    o = np.concatenate([res[0][1], res[1][1]], axis=2)
    assert np.allclose(o, ro.numpy(), rtol=0, atol=1e-10)
    for _, _, hT in res:
        assert np.allclose(hT, rh.numpy(), rtol=0, atol=1e-10)
