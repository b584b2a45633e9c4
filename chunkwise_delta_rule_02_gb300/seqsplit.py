"""Gated DeltaNet forward split along the sequence over ranks, with one exchange step.

The recurrence S_t = S_{t-1} alpha_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
("Gated DeltaNet: Improving Mamba2 with Delta Rule", rebuttal Table 1, row "Gated
DeltaNet"; stored here transposed, d_k x d_v) is linear in the state.  So the state
leaving a span of tokens is an affine function of the state entering it,

    S_out = A S_in + B,

with A (d_k x d_k) the product of the span's transitions and B (d_k x d_v) the span's
own final state from zero.  Both come out of the ordinary forward: A is the final
state of a call with v = 0 and h0 = I, B the final state of a call with h0 = 0.

Rank r holds the tokens [t_r, t_{r+1}) of every (batch row, head) — its shard, the
boundaries on chunk multiples so that the chunking matches the unsplit call.  Then:

  1. rank 0, whose entering state h0 is known, runs its shard's forward at once and
     sends (A_0, B_0) = (0, its final state); every other rank sends the map (A_r, B_r)
     of its shard;
  2. one all-gather of the maps (the only exchange);
  3. every rank composes the maps in rank order (an exclusive scan, dn_state_affine):
     S_in(r) = A_{r-1} S_in(r-1) + B_{r-1}, and the final state after the last shard;
  4. rank r > 0 runs its shard's forward from S_in(r) for its outputs.

Each rank therefore runs three forward calls on its shard (rank 0 one), and the
compositions are small batched d_k x d_k by d_k x d_v products.  Fixed-length input
[B, H, T, d] only (packed sequences are not split).  The collective is
torch.distributed's all_gather (NCCL between GPUs, gloo on the CPU); the per-shard
work runs in the library's kernels through ``library_ops``.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch


def shard_bounds(T: int, world: int, chunk: int = 64) -> List[Tuple[int, int]]:
    """Contiguous token ranges [t0, t1) of the `world` shards of a sequence of T
    tokens, as even as possible in whole chunks (the last shard takes a ragged tail;
    shards may be empty when there are fewer chunks than ranks)."""
    if T < 0 or world < 1 or chunk < 1:
        raise ValueError("bad shard geometry")
    nch = (T + chunk - 1) // chunk
    base, extra = divmod(nch, world)
    out, c = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        t0, t1 = min(T, c * chunk), min(T, (c + n) * chunk)
        out.append((t0, t1))
        c += n
    return out


class LibraryOps:
    """The per-shard operations on the library's kernels (device tensors)."""

    def __init__(self, chunk: int = 64, scale: float = 1.0, qk_l2norm: bool = True,
                 eps: float = 1e-6, longhorn: bool = False):
        self.kw = dict(chunk=chunk, scale=scale, qk_l2norm=qk_l2norm, eps=eps, longhorn=longhorn)

    def forward(self, q, k, v, beta, g, h0):
        from . import binding
        return binding.forward(q, k, v, beta, g, h0, **self.kw)

    def affine(self, A, S, B):
        from . import binding
        out = torch.empty_like(B if B is not None else S)
        binding.dn_state_affine(A.contiguous(), S.contiguous(),
                                None if B is None else B.contiguous(), out)
        return out


def shard_map(q, k, v, beta, g, ops) -> Tuple[torch.Tensor, torch.Tensor]:
    """(A, B) of one shard for every (batch row, head): S_out = A S_in + B."""
    Bn, H, _, dk = q.shape
    eye = torch.eye(dk, dtype=torch.float32, device=q.device)
    eye = eye.to(torch.float64) if q.dtype == torch.float64 else eye
    eye = eye.expand(Bn, H, dk, dk).contiguous()
    zv = torch.zeros(q.shape[:-1] + (dk,), dtype=v.dtype, device=v.device)
    _, A = ops.forward(q, k, zv, beta, g, eye)
    _, Bm = ops.forward(q, k, v, beta, g, None)
    return A, Bm


def compose(maps: Sequence[Tuple[torch.Tensor, torch.Tensor]], h0: Optional[torch.Tensor], ops,
            upto: Optional[int] = None) -> List[torch.Tensor]:
    """Entering states S_in(0..upto) (upto defaults to len(maps): the last entry is then
    the state after every shard), S_in(0) = h0 (zero if None)."""
    A0, B0 = maps[0]
    S = torch.zeros_like(B0) if h0 is None else h0.to(B0.dtype)
    out = [S]
    n = len(maps) if upto is None else upto
    for r in range(n):
        A, Bm = maps[r]
        S = ops.affine(A, S, Bm)
        out.append(S)
    return out


def torch_all_gather(group=None) -> Callable:
    """The exchange over a torch.distributed process group: every rank's (A, B),
    packed into one tensor, gathered by one all_gather."""
    import torch.distributed as dist

    def gather(A, Bm):
        dk = A.shape[-1]
        packed = torch.cat([A, Bm], dim=-1).contiguous()
        parts = [torch.empty_like(packed) for _ in range(dist.get_world_size(group))]
        dist.all_gather(parts, packed, group=group)
        return [(p[..., :dk].contiguous(), p[..., dk:].contiguous()) for p in parts]

    return gather


def forward_seqsplit(q, k, v, beta, g, h0, rank: int, world: int, gather: Callable,
                     ops=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """This rank's outputs o [B, H, t_{r+1} - t_r, dv] and the final state of the whole
    sequence [B, H, dk, dv] (on every rank).  q, k, v, beta, g are this rank's shard;
    h0 is the sequence's initial state (used by rank 0; others may pass None)."""
    ops = ops or LibraryOps()
    if rank == 0:
        o, hT0 = ops.forward(q, k, v, beta, g, h0)
        A = torch.zeros(q.shape[:2] + (q.shape[-1], q.shape[-1]), dtype=hT0.dtype, device=hT0.device)
        mine = (A, hT0)
    else:
        mine = shard_map(q, k, v, beta, g, ops)
    maps = gather(*mine)
    if len(maps) != world:
        raise RuntimeError("the exchange returned %d maps for %d ranks" % (len(maps), world))
    states = compose(maps, None, ops)
    if rank > 0:
        o, _ = ops.forward(q, k, v, beta, g, states[rank])
    return o, states[world]
