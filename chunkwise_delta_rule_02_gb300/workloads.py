"""Seeded synthetic inputs for the (gated) delta-rule workloads.

This module holds the shapes, seeds and value distributions of the
workloads and nothing of the method's arithmetic: it draws q, k, v, beta, the
log-gate g, the initial state, packed sequence lengths and upstream gradients.
Both the CUDA path's tests/benchmark and the fp64 oracle take their inputs from
here, so the two sides see the same values.

Distributions (the 1.3B-scale layer shape of the DeltaNet page, d_head 128 and
16 heads, as the synthetic stand-in for the pages' training data):
  q, k, v ~ N(0, 1) (q and k are normalised inside the kernels, not here);
  beta = sigmoid(N(0, 1));
  g = -softplus(N(0, 1)) / 16 (fp32 log-gate, alpha = exp(g) in (0, 1));
  initial state ~ N(0, 0.02^2) fp32 where a workload has one;
  upstream gradients do ~ N(0, 1), dhT ~ N(0, 0.01^2).
All draws come from one CPU ``torch.Generator`` per workload, in a fixed order,
in float32; 16-bit workloads then round q, k, v, beta (and do) to bfloat16.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dtype: str            # "f32" or "bf16"
    gated: bool
    with_h0: bool
    seed: int
    chunk: int = 64
    varlen_total: int = 0  # >0: packed sequences summing to this many tokens (B == 1)
    varlen_n: int = 0
    backward: bool = False

    @property
    def tokens(self) -> int:
        return self.varlen_total if self.varlen_total else self.B * self.T


WORKLOADS: Dict[str, Workload] = {
    # DeltaNet forward, fp32, B1 H2 T256 d64, seed 0
    "dn_fwd_f32_b1h2t256d64": Workload("dn_fwd_f32_b1h2t256d64", 1, 2, 256, 64, "f32",
                                       False, False, 0),
    # DeltaNet forward, bf16, B8 H16 T2048 d128
    "dn_fwd_bf16_b8h16t2048d128": Workload("dn_fwd_bf16_b8h16t2048d128", 8, 16, 2048, 128,
                                           "bf16", False, False, 1),
    # Gated DeltaNet forward, bf16, B4 H16 T8192 d128, with initial state
    "gdn_fwd_bf16_b4h16t8192d128_h0": Workload("gdn_fwd_bf16_b4h16t8192d128_h0", 4, 16, 8192,
                                               128, "bf16", True, True, 2),
    # Gated DeltaNet forward, bf16, packed: H32, 8 sequences, 65536 tokens
    "gdn_fwd_bf16_varlen_h32_n8_t65536": Workload("gdn_fwd_bf16_varlen_h32_n8_t65536", 1, 32,
                                                  65536, 128, "bf16", True, False, 3,
                                                  varlen_total=65536, varlen_n=8),
    # Gated DeltaNet forward + backward, bf16, B8 H16 T4096 d128
    "gdn_fwdbwd_bf16_b8h16t4096d128": Workload("gdn_fwdbwd_bf16_b8h16t4096d128", 8, 16, 4096,
                                               128, "bf16", True, True, 4, backward=True),
    # chunk 32 (the DeltaNet page's best chunk on A100) on the B4 H16 T8192 d128 forward
    "gdn_fwd_bf16_b4h16t8192d128_c32_h0": Workload("gdn_fwd_bf16_b4h16t8192d128_c32_h0", 4, 16,
                                                   8192, 128, "bf16", True, True, 5, chunk=32),
    # head dim 256 (the Gated DeltaNet page's head size) at the same width, 8 heads x 256 =
    # 16 x 128, chunk 32
    "gdn_fwd_bf16_b4h8t8192d256_c32_h0": Workload("gdn_fwd_bf16_b4h8t8192d256_c32_h0", 4, 8, 8192,
                                                  256, "bf16", True, True, 6, chunk=32),
}

WORKLOAD_ORDER: List[str] = list(WORKLOADS)


def varlen_lengths(total: int, n: int, seed: int, lo: int = 1024, hi: int = 16384) -> List[int]:
    """n lengths drawn uniformly from [lo, hi], rescaled to sum to ``total``,
    clamped to [lo, hi]; whatever rounding leaves over goes to the last one
    (and, if that would leave [lo, hi], is spread over the others)."""
    gen = torch.Generator().manual_seed(seed)
    raw = torch.randint(lo, hi + 1, (n,), generator=gen).tolist()
    s = float(sum(raw))
    lens = [min(hi, max(lo, int(round(x * total / s)))) for x in raw]
    lens[-1] += total - sum(lens)
    i = 0
    while not (lo <= lens[-1] <= hi):
        j = i % (n - 1)
        step = 1 if lens[-1] > hi else -1
        if lo <= lens[j] + step <= hi:
            lens[j] += step
            lens[-1] -= step
        i += 1
    return lens


def cu_seqlens_of(lengths: List[int]) -> torch.Tensor:
    out = [0]
    for L in lengths:
        out.append(out[-1] + L)
    return torch.tensor(out, dtype=torch.int32)


def generate(w: Workload, B: Optional[int] = None, H: Optional[int] = None,
             T: Optional[int] = None, d: Optional[int] = None,
             lengths: Optional[List[int]] = None, seed: Optional[int] = None) -> dict:
    """Draw one workload's inputs on the CPU.  Overrides (B, H, T, d, lengths,
    seed) give the same distributions at other sizes (small parity cases).

    Returns a dict of CPU tensors: q, k, v [NB,H,T,d] and beta [NB,H,T] in the
    workload dtype (bf16 values are the rounded fp32 draws); g [NB,H,T] fp32 or
    None; h0 [N,H,d,d] fp32 or None; cu_seqlens int32 or None; do, dhT for
    backward workloads; plus 'dtype' and 'lengths'."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    d = w.d if d is None else d
    seed = w.seed if seed is None else seed
    if w.varlen_total or lengths is not None:
        if lengths is None:
            lengths = varlen_lengths(w.varlen_total, w.varlen_n, w.seed)
        NB, Ttot, N = 1, int(sum(lengths)), len(lengths)
        cu = cu_seqlens_of(lengths)
    else:
        T = w.T if T is None else T
        NB, Ttot, N = B, T, B
        cu = None
    gen = torch.Generator().manual_seed(seed)
    f32 = torch.float32
    q = torch.randn((NB, H, Ttot, d), generator=gen, dtype=f32)
    k = torch.randn((NB, H, Ttot, d), generator=gen, dtype=f32)
    v = torch.randn((NB, H, Ttot, d), generator=gen, dtype=f32)
    beta = torch.sigmoid(torch.randn((NB, H, Ttot), generator=gen, dtype=f32))
    g = None
    if w.gated:
        g = -torch.nn.functional.softplus(torch.randn((NB, H, Ttot), generator=gen, dtype=f32)) / 16.0
    h0 = None
    if w.with_h0:
        h0 = 0.02 * torch.randn((N, H, d, d), generator=gen, dtype=f32)
    do = dhT = None
    if w.backward:
        do = torch.randn((NB, H, Ttot, d), generator=gen, dtype=f32)
        dhT = 0.01 * torch.randn((N, H, d, d), generator=gen, dtype=f32)
    if w.dtype == "bf16":
        q, k, v, beta = (x.to(torch.bfloat16) for x in (q, k, v, beta))
        if do is not None:
            do = do.to(torch.bfloat16)
    return dict(q=q, k=k, v=v, beta=beta, g=g, h0=h0, cu_seqlens=cu, do=do, dhT=dhT,
                dtype=w.dtype, lengths=lengths)
