"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the fp64 oracle on the same (bf16-rounded, upcast) inputs, compare."""
import numpy as np
import torch

import oracle

TOL = {"f32": 1e-4, "bf16": 2e-2}   # relative Frobenius error bound per tensor


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    if nb == 0.0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def f64(t):
    return None if t is None else t.detach().to("cpu").double().numpy()


def to_dev(x, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def oracle_fwd(x, scale=1.0, sel=None):
    """Oracle forward on the generated inputs; sel = list of (b, h) (fixed length) to
    restrict to sampled items.  Returns (o, hT) arrays aligned with sel."""
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].numpy().astype(np.int64)
    if sel is None:
        return oracle.fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["beta"]), f64(x["g"]),
                          f64(x["h0"]), cu_seqlens=cu, scale=scale)
    outs = []
    for b, h in sel:
        sl = lambda t: None if t is None else t[b:b + 1, h:h + 1]
        outs.append(oracle.fwd(f64(sl(x["q"])), f64(sl(x["k"])), f64(sl(x["v"])),
                               f64(sl(x["beta"])), f64(sl(x["g"])), f64(sl(x["h0"])), scale=scale))
    return outs


def oracle_bwd(x, scale=1.0, sel=None):
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].numpy().astype(np.int64)
    if sel is None:
        return oracle.bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["beta"]), f64(x["g"]),
                          f64(x["h0"]), f64(x["do"]), f64(x["dhT"]), cu_seqlens=cu, scale=scale)
    outs = []
    for b, h in sel:
        sl = lambda t: None if t is None else t[b:b + 1, h:h + 1]
        outs.append(oracle.bwd(f64(sl(x["q"])), f64(sl(x["k"])), f64(sl(x["v"])),
                               f64(sl(x["beta"])), f64(sl(x["g"])), f64(sl(x["h0"])),
                               f64(sl(x["do"])), f64(sl(x["dhT"])), scale=scale))
    return outs
