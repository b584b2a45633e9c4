"""Thin ctypes binding of libgdn_gb300.so (include/gdn.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, and every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if the library is missing, or a
call returns an error status, these functions raise.

The names match the C ABI: dn_workspace_size, dn_chunk_fwd, gdn_chunk_fwd,
gdn_chunk_bwd, dn_saved_size, gdn_chunk_fwd_save, gdn_chunk_bwd_saved,
dn_host_arena_size, gdn_chunk_fwd_host, dn_device_status, dn_uses_fast_path,
dn_plan, gdn_chunk_fwd_noalloc, dn_noalloc_status, gdn_decode_step,
dn_state_affine.  ``forward`` / ``backward`` additionally
allocate outputs and the workspace with torch (device memory only) and, unless
told not to, read the device status word after the call (which synchronises the
stream) so that a bounded wait that ran out, malformed packed offsets or a
log-gate outside its domain raise instead of returning invalid results.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from ._build import LIB

(DN_OK, DN_ERR_INVALID_ARG, DN_ERR_UNSUPPORTED, DN_ERR_WORKSPACE, DN_ERR_CUDA, DN_ERR_TIMEOUT,
 DN_ERR_DOMAIN) = range(7)
DN_F32, DN_BF16 = 0, 1
DN_BETA_DELTA, DN_BETA_LONGHORN = 0, 1

EXPORTS = ["dn_workspace_size", "dn_chunk_fwd", "gdn_chunk_fwd", "gdn_chunk_bwd", "dn_saved_size",
           "gdn_chunk_fwd_save", "gdn_chunk_bwd_saved",
           "dn_host_arena_size", "gdn_chunk_fwd_host", "dn_device_status", "dn_status_str",
           "dn_uses_fast_path", "gdn_chunk_fwd_noalloc", "dn_noalloc_status", "dn_plan",
           "gdn_decode_step", "dn_state_affine"]


class DnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("T", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p),
                ("num_seqs", ctypes.c_int32), ("qk_l2norm", ctypes.c_int32),
                ("scale", ctypes.c_float), ("eps", ctypes.c_float), ("beta_mode", ctypes.c_int32)]


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (where, status_str(status), status))


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return LIB


def lib():
    """Load libgdn_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError("libgdn_gb300.so is not built (call __graft_entry__.build() or "
                                   "chunkwise_delta_rule_02_gb300._build.build()); there is no fallback")
            L = ctypes.CDLL(LIB)
            P, S, I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            SP = ctypes.POINTER(DnShape)
            L.dn_workspace_size.argtypes = [SP, I]
            L.dn_workspace_size.restype = S
            L.dn_uses_fast_path.argtypes = [SP, I]
            L.dn_uses_fast_path.restype = I
            L.dn_plan.argtypes = [SP, I, ctypes.POINTER(ctypes.c_int)]
            L.dn_plan.restype = I
            L.dn_chunk_fwd.argtypes = [SP, P, P, P, P, P, P, P, P, S, P]
            L.dn_chunk_fwd.restype = I
            L.gdn_chunk_fwd.argtypes = [SP, P, P, P, P, P, P, P, P, P, S, P]
            L.gdn_chunk_fwd.restype = I
            L.gdn_chunk_bwd.argtypes = [SP, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, S, P]
            L.gdn_chunk_bwd.restype = I
            L.dn_saved_size.argtypes = [SP]
            L.dn_saved_size.restype = S
            L.gdn_chunk_fwd_save.argtypes = [SP, P, P, P, P, P, P, P, P, P, S, P, S, P]
            L.gdn_chunk_fwd_save.restype = I
            L.gdn_chunk_bwd_saved.argtypes = [SP, P, P, P, P, P, P, P, P, S, P, P, P, P, P, P, P, S, P]
            L.gdn_chunk_bwd_saved.restype = I
            L.dn_host_arena_size.argtypes = [SP, I, I]
            L.dn_host_arena_size.restype = S
            L.gdn_chunk_fwd_host.argtypes = [SP, P, P, P, P, P, P, P, P, P, S, P, S, P]
            L.gdn_chunk_fwd_host.restype = I
            L.gdn_chunk_fwd_noalloc.argtypes = [SP, P, P, P, P, P, P, P, P, P]
            L.gdn_chunk_fwd_noalloc.restype = I
            L.gdn_decode_step.argtypes = [SP, P, P, P, P, P, P, P, P, P]
            L.gdn_decode_step.restype = I
            L.dn_device_status.argtypes = [P, P]
            L.dn_device_status.restype = I
            L.dn_noalloc_status.argtypes = [P]
            L.dn_noalloc_status.restype = I
            L.dn_state_affine.argtypes = [P, P, P, P, I, I, I, P]
            L.dn_state_affine.restype = I
            L.dn_status_str.argtypes = [I]
            L.dn_status_str.restype = ctypes.c_char_p
            _lib = L
    return _lib


def status_str(s: int) -> str:
    try:
        return lib().dn_status_str(int(s)).decode()
    except Exception:
        return "status %d" % s


def _p(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != DN_OK:
        raise GdnError(rc, where)


def make_shape(q: torch.Tensor, v: torch.Tensor, chunk: int = 64, cu_seqlens=None,
               scale: float = 1.0, qk_l2norm: bool = True, eps: float = 1e-6,
               longhorn: bool = False) -> DnShape:
    """Shape record for q [B,H,T,dk], v [B,H,T,dv]; cu_seqlens a device int32 tensor;
    longhorn: step size beta / (1 + beta k^T k) (DN_BETA_LONGHORN) instead of beta."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if q.dtype == torch.float32:
        dt = DN_F32
    elif q.dtype == torch.bfloat16:
        dt = DN_BF16
    else:
        raise TypeError("q must be float32 or bfloat16")
    s = DnShape(B, H, T, dk, dv, chunk, dt, None, 0, int(bool(qk_l2norm)), float(scale), float(eps),
                DN_BETA_LONGHORN if longhorn else DN_BETA_DELTA)
    if cu_seqlens is not None:
        s.cu_seqlens = _p(cu_seqlens)
        s.num_seqs = int(cu_seqlens.numel()) - 1
    return s


def dn_workspace_size(shape: DnShape, for_backward=False) -> int:
    """for_backward: False / True (gdn_chunk_bwd) or 2 (gdn_chunk_bwd_saved)."""
    return int(lib().dn_workspace_size(ctypes.byref(shape), int(for_backward)))


def dn_uses_fast_path(shape: DnShape, for_backward: bool = False) -> int:
    return int(lib().dn_uses_fast_path(ctypes.byref(shape), int(bool(for_backward))))


DN_PATH_GENERAL, DN_PATH_FUSED, DN_PATH_COOP = 0, 1, 2
PATH_NAMES = {DN_PATH_GENERAL: "general", DN_PATH_FUSED: "fused", DN_PATH_COOP: "coop"}


def dn_plan(shape: DnShape, for_backward=False):
    """(path, kernels per call): DN_PATH_* and the number of library kernels one call
    launches; for_backward as in dn_workspace_size."""
    n = ctypes.c_int(0)
    path = int(lib().dn_plan(ctypes.byref(shape), int(for_backward), ctypes.byref(n)))
    return path, int(n.value)


def dn_host_arena_size(shape: DnShape, gated: bool, with_h0: bool) -> int:
    return int(lib().dn_host_arena_size(ctypes.byref(shape), int(gated), int(with_h0)))


def dn_chunk_fwd(shape, q, k, v, beta, h0, o, hT, ws, stream=None):
    rc = lib().dn_chunk_fwd(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(beta), _p(h0), _p(o),
                            _p(hT), _p(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "dn_chunk_fwd")


def gdn_chunk_fwd(shape, q, k, v, beta, g, h0, o, hT, ws, stream=None):
    rc = lib().gdn_chunk_fwd(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(beta), _p(g), _p(h0),
                             _p(o), _p(hT), _p(ws), ws.numel() * ws.element_size(),
                             _stream(stream))
    _check(rc, "gdn_chunk_fwd")


def gdn_chunk_bwd(shape, q, k, v, beta, g, h0, dO, dhT, dq, dk, dv, dbeta, dg, dh0, ws,
                  stream=None):
    rc = lib().gdn_chunk_bwd(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(beta), _p(g), _p(h0),
                             _p(dO), _p(dhT), _p(dq), _p(dk), _p(dv), _p(dbeta), _p(dg),
                             _p(dh0), _p(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "gdn_chunk_bwd")


def dn_saved_size(shape) -> int:
    """Bytes of the buffer gdn_chunk_fwd_save fills (0: no saved path for the shape)."""
    return int(lib().dn_saved_size(ctypes.byref(shape)))


def gdn_chunk_fwd_save(shape, q, k, v, beta, g, h0, o, hT, saved, ws, stream=None):
    rc = lib().gdn_chunk_fwd_save(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(beta), _p(g), _p(h0),
                                  _p(o), _p(hT), _p(saved), saved.numel() * saved.element_size(),
                                  _p(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "gdn_chunk_fwd_save")


def gdn_chunk_bwd_saved(shape, q, k, v, beta, g, dO, dhT, saved, dq, dk, dv, dbeta, dg, dh0, ws,
                        stream=None):
    rc = lib().gdn_chunk_bwd_saved(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(beta), _p(g), _p(dO),
                                   _p(dhT), _p(saved), saved.numel() * saved.element_size(), _p(dq),
                                   _p(dk), _p(dv), _p(dbeta), _p(dg), _p(dh0), _p(ws),
                                   ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "gdn_chunk_bwd_saved")


def gdn_chunk_fwd_host(shape, q, k, v, beta, g, h0, o, hT, arena, ws, stream=None):
    """Host (pinned CPU) tensors in and out; arena and ws are device tensors."""
    rc = lib().gdn_chunk_fwd_host(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(beta), _p(g),
                                  _p(h0), _p(o), _p(hT), _p(arena),
                                  arena.numel() * arena.element_size(), _p(ws),
                                  ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "gdn_chunk_fwd_host")


def gdn_chunk_fwd_noalloc(shape, q, k, v, beta, g, h0, o, hT, stream=None):
    """Forward without workspace or allocation (scratch in the library's static
    device array; bf16, d = 128, chunk 64 only)."""
    rc = lib().gdn_chunk_fwd_noalloc(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(beta), _p(g),
                                     _p(h0), _p(o), _p(hT), _stream(stream))
    _check(rc, "gdn_chunk_fwd_noalloc")


def gdn_decode_step(shape, q, k, v, beta, g, state_in, state_out, o, stream=None):
    """One recurrent step per sequence: q, k [N,H,dk], v [N,H,dv], beta [N,H], g [N,H] or
    None, states [N,H,dk,dv] float32 (state_out may be state_in), o [N,H,dv]."""
    rc = lib().gdn_decode_step(ctypes.byref(shape), _p(q), _p(k), _p(v), _p(beta), _p(g),
                               _p(state_in), _p(state_out), _p(o), _stream(stream))
    _check(rc, "gdn_decode_step")


def decode_step(q, k, v, beta, g=None, state=None, out_state=None, scale=1.0, qk_l2norm=True,
                eps=1e-6, longhorn=False):
    """Allocate o (and the new state unless out_state is given; pass out_state=state for an
    in-place update) and run gdn_decode_step.  q, k [N,H,dk].  Returns (o, new_state)."""
    N, H, dk = q.shape
    dv = v.shape[-1]
    shape = make_shape(q.view(N, H, 1, dk), v.view(N, H, 1, dv), 64, None, scale, qk_l2norm, eps,
                       longhorn)
    o = torch.empty((N, H, dv), dtype=v.dtype, device=v.device)
    if out_state is None:
        out_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    gdn_decode_step(shape, q, k, v, beta, g, state, out_state, o)
    return o, out_state


def dn_state_affine(A, S, B, out, stream=None):
    """out_i = A_i S_i + B_i over the leading dimensions: A [..., dk, dk], S, B, out
    [..., dk, dv], float32 device tensors (B may be None)."""
    dk, dv = S.shape[-2], S.shape[-1]
    count = S.numel() // (dk * dv) if S.numel() else 0
    for t in (A, S, B, out):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise TypeError("dn_state_affine takes contiguous float32 tensors")
    rc = lib().dn_state_affine(_p(A), _p(S), _p(B), _p(out), count, dk, dv, _stream(stream))
    _check(rc, "dn_state_affine")


def dn_device_status(ws, stream=None) -> int:
    return int(lib().dn_device_status(_p(ws), _stream(stream)))


def dn_noalloc_status(stream=None) -> int:
    """Status word of the most recent gdn_chunk_fwd_noalloc call (syncs the stream)."""
    return int(lib().dn_noalloc_status(_stream(stream)))


def alloc_workspace(shape: DnShape, for_backward, device) -> torch.Tensor:
    """for_backward: False / True (gdn_chunk_bwd) or 2 (gdn_chunk_bwd_saved)."""
    n = dn_workspace_size(shape, int(for_backward))
    if n == 0:
        raise GdnError(DN_ERR_INVALID_ARG, "dn_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _nseq(q, cu_seqlens):
    return q.shape[0] if cu_seqlens is None else int(cu_seqlens.numel()) - 1


def saved_supported(q, v, chunk=64, cu_seqlens=None, scale=1.0, qk_l2norm=True, eps=1e-6,
                    longhorn=False) -> bool:
    """Whether forward(save=True) / backward(saved=...) run for these inputs."""
    return dn_saved_size(make_shape(q, v, chunk, cu_seqlens, scale, qk_l2norm, eps, longhorn)) > 0


def forward(q, k, v, beta, g=None, h0=None, cu_seqlens=None, chunk=64, scale=1.0,
            qk_l2norm=True, eps=1e-6, want_state=True, ws=None, longhorn=False,
            check_status=True, save=False):
    """Allocate o (and hT) and run gdn_chunk_fwd / dn_chunk_fwd.  Returns (o, hT).
    check_status: read the device status word afterwards (synchronises the stream)
    and raise GdnError if the kernels flagged anything.  save=True runs
    gdn_chunk_fwd_save and returns (o, hT, saved) for backward(saved=saved)."""
    shape = make_shape(q, v, chunk, cu_seqlens, scale, qk_l2norm, eps, longhorn)
    if save:
        n = dn_saved_size(shape)
        if n == 0:
            raise GdnError(DN_ERR_UNSUPPORTED, "gdn_chunk_fwd_save")
        saved = torch.empty(n, dtype=torch.uint8, device=q.device)
        o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
        hT = torch.empty((_nseq(q, cu_seqlens), q.shape[1], q.shape[-1], v.shape[-1]), dtype=torch.float32,
                         device=q.device) if want_state else None
        if ws is None:
            ws = alloc_workspace(shape, False, q.device)
        gdn_chunk_fwd_save(shape, q, k, v, beta, g, h0, o, hT, saved, ws)
        if check_status:
            _check(dn_device_status(ws), "gdn_chunk_fwd_save (device status)")
        return o, hT, saved
    o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    N = _nseq(q, cu_seqlens)
    hT = torch.empty((N, q.shape[1], q.shape[-1], v.shape[-1]), dtype=torch.float32,
                     device=q.device) if want_state else None
    if ws is None:
        ws = alloc_workspace(shape, False, q.device)
    if g is None:
        dn_chunk_fwd(shape, q, k, v, beta, h0, o, hT, ws)
    else:
        gdn_chunk_fwd(shape, q, k, v, beta, g, h0, o, hT, ws)
    if check_status:
        _check(dn_device_status(ws), "gdn_chunk_fwd (device status)")
    return o, hT


def backward(q, k, v, beta, g, h0, dO, dhT, cu_seqlens=None, chunk=64, scale=1.0,
             qk_l2norm=True, eps=1e-6, ws=None, longhorn=False, check_status=True, saved=None):
    """Allocate the gradients and run gdn_chunk_bwd (or, with the buffer of
    forward(save=True), gdn_chunk_bwd_saved).  Returns a dict.  check_status as in
    forward."""
    shape = make_shape(q, v, chunk, cu_seqlens, scale, qk_l2norm, eps, longhorn)
    out = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
               dbeta=torch.empty_like(beta),
               dg=torch.empty_like(g) if g is not None else None,
               dh0=torch.empty((_nseq(q, cu_seqlens), q.shape[1], q.shape[-1], v.shape[-1]),
                               dtype=torch.float32, device=q.device))
    if saved is not None:
        if ws is None:
            ws = alloc_workspace(shape, 2, q.device)
        gdn_chunk_bwd_saved(shape, q, k, v, beta, g, dO, dhT, saved, out["dq"], out["dk"], out["dv"],
                            out["dbeta"], out["dg"], out["dh0"], ws)
        if check_status:
            _check(dn_device_status(ws), "gdn_chunk_bwd_saved (device status)")
        return out
    if ws is None:
        ws = alloc_workspace(shape, True, q.device)
    gdn_chunk_bwd(shape, q, k, v, beta, g, h0, dO, dhT, out["dq"], out["dk"], out["dv"],
                  out["dbeta"], out["dg"], out["dh0"], ws)
    if check_status:
        _check(dn_device_status(ws), "gdn_chunk_bwd (device status)")
    return out
