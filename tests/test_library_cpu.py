"""Host-side checks that need no GPU: the C ABI library loads, exports every
function include/gdn.h declares, sizes its workspace, and rejects bad arguments
with a status code before touching the device.  Also the seeded input
generators."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gdn():
    import __graft_entry__
    __graft_entry__.build()
    from chunkwise_delta_rule_02_gb300 import binding
    return binding


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z][a-z0-9_]+)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("dn_chunk_fwd", "gdn_chunk_fwd", "gdn_chunk_bwd", "dn_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(gdn):
    lib = ctypes.CDLL(gdn.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name
    for name in gdn.EXPORTS:
        assert hasattr(lib, name), name


def _shape(gdn, B=2, H=3, T=100, d=64, dtype=1, chunk=64, cu=None, N=0, beta_mode=0):
    s = gdn.DnShape(B, H, T, d, d, chunk, dtype, cu, N, 1, 1.0, 1e-6, beta_mode)
    return s


def test_workspace_size_and_validation(gdn):
    s = _shape(gdn)
    n_f = gdn.dn_workspace_size(s, False)
    n_b = gdn.dn_workspace_size(s, True)
    assert 0 < n_f < n_b
    assert n_f % 256 == 0
    bad = [_shape(gdn, B=0), _shape(gdn, d=257), _shape(gdn, chunk=48), _shape(gdn, dtype=7),
           _shape(gdn, H=0), _shape(gdn, T=-1)]
    for b in bad:
        assert gdn.dn_workspace_size(b, False) == 0
        assert gdn.dn_uses_fast_path(b, False) == -1
    assert gdn.dn_workspace_size(_shape(gdn, B=2, cu=16, N=3), False) == 0   # packed needs B == 1
    assert gdn.dn_workspace_size(_shape(gdn, B=1, cu=16, N=3), False) > 0


def test_host_arena_size(gdn):
    """gdn_chunk_fwd_host's device arena: q, k, v, o, beta, g and the states each in a
    256-byte aligned block, the states being h0, h_T and the two that carry the state
    between the time segments of the pipelined call; 0 on bad arguments."""
    a256 = lambda n: (n + 255) // 256 * 256
    B, H, T, d = 2, 3, 1000, 128
    s = _shape(gdn, B=B, H=H, T=T, d=d)
    tok, st = B * H * T, B * H * d * d * 4
    base = 4 * a256(tok * d * 2) + a256(tok * 2) + 3 * a256(st)   # q k v o, beta, hT + 2 between
    assert gdn.dn_host_arena_size(s, False, False) == base
    assert gdn.dn_host_arena_size(s, True, False) == base + a256(tok * 4)
    assert gdn.dn_host_arena_size(s, True, True) == base + a256(tok * 4) + a256(st)
    assert gdn.dn_host_arena_size(_shape(gdn, B=0), True, True) == 0


def test_beta_mode_is_validated(gdn):
    """DN_BETA_DELTA and DN_BETA_LONGHORN are the two step-size modes; any other value
    is rejected before any device work, and Longhorn's needs no extra workspace
    beyond the per-token step sizes every general-path call records."""
    for mode in (gdn.DN_BETA_DELTA, gdn.DN_BETA_LONGHORN):
        for bwd in (False, True):
            assert gdn.dn_workspace_size(_shape(gdn, beta_mode=mode), bwd) == \
                gdn.dn_workspace_size(_shape(gdn), bwd)
    for mode in (2, -1, 7):
        assert gdn.dn_workspace_size(_shape(gdn, beta_mode=mode), False) == 0
        assert gdn.dn_uses_fast_path(_shape(gdn, beta_mode=mode), False) == -1


def test_plan_reports_path_and_kernel_count(gdn):
    # fp32 runs the three general kernels, the backward six; packed input adds k_cstart
    assert gdn.dn_plan(_shape(gdn, dtype=0), False) == (gdn.DN_PATH_GENERAL, 3)
    assert gdn.dn_plan(_shape(gdn, d=128), True) == (gdn.DN_PATH_GENERAL, 6)
    assert gdn.dn_plan(_shape(gdn, B=1, dtype=0, cu=16, N=3), False) == (gdn.DN_PATH_GENERAL, 4)
    # bf16 d = 128 takes one of the tcgen05 kernels on an sm_103 device (one launch, plus
    # two for packed input); without such a device it falls to the general kernels
    fused = (gdn.DN_PATH_FUSED, gdn.DN_PATH_COOP)
    path, n = gdn.dn_plan(_shape(gdn, d=128), False)
    assert (path in fused and n == 1) or (path == gdn.DN_PATH_GENERAL and n == 3)
    path, n = gdn.dn_plan(_shape(gdn, B=1, d=128, cu=16, N=3), False)
    assert (path in fused and n == 3) or (path == gdn.DN_PATH_GENERAL and n == 4)
    assert gdn.dn_plan(_shape(gdn, B=0), False)[0] == -1


def test_status_codes_without_device_work(gdn):
    L = gdn.lib()
    s = _shape(gdn)
    # null shape
    assert L.gdn_chunk_fwd(None, 16, 16, 16, 16, None, None, 16, None, 16, 1 << 40, None) == gdn.DN_ERR_INVALID_ARG
    # null input pointer
    assert L.gdn_chunk_fwd(ctypes.byref(s), None, 16, 16, 16, None, None, 16, None, 16, 1 << 40, None) == gdn.DN_ERR_INVALID_ARG
    # misaligned pointer
    assert L.gdn_chunk_fwd(ctypes.byref(s), 18, 16, 16, 16, None, None, 16, None, 16, 1 << 40, None) == gdn.DN_ERR_INVALID_ARG
    # workspace missing / too small
    assert L.gdn_chunk_fwd(ctypes.byref(s), 16, 16, 16, 16, None, None, 16, None, None, 0, None) == gdn.DN_ERR_WORKSPACE
    assert L.gdn_chunk_fwd(ctypes.byref(s), 16, 16, 16, 16, None, None, 16, None, 16, 64, None) == gdn.DN_ERR_WORKSPACE
    # unsupported head dim
    s2 = _shape(gdn, d=512)
    assert L.dn_chunk_fwd(ctypes.byref(s2), 16, 16, 16, 16, None, 16, None, 16, 1 << 40, None) == gdn.DN_ERR_UNSUPPORTED
    # backward: dg without g
    assert L.gdn_chunk_bwd(ctypes.byref(s), 16, 16, 16, 16, None, None, 16, None, 16, 16, 16, 16,
                           16, None, 16, 1 << 40, None) == gdn.DN_ERR_INVALID_ARG
    for code in range(6):
        assert gdn.status_str(code)


def test_workloads_are_seeded_and_shaped():
    from chunkwise_delta_rule_02_gb300 import workloads as W
    for name, w in W.WORKLOADS.items():
        x = W.generate(w, B=1 if not w.varlen_total else None, H=2, T=70 if not w.varlen_total else None,
                       lengths=[5, 70, 0, 9] if w.varlen_total else None)
        y = W.generate(w, B=1 if not w.varlen_total else None, H=2, T=70 if not w.varlen_total else None,
                       lengths=[5, 70, 0, 9] if w.varlen_total else None)
        for key in ("q", "k", "v", "beta", "g", "h0", "do", "dhT"):
            if x[key] is not None:
                assert torch.equal(x[key], y[key]), (name, key)
        assert (x["g"] is not None) == w.gated
        if x["g"] is not None:
            assert float(x["g"].max()) < 0.0
        want = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        assert x["q"].dtype == want and x["beta"].dtype == want
    lens = W.varlen_lengths(65536, 8, 3)
    assert sum(lens) == 65536 and len(lens) == 8
    assert all(1024 <= L <= 16384 for L in lens)
    full = W.generate(W.WORKLOADS["gdn_fwd_bf16_varlen_h32_n8_t65536"])
    assert full["q"].shape == (1, 32, 65536, 128)
    assert full["cu_seqlens"].tolist()[-1] == 65536


def test_state_affine_checks_its_arguments_on_the_host(gdn):
    """dn_state_affine rejects bad sizes, misaligned pointers and an output that
    overlaps A or S before launching anything (no device is touched here)."""
    lib = gdn.lib()
    base = 1 << 20
    ok_ptrs = (base, base + 0x100000, base + 0x200000, base + 0x300000)
    assert lib.dn_state_affine(*ok_ptrs[:4], 0, 16, 16, None) == gdn.DN_OK          # nothing to do
    assert lib.dn_state_affine(*ok_ptrs[:4], -1, 16, 16, None) == gdn.DN_ERR_INVALID_ARG
    assert lib.dn_state_affine(*ok_ptrs[:4], 2, 300, 16, None) == gdn.DN_ERR_INVALID_ARG
    assert lib.dn_state_affine(*ok_ptrs[:4], 70000, 16, 16, None) == gdn.DN_ERR_UNSUPPORTED
    assert lib.dn_state_affine(base + 2, *ok_ptrs[1:4], 2, 16, 16, None) == gdn.DN_ERR_INVALID_ARG
    # out overlapping S, then A
    assert lib.dn_state_affine(base, base + 0x100000, None, base + 0x100000 + 64, 2, 16, 16,
                               None) == gdn.DN_ERR_INVALID_ARG
    assert lib.dn_state_affine(base, base + 0x100000, None, base + 1024, 2, 16, 16,
                               None) == gdn.DN_ERR_INVALID_ARG
