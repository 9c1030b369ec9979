"""The C-ABI library builds, loads and exports every entry point include/attn.h declares;
host-side argument checks reject bad calls before any CUDA work (no GPU needed)."""
import ctypes
import os
import re

import pytest

import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import build as ofa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ofa_build.build()
    return ofa.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_decode_splitkv", "attn_merge_states",
              "attn_decode_workspace_bytes", "attn_last_error", "attn_device_error_flags"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/attn.h but not exported"


def test_version_and_workspace_size(lib):
    assert lib.attn_version() >= 100
    assert ofa.decode_workspace_bytes(64, 32, 128, 16) == 64 * 32 * 16 * 130 * 4
    assert ofa.decode_workspace_bytes(-1, 32, 128, 16) == 0
    assert ofa.decode_workspace_bytes(64, 32, 128, 16, Nq=4) == 4 * 64 * 32 * 16 * 130 * 4
    assert ofa.decode_workspace_bytes(64, 32, 128, 16, Nq=0) == 0
    # the fused decode: the same partial states (rounded up to 16 bytes), then a uint64 per (b, h)
    assert ofa.decode_fused_workspace_bytes(64, 32, 128, 16) == 64 * 32 * 16 * 130 * 4 + 64 * 32 * 8
    assert ofa.decode_fused_workspace_bytes(3, 1, 64, 1) == 16 * ((3 * 66 * 4 + 15) // 16) + 3 * 8
    assert ofa.decode_fused_workspace_bytes(3, 1, 64, 0) == 0


def test_fused_decode_checks_its_workspace_on_the_host(lib):
    p = _params(Nq=1, Nk=64)
    need = ofa.decode_fused_workspace_bytes(1, 1, 128, 4)
    assert lib.attn_decode_splitkv_fused(ctypes.byref(p), 4, ctypes.c_void_p(0x50000), need - 4, None) \
        == ofa.Status.WORKSPACE
    assert lib.attn_decode_splitkv_fused(ctypes.byref(p), 4, ctypes.c_void_p(0x50008), need, None) \
        == ofa.Status.WORKSPACE
    assert lib.attn_decode_splitkv_fused(ctypes.byref(p), 0, ctypes.c_void_p(0x50000), need, None) \
        == ofa.Status.INVALID_ARG


def _params(**kw):
    p = ofa.Params()
    p.dtype, p.causal = 1, 0
    p.B, p.H, p.Nq, p.Nk, p.dk, p.dv = 1, 1, 16, 16, 128, 128
    p.q, p.k, p.v, p.o = 0x10000, 0x20000, 0x30000, 0x40000
    for s in ("q_stride", "k_stride", "v_stride", "o_stride"):
        setattr(p, s, (ctypes.c_int64 * 3)(16 * 128, 128, 128))
    p.scale = 0.088
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=7), ofa.Status.INVALID_ARG),
    (dict(causal=2), ofa.Status.INVALID_ARG),
    (dict(B=-1), ofa.Status.INVALID_ARG),
    (dict(dk=0), ofa.Status.INVALID_ARG),
    (dict(scale=float("nan")), ofa.Status.INVALID_ARG),
    (dict(q=None), ofa.Status.INVALID_ARG),
    (dict(dk=96, dv=96), ofa.Status.UNSUPPORTED),
    (dict(dv=192), ofa.Status.UNSUPPORTED),
    (dict(scale=-1.0), ofa.Status.UNSUPPORTED),
    (dict(q=0x10002), ofa.Status.MISALIGNED),
    (dict(k_stride=(ctypes.c_int64 * 3)(16 * 128, 132, 128)), ofa.Status.MISALIGNED),
    (dict(block_k=16), ofa.Status.INVALID_ARG),
    (dict(dtype=0, block_k=48), ofa.Status.INVALID_ARG),
    (dict(dtype=0, dk=300), ofa.Status.UNSUPPORTED),
])
def test_fwd_rejects_bad_arguments_on_the_host(lib, kw, status):
    p = _params(**kw)
    st = lib.attn_fwd(ctypes.byref(p), None)
    assert st == status, ofa.last_error()
    assert ofa.last_error()


def test_null_params_and_empty_problem(lib):
    assert lib.attn_fwd(None, None) == ofa.Status.INVALID_ARG
    p = _params(Nq=0)
    assert lib.attn_fwd(ctypes.byref(p), None) == ofa.Status.OK  # nothing to do


def test_decode_rejects_bad_arguments_on_the_host(lib):
    p = _params(Nq=1)
    ws = ctypes.c_void_p(0x50000)
    assert lib.attn_decode_splitkv(ctypes.byref(p), 0, ws, 1 << 20, None) == ofa.Status.INVALID_ARG
    assert lib.attn_decode_splitkv(ctypes.byref(p), 300, ws, 1 << 20, None) == ofa.Status.INVALID_ARG
    assert lib.attn_decode_splitkv(ctypes.byref(p), 4, ws, 16, None) == ofa.Status.WORKSPACE
    assert lib.attn_decode_splitkv(ctypes.byref(p), 4, None, 1 << 20, None) == ofa.Status.WORKSPACE
    p2 = _params(Nq=9)  # more query rows than the decode takes
    assert lib.attn_decode_splitkv(ctypes.byref(p2), 4, ws, 1 << 20, None) == ofa.Status.INVALID_ARG
    p2 = _params(Nq=0)
    assert lib.attn_decode_splitkv(ctypes.byref(p2), 4, ws, 1 << 20, None) == ofa.Status.INVALID_ARG
    # Nq rows need Nq times the partial states of one row
    p2 = _params(Nq=3)
    one = lib.attn_decode_workspace_bytes(p2.B, p2.H, p2.dv, 4)
    assert lib.attn_decode_workspace_bytes_rows(p2.B, p2.H, 3, p2.dv, 4) == 3 * one
    assert lib.attn_decode_splitkv(ctypes.byref(p2), 4, ws, 3 * one - 16, None) == ofa.Status.WORKSPACE
    p3 = _params(Nq=1, dtype=0)
    assert lib.attn_decode_splitkv(ctypes.byref(p3), 4, ws, 1 << 20, None) == ofa.Status.UNSUPPORTED
    p4 = _params(Nq=1, dk=128, dv=64)
    assert lib.attn_decode_splitkv(ctypes.byref(p4), 4, ws, 1 << 20, None) == ofa.Status.UNSUPPORTED


def test_merge_rejects_bad_arguments_on_the_host(lib):
    st = (ctypes.c_int64 * 3)(128, 128, 128)
    assert lib.attn_merge_states(None, 1, 1, 4, 128, 1, ctypes.c_void_p(0x1000), st, None,
                                 None) == ofa.Status.INVALID_ARG
    assert lib.attn_merge_states(ctypes.c_void_p(0x1000), 1, 1, 0, 128, 1, ctypes.c_void_p(0x1000),
                                 st, None, None) == ofa.Status.INVALID_ARG
    assert lib.attn_merge_states(ctypes.c_void_p(0x1000), 1, 1, 4, 128, 5, ctypes.c_void_p(0x1000),
                                 st, None, None) == ofa.Status.INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 4, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ofa.attn_fwd(q, q, q)


def test_bwd_rejects_bad_arguments_on_the_host(lib):
    def bp(**kw):
        p = ofa.BwdParams()
        p.fwd = _params(Nq=64, Nk=64, **kw)
        p.fwd.lse = 0x60000
        for name, addr in (("dout", 0x70000), ("dq", 0x80000), ("dk", 0x90000), ("dv", 0xA0000)):
            setattr(p, name, addr)
            setattr(p, name + "_stride", (ctypes.c_int64 * 3)(16 * 128, 128, 128))
        return p
    ws = ctypes.c_void_p(0xB0000)
    need = lib.attn_bwd_workspace_bytes(1, 1, 64, 128)
    # fp32 dQ accumulator, c per row, and lse * log2 e with rows padded to a multiple of 128
    assert need == 64 * 128 * 4 + 64 * 4 + 128 * 4
    assert lib.attn_bwd(None, ws, need, None) == ofa.Status.INVALID_ARG
    assert lib.attn_bwd(ctypes.byref(bp(dtype=0)), ws, need, None) == ofa.Status.UNSUPPORTED
    assert lib.attn_bwd(ctypes.byref(bp(dk=192)), ws, need, None) == ofa.Status.UNSUPPORTED
    assert lib.attn_bwd(ctypes.byref(bp()), ws, need - 4, None) == ofa.Status.WORKSPACE
    assert lib.attn_bwd(ctypes.byref(bp()), None, need, None) == ofa.Status.WORKSPACE
    p = bp()
    p.fwd.lse = None
    assert lib.attn_bwd(ctypes.byref(p), ws, need, None) == ofa.Status.INVALID_ARG
    p = bp()
    p.dq = 0x80004  # not 16-byte aligned
    assert lib.attn_bwd(ctypes.byref(p), ws, need, None) == ofa.Status.MISALIGNED
    assert lib.attn_bwd_workspace_bytes(-1, 1, 64, 128) == 0


def _mask_stride(nb=16):
    return (ctypes.c_int64 * 3)(16 * nb, 16 * nb, nb)


@pytest.mark.parametrize("kw,status", [
    (dict(dropout_p=0.1), ofa.Status.INVALID_ARG),                                  # p without a mask
    (dict(dropout_mask=0x100000, dropout_p=1.0), ofa.Status.INVALID_ARG),           # p outside [0, 1)
    (dict(dropout_mask=0x100000, dropout_p=-0.1), ofa.Status.INVALID_ARG),
    (dict(dropout_mask=0x100000, dropout_p=float("nan")), ofa.Status.INVALID_ARG),
    (dict(dropout_mask=0x100000, dropout_p=0.1,
          dropout_mask_stride=(ctypes.c_int64 * 3)(256, 16, -16)), ofa.Status.INVALID_ARG),
    (dict(dropout_mask=0x100008, dropout_p=0.1), ofa.Status.MISALIGNED),            # base not 16-aligned
    (dict(dropout_mask=0x100000, dropout_p=0.1,
          dropout_mask_stride=(ctypes.c_int64 * 3)(256, 16, 8)), ofa.Status.MISALIGNED),
    (dict(dropout_mask=0x100000, dropout_p=0.1, dk=192), ofa.Status.UNSUPPORTED),   # dk = 192: not built
])
def test_fwd_rejects_bad_dropout_arguments_on_the_host(lib, kw, status):
    kw.setdefault("dropout_mask_stride", _mask_stride())
    p = _params(**kw)
    st = lib.attn_fwd(ctypes.byref(p), None)
    assert st == status, ofa.last_error()


def test_decode_refuses_and_bwd_restricts_a_dropout_mask(lib):
    ws = ctypes.c_void_p(0x50000)
    p = _params(Nq=1, dropout_mask=0x100000, dropout_mask_stride=_mask_stride(), dropout_p=0.1)
    assert lib.attn_decode_splitkv(ctypes.byref(p), 4, ws, 1 << 20, None) == ofa.Status.UNSUPPORTED

    def bp(mask=0x100000, stride=None, **kw):
        b = ofa.BwdParams()
        b.fwd = _params(Nq=64, Nk=64, dropout_mask=mask, dropout_mask_stride=stride or _mask_stride(),
                        dropout_p=0.1, **kw)
        b.fwd.lse = 0x60000
        for name, addr in (("dout", 0x70000), ("dq", 0x80000), ("dk", 0x90000), ("dv", 0xA0000)):
            setattr(b, name, addr)
            setattr(b, name + "_stride", (ctypes.c_int64 * 3)(16 * 128, 128, 128))
        return b
    wsb = ctypes.c_void_p(0xB0000)
    need = lib.attn_bwd_workspace_bytes(1, 1, 64, 64)
    # the backward of a dropout forward takes no bias
    b = bp()
    b.fwd.bias = 0xC0000
    assert lib.attn_bwd(ctypes.byref(b), wsb, 1 << 20, None) == ofa.Status.UNSUPPORTED
    assert lib.attn_bwd(ctypes.byref(bp(mask=0x100004)), wsb, 1 << 20, None) == ofa.Status.MISALIGNED
    assert lib.attn_bwd(ctypes.byref(bp(stride=(ctypes.c_int64 * 3)(256, 16, 4))), wsb, 1 << 20,
                        None) == ofa.Status.MISALIGNED
