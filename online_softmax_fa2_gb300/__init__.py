"""Exact attention forward on NVIDIA GB300 (sm_103a): thin Python binding over the C ABI.

Every step of the computation runs in the CUDA kernels of ``libattn_gb300.so`` (declared in
``include/attn.h``); this module only marshals torch tensors into the C structs and calls the
library on torch's current CUDA stream.  There is no CPU path: without the built library or a
CUDA device every call raises.

    o, lse = attn_fwd(q, k, v, bias=None, kv_lens=None, causal=False, scale=None)
    o, lse = attn_decode_splitkv(q, k_cache, v_cache, kv_lens, num_splits=16)
    o, lse = attn_merge_states(partials)

Shapes: q [B, Nq, H, dk], k [B, Nk, H, dk], v [B, Nk, H, dv] (any strides with the last
dimension contiguous), bias [B, H, Nq, Nk] fp32 (any strides with the last dimension
contiguous, 0 strides broadcast), kv_lens int32 [B].  Outputs o [B, Nq, H, dv] in q's dtype
and lse [B, H, Nq] fp32.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

__all__ = ["attn_fwd", "attn_fwd_partial", "attn_merge_states_rows", "attn_bwd", "attn_decode_splitkv",
           "attn_decode_splitkv_fused", "attn_decode_splitkv_noalloc",
           "attn_merge_states", "decode_workspace_bytes", "bwd_workspace_bytes",
           "device_error_flags", "last_error", "library_path", "load", "AttnError", "Status"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libattn_gb300.so")
_lib = None
_lock = threading.Lock()


class Status:
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    MISALIGNED = 3
    CUDA = 4
    DEVICE_TIMEOUT = 5
    WORKSPACE = 6


F32, BF16 = 0, 1


class AttnError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"attn status {status}: {msg}")
        self.status = status


class Params(ctypes.Structure):
    """Mirror of attn_fwd_params_t (include/attn.h)."""
    _fields_ = [
        ("dtype", ctypes.c_int32), ("causal", ctypes.c_int32),
        ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("Nq", ctypes.c_int64),
        ("Nk", ctypes.c_int64), ("dk", ctypes.c_int64), ("dv", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3),
        ("lse", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("bias_stride", ctypes.c_int64 * 3),
        ("kv_lens", ctypes.c_void_p),
        ("scale", ctypes.c_float), ("block_k", ctypes.c_int32),
        ("dropout_mask", ctypes.c_void_p), ("dropout_mask_stride", ctypes.c_int64 * 3),
        ("dropout_p", ctypes.c_float), ("dropout_rng", ctypes.c_int32),
        ("dropout_seed", ctypes.c_uint64), ("dropout_offset", ctypes.c_uint64),
    ]


class BwdParams(ctypes.Structure):
    """Mirror of attn_bwd_params_t (include/attn.h)."""
    _fields_ = [
        ("fwd", Params),
        ("dout", ctypes.c_void_p), ("dout_stride", ctypes.c_int64 * 3),
        ("dq", ctypes.c_void_p), ("dq_stride", ctypes.c_int64 * 3),
        ("dk", ctypes.c_void_p), ("dk_stride", ctypes.c_int64 * 3),
        ("dv", ctypes.c_void_p), ("dv_stride", ctypes.c_int64 * 3),
    ]


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libattn_gb300.so (built by ``online_softmax_fa2_gb300.build``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER(Params)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.attn_fwd.argtypes = [P, vp]
        lib.attn_fwd.restype = i32
        lib.attn_decode_workspace_bytes.argtypes = [i64, i64, i64, i32]
        lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_decode_workspace_bytes_rows.argtypes = [i64, i64, i64, i64, i32]
        lib.attn_decode_workspace_bytes_rows.restype = ctypes.c_size_t
        lib.attn_decode_splitkv.argtypes = [P, i32, vp, ctypes.c_size_t, vp]
        lib.attn_decode_splitkv.restype = i32
        lib.attn_decode_fused_workspace_bytes.argtypes = [i64, i64, i64, i64, i32]
        lib.attn_decode_fused_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_decode_splitkv_fused.argtypes = [P, i32, vp, ctypes.c_size_t, vp]
        lib.attn_decode_splitkv_fused.restype = i32
        lib.attn_decode_splitkv_noalloc.argtypes = [P, i32, vp]
        lib.attn_decode_splitkv_noalloc.restype = i32
        lib.attn_merge_states.argtypes = [vp, i64, i64, i32, i64, i32, vp,
                                          ctypes.POINTER(ctypes.c_int64), vp, vp]
        lib.attn_merge_states.restype = i32
        lib.attn_fwd_partial.argtypes = [P, i64, i64, vp, vp]
        lib.attn_fwd_partial.restype = i32
        lib.attn_merge_states_rows.argtypes = [vp, i64, i64, i64, i32, i64, i64, i64, i32, vp,
                                               ctypes.POINTER(ctypes.c_int64), vp, vp]
        lib.attn_merge_states_rows.restype = i32
        lib.attn_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64]
        lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.attn_bwd.argtypes = [ctypes.POINTER(BwdParams), vp, ctypes.c_size_t, vp]
        lib.attn_bwd.restype = i32
        lib.attn_last_error.argtypes = []
        lib.attn_last_error.restype = ctypes.c_char_p
        lib.attn_device_error_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        lib.attn_device_error_flags.restype = i32
        lib.attn_version.argtypes = []
        lib.attn_version.restype = i32
        _lib = lib
        return lib


def last_error() -> str:
    return load().attn_last_error().decode()


def _check(st):
    if st != Status.OK:
        raise AttnError(st, last_error())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.float32 or torch.bfloat16")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _bnhd_strides(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, N, H, d], got {tuple(t.shape)}")
    if t.shape[3] > 1 and t.stride(3) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("every tensor must be on a CUDA device (there is no CPU path)")


def make_params(q, k, v, o, lse=None, bias=None, kv_lens=None, causal=False, scale=None,
                block_k=0, dropout_mask=None, dropout_p=0.0, dropout_seed=None, dropout_offset=0) -> Params:
    """Fill an attn_fwd_params_t from tensors (no computation)."""
    _require_cuda(q, k, v, o, lse, bias, kv_lens, dropout_mask)
    B, Nq, H, dk = q.shape
    Nk, dv = k.shape[1], v.shape[3]
    if k.shape != (B, Nk, H, dk) or v.shape != (B, Nk, H, dv) or o.shape != (B, Nq, H, dv):
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} "
                         f"v{tuple(v.shape)} o{tuple(o.shape)}")
    if not (q.dtype == k.dtype == v.dtype == o.dtype):
        raise TypeError("q, k, v and o must share one dtype")
    p = Params()
    p.dtype = _dtype_code(q)
    p.causal = 1 if causal else 0
    p.B, p.H, p.Nq, p.Nk, p.dk, p.dv = B, H, Nq, Nk, dk, dv
    p.q, p.k, p.v, p.o = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
    p.q_stride = _bnhd_strides(q, "q")
    p.k_stride = _bnhd_strides(k, "k")
    p.v_stride = _bnhd_strides(v, "v")
    p.o_stride = _bnhd_strides(o, "o")
    if lse is not None:
        if lse.dtype != torch.float32 or lse.shape != (B, H, Nq) or not lse.is_contiguous():
            raise ValueError("lse must be contiguous float32 [B, H, Nq]")
        p.lse = lse.data_ptr()
    if bias is not None:
        if bias.dtype != torch.float32 or bias.dim() != 4:
            raise ValueError("bias must be float32 [B, H, Nq, Nk] (broadcast dims allowed)")
        bb = bias.expand(B, H, Nq, Nk)
        if Nk > 1 and bb.stride(3) != 1:
            raise ValueError("bias: the key dimension must be contiguous")
        p.bias = bb.data_ptr()
        p.bias_stride = (ctypes.c_int64 * 3)(bb.stride(0), bb.stride(1), bb.stride(2))
    if kv_lens is not None:
        if kv_lens.dtype != torch.int32 or kv_lens.shape != (B,) or not kv_lens.is_contiguous():
            raise ValueError("kv_lens must be contiguous int32 [B]")
        p.kv_lens = kv_lens.data_ptr()
    p.scale = float(1.0 / math.sqrt(dk) if scale is None else scale)
    p.block_k = int(block_k)
    if dropout_mask is not None:
        nb = 16 * ((Nk + 127) // 128)
        if dropout_mask.dtype != torch.uint8 or dropout_mask.dim() != 4 or dropout_mask.shape[3] < nb:
            raise ValueError(f"dropout_mask must be uint8 [B, H, Nq, >= {nb}] (bit j % 8 of byte j // 8 "
                             "keeps key j; see workloads.pack_keep_mask)")
        mm = dropout_mask.expand(B, H, Nq, dropout_mask.shape[3])
        if mm.stride(3) != 1:
            raise ValueError("dropout_mask: the byte dimension must be contiguous")
        p.dropout_mask = mm.data_ptr()
        p.dropout_mask_stride = (ctypes.c_int64 * 3)(mm.stride(0), mm.stride(1), mm.stride(2))
    p.dropout_p = float(dropout_p)
    if dropout_seed is not None:  # keep decisions drawn in-kernel (Philox4x32-10; see attn.h)
        p.dropout_rng = 1
        p.dropout_seed = int(dropout_seed) & 0xFFFFFFFFFFFFFFFF
        p.dropout_offset = int(dropout_offset) & 0xFFFFFFFFFFFFFFFF
    return p


def attn_fwd(q, k, v, bias=None, kv_lens=None, causal=False, scale=None, block_k=0, out=None,
             lse=None, stream=None, dropout_mask=None, dropout_p=0.0, dropout_seed=None, dropout_offset=0):
    """Exact attention forward; returns (o, lse).  See include/attn.h, attn_fwd.  With a
    dropout_mask (uint8 [B, H, Nq, 16 * ceil(Nk / 128)], workloads.pack_keep_mask) the kept
    weights are scaled by 1 / (1 - dropout_p) and the dropped ones count 0 in o; lse is the
    undropped one.  With dropout_seed (and dropout_offset) instead of a mask the keep
    decisions are drawn in-kernel (Philox4x32-10, p quantised to round(256 p) / 256); the
    backward given the same seed and offset draws the same ones."""
    lib = load()
    B, Nq, H, _ = q.shape
    dv = v.shape[3]
    if out is None:
        out = torch.empty((B, Nq, H, dv), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    p = make_params(q, k, v, out, lse, bias, kv_lens, causal, scale, block_k, dropout_mask, dropout_p,
                    dropout_seed, dropout_offset)
    _check(lib.attn_fwd(ctypes.byref(p), _stream(stream)))
    return out, lse


def attn_fwd_partial(q, k, v, key_offset, nk_total, kv_lens=None, bias=None, causal=False, scale=None,
                     out=None, stream=None):
    """The state (m, l, u) of every query row over one shard of the keys: k, v (and bias) hold
    keys [key_offset, key_offset + k.shape[1]) of sequences of nk_total keys; kv_lens and the
    causal mask are in global positions.  Returns fp32 [B, H, Nq, 2 + dv]."""
    lib = load()
    B, Nq, H, _ = q.shape
    dv = v.shape[3]
    if out is None:
        out = torch.empty((B, H, Nq, 2 + dv), dtype=torch.float32, device=q.device)
    _require_cuda(out)
    if out.shape != (B, H, Nq, 2 + dv) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 [B, H, Nq, 2 + dv] tensor")
    if q.shape[3] != dv:
        raise ValueError("partial states need dk == dv")
    # o is not written (q fills the o fields, which the call ignores)
    p = make_params(q, k, v, q, None, bias, kv_lens, causal, scale, 0)
    p.o = None
    _check(lib.attn_fwd_partial(ctypes.byref(p), int(key_offset), int(nk_total), _ptr(out), _stream(stream)))
    return out


def attn_merge_states_rows(partials, B, H, Nq, dv, num_splits, row_stride=0, split_stride=0, out=None,
                           lse=None, dtype=torch.bfloat16, stream=None):
    """Merge num_splits states per row (state s of row r = (b*H + h)*Nq + i at
    partials[r*row_stride + s*split_stride], in floats; 0, 0: the decode layout) into
    (o [B, Nq, H, dv] of dtype, lse [B, H, Nq])."""
    lib = load()
    _require_cuda(partials)
    if partials.dtype != torch.float32:
        raise TypeError("partials must be float32")
    if out is None:
        out = torch.empty((B, Nq, H, dv), dtype=dtype, device=partials.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=partials.device)
    os_ = (ctypes.c_int64 * 3)(out.stride(0), out.stride(1), out.stride(2))
    _check(lib.attn_merge_states_rows(_ptr(partials), int(B), int(H), int(Nq), int(num_splits), int(dv),
                                      int(row_stride), int(split_stride), _dtype_code(out), _ptr(out), os_,
                                      _ptr(lse), _stream(stream)))
    return out, lse


def decode_workspace_bytes(B, H, dv, num_splits, Nq=1) -> int:
    return int(load().attn_decode_workspace_bytes_rows(B, H, Nq, dv, num_splits))


def attn_decode_splitkv(q, k, v, kv_lens=None, num_splits=16, bias=None, scale=None,
                        workspace=None, out=None, lse=None, stream=None, causal=False):
    """Split-KV decode (q [B, Nq, H, d], 1 <= Nq <= 8); returns (o, lse, workspace).

    k, v are [B, L, H, d]-indexed views (a [B, H, L, d] cache passes as
    ``cache.permute(0, 2, 1, 3)``).  causal applies the bottom-right mask (row i sees keys
    j <= i + kv_len - Nq).  The workspace holds the partial states
    [B, H, Nq, num_splits, 2 + dv] (m, l, u) after the call."""
    lib = load()
    B, Nq, H, _ = q.shape
    dv = v.shape[3]
    if out is None:
        out = torch.empty((B, Nq, H, dv), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    need = decode_workspace_bytes(B, H, dv, num_splits, Nq)
    if workspace is None:
        workspace = torch.empty((max(need, 16) + 3) // 4, dtype=torch.float32, device=q.device)
    _require_cuda(workspace)
    p = make_params(q, k, v, out, lse, bias, kv_lens, causal, scale, 0)
    _check(lib.attn_decode_splitkv(ctypes.byref(p), int(num_splits), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse, workspace


def decode_fused_workspace_bytes(B, H, dv, num_splits, Nq=1) -> int:
    return int(load().attn_decode_fused_workspace_bytes(B, H, Nq, dv, num_splits))


def attn_decode_splitkv_fused(q, k, v, kv_lens=None, num_splits=16, bias=None, scale=None,
                              workspace=None, out=None, lse=None, stream=None, causal=False):
    """Split-KV decode with the merge done by the split kernel (one launch); returns
    (o, lse, workspace).  The workspace holds the partial states, then one counter per
    (b, h); its contents on entry do not matter, so the returned workspace can be passed to
    later calls of any shape that fits."""
    lib = load()
    B, Nq, H, _ = q.shape
    dv = v.shape[3]
    if out is None:
        out = torch.empty((B, Nq, H, dv), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    need = decode_fused_workspace_bytes(B, H, dv, num_splits, Nq)
    if workspace is None:
        workspace = torch.empty((max(need, 16) + 3) // 4, dtype=torch.float32, device=q.device)
    _require_cuda(workspace)
    p = make_params(q, k, v, out, lse, bias, kv_lens, causal, scale, 0)
    _check(lib.attn_decode_splitkv_fused(ctypes.byref(p), int(num_splits), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse, workspace


def attn_decode_splitkv_noalloc(q, k, v, kv_lens=None, num_splits=16, bias=None, scale=None,
                                out=None, lse=None, stream=None, causal=False):
    """Split-KV decode that allocates no device memory in the library: for callers that
    cannot allocate while decoding.  The partial states go to a 32 MiB device array built
    into the library (shared by every call: order calls on one stream).  The first call from a
    CUDA context looks up that array's address.  Returns (o, lse); o and lse are allocated here
    only when not passed in."""
    lib = load()
    B, Nq, H, _ = q.shape
    dv = v.shape[3]
    if out is None:
        out = torch.empty((B, Nq, H, dv), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    p = make_params(q, k, v, out, lse, bias, kv_lens, causal, scale, 0)
    _check(lib.attn_decode_splitkv_noalloc(ctypes.byref(p), int(num_splits), _stream(stream)))
    return out, lse


def bwd_workspace_bytes(B, H, Nq, dk) -> int:
    return int(load().attn_bwd_workspace_bytes(B, H, Nq, dk))


def attn_bwd(q, k, v, o, lse, dout, bias=None, kv_lens=None, causal=False, scale=None,
             dq=None, dk=None, dv=None, workspace=None, stream=None, dropout_mask=None, dropout_p=0.0,
             dropout_seed=None, dropout_offset=0):
    """Gradients (dq, dk, dv) of a loss through o = attn_fwd(q, k, v, ...), given dout = dL/do
    and the forward's o and lse (bfloat16, dk == dv in {64, 128}).  The mask, bias, kv_lens,
    causal and dropout settings must be the forward's (dropout: without a bias);
    the bias gets no gradient."""
    lib = load()
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    if dout.shape != o.shape or dout.dtype != q.dtype:
        raise ValueError("dout must have o's shape and dtype")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_bytes(B, H, Nq, d)
    if workspace is None:
        workspace = torch.empty((max(need, 16) + 3) // 4, dtype=torch.float32, device=q.device)
    _require_cuda(dout, dq, dk, dv, workspace)
    p = BwdParams()
    p.fwd = make_params(q, k, v, o, lse, bias, kv_lens, causal, scale, 0, dropout_mask, dropout_p, dropout_seed,
                        dropout_offset)
    p.dout, p.dout_stride = dout.data_ptr(), _bnhd_strides(dout, "dout")
    p.dq, p.dq_stride = dq.data_ptr(), _bnhd_strides(dq, "dq")
    p.dk, p.dk_stride = dk.data_ptr(), _bnhd_strides(dk, "dk")
    p.dv, p.dv_stride = dv.data_ptr(), _bnhd_strides(dv, "dv")
    _check(lib.attn_bwd(ctypes.byref(p), _ptr(workspace), workspace.numel() * workspace.element_size(),
                        _stream(stream)))
    return dq, dk, dv


def attn_merge_states(partials, out_dtype=torch.bfloat16, out=None, lse=None, stream=None):
    """Merge partial states [B, H, S, 2 + dv] (float32, contiguous) into (o [B, 1, H, dv],
    lse [B, H, 1])."""
    lib = load()
    _require_cuda(partials)
    if partials.dtype != torch.float32 or partials.dim() != 4 or not partials.is_contiguous():
        raise ValueError("partials must be contiguous float32 [B, H, S, 2 + dv]")
    B, H, S, w = partials.shape
    dv = w - 2
    if out is None:
        out = torch.empty((B, 1, H, dv), dtype=out_dtype, device=partials.device)
    if lse is None:
        lse = torch.empty((B, H, 1), dtype=torch.float32, device=partials.device)
    _require_cuda(out, lse)
    ost = (ctypes.c_int64 * 3)(out.stride(0), out.stride(1), out.stride(2))
    _check(lib.attn_merge_states(_ptr(partials), B, H, S, dv, _dtype_code(out), _ptr(out), ost,
                                 _ptr(lse), _stream(stream)))
    return out, lse


def device_error_flags(clear=True) -> int:
    """Device error word (bit 0: a bounded wait gave up; bit 1: kv_lens clamped)."""
    v = ctypes.c_uint32(0)
    _check(load().attn_device_error_flags(ctypes.byref(v), 1 if clear else 0))
    return int(v.value)
