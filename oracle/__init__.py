"""float64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use this package.  The GPU library (``online_softmax_fa2_gb300``) never
imports it and shares no code with it.

``attn_oracle.c`` holds the arithmetic (the plain definition of the operator, row by row,
in float64); this module compiles it with gcc on first use and wraps it with ctypes.
``online_ref`` holds a pure-Python restatement of the online method as a merge of per-key-set
(m, l, u) states over any partition of the keys, used to pin the definition against the
method's own claim that the pieces combine to the whole.

Readings of the pages that the oracle takes (bias not scaled; bottom-right causal aligned
to each sequence's own key length; bias -inf masks; empty row -> o = +0.0, lse = -inf) are
listed in ``attn_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "_attn_oracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: every double operation rounds on its own, the same on x86 and Arm.
GCC_FLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
             "-fvisibility=hidden", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into _attn_oracle.so (if missing or stale); return its path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def bind(path: str):
    """Load an oracle shared object from ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    i64, f64, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_int
    vp = ctypes.c_void_p
    lib.oracle_attn_fwd.argtypes = [i64] * 6 + [vp] * 5 + [i32, f64, vp, i64, vp, vp, i32]
    lib.oracle_attn_fwd.restype = i32
    lib.oracle_attn_probs.argtypes = [i64] * 6 + [vp] * 5 + [i32, f64, vp]
    lib.oracle_attn_probs.restype = i32
    lib.oracle_key_state.argtypes = [i64] * 6 + [vp] * 5 + [i32, f64, i64, i64, vp]
    lib.oracle_key_state.restype = i32
    lib.oracle_merge_states.argtypes = [i64, i64, i64, vp, vp, vp]
    lib.oracle_merge_states.restype = i32
    lib.oracle_attn_bwd.argtypes = [i64] * 6 + [vp] * 5 + [i32, f64, vp, vp, vp, vp, i32]
    lib.oracle_attn_bwd.restype = i32
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
        return _lib


def _f32(x):
    """Contiguous float32 numpy view of x (a numpy array or a CPU torch tensor), or None.

    bfloat16 and float16 widen to float32 exactly, so the oracle sees the rounded inputs.
    """
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").float().contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _kvl(kv_lens):
    if kv_lens is None:
        return None
    if hasattr(kv_lens, "detach"):
        kv_lens = kv_lens.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int32))


def _shapes(q, k, v):
    B, Nq, H, dk = q.shape
    Nk = k.shape[1]
    dv = v.shape[3]
    if k.shape != (B, Nk, H, dk) or v.shape != (B, Nk, H, dv):
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    return B, H, Nq, Nk, dk, dv


def attn_fwd(q, k, v, bias=None, kv_lens=None, causal=False, scale=None, rows=None,
             threads=0, lib=None):
    """Exact attention in float64.

    q [B, Nq, H, dk], k [B, Nk, H, dk], v [B, Nk, H, dv], bias [B, H, Nq, Nk] or None,
    kv_lens [B] or None.  scale defaults to 1/sqrt(dk).
    rows: optional flat row indices (b*H + h)*Nq + i; then O is [n, dv] and lse [n].
    Returns (O float64 [B, Nq, H, dv], lse float64 [B, H, Nq], threads used).
    """
    q, k, v, bias = _f32(q), _f32(k), _f32(v), _f32(bias)
    kvl = _kvl(kv_lens)
    B, H, Nq, Nk, dk, dv = _shapes(q, k, v)
    if bias is not None and bias.shape != (B, H, Nq, Nk):
        raise ValueError(f"bias shape {bias.shape}")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    if rows is not None:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        o = np.empty((rows.size, dv), np.float64)
        lse = np.empty((rows.size,), np.float64)
    else:
        o = np.empty((B, Nq, H, dv), np.float64)
        lse = np.empty((B, H, Nq), np.float64)
    used = (lib or _load()).oracle_attn_fwd(B, H, Nq, Nk, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(bias),
                                   _ptr(kvl), int(bool(causal)), float(scale), _ptr(rows),
                                   0 if rows is None else rows.size, _ptr(o), _ptr(lse),
                                   int(threads))
    if used < 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return o, lse, used


def attn_bwd(q, k, v, dout, bias=None, kv_lens=None, causal=False, scale=None, threads=0,
             lib=None):
    """Gradients of sum(dout * O) in float64: returns (dQ [B, Nq, H, dk], dK [B, Nk, H, dk],
    dV [B, Nk, H, dv], threads used).  dout [B, Nq, H, dv]; other arguments as attn_fwd.  The
    bias is fixed (no gradient); empty rows pass no gradient."""
    q, k, v, bias, dout = _f32(q), _f32(k), _f32(v), _f32(bias), _f32(dout)
    kvl = _kvl(kv_lens)
    B, H, Nq, Nk, dk, dv = _shapes(q, k, v)
    if dout.shape != (B, Nq, H, dv):
        raise ValueError(f"dout shape {dout.shape}")
    if bias is not None and bias.shape != (B, H, Nq, Nk):
        raise ValueError(f"bias shape {bias.shape}")
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    dq = np.empty((B, Nq, H, dk), np.float64)
    dkk = np.empty((B, Nk, H, dk), np.float64)
    dvv = np.empty((B, Nk, H, dv), np.float64)
    used = (lib or _load()).oracle_attn_bwd(B, H, Nq, Nk, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(bias),
                                   _ptr(kvl), int(bool(causal)), float(scale), _ptr(dout), _ptr(dq),
                                   _ptr(dkk), _ptr(dvv), int(threads))
    if used < 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return dq, dkk, dvv, used


def attn_probs(q, k, v, bias=None, kv_lens=None, causal=False, scale=None, lib=None):
    """The weight matrix P [B, H, Nq, Nk] in float64 (small inputs only)."""
    q, k, v, bias = _f32(q), _f32(k), _f32(v), _f32(bias)
    kvl = _kvl(kv_lens)
    B, H, Nq, Nk, dk, dv = _shapes(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    p = np.empty((B, H, Nq, Nk), np.float64)
    rc = (lib or _load()).oracle_attn_probs(B, H, Nq, Nk, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(bias),
                                   _ptr(kvl), int(bool(causal)), float(scale), _ptr(p))
    if rc:
        raise ValueError("oracle_attn_probs rejected its arguments")
    return p


def attn_fwd_dropout(q, k, v, keep, p_drop, bias=None, kv_lens=None, causal=False, scale=None,
                     lib=None):
    """Attention with dropout on the normalised weights, in float64 (small inputs only).

    "How Does FlashAttention Preserve Global Softmax Across Tiles?", section 6, disables
    dropout and adds that with training dropout the backward recomputation must reproduce the
    forward's random mask and scaling.  The reading taken here is inverted dropout of the
    weights: keep [B, H, Nq, Nk] (nonzero = kept) is an input, so forward and backward see
    the same mask; O_i = sum_j keep_ij / (1 - p_drop) * P_ij v_j with P the weights of
    attn_probs (the row's undropped softmax); lse is the undropped log-sum-exp of attn_fwd.
    Returns (O float64 [B, Nq, H, dv], lse float64 [B, H, Nq])."""
    if not 0.0 <= p_drop < 1.0:
        raise ValueError("p_drop must be in [0, 1)")
    P = attn_probs(q, k, v, bias=bias, kv_lens=kv_lens, causal=causal, scale=scale, lib=lib)
    keep = np.asarray(keep.cpu().numpy() if hasattr(keep, "cpu") else keep) != 0
    if keep.shape != P.shape:
        raise ValueError(f"keep shape {keep.shape}, expected {P.shape}")
    w = np.where(keep, P, 0.0) / (1.0 - p_drop)
    # the sum runs over visible keys only: value rows past a sequence's key length are no
    # part of it (they may hold anything), so they are left out, not multiplied by zero
    v64 = _f32(v).astype(np.float64)
    kvl = _kvl(kv_lens)
    if kvl is not None:
        for b in range(v64.shape[0]):
            v64[b, min(max(int(kvl[b]), 0), v64.shape[1]):] = 0.0
    o = np.einsum("bhij,bjhd->bihd", w, v64)
    _, lse, _ = attn_fwd(q, k, v, bias=bias, kv_lens=kv_lens, causal=causal, scale=scale, lib=lib)
    return o, lse


def attn_bwd_dropout(q, k, v, dout, keep, p_drop, bias=None, kv_lens=None, causal=False,
                     scale=None, lib=None):
    """Gradients of sum(dout * O) for attn_fwd_dropout's output, in float64 (small inputs only).

    The chain rule through W = keep / (1 - p_drop) * P (P the undropped weights, O = W V):
    dV = W^T G; the gradient reaching P_ij is keep_ij / (1 - p_drop) * g_i . v_j, and the
    softmax Jacobian turns it into dS_ij = P_ij (keep_ij / (1 - p_drop) * g_i . v_j - c_i) with
    c_i = g_i . o_i; dQ = scale * dS K, dK = scale * dS^T Q ("How Does FlashAttention Preserve
    Global Softmax Across Tiles?", section 7, with the mask its section 6 asks the backward to
    reproduce).  Returns (dQ [B, Nq, H, dk], dK [B, Nk, H, dk], dV [B, Nk, H, dv])."""
    if not 0.0 <= p_drop < 1.0:
        raise ValueError("p_drop must be in [0, 1)")
    q64, k64, v64 = (_f32(t).astype(np.float64) for t in (q, k, v))
    g64 = _f32(dout).astype(np.float64)
    B, H, Nq, Nk, dk, dv = _shapes(_f32(q), _f32(k), _f32(v))
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    kvl = _kvl(kv_lens)
    if kvl is not None:  # rows past a sequence's key length are no part of any sum
        for b in range(B):
            n = min(max(int(kvl[b]), 0), Nk)
            k64[b, n:] = 0.0
            v64[b, n:] = 0.0
    P = attn_probs(q, k, v, bias=bias, kv_lens=kv_lens, causal=causal, scale=scale, lib=lib)
    keep = np.asarray(keep.cpu().numpy() if hasattr(keep, "cpu") else keep) != 0
    zs = np.where(keep, 1.0 / (1.0 - p_drop), 0.0)
    W = P * zs
    O = np.einsum("bhij,bjhd->bihd", W, v64)
    dV = np.einsum("bhij,bihd->bjhd", W, g64)
    GV = np.einsum("bihd,bjhd->bhij", g64, v64)
    c = np.einsum("bihd,bihd->bhi", g64, O)
    dS = P * (zs * GV - c[..., None])
    dQ = scale * np.einsum("bhij,bjhd->bihd", dS, k64)
    dK = scale * np.einsum("bhij,bihd->bjhd", dS, q64)
    return dQ, dK, dV


def key_state(q, k, v, j0, j1, bias=None, kv_lens=None, causal=False, scale=None,
              lib=None):
    """State (m, l, u) of every row over the visible keys in [j0, j1): [B, H, Nq, 2 + dv]."""
    q, k, v, bias = _f32(q), _f32(k), _f32(v), _f32(bias)
    kvl = _kvl(kv_lens)
    B, H, Nq, Nk, dk, dv = _shapes(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(dk)
    st = np.empty((B, H, Nq, 2 + dv), np.float64)
    rc = (lib or _load()).oracle_key_state(B, H, Nq, Nk, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(bias),
                                  _ptr(kvl), int(bool(causal)), float(scale), int(j0), int(j1),
                                  _ptr(st))
    if rc:
        raise ValueError("oracle_key_state rejected its arguments")
    return st


def merge_states(states, lib=None):
    """Merge states [..., S, 2 + dv] along S and finalise; returns (O [..., dv], lse [...])."""
    st = np.ascontiguousarray(np.asarray(states, dtype=np.float64))
    lead = st.shape[:-2]
    S, w = st.shape[-2], st.shape[-1]
    dv = w - 2
    n = int(np.prod(lead)) if lead else 1
    o = np.empty((n, dv), np.float64)
    lse = np.empty((n,), np.float64)
    rc = (lib or _load()).oracle_merge_states(n, S, dv, _ptr(st), _ptr(o), _ptr(lse))
    if rc:
        raise ValueError("oracle_merge_states rejected its arguments")
    return o.reshape(*lead, dv), lse.reshape(lead)


def max_threads() -> int:
    return int(_load().oracle_max_threads())
