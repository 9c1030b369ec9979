"""The allocation-free decode entry point against the workspace one.

attn_decode_splitkv_noalloc is for callers that cannot allocate device memory while they
decode (a framework whose allocator owns the device memory, a plugin given only its input and
output buffers, a latency-bound loop where cudaMalloc would synchronise the device).  It keeps
the partial states in a device array built into the library and runs the same kernels as
attn_decode_splitkv, so its outputs must equal that entry point's bit for bit; one case is
also compared with the oracle directly.  This file is collected last so that a run stopping
at its first failure has already run every other test; it also passes when run alone in a
fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL, cpu32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def call_noalloc(lib, a, num_splits):
    """Through the C ABI: returns (o, lse) written by attn_decode_splitkv_noalloc."""
    o = torch.full((a.B, a.Nq, a.H, a.dv), float("nan"), dtype=a.q.dtype, device=DEV)
    lse = torch.full((a.B, a.H, a.Nq), float("nan"), dtype=torch.float32, device=DEV)
    p = ofa.make_params(a.q, a.k, a.v, o, lse, None, a.kv_lens, a.causal, a.scale, 0)
    st = lib.attn_decode_splitkv_noalloc(ctypes.byref(p), num_splits,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ofa.Status.OK, ofa.last_error()
    return o, lse


def call_workspace(a, num_splits):
    o, lse, _ = ofa.attn_decode_splitkv(a.q, a.k, a.v, kv_lens=a.kv_lens, num_splits=num_splits,
                                        scale=a.scale, causal=a.causal)
    return o, lse


def test_noalloc_equals_workspace_entry_point_twice_in_a_row():
    lib = ofa.load()
    # different problems back to back (one row, then four causal rows per sequence): the
    # shared scratch must not carry anything from one call into the next
    cases = [wl.decode(DEV, seed=41, B=6, H=4, L=1500, d=128, num_splits=16,
                       lens=[1500, 1, 0, 777, 1024, 9]),
             wl.decode(DEV, seed=42, B=3, H=8, L=900, d=64, num_splits=7, lens=[5, 900, 450],
                       nq=4, causal=True),
             wl.decode(DEV, seed=41, B=6, H=4, L=1500, d=128, num_splits=16,
                       lens=[1500, 1, 0, 777, 1024, 9])]
    for a in cases:
        o1, l1 = call_noalloc(lib, a, a.num_splits)
        o2, l2 = call_workspace(a, a.num_splits)
        torch.cuda.synchronize()
        assert ofa.device_error_flags() & 1 == 0
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)), a.name
        assert torch.equal(l1.view(torch.int32), l2.view(torch.int32)), a.name


def test_noalloc_matches_oracle():
    lib = ofa.load()
    a = wl.decode(DEV, seed=44, B=5, H=3, L=700, d=128, num_splits=16, lens=[700, 1, 0, 333, 64],
                  nq=4, causal=True)
    o, lse = call_noalloc(lib, a, a.num_splits)
    torch.cuda.synchronize()
    o_ref, l_ref, _ = oracle.attn_fwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), kv_lens=a.kv_lens.cpu(),
                                      causal=True, scale=a.scale)
    tol = TOL[torch.bfloat16]
    og = o.float().cpu().numpy()
    lg = lse.cpu().numpy()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.all(o.view(torch.int16).cpu().numpy().transpose(0, 2, 1, 3)[~fin] == 0)
    assert np.max(np.abs(og - o_ref)) <= tol["o"]
    assert np.max(np.abs(lg[fin] - l_ref[fin])) <= tol["lse"]


def test_noalloc_checks_arguments_before_its_size():
    lib = ofa.load()
    a = wl.decode(DEV, seed=43, B=64, H=32, L=64, d=128, num_splits=16)
    o = torch.empty((a.B, 1, a.H, a.dv), dtype=a.q.dtype, device=DEV)
    lse = torch.empty((a.B, a.H, 1), dtype=torch.float32, device=DEV)
    p = ofa.make_params(a.q, a.k, a.v, o, lse, None, a.kv_lens, False, a.scale, 0)
    # 64 * 32 * 256 splits * 130 floats * 4 bytes = 272 MB > 32 MiB
    assert lib.attn_decode_splitkv_noalloc(ctypes.byref(p), 256, None) == ofa.Status.WORKSPACE
    assert "scratch" in ofa.last_error()
    # a bad argument is reported as such, even where the problem would not fit either
    assert lib.attn_decode_splitkv_noalloc(ctypes.byref(p), 257, None) == ofa.Status.INVALID_ARG
    assert lib.attn_decode_splitkv_noalloc(ctypes.byref(p), 0, None) == ofa.Status.INVALID_ARG
    p.Nq = 9
    assert lib.attn_decode_splitkv_noalloc(ctypes.byref(p), 16, None) == ofa.Status.INVALID_ARG
