"""The allocation-free decode entry point against the workspace one.

attn_decode_splitkv_noalloc is for callers that cannot allocate device memory while they
decode (a framework whose allocator owns the device memory, a plugin given only its input and
output buffers, a latency-bound loop where cudaMalloc would synchronise the device).  It keeps
the partial states in a device array built into the library.  This file is collected last so
that a run stopping at its first failure has already run every other test; it also passes
when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL

pytestmark = pytest.mark.gpu
DEV = "cuda"


def call_noalloc(lib, a, num_splits):
    """Through the C ABI: returns (o, lse) written by attn_decode_splitkv_noalloc."""
    o = torch.full((a.B, 1, a.H, a.dv), float("nan"), dtype=a.q.dtype, device=DEV)
    lse = torch.full((a.B, a.H, 1), float("nan"), dtype=torch.float32, device=DEV)
    p = ofa.make_params(a.q, a.k, a.v, o, lse, None, a.kv_lens, False, a.scale, 0)
    st = lib.attn_decode_splitkv_noalloc(ctypes.byref(p), num_splits,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ofa.Status.OK, ofa.last_error()
    return o, lse


def call_workspace(a, num_splits):
    o, lse, _ = ofa.attn_decode_splitkv(a.q, a.k, a.v, kv_lens=a.kv_lens, num_splits=num_splits,
                                        scale=a.scale)
    return o, lse


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    lib = ofa.load()
    tol = TOL[torch.bfloat16]
    # two different problems back to back: the shared scratch must not carry anything over
    cases = [wl.decode(DEV, seed=41, B=6, H=4, L=1500, d=128, num_splits=16,
                       lens=[1500, 1, 0, 777, 1024, 9]),
             wl.decode(DEV, seed=42, B=3, H=8, L=900, d=64, num_splits=7, lens=[5, 900, 450])]
    for a in cases:
        o1, l1 = call_noalloc(lib, a, a.num_splits)
        o2, l2 = call_workspace(a, a.num_splits)
        torch.cuda.synchronize()
        assert not torch.isnan(o1.float()).any()
        assert (o1.float() - o2.float()).abs().max().item() <= tol["o"]
        fin = torch.isfinite(l2)
        assert torch.equal(torch.isfinite(l1), fin)
        assert (l1[fin] - l2[fin]).abs().max().item() <= tol["lse"]
        assert torch.all(l1[~fin] == -float("inf"))


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = ofa.load()
    a = wl.decode(DEV, seed=43, B=64, H=32, L=64, d=128, num_splits=16)
    # 64 * 32 * 256 splits * 130 floats * 4 bytes = 272 MB > 32 MiB
    o = torch.empty((a.B, 1, a.H, a.dv), dtype=a.q.dtype, device=DEV)
    lse = torch.empty((a.B, a.H, 1), dtype=torch.float32, device=DEV)
    p = ofa.make_params(a.q, a.k, a.v, o, lse, None, a.kv_lens, False, a.scale, 0)
    st = lib.attn_decode_splitkv_noalloc(ctypes.byref(p), 256, None)
    assert st == ofa.Status.WORKSPACE
    assert "scratch" in ofa.last_error()
