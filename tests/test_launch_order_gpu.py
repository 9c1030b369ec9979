"""Chained calls on one stream: every kernel of the library is launched as a programmatic
dependent of the kernel before it, so its CTAs may start while that kernel drains; each
waits (griddepcontrol.wait) before its first global access.  Here each call reads the output
of the call before it with no synchronisation in between, and the chain must give the same
bits as the same calls with the device synchronised after each one."""
import pytest
import torch

import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def chain(a, b, sync):
    """o1 = attn(q, k, v) (two-tile kernel); o2 = attn(q2, k2, o1) with dk = 192 (one-tile
    kernel, o1 as its values); o3 = attn(o2, k, v) (o2 as queries); a decode of o3's last row
    against the cache (split and merge kernels); a backward through the first call."""
    def s():
        if sync:
            torch.cuda.synchronize()
    o1, l1 = ofa.attn_fwd(a.q, a.k, a.v, causal=True, scale=a.scale)
    s()
    o2, l2 = ofa.attn_fwd(b.q, b.k, o1, causal=False, scale=b.scale)
    s()
    o3, l3 = ofa.attn_fwd(o2, a.k, a.v, causal=True, scale=a.scale)
    s()
    od, ld, _ = ofa.attn_decode_splitkv(o3[:, -1:].contiguous(), a.k, a.v, num_splits=5, scale=a.scale)
    s()
    g = o3.clone()
    s()
    dq, dk, dv = ofa.attn_bwd(a.q, a.k, a.v, o1, l1, g, causal=True, scale=a.scale)
    torch.cuda.synchronize()
    return [o1, l1, o2, l2, o3, l3, od, ld, dk, dv]


def test_chained_calls_read_their_predecessors_outputs():
    a = wl.make_prefill(2, 4, 640, 640, 128, 128, torch.bfloat16, causal=True, seed=71, device=DEV)
    b = wl.make_prefill(2, 4, 640, 640, 192, 128, torch.bfloat16, causal=False, seed=72, device=DEV)
    free = chain(a, b, sync=False)
    assert ofa.device_error_flags() & 1 == 0
    ordered = chain(a, b, sync=True)
    for x, y in zip(free, ordered):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)
