"""GPU parity of the fused split-KV decode (the merge done by the split kernel's last CTA of
each (b, h)) against the oracle and against the two-launch decode.

"How Does FlashAttention Preserve Global Softmax Across Tiles?", section 8 (split-KV decode,
its partial round trip and merge launch) and section 3 (the merge).  The fused call runs the
same split kernel and the same merge arithmetic as attn_decode_splitkv, so its outputs must
equal that call's bit for bit.  Its per-(b, h) counters carry each call's own tag, so the
workspace's contents on entry must not matter: the tests fill it with garbage first."""
import numpy as np
import pytest
import torch

import oracle
import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL, cpu32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def garbage_workspace(nbytes, seed):
    """A fused-decode workspace holding arbitrary bits (its contents on entry must not matter)."""
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    ws = torch.empty((nbytes + 3) // 4 + 4, dtype=torch.int32, device=DEV)
    ws.random_(-2 ** 31, 2 ** 31 - 1, generator=g)
    return ws.view(torch.float32)


def oracle_check(a, o, lse):
    o_ref, l_ref, _ = oracle.attn_fwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), bias=cpu32(a.bias),
                                      kv_lens=a.kv_lens.cpu(), causal=a.causal, scale=a.scale)
    og, lg = o.float().cpu().numpy(), lse.cpu().numpy()
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    bits = o.view(torch.int16).cpu().numpy().transpose(0, 2, 1, 3)
    assert np.all(bits[~fin] == 0)  # empty rows: +0.0 exactly
    assert np.max(np.abs(og - o_ref)) <= TOL[torch.bfloat16]["o"]
    assert np.max(np.abs(lg[fin] - l_ref[fin])) <= TOL[torch.bfloat16]["lse"]


@pytest.mark.parametrize("num_splits", [1, 2, 16, 37])
@pytest.mark.parametrize("nq,causal", [(1, False), (4, True)])
def test_fused_equals_two_launch_decode_and_matches_oracle(num_splits, nq, causal):
    # keys past each length hold NaN (the workload's poison): nothing may read them
    a = wl.decode(DEV, seed=50 + num_splits, B=5, H=4, L=1200, d=128, num_splits=num_splits,
                  lens=[1200, 1, 0, 500, 37], nq=nq, causal=causal)
    ws = garbage_workspace(ofa.decode_fused_workspace_bytes(a.B, a.H, a.dv, num_splits, nq), num_splits)
    o1, l1, _ = ofa.attn_decode_splitkv_fused(a.q, a.k, a.v, kv_lens=a.kv_lens, num_splits=num_splits,
                                              scale=a.scale, causal=causal, workspace=ws)
    o2, l2, _ = ofa.attn_decode_splitkv(a.q, a.k, a.v, kv_lens=a.kv_lens, num_splits=num_splits,
                                        scale=a.scale, causal=causal)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    oracle_check(a, o1, l1)


def test_fused_reuses_its_workspace_across_calls_of_other_lengths():
    a = wl.decode(DEV, seed=61, B=6, H=3, L=900, d=64, num_splits=16, lens=[900, 3, 450, 0, 77, 899])
    b = wl.decode(DEV, seed=62, B=6, H=3, L=900, d=64, num_splits=7, lens=[1, 900, 300, 64, 0, 512], nq=4,
                  causal=True)
    nbytes = max(ofa.decode_fused_workspace_bytes(a.B, a.H, a.dv, 16, 1),
                 ofa.decode_fused_workspace_bytes(b.B, b.H, b.dv, 7, 4))
    ws = garbage_workspace(nbytes, 7)
    o, lse, _ = ofa.attn_decode_splitkv_fused(a.q, a.k, a.v, kv_lens=a.kv_lens, num_splits=16, scale=a.scale,
                                              workspace=ws)
    torch.cuda.synchronize()
    oracle_check(a, o, lse)
    # the same workspace again: other lengths, fewer splits, four causal rows (its counters now
    # sit where the first call left partial states), then the first problem once more
    for c, ns, causal in ((b, 7, True), (a, 16, False)):
        o, lse, ws2 = ofa.attn_decode_splitkv_fused(c.q, c.k, c.v, kv_lens=c.kv_lens, num_splits=ns,
                                                    scale=c.scale, causal=causal, workspace=ws)
        torch.cuda.synchronize()
        assert ws2 is ws
        assert ofa.device_error_flags() & 1 == 0
        oracle_check(c, o, lse)


def test_fused_full_size_decode_sampled_heads():
    a = wl.decode(DEV)  # B=64, H=32, L=8192, 16 splits
    o1, l1, _ = ofa.attn_decode_splitkv_fused(a.q, a.k, a.v, kv_lens=a.kv_lens, num_splits=a.num_splits,
                                              scale=a.scale)
    o2, l2, _ = ofa.attn_decode_splitkv(a.q, a.k, a.v, kv_lens=a.kv_lens, num_splits=a.num_splits,
                                        scale=a.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
