"""GPU parity of attention over key shards: attn_fwd_partial on every shard of the key axis,
then attn_merge_states_rows on the gathered states, against attn_fwd and the oracle.

The shards stand in for the ranks of sequence parallelism (each would hold one); here they run
one after another on one GPU.  Each shard's states are also checked against the oracle's
key_state over the same keys ("How Does FlashAttention Preserve Global Softmax Across
Tiles?", section 3: the state of a key subset; sections 3-4: disjoint states merge to the
whole).  Empty rows are exact: (-inf, 0, 0) in a state, +0.0 and -inf after the merge."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL, compare, cpu32, empty_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def shard_states(a, cuts):
    """States of every shard [cuts[r], cuts[r+1]), stacked [R, B, H, Nq, 2 + dv] as a gather
    would leave them."""
    parts = []
    for c0, c1 in zip(cuts[:-1], cuts[1:]):
        b = None if a.bias is None else a.bias[..., c0:c1]
        parts.append(ofa.attn_fwd_partial(a.q, a.k[:, c0:c1], a.v[:, c0:c1], c0, a.Nk, kv_lens=a.kv_lens,
                                          bias=b, causal=a.causal, scale=a.scale))
    return torch.stack(parts)


def merge(a, allp):
    R = allp.shape[0]
    return ofa.attn_merge_states_rows(allp, a.B, a.H, a.Nq, a.dv, R, row_stride=2 + a.dv,
                                      split_stride=allp[0].numel())


def check_states(a, allp, cuts):
    """Each shard's states against the oracle's key_state over the same keys: m + ln l and u / l
    within the bf16 tolerances, and empty states exactly (-inf, 0, 0)."""
    kvl = None if a.kv_lens is None else a.kv_lens.cpu()
    for r, (c0, c1) in enumerate(zip(cuts[:-1], cuts[1:])):
        ref = oracle.key_state(cpu32(a.q), cpu32(a.k), cpu32(a.v), c0, c1, bias=cpu32(a.bias), kv_lens=kvl,
                               causal=a.causal, scale=a.scale)
        got = allp[r].double().cpu().numpy()
        empty = ref[..., 1] == 0
        assert np.array_equal(got[..., 1] == 0, empty), f"shard {r}: empty rows differ"
        assert np.all(got[empty][:, 0] == -np.inf) and np.all(got[empty][:, 1:] == 0), f"shard {r}"
        lse_g = got[~empty][:, 0] + np.log(got[~empty][:, 1])
        lse_r = ref[~empty][:, 0] + np.log(ref[~empty][:, 1])
        assert np.max(np.abs(lse_g - lse_r), initial=0) <= TOL[torch.bfloat16]["lse"], f"shard {r}"
        o_g = got[~empty][:, 2:] / got[~empty][:, 1:2]
        o_r = ref[~empty][:, 2:] / ref[~empty][:, 1:2]
        assert np.max(np.abs(o_g - o_r), initial=0) <= TOL[torch.bfloat16]["o"], f"shard {r}"


@pytest.mark.parametrize("d,causal,cuts_frac", [
    (128, True, [0, 0.4, 1]),
    (128, False, [0, 0.25, 0.5, 1]),
    (64, True, [0, 0.1, 0.6, 1]),
])
def test_shards_merge_to_the_whole_forward(d, causal, cuts_frac):
    a = wl.make_prefill(3, 2, 300, 520, d, d, torch.bfloat16, causal=causal, kv_lens=[520, 130, 0], seed=71,
                        device=DEV)
    cuts = [int(round(f * a.Nk / 8)) * 8 for f in cuts_frac]  # 16-byte aligned shard starts
    allp = shard_states(a, cuts)
    o, lse = merge(a, allp)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    check_states(a, allp, cuts)
    o_ref, l_ref, _ = oracle.attn_fwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), kv_lens=a.kv_lens.cpu(), causal=causal,
                                      scale=a.scale)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, empty=empty_rows(a), what="merged shards")
    # and against the whole-sequence kernel
    o1, l1 = ofa.attn_fwd(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=causal, scale=a.scale)
    torch.cuda.synchronize()
    assert (o.float() - o1.float()).abs().max().item() <= TOL[torch.bfloat16]["o"]


def test_shards_with_bias_and_masked_keys():
    a = wl.make_prefill(2, 2, 200, 384, 128, 128, torch.bfloat16, causal=True, bias=True, kv_lens=[384, 250],
                        seed=72, device=DEV, bias_mask_p=0.1)
    cuts = [0, 128, 200, 384]
    allp = shard_states(a, cuts)
    o, lse = merge(a, allp)
    torch.cuda.synchronize()
    check_states(a, allp, cuts)
    o_ref, l_ref, _ = oracle.attn_fwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), bias=cpu32(a.bias),
                                      kv_lens=a.kv_lens.cpu(), causal=True, scale=a.scale)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, what="merged shards with bias")


def test_one_shard_is_the_forward_and_a_shard_past_the_sequence_is_empty():
    a = wl.make_prefill(2, 3, 260, 256, 128, 128, torch.bfloat16, causal=True, kv_lens=[256, 100], seed=73,
                        device=DEV)
    allp = shard_states(a, [0, a.Nk])
    o, lse = merge(a, allp)
    o1, l1 = ofa.attn_fwd(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=True, scale=a.scale)
    torch.cuda.synchronize()
    assert (o.float() - o1.float()).abs().max().item() <= TOL[torch.bfloat16]["o"]
    fin = torch.isfinite(l1)
    assert torch.equal(torch.isfinite(lse), fin) and torch.all(o.view(torch.int16).permute(0, 2, 1, 3)[~fin] == 0)
    # keys [128, 256) of sequence 1 (100 keys long) hold nothing it can see: empty states
    part = ofa.attn_fwd_partial(a.q, a.k[:, 128:], a.v[:, 128:], 128, a.Nk, kv_lens=a.kv_lens, causal=True,
                                scale=a.scale)
    torch.cuda.synchronize()
    p1 = part[1].cpu()
    assert torch.all(p1[..., 0] == -math.inf) and torch.all(p1[..., 1:] == 0)


def test_causal_b4_h16_n2048_d128_two_shards_sampled_heads():
    a = wl.causal_2k(DEV)
    allp = shard_states(a, [0, 1024, 2048])
    o, lse = merge(a, allp)
    o1, l1 = ofa.attn_fwd(a.q, a.k, a.v, causal=True, scale=a.scale)
    torch.cuda.synchronize()
    assert (o.float() - o1.float()).abs().max().item() <= TOL[torch.bfloat16]["o"]
    assert (lse - l1).abs().max().item() <= TOL[torch.bfloat16]["lse"]
    for b, h in ((0, 0), (3, 15)):
        sub = lambda t: cpu32(t[b:b + 1, :, h:h + 1])
        o_ref, l_ref, _ = oracle.attn_fwd(sub(a.q), sub(a.k), sub(a.v), causal=True, scale=a.scale)
        assert np.max(np.abs(o[b:b + 1, :, h:h + 1].float().cpu().numpy() - o_ref)) <= TOL[torch.bfloat16]["o"]
        assert np.max(np.abs(lse[b, h].cpu().numpy() - l_ref[0, 0])) <= TOL[torch.bfloat16]["lse"]


def test_sequence_parallel_attn_on_a_one_rank_nccl_group():
    # the whole path of seqpar.sequence_parallel_attn (partial kernel, NCCL all-gather, merge)
    # on a one-rank group holding every key, on a side stream: it must give attn_fwd's bits
    import socket
    import torch.distributed as dist
    from online_softmax_fa2_gb300 import seqpar

    a = wl.make_prefill(2, 3, 300, 333, 128, 128, torch.bfloat16, causal=True, kv_lens=[333, 100],
                        seed=81, device=DEV)
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        o, lse = seqpar.sequence_parallel_attn(a.q, a.k, a.v, 0, a.Nk, kv_lens=a.kv_lens, causal=True,
                                               scale=a.scale, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    allp = shard_states(a, [0, a.Nk])
    o2, l2 = merge(a, allp)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse, l2)
    o_ref, l_ref, _ = oracle.attn_fwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), kv_lens=a.kv_lens.cpu(), causal=True,
                                      scale=a.scale)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, empty=empty_rows(a), what="seqpar one rank")
