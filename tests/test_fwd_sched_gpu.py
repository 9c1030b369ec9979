"""GPU parity of attn_fwd where the bf16 kernels schedule work: the two-tile kernel is
persistent (one CTA per SM walks a fixed list of 256-row items, several per CTA), and both
kernels must give the same rows whatever stream, graph or item order they run in.

Every case compares with the float64 oracle (sampled rows where the problem is large):
|o| within 2e-2 and |lse| within 1e-2, empty rows exactly +0.0 / -inf.
"""
import math

import numpy as np
import pytest
import torch

import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import compare, compare_rows, empty_rows, gather_rows, oracle_full, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(a, stream=None):
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal,
                          scale=a.scale, stream=stream)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0, "a kernel gave up a bounded wait"
    return o, lse


def check_sampled(a, o, lse, what, n_per_head=6, seed=0):
    rows = sample_rows(a, n_per_head=n_per_head, seed=seed)
    o_s, l_s = gather_rows(o, lse, rows, a.H, a.Nq)
    o_ref, l_ref, _ = oracle_full(a, rows=rows)
    compare_rows(o_s, l_s, o_ref, l_ref, torch.bfloat16, what=what)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_items_outnumber_sms(causal):
    # 2 x 48 heads x 4 items of 256 rows: every CTA of the persistent kernel walks several
    # items, so barrier phases and buffers carry over between items
    a = wl.make_prefill(2, 48, 1024, 1024, 128, 128, torch.bfloat16, causal=causal, seed=31,
                        device=DEV)
    o, lse = run(a)
    check_sampled(a, o, lse, f"many items causal={causal}")


def test_bf16_items_of_uneven_length_padded():
    # per-sequence key lengths give items of 0 to 8 key tiles in one launch
    lens = [1024, 0, 37, 511, 129, 900, 256, 1]
    a = wl.make_prefill(8, 20, 512, 1024, 128, 128, torch.bfloat16, causal=False, kv_lens=lens,
                        seed=32, device=DEV)
    o, lse = run(a)
    check_sampled(a, o, lse, "uneven items")


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128)])
def test_bf16_causal_keys_shorter_than_queries(dk, dv):
    # bottom-right causal with kv_len < Nq: leading query tiles see no key at all, and items
    # where tile A is empty while tile B is not
    a = wl.make_prefill(3, 2, 700, 700, dk, dv, torch.bfloat16, causal=True,
                        kv_lens=[100, 700, 0], seed=33, device=DEV)
    o, lse = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, empty=empty_rows(a), what=f"short keys {dk}/{dv}")


def test_bf16_two_streams_at_once():
    # two problems queued on two streams without synchronising in between
    a1 = wl.make_prefill(2, 8, 1024, 1024, 128, 128, torch.bfloat16, causal=True, seed=34, device=DEV)
    a2 = wl.make_prefill(4, 3, 700, 900, 192, 128, torch.bfloat16, causal=False, seed=35, device=DEV)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for _ in range(3):
        for a, s in ((a1, s1), (a2, s2)):
            with torch.cuda.stream(s):
                outs.append((a, ofa.attn_fwd(a.q, a.k, a.v, causal=a.causal, scale=a.scale, stream=s)))
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    for n, (a, (o, lse)) in enumerate(outs):
        check_sampled(a, o, lse, f"stream launch {n}", n_per_head=4, seed=n)


def test_bf16_cuda_graph_replay():
    # attn_fwd captured once into a CUDA graph and replayed on new inputs copied into the
    # captured buffers
    a = wl.make_prefill(2, 4, 600, 600, 128, 128, torch.bfloat16, causal=True, seed=36, device=DEV)
    q, k, v = a.q.clone(), a.k.clone(), a.v.clone()
    o = torch.empty((a.B, a.Nq, a.H, a.dv), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((a.B, a.H, a.Nq), dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ofa.attn_fwd(q, k, v, causal=True, scale=a.scale, out=o, lse=lse, stream=s)  # warm-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ofa.attn_fwd(q, k, v, causal=True, scale=a.scale, out=o, lse=lse, stream=s)
    for seed in (37, 38):
        b = wl.make_prefill(2, 4, 600, 600, 128, 128, torch.bfloat16, causal=True, seed=seed,
                            device=DEV)
        q.copy_(b.q)
        k.copy_(b.k)
        v.copy_(b.v)
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert ofa.device_error_flags() & 1 == 0
        o_ref, l_ref, _ = oracle_full(b)
        compare(o, lse, o_ref, l_ref, torch.bfloat16, what=f"graph replay seed {seed}")


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_bias_in_the_two_tile_kernel(dk, dv, causal):
    # fp32 bias with explicit -inf masks and padded sequences, several items per CTA; with one
    # visible key in the last sequence some rows are emptied by the bias alone, and the oracle's
    # -inf lse marks them (compare checks those rows are exactly +0.0 / -inf)
    a = wl.make_prefill(3, 6, 600, 650, dk, dv, torch.bfloat16, causal=causal, bias=True,
                        kv_lens=[650, 333, 1], seed=39, device=DEV, bias_mask_p=0.05)
    o, lse = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    assert np.all(np.isinf(l_ref)[empty_rows(a)])  # every row the mask empties is among them
    compare(o, lse, o_ref, l_ref, torch.bfloat16, what=f"bias {dk}/{dv} causal={causal}")


@pytest.mark.parametrize("dk", [128, 192])
def test_bf16_broadcast_bias_over_batch_and_heads(dk):
    # one [Nq, Nk] bias for every (b, h): batch and head strides 0 (with dk = 192 the bias
    # cannot go through a tensor map and is read with plain loads)
    a = wl.make_prefill(2, 4, 400, 400, dk, 128, torch.bfloat16, causal=False, seed=40,
                        device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(41)
    base = torch.randn((1, 1, 400, 400), generator=g, device=DEV, dtype=torch.float32)
    a.bias = base.expand(a.B, a.H, 400, 400)
    o, lse = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, what=f"broadcast bias dk={dk}")
