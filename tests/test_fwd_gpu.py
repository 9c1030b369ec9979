"""GPU parity of attn_fwd (float32 SIMT path and bfloat16 tcgen05 path) against the oracle.

Every case calls the library through its C ABI (ctypes) on seeded inputs and compares with
the float64 oracle element by element: bf16 within |o| 2e-2 and |lse| 1e-2, fp32 within
1e-5; empty rows must be +0.0 / -inf exactly.
"""
import math

import numpy as np
import pytest
import torch

import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import (TOL, compare, compare_rows, empty_rows, gather_rows, oracle_full,
                     sample_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(a, block_k=0):
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal,
                          scale=a.scale, block_k=block_k)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0, "a kernel gave up a bounded wait"
    return o, lse


# ------------------------------------------------------------------------ float32 path

@pytest.mark.parametrize("block_k", [16, 32, 64])
def test_fp32_n128_d64_each_tile_size_matches_oracle(block_k):
    a = wl.fp32_small(DEV)
    o, lse = run(a, block_k)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.float32, what=f"fp32 B_k={block_k}")


def test_fp32_tile_sizes_agree_with_each_other():
    a = wl.fp32_small(DEV)
    outs = [run(a, bk) for bk in (16, 32, 64)]
    for o, l in outs[1:]:
        assert (o - outs[0][0]).abs().max().item() <= 1e-5
        assert (l - outs[0][1]).abs().max().item() <= 1e-5


FAMILIES = [  # page-1 section-9 check families (shape Nq/Nk/dk/dv) plus masks
    dict(Nq=5, Nk=9, dk=4, dv=3),
    dict(Nq=7, Nk=7, dk=5, dv=2, causal=True),
    dict(Nq=2, Nk=6, dk=1, dv=1, causal=True),
    dict(Nq=5, Nk=2, dk=1, dv=1, causal=True),
    dict(Nq=2, Nk=4, dk=3, dv=2, kv=[1]),
    dict(Nq=4, Nk=7, dk=3, dv=4, kv=[3], causal=True),
    dict(Nq=2, Nk=0, dk=3, dv=2),
    dict(Nq=1, Nk=5, dk=1, dv=1, bias=True),
    dict(Nq=3, Nk=6, dk=4, dv=3),
]


@pytest.mark.parametrize("fam", FAMILIES, ids=lambda f: "_".join(f"{k}{v}" for k, v in f.items()))
def test_fp32_small_families(fam):
    f = dict(fam)
    kv = f.pop("kv", None)
    bias = f.pop("bias", False)
    causal = f.pop("causal", False)
    a = wl.make_prefill(1, 2, f["Nq"], f["Nk"], f["dk"], f["dv"], torch.float32, causal=causal,
                        bias=bias, kv_lens=kv, seed=11, device=DEV)
    for bk in (16, 64):
        o, lse = run(a, bk)
        o_ref, l_ref, _ = oracle_full(a)
        compare(o, lse, o_ref, l_ref, torch.float32, what=str(fam))


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_masks_bias_padding(causal):
    a = wl.make_prefill(3, 2, 77, 130, 40, 24, torch.float32, causal=causal, bias=True,
                        kv_lens=[130, 45, 0], seed=12, device=DEV, bias_mask_p=0.1)
    for bk in (16, 32, 64):
        o, lse = run(a, bk)
        o_ref, l_ref, _ = oracle_full(a)
        compare(o, lse, o_ref, l_ref, torch.float32, what=f"fp32 masks bk={bk}")


def test_fp32_head_dims_256():
    a = wl.make_prefill(1, 1, 33, 70, 256, 256, torch.float32, causal=True, seed=13, device=DEV)
    o, lse = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.float32, what="fp32 d=256")


# ------------------------------------------------------------------------ bfloat16 path

DIMS = [(64, 64), (128, 128), (192, 128), (192, 64), (128, 64), (64, 128)]


@pytest.mark.parametrize("dk,dv", DIMS)
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_multi_tile_ragged(dk, dv, causal):
    # several 128-row / 128-key tiles and a ragged tail on both axes
    a = wl.make_prefill(2, 2, 300, 300, dk, dv, torch.bfloat16, causal=causal, seed=21,
                        device=DEV)
    o, lse = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, empty=empty_rows(a), what=f"bf16 {dk}/{dv}")


@pytest.mark.parametrize("B,causal,bias", [(40, True, False), (12, False, True)])
def test_bf16_dk192_many_items_per_cta(B, causal, bias):
    # the persistent dk = 192 kernel walks several items per CTA: per-sequence lengths with
    # empty and one-key sequences, more than 32 sequences (no length ranking) or fewer, and
    # every ring running on across items; rows spread over all sequences are checked
    lens = [(37 * b) % 400 for b in range(B)]
    lens[1], lens[2] = 0, 1
    a = wl.make_prefill(B, 3, 390, 400, 192, 128, torch.bfloat16, causal=causal, bias=bias, kv_lens=lens,
                        seed=25, device=DEV)
    o, lse = run(a)
    rows = sample_rows(a, n_per_head=24, heads=[(b, h) for b in range(B) for h in range(3)])
    o_ref, l_ref, _ = oracle_full(a, rows=rows)
    o_s, l_s = gather_rows(o, lse, rows, a.H, a.Nq)
    compare_rows(o_s, l_s, o_ref, l_ref, torch.bfloat16, what=f"dk192 B={B} causal={causal} bias={bias}")


@pytest.mark.parametrize("dk,dv", [(128, 128), (192, 128)])
@pytest.mark.parametrize("Nq,Nk", [(200, 450), (450, 200), (1, 129), (129, 1), (128, 128), (700, 300)])
def test_bf16_rectangular_bottom_right(Nq, Nk, dk, dv):
    # with Nq > Nk the first query tiles see no key: some CTAs of the dk = 192 kernel hold an
    # empty query tile followed by one with keys
    a = wl.make_prefill(1, 3, Nq, Nk, dk, dv, torch.bfloat16, causal=True, seed=22, device=DEV)
    o, lse = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, empty=empty_rows(a), what=f"rect {Nq}x{Nk}")


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_padding_bias_and_bias_masks(causal):
    a = wl.make_prefill(4, 2, 260, 390, 192, 128, torch.bfloat16, causal=causal, bias=True,
                        kv_lens=[390, 0, 129, 200], seed=23, device=DEV, bias_mask_p=0.05)
    o, lse = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, what="bias+padding")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nk", [392, 1024])
def test_bf16_dk192_bias_staged_by_tma(causal, Nk):
    # bias rows 16-byte aligned (Nk a multiple of 4): the bias tile goes through TMA
    a = wl.make_prefill(3, 2, 300, Nk, 192, 128, torch.bfloat16, causal=causal, bias=True,
                        kv_lens=[Nk, 129, Nk - 1], seed=28, device=DEV, bias_mask_p=0.05)
    o, lse = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, what=f"staged bias Nk={Nk}")


def test_bf16_dk192_staged_bias_masked_positions_bit_exact():
    kw = dict(B=3, H=2, Nq=257, Nk=336, dk=192, dv=128, dtype=torch.bfloat16, causal=True,
              bias=True, kv_lens=[336, 150, 77], seed=29, device=DEV)
    clean = wl.make_prefill(**kw, poison=False)
    dirty = wl.make_prefill(**kw, poison=True)
    o1, l1 = run(clean)
    o2, l2 = run(dirty)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    o_ref, l_ref, _ = oracle_full(clean)
    compare(o2, l2, o_ref, l_ref, torch.bfloat16, what="staged bias, poisoned")


def test_bf16_masked_positions_bit_exact():
    # NaN stored at every masked position (keys/values past kv_len, bias at masked (i, j))
    # must leave every output bit unchanged
    kw = dict(B=3, H=2, Nq=257, Nk=333, dk=128, dv=128, dtype=torch.bfloat16, causal=True,
              bias=True, kv_lens=[333, 150, 77], seed=24, device=DEV)
    clean = wl.make_prefill(**kw, poison=False)
    dirty = wl.make_prefill(**kw, poison=True)
    assert torch.isnan(dirty.k).any() and torch.isnan(dirty.bias).any()
    o1, l1 = run(clean)
    o2, l2 = run(dirty)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    o_ref, l_ref, _ = oracle_full(clean)
    compare(o2, l2, o_ref, l_ref, torch.bfloat16, what="poisoned")


@pytest.mark.parametrize("dk,dv,causal", [(128, 128, True), (128, 64, False), (64, 64, True), (64, 128, True)])
def test_bf16_staged_bias_at_dk_up_to_128(dk, dv, causal):
    # bias rows 16-byte aligned (Nk a multiple of 4): with dk >= dv the bias is staged by TMA in
    # the one-tile kernel, with dk < dv it is read into registers by the two-tile kernel; NaN
    # stored at every masked position must change no output bit either way
    kw = dict(B=3, H=2, Nq=300, Nk=336, dk=dk, dv=dv, dtype=torch.bfloat16, causal=causal, bias=True,
              kv_lens=[336, 150, 77], seed=31, device=DEV, bias_mask_p=0.05)
    clean = wl.make_prefill(**kw, poison=False)
    dirty = wl.make_prefill(**kw, poison=True)
    o1, l1 = run(clean)
    o2, l2 = run(dirty)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    o_ref, l_ref, _ = oracle_full(clean)
    compare(o2, l2, o_ref, l_ref, torch.bfloat16, empty=empty_rows(clean), what=f"staged bias {dk}/{dv}")


def test_bf16_empty_cases():
    # no keys at all
    a = wl.make_prefill(2, 2, 130, 0, 128, 128, torch.bfloat16, seed=25, device=DEV)
    o, lse = run(a)
    assert torch.all(o.view(torch.int16) == 0) and torch.all(lse == -math.inf)
    # every sequence padded to zero keys
    a = wl.make_prefill(2, 2, 130, 200, 128, 128, torch.bfloat16, kv_lens=[0, 0], seed=25,
                        device=DEV)
    o, lse = run(a)
    assert torch.all(o.view(torch.int16) == 0) and torch.all(lse == -math.inf)


def test_bf16_deterministic():
    a = wl.make_prefill(2, 4, 384, 384, 128, 128, torch.bfloat16, causal=True, seed=26,
                        device=DEV)
    o1, l1 = run(a)
    o2, l2 = run(a)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_bf16_strided_packed_qkv():
    # q, k, v as views into one packed [B, N, 3, H, d] tensor (non-contiguous strides)
    g = torch.Generator(device=DEV)
    g.manual_seed(27)
    B, N, H, d = 2, 200, 3, 128
    qkv = torch.randn((B, N, 3, H, d), generator=g, device=DEV).to(torch.bfloat16)
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    o, lse = ofa.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    a = wl.Attn("packed", torch.bfloat16, B, H, N, N, d, d, True, 1 / math.sqrt(d), q, k, v)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, what="packed qkv")


def test_bf16_unsupported_head_dim_raises():
    a = wl.make_prefill(1, 1, 16, 16, 96, 96, torch.bfloat16, seed=1, device=DEV)
    with pytest.raises(ofa.AttnError) as e:
        ofa.attn_fwd(a.q, a.k, a.v)
    assert e.value.status == ofa.Status.UNSUPPORTED


# ------------------------------------------------------------------------ full-size workloads

def test_causal_b4_h16_n2048_d128():
    a = wl.causal_2k(DEV)
    o, lse = run(a)
    heads = [(0, 0), (3, 15)] + [(b, h) for b in range(4) for h in (5, 11)]
    rows = sample_rows(a, n_per_head=64, heads=heads)
    # all rows of two heads as well
    full = np.concatenate([np.arange(a.Nq) + (b * a.H + h) * a.Nq for b, h in [(1, 7), (2, 3)]])
    rows = np.unique(np.concatenate([rows, full]))
    o_ref, l_ref, _ = oracle_full(a, rows=rows)
    o_s, l_s = gather_rows(o, lse, rows, a.H, a.Nq)
    compare_rows(o_s, l_s, o_ref, l_ref, torch.bfloat16, what="causal 2k")
    # properties at every row: finite, lse >= the row's logit of the diagonal key
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_padbias_b8_h8_n1024_dk192_dv128():
    a = wl.padded_bias(DEV)
    o, lse = run(a)
    rows = sample_rows(a, n_per_head=40)
    o_ref, l_ref, _ = oracle_full(a, rows=rows)
    o_s, l_s = gather_rows(o, lse, rows, a.H, a.Nq)
    compare_rows(o_s, l_s, o_ref, l_ref, torch.bfloat16, what="padded bias")
    # sequence 0 has kv_len 0: every one of its rows is empty, exactly
    assert torch.all(o[0].view(torch.int16) == 0) and torch.all(lse[0] == -math.inf)


def test_long_causal_b1_h32_n16384_d128():
    a = wl.long_causal(DEV)
    o, lse = run(a)
    # every row of heads 0 and 31, the last 256 rows of every head (where the lazy rescale
    # has run longest and most +8 keys were met), and a seeded sample of each head
    rows = sample_rows(a, n_per_head=48, heads=[(0, h) for h in range(a.H)])
    whole = np.concatenate([np.arange(a.Nq) + h * a.Nq for h in (0, a.H - 1)])
    last = np.concatenate([np.arange(a.Nq - 256, a.Nq) + h * a.Nq for h in range(a.H)])
    rows = np.unique(np.concatenate([rows, whole, last]))
    o_ref, l_ref, _ = oracle_full(a, rows=rows)
    o_s, l_s = gather_rows(o, lse, rows, a.H, a.Nq)
    compare_rows(o_s, l_s, o_ref, l_ref, torch.bfloat16, what="long causal")
