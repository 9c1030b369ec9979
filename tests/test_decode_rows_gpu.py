"""GPU parity of split-KV decode with several query rows per sequence (1 < Nq <= 8): every
cache row is read once for all rows, and with causal=True row i sees keys
j <= i + kv_len - Nq (bottom-right, "How Does FlashAttention Preserve Global Softmax Across
Tiles?", section 6), so rows of a sequence shorter than Nq can be empty."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL, compare, cpu32, empty_rows, oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(a, num_splits=None, **kw):
    o, lse, ws = ofa.attn_decode_splitkv(a.q, a.k, a.v, kv_lens=a.kv_lens, bias=a.bias,
                                         num_splits=num_splits or a.num_splits, scale=a.scale,
                                         causal=a.causal, **kw)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    return o, lse, ws


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("nq", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_rows_match_oracle(d, nq, causal):
    # kv_len 0, shorter than nq (leading rows empty under causal), one split's worth, long
    lens = [0, 1, nq - 1, 17, 700, 333]
    for splits in (1, 16):
        a = wl.decode(DEV, seed=40 + nq, B=6, H=3, L=700, d=d, num_splits=splits, lens=lens, nq=nq,
                      causal=causal)
        o, lse, _ = run(a)
        o_ref, l_ref, _ = oracle_full(a)
        compare(o, lse, o_ref, l_ref, torch.bfloat16, empty=empty_rows(a),
                what=f"decode rows nq={nq} d={d} causal={causal} S={splits}")


def test_decode_rows_partials_are_the_split_states():
    # workspace [B, H, Nq, S, 2 + dv]: row i's state over the keys of split s it can see
    S, nq = 5, 4
    a = wl.decode(DEV, seed=41, B=3, H=2, L=300, d=128, num_splits=S, lens=[300, 3, 129], nq=nq,
                  causal=True)
    _, _, ws = run(a)
    part = ws[: 3 * 2 * nq * S * 130].view(3, 2, nq, S, 130).cpu().double().numpy()
    for b, n in enumerate(a.kv_len_list()):
        kvl = torch.tensor([n], dtype=torch.int32)
        for h in range(2):
            q = cpu32(a.q[b:b + 1, :, h:h + 1])
            k = cpu32(a.k[b:b + 1, :, h:h + 1])
            v = cpu32(a.v[b:b + 1, :, h:h + 1])
            for s in range(S):
                lo, hi = (s * n) // S, ((s + 1) * n) // S
                st = oracle.key_state(q, k, v, lo, hi, kv_lens=kvl, causal=True, scale=a.scale)[0, 0]
                for i in range(nq):
                    g = part[b, h, i, s]
                    if st[i, 1] == 0:
                        assert g[0] == -np.inf and g[1] == 0 and np.all(g[2:] == 0), (b, h, s, i)
                        continue
                    f = math.exp(g[0] - st[i, 0])
                    assert abs(g[0] - st[i, 0]) < 1e-4
                    assert abs(f * g[1] - st[i, 1]) <= 1e-3 * st[i, 1]
                    assert np.max(np.abs(f * g[2:] - st[i, 2:])) <= 2e-3 * max(1.0, st[i, 1])


@pytest.mark.parametrize("causal", [False, True])
def test_decode_rows_bias_and_masks(causal):
    nq = 4
    a = wl.decode(DEV, seed=42, B=3, H=2, L=300, d=128, num_splits=7, lens=[300, 40, 2], nq=nq,
                  causal=causal)
    g = torch.Generator(device=DEV)
    g.manual_seed(6)
    bias = torch.randn((3, 2, nq, 300), generator=g, device=DEV)
    bias[:, :, :, ::5] = -math.inf
    a.bias = bias
    o, lse, _ = run(a)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, what=f"decode rows bias causal={causal}")


def test_decode_rows_split_invariance_and_poison():
    kw = dict(seed=43, B=3, H=4, L=1000, d=128, num_splits=16, lens=[1000, 999, 3], nq=8, causal=True)
    a = wl.decode(DEV, **kw)
    outs = [run(a, S)[:2] for S in (1, 3, 16, 37)]
    fin = torch.isfinite(outs[0][1])
    for o, l in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert torch.equal(torch.isfinite(l), fin)
        assert (l[fin] - outs[0][1][fin]).abs().max().item() <= 1e-3
    o1, l1, _ = run(wl.decode(DEV, poison=False, **kw))
    o2, l2, _ = run(a)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_decode_rows_one_row_is_the_single_row_decode():
    # the first row of a non-causal Nq=4 decode is the Nq=1 decode of that row (the two take
    # different kernels, P in bf16 on the tensor cores against fp32 on the FMA pipe: equal
    # within the bf16 tolerance, and the empty sequence exactly)
    a4 = wl.decode(DEV, seed=44, B=4, H=3, L=500, d=128, num_splits=16, lens=[500, 9, 0, 250], nq=4)
    o4, l4, _ = run(a4)
    q1 = a4.q[:, :1].contiguous()
    o1, l1, _ = ofa.attn_decode_splitkv(q1, a4.k, a4.v, kv_lens=a4.kv_lens, num_splits=16,
                                        scale=a4.scale)
    torch.cuda.synchronize()
    fin = torch.isfinite(l1[:, :, 0])
    assert torch.equal(fin, torch.isfinite(l4[:, :, 0])) and not fin[2].any()
    assert torch.all(o4[2].view(torch.int16) == 0)
    assert (o1[:, 0].float() - o4[:, 0].float()).abs().max().item() <= TOL[torch.bfloat16]["o"]
    assert (l1[:, :, 0][fin] - l4[:, :, 0][fin]).abs().max().item() <= TOL[torch.bfloat16]["lse"]


def test_decode_rows_rejects_too_many_rows():
    a = wl.decode(DEV, seed=45, B=1, H=1, L=64, d=128, num_splits=2, lens=[64], nq=9)
    with pytest.raises(ofa.AttnError):
        run(a)


def test_decode_b64_h32_l8192_d128_nq4_causal_sampled():
    a = wl.decode(DEV, nq=4, causal=True)
    o, lse, _ = run(a)
    rng = np.random.default_rng(46)
    heads = {(0, 0), (63, 31), (0, 31), (63, 0)}
    heads |= {(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 24), rng.integers(0, 32, 24))}
    lens = a.kv_len_list()
    for b, h in sorted(heads):
        n = lens[b]
        kvl = torch.tensor([n], dtype=torch.int32)
        o_ref, l_ref, _ = oracle.attn_fwd(cpu32(a.q[b:b + 1, :, h:h + 1]), cpu32(a.k[b:b + 1, :n, h:h + 1]),
                                          cpu32(a.v[b:b + 1, :n, h:h + 1]), kv_lens=kvl, causal=True,
                                          scale=a.scale)
        for i in range(4):
            if not np.isfinite(l_ref[0, 0, i]):
                assert lse[b, h, i].item() == -math.inf
                assert torch.all(o[b, i, h].view(torch.int16) == 0)
                continue
            err = np.max(np.abs(o[b, i, h].float().cpu().numpy() - o_ref[0, i, 0]))
            assert err <= TOL[torch.bfloat16]["o"], (b, h, i, n, err)
            assert abs(lse[b, h, i].item() - l_ref[0, 0, i]) <= TOL[torch.bfloat16]["lse"]
