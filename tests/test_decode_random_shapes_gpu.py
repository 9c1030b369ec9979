"""Seeded random decode shapes against the float64 oracle, through the two-launch, fused and
allocation-free entry points: 1 to 8 query rows per sequence (bottom-right causal when more
than one), d = 64 or 128, 1 to 64 splits, ragged sequence lengths (some 0 or 1), with or
without a bias (with -inf entries); the three entry points must also agree bit for bit."""
import math

import numpy as np
import pytest
import torch

import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL, compare, empty_rows, oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("seed", range(12))
def test_random_decode(seed):
    r = np.random.default_rng(4000 + seed)
    d = int(r.choice([64, 128]))
    B, H = int(r.integers(1, 5)), int(r.integers(1, 5))
    L = int(r.integers(1, 1500))
    nq = int(r.integers(1, 9))
    S = int(r.integers(1, 65))
    lens = [int(x) for x in r.integers(0, L + 1, B)]
    if B > 1:
        lens[0] = 1
    a = wl.decode(DEV, seed=seed, B=B, H=H, L=L, d=d, num_splits=S, lens=lens, nq=nq, causal=nq > 1)
    if seed % 2:
        g = torch.Generator(device=DEV).manual_seed(seed)
        bias = torch.randn((B, H, nq, L), generator=g, device=DEV)
        bias[..., seed % 5::5] = -math.inf
        a.bias = bias
    kw = dict(kv_lens=a.kv_lens, num_splits=S, bias=a.bias, scale=a.scale, causal=a.causal)
    o1, l1, _ = ofa.attn_decode_splitkv(a.q, a.k, a.v, **kw)
    o2, l2, _ = ofa.attn_decode_splitkv_fused(a.q, a.k, a.v, **kw)
    o3, l3 = ofa.attn_decode_splitkv_noalloc(a.q, a.k, a.v, **kw)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    for o, l in ((o2, l2), (o3, l3)):
        assert torch.equal(o.view(torch.int16), o1.view(torch.int16))
        assert torch.equal(l, l1)
    o_ref, l_ref, _ = oracle_full(a)
    compare(o1, l1, o_ref, l_ref, torch.bfloat16, empty=None if a.bias is not None else empty_rows(a),
            what=f"seed {seed}")
