"""Seeded random shapes through every forward dispatch path against the float64 oracle: head
dimensions 64, 128 and 192 with dv <= dk or dv > dk (two-tile kernel, one-tile kernel, staged
or per-row bias), causal or not, with or without per-sequence lengths (some 0, some past the
query count) and a bias (aligned rows or not, some -inf), Nq and Nk from 1 to a few tiles."""
import numpy as np
import pytest
import torch

import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL, compare, empty_rows, oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda"
DIMS = [(64, 64), (128, 128), (128, 64), (64, 128), (192, 128), (192, 64)]


def case(seed):
    r = np.random.default_rng(seed)
    dk, dv = DIMS[r.integers(len(DIMS))]
    B, H = int(r.integers(1, 4)), int(r.integers(1, 4))
    Nq, Nk = int(r.integers(1, 520)), int(r.integers(1, 520))
    causal = bool(r.integers(2))
    bias = bool(r.integers(2))
    lens = None
    if r.integers(2):
        lens = [int(x) for x in r.integers(0, Nk + 1, B)]
    return dict(B=B, H=H, Nq=Nq, Nk=Nk, dk=dk, dv=dv, causal=causal, bias=bias, kv_lens=lens,
                bias_mask_p=0.03 if bias else 0.0)


@pytest.mark.parametrize("seed", range(24))
def test_random_shape(seed):
    c = case(1000 + seed)
    a = wl.make_prefill(c["B"], c["H"], c["Nq"], c["Nk"], c["dk"], c["dv"], torch.bfloat16,
                        causal=c["causal"], bias=c["bias"], kv_lens=c["kv_lens"], seed=seed, device=DEV,
                        bias_mask_p=c["bias_mask_p"])
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal, scale=a.scale)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    o_ref, l_ref, _ = oracle_full(a)
    # rows that a -inf bias empties are not in empty_rows (masks only): the oracle decides those
    compare(o, lse, o_ref, l_ref, torch.bfloat16, empty=None if c["bias"] else empty_rows(a), what=str(c))
