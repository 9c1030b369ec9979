"""Seeded random shapes through the tcgen05 backward against the float64 oracle: d = 64 or 128,
causal or not, with or without per-sequence lengths (some 0), a bias (some -inf entries) or
dropout drawn in-kernel, Nq and Nk from 1 to a few tiles; the gradient bound of helpers."""
import numpy as np
import pytest
import torch

import oracle
import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from oracle import philox
from helpers import check_grad, cpu32, dq_c_term

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("seed", range(12))
def test_random_shape_backward(seed):
    r = np.random.default_rng(2000 + seed)
    d = int(r.choice([64, 128]))
    B, H = int(r.integers(1, 3)), int(r.integers(1, 3))
    Nq, Nk = int(r.integers(1, 400)), int(r.integers(1, 400))
    causal = bool(r.integers(2))
    mode = ["plain", "bias", "dropout"][seed % 3]
    lens = [int(x) for x in r.integers(0, Nk + 1, B)] if r.integers(2) else None
    a = wl.make_prefill(B, H, Nq, Nk, d, d, torch.bfloat16, causal=causal, bias=mode == "bias", kv_lens=lens,
                        seed=seed, device=DEV, bias_mask_p=0.03 if mode == "bias" else 0.0)
    drop = dict(dropout_p=0.2, dropout_seed=77 + seed, dropout_offset=seed) if mode == "dropout" else {}
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=causal, scale=a.scale, **drop)
    g = torch.Generator(device=DEV)
    g.manual_seed(3000 + seed)
    dout = torch.randn(o.shape, generator=g, device=DEV).to(o.dtype)
    dq, dk, dv = ofa.attn_bwd(a.q, a.k, a.v, o, lse, dout, bias=a.bias, kv_lens=a.kv_lens, causal=causal,
                              scale=a.scale, **drop)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    kvl = None if a.kv_lens is None else a.kv_lens.cpu()
    if mode == "dropout":
        keep, p_real = philox.keep_mask(drop["dropout_seed"], drop["dropout_offset"], B, H, Nq, Nk, 0.2)
        refs = oracle.attn_bwd_dropout(cpu32(a.q), cpu32(a.k), cpu32(a.v), cpu32(dout), torch.from_numpy(keep),
                                       p_real, kv_lens=kvl, causal=causal, scale=a.scale)
    else:
        refs = oracle.attn_bwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), cpu32(dout), bias=cpu32(a.bias), kv_lens=kvl,
                               causal=causal, scale=a.scale)[:3]
    ct = dq_c_term(dout, o, a.k, a.scale, a.kv_lens)
    what = f"d={d} B={B} H={H} {Nq}x{Nk} causal={causal} {mode} lens={lens}"
    check_grad(dq, refs[0], "dq " + what, extra=ct)
    check_grad(dk, refs[1], "dk " + what)
    check_grad(dv, refs[2], "dv " + what)
