"""GPU parity of the attention backward (dQ, dK, dV) against the float64 oracle.

Tolerance: the backward forms P and dS in bf16 for the tensor cores and writes bf16
gradients; every element is held to |g - ref| <= 2^-6 |ref| + 2^-4 rms(its row) +
2^-10 rms(tensor) (plus, for dQ, the reach of the bf16 O through c), and every tensor to a
relative Frobenius error of 1e-2 (helpers.check_grad, which derives both from the rounding and
calibrates them against a bf16-rounding emulation).
What the masks fix is exact: a key that no row sees gets dK = dV = +0.0, and an empty row gets
dQ = +0.0."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import check_grad, cpu32, dq_c_term

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_bwd(a, seed=0):
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal, scale=a.scale)
    g = torch.Generator(device=DEV)
    g.manual_seed(1000 + seed)
    dout = torch.randn(o.shape, generator=g, device=DEV).to(o.dtype)
    dq, dk, dv = ofa.attn_bwd(a.q, a.k, a.v, o, lse, dout, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal,
                              scale=a.scale)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    run_bwd.last_o = o
    return dout, dq, dk, dv


def oracle_bwd(a, dout):
    return oracle.attn_bwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), cpu32(dout), bias=cpu32(a.bias),
                           kv_lens=None if a.kv_lens is None else a.kv_lens.cpu(), causal=a.causal,
                           scale=a.scale)[:3]


def unseen_keys(a):
    """[B, Nk]: keys no row can see (past the sequence's key length; the last row of a
    bottom-right causal mask sees every key before it)."""
    z = np.zeros((a.B, a.Nk), bool)
    for b, n in enumerate(a.kv_len_list()):
        z[b, n:] = True
    return z


def empty_query_rows(a):
    """[B, Nq]: rows that see no key (masks only; the same for every head)."""
    z = np.zeros((a.B, a.Nq), bool)
    for b, n in enumerate(a.kv_len_list()):
        for i in range(a.Nq):
            last = n - 1 if not a.causal else min(n - 1, i + n - a.Nq)
            z[b, i] = last < 0
    return z


def check_all(a, dq, dk, dv, rq, rk, rv, what, dout):
    ct = dq_c_term(dout, run_bwd.last_o, a.k, a.scale, a.kv_lens)
    check_grad(dq, rq, "dq " + what, empty_query_rows(a), extra=ct)
    check_grad(dk, rk, "dk " + what, unseen_keys(a))
    check_grad(dv, rv, "dv " + what, unseen_keys(a))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(100, 150), (150, 100), (64, 64), (33, 257)])
def test_bwd_matches_oracle(d, causal, Nq, Nk):
    a = wl.make_prefill(2, 2, Nq, Nk, d, d, torch.bfloat16, causal=causal, seed=60 + Nq + Nk, device=DEV)
    dout, dq, dk, dv = run_bwd(a)
    rq, rk, rv = oracle_bwd(a, dout)
    check_all(a, dq, dk, dv, rq, rk, rv, f"d={d} causal={causal} {Nq}x{Nk}", dout)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_padding_bias_and_masks(causal, d):
    a = wl.make_prefill(4, 2, 130, 200, d, d, torch.bfloat16, causal=causal, bias=True,
                        kv_lens=[200, 0, 65, 1], seed=61, device=DEV, bias_mask_p=0.05)
    dout, dq, dk, dv = run_bwd(a, 1)
    rq, rk, rv = oracle_bwd(a, dout)
    check_all(a, dq, dk, dv, rq, rk, rv, "bias+padding", dout)


def test_bwd_dk_dv_deterministic_and_poison_free():
    a = wl.make_prefill(2, 3, 200, 300, 128, 128, torch.bfloat16, causal=True, kv_lens=[300, 123],
                        seed=62, device=DEV)
    _, dq1, dk1, dv1 = run_bwd(a, 2)
    _, dq2, dk2, dv2 = run_bwd(a, 2)
    assert torch.equal(dk1.view(torch.int16), dk2.view(torch.int16))
    assert torch.equal(dv1.view(torch.int16), dv2.view(torch.int16))
    assert (dq1.float() - dq2.float()).abs().max().item() <= 1e-2
    # keys past kv_len hold NaN (the workload's poison): no gradient reads them
    assert torch.isfinite(dq1.float()).all() and torch.isfinite(dk1.float()).all()


@pytest.mark.parametrize("d,bias", [(64, False), (128, True)])
def test_bwd_full_size_shapes_sampled_heads(d, bias):
    # the 2k causal shape at d = 64, and at d = 128 with a broadcast-free fp32 bias (two heads
    # against the oracle each)
    a = wl.make_prefill(2, 8, 2048, 2048, d, d, torch.bfloat16, causal=True, bias=bias, seed=63, device=DEV)
    dout, dq, dk, dv = run_bwd(a, 4)
    o = run_bwd.last_o
    for b, h in ((0, 0), (1, 7)):
        sub = lambda t: cpu32(t[b:b + 1, :, h:h + 1])
        bsub = cpu32(a.bias[b:b + 1, h:h + 1]) if bias else None
        rq, rk, rv, _ = oracle.attn_bwd(sub(a.q), sub(a.k), sub(a.v), sub(dout), bias=bsub, causal=True,
                                        scale=a.scale)
        ct = dq_c_term(sub(dout), sub(o), sub(a.k), a.scale)
        check_grad(dq[b:b + 1, :, h:h + 1], rq, f"dq d={d} bias={bias} head {b},{h}", extra=ct)
        check_grad(dk[b:b + 1, :, h:h + 1], rk, f"dk d={d} bias={bias} head {b},{h}")
        check_grad(dv[b:b + 1, :, h:h + 1], rv, f"dv d={d} bias={bias} head {b},{h}")


def test_bwd_causal_b4_h16_n2048_d128_sampled_heads():
    a = wl.causal_2k(DEV)
    dout, dq, dk, dv = run_bwd(a, 3)
    o = run_bwd.last_o
    for b, h in ((0, 0), (3, 15), (2, 7)):
        sub = lambda t: cpu32(t[b:b + 1, :, h:h + 1])
        rq, rk, rv, _ = oracle.attn_bwd(sub(a.q), sub(a.k), sub(a.v), sub(dout), causal=True, scale=a.scale)
        ct = dq_c_term(sub(dout), sub(o), sub(a.k), a.scale)
        check_grad(dq[b:b + 1, :, h:h + 1], rq, f"dq head {b},{h}", extra=ct)
        check_grad(dk[b:b + 1, :, h:h + 1], rk, f"dk head {b},{h}")
        check_grad(dv[b:b + 1, :, h:h + 1], rv, f"dv head {b},{h}")
