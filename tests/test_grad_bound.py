"""The gradient bound of the GPU backward tests, checked on the CPU against both of its sides.

helpers.check_grad holds each gradient element to 2^-6 |ref| + 2^-4 rms(its row) +
2^-10 rms(tensor), plus for dQ the reach of the bf16 O's rounding through c_i = dO_i . O_i
(helpers.dq_c_term), and each tensor to a relative Frobenius error of 1e-2.  Here:
  - a backward that rounds exactly where the kernels round (P and dS to bf16 before the
    products, c from the bf16 O, the gradients stored in bf16; torch float32 otherwise)
    passes it on causal, rectangular and non-causal heads, so the bound does not reject
    honest bf16 arithmetic;
  - plausible mistakes applied to that output (small entries zeroed or halved, a dropped
    scale, c left out, unnormalised weights, a one-row sign error, a 3 % gain) each fail it,
    so the bound does reject a wrong gradient, including one wrong only in the bulk of small
    elements.
The reference is the float64 oracle ("How Does FlashAttention Preserve Global Softmax Across
Tiles?", section 7)."""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import GRAD_FRO, dq_c_term, grad_bound_violations


def bf(x):
    return x.to(torch.bfloat16).float()


def emulate(q, k, v, g, causal, scale, mistake=None):
    """bf16-rounding backward of one head: q [Nq, d], k, v [Nk, d], g [Nq, d] (bf16 values in
    float32).  Returns dq, dk, dv as float64 arrays [Nq or Nk, d]."""
    nq, nk = q.shape[0], k.shape[0]
    i = torch.arange(nq)[:, None]
    j = torch.arange(nk)[None, :]
    hidden = (j > i + nk - nq) if causal else torch.zeros(nq, nk, dtype=torch.bool)
    empty = hidden.all(1)
    s = ((q @ k.T) * scale).masked_fill(hidden, -math.inf)
    m = torch.where(empty, torch.zeros(()), s.max(1).values)
    w = torch.exp(s - m[:, None])                      # masked keys: exp(-inf) = 0
    l = w.sum(1)
    # the forward as the kernels run it: bf16 weights in the value product, one division,
    # O stored in bf16, lse = m + ln l (an empty row: O = 0, lse = -inf)
    o = bf(torch.where(empty[:, None], torch.zeros(()), (bf(w) @ v) / l.clamp_min(1e-30)[:, None]))
    lse = torch.where(empty, torch.full((), -math.inf), m + torch.log(l.clamp_min(1e-30)))
    ref_pt = m if mistake == "unnormalised" else lse
    p = torch.where(empty[:, None], torch.zeros(()), torch.exp(s - ref_pt[:, None]))
    dv = bf(bf(p).T @ g)
    dp = g @ v.T
    c = (g * o).sum(1)
    ds = bf(p * dp) if mistake == "no_c" else bf(p * (dp - c[:, None]))
    dq = bf((1.0 if mistake == "no_scale_dq" else scale) * (ds @ k))
    dk = bf(scale * (ds.T @ q))
    emulate.last_o = o
    return dq.double().numpy(), dk.double().numpy(), dv.double().numpy()


def head(nq, nk, d, causal, seed):
    gen = torch.Generator().manual_seed(seed)
    q, k, v = (bf(torch.randn(n, d, generator=gen)) for n in (nq, nk, nk))
    g = bf(torch.randn(nq, d, generator=gen))
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attn_bwd(q[None, :, None], k[None, :, None], v[None, :, None], g[None, :, None],
                          causal=causal, scale=scale)[:3]
    ref = [np.asarray(r, np.float64)[0, :, 0] for r in ref]
    return (q, k, v, g, scale), ref


def extras(q, k, v, g, scale):
    """Per-tensor additions to the limit: the c term for dQ (from the emulated forward's O)."""
    ct = dq_c_term(g[None, :, None], emulate.last_o[None, :, None], k[None, :, None], scale)[0, :, 0]
    return (ct, None, None)


def passes(got, ref, extra=None):
    bad, fro = grad_bound_violations(got, ref, extra)
    return bad == 0 and fro <= GRAD_FRO


CASES = [(384, 384, 128, True, 1), (200, 333, 64, True, 2), (256, 256, 64, False, 3),
         (333, 200, 128, True, 4), (512, 512, 128, True, 13), (1024, 1024, 64, True, 8)]


@pytest.mark.parametrize("nq,nk,d,causal,seed", CASES)
def test_bf16_rounding_backward_passes(nq, nk, d, causal, seed):
    (q, k, v, g, scale), ref = head(nq, nk, d, causal, seed)
    got = emulate(q, k, v, g, causal, scale)
    for x, r, e, name in zip(got, ref, extras(q, k, v, g, scale), ("dq", "dk", "dv")):
        bad, fro = grad_bound_violations(x, r, e)
        assert bad == 0 and fro <= GRAD_FRO, (name, bad, fro)
        assert fro < GRAD_FRO / 3, (name, fro)  # the honest error sits well inside the bound


def planted(name, x, r):
    """A mistake applied to an honest gradient x (reference r); None if it does not apply."""
    if name == "zero_small":       # every entry below 0.05 in magnitude lost
        return np.where(np.abs(r) < 0.05, 0.0, x)
    if name == "halve_small":      # a missing factor on the entries below the median only
        return np.where(np.abs(r) < np.median(np.abs(r)), 0.5 * x, x)
    if name == "gain":             # a 3 % error in a scale factor
        return x * 1.03
    if name == "row_sign":         # one row's sign flipped
        y = x.copy()
        nz = np.flatnonzero(np.abs(r).sum(1) > 0)
        y[nz[len(nz) // 2]] *= -1.0
        return y
    raise KeyError(name)


@pytest.mark.parametrize("mistake", ["zero_small", "halve_small", "gain", "row_sign"])
@pytest.mark.parametrize("nq,nk,d,causal,seed", CASES[:2])
def test_planted_output_mistakes_fail(mistake, nq, nk, d, causal, seed):
    (q, k, v, g, scale), ref = head(nq, nk, d, causal, seed)
    got = emulate(q, k, v, g, causal, scale)
    for x, r, e, name in zip(got, ref, extras(q, k, v, g, scale), ("dq", "dk", "dv")):
        assert passes(x, r, e)
        assert not passes(planted(mistake, x, r), r, e), (mistake, name)


@pytest.mark.parametrize("mistake,which", [("no_scale_dq", (0,)), ("no_c", (0, 1)),
                                           ("unnormalised", (0, 1, 2))])
def test_planted_arithmetic_mistakes_fail(mistake, which):
    (q, k, v, g, scale), ref = head(256, 320, 128, True, 5)
    got = emulate(q, k, v, g, True, scale, mistake=mistake)
    ex = extras(q, k, v, g, scale)
    for t in which:
        assert not passes(got[t], ref[t], ex[t]), (mistake, t)
