"""Pins of the oracle's dropout forward (no GPU).

The pages disable dropout ("How Does FlashAttention Preserve Global Softmax Across Tiles?",
section 6) and only require that with it the backward reproduce the forward's random mask and
scaling; the oracle reads that as inverted dropout of the normalised weights with the keep
mask as an input.  These tests tie that reading to the already pinned forward (all kept, none
kept, disjoint masks) and to the defining property of inverted dropout (the mean over random
masks is the undropped output), so that a missing 1/(1 - p), a row sum taken over the kept
keys only, or a mask read at the wrong position fails one of them."""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_fa2_gb300 import workloads as wl

def small(causal=True, lens=None, seed=11, B=2, H=2, N=37, d=16):
    return wl.make_prefill(B, H, N, N, d, d, torch.float32, causal=causal, kv_lens=lens, seed=seed,
                           device="cpu")


def run(a, keep, p):
    return oracle.attn_fwd_dropout(a.q, a.k, a.v, keep, p, kv_lens=a.kv_lens, causal=a.causal,
                                   scale=a.scale)


def plain(a):
    o, lse, _ = oracle.attn_fwd(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=a.causal, scale=a.scale)
    return o, lse


@pytest.mark.parametrize("p", [0.0, 0.1, 0.5])
def test_all_kept_is_the_forward_scaled(p):
    a = small(lens=[37, 20])
    keep = torch.ones((a.B, a.H, a.Nq, a.Nk), dtype=torch.bool)
    o, lse = run(a, keep, p)
    o0, lse0 = plain(a)
    assert np.allclose(o, o0 / (1.0 - p), rtol=1e-12, atol=1e-12)
    assert np.array_equal(np.isfinite(lse), np.isfinite(lse0))
    assert np.allclose(lse[np.isfinite(lse)], lse0[np.isfinite(lse0)], rtol=0, atol=0)


def test_none_kept_gives_zero_and_keeps_lse():
    a = small(lens=[37, 5])
    keep = torch.zeros((a.B, a.H, a.Nq, a.Nk), dtype=torch.bool)
    o, lse = run(a, keep, 0.3)
    _, lse0 = plain(a)
    assert np.all(o == 0.0) and not np.any(np.signbit(o))
    fin = np.isfinite(lse0)
    assert np.array_equal(np.isfinite(lse), fin) and np.all(lse[fin] == lse0[fin])


def test_disjoint_masks_add():
    a = small(causal=False, seed=12)
    g = torch.Generator().manual_seed(3)
    u = torch.rand((a.B, a.H, a.Nq, a.Nk), generator=g)
    ka, kb = u < 0.4, (u >= 0.4) & (u < 0.7)
    oa, _ = run(a, ka, 0.25)
    ob, _ = run(a, kb, 0.25)
    oab, _ = run(a, ka | kb, 0.25)
    assert np.allclose(oa + ob, oab, rtol=1e-12, atol=1e-12)


def test_mean_over_masks_is_the_undropped_output():
    a = small(B=1, H=1, N=12, d=8, lens=None, seed=13)
    o0, _ = plain(a)
    p, n = 0.4, 4000
    g = torch.Generator().manual_seed(4)
    keeps = torch.rand((n, a.Nq, a.Nk), generator=g) >= p
    P = oracle.attn_probs(a.q, a.k, a.v, causal=a.causal, scale=a.scale)[0, 0]
    v = a.v[0, :, 0].double().numpy()
    # per mask the oracle's output; their mean against the undropped forward
    acc = np.zeros_like(o0[0, :, 0])
    for t in range(0, n, 500):
        for kt in keeps[t:t + 500]:
            o, _ = run(a, kt[None, None], p)
            acc += o[0, :, 0]
    mean = acc / n
    # each output is a sum of kept terms w_j v_j / (1 - p): its standard deviation per mask
    sd = np.sqrt(p / (1 - p) * (P ** 2) @ (v ** 2))
    assert np.all(np.abs(mean - o0[0, :, 0]) <= 5 * sd / np.sqrt(n) + 1e-12)


def test_mask_bits_at_hidden_positions_do_not_matter():
    a = small(lens=[30, 9], seed=14)
    g = torch.Generator().manual_seed(5)
    keep = torch.rand((a.B, a.H, a.Nq, a.Nk), generator=g) >= 0.3
    P = oracle.attn_probs(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=a.causal, scale=a.scale)
    hidden = torch.from_numpy(P == 0.0)
    flipped = torch.where(hidden, ~keep, keep)
    o1, _ = run(a, keep, 0.3)
    o2, _ = run(a, flipped, 0.3)
    assert np.array_equal(o1, o2)


def test_packed_mask_round_trip():
    keep = wl.dropout_keep(2, 3, 5, 300, 0.35, seed=6)
    packed = wl.pack_keep_mask(keep)
    assert packed.dtype == torch.uint8 and packed.shape == (2, 3, 5, 16 * 3)
    bits = np.unpackbits(packed.numpy(), axis=-1, bitorder="little")
    assert np.array_equal(bits[..., :300].astype(bool), keep.numpy())
    assert not bits[..., 300:].any()


# ---- backward of the dropout forward


def grads(a, keep, p, dout):
    return oracle.attn_bwd_dropout(a.q, a.k, a.v, dout, keep, p, kv_lens=a.kv_lens, causal=a.causal,
                                   scale=a.scale)


def test_bwd_all_kept_no_drop_is_the_backward():
    a = small(lens=[37, 20], seed=21)
    dout = torch.randn(a.B, a.Nq, a.H, a.dv, generator=torch.Generator().manual_seed(1))
    keep = torch.ones((a.B, a.H, a.Nq, a.Nk), dtype=torch.bool)
    got = grads(a, keep, 0.0, dout)
    want = oracle.attn_bwd(a.q, a.k, a.v, dout, kv_lens=a.kv_lens, causal=a.causal, scale=a.scale)[:3]
    for x, y in zip(got, want):
        assert np.allclose(x, y, rtol=1e-12, atol=1e-12)


def test_bwd_none_kept_passes_no_gradient():
    a = small(lens=[37, 11], seed=22)
    dout = torch.randn(a.B, a.Nq, a.H, a.dv, generator=torch.Generator().manual_seed(2))
    keep = torch.zeros((a.B, a.H, a.Nq, a.Nk), dtype=torch.bool)
    for x in grads(a, keep, 0.4, dout):
        assert np.all(x == 0.0)


def test_bwd_matches_finite_differences_of_the_dropout_forward():
    # central differences of L = sum(dout * O_drop) in float64, at a few entries of q, k, v
    a = wl.make_prefill(1, 2, 9, 11, 6, 5, torch.float32, causal=True, kv_lens=[10], seed=23,
                        device="cpu", poison=False)
    g = torch.Generator().manual_seed(3)
    dout = torch.randn(a.B, a.Nq, a.H, a.dv, generator=g).double().numpy()
    keep = torch.rand((a.B, a.H, a.Nq, a.Nk), generator=g) >= 0.3
    p = 0.3
    dQ, dK, dV = grads(a, keep, p, torch.from_numpy(dout))
    base = {"q": a.q.double().numpy().copy(), "k": a.k.double().numpy().copy(), "v": a.v.double().numpy().copy()}

    def loss(t):
        o, _ = oracle.attn_fwd_dropout(t["q"], t["k"], t["v"], keep, p, kv_lens=a.kv_lens,
                                       causal=a.causal, scale=a.scale)
        return float(np.sum(dout * o))

    # the oracle takes float32 inputs, so a perturbed entry is rounded to float32: a step of
    # 2^-10 and the 2e-4 of the forward oracle's own finite-difference pin
    eps = 2.0 ** -10
    rng = np.random.default_rng(4)
    for name, grad in (("q", dQ), ("k", dK), ("v", dV)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in base[name].shape)
            if name in ("k", "v") and idx[1] >= 10:  # past the key length: no part of the loss
                assert grad[idx] == 0.0
                continue
            t1 = {k_: v_.copy() for k_, v_ in base.items()}
            t2 = {k_: v_.copy() for k_, v_ in base.items()}
            t1[name][idx] += eps
            t2[name][idx] -= eps
            fd = (loss(t1) - loss(t2)) / (2 * eps)
            assert abs(fd - grad[idx]) <= 2e-4 * max(1.0, abs(fd)), (name, idx, fd, grad[idx])


def test_mask_bits_under_a_minus_inf_bias_do_not_matter():
    a = wl.make_prefill(2, 2, 21, 23, 8, 8, torch.float32, causal=False, bias=True, kv_lens=[23, 15],
                        seed=15, device="cpu", bias_mask_p=0.3)
    g = torch.Generator().manual_seed(6)
    keep = torch.rand((a.B, a.H, a.Nq, a.Nk), generator=g) >= 0.25
    hidden = torch.isinf(a.bias) & (a.bias < 0)
    assert hidden.any()
    flipped = torch.where(hidden, ~keep, keep)
    kw = dict(bias=a.bias, kv_lens=a.kv_lens, causal=False, scale=a.scale)
    o1, _ = oracle.attn_fwd_dropout(a.q, a.k, a.v, keep, 0.25, **kw)
    o2, _ = oracle.attn_fwd_dropout(a.q, a.k, a.v, flipped, 0.25, **kw)
    assert np.array_equal(o1, o2)
    d1 = oracle.attn_bwd_dropout(a.q, a.k, a.v, torch.ones(a.B, a.Nq, a.H, a.dv), keep, 0.25, **kw)
    d2 = oracle.attn_bwd_dropout(a.q, a.k, a.v, torch.ones(a.B, a.Nq, a.H, a.dv), flipped, 0.25, **kw)
    for x, y in zip(d1, d2):
        assert np.array_equal(x, y)
