"""GPU parity of the dropout forward (keep mask as an input) against the oracle.

The kernels read the bit-packed mask (workloads.pack_keep_mask); the oracle reads the same
keep decisions unpacked.  Kept weights are scaled by 1 / (1 - p), the row sum and lse are the
undropped ones; empty rows stay +0.0 / -inf."""
import numpy as np
import pytest
import torch

import oracle
import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL, check_grad, compare, cpu32, dq_c_term, empty_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(a, keep, p, **kw):
    mask = wl.pack_keep_mask(keep)
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=a.causal,
                          scale=a.scale, dropout_mask=mask, dropout_p=p, **kw)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    return o, lse


def ref(a, keep, p):
    return oracle.attn_fwd_dropout(cpu32(a.q), cpu32(a.k), cpu32(a.v), keep.cpu(), p, bias=cpu32(a.bias),
                                   kv_lens=None if a.kv_lens is None else a.kv_lens.cpu(),
                                   causal=a.causal, scale=a.scale)


@pytest.mark.parametrize("dk,dv,causal,bias,p", [
    (128, 128, True, False, 0.2),
    (64, 64, False, True, 0.5),
    (128, 64, True, False, 0.1),
    (64, 128, True, True, 0.3),
])
def test_bf16_dropout_matches_oracle(dk, dv, causal, bias, p):
    a = wl.make_prefill(2, 3, 300, 333, dk, dv, torch.bfloat16, causal=causal, bias=bias,
                        kv_lens=[333, 170], seed=41, device=DEV)
    keep = wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, p, seed=7, device=DEV)
    o, lse = run(a, keep, p)
    o_ref, l_ref = ref(a, keep, p)
    tol = TOL[torch.bfloat16]["o"] / (1.0 - p)  # kept weights are scaled up by 1 / (1 - p)
    err = float(np.max(np.abs(o.float().cpu().numpy() - o_ref)))
    assert err <= tol, (err, tol)
    compare(torch.zeros_like(o), lse, np.zeros_like(o_ref), l_ref, torch.bfloat16, empty=empty_rows(a),
            what="lse with dropout")


def test_bf16_dropout_all_kept_is_bitwise_the_forward():
    a = wl.make_prefill(2, 2, 260, 260, 128, 128, torch.bfloat16, causal=True, kv_lens=[260, 99],
                        seed=42, device=DEV)
    keep = torch.ones((a.B, a.H, a.Nq, a.Nk), dtype=torch.bool, device=DEV)
    o1, l1 = run(a, keep, 0.0)
    o0, l0 = ofa.attn_fwd(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=True, scale=a.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o0.view(torch.int16)) and torch.equal(l1, l0)


def test_bf16_dropout_lse_is_the_undropped_one():
    a = wl.make_prefill(1, 2, 200, 200, 128, 128, torch.bfloat16, causal=True, seed=43, device=DEV)
    o0, l0 = ofa.attn_fwd(a.q, a.k, a.v, causal=True, scale=a.scale)
    keep = wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, 0.6, seed=8, device=DEV)
    _, l1 = run(a, keep, 0.6)
    assert torch.equal(l0, l1)


def test_fp32_dropout_matches_oracle():
    a = wl.make_prefill(1, 2, 70, 90, 32, 48, torch.float32, causal=True, kv_lens=[77], seed=44,
                        device=DEV)
    keep = wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, 0.25, seed=9, device=DEV)
    o, lse = run(a, keep, 0.25, block_k=32)
    o_ref, l_ref = ref(a, keep, 0.25)
    compare(o, lse, o_ref, l_ref, torch.float32, what="fp32 dropout")


def test_bf16_dropout_full_size_sampled_heads():
    # the 2k causal prefill workload with p = 0.1, two heads checked against the oracle
    a = wl.causal_2k(DEV)
    keep = wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, 0.1, seed=10, device=DEV)
    o, lse = run(a, keep, 0.1)
    for (b, h) in [(0, 0), (3, 15)]:
        sub = wl.make_prefill(1, 1, a.Nq, a.Nk, a.dk, a.dv, torch.bfloat16, causal=True, seed=0, device="cpu")
        sub.q, sub.k, sub.v = (t[b:b + 1, :, h:h + 1].cpu() for t in (a.q, a.k, a.v))
        o_ref, l_ref = ref(sub, keep[b:b + 1, h:h + 1], 0.1)
        err = float(np.max(np.abs(o[b, :, h].float().cpu().numpy() - o_ref[0, :, 0])))
        assert err <= TOL[torch.bfloat16]["o"] / 0.9, (b, h, err)
        assert float(np.max(np.abs(lse[b, h].cpu().numpy() - l_ref[0, 0]))) <= TOL[torch.bfloat16]["lse"]


# ---- backward of the dropout forward (the d = 128 tcgen05 kernel)

def run_bwd_drop(a, keep, p, seed=0):
    mask = wl.pack_keep_mask(keep)
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=a.causal, scale=a.scale,
                          dropout_mask=mask, dropout_p=p)
    g = torch.Generator(device=DEV)
    g.manual_seed(2000 + seed)
    dout = torch.randn(o.shape, generator=g, device=DEV).to(o.dtype)
    grads = ofa.attn_bwd(a.q, a.k, a.v, o, lse, dout, kv_lens=a.kv_lens, causal=a.causal, scale=a.scale,
                         dropout_mask=mask, dropout_p=p)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    run_bwd_drop.last_o = o
    return dout, grads


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,p,lens", [(True, 0.2, [333, 170]), (False, 0.5, [301, 333])])
def test_bwd_dropout_matches_oracle(causal, p, lens, d):
    a = wl.make_prefill(2, 2, 300, 333, d, d, torch.bfloat16, causal=causal, kv_lens=lens, seed=45,
                        device=DEV)
    keep = wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, p, seed=11, device=DEV)
    dout, grads = run_bwd_drop(a, keep, p)
    refs = oracle.attn_bwd_dropout(cpu32(a.q), cpu32(a.k), cpu32(a.v), cpu32(dout), keep.cpu(), p,
                                   kv_lens=a.kv_lens.cpu(), causal=causal, scale=a.scale)
    ct = dq_c_term(dout, run_bwd_drop.last_o, a.k, a.scale, a.kv_lens)
    for got, ref, name in zip(grads, refs, ("dq", "dk", "dv")):
        check_grad(got, ref, f"{name} causal={causal} p={p}", extra=ct if name == "dq" else None)
    # keys past the sequence get +0.0 exactly
    for t in grads[1:]:
        bits = t.view(torch.int16).cpu().numpy()
        assert np.all(bits[1, lens[1]:] == 0)


def test_bwd_dropout_all_kept_is_bitwise_the_backward():
    a = wl.make_prefill(2, 2, 260, 260, 128, 128, torch.bfloat16, causal=True, kv_lens=[260, 99], seed=46,
                        device=DEV)
    keep = torch.ones((a.B, a.H, a.Nq, a.Nk), dtype=torch.bool, device=DEV)
    dout, (dq1, dk1, dv1) = run_bwd_drop(a, keep, 0.0)
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=True, scale=a.scale)
    dq0, dk0, dv0 = ofa.attn_bwd(a.q, a.k, a.v, o, lse, dout, kv_lens=a.kv_lens, causal=True, scale=a.scale)
    torch.cuda.synchronize()
    assert torch.equal(dk1.view(torch.int16), dk0.view(torch.int16))
    assert torch.equal(dv1.view(torch.int16), dv0.view(torch.int16))
    # dQ is added with atomics in a varying order: equal within its last bits
    assert (dq1.float() - dq0.float()).abs().max().item() <= 1e-2 * max(1.0, dq0.float().abs().max().item())


def test_bwd_dropout_full_size_one_head():
    # the 2k causal workload with p = 0.1: one (b, h) head against the oracle
    a = wl.causal_2k(DEV)
    keep = wl.dropout_keep(a.B, a.H, a.Nq, a.Nk, 0.1, seed=12, device=DEV)
    dout, grads = run_bwd_drop(a, keep, 0.1, seed=3)
    b, h = 2, 9
    sl = lambda t: cpu32(t[b:b + 1, :, h:h + 1])
    refs = oracle.attn_bwd_dropout(sl(a.q), sl(a.k), sl(a.v), sl(dout), keep[b:b + 1, h:h + 1].cpu(), 0.1,
                                   causal=True, scale=a.scale)
    ct = dq_c_term(sl(dout), sl(run_bwd_drop.last_o), sl(a.k), a.scale)
    for got, ref, name in zip(grads, refs, ("dq", "dk", "dv")):
        check_grad(got[b:b + 1, :, h:h + 1], ref, f"{name} full-size head", extra=ct if name == "dq" else None)


# ---------------------------------------------------------------- keep decisions drawn in-kernel
# (Philox4x32-10, include/attn.h dropout_rng).  The oracle restates the generator
# (oracle/philox.py, pinned to the published known-answer vectors) and draws the same
# decisions; feeding them to the kernel as a mask must give the same output bit for bit, and
# both must match the dropout oracle.

from oracle import philox as _philox  # noqa: E402


def _rng_keep(a, seed, offset, p):
    keep, p_real = _philox.keep_mask(seed, offset, a.B, a.H, a.Nq, a.Nk, p)
    return torch.from_numpy(keep).to(DEV), p_real


@pytest.mark.parametrize("dk,dv,causal,bias,p", [
    (128, 128, True, False, 0.2),
    (64, 64, False, True, 0.5),
    (128, 64, True, False, 0.1),
])
def test_bf16_in_kernel_draws_equal_the_oracles_generator(dk, dv, causal, bias, p):
    a = wl.make_prefill(2, 3, 300, 333, dk, dv, torch.bfloat16, causal=causal, bias=bias,
                        kv_lens=[333, 170], seed=47, device=DEV)
    seed, offset = 0x0123_4567_89AB_CDEF, 11
    o1, l1 = ofa.attn_fwd(a.q, a.k, a.v, bias=a.bias, kv_lens=a.kv_lens, causal=causal, scale=a.scale,
                          dropout_p=p, dropout_seed=seed, dropout_offset=offset)
    keep, p_real = _rng_keep(a, seed, offset, p)
    o2, l2 = run(a, keep, p_real)  # the same decisions, as a keep mask
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)
    o_ref, l_ref = ref(a, keep, p_real)
    err = float(np.max(np.abs(o1.float().cpu().numpy() - o_ref)))
    assert err <= TOL[torch.bfloat16]["o"] / (1.0 - p_real), err


def test_fp32_in_kernel_draws_equal_the_oracles_generator():
    a = wl.make_prefill(1, 2, 100, 130, 64, 64, torch.float32, causal=True, kv_lens=[130], seed=48, device=DEV)
    seed, offset, p = 99, 3, 0.3
    o1, l1 = ofa.attn_fwd(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=True, scale=a.scale, dropout_p=p,
                          dropout_seed=seed, dropout_offset=offset)
    keep, p_real = _rng_keep(a, seed, offset, p)
    o_ref, l_ref = ref(a, keep, p_real)
    torch.cuda.synchronize()
    assert np.max(np.abs(o1.cpu().numpy() - o_ref)) <= 1e-5 / (1.0 - p_real)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,p,lens", [(True, 0.2, [333, 170]), (False, 0.5, [301, 333])])
def test_bwd_in_kernel_draws_match_oracle(causal, p, lens, d):
    a = wl.make_prefill(2, 2, 300, 333, d, d, torch.bfloat16, causal=causal, kv_lens=lens, seed=49,
                        device=DEV)
    seed, offset = 1234567, 5
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, kv_lens=a.kv_lens, causal=causal, scale=a.scale, dropout_p=p,
                          dropout_seed=seed, dropout_offset=offset)
    g = torch.Generator(device=DEV)
    g.manual_seed(2100)
    dout = torch.randn(o.shape, generator=g, device=DEV).to(o.dtype)
    grads = ofa.attn_bwd(a.q, a.k, a.v, o, lse, dout, kv_lens=a.kv_lens, causal=causal, scale=a.scale,
                         dropout_p=p, dropout_seed=seed, dropout_offset=offset)
    keep, p_real = _rng_keep(a, seed, offset, p)
    # the backward with the oracle's decisions as a mask: bit for bit the same dK and dV
    grads_m = ofa.attn_bwd(a.q, a.k, a.v, o, lse, dout, kv_lens=a.kv_lens, causal=causal, scale=a.scale,
                           dropout_mask=wl.pack_keep_mask(keep), dropout_p=p_real)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    assert torch.equal(grads[1].view(torch.int16), grads_m[1].view(torch.int16))
    assert torch.equal(grads[2].view(torch.int16), grads_m[2].view(torch.int16))
    refs = oracle.attn_bwd_dropout(cpu32(a.q), cpu32(a.k), cpu32(a.v), cpu32(dout), keep.cpu(), p_real,
                                   kv_lens=a.kv_lens.cpu(), causal=causal, scale=a.scale)
    ct = dq_c_term(dout, o, a.k, a.scale, a.kv_lens)
    for got, r, name in zip(grads, refs, ("dq", "dk", "dv")):
        check_grad(got, r, f"{name} in-kernel draws causal={causal} p={p}", extra=ct if name == "dq" else None)


def test_full_size_forward_in_kernel_draws_one_head():
    a = wl.causal_2k(DEV)
    seed, offset, p = 77, 1, 0.1
    o, lse = ofa.attn_fwd(a.q, a.k, a.v, causal=True, scale=a.scale, dropout_p=p, dropout_seed=seed,
                          dropout_offset=offset)
    torch.cuda.synchronize()
    b, h = 1, 6
    keep, p_real = _philox.keep_mask(seed, offset, a.B, a.H, a.Nq, a.Nk, p, heads=[(b, h)])
    sl = lambda t: cpu32(t[b:b + 1, :, h:h + 1])
    o_ref, l_ref = oracle.attn_fwd_dropout(sl(a.q), sl(a.k), sl(a.v), torch.from_numpy(keep)[None], p_real,
                                           causal=True, scale=a.scale)
    err = float(np.max(np.abs(o[b:b + 1, :, h:h + 1].float().cpu().numpy() - o_ref)))
    assert err <= TOL[torch.bfloat16]["o"] / (1.0 - p_real), err
