"""GPU parity of split-KV decode and of the (m, l, u) merge kernel against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import online_softmax_fa2_gb300 as ofa
from online_softmax_fa2_gb300 import workloads as wl
from helpers import TOL, compare, cpu32, oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_decode(a, num_splits=None):
    o, lse, ws = ofa.attn_decode_splitkv(a.q, a.k, a.v, kv_lens=a.kv_lens, bias=a.bias,
                                         num_splits=num_splits or a.num_splits, scale=a.scale)
    torch.cuda.synchronize()
    assert ofa.device_error_flags() & 1 == 0
    return o, lse, ws


def oracle_head(a, b, h):
    """Oracle on one (b, h) of a decode workload, keys cut at that sequence's kv_len."""
    n = a.kv_len_list()[b]
    q = cpu32(a.q[b:b + 1, :, h:h + 1])
    k = cpu32(a.k[b:b + 1, :n, h:h + 1])
    v = cpu32(a.v[b:b + 1, :n, h:h + 1])
    bias = None if a.bias is None else cpu32(a.bias[b:b + 1, h:h + 1, :, :n])
    o, lse, _ = oracle.attn_fwd(q, k, v, bias=bias, scale=a.scale)
    return o[0, 0, 0], lse[0, 0, 0]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [1, 2, 16, 37])
def test_decode_small_matches_oracle(d, splits):
    a = wl.decode(DEV, seed=31, B=5, H=3, L=700, d=d, num_splits=splits,
                  lens=[1, 700, 0, 333, 17])
    o, lse, ws = run_decode(a)
    # the oracle on the whole problem (kv_len 0 gives empty rows)
    o_ref, l_ref, _ = oracle.attn_fwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), kv_lens=a.kv_lens.cpu(),
                                      scale=a.scale)
    compare(o, lse, o_ref, l_ref, torch.bfloat16, what=f"decode d={d} S={splits}")


def test_decode_partials_are_the_split_states():
    # the workspace holds each split's (m, l, u) over keys [s*n/S, (s+1)*n/S)
    S = 16
    a = wl.decode(DEV, seed=32, B=4, H=2, L=600, d=128, num_splits=S, lens=[600, 5, 0, 257])
    _, _, ws = run_decode(a)
    part = ws[: 4 * 2 * S * 130].view(4, 2, S, 130).cpu().double().numpy()
    for b, n in enumerate(a.kv_len_list()):
        for h in range(2):
            q = cpu32(a.q[b:b + 1, :, h:h + 1])
            k = cpu32(a.k[b:b + 1, :, h:h + 1])
            v = cpu32(a.v[b:b + 1, :, h:h + 1])
            for s in range(S):
                lo, hi = (s * n) // S, ((s + 1) * n) // S
                st = oracle.key_state(q, k, v, lo, hi, scale=a.scale)[0, 0, 0]
                g = part[b, h, s]
                if hi == lo:
                    assert g[0] == -np.inf and g[1] == 0 and np.all(g[2:] == 0)
                    continue
                # states are compared after a common re-basing to the oracle's maximum
                f = math.exp(g[0] - st[0])
                assert abs(g[0] - st[0]) < 1e-4
                assert abs(f * g[1] - st[1]) <= 1e-3 * st[1]
                assert np.max(np.abs(f * g[2:] - st[2:])) <= 2e-3 * max(1.0, st[1])


def test_decode_bias_and_masks():
    a = wl.decode(DEV, seed=33, B=3, H=2, L=300, d=128, num_splits=7, lens=[300, 40, 299])
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    bias = torch.randn((3, 2, 1, 300), generator=g, device=DEV)
    bias[:, :, :, ::7] = -math.inf
    a.bias = bias
    o, lse, _ = run_decode(a)
    for b in range(3):
        for h in range(2):
            o_ref, l_ref = oracle_head(a, b, h)
            assert np.max(np.abs(o[b, 0, h].float().cpu().numpy() - o_ref)) <= TOL[torch.bfloat16]["o"]
            assert abs(lse[b, h, 0].item() - l_ref) <= TOL[torch.bfloat16]["lse"]


def test_decode_split_invariance_and_poison():
    a = wl.decode(DEV, seed=34, B=3, H=4, L=1000, d=128, num_splits=16, lens=[1000, 999, 3])
    outs = [run_decode(a, S)[:2] for S in (1, 2, 16, 37)]
    for o, l in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert (l - outs[0][1]).abs().max().item() <= 1e-3
    clean = wl.decode(DEV, seed=34, B=3, H=4, L=1000, d=128, num_splits=16, lens=[1000, 999, 3],
                      poison=False)
    o1, l1, _ = run_decode(clean)
    o2, l2, _ = run_decode(a)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_merge_kernel_matches_oracle_merge():
    rng = np.random.default_rng(35)
    B, H, S, dv = 3, 5, 9, 128
    st = np.zeros((B, H, S, 2 + dv), np.float32)
    st[..., 0] = rng.normal(0, 5, (B, H, S))
    st[..., 1] = rng.uniform(1, 50, (B, H, S))
    st[..., 2:] = rng.normal(0, 3, (B, H, S, dv))
    empty = rng.random((B, H, S)) < 0.3
    empty[1, 2, :] = True  # a row whose parts are all empty
    st[empty, 0] = -np.inf
    st[empty, 1] = 0
    st[empty, 2:] = 0
    part = torch.from_numpy(st).to(DEV)
    for dt in (torch.float32, torch.bfloat16):
        o, lse = ofa.attn_merge_states(part, out_dtype=dt)
        torch.cuda.synchronize()
        o_ref, l_ref = oracle.merge_states(st.astype(np.float64))
        og = o[:, 0].float().cpu().numpy()
        lg = lse[:, :, 0].cpu().numpy()
        fin = np.isfinite(l_ref)
        tol = 1e-5 if dt == torch.float32 else 2e-2
        assert np.max(np.abs(og - o_ref) / (1 + np.abs(o_ref))) <= tol
        assert np.max(np.abs(lg[fin] - l_ref[fin])) <= 1e-5 * (1 + np.max(np.abs(l_ref[fin])))
        assert np.all(lg[~fin] == -np.inf) and np.all(og[~fin] == 0)


def test_decode_b64_h32_l8192_d128_sampled():
    a = wl.decode(DEV)
    o, lse, _ = run_decode(a)
    lens = a.kv_len_list()
    rng = np.random.default_rng(36)
    pairs = {(0, 0), (63, 31), (0, 31), (63, 0)}
    pairs |= {(int(b), int(h)) for b, h in zip(rng.integers(0, 64, 40), rng.integers(0, 32, 40))}
    for b, h in sorted(pairs):
        o_ref, l_ref = oracle_head(a, b, h)
        err = np.max(np.abs(o[b, 0, h].float().cpu().numpy() - o_ref))
        assert err <= TOL[torch.bfloat16]["o"], (b, h, lens[b], err)
        assert abs(lse[b, h, 0].item() - l_ref) <= TOL[torch.bfloat16]["lse"]
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
