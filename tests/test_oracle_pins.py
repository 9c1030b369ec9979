"""Pins of the float64 oracle to facts the pages and the mathematics fix.

Every check here runs on the CPU (no GPU, no CUDA library).  Each one pins the oracle to
something other than itself: a value a page prints for a worked example (fixtures under
tests/golden/, each with its source), a closed form, an invariant, a special case that a
library routine computes independently (torch's float64 math attention), or the pages'
own merge of per-key-set states restated in pure Python.
"""
import itertools
import json
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
from oracle import online_ref

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def printed_tol(g):
    # values printed with d decimals, "rounded after calculation at full precision"
    return 0.5 * 10.0 ** (-g.get("printed_decimals", 3)) + 1e-12


def one_query(scores, values, scale=1.0):
    """Encode one query row with given logits: dk = 1, q = [1], k_j = [s_j]."""
    q = np.ones((1, 1, 1, 1), np.float32)
    k = np.asarray(scores, np.float32).reshape(1, -1, 1, 1)
    v = np.asarray(values, np.float32).reshape(1, len(values), 1, -1)
    return q, k, v, scale


# ---------------------------------------------------------------- worked examples

def test_p1_s2_global_output_three_quarters():
    g = gold("p1_s2_tile_local_counterexample.json")
    q, k, v, _ = one_query([0.0, 1.0], g["values"])
    o, lse, _ = oracle.attn_fwd(q, k, v, scale=math.log(3.0))
    assert abs(o[0, 0, 0, 0] - g["printed"]["output"]) < 1e-15
    assert abs(lse[0, 0, 0] - math.log(4.0)) < 1e-15
    p = oracle.attn_probs(q, k, v, scale=math.log(3.0))[0, 0, 0]
    assert np.allclose(p, g["printed"]["global_weights"], atol=1e-15, rtol=0)
    # each one-key tile alone: local weight one, local outputs 0 and 1
    locals_ = []
    for j in range(2):
        oj, _, _ = oracle.attn_fwd(q, k[:, j:j + 1], v[:, j:j + 1], scale=math.log(3.0))
        locals_.append(oj[0, 0, 0, 0])
    assert locals_ == g["printed"]["tile_local_outputs"]
    assert sum(locals_) == g["printed"]["tile_local_sum"]
    assert sum(locals_) / 2 == g["printed"]["tile_local_average"]
    # the correct answer is neither of the wrong combinations
    assert abs(o[0, 0, 0, 0] - sum(locals_)) > 0.2
    assert abs(o[0, 0, 0, 0] - sum(locals_) / 2) > 0.2


def _rescale_l_only(scores, values):
    """The wrong update of section 4: rescales l but not u (planted here, never in code)."""
    m, l, u = -math.inf, 0.0, [0.0] * len(values[0])
    for s, vv in zip(scores, values):
        mn = max(m, s)
        alpha = math.exp(m - mn) if m > -math.inf else 0.0
        l = alpha * l + math.exp(s - mn)
        u = [c + math.exp(s - mn) * x for c, x in zip(u, vv)]  # u NOT rescaled
        m = mn
    return [c / l for c in u]


def test_p1_s4_both_accumulators_rescaled():
    g = gold("p1_s4_rescale_u_counterexample.json")
    q, k, v, _ = one_query([0.0, 1.0], g["values"])
    o, _, _ = oracle.attn_fwd(q, k, v, scale=math.log(3.0))
    assert abs(o[0, 0, 0, 0] - g["printed"]["output"]) < 1e-15
    # the planted bug gives the printed wrong answer, and the oracle does not
    bad = _rescale_l_only([0.0, math.log(3.0)], g["values"])[0]
    assert abs(bad - g["printed"]["rescale_l_only_output"]) < 1e-15
    assert abs(o[0, 0, 0, 0] - bad) > 0.4
    # alpha = exp(m_old - m_new) = 1/3
    s0 = oracle.key_state(q, k[:, :1], v[:, :1], 0, 1, scale=math.log(3.0))[0, 0, 0]
    sall = oracle.key_state(q, k, v, 0, 2, scale=math.log(3.0))[0, 0, 0]
    assert abs(math.exp(s0[0] - sall[0]) - g["printed"]["alpha"]) < 1e-15


def test_p3_fig1_deferred_division():
    g = gold("p3_fig1_deferred_division.json")
    t = printed_tol(g)
    q, k, v, _ = one_query(g["scores"], g["values"])
    o, lse, _ = oracle.attn_fwd(q, k, v, scale=1.0)
    st = oracle.key_state(q, k, v, 0, 2, scale=1.0)[0, 0, 0]
    pr = g["printed"]
    assert st[0] == pr["m"]
    assert abs(st[1] - pr["l"]) <= t
    assert np.all(np.abs(st[2:] - pr["a"]) <= t)
    assert np.all(np.abs(o[0, 0, 0] - pr["output"]) <= t)
    p = oracle.attn_probs(q, k, v, scale=1.0)[0, 0, 0]
    assert np.all(np.abs(p - pr["probs"]) <= t)
    # closed form: o = (e^-1 * [2,0] + [0,2]) / (1 + e^-1)
    e = math.exp(-1.0)
    assert np.allclose(o[0, 0, 0], [2 * e / (1 + e), 2 / (1 + e)], atol=1e-15, rtol=0)
    assert abs(lse[0, 0, 0] - (2.0 + math.log(1 + e))) < 1e-15


def test_p3_fig2_states_after_each_chunk():
    g = gold("p3_fig2_six_scores_three_chunks.json")
    t = printed_tol(g)
    q, k, v, _ = one_query(g["scores"], g["values"])
    pr = g["printed"]
    for ch in pr["after_chunk"]:
        j0, j1 = ch["keys"]
        st = oracle.key_state(q, k, v, j0, j1, scale=1.0)[0, 0, 0]
        assert st[0] == ch["m"]
        assert abs(st[1] - ch["l"]) <= t
        assert np.all(np.abs(st[2:] - ch["a"]) <= t)
    c2 = oracle.key_state(q, k, v, 2, 4, scale=1.0)[0, 0, 0]  # chunk 2 alone, m = 1
    # chunk 2's mass and weighted sum measured against the running maximum 2
    f = math.exp(c2[0] - 2.0)
    assert abs(f * c2[1] - pr["chunk2_mass"]) <= t
    assert np.all(np.abs(f * c2[2:] - pr["chunk2_weighted"]) <= t)
    s4 = oracle.key_state(q, k, v, 0, 4, scale=1.0)[0, 0, 0]
    alpha = math.exp(s4[0] - 3.0)
    assert abs(alpha - pr["rescale_factor"]) <= t
    assert abs(alpha * s4[1] - pr["rescaled_l"]) <= t
    assert np.all(np.abs(alpha * s4[2:] - pr["rescaled_a"]) <= t)
    c3 = oracle.key_state(q, k, v, 4, 6, scale=1.0)[0, 0, 0]
    assert c3[0] == 3.0
    assert abs(c3[1] - pr["chunk3_mass"]) <= t
    assert np.all(np.abs(c3[2:] - pr["chunk3_weighted"]) <= t)
    o, _, _ = oracle.attn_fwd(q, k, v, scale=1.0)
    assert np.all(np.abs(o[0, 0, 0] - pr["output"]) <= t)


def test_p2_step6_two_tiles_merge():
    g = gold("p2_step6_two_tiles.json")
    t = printed_tol(g)
    q = np.asarray(g["q"], np.float32).reshape(1, 1, 1, 2)
    k = np.asarray(g["k"], np.float32).reshape(1, 4, 1, 2)
    v = np.asarray(g["values"], np.float32).reshape(1, 4, 1, 2)
    sc = 1.0 / math.sqrt(2.0)
    pr = g["printed"]
    states = []
    for tile in pr["tiles"]:
        j0, j1 = tile["keys"]
        st = oracle.key_state(q, k, v, j0, j1, scale=sc)[0, 0, 0]
        assert abs(st[0] - tile["m"]) <= t
        assert abs(st[1] - tile["l"]) <= t
        assert np.all(np.abs(st[2:] - tile["o_tilde"]) <= t)
        states.append(st)
    whole = oracle.key_state(q, k, v, 0, 4, scale=sc)[0, 0, 0]
    assert abs(whole[1] - pr["merged_l"]) <= t
    assert np.all(np.abs(whole[2:] - pr["merged_o_tilde"]) <= t)
    o, _, _ = oracle.attn_fwd(q, k, v, scale=sc)
    assert np.all(np.abs(o[0, 0, 0] - pr["output"]) <= t)
    om, _ = oracle.merge_states(np.stack(states)[None])
    assert np.allclose(om[0], o[0, 0, 0], atol=1e-15, rtol=0)


def test_p3_fig3_two_queries():
    g = gold("p3_fig3_two_queries_two_tiles.json")
    t = printed_tol(g)
    q = np.asarray(g["q"], np.float32).reshape(1, 2, 1, 2)
    k = np.asarray(g["k"], np.float32).reshape(1, 4, 1, 2)
    v = np.asarray(g["values"], np.float32).reshape(1, 4, 1, 2)
    pr = g["printed"]
    # the printed score tiles are reproduced by the inferred K
    s = q[0, :, 0] @ k[0, :, 0].T
    assert np.array_equal(s[:, :2], pr["tile1_scores"])
    assert np.array_equal(s[:, 2:], pr["tile2_scores"])
    t1 = oracle.key_state(q, k, v, 0, 2, scale=1.0)[0, 0]
    assert np.all(np.abs(t1[:, 1] - pr["tile1_l"]) <= t)
    assert np.all(np.abs(t1[:, 2:] - np.asarray(pr["tile1_a"])) <= t)
    fin = oracle.key_state(q, k, v, 0, 4, scale=1.0)[0, 0]
    assert np.all(np.abs(fin[:, 1] - pr["final_l"]) <= t)
    assert np.all(np.abs(fin[:, 2:] - np.asarray(pr["final_a"])) <= t)
    o, _, _ = oracle.attn_fwd(q, k, v, scale=1.0)
    assert np.all(np.abs(o[0, :, 0] - np.asarray(pr["output"])) <= t)


def test_p1_s6_bottom_right_visible_sets():
    g = gold("p1_s6_bottom_right_mask.json")
    rng = np.random.default_rng(7)
    for case in g["cases"]:
        nq, nk = case["Nq"], case["Nk"]
        q = rng.standard_normal((1, nq, 1, 3)).astype(np.float32)
        k = rng.standard_normal((1, nk, 1, 3)).astype(np.float32)
        v = rng.standard_normal((1, nk, 1, 2)).astype(np.float32)
        p = oracle.attn_probs(q, k, v, causal=True)[0, 0]
        for i in range(nq):
            vis = [j for j in range(nk) if p[i, j] > 0]
            assert vis == case["visible"][i]
            assert all(p[i, j] == 0.0 for j in range(nk) if j not in vis)
        if "top_left_visible" in case:
            assert case["top_left_visible"] != case["visible"]
        o, lse, _ = oracle.attn_fwd(q, k, v, causal=True)
        for i in range(nq):
            if not case["visible"][i]:
                assert np.all(o[0, i, 0] == 0.0) and not np.any(np.signbit(o[0, i, 0]))
                assert lse[0, 0, i] == -math.inf


# ---------------------------------------------------------------- closed forms, invariants

def rand_problem(rng, B, H, Nq, Nk, dk, dv, bias=False, kv=None, mask_p=0.0):
    q = rng.standard_normal((B, Nq, H, dk)).astype(np.float32)
    k = rng.standard_normal((B, Nk, H, dk)).astype(np.float32)
    v = rng.standard_normal((B, Nk, H, dv)).astype(np.float32)
    b = None
    if bias:
        b = rng.standard_normal((B, H, Nq, Nk)).astype(np.float32)
        if mask_p > 0:
            b[rng.random(b.shape) < mask_p] = -np.inf
    kvl = None if kv is None else np.asarray(kv, np.int32)
    return q, k, v, b, kvl


def test_empty_key_axis_and_empty_rows_exact():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((2, 2, 1, 3)).astype(np.float32)
    k = np.zeros((2, 0, 1, 3), np.float32)
    v = np.zeros((2, 0, 1, 2), np.float32)
    o, lse, _ = oracle.attn_fwd(q, k, v)
    assert np.all(o == 0.0) and not np.any(np.signbit(o))
    assert np.all(lse == -np.inf)
    # kv_len = 0 on one sequence and a row whose whole bias is -inf
    q, k, v, b, kvl = rand_problem(rng, 2, 2, 3, 4, 3, 2, bias=True, kv=[0, 4])
    b[1, 1, 2, :] = -np.inf
    o, lse, _ = oracle.attn_fwd(q, k, v, bias=b, kv_lens=kvl)
    assert np.all(o[0] == 0.0) and np.all(lse[0] == -np.inf)
    assert np.all(o[1, 2, 1] == 0.0) and lse[1, 1, 2] == -np.inf
    assert np.all(np.isfinite(lse[1, 0])) and np.all(np.isfinite(o[1, :, 0]))


def test_all_logits_equal_gives_plain_mean():
    # Visual walkthrough, Step 7: equal scores -> every exponent 1, l = count, plain average
    rng = np.random.default_rng(2)
    q = np.zeros((1, 3, 1, 4), np.float32)
    k = rng.standard_normal((1, 7, 1, 4)).astype(np.float32)
    v = rng.standard_normal((1, 7, 1, 3)).astype(np.float32)
    o, lse, _ = oracle.attn_fwd(q, k, v, causal=True)
    for i in range(3):
        n = i + 7 - 3 + 1
        assert np.allclose(o[0, i, 0], v[0, :n, 0].astype(np.float64).mean(0), atol=1e-15,
                           rtol=0)
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-15
    st = oracle.key_state(q, k, v, 0, 7)[0, 0]
    assert np.all(st[:, 0] == 0.0) and np.all(st[:, 1] == 7.0)


def test_one_dominating_logit_selects_its_value():
    # Visual walkthrough, Step 7 and the page-1 counterexample: a growing gap drives the
    # output to the dominating key's value
    rng = np.random.default_rng(3)
    v = rng.standard_normal((1, 5, 1, 3)).astype(np.float32)
    for gap in (10.0, 30.0, 700.0):
        scores = [0.0, 1.0, gap, -2.0, 0.5]
        q, k, _, _ = one_query(scores, np.zeros((5, 3)))
        o, lse, _ = oracle.attn_fwd(q, k, v, scale=1.0)
        err = np.max(np.abs(o[0, 0, 0] - v[0, 2, 0]))
        assert err <= 5.0 * math.exp(-(gap - 1.0)) * np.max(np.abs(v)) + 1e-15
        assert abs(lse[0, 0, 0] - gap) < 1e-12 * gap + 5 * math.exp(-(gap - 1.0))


def test_common_logit_shift_and_wide_span():
    # page 1, section 9 family "common logit shifts and wide span": adding c to a row's
    # logits leaves O unchanged and moves lse by c; huge logits do not overflow
    rng = np.random.default_rng(4)
    q, k, v, b, _ = rand_problem(rng, 1, 2, 3, 5, 2, 2, bias=True)
    b = (np.round(b * 1024.0) / 1024.0).astype(np.float32)  # so that b + c is exact in fp32
    o0, l0, _ = oracle.attn_fwd(q, k, v, bias=b)
    for c in (-50.0, 3.0, 600.0):
        o1, l1, _ = oracle.attn_fwd(q, k, v, bias=b + np.float32(c))
        assert np.allclose(o1, o0, atol=1e-12, rtol=0)
        assert np.allclose(l1 - l0, c, atol=1e-12 * (1 + abs(c)), rtol=0)
    # wide span: logits 0 and 1000 (exp(1000) overflows binary64 without the max shift)
    q, k, v2, _ = one_query([0.0, 1000.0, 990.0], [[1.0], [2.0], [3.0]])
    o, lse, _ = oracle.attn_fwd(q, k, v2, scale=1.0)
    e = math.exp(-10.0)
    assert abs(o[0, 0, 0, 0] - (2.0 + 3.0 * e + math.exp(-1000.0)) / (1.0 + e)) < 1e-14
    assert abs(lse[0, 0, 0] - (1000.0 + math.log1p(e))) < 1e-12


def test_weights_sum_to_one_masked_zero_and_l_bounds():
    # page 1, sections 1 and 3: weights sum to one on every nonempty row, masked positions
    # weigh zero, and 1 <= l <= n for n visible logits in the max frame
    rng = np.random.default_rng(5)
    q, k, v, b, kvl = rand_problem(rng, 2, 3, 6, 9, 4, 3, bias=True, kv=[9, 5], mask_p=0.2)
    for causal in (False, True):
        p = oracle.attn_probs(q, k, v, bias=b, kv_lens=kvl, causal=causal)
        st = oracle.key_state(q, k, v, 0, 9, bias=b, kv_lens=kvl, causal=causal)
        for bb in range(2):
            n = int(kvl[bb])
            for h in range(3):
                for i in range(6):
                    vis = [j for j in range(9) if j < n and not np.isneginf(b[bb, h, i, j])
                           and (not causal or j <= i + n - 6)]
                    row = p[bb, h, i]
                    assert np.all(row[[j for j in range(9) if j not in vis]] == 0.0)
                    if vis:
                        assert abs(row.sum() - 1.0) < 1e-14
                        assert np.all(row[vis] > 0)
                        assert 1.0 <= st[bb, h, i, 1] <= len(vis)
                    else:
                        assert np.all(row == 0.0) and st[bb, h, i, 1] == 0.0


def test_masked_positions_are_never_read():
    # page 1, sections 1 and 6: masked positions have zero weight, so whatever is stored
    # there (NaN, inf) must not change a single bit of the result
    rng = np.random.default_rng(6)
    q, k, v, b, kvl = rand_problem(rng, 3, 2, 5, 8, 3, 4, bias=True, kv=[8, 3, 0])
    o0, l0, _ = oracle.attn_fwd(q, k, v, bias=b, kv_lens=kvl, causal=True)
    k2, v2, b2 = k.copy(), v.copy(), b.copy()
    for bb, n in enumerate(kvl):
        k2[bb, n:] = np.nan
        v2[bb, n:] = np.inf
        for i in range(5):
            for j in range(8):
                if j >= n or j > i + n - 5:
                    b2[bb, :, i, j] = np.nan
    o1, l1, _ = oracle.attn_fwd(q, k2, v2, bias=b2, kv_lens=kvl, causal=True)
    assert o0.tobytes() == o1.tobytes() and l0.tobytes() == l1.tobytes()


def test_matches_library_attention_in_float64():
    # special case that a library routine computes independently: torch's float64 math
    # attention (an additive float mask is a bias that is not scaled; is_causal on a square
    # problem is the same as bottom-right)
    rng = np.random.default_rng(8)
    for (B, H, Nq, Nk, dk, dv, causal, bias) in [
            (2, 3, 7, 7, 5, 2, True, False), (1, 2, 5, 9, 4, 3, False, True),
            (2, 1, 16, 16, 8, 6, True, False), (1, 1, 4, 11, 3, 7, False, False)]:
        q, k, v, b, _ = rand_problem(rng, B, H, Nq, Nk, dk, dv, bias=bias)
        o, lse, _ = oracle.attn_fwd(q, k, v, bias=b, causal=causal)
        tq = torch.from_numpy(q).double().permute(0, 2, 1, 3)
        tk = torch.from_numpy(k).double().permute(0, 2, 1, 3)
        tv = torch.from_numpy(v).double().permute(0, 2, 1, 3)
        mask = None if b is None else torch.from_numpy(b).double()
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                               is_causal=causal)
        assert np.allclose(o, ref.permute(0, 2, 1, 3).numpy(), atol=1e-13, rtol=0)
        s = (tq @ tk.transpose(-1, -2)) / math.sqrt(dk)
        if mask is not None:
            s = s + mask
        if causal:
            s = s.masked_fill(torch.ones(Nq, Nk, dtype=torch.bool).triu(1), -math.inf)
        assert np.allclose(lse, torch.logsumexp(s, -1).numpy(), atol=1e-13, rtol=0)


def test_row_subset_equals_full():
    rng = np.random.default_rng(9)
    q, k, v, b, kvl = rand_problem(rng, 2, 3, 6, 7, 4, 5, bias=True, kv=[7, 2])
    o, lse, _ = oracle.attn_fwd(q, k, v, bias=b, kv_lens=kvl, causal=True)
    rows = [0, 5, 17, 35, 20]
    os_, ls_, _ = oracle.attn_fwd(q, k, v, bias=b, kv_lens=kvl, causal=True, rows=rows)
    for t, r in enumerate(rows):
        bb, h, i = r // 18, (r // 6) % 3, r % 6
        assert np.array_equal(os_[t], o[bb, i, h]) and (ls_[t] == lse[bb, h, i])


# ------------------------------------------------- merge of per-piece states (page 1 s3, s4, s9)

def _tol_ok(x, y):
    x, y = np.asarray(x, np.float64), np.asarray(y, np.float64)
    assert x.shape == y.shape
    with np.errstate(invalid="ignore"):
        return _tol_ok_inner(x, y)


def _tol_ok_inner(x, y):
    both_inf = np.isinf(x) & np.isinf(y) & (np.sign(x) == np.sign(y))
    d = np.abs(np.where(both_inf, 0.0, x - y))
    lim = 2e-12 + 2e-12 * np.maximum(np.abs(np.where(both_inf, 0, x)),
                                     np.abs(np.where(both_inf, 0, y)))
    return bool(np.all(d <= lim))


def _online_vs_oracle(q, k, v, causal, kv_len, tiles, allowed=None, bias=None, scale=None, tree=False):
    """q [Nq, dk], k [Nk, dk], v [Nk, dv] for one head; returns True if they agree."""
    nq, nk = q.shape[0], k.shape[0]
    sc = 1.0 / math.sqrt(q.shape[1]) if scale is None else scale
    vis = online_ref.bottom_right_visible(nq, kv_len, causal, allowed)
    bfun = None if bias is None else (lambda i, j: float(bias[i, j]))
    o_on, lse_on, _ = online_ref.online_rows(q.astype(np.float64).tolist(),
                                             k.astype(np.float64).tolist(),
                                             v.astype(np.float64).tolist(), tiles, vis, sc,
                                             bias=bfun, dv=v.shape[1], tree=tree)
    bias4 = None
    if bias is not None or allowed is not None:
        bb = np.zeros((nq, nk), np.float32) if bias is None else bias.astype(np.float32).copy()
        if allowed is not None:
            for i in range(nq):
                for j in range(nk):
                    if not allowed(i, j):
                        bb[i, j] = -np.inf
        bias4 = bb[None, None]
    o, lse, _ = oracle.attn_fwd(q[None, :, None], k[None, :, None], v[None, :, None],
                                bias=bias4, kv_lens=[kv_len], causal=causal, scale=sc)
    return _tol_ok(o[0, :, 0], o_on) and _tol_ok(lse[0, 0], lse_on)


def _partitions(nk, rng, count):
    out = [[list(range(nk))], [[j] for j in range(nk)]]
    for _ in range(count):
        cuts = sorted(rng.sample(range(1, nk), rng.randint(0, max(0, nk - 1)))) if nk > 1 else []
        edges = [0] + cuts + [nk]
        tiles = [list(range(a, b)) for a, b in zip(edges[:-1], edges[1:])]
        tiles.insert(rng.randint(0, len(tiles)), [])  # an empty tile somewhere
        rng.shuffle(tiles)
        out.append(tiles)
    return out


@pytest.mark.parametrize("family,shape,causal,pad", [
    ("noncausal irregular tiles", (5, 9, 4, 3), False, None),
    ("square global causal", (7, 7, 5, 2), True, None),
    ("rectangular bottom-right, empty prefix rows", (2, 6, 1, 1), True, None),
    ("rectangular bottom-right, empty prefix rows", (5, 2, 1, 1), True, None),
    ("padding, empty tiles and rows", (2, 4, 3, 2), False, 1),
    ("padding, empty tiles and rows", (4, 7, 3, 4), True, 3),
    ("empty key axis", (2, 0, 3, 2), False, None),
    ("common logit shifts and wide span", (1, 5, 1, 1), False, None),
    ("common logit shifts and wide span", (1, 5, 1, 2), False, None),
])
def test_online_families_agree_with_oracle(family, shape, causal, pad):
    # "How Does FlashAttention Preserve Global Softmax Across Tiles?", section 9 table
    nq, nk, dk, dv = shape
    rng = random.Random(hash(shape) & 0xFFFF)
    nrng = np.random.default_rng(abs(hash(shape)) & 0xFFFF)
    q = nrng.standard_normal((nq, dk)).astype(np.float32)
    k = nrng.standard_normal((nk, dk)).astype(np.float32)
    v = nrng.standard_normal((nk, dv)).astype(np.float32)
    kv_len = nk if pad is None else pad
    bias = None
    if family.startswith("common"):
        bias = (nrng.standard_normal((nq, nk)) * 300.0).astype(np.float32)  # wide span
    for tiles in _partitions(nk, rng, 6):
        for tree in (False, True):  # pieces combined one after another, and as a merge tree
            assert _online_vs_oracle(q, k, v, causal, kv_len, tiles, bias=bias, tree=tree), (family, tiles)
    if family.startswith("common"):
        assert _online_vs_oracle(q, k, v, causal, kv_len, [list(range(nk))],
                                 bias=bias + np.float32(1000.0))


def test_all_six_three_tile_orders():
    # section 9: "all six three-tile orders", shape 3/6/4/3
    nrng = np.random.default_rng(36)
    q = nrng.standard_normal((3, 4)).astype(np.float32)
    k = nrng.standard_normal((6, 4)).astype(np.float32)
    v = nrng.standard_normal((6, 3)).astype(np.float32)
    tiles = [[0, 1], [2, 3], [4, 5]]
    for perm in itertools.permutations(tiles):
        assert _online_vs_oracle(q, k, v, False, 6, list(perm))


def test_sixteen_seeded_shapes():
    # section 9 lists 16 fixed-seed shapes whose script is not available; these are 16
    # seeded shapes of the same kind (the tolerance and method are the page's)
    rng = random.Random(16)
    for t in range(16):
        nq, nk, dk, dv = rng.randint(1, 7), rng.randint(0, 9), rng.randint(1, 5), rng.randint(1, 4)
        nrng = np.random.default_rng(1000 + t)
        q = nrng.standard_normal((nq, dk)).astype(np.float32)
        k = nrng.standard_normal((nk, dk)).astype(np.float32)
        v = nrng.standard_normal((nk, dv)).astype(np.float32)
        causal = bool(t % 2)
        kv_len = rng.randint(0, nk) if t % 3 == 0 else nk
        allowed = (lambda i, j, s=t: (i * 7 + j * 3 + s) % 5 != 0) if t % 4 == 1 else None
        for tiles in _partitions(nk, rng, 3):
            assert _online_vs_oracle(q, k, v, causal, kv_len, tiles, allowed=allowed)


# ---------------------------------------------------------------- merge of key-subset states

def test_merge_of_disjoint_subsets_equals_whole_in_any_order():
    # page 1, section 4: merging disjoint subsets is associative and order-free; a key
    # included twice counts twice
    rng = np.random.default_rng(10)
    q, k, v, b, kvl = rand_problem(rng, 2, 2, 1, 37, 8, 8, bias=True, kv=[37, 20])
    o, lse, _ = oracle.attn_fwd(q, k, v, bias=b, kv_lens=kvl)
    for n_splits in (1, 2, 16, 37):
        edges = [round(s * 37 / n_splits) for s in range(n_splits + 1)]
        st = np.stack([oracle.key_state(q, k, v, a, c, bias=b, kv_lens=kvl)
                       for a, c in zip(edges[:-1], edges[1:])], axis=3)  # [B,H,1,S,2+dv]
        perm = rng.permutation(n_splits)
        om, lm = oracle.merge_states(st[:, :, :, perm])
        assert np.allclose(om[:, :, 0], o[:, 0], atol=1e-13, rtol=0)
        assert np.allclose(lm[:, :, 0], lse[:, :, 0], atol=1e-13, rtol=0)
    # duplicated key: merge [0, 20) with [10, 37): keys 10..19 counted twice
    s1 = oracle.key_state(q, k, v, 0, 20, bias=b, kv_lens=kvl)
    s2 = oracle.key_state(q, k, v, 10, 37, bias=b, kv_lens=kvl)
    od, _ = oracle.merge_states(np.stack([s1, s2], axis=3))
    assert np.max(np.abs(od[:, :, 0] - o[:, 0])) > 1e-3


def test_merge_skips_empty_states_and_all_empty_row():
    st = np.zeros((3, 4, 2 + 3))
    st[:, :, 0] = -np.inf
    st[1, 2] = [0.5, 2.0, 1.0, 2.0, 3.0]
    st[2, 0] = [1.0, 1.0, 1.0, 1.0, 1.0]
    st[2, 3] = [3.0, 1.0, 0.0, 0.0, 0.0]
    o, lse = oracle.merge_states(st)
    assert np.all(o[0] == 0.0) and lse[0] == -np.inf
    assert np.allclose(o[1], [0.5, 1.0, 1.5], atol=1e-15)
    assert abs(lse[1] - (0.5 + math.log(2.0))) < 1e-15
    e = math.exp(-2.0)
    assert np.allclose(o[2], [e / (e + 1)] * 3, atol=1e-15)
    assert abs(lse[2] - (3.0 + math.log1p(e))) < 1e-15
