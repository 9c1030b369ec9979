"""Pins of the oracle's backward (dQ, dK, dV of sum(dout * O)), against things other than its
own formulas ("How Does FlashAttention Preserve Global Softmax Across Tiles?", section 7):

  - torch float64 autograd through an explicitly written masked softmax (a library routine);
  - central finite differences of the forward oracle itself (no backward formula involved);
  - the q/k scaling symmetry: O depends on q and k only through q_i . k_j, so scaling q by
    (1 + e) and k by 1 / (1 + e) changes nothing, and sum_i q_i . dQ_i = sum_j k_j . dK_j;
  - exact zeros: a key no row sees gets dK = dV = 0, an empty row gets dQ = 0;
  - planted mistakes in a copy of the C source (dropped row reduction, missing scale,
    unnormalised weights, dQ built from v) each fail one of these.
No GPU needed."""
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")


def rand(rng, *shape, s=1.0):
    return (rng.standard_normal(shape) * s).astype(np.float32)


def visible_mask(B, H, Nq, Nk, kv_lens, causal, bias):
    m = np.ones((B, H, Nq, Nk), bool)
    lens = [Nk] * B if kv_lens is None else [int(x) for x in kv_lens]
    for b, n in enumerate(lens):
        for i in range(Nq):
            for j in range(Nk):
                if j >= n or (causal and j > i + n - Nq):
                    m[b, :, i, j] = False
    if bias is not None:
        m &= ~np.isneginf(bias)
    return m


def torch_grads(q, k, v, g, bias=None, kv_lens=None, causal=False, scale=None):
    """float64 autograd of sum(g * O) with O written as masked softmax(scale q k^T + b) v;
    rows with no visible key are left out of the softmax (their output is zero)."""
    B, Nq, H, dk = q.shape
    Nk = k.shape[1]
    scale = 1 / math.sqrt(dk) if scale is None else scale
    vis = torch.from_numpy(visible_mask(B, H, Nq, Nk, kv_lens, causal, bias))
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    x = scale * torch.einsum("bihc,bjhc->bhij", qt, kt)
    if bias is not None:
        x = x + torch.from_numpy(np.where(np.isneginf(bias), 0.0, bias)).double()
    x = x.masked_fill(~vis, -math.inf)
    nonempty = vis.any(-1, keepdim=True)
    x = torch.where(nonempty, x, torch.zeros_like(x))
    p = torch.softmax(x, -1) * nonempty * vis
    o = torch.einsum("bhij,bjhc->bihc", p, vt)
    (o * torch.from_numpy(g).double()).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def loss(q, k, v, g, **kw):
    o, _, _ = oracle.attn_fwd(q, k, v, **kw)
    return float(np.sum(o * g.astype(np.float64)))


CASES = [
    dict(B=1, H=2, Nq=5, Nk=7, dk=4, dv=3, causal=False),
    dict(B=2, H=1, Nq=6, Nk=6, dk=3, dv=5, causal=True),
    dict(B=2, H=2, Nq=7, Nk=4, dk=2, dv=2, causal=True),              # Nq > Nk: empty rows
    dict(B=3, H=1, Nq=4, Nk=9, dk=3, dv=2, causal=True, kv_lens=[9, 2, 0]),
    dict(B=1, H=2, Nq=4, Nk=6, dk=5, dv=4, causal=False, bias=True),
]


def make(case, seed):
    rng = np.random.default_rng(seed)
    B, H, Nq, Nk, dk, dv = (case[x] for x in ("B", "H", "Nq", "Nk", "dk", "dv"))
    q, k, v = rand(rng, B, Nq, H, dk), rand(rng, B, Nk, H, dk), rand(rng, B, Nk, H, dv)
    g = rand(rng, B, Nq, H, dv)
    kw = dict(causal=case["causal"])
    if case.get("kv_lens") is not None:
        kw["kv_lens"] = np.array(case["kv_lens"], np.int32)
    if case.get("bias"):
        bias = rand(rng, B, H, Nq, Nk)
        bias[..., ::3] = -np.inf
        kw["bias"] = bias
    return q, k, v, g, kw


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_matches_torch_autograd(ci):
    q, k, v, g, kw = make(CASES[ci], 100 + ci)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, g, **kw)
    tq, tk, tv = torch_grads(q, k, v, g, **kw)
    for a, b in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.max(np.abs(a - b)) <= 1e-12 * (1 + np.max(np.abs(b)))


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_matches_finite_differences_of_the_forward(ci):
    q, k, v, g, kw = make(CASES[ci], 200 + ci)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, g, **kw)
    rng = np.random.default_rng(300 + ci)
    eps = 2.0 ** -9
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            h = float(xp[idx]) - float(xm[idx])  # the step as float32 holds it
            args = {"q": q, "k": k, "v": v}
            fd = (loss(**{**args, name: xp}, g=g, **kw) - loss(**{**args, name: xm}, g=g, **kw)) / h
            assert abs(fd - grad[idx]) <= 2e-4 * (1 + abs(grad[idx])), (name, idx, fd, grad[idx])


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_scaling_symmetry_of_q_and_k(ci):
    q, k, v, g, kw = make(CASES[ci], 400 + ci)
    dq, dk, _, _ = oracle.attn_bwd(q, k, v, g, **kw)
    lhs = np.sum(q.astype(np.float64) * dq)
    rhs = np.sum(k.astype(np.float64) * dk)
    assert abs(lhs - rhs) <= 1e-12 * (1 + abs(lhs))


def test_exact_zeros_for_unseen_keys_and_empty_rows():
    # causal, Nq > Nk and a padded sequence: the first rows see nothing; keys past kv_len and
    # keys no row reaches have zero gradient, exactly
    rng = np.random.default_rng(7)
    B, H, Nq, Nk, d = 2, 2, 6, 4, 3
    q, k, v, g = rand(rng, B, Nq, H, d), rand(rng, B, Nk, H, d), rand(rng, B, Nk, H, d), rand(rng, B, Nq, H, d)
    kvl = np.array([4, 2], np.int32)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, g, kv_lens=kvl, causal=True)
    # batch 0: row i sees j <= i - 2, so rows 0, 1 are empty; batch 1: j <= i - 4 and j < 2
    assert np.all(dq[0, :2] == 0) and np.all(dq[1, :4] == 0)
    assert np.all(dk[1, 2:] == 0) and np.all(dv[1, 2:] == 0)
    assert np.any(dq[0, 2:] != 0) and np.any(dk[0] != 0)


def test_one_key_per_row_passes_no_q_or_k_gradient():
    # with one visible key a row's weight is 1 whatever the logit: dQ = 0, dK = 0, dV_j = g_i
    rng = np.random.default_rng(8)
    q, k, v, g = rand(rng, 1, 1, 1, 4), rand(rng, 1, 1, 1, 4), rand(rng, 1, 1, 1, 3), rand(rng, 1, 1, 1, 3)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, g)
    assert np.all(dq == 0) and np.all(dk == 0)
    assert np.array_equal(dv[0, 0, 0], g[0, 0, 0].astype(np.float64))


MUTANTS = {
    "row reduction dropped": ("const double ds = prow[j] * (dprow[j] - c);",
                              "const double ds = prow[j] * dprow[j];"),
    "scale missing on dK": ("dkj[t] += scale * ds * (double)qi[t];", "dkj[t] += ds * (double)qi[t];"),
    "weights not normalised": ("for (int64_t j = 0; j < Nk; ++j) prow[j] /= l;\n                /* dP_ij",
                               "/* dP_ij"),
    "dV from the un-normalised weight": ("for (int64_t t = 0; t < dv; ++t) dvj[t] += prow[j] * (double)gi[t];",
                                         "for (int64_t t = 0; t < dv; ++t) dvj[t] += prow[j] * l * (double)gi[t];"),
    "dQ from q instead of k": ("dqi[t] += scale * ds * (double)kj[t];", "dqi[t] += scale * ds * (double)qi[t];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_backward_mistakes_fail_a_pin(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "m.so")
        with open(c, "w") as f:
            f.write(src.replace(old, new))
        subprocess.run(["gcc", *oracle.GCC_FLAGS, c, "-o", so, "-lm"], check=True, capture_output=True)
        lib = oracle.bind(so)
        failed = False
        for ci in (0, 1, 3):
            q, k, v, g, kw = make(CASES[ci], 500 + ci)
            dq, dk, dv, _ = oracle.attn_bwd(q, k, v, g, lib=lib, **kw)
            tq, tk, tv = torch_grads(q, k, v, g, **kw)
            if any(np.max(np.abs(a - b)) > 1e-9 * (1 + np.max(np.abs(b))) for a, b in ((dq, tq), (dk, tk), (dv, tv))):
                failed = True
        assert failed, f"mutant '{name}' passed every pin"
