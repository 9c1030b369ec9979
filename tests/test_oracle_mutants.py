"""Plausible mistakes planted in a copy of the oracle must each fail a pin.

Each mutant is the oracle's C source with one edit (a dropped term, a wrong sign or index,
a transposed operand, a wrong mask convention).  It is compiled on the CPU into a temporary
shared object and run through a compact set of the pins; the test passes only if at least
one pin rejects it.  Nothing here touches the repository's own oracle build.
"""
import math
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "scale dropped": ("double x = p->scale * dot;", "double x = dot;"),
    "bias scaled": ("if (p->bias) x += bias_at(p, b, h, i, j);",
                    "if (p->bias) x += p->scale * bias_at(p, b, h, i, j);"),
    "top-left causal": ("if (p->causal && j > i + n - p->Nq) return 0;",
                        "if (p->causal && j > i) return 0;"),
    "causal off by one": ("if (p->causal && j > i + n - p->Nq) return 0;",
                          "if (p->causal && j >= i + n - p->Nq) return 0;"),
    "padding off by one": ("if (j >= n) return 0;                                 /* padding */",
                           "if (j > n) return 0;"),
    "exp sign flipped": ("double w = exp(xbuf[j] - m);", "double w = exp(m - xbuf[j]);"),
    "no max shift": ("double w = exp(xbuf[j] - m);", "double w = exp(xbuf[j]);"),
    "lse in log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "lse without max": ("*lse = m + log(l);", "*lse = log(l);"),
    "value rows strided by dk": ("return p->v + ((b * p->Nk + j) * p->H + h) * p->dv;",
                                 "return p->v + ((b * p->Nk + j) * p->H + h) * p->dk;"),
    "q and k swapped in layout": (
        "const float *kj = p->k + ((b * p->Nk + j) * p->H + h) * p->dk;",
        "const float *kj = p->k + ((b * p->Nk + i) * p->H + h) * p->dk;"),
    "empty row lse zero": ("        *lse = -INFINITY;\n        return;",
                           "        *lse = 0.0;\n        return;"),
    "no final division": ("for (int64_t c = 0; c < p->dv; ++c) o[c] /= l;\n    *lse",
                          "*lse"),
    "merge forgets to rescale u": ("for (int64_t c = 0; c < dv; ++c) orow[c] += a * x[2 + c];",
                                   "for (int64_t c = 0; c < dv; ++c) orow[c] += x[2 + c];"),
    "merge forgets to rescale l": ("l += a * x[1];", "l += x[1];"),
    "state l not shifted": ("s[1] += w;", "s[1] += exp(logit(&p, b, h, i, j));"),
}


def _compile(src_text, out):
    with tempfile.NamedTemporaryFile("w", suffix=".c", delete=False) as f:
        f.write(src_text)
        path = f.name
    try:
        subprocess.run(["gcc", *oracle.GCC_FLAGS, path, "-o", out, "-lm"], check=True,
                       capture_output=True)
    finally:
        os.unlink(path)


def _pins(lib):
    """Compact pins (a subset of test_oracle_pins); returns the list of those that fail."""
    fails = []
    # page 1 s2 / s4 worked examples (exact)
    q = np.ones((1, 1, 1, 1), np.float32)
    k = np.array([0, 1], np.float32).reshape(1, 2, 1, 1)
    for vals, want in (([0.0, 1.0], 0.75), ([1.0, 0.0], 0.25)):
        v = np.array(vals, np.float32).reshape(1, 2, 1, 1)
        o, lse, _ = oracle.attn_fwd(q, k, v, scale=math.log(3.0), lib=lib)
        if abs(o[0, 0, 0, 0] - want) > 1e-15 or abs(lse[0, 0, 0] - math.log(4)) > 1e-15:
            fails.append("page1 worked example")
    # library attention with bias, causal, dk != dv, wide logits
    rng = np.random.default_rng(8)
    for (B, H, Nq, Nk, dk, dv, causal, bias, big) in [(2, 3, 7, 7, 5, 2, True, False, 1),
                                                       (1, 2, 5, 9, 4, 3, False, True, 1),
                                                       (1, 1, 3, 4, 2, 3, False, False, 400)]:
        qq = (rng.standard_normal((B, Nq, H, dk)) * big).astype(np.float32)
        kk = (rng.standard_normal((B, Nk, H, dk)) * big).astype(np.float32)
        vv = rng.standard_normal((B, Nk, H, dv)).astype(np.float32)
        bb = rng.standard_normal((B, H, Nq, Nk)).astype(np.float32) if bias else None
        o, lse, _ = oracle.attn_fwd(qq, kk, vv, bias=bb, causal=causal, lib=lib)
        t = lambda a: torch.from_numpy(a).double().permute(0, 2, 1, 3)
        ref = torch.nn.functional.scaled_dot_product_attention(
            t(qq), t(kk), t(vv), attn_mask=None if bb is None else torch.from_numpy(bb).double(),
            is_causal=causal).permute(0, 2, 1, 3).numpy()
        if not np.allclose(o, ref, atol=1e-12, rtol=0):
            fails.append("library attention")
        s = (t(qq) @ t(kk).transpose(-1, -2)) / math.sqrt(dk)
        if bb is not None:
            s = s + torch.from_numpy(bb).double()
        if causal:
            s = s.masked_fill(torch.ones(Nq, Nk, dtype=torch.bool).triu(1), -math.inf)
        if not np.allclose(lse, torch.logsumexp(s, -1).numpy(), atol=1e-10, rtol=1e-12):
            fails.append("library lse")
    # bottom-right rectangular mask and empty rows (page 1 s6)
    qq = rng.standard_normal((1, 5, 1, 3)).astype(np.float32)
    kk = rng.standard_normal((1, 2, 1, 3)).astype(np.float32)
    vv = rng.standard_normal((1, 2, 1, 2)).astype(np.float32)
    o, lse, _ = oracle.attn_fwd(qq, kk, vv, causal=True, lib=lib)
    if not (np.all(o[0, :3] == 0) and np.all(lse[0, 0, :3] == -np.inf)
            and np.all(np.isfinite(lse[0, 0, 3:]))):
        fails.append("empty rows")
    p = oracle.attn_probs(qq[:, :2], rng.standard_normal((1, 5, 1, 3)).astype(np.float32),
                          rng.standard_normal((1, 5, 1, 2)).astype(np.float32), causal=True,
                          lib=lib)[0, 0]
    if not ((p[0] > 0).tolist() == [1, 1, 1, 1, 0] and (p[1] > 0).all()):
        fails.append("bottom-right visible sets")
    # padding
    kvl = np.array([3], np.int32)
    kk = rng.standard_normal((1, 6, 1, 3)).astype(np.float32)
    vv = rng.standard_normal((1, 6, 1, 2)).astype(np.float32)
    o1, _, _ = oracle.attn_fwd(qq, kk, vv, kv_lens=kvl, lib=lib)
    o2, _, _ = oracle.attn_fwd(qq, kk[:, :3], vv[:, :3], lib=lib)
    if not np.allclose(o1, o2, atol=1e-15):
        fails.append("padding")
    # split states merged equal the whole, and states obey 1 <= l <= n
    qq = rng.standard_normal((1, 1, 1, 4)).astype(np.float32)
    kk = rng.standard_normal((1, 9, 1, 4)).astype(np.float32)
    vv = rng.standard_normal((1, 9, 1, 3)).astype(np.float32)
    o, _, _ = oracle.attn_fwd(qq, kk, vv, lib=lib)
    st = np.stack([oracle.key_state(qq, kk, vv, a, b, lib=lib) for a, b in ((0, 4), (4, 9))], 3)
    om, _ = oracle.merge_states(st, lib=lib)
    if not np.allclose(om[:, :, 0], o[:, 0], atol=1e-14):
        fails.append("merge")
    if not all(1.0 <= s[1] <= 5.0 for s in st[0, 0, 0]):
        fails.append("l bounds")
    return fails


def test_unmodified_oracle_passes_compact_pins(tmp_path):
    out = str(tmp_path / "orig.so")
    _compile(open(SRC).read(), out)
    assert _pins(oracle.bind(out)) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    out = str(tmp_path / "mutant.so")
    _compile(src.replace(old, new), out)
    with np.errstate(all="ignore"):
        fails = _pins(oracle.bind(out))
    assert fails, f"mutant '{name}' passed every pin"
