"""Pins of the oracle's Philox4x32-10 and of the dropout keep convention drawn from it.

The generator is Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
(SC'11); its published known-answer vectors (tests/golden/philox4x32_10_kat.json) fix it, and
plausible slips (swapped multipliers, a missing key bump, outputs in the wrong order, nine
rounds) each fail them.  The keep convention is pinned by a direct single-counter check, by
its rate (1 - p8/256) and by its determinism in (seed, offset)."""
import json
import os

import numpy as np
import pytest

from oracle import philox

GOLD = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")


def kat_cases():
    with open(GOLD) as f:
        g = json.load(f)
    for c in g["cases"]:
        yield (np.array([int(x, 16) for x in c["ctr"]], np.uint64), np.array([int(x, 16) for x in c["key"]], np.uint64),
               [int(x, 16) for x in c["out"]])


def test_known_answer_vectors():
    for ctr, key, want in kat_cases():
        assert [int(x) for x in philox.philox4x32_10(ctr, key)] == want


def _variant(ctr, key, m0, m1, bump=True, order=(0, 1, 2, 3), rounds=10):
    x0, x1, x2, x3 = (int(c) for c in ctr)
    k0, k1 = (int(k) for k in key)
    for r in range(rounds):
        if r and bump:
            k0, k1 = (k0 + philox.W0) & philox.MASK, (k1 + philox.W1) & philox.MASK
        p0, p1 = m0 * x0, m1 * x2
        x0, x1, x2, x3 = ((p1 >> 32) ^ x1 ^ k0, p1 & philox.MASK, (p0 >> 32) ^ x3 ^ k1, p0 & philox.MASK)
    out = (x0, x1, x2, x3)
    return [out[t] for t in order]


def test_the_restatement_and_its_mutants():
    cases = list(kat_cases())
    # the scalar restatement in this file agrees with the oracle's on every vector
    for ctr, key, want in cases:
        assert _variant(ctr, key, philox.M0, philox.M1) == want
    mutants = {
        "multipliers swapped": dict(m0=philox.M1, m1=philox.M0),
        "no key bump": dict(m0=philox.M0, m1=philox.M1, bump=False),
        "outputs reversed": dict(m0=philox.M0, m1=philox.M1, order=(3, 2, 1, 0)),
        "nine rounds": dict(m0=philox.M0, m1=philox.M1, rounds=9),
    }
    for name, kw in mutants.items():
        assert any(_variant(ctr, key, **kw) != want for ctr, key, want in cases), name


def test_keep_convention_single_counter():
    # row 3, keys 16..31 of head (b, h) = (1, 2) with H = 4: counter (3, 1, 1 * 4 + 2, offset)
    seed, offset, p = 0x1234_5678_9ABC_DEF0, 77, 0.3
    keep, p_real = philox.keep_mask(seed, offset, 2, 4, 5, 40, p)
    p8 = philox.quantise(p)
    assert p8 == 77 and p_real == 77 / 256
    words = philox.philox4x32_10(np.array([3, 1, 6, offset], np.uint64),
                                 np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint64))
    by = [(int(words[t // 4]) >> (8 * (t % 4))) & 0xFF for t in range(16)]
    assert list(keep[1, 2, 3, 16:32]) == [b >= p8 for b in by]


def test_keep_rate_determinism_and_edges():
    keep, p_real = philox.keep_mask(7, 0, 2, 2, 64, 1000, 0.1)
    n = keep.size
    rate = keep.mean()
    sigma = np.sqrt(p_real * (1 - p_real) / n)
    assert abs((1 - rate) - p_real) < 5 * sigma
    again, _ = philox.keep_mask(7, 0, 2, 2, 64, 1000, 0.1)
    assert np.array_equal(keep, again)
    other, _ = philox.keep_mask(7, 1, 2, 2, 64, 1000, 0.1)  # another offset: other draws
    assert 0.7 < (keep == other).mean() < 0.9
    allk, p0 = philox.keep_mask(7, 0, 1, 1, 8, 100, 0.0)
    assert p0 == 0.0 and allk.all()
    assert philox.quantise(0.999) == 255
    with pytest.raises(ValueError):
        philox.quantise(1.0)
