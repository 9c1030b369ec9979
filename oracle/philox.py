"""The counter-based generator Philox4x32-10 and the dropout keep decisions drawn from it.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): the tests draw the keep decisions the
library's kernels draw in-kernel, from this independent restatement, and feed them to the
float64 dropout oracle.

Philox4x32-10 is the generator of J. K. Salmon, M. A. Moraes, R. O. Dror and D. E. Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), restated here from the paper's
definition: a 128-bit counter (x0, x1, x2, x3) and a 64-bit key (k0, k1) pass through ten
rounds; a round multiplies x0 and x2 by the constants M0 and M1 into 64-bit products and
outputs (hi(M1 x2) ^ x1 ^ k0, lo(M1 x2), hi(M0 x0) ^ x3 ^ k1, lo(M0 x0)); the key is bumped by
the Weyl constants (W0, W1) between rounds.  The tests pin it to the paper's known-answer
vectors.

Dropout keep decisions (the library's convention): the drop probability p is quantised to
p8 / 256 with p8 = round(256 p), at most 255.  Key j of query row i of head (b, h) is kept iff
byte (j % 16) of Philox4x32-10 at counter (i, j // 16, b * H + h, offset mod 2^32) and key
(seed mod 2^32, seed div 2^32) -- the four output words in order, each little-endian -- is at
least p8.  A kept weight is scaled by 256 / (256 - p8).
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32-10 of counters ctr (uint32 [..., 4]) under keys key (uint32 [..., 2], broadcast);
    returns uint32 [..., 4]."""
    ctr = np.asarray(ctr, dtype=np.uint64)
    key = np.asarray(key, dtype=np.uint64)
    x0, x1, x2, x3 = (ctr[..., t] for t in range(4))
    k0, k1 = key[..., 0], key[..., 1]
    for rnd in range(10):
        if rnd:
            k0 = (k0 + W0) & MASK
            k1 = (k1 + W1) & MASK
        p0 = np.uint64(M0) * x0
        p1 = np.uint64(M1) * x2
        x0, x1, x2, x3 = ((p1 >> np.uint64(32)) ^ x1 ^ k0, p1 & np.uint64(MASK),
                          (p0 >> np.uint64(32)) ^ x3 ^ k1, p0 & np.uint64(MASK))
    return np.stack([x0, x1, x2, x3], axis=-1).astype(np.uint32)


def quantise(p_drop: float) -> int:
    """p8 of the library's convention: round(256 p), at most 255 (p in [0, 1))."""
    if not 0.0 <= p_drop < 1.0:
        raise ValueError("p_drop must be in [0, 1)")
    return min(255, int(np.floor(p_drop * 256.0 + 0.5)))


def keep_mask(seed: int, offset: int, B: int, H: int, Nq: int, Nk: int, p_drop: float,
              heads=None):
    """Keep decisions [B, H, Nq, Nk] (bool) of the library's in-kernel dropout, and the realised
    drop probability p8 / 256.  heads: optional list of (b, h) to draw ([len, Nq, Nk] then)."""
    p8 = quantise(p_drop)
    G = (Nk + 15) // 16
    key = np.array([seed & MASK, (seed >> 32) & MASK], dtype=np.uint64)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    out = np.empty((len(pairs), Nq, Nk), dtype=bool)
    i = np.arange(Nq, dtype=np.uint64)[:, None]
    g = np.arange(G, dtype=np.uint64)[None, :]
    for t, (b, h) in enumerate(pairs):
        ctr = np.stack(np.broadcast_arrays(i, g, np.uint64(b * H + h), np.uint64(offset & MASK)), axis=-1)
        words = philox4x32_10(ctr, key)                      # [Nq, G, 4]
        by = words.astype("<u4").view(np.uint8).reshape(Nq, G * 16)
        out[t] = by[:, :Nk] >= p8
    if heads is None:
        out = out.reshape(B, H, Nq, Nk)
    return out, p8 / 256.0
