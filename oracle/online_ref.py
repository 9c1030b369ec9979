"""Pure-Python (binary64) restatement of the tiled online-softmax forward.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  The tests use it to pin the
materialised oracle against the pages' own online formulation: for any complete,
non-duplicated partition of the key axis into tiles, visited in any order, the online
result must equal the dense one within binary64 rounding
("How Does FlashAttention Preserve Global Softmax Across Tiles?", section 9: element-wise
|x - y| <= 2e-12 + 2e-12 * max(|x|, |y|)).

The loop follows that page's section 5 outline, in its order:
  for each query tile: every row starts from the empty state;
  for each key/value tile: form the scaled logits under the global-position mask;
    for each row that sees at least one key of this tile: take the new maximum,
    rescale both the old l and the old u by exp(m_old - m_new), add this tile's
    exponential mass and weighted values;
  after the loop, divide each nonempty row once; empty rows are handled explicitly.
The first update of a row takes an explicit branch instead of evaluating
exp(-inf - (-inf)) (same page, section 6).  The state itself is that page's section 3
(m, l, u) and "Reducing Memory Traffic with Output Accumulation in FlashAttention",
"Updating the Exponential Sum and Weighted Sum Together".
"""
from __future__ import annotations

import math
from typing import Callable, List, Sequence, Tuple

Row = List[float]


def dot(a: Sequence[float], b: Sequence[float]) -> float:
    s = 0.0
    for x, y in zip(a, b):
        s += x * y
    return s


def online_rows(q: Sequence[Row], k: Sequence[Row], v: Sequence[Row],
                key_tiles: Sequence[Sequence[int]], visible: Callable[[int, int], bool],
                scale: float, bias: Callable[[int, int], float] | None = None,
                query_tiles: Sequence[Sequence[int]] | None = None, dv: int | None = None,
                ) -> Tuple[List[Row], List[float], List[Tuple[float, float]]]:
    """Online forward for one head.

    q, k, v: lists of rows; key_tiles: the key axis cut into tiles (lists of key indices,
    any sizes, any order; empty tiles allowed); visible(i, j): the mask; bias(i, j): the
    additive bias (not scaled); dv: the value width (needed when there are no keys).
    Returns (O rows, lse per row, final (m, l) per row).
    """
    nq = len(q)
    if dv is None:
        dv = len(v[0])
    if query_tiles is None:
        query_tiles = [list(range(nq))]
    out: List[Row] = [[0.0] * dv for _ in range(nq)]
    lse = [-math.inf] * nq
    stats: List[Tuple[float, float]] = [(-math.inf, 0.0)] * nq
    for qt in query_tiles:
        # empty state per row: no mass yet
        m = {i: -math.inf for i in qt}
        l = {i: 0.0 for i in qt}
        u = {i: [0.0] * dv for i in qt}
        has = {i: False for i in qt}
        for kt in key_tiles:
            for i in qt:
                cols = [j for j in kt if visible(i, j)]
                if not cols:
                    continue  # no allowed key in this tile: keep the state as it is
                x = {}
                for j in cols:
                    s = scale * dot(q[i], k[j])
                    if bias is not None:
                        s += bias(i, j)
                    x[j] = s
                tile_max = max(x.values())
                if has[i]:
                    m_new = max(m[i], tile_max)
                    alpha = math.exp(m[i] - m_new)
                    l[i] = alpha * l[i]
                    u[i] = [alpha * c for c in u[i]]
                else:
                    m_new = tile_max  # first update: the old state has zero mass
                    has[i] = True
                for j in cols:
                    e = math.exp(x[j] - m_new)
                    l[i] += e
                    u[i] = [c + e * vv for c, vv in zip(u[i], v[j])]
                m[i] = m_new
        for i in qt:
            if has[i]:
                out[i] = [c / l[i] for c in u[i]]
                lse[i] = m[i] + math.log(l[i])
                stats[i] = (m[i], l[i])
            else:
                out[i] = [0.0] * dv
                lse[i] = -math.inf
    return out, lse, stats


def bottom_right_visible(nq: int, nk_valid: int, causal: bool,
                         allowed: Callable[[int, int], bool] | None = None):
    """Mask in global positions: key j is visible to query i iff j < nk_valid, and, when
    causal, j <= i + (nk_valid - nq) (both sequences' ends aligned); ``allowed`` adds an
    explicit Boolean mask on top."""
    def vis(i: int, j: int) -> bool:
        if j >= nk_valid:
            return False
        if causal and j > i + nk_valid - nq:
            return False
        return True if allowed is None else bool(allowed(i, j))
    return vis
