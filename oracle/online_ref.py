"""Pure-Python (binary64) restatement of the online softmax as a merge of per-key-set states.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  The tests use it to pin the
materialised oracle against the method's own claim: the state (m, l, u) of a set of keys
(the largest logit, the exponential mass measured against it, and the value sum weighted the
same way) can be formed piece by piece and combined, and combining the states of the pieces
of any complete, non-duplicated partition of the key set, in any grouping and any order,
gives the state of the whole set; dividing u by l once gives the dense result
("How Does FlashAttention Preserve Global Softmax Across Tiles?", sections 3 and 4; the
acceptance bound of its section 9, element-wise |x - y| <= 2e-12 + 2e-12 * max(|x|, |y|)).

Structure: a row's state over one piece of the key axis is built from its visible keys
(``piece_state``); two states are combined by bringing both to their common maximum
(``combine``: the larger m is kept and each side's l and u are multiplied by
exp(m_side - m)); the pieces of a partition are combined either one after another or as a
balanced binary tree (``fold``).  An empty piece, or one with no visible key, has no mass
and is skipped by ``combine`` instead of evaluating exp(-inf - (-inf)) (same page, section
6).  The empty-row policy (o = 0, lse = -inf) is that page's section 6, and the single final
division is "Reducing Memory Traffic with Output Accumulation in FlashAttention",
"Computing the Value Weighted Sum First".
"""
from __future__ import annotations

import math
from typing import Callable, List, Optional, Sequence, Tuple

Row = List[float]
# (m, l, u): m = -inf and l = 0 for a state without mass
State = Tuple[float, float, Row]


def dot(a: Sequence[float], b: Sequence[float]) -> float:
    s = 0.0
    for x, y in zip(a, b):
        s += x * y
    return s


def no_mass(dv: int) -> State:
    return (-math.inf, 0.0, [0.0] * dv)


def piece_state(logits: Sequence[float], values: Sequence[Row], dv: int) -> State:
    """State of one piece from the logits of its visible keys and their value rows."""
    if not logits:
        return no_mass(dv)
    m = max(logits)
    w = [math.exp(x - m) for x in logits]
    u = [0.0] * dv
    for wj, vj in zip(w, values):
        u = [c + wj * e for c, e in zip(u, vj)]
    return (m, math.fsum(w), u)


def combine(a: State, b: State) -> State:
    """State of the union of two disjoint key sets (section 3 of the first page)."""
    if a[1] == 0.0:
        return b
    if b[1] == 0.0:
        return a
    m = max(a[0], b[0])
    fa, fb = math.exp(a[0] - m), math.exp(b[0] - m)
    return (m, fa * a[1] + fb * b[1], [fa * x + fb * y for x, y in zip(a[2], b[2])])


def fold(states: Sequence[State], dv: int, tree: bool = False) -> State:
    """Combine the states of a partition's pieces: left to right, or as a balanced tree."""
    if not states:
        return no_mass(dv)
    if not tree:
        acc = no_mass(dv)
        for s in states:
            acc = combine(acc, s)
        return acc
    level = list(states)
    while len(level) > 1:
        nxt = [combine(level[t], level[t + 1]) for t in range(0, len(level) - 1, 2)]
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    return level[0]


def finish(s: State, dv: int) -> Tuple[Row, float]:
    """o = u / l and lse = m + ln l; a state without mass is an empty row: (0, -inf)."""
    if s[1] == 0.0:
        return [0.0] * dv, -math.inf
    return [c / s[1] for c in s[2]], s[0] + math.log(s[1])


def online_rows(q: Sequence[Row], k: Sequence[Row], v: Sequence[Row],
                key_tiles: Sequence[Sequence[int]], visible: Callable[[int, int], bool],
                scale: float, bias: Optional[Callable[[int, int], float]] = None,
                dv: Optional[int] = None, tree: bool = False,
                ) -> Tuple[List[Row], List[float], List[Tuple[float, float]]]:
    """Attention of one head from the pieces of a key partition.

    q, k, v: lists of rows; key_tiles: the key axis cut into pieces (lists of key indices,
    any sizes, any order; empty pieces allowed); visible(i, j): the mask; bias(i, j): the
    additive bias (not scaled); dv: the value width (needed when there are no keys); tree:
    combine the pieces as a balanced binary tree instead of one after another.
    Returns (O rows, lse per row, final (m, l) per row).
    """
    if dv is None:
        dv = len(v[0])
    out: List[Row] = []
    lse: List[float] = []
    stats: List[Tuple[float, float]] = []
    for i, qi in enumerate(q):
        pieces = []
        for tile in key_tiles:
            keys = [j for j in tile if visible(i, j)]
            logits = [scale * dot(qi, k[j]) + (bias(i, j) if bias is not None else 0.0) for j in keys]
            pieces.append(piece_state(logits, [v[j] for j in keys], dv))
        st = fold(pieces, dv, tree)
        o_i, lse_i = finish(st, dv)
        out.append(o_i)
        lse.append(lse_i)
        stats.append((st[0], st[1]))
    return out, lse, stats


def bottom_right_visible(nq: int, nk_valid: int, causal: bool,
                         allowed: Optional[Callable[[int, int], bool]] = None):
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
