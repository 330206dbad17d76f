"""Pure-Python brute force of one ZoomR decode step, for tiny inputs only.

It pins the oracle from outside: it never pages (it reads the logical,
unpaged K/V the generator drew), it decides membership of every token with a
per-token predicate instead of a union of ranges, it ranks segments on their
exact rational scores (``fractions.Fraction``) instead of the fp32 key, and it
sums with ``math.fsum`` in Python floats. None of it is shared with
``oracle/``.
"""

from __future__ import annotations

import math
from fractions import Fraction
from itertools import combinations
from typing import List, Sequence


def exact_dot(a: Sequence[float], b: Sequence[float]) -> Fraction:
    return sum((Fraction(float(x)) * Fraction(float(y)) for x, y in zip(a, b)), Fraction(0))


def exact_scores(q_group, sum_k_rows) -> List[Fraction]:
    """max over the group's heads of the exact q . s for every segment."""
    return [max(exact_dot(q, s) for q in q_group) for s in sum_k_rows]


def dominant_subset(scores: Sequence, k: int) -> List[int]:
    """The one k-subset S with: i in S, j not in S => s_i > s_j or (s_i == s_j and i < j).

    Found by enumerating every k-subset (tiny n only)."""
    n = len(scores)
    k = max(0, min(k, n))
    found = []
    for S in combinations(range(n), k):
        inside = set(S)
        ok = all(scores[i] > scores[j] or (scores[i] == scores[j] and i < j)
                 for i in inside for j in range(n) if j not in inside)
        if ok:
            found.append(list(S))
    assert len(found) == 1, found
    return found[0]


def segment_of(bounds: Sequence[int], t: int) -> int:
    for i in range(len(bounds) - 1):
        if bounds[i] <= t < bounds[i + 1]:
            return i
    raise ValueError(t)


def in_gather_set(t: int, L: int, w: int, bounds, selected: set) -> bool:
    return t >= L - w or segment_of(bounds, t) in selected


def brute_unit(q_group, k_logical, v_logical, bounds, sum_k_rows, sum_v_rows, k: int, w: int, selected=None):
    """Output [G][d] (Python floats) of one unit, attending over the gathered
    tokens (logical K/V rows) and the summaries of the non-selected segments."""
    L = int(bounds[-1])
    n = len(bounds) - 1
    if selected is None:
        selected = dominant_subset(exact_scores(q_group, sum_k_rows), k)
    selected = set(selected)
    rows_k, rows_v = [], []
    for t in range(L):
        if in_gather_set(t, L, w, bounds, selected):
            rows_k.append(k_logical[t])
            rows_v.append(v_logical[t])
    for i in range(n):
        if i not in selected:
            rows_k.append(sum_k_rows[i])
            rows_v.append(sum_v_rows[i])
    d = len(q_group[0])
    outs = []
    for q in q_group:
        logits = [math.fsum(float(a) * float(b) for a, b in zip(q, r)) / math.sqrt(d) for r in rows_k]
        m = max(logits)
        e = [math.exp(x - m) for x in logits]
        z = math.fsum(e)
        outs.append([math.fsum(e[j] * float(rows_v[j][c]) for j in range(len(e))) / z for c in range(d)])
    return outs, sorted(selected), len(rows_k)
