"""CPU oracle for one ZoomR decode step over a paged KV cache.

TEST INFRASTRUCTURE. This module is the oracle, not the product: only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it. It shares no code with the CUDA path and imports nothing from it.

It is written to be read against the ZoomR page ("ZoomR: Memory Efficient
Reasoning through Multi-Granularity Key Value Retrieval") and the
"KV-cache management" page, step by step, per unit = (layer, sequence b,
KV head g), with no blocking, fusion or reordering beyond what each step
states:

1. ``summary_keys``   ZoomR 3.3, "Per-Head Importance Scoring and Voting",
   the equation alpha_i = q_t^T kbar_i: the inner product of the query with
   every mean summary key. Readings: per KV head the score is the maximum over
   the GQA group's query heads; the division by sqrt(d) is dropped from the
   ranking key (a positive scale does not change an order). The key is the
   exact real value of that inner product on the stored inputs: every product
   of two stored values (bf16 or fp32) is exact in fp64, the d products are
   summed in fp64 with a TwoSum error term after every add, and any sum whose
   error terms are not all zero is recomputed with ``fractions.Fraction``.
2. ``select_top_k``   ZoomR 3.3, the equation I_top-k = argtop-k(alpha):
   the k largest keys; ties go to the lower segment index; the result is
   returned in ascending index order. k >= n selects every segment.
3. ``gather_set``     ZoomR 3.3, "Constructing the Final Multi-Granularity
   Context", the equation for I_f: the union of the recent window and the
   token ranges of the selected segments, as a deduplicated sorted set; every
   segment that is not selected contributes its one summary vector instead.
   The window is the last min(w, L) cached positions [L - w, L).
4. ``attend``         ZoomR 2 "Background", the equation
   A = softmax(q K^T / sqrt(d)) V, restricted to the gathered set; K/V rows
   are fetched through the block table as on the "KV-cache management" page,
   "Paged KV cache (PagedAttention)". fp64 throughout.

Every step above is pinned from outside the oracle (closed forms checked
against a library attention routine, exact rational scores, a pure-Python
brute force, hand-computed cancellation cases and invariants) in
``tests/test_oracle_pins.py``; no step is left unpinned.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from fractions import Fraction
from typing import List, Sequence

import numpy as np

BLOCK_SIZE = 16


def _two_sum(a: np.ndarray, b: np.ndarray):
    """fp64 a + b and its exact rounding error (Knuth's TwoSum, round to nearest)."""
    s = a + b
    bb = s - a
    return s, (a - (s - bb)) + (b - bb)


def exact_dots(q_group: np.ndarray, sum_k: np.ndarray):
    """Exact q_h . s_i for every segment i and group head h.

    q_group: [G, d], sum_k: [n, d], holding the exact stored values. Returns
    (dots, inexact): dots is an object array [n, G] of Python floats (where the
    fp64 sum was exact) or Fractions (where it was not), inexact the bool [n, G]
    flags of the entries that took the Fraction route.
    """
    q = np.asarray(q_group, dtype=np.float64)  # bf16 and fp32 widen exactly
    s = np.asarray(sum_k, dtype=np.float64)
    assert np.all(np.isfinite(q)) and np.all(np.isfinite(s)), "non-finite ranking inputs are unsupported"
    n, d = s.shape
    G = q.shape[0]
    acc = np.zeros((n, G), dtype=np.float64)
    inexact = np.zeros((n, G), dtype=bool)
    for t in range(d):
        prod = s[:, t:t + 1] * q[None, :, t]  # two <= 24-bit significands: exact in fp64
        acc, err = _two_sum(acc, prod)
        inexact |= err != 0
    dots = np.empty((n, G), dtype=object)
    for i in range(n):
        for h in range(G):
            if inexact[i, h]:
                dots[i, h] = sum((Fraction(float(s[i, t])) * Fraction(float(q[h, t])) for t in range(d)), Fraction(0))
            else:
                dots[i, h] = float(acc[i, h])
    return dots, inexact


def summary_keys(q_group: np.ndarray, sum_k: np.ndarray) -> np.ndarray:
    """Ranking key of every segment for one KV head: max over the G heads of the
    exact dot product (object array [n] of Python floats or Fractions; Python
    compares the two kinds exactly)."""
    dots, _ = exact_dots(q_group, sum_k)
    keys = np.empty(dots.shape[0], dtype=object)
    for i in range(dots.shape[0]):
        keys[i] = max(dots[i])
    return keys


def select_top_k(keys: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest keys, ties to the lower index, ascending order."""
    n = len(keys)
    order = sorted(range(n), key=lambda i: (-keys[i], i))
    chosen = order[:max(0, min(int(k), n))]
    return np.array(sorted(chosen), dtype=np.int64)


def gather_set(bounds: np.ndarray, sel: np.ndarray, L: int, w: int):
    """Token set T (sorted) and summary list Sigma (ascending) for one unit.

    bounds: the n+1 ascending segment bounds of the sequence (first 0, last L).
    """
    tokens = set(range(max(0, L - int(w)), L))
    chosen = set(int(i) for i in sel)
    for i in chosen:
        tokens.update(range(int(bounds[i]), int(bounds[i + 1])))
    n = len(bounds) - 1
    summaries = [i for i in range(n) if i not in chosen]
    return np.array(sorted(tokens), dtype=np.int64), np.array(summaries, dtype=np.int64)


def token_ranges(tokens: np.ndarray) -> np.ndarray:
    """Maximal runs [start, end) of a sorted token list (int64 [R, 2])."""
    if len(tokens) == 0:
        return np.zeros((0, 2), dtype=np.int64)
    breaks = np.nonzero(np.diff(tokens) != 1)[0]
    starts = np.concatenate([[tokens[0]], tokens[breaks + 1]])
    ends = np.concatenate([tokens[breaks] + 1, [tokens[-1] + 1]])
    return np.stack([starts, ends], axis=1)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """softmax(q K^T / sqrt(d)) V in fp64. Returns (o [d], p [R])."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    d = q.shape[0]
    logits = (K @ q) / math.sqrt(d)
    m = logits.max()
    e = np.exp(logits - m)
    p = e / e.sum()
    return p @ V, p


def paged_rows(pool: np.ndarray, block_table_row: np.ndarray, g: int, tokens: np.ndarray) -> np.ndarray:
    """Rows of KV head g for logical tokens, read through the block table.

    pool: [num_blocks, Hkv, 16, d]; token t lives in physical block
    block_table_row[t // 16], slot t % 16.
    """
    phys = np.asarray(block_table_row)[tokens // BLOCK_SIZE]
    return pool[phys, g, tokens % BLOCK_SIZE, :]


@dataclass
class UnitResult:
    keys: np.ndarray  # object [n]: exact keys (Python float or Fraction)
    sel: np.ndarray  # int64 ascending
    tokens: np.ndarray  # int64 sorted
    summaries: np.ndarray  # int64 ascending
    out: np.ndarray  # float64 [G, d]
    probs: np.ndarray  # float64 [G, |T| + |Sigma|]


def decode_unit(q_group, k_pool, v_pool, block_table_row, g, bounds, sum_k_rows, sum_v_rows, k, w) -> UnitResult:
    """All four steps for one (sequence, KV head).

    q_group [G, d]; k_pool/v_pool [num_blocks, Hkv, 16, d]; bounds [n+1];
    sum_k_rows/sum_v_rows [n, d] (this sequence's segments, KV head g).
    """
    L = int(bounds[-1])
    keys = summary_keys(q_group, sum_k_rows)
    sel = select_top_k(keys, k)
    tokens, summaries = gather_set(bounds, sel, L, w)
    K = np.concatenate([paged_rows(k_pool, block_table_row, g, tokens), np.asarray(sum_k_rows)[summaries]], axis=0)
    V = np.concatenate([paged_rows(v_pool, block_table_row, g, tokens), np.asarray(sum_v_rows)[summaries]], axis=0)
    outs, probs = [], []
    for h in range(q_group.shape[0]):
        o, p = attend(q_group[h], K, V)
        outs.append(o)
        probs.append(p)
    return UnitResult(keys, sel, tokens, summaries, np.stack(outs), np.stack(probs))


@dataclass
class StepResult:
    out: np.ndarray  # float64 [B, Hq, d]
    sel: np.ndarray  # int32 [B, Hkv, k_max], ascending, -1 padded
    units: List[List[UnitResult]]  # [B][Hkv]


def decode_step(q, k_pool, v_pool, block_tables, seg_ptr, seg_bounds, sum_k, sum_v, topk, window,
                units: Sequence[tuple] | None = None) -> StepResult:
    """One decode step of one layer for every (or the listed) (b, g) unit.

    Arrays are host numpy arrays holding the exact stored values:
    q [B, Hq, d]; k_pool/v_pool [num_blocks, Hkv, 16, d]; block_tables
    [B, max_blocks]; seg_ptr [B+1] (CSR over segments); seg_bounds (sequence b's
    n_b+1 bounds start at seg_ptr[b] + b); sum_k/sum_v [total_segments, Hkv, d];
    topk [B]; window w.
    """
    B, Hq, d = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    k_clip = [min(int(topk[b]), int(seg_ptr[b + 1] - seg_ptr[b])) for b in range(B)]
    k_max = max(k_clip) if B else 0
    out = np.full((B, Hq, d), np.nan)
    sel_all = np.full((B, Hkv, max(k_max, 0)), -1, dtype=np.int32)
    todo = units if units is not None else [(b, g) for b in range(B) for g in range(Hkv)]
    res: List[List[UnitResult]] = [[None] * Hkv for _ in range(B)]
    for (b, g) in todo:
        s0, s1 = int(seg_ptr[b]), int(seg_ptr[b + 1])
        n = s1 - s0
        bounds = np.asarray(seg_bounds[s0 + b: s0 + b + n + 1])
        r = decode_unit(q[b, g * G:(g + 1) * G], k_pool, v_pool, block_tables[b], g, bounds,
                        sum_k[s0:s1, g], sum_v[s0:s1, g], int(topk[b]), int(window))
        out[b, g * G:(g + 1) * G] = r.out
        sel_all[b, g, :len(r.sel)] = r.sel
        res[b][g] = r
    return StepResult(out, sel_all, res)
