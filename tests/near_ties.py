"""Planted near-ties at the top-k boundary, for tests of the exact ranking key.

A near-tie is a summary key copied from the last selected segment i onto the
first unselected segment j, then nudged by one unit in the last place in two
components whose changes nearly cancel. The pair is chosen so that the exact
scores differ by a tiny amount while an fp32 chain (each product and partial sum
rounded, components in ascending order) loses the difference and ranks the pair
by the tie rule instead. Exact arithmetic and that fp32 chain then pick
different segments.

This module draws test inputs and computes nothing the oracle or the kernels
compute: the exact comparison of the planted pair uses ``fractions.Fraction``,
and ``fp32_chain_keys`` is the ranking a plain fp32 loop would give, kept only
to show that the two orders really disagree.
"""

from __future__ import annotations

from fractions import Fraction
from typing import List, Optional, Tuple

import numpy as np
import torch

from hierarchical_sparse_kv_gb300 import workloads as W


def fp32_chain_keys(q_group: np.ndarray, sum_k: np.ndarray) -> np.ndarray:
    """max over the group of the fp32 dot, rounded after every product and add, ascending components."""
    q32 = np.asarray(q_group, dtype=np.float32)
    s32 = np.asarray(sum_k, dtype=np.float32)
    acc = np.zeros((s32.shape[0], q32.shape[0]), dtype=np.float32)
    for t in range(s32.shape[1]):
        acc = acc + s32[:, t:t + 1] * q32[None, :, t]
    return acc.max(axis=1)


def _exact(q_group, row) -> Fraction:
    return max(sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(qh, row)), Fraction(0))
               for qh in q_group)


def _nudged(x: np.float32, up: bool, dtype: str) -> np.float32:
    """x moved one unit in the last place of the storage dtype, away from (up) or toward zero."""
    bits = np.array([x], dtype=np.float32).view(np.uint32)[0]
    step = np.uint32(1 << 16) if dtype == "bf16" else np.uint32(1)
    bits = bits + step if up else bits - step
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def _rank_pair(keys: np.ndarray, k: int) -> Tuple[int, int]:
    order = sorted(range(len(keys)), key=lambda i: (-float(keys[i]), i))
    return order[k - 1], order[k]


def near_tie_row(q: np.ndarray, sk: np.ndarray, i: int, j: int, dtype: str) -> Optional[np.ndarray]:
    """A nudged copy of summary key sk[i] to put in row j, or None if none is found.

    q [G, d] holds the group's queries and sk [n, d] the unit's summary keys (exact stored values). With
    the copy in row j, the exact keys of i and j differ, the exact order favours the higher index of the
    two (where the tie rule would not), an ascending fp32 chain ranks them the other way, and no other
    row's exact key lies between theirs.
    """
    n = sk.shape[0]
    approx = (sk.astype(np.float64) @ q.astype(np.float64).T).max(axis=1)
    hstar = int(np.argmax(sk[i].astype(np.float64) @ q.astype(np.float64).T))
    ki = _exact(q, sk[i])
    want_j_above = j > i
    # one-ulp nudges of single components, and the change each makes to q_h* . s (exact in fp64)
    nudges = []
    for t in range(sk.shape[1]):
        if sk[i, t] == 0:
            continue
        for up in (True, False):
            x = _nudged(sk[i, t], up, dtype)
            nudges.append((float(q[hstar, t]) * (float(x) - float(sk[i, t])), t, up))
    # pairs of nudges on different components whose changes nearly cancel: smallest sum first
    nudges.sort()
    vals = np.array([v for v, _, _ in nudges])
    pairs = []
    for va, ta, ua in nudges:
        m = int(np.searchsorted(vals, -va))
        for c in (m - 1, m, m + 1):
            if 0 <= c < len(nudges) and nudges[c][1] != ta and va + nudges[c][0] != 0:
                pairs.append((abs(va + nudges[c][0]), (ta, ua), (nudges[c][1], nudges[c][2])))
    pairs.sort()
    for _, (t1, u1), (t2, u2) in pairs[:64]:
        row = sk[i].copy()
        row[t1] = _nudged(row[t1], u1, dtype)
        row[t2] = _nudged(row[t2], u2, dtype)
        kj = _exact(q, row)
        if kj == ki or (kj > ki) != want_j_above:
            continue
        trial = sk.copy()
        trial[j] = row
        f32 = fp32_chain_keys(q, trial)
        f32_j_above = f32[j] > f32[i] or (f32[j] == f32[i] and j < i)
        if f32_j_above == want_j_above:
            continue  # the fp32 chain kept the difference: not a disagreement
        lo, hi = min(ki, kj), max(ki, kj)
        others = [m for m in range(n) if m not in (i, j) and abs(approx[m] - float(ki)) < 1e-3]
        if any(lo <= _exact(q, sk[m]) <= hi for m in others):
            continue
        return row
    return None


def boundary_pair(q: np.ndarray, sk: np.ndarray, k: int) -> Tuple[int, int]:
    """The k-th and (k+1)-th rows in (key desc, index asc), keys estimated in fp64."""
    return _rank_pair((sk.astype(np.float64) @ q.astype(np.float64).T).max(axis=1), k)


def plant_near_ties(st: W.Structure, lt: W.LayerTensors, max_units: int = 64) -> List[Tuple[int, int, int, int]]:
    """Plant a near-tie into up to ``max_units`` units of ``lt`` (in place, on its device).

    Returns (b, g, i, j) for every planted unit: segment j now holds the row ``near_tie_row`` built
    from segment i's summary key, i and j being the unit's k-th and (k+1)-th segments.
    """
    spec = st.spec
    G = spec.num_q_heads // spec.num_kv_heads
    q_all = W.to_numpy32(lt.q)
    sk_all = W.to_numpy32(lt.sum_k)
    planted = []
    for b in range(st.batch):
        s0, n = int(st.seg_ptr[b]), st.num_segments(b)
        k = min(int(st.topk[b]), n)
        if not (0 < k < n):
            continue
        for g in range(spec.num_kv_heads):
            if len(planted) >= max_units:
                break
            q = q_all[b, g * G:(g + 1) * G]
            sk = sk_all[s0:s0 + n, g]
            i, j = boundary_pair(q, sk, k)
            row = near_tie_row(q, sk, i, j, spec.dtype)
            if row is None:
                continue
            lt.sum_k[s0 + j, g] = torch.from_numpy(row).to(lt.sum_k.dtype).to(lt.sum_k.device)
            planted.append((b, g, i, j))
    return planted
