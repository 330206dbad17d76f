"""CPU oracle for the decode step with the prompt kept as an attention sink.

TEST INFRASTRUCTURE. This module is the oracle, not the product: only the
tests and the benchmark may import it. It shares no code with the CUDA path and
imports nothing from it (it reuses the decode oracle's steps).

The ZoomR page keeps the initial prompt tokens I_p in every final set as an
attention sink (3.3 "Constructing the Final Multi-Granularity Context", the I_f
equation; 3.4 "Prefill Stage": the prompt's cache is retained in full), and
segments only the generated tokens.

Reading: with a sink of N_s prompt tokens the segments partition [N_s, L) (the
first segment bound is N_s), and the token set of a unit is
[0, N_s) + the recent window [max(0, L - w), L) + the selected segments' ranges,
deduplicated; every segment that is not selected contributes its one summary
row, as in the decode step. Scoring, top-k and attention are the decode
oracle's.

Pins: ``tests/test_sink_pins.py`` (N_s = 0 is the decode step, a per-token
predicate, the dense case against a library attention routine).
"""

from __future__ import annotations

from typing import Sequence

import numpy as np

from oracle import zoomr_oracle as O


def gather_set_sink(bounds: np.ndarray, sel: np.ndarray, L: int, w: int, sink: int):
    """Token set T (sorted) and summary list (ascending) with the sink [0, sink) always in T."""
    tokens, summaries = O.gather_set(bounds, sel, L, w)
    return np.array(sorted(set(tokens.tolist()) | set(range(int(sink)))), dtype=np.int64), summaries


def decode_unit_sink(q_group, k_pool, v_pool, block_table_row, g, bounds, sum_k_rows, sum_v_rows, k, w,
                     sink) -> O.UnitResult:
    keys = O.summary_keys(q_group, sum_k_rows)
    sel = O.select_top_k(keys, k)
    tokens, summaries = gather_set_sink(bounds, sel, int(bounds[-1]), w, sink)
    K = np.concatenate([O.paged_rows(k_pool, block_table_row, g, tokens), np.asarray(sum_k_rows)[summaries]], axis=0)
    V = np.concatenate([O.paged_rows(v_pool, block_table_row, g, tokens), np.asarray(sum_v_rows)[summaries]], axis=0)
    outs, probs = [], []
    for h in range(q_group.shape[0]):
        o, p = O.attend(q_group[h], K, V)
        outs.append(o)
        probs.append(p)
    return O.UnitResult(keys, sel, tokens, summaries, np.stack(outs), np.stack(probs))


def decode_step_sink(q, k_pool, v_pool, block_tables, seg_ptr, seg_bounds, sum_k, sum_v, topk, window,
                     sink_lens, units: Sequence[tuple] | None = None):
    """As ``zoomr_oracle.decode_step`` with sequence b's sink of sink_lens[b] tokens."""
    B, Hq, d = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, d), np.nan)
    res = [[None] * Hkv for _ in range(B)]
    todo = units if units is not None else [(b, g) for b in range(B) for g in range(Hkv)]
    for (b, g) in todo:
        s0, s1 = int(seg_ptr[b]), int(seg_ptr[b + 1])
        bounds = np.asarray(seg_bounds[s0 + b: s0 + b + (s1 - s0) + 1])
        r = decode_unit_sink(q[b, g * G:(g + 1) * G], k_pool, v_pool, block_tables[b], g, bounds, sum_k[s0:s1, g],
                             sum_v[s0:s1, g], int(topk[b]), int(window), int(sink_lens[b]))
        out[b, g * G:(g + 1) * G] = r.out
        res[b][g] = r
    return out, res
