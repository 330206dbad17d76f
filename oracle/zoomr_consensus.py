"""CPU oracle for ZoomR's consensus selection and the attention over its final set.

TEST INFRASTRUCTURE. This module is the oracle, not the product: only the
tests and the benchmark may import it. It shares no code with the CUDA path and
imports nothing from it (it reuses the decode oracle's exact key, top-k, paged
row and fp64 attention steps).

It follows the ZoomR page ("ZoomR: Memory Efficient Reasoning through
Multi-Granularity Key Value Retrieval"), section 3.3, and its Algorithm 1:

Layout (reading). A sequence of L cached tokens holds the prompt [0, N_p), then
n pairs of a regular segment R_i and its summary segment S_i laid end to end,
each summary right after the paragraph it summarises, then possibly a tail that
has no summary yet. With the 2n + 1 ascending bounds bd (bd[0] = N_p,
bd[2n] <= L): R_i = [bd[2i], bd[2i+1]) and S_i = [bd[2i+1], bd[2i+2]).

1. ``head_top_k``  3.3 "Per-Head Importance Scoring and Voting": for every layer
   l and query head h, alpha_i = q^(l,h) . kbar_i^(l,h) over the n summaries and
   the indices of the k largest (ties to the lower index). kbar_i is the mean
   summary key of S_i for the KV head that query head h reads (GQA). The key is
   the decode oracle's exact dot product (fp64 where that sum is exact, Fraction
   elsewhere); k >= n gives every index.
2. ``consensus``   3.3 "Global Aggregation and Consensus": I_all is the union of
   all (layer, head) top-k sets; v_i counts the sets that contain i; I_c is the
   c members of I_all with the most votes (ties to the lower index; c >= |I_all|
   takes all of them); I_s = I_all minus I_c.
3. ``final_tokens`` 3.3 "Constructing the Final Multi-Granularity Context", the
   I_f equation: the prompt, the recent window [max(0, L - w), L), the regular
   segments of I_c and the summary segments of I_s, as one sorted set of token
   indices. Segments outside I_all contribute nothing.
4. ``attend_final`` ZoomR 2 "Background": for every layer and query head,
   softmax(q K^T / sqrt(d)) V over the K/V rows of I_f (the query head's KV
   head, read through the block table), in fp64. The same I_f serves every
   layer and head of the sequence.

Pins: ``tests/test_consensus_pins.py`` (integer-valued brute force of the votes
and the consensus, vote-count invariants, closed forms for k >= n, c = 0 and
c >= |I_all|, a dense case against a library attention routine, exact ties).
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence

import numpy as np

from oracle import zoomr_oracle as O


def head_top_k(q_head: np.ndarray, kbar: np.ndarray, k: int) -> np.ndarray:
    """Top-k summary indices of one (layer, query head): q_head [d], kbar [n, d] (its KV head's mean
    summary keys). Ascending index order."""
    keys = O.summary_keys(np.asarray(q_head)[None, :], kbar)  # a group of one head: its own exact key
    return O.select_top_k(keys, k)


def consensus(topk_sets: Sequence[np.ndarray], n: int, c: int):
    """Votes v [n], I_all, I_c and I_s (ascending int64 arrays) from all (layer, head) top-k sets."""
    votes = np.zeros(n, dtype=np.int64)
    for s in topk_sets:
        for i in s:
            votes[int(i)] += 1
    i_all = [i for i in range(n) if votes[i] > 0]
    ranked = sorted(i_all, key=lambda i: (-int(votes[i]), i))
    i_c = sorted(ranked[:max(0, min(int(c), len(i_all)))])
    i_s = [i for i in i_all if i not in set(i_c)]
    as_arr = lambda x: np.array(x, dtype=np.int64)
    return votes, as_arr(i_all), as_arr(i_c), as_arr(i_s)


def final_tokens(bounds: np.ndarray, prompt_len: int, L: int, w: int, i_c: np.ndarray, i_s: np.ndarray) -> np.ndarray:
    """I_f as a sorted array of token indices. bounds: the 2n+1 pair bounds (bd[0] = prompt_len)."""
    tokens = set(range(0, int(prompt_len)))
    tokens.update(range(max(0, L - int(w)), L))
    for i in i_c:
        tokens.update(range(int(bounds[2 * i]), int(bounds[2 * i + 1])))       # R_i
    for i in i_s:
        tokens.update(range(int(bounds[2 * i + 1]), int(bounds[2 * i + 2])))   # S_i
    return np.array(sorted(tokens), dtype=np.int64)


def attend_final(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, block_table_row: np.ndarray,
                 tokens: np.ndarray, G: int) -> np.ndarray:
    """fp64 outputs [Hq, d] of one layer for one sequence: q [Hq, d]; query head h reads KV head h // G."""
    outs = []
    for h in range(q.shape[0]):
        g = h // G
        K = O.paged_rows(k_pool, block_table_row, g, tokens)
        V = O.paged_rows(v_pool, block_table_row, g, tokens)
        o, _ = O.attend(q[h], K, V)
        outs.append(o)
    return np.stack(outs)


@dataclass
class SequenceResult:
    votes: np.ndarray   # int64 [n]
    i_all: np.ndarray
    i_c: np.ndarray
    i_s: np.ndarray
    tokens: np.ndarray  # I_f, sorted
    out: np.ndarray     # float64 [layers, Hq, d] (NaN for layers not attended)


def consensus_step(qs: Sequence[np.ndarray], kbars: Sequence[np.ndarray], k_pools, v_pools, block_tables,
                   seg_ptr, seg_bounds, prompt_lens, seq_lens, topk, consensus_c, window,
                   attend_layers: Sequence[int] | None = None, batch: Sequence[int] | None = None) -> List[SequenceResult]:
    """One consensus decode step for every (or the listed) sequence.

    qs[l] [B, Hq, d]; kbars[l] [seg_ptr[B], Hkv, d] (mean summary keys, CSR over segments);
    k_pools[l]/v_pools[l] [num_blocks, Hkv, 16, d]; block_tables [B, max_blocks]; seg_ptr [B+1];
    seg_bounds: sequence b's 2 n_b + 1 pair bounds start at 2 seg_ptr[b] + b; prompt_lens, seq_lens,
    topk, consensus_c [B]; window w. The votes use every layer in qs; the attention runs for
    ``attend_layers`` (default: all). Returns one SequenceResult per sequence in ``batch``.
    """
    nl = len(qs)
    B, Hq, d = qs[0].shape
    Hkv = kbars[0].shape[1]
    G = Hq // Hkv
    todo_layers = list(range(nl)) if attend_layers is None else list(attend_layers)
    out = []
    for b in (range(B) if batch is None else batch):
        s0, s1 = int(seg_ptr[b]), int(seg_ptr[b + 1])
        n = s1 - s0
        bd = np.asarray(seg_bounds[2 * s0 + b: 2 * s0 + b + 2 * n + 1])
        sets = []
        for l in range(nl):
            for h in range(Hq):
                sets.append(head_top_k(qs[l][b, h], kbars[l][s0:s1, h // G], int(topk[b])))
        votes, i_all, i_c, i_s = consensus(sets, n, int(consensus_c[b]))
        L = int(seq_lens[b])
        tokens = final_tokens(bd, int(prompt_lens[b]), L, int(window), i_c, i_s)
        o = np.full((nl, Hq, d), np.nan)
        for l in todo_layers:
            o[l] = attend_final(qs[l][b], k_pools[l], v_pools[l], block_tables[b], tokens, G)
        out.append(SequenceResult(votes, i_all, i_c, i_s, tokens, o))
    return out
