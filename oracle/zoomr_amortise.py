"""CPU oracle for the decode steps between two selections (semantic-boundary amortisation).

TEST INFRASTRUCTURE. This module is the oracle, not the product: only the
tests and the benchmark may import it. It shares no code with the CUDA path and
imports nothing from it (it reuses the decode and consensus oracles' steps).

The ZoomR page, 3.4 "Decoding Stage", recomputes the selection set only at
semantic boundaries and reuses it for the steps in between; appendix A.3
"Semantic Boundaries" puts the boundaries at punctuation tokens, about 35 tokens
apart. In Algorithm 1 the final set is rebuilt only at a boundary, while its
recent window {t-w+1, ..., t-1} is defined from the current step t.

Reading: between selections the selected parts stay fixed (the decode step's
selected segments and its summary rows; the consensus path's prompt, zoomed
regular segments and candidate summary segments), and the recent window follows
the newest token: with L' cached tokens it is [max(0, L' - w), L'). Tokens
appended since the selection belong to no segment yet and are reached only
through the window.

1. ``reuse_unit``         the decode step of one (sequence, KV head) with the
   selection held fixed and L' cached tokens.
2. ``reuse_final_tokens`` the consensus path's final set with I_c and I_s held
   fixed and L' cached tokens.

Pins: ``tests/test_amortise_pins.py`` (equal to the full step when L' = L, a
per-token brute force, the dense case against a library attention routine).
"""

from __future__ import annotations

import numpy as np

from oracle import zoomr_consensus as OC
from oracle import zoomr_oracle as O


def reuse_unit(q_group, k_pool, v_pool, block_table_row, g, bounds, sum_k_rows, sum_v_rows, sel, L_new: int,
               w: int) -> O.UnitResult:
    """Attention of one unit over the fixed selection ``sel`` (ascending segment indices) and the window of a
    sequence that now holds L_new tokens. bounds: the segment bounds of the selection step."""
    tokens, summaries = O.gather_set(bounds, np.asarray(sel), int(L_new), int(w))
    K = np.concatenate([O.paged_rows(k_pool, block_table_row, g, tokens), np.asarray(sum_k_rows)[summaries]], axis=0)
    V = np.concatenate([O.paged_rows(v_pool, block_table_row, g, tokens), np.asarray(sum_v_rows)[summaries]], axis=0)
    outs, probs = [], []
    for h in range(q_group.shape[0]):
        o, p = O.attend(q_group[h], K, V)
        outs.append(o)
        probs.append(p)
    return O.UnitResult(np.zeros(0, np.float32), np.asarray(sel), tokens, summaries, np.stack(outs), np.stack(probs))


def reuse_final_tokens(bounds: np.ndarray, prompt_len: int, L_new: int, w: int, i_c, i_s) -> np.ndarray:
    """The consensus path's final set for a sequence that now holds L_new tokens, I_c and I_s held fixed."""
    return OC.final_tokens(bounds, prompt_len, int(L_new), int(w), np.asarray(i_c), np.asarray(i_s))
