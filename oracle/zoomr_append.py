"""CPU oracle for the append path of a paged KV cache and the mean summary keys.

TEST INFRASTRUCTURE. This module is the oracle, not the product: only the
tests and the benchmark may import it. It shares no code with the CUDA path and
imports nothing from it.

It follows the "KV-cache management" page and the ZoomR page ("ZoomR: Memory
Efficient Reasoning through Multi-Granularity Key Value Retrieval"):

1. ``append_kv``     "KV-cache management", "Paged KV cache (PagedAttention)":
   the K and V rows of the token at position t of sequence b go to physical
   block block_tables[b][t // 16], slot t % 16, for every KV head. A negative
   position means that sequence appends nothing.
2. ``copy_blocks``   "KV-cache management", "Block sharing with reference counts
   and copy-on-write": before a write into a last block that other sequences
   share, the block is copied whole into a private block; the copies of one
   step are made together. Each (src, dst) pair copies every KV head's 16 rows
   of K and of V.
3. ``segment_mean``  ZoomR 3.3, "Representing Context with Mean Summary Keys":
   the mean summary key of a segment is the average of the key vectors of its
   tokens, per KV head; the summary value row is the same average over the V
   rows (the reading under which every unselected segment contributes one
   summary K row and one summary V row). Precision: the rows are summed in fp64
   in ascending token order, the sum is divided by the token count in fp64, and
   the result is rounded to fp32 and then to the storage dtype, each time to
   nearest even.

Pins: ``tests/test_append_pins.py`` (exact rational means, read-back through
the decode oracle's paged reads, copy-on-write isolation, invariants).
"""

from __future__ import annotations

from typing import Iterable, Sequence, Tuple

import numpy as np
import torch

BLOCK_SIZE = 16


def append_kv(k_pool: np.ndarray, v_pool: np.ndarray, block_tables: np.ndarray, positions: Sequence[int],
              k_new: np.ndarray, v_new: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """New K/V pools after writing one token per sequence.

    k_pool, v_pool: [num_blocks, Hkv, 16, d]; block_tables: [B, max_blocks];
    positions: [B] token index of each sequence's new row (negative: none);
    k_new, v_new: [B, Hkv, d]. Returns copies; the inputs are not modified.
    """
    kp, vp = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    for b, t in enumerate(positions):
        t = int(t)
        if t < 0:
            continue
        blk = int(block_tables[b][t // BLOCK_SIZE])
        kp[blk, :, t % BLOCK_SIZE, :] = k_new[b]
        vp[blk, :, t % BLOCK_SIZE, :] = v_new[b]
    return kp, vp


def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray,
                pairs: Iterable[Tuple[int, int]]) -> Tuple[np.ndarray, np.ndarray]:
    """New K/V pools after copying whole blocks src -> dst (every KV head, all 16 rows)."""
    kp, vp = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
    for src, dst in pairs:
        kp[int(dst)] = k_pool[int(src)]
        vp[int(dst)] = v_pool[int(src)]
    return kp, vp


def segment_mean(pool: np.ndarray, block_table_row: np.ndarray, g: int, start: int, end: int) -> np.ndarray:
    """fp64 mean of KV head g's rows of tokens [start, end) of one sequence, read through its
    block table; the rows are added one token at a time in ascending order."""
    assert end > start
    acc = np.zeros(pool.shape[-1], dtype=np.float64)
    for t in range(start, end):
        acc = acc + pool[int(block_table_row[t // BLOCK_SIZE]), g, t % BLOCK_SIZE, :].astype(np.float64)
    return acc / float(end - start)


def round_to_dtype(x64: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> fp32 -> storage dtype, each to nearest even; returned as float32 values."""
    x32 = np.asarray(x64, dtype=np.float64).astype(np.float32)
    if dtype == "f32":
        return x32
    return torch.from_numpy(x32).to(torch.bfloat16).to(torch.float32).numpy()


def segment_summaries(k_pool: np.ndarray, v_pool: np.ndarray, block_tables: np.ndarray,
                      segs: Sequence[Tuple[int, int, int, int]], dtype: str, num_rows: int):
    """Summary rows of the given segments: segs[i] = (sequence b, start, end, output row).

    Returns (sum_k, sum_v) float32 arrays [num_rows, Hkv, d] holding the rounded means in the
    listed rows and NaN elsewhere (rows no segment writes)."""
    Hkv, d = k_pool.shape[1], k_pool.shape[3]
    sk = np.full((num_rows, Hkv, d), np.nan, dtype=np.float32)
    sv = np.full((num_rows, Hkv, d), np.nan, dtype=np.float32)
    for b, s, e, row in segs:
        for g in range(Hkv):
            sk[row, g] = round_to_dtype(segment_mean(k_pool, block_tables[b], g, s, e), dtype)
            sv[row, g] = round_to_dtype(segment_mean(v_pool, block_tables[b], g, s, e), dtype)
    return sk, sv
