"""Token and byte accounting for the ZoomR decode step.

These counters feed the benchmark's roofline (algorithmic bytes per launch)
and restate the sizing formulas the pages print, so that tests can pin them to
the pages' worked numbers.
"""

from __future__ import annotations

from typing import Iterable


def memory_savings(n_prompt: int, n_gen: int, n_window: int, c: int, mean_regular_len: float,
                   mean_summary_len: float, n_candidates: int) -> float:
    """ZoomR page, "3.5 Theoretical Memory Analysis", the MS equation.

    Full cache (prompt + generated tokens) over ZoomR's active set: the prompt,
    c zoomed-in regular segments, the remaining candidates' summary segments
    and the recent window.
    """
    active = n_prompt + c * mean_regular_len + (n_candidates - c) * mean_summary_len + n_window
    return (n_prompt + n_gen) / active


def dense_kv_bytes(layers: int, tokens: int, kv_heads: int, head_dim: int, bytes_per_elem: int,
                   sequences: int = 1) -> int:
    """"KV-cache management" page, "Sizing the dense cache (planning formula)":
    layers x 2 (K and V) x tokens x KV heads x head dim x bytes, linear in sequences."""
    return layers * 2 * tokens * kv_heads * head_dim * bytes_per_elem * sequences


def distinct_blocks(tokens: Iterable[int], block_size: int = 16) -> int:
    """Number of distinct logical blocks a sorted token list touches."""
    last = -1
    n = 0
    for t in tokens:
        blk = int(t) // block_size
        if blk != last:
            n += 1
            last = blk
    return n


def attend_bytes_per_unit(n_tokens: int, n_summaries: int, n_blocks_touched: int, group: int, head_dim: int,
                          elem_bytes: int) -> int:
    """Algorithmic bytes the gather-attention kernel must read for one
    (sequence, KV head) unit: the K and V rows of the gathered tokens, the
    summary K and V rows of the non-selected segments, one block-table entry
    per distinct logical block, and the group's queries."""
    row = head_dim * elem_bytes
    return (2 * (n_tokens + n_summaries) * row + 4 * n_blocks_touched + group * row)


def select_bytes_per_unit(n_segments: int, group: int, head_dim: int, elem_bytes: int) -> int:
    """Algorithmic bytes of the score + select step for one unit: every summary
    key of the sequence for this KV head, plus the group's queries."""
    row = head_dim * elem_bytes
    return n_segments * row + group * row


def ranges_token_count(ranges) -> int:
    return int(sum(int(e) - int(s) for s, e in ranges))


def ranges_block_count(ranges, block_size: int = 16) -> int:
    """Distinct logical blocks covered by sorted, disjoint [start, end) ranges."""
    n = 0
    last = -1
    for s, e in ranges:
        s, e = int(s), int(e)
        if e <= s:
            continue
        b0, b1 = s // block_size, (e - 1) // block_size
        if b0 == last:
            b0 += 1
        if b1 >= b0:
            n += b1 - b0 + 1
        last = max(last, (e - 1) // block_size)
    return n
