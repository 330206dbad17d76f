"""How the gather-attention kernels share a call's rows among their warps, modelled on the host (no GPU): the
even split's shares, partial slots and the merge's warp ranges, and the dynamic split's claim protocol on its
per-unit batch counter.

Each of a unit's H home warps claims 32-row batches with an atomic add on one counter: a first claim, then one
claim at a time, each issued only after the previous one succeeded, until its first failing claim (a value >= T,
the unit's batch count). The model runs the warps under random interleavings and checks what the kernel relies
on: every batch is handed out exactly once, every warp fails exactly once, the counter ends at T + H, and exactly
one claim (the last increment of the call) sees T + H - 1 and stores 0, leaving the counter ready for the next
call. A planted mistake (a warp that stops after a success) must break it.
"""

from __future__ import annotations

import random

import pytest


def _run(T: int, H: int, rng: random.Random, stop_early: int = -1):
    """Interleave H warps' claims; returns (batches handed out, failures per warp, final counter, resets,
    whether the planted mistake happened)."""
    counter = 0
    handed, failures, resets, planted = [], [0] * H, 0, False
    live = list(range(H))
    while live:
        w = rng.choice(live)
        c = counter
        counter += 1  # the atomic add
        if c < T:
            handed.append(c)
            if w == stop_early:  # planted mistake: this warp stops after a success, without its failing claim
                planted = True
                live.remove(w)
        else:
            failures[w] += 1
            if c + 1 == T + H:
                resets += 1
                counter = 0  # the store of the warp whose failing claim is the call's last increment
            live.remove(w)
    return handed, failures, counter, resets, planted


@pytest.mark.parametrize("T,H", [(1, 1), (5, 28), (138, 28), (40, 1), (3, 60), (0, 4)])
def test_every_batch_once_and_the_counter_returns_to_zero(T, H):
    rng = random.Random(T * 1000 + H)
    for _ in range(200):
        handed, failures, counter, resets, _ = _run(T, H, rng)
        assert sorted(handed) == list(range(T))
        assert failures == [1] * H
        assert resets == 1 and counter == 0


def test_a_warp_that_skips_its_failing_claim_leaves_the_counter_dirty():
    rng = random.Random(7)
    runs = 0
    for _ in range(200):
        _, _, counter, resets, planted = _run(10, 6, rng, stop_early=2)
        if planted:
            runs += 1
            assert counter != 0 and resets == 0
    assert runs > 100


# ---------------------------------------------------------------- the even split's bookkeeping
# The attend kernels split the cost coordinate (every unit's rows, each unit preceded by X virtual rows) evenly over
# N warps: warp w takes [floor(w C / N), floor((w + 1) C / N)). A warp writes one partial per unit whose rows its share
# meets, into slot u + w; the merge (and the dynamic split, for its home-warp count H) finds a unit's first and last
# warp from the unit's first row c0 and last row c1 alone: the warp holding position c is ceil((c + 1) N / C) - 1.

def _shares(C: int, N: int):
    return [(w * C // N, (w + 1) * C // N) for w in range(N)]


def _merge_range(c0: int, c1: int, C: int, N: int):
    wf = ((c0 + 1) * N + C - 1) // C - 1
    wl = ((c1 + 1) * N + C - 1) // C - 1
    return wf, wl


@pytest.mark.parametrize("seed", range(12))
def test_merge_range_and_slots_match_brute_force(seed):
    rng = random.Random(seed)
    U = rng.choice([1, 2, 7, 64, 300])
    X = rng.choice([0, 48])
    rows = [rng.randint(1, rng.choice([20, 600, 5000])) for _ in range(U)]
    C = sum(rows) + U * X
    N = min(rng.choice([1, 5, 456, 1824, 4096]), C)
    shares = _shares(C, N)
    assert shares[0][0] == 0 and shares[-1][1] == C and all(s < e for s, e in shares)
    slots = set()
    P = 0
    for u, R in enumerate(rows):
        c0 = P + X  # the unit's first row in the cost coordinate
        brute = [w for w, (s, e) in enumerate(shares) if s < c0 + R and e > c0]
        wf, wl = _merge_range(c0, c0 + R - 1, C, N)
        assert brute == list(range(wf, wl + 1))
        for w in brute:
            assert u + w not in slots and u + w < U + N
            slots.add(u + w)
        P = c0 + R
