"""GPU parity of the append path (``zr_append_kv``, ``zr_copy_blocks``,
``zr_segment_summaries``) against ``oracle/zoomr_append.py``: every pool row and
every summary row bit-exact, device-detected bad indices reported and skipped,
and the decode step over a cache maintained by these calls equal to the oracle's.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z
from oracle import zoomr_append as A
from oracle import zoomr_oracle as O
from tests import gpu_common as C

pytestmark = pytest.mark.gpu

BAD_BLOCK, BAD_INDEX = 1, 2


def _np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float32).cpu().numpy()


def _same(a: np.ndarray, b: np.ndarray) -> bool:
    """Bitwise equality of float32 arrays (NaN == NaN)."""
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


def _setup(dtype="bf16", d=128, seed=11, batch=4, spare=12, seq_len_range=(33, 210), seg_len_range=(1, 40),
           extra_cols=1):
    spec = W.small_spec(dtype=dtype, head_dim=d, batch=batch, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=seq_len_range, seg_len_range=seg_len_range, topk=3, window=8, seed=seed)
    st = W.make_structure(spec, spare_blocks=spare)
    if extra_cols:
        st = dataclasses.replace(st, block_tables=np.concatenate(
            [st.block_tables, np.full((st.batch, extra_cols), -1, np.int32)], axis=1))
    lt = W.make_layer(st, 0, "cuda")
    return st, lt


def _cfg(st: W.Structure) -> Z.zr_config:
    sp = st.spec
    return Z.cache_config(batch=st.batch, num_kv_heads=sp.num_kv_heads, head_dim=sp.head_dim,
                          num_blocks=st.num_blocks, max_blocks_per_seq=st.max_blocks_per_seq, dtype=sp.dtype,
                          num_q_heads=sp.num_q_heads, window=st.window)


def _free_blocks(st: W.Structure):
    used = set(int(x) for x in st.block_tables.ravel() if x >= 0)
    return [b for b in range(st.num_blocks) if b not in used]


def _grow_tables(st: W.Structure, positions):
    """Block tables in which every sequence owns the block its position falls in (new blocks from the spares)."""
    bt = st.block_tables.copy()
    free = _free_blocks(st)
    for b, t in enumerate(positions):
        if t >= 0 and bt[b, t // 16] < 0:
            bt[b, t // 16] = free.pop(0)
    return bt


def _rand_rows(st, seed):
    sp = st.spec
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    shape = (st.batch, sp.num_kv_heads, sp.head_dim)
    dt = W.torch_dtype(sp.dtype)
    return (torch.randn(shape, generator=g, device="cuda").to(dt),
            torch.randn(shape, generator=g, device="cuda").to(dt))


def _all_segments(st: W.Structure):
    segs = []
    for b in range(st.batch):
        bnd = st.bounds(b)
        for i in range(len(bnd) - 1):
            segs.append((b, int(bnd[i]), int(bnd[i + 1]), int(st.seg_ptr[b]) + i))
    return segs


# ------------------------------------------------------------------ zr_append_kv
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 64)])
def test_append_matches_the_oracle(dtype, d):
    st, lt = _setup(dtype, d)
    L = st.seq_lens.astype(int)
    # the next token of every sequence but one (skipped), and an overwrite inside sequence 2
    pos = [int(L[b]) for b in range(st.batch)]
    pos[1] = -1
    pos[2] = int(L[2]) // 2
    bt = _grow_tables(st, pos)
    cfg = _cfg(st)
    kn, vn = _rand_rows(st, 5)
    kp0, vp0 = _np32(lt.k_pool), _np32(lt.v_pool)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_append_kv(cfg, torch.tensor(pos, dtype=torch.int32, device="cuda"), kn, vn,
                   torch.from_numpy(bt).cuda(), lt.k_pool, lt.v_pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wk, wv = A.append_kv(kp0, vp0, bt, pos, _np32(kn), _np32(vn))
    assert _same(_np32(lt.k_pool), wk) and _same(_np32(lt.v_pool), wv)


def test_append_bad_positions_and_blocks_are_reported_and_skipped():
    st, lt = _setup("bf16", 128, batch=5)
    L = st.seq_lens.astype(int)
    mb = st.max_blocks_per_seq
    pos = [int(L[b]) for b in range(st.batch)]
    bt = _grow_tables(st, pos)
    pos[0] = 16 * mb              # past the table: bad index
    bt[1, pos[1] // 16] = -1       # unmapped block: bad block
    bt[3, pos[3] // 16] = st.num_blocks  # block id past the pool: bad block
    cfg = _cfg(st)
    kn, vn = _rand_rows(st, 6)
    kp0, vp0 = _np32(lt.k_pool), _np32(lt.v_pool)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_append_kv(cfg, torch.tensor(pos, dtype=torch.int32, device="cuda"), kn, vn,
                   torch.from_numpy(bt).cuda(), lt.k_pool, lt.v_pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == BAD_BLOCK | BAD_INDEX
    good = [p if b in (2, 4) else -1 for b, p in enumerate(pos)]
    wk, wv = A.append_kv(kp0, vp0, bt, good, _np32(kn), _np32(vn))
    assert _same(_np32(lt.k_pool), wk) and _same(_np32(lt.v_pool), wv)


# ---------------------------------------------------------------- zr_copy_blocks
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_copy_blocks_match_the_oracle(dtype, d):
    st, lt = _setup(dtype, d, spare=20)
    free = _free_blocks(st)
    used = [int(x) for x in st.block_tables.ravel() if x >= 0]
    rng = np.random.default_rng(2)
    src = rng.choice(used, size=9, replace=False)
    dst = free[:9]
    pairs = np.stack([src, dst], 1).astype(np.int32)
    kp0, vp0 = _np32(lt.k_pool), _np32(lt.v_pool)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_copy_blocks(_cfg(st), torch.from_numpy(pairs).cuda(), lt.k_pool, lt.v_pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wk, wv = A.copy_blocks(kp0, vp0, [tuple(p) for p in pairs])
    assert _same(_np32(lt.k_pool), wk) and _same(_np32(lt.v_pool), wv)
    # an empty batch is a no-op
    Z.zr_copy_blocks(_cfg(st), None, lt.k_pool, lt.v_pool, err)
    torch.cuda.synchronize()
    assert _same(_np32(lt.k_pool), wk)


def test_copy_blocks_bad_pairs_are_reported_and_skipped():
    st, lt = _setup("bf16", 128, spare=8)
    free = _free_blocks(st)
    used = [int(x) for x in st.block_tables.ravel() if x >= 0]
    pairs = np.array([[used[0], free[0]], [-1, free[1]], [used[1], st.num_blocks], [used[2], free[2]]], np.int32)
    kp0, vp0 = _np32(lt.k_pool), _np32(lt.v_pool)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_copy_blocks(_cfg(st), torch.from_numpy(pairs).cuda(), lt.k_pool, lt.v_pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == BAD_BLOCK
    wk, wv = A.copy_blocks(kp0, vp0, [tuple(pairs[0]), tuple(pairs[3])])
    assert _same(_np32(lt.k_pool), wk) and _same(_np32(lt.v_pool), wv)


def test_copy_on_write_fork_then_append():
    """A forked child copies its shared last block, then appends: the parent's rows stay as they were."""
    st, lt = _setup("bf16", 128, batch=1, seq_len_range=(40, 40), spare=4)
    L = 40
    alloc = W.PagedBlockAllocator(st.num_blocks, np.random.default_rng(0))
    # rebuild the allocator's state from the structure's table: the parent owns its blocks
    parent = [int(x) for x in st.block_tables[0] if x >= 0]
    alloc.free_list = [b for b in alloc.free_list if b not in parent]
    alloc.ref_count[parent] = 1
    child = alloc.fork(parent)
    copies = alloc.append_block(child)
    assert len(copies) == 1
    mb = st.max_blocks_per_seq
    tables = np.full((2, mb), -1, np.int32)
    tables[0, :len(parent)] = parent
    tables[1, :len(child)] = child
    cfg = Z.cache_config(batch=2, num_kv_heads=2, head_dim=128, num_blocks=st.num_blocks, max_blocks_per_seq=mb,
                         dtype="bf16")
    kp0, vp0 = _np32(lt.k_pool), _np32(lt.v_pool)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_copy_blocks(cfg, torch.tensor(copies, dtype=torch.int32, device="cuda"), lt.k_pool, lt.v_pool, err)
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    kn = torch.randn((2, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn((2, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    pos = [-1, L]
    Z.zr_append_kv(cfg, torch.tensor(pos, dtype=torch.int32, device="cuda"), kn, vn, torch.from_numpy(tables).cuda(),
                   lt.k_pool, lt.v_pool, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k1, v1 = A.copy_blocks(kp0, vp0, copies)
    wk, wv = A.append_kv(k1, v1, tables, pos, _np32(kn), _np32(vn))
    kp, vp = _np32(lt.k_pool), _np32(lt.v_pool)
    assert _same(kp, wk) and _same(vp, wv)
    toks = np.arange(L)
    for h in range(2):
        assert _same(O.paged_rows(kp, tables[0], h, toks), O.paged_rows(kp0, tables[0], h, toks))
        assert _same(O.paged_rows(kp, tables[1], h, toks), O.paged_rows(kp0, tables[0], h, toks))


# ---------------------------------------------------------- zr_segment_summaries
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 64)])
def test_summaries_of_every_segment_match_the_oracle(dtype, d):
    st, lt = _setup(dtype, d, extra_cols=0)
    segs = _all_segments(st)
    rows = st.total_segments
    sk = torch.full((rows, 2, d), 7.0, dtype=W.torch_dtype(dtype), device="cuda")
    sv = torch.full_like(sk, 7.0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_segment_summaries(_cfg(st), torch.tensor(segs, dtype=torch.int32, device="cuda"),
                           C.device_tables(st), lt.k_pool, lt.v_pool, sk, sv, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wk, wv = A.segment_summaries(_np32(lt.k_pool), _np32(lt.v_pool), st.block_tables, segs, dtype, rows)
    assert _same(_np32(sk), wk) and _same(_np32(sv), wv)


def test_summaries_with_values_outside_the_exact_window_match_the_oracle():
    """Tiny (far below the int64 window), large (above it) and subnormal values, exact zeros and negative zeros,
    and a sum that fp64 cannot hold exactly (1 + 2^-60): every summary row still equals the oracle's fp64 loop."""
    st, lt = _setup("bf16", 128, extra_cols=0)
    segs = _all_segments(st)
    long_segs = [sg for sg in segs if sg[2] - sg[1] >= 4]
    bt = st.block_tables

    def at(b, t):
        return int(bt[b, t // 16]), t % 16

    plants = [
        (long_segs[0], "k", 3e-12), (long_segs[1], "v", 3000.0), (long_segs[2], "k", 1e-40),
        (long_segs[3], "v", 2.0 ** -60), (long_segs[4], "k", 0.0), (long_segs[5], "v", -0.0),
    ]
    for (b, s0, _, _), which, val in plants:
        pool = lt.k_pool if which == "k" else lt.v_pool
        blk, slot = at(b, s0 + 1)
        pool[blk, 1, slot, 3] = val
        pool[blk, 0, slot, 64:96] = val
    # an all-zero token row, and a segment whose values are all exactly 1 apart from one 2^-60
    b, s0, e0, _ = long_segs[6]
    blk, slot = at(b, s0)
    lt.k_pool[blk, :, slot, :] = 0.0
    b, s0, e0, _ = long_segs[7]
    for t in range(s0, e0):
        blk, slot = at(b, t)
        lt.v_pool[blk, :, slot, :] = 1.0
    blk, slot = at(b, s0 + 2)
    lt.v_pool[blk, :, slot, 5] = 2.0 ** -60
    torch.cuda.synchronize()
    rows = st.total_segments
    sk = torch.empty_like(lt.sum_k)
    sv = torch.empty_like(lt.sum_v)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_segment_summaries(_cfg(st), torch.tensor(segs, dtype=torch.int32, device="cuda"), C.device_tables(st),
                           lt.k_pool, lt.v_pool, sk, sv, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wk, wv = A.segment_summaries(_np32(lt.k_pool), _np32(lt.v_pool), st.block_tables, segs, "bf16", rows)
    assert _same(_np32(sk), wk) and _same(_np32(sv), wv)


def test_summaries_of_chosen_spans_leave_other_rows_alone():
    """Arbitrary spans (one token, a whole block, across blocks, a whole sequence), rows out of order."""
    st, lt = _setup("bf16", 128, extra_cols=0)
    L = st.seq_lens.astype(int)
    segs = [(0, 0, 1, 5), (1, 16, 32, 0), (2, 13, 35, 3), (3, 0, int(L[3]), 7), (0, int(L[0]) - 1, int(L[0]), 1),
            (1, 5, 6, 9)]
    rows = 12
    sk = torch.full((rows, 2, 128), -3.0, dtype=torch.bfloat16, device="cuda")
    sv = torch.full_like(sk, -3.0)
    Z.zr_segment_summaries(_cfg(st), torch.tensor(segs, dtype=torch.int32, device="cuda"), C.device_tables(st),
                           lt.k_pool, lt.v_pool, sk, sv)
    torch.cuda.synchronize()
    wk, wv = A.segment_summaries(_np32(lt.k_pool), _np32(lt.v_pool), st.block_tables, segs, "bf16", rows)
    untouched = np.isnan(wk)
    wk[untouched] = -3.0
    wv[untouched] = -3.0
    assert _same(_np32(sk), wk) and _same(_np32(sv), wv)


def test_bad_segments_are_reported_and_not_written():
    st, lt = _setup("f32", 64, extra_cols=1)
    mb = st.max_blocks_per_seq
    nb3 = (int(st.seq_lens[3]) + 15) // 16
    assert nb3 < mb and st.block_tables[3, nb3] == -1
    rows = 8
    segs = [
        (0, 0, 4, 0),                 # good
        (st.batch, 0, 4, 1),          # sequence out of range
        (1, 5, 5, 2),                 # empty
        (1, 8, 3, 2),                 # reversed
        (1, -1, 3, 2),                # negative start
        (2, 0, 16 * mb + 1, 2),       # past the table
        (2, 0, 4, rows),              # row out of range
        (3, 16 * nb3 - 1, 16 * nb3 + 1, 4),    # runs into the unmapped extra block
        (3, 1, 9, 6),                 # good
    ]
    sk = torch.full((rows, 2, 64), 1.5, dtype=torch.float32, device="cuda")
    sv = torch.full_like(sk, 1.5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_segment_summaries(_cfg(st), torch.tensor(segs, dtype=torch.int32, device="cuda"), C.device_tables(st),
                           lt.k_pool, lt.v_pool, sk, sv, err)
    torch.cuda.synchronize()
    assert int(err.item()) == BAD_BLOCK | BAD_INDEX
    good = [segs[0], segs[-1]]
    wk, wv = A.segment_summaries(_np32(lt.k_pool), _np32(lt.v_pool), st.block_tables, good, "f32", rows)
    wk[np.isnan(wk)] = 1.5
    wv[np.isnan(wv)] = 1.5
    assert _same(_np32(sk), wk) and _same(_np32(sv), wv)


def test_summaries_at_full_size_on_sampled_segments():
    """Every segment of the 16K-token, batch-8, 8-KV-head, d=128 bf16 layer on the device; a seeded sample of
    segments (all heads) against the oracle."""
    st = W.make_structure(W.WORKLOADS[2])
    lt = W.make_layer(st, 0, "cuda")
    segs = _all_segments(st)
    rows = st.total_segments
    sk = torch.empty((rows, 8, 128), dtype=torch.bfloat16, device="cuda")
    sv = torch.empty_like(sk)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_segment_summaries(_cfg(st), torch.tensor(segs, dtype=torch.int32, device="cuda"), C.device_tables(st),
                           lt.k_pool, lt.v_pool, sk, sv, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    pick = np.random.default_rng(4).choice(len(segs), size=24, replace=False)
    chosen = [segs[i] for i in sorted(pick)]
    kp, vp = _np32(lt.k_pool), _np32(lt.v_pool)
    wk, wv = A.segment_summaries(kp, vp, st.block_tables, chosen, "bf16", rows)
    gk, gv = _np32(sk), _np32(sv)
    for (_, _, _, r) in chosen:
        assert _same(gk[r], wk[r]) and _same(gv[r], wv[r]), r


# ------------------------------------------------- the decode over a maintained cache
def _decode_parity(st: W.Structure, lt: W.LayerTensors):
    plan = Z.DecodePlan.from_structure(st)
    try:
        return C.parity(st, lt, plan)
    finally:
        plan.close()


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_decode_over_device_summaries_matches_the_oracle(dtype, d):
    """Summaries computed on the device (bit-equal to the oracle's) feed the decode step."""
    st, lt = _setup(dtype, d, extra_cols=0)
    segs = _all_segments(st)
    rows = st.total_segments
    sk = torch.empty_like(lt.sum_k)
    sv = torch.empty_like(lt.sum_v)
    Z.zr_segment_summaries(_cfg(st), torch.tensor(segs, dtype=torch.int32, device="cuda"), C.device_tables(st),
                           lt.k_pool, lt.v_pool, sk, sv)
    torch.cuda.synchronize()
    wk, wv = A.segment_summaries(_np32(lt.k_pool), _np32(lt.v_pool), st.block_tables, segs, dtype, rows)
    assert _same(_np32(sk), wk) and _same(_np32(sv), wv)
    _decode_parity(st, dataclasses.replace(lt, sum_k=sk, sum_v=sv))


def test_generation_steps_append_close_segments_and_decode():
    """Three generation steps: every sequence appends a token (a new block when its last one is full); a
    sequence whose last segment reaches 6 tokens closes it and opens a new one; the closed (and the open)
    segments' summaries are recomputed on the device; the decode over the result matches the oracle's."""
    st, lt = _setup("bf16", 128, extra_cols=1, seq_len_range=(30, 100))
    kp_h, vp_h = _np32(lt.k_pool), _np32(lt.v_pool)
    for step in range(3):
        L = st.seq_lens.astype(int)
        pos = [int(L[b]) for b in range(st.batch)]
        bt = _grow_tables(st, pos)
        cfg = _cfg(dataclasses.replace(st, block_tables=bt))
        kn, vn = _rand_rows(st, 100 + step)
        Z.zr_append_kv(cfg, torch.tensor(pos, dtype=torch.int32, device="cuda"), kn, vn, torch.from_numpy(bt).cuda(),
                       lt.k_pool, lt.v_pool)
        kp_h, vp_h = A.append_kv(kp_h, vp_h, bt, pos, _np32(kn), _np32(vn))
        # new bounds: the last segment grows by one token; at 6 tokens it closes and a 1-token segment opens
        bl, nseg = [], []
        for b in range(st.batch):
            bnd = list(int(x) for x in st.bounds(b))
            bnd[-1] = pos[b] + 1
            if bnd[-1] - bnd[-2] > 6:
                bnd.insert(-1, pos[b])
            bl.append(bnd)
            nseg.append(len(bnd) - 1)
        seg_ptr = np.concatenate([[0], np.cumsum(nseg)]).astype(np.int32)
        st = dataclasses.replace(st, seq_lens=np.array([p + 1 for p in pos], np.int32), seg_ptr=seg_ptr,
                                 seg_bounds=np.concatenate(bl).astype(np.int32), block_tables=bt)
        # every summary row of the new CSR layout, recomputed on the device
        segs = _all_segments(st)
        rows = st.total_segments
        sk = torch.empty((rows, 2, 128), dtype=torch.bfloat16, device="cuda")
        sv = torch.empty_like(sk)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        Z.zr_segment_summaries(_cfg(st), torch.tensor(segs, dtype=torch.int32, device="cuda"), C.device_tables(st),
                               lt.k_pool, lt.v_pool, sk, sv, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert _same(_np32(lt.k_pool), kp_h) and _same(_np32(lt.v_pool), vp_h), step
        wk, wv = A.segment_summaries(kp_h, vp_h, st.block_tables, segs, "bf16", rows)
        assert _same(_np32(sk), wk) and _same(_np32(sv), wv), step
        _decode_parity(st, dataclasses.replace(lt, sum_k=sk, sum_v=sv))
