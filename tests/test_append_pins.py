"""Pins of the append-path oracle (``oracle/zoomr_append.py``) from outside it.

- Segment means against exact rational arithmetic (``fractions.Fraction``), and
  against a plain vectorised mean over the generator's logical (unpaged) rows.
- Appended rows read back through the decode oracle's paged reads, with every
  other row unchanged.
- Copy-on-write: a forked child's append leaves the parent's rows untouched.
- Invariants: constant segments, a permuted physical pool.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from oracle import zoomr_append as A
from oracle import zoomr_oracle as O


def _layer(dtype="bf16", **kw):
    base = dict(dtype=dtype, head_dim=64, batch=3, num_q_heads=4, num_kv_heads=2, seq_len=None,
                seq_len_range=(40, 130), seg_len_range=(5, 30), topk=2, window=8, seed=7)
    base.update(kw)
    st = W.make_structure(W.small_spec(**base), spare_blocks=6)
    lt = W.make_layer(st, 0, "cpu", keep_logical=True)
    return st, lt


def _np(x):
    return x.to(torch.float32).numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_segment_mean_is_the_exact_rational_mean_rounded(dtype):
    st, lt = _layer(dtype)
    kp = _np(lt.k_pool)
    for b in range(st.batch):
        L = int(st.seq_lens[b])
        for (s, e) in [(0, 1), (0, 16), (3, 35), (L - 13, L), (5, 37)]:
            if not 0 <= s < e <= L:
                continue
            for g in range(2):
                got = A.round_to_dtype(A.segment_mean(kp, st.block_tables[b], g, s, e), dtype)
                for c in range(0, kp.shape[-1], 9):
                    exact = sum(Fraction(float(kp[st.block_tables[b][t // 16], g, t % 16, c])) for t in range(s, e))
                    exact /= (e - s)
                    want32 = np.float32(float(exact))  # Fraction -> nearest double -> nearest float32
                    want = A.round_to_dtype(np.array([float(want32)]), dtype)[0]
                    assert got[c] == want, (b, s, e, g, c, got[c], want)


def test_segment_mean_matches_a_vectorised_mean_over_logical_rows():
    st, lt = _layer("bf16")
    kp, vp = _np(lt.k_pool), _np(lt.v_pool)
    for b in range(st.batch):
        lk = lt.logical_k[b].to(torch.float64).numpy()
        lv = lt.logical_v[b].to(torch.float64).numpy()
        bnd = st.bounds(b)
        for i in range(len(bnd) - 1):
            s, e = int(bnd[i]), int(bnd[i + 1])
            for g in range(2):
                assert np.array_equal(A.segment_mean(kp, st.block_tables[b], g, s, e), lk[s:e, g].mean(axis=0))
                assert np.array_equal(A.segment_mean(vp, st.block_tables[b], g, s, e), lv[s:e, g].mean(axis=0))


def test_appended_rows_read_back_through_the_block_tables_and_nothing_else_moves():
    st, lt = _layer("bf16")
    kp, vp = _np(lt.k_pool), _np(lt.v_pool)
    rng = np.random.default_rng(3)
    B, Hkv, d = st.batch, 2, kp.shape[-1]
    # append at each sequence's current end when it still fits in its blocks, else skip
    pos = [int(st.seq_lens[b]) if int(st.seq_lens[b]) % 16 else -1 for b in range(B)]
    kn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
    vn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
    kp2, vp2 = A.append_kv(kp, vp, st.block_tables, pos, kn, vn)
    for b in range(B):
        L = int(st.seq_lens[b])
        old = np.arange(L)
        for g in range(Hkv):
            assert np.array_equal(O.paged_rows(kp2, st.block_tables[b], g, old), O.paged_rows(kp, st.block_tables[b], g, old))
            if pos[b] >= 0:
                assert np.array_equal(O.paged_rows(kp2, st.block_tables[b], g, np.array([L]))[0], kn[b, g])
                assert np.array_equal(O.paged_rows(vp2, st.block_tables[b], g, np.array([L]))[0], vn[b, g])
    changed = np.argwhere(np.any(kp2 != kp, axis=(1, 2, 3))).ravel()
    want = sorted({int(st.block_tables[b][pos[b] // 16]) for b in range(B) if pos[b] >= 0})
    assert sorted(changed.tolist()) == want


def test_copy_on_write_leaves_the_parent_untouched():
    rng = np.random.default_rng(5)
    alloc = W.PagedBlockAllocator(12, rng)
    Hkv, d = 2, 8
    kp = rng.standard_normal((12, Hkv, 16, d)).astype(np.float32)
    vp = rng.standard_normal((12, Hkv, 16, d)).astype(np.float32)
    parent = alloc.alloc(3)  # 40 tokens: the last block holds 8
    L = 40
    child = alloc.fork(parent)
    copies = alloc.append_block(child)  # the child's last block is shared: copy it first
    assert len(copies) == 1 and child[-1] != parent[-1]
    kp2, vp2 = A.copy_blocks(kp, vp, copies)
    kn = rng.standard_normal((1, Hkv, d)).astype(np.float32)
    vn = rng.standard_normal((1, Hkv, d)).astype(np.float32)
    tabs = np.array([child], dtype=np.int64)
    kp3, vp3 = A.append_kv(kp2, vp2, tabs, [L], kn, vn)
    for g in range(Hkv):
        toks = np.arange(L)
        assert np.array_equal(O.paged_rows(kp3, np.array(parent), g, toks), O.paged_rows(kp, np.array(parent), g, toks))
        assert np.array_equal(O.paged_rows(kp3, np.array(child), g, toks), O.paged_rows(kp, np.array(parent), g, toks))
        assert np.array_equal(O.paged_rows(kp3, np.array(child), g, np.array([L]))[0], kn[0, g])
        assert np.array_equal(O.paged_rows(vp3, np.array(child), g, np.array([L]))[0], vn[0, g])


def test_constant_segment_and_permuted_pool():
    st, lt = _layer("f32")
    kp = _np(lt.k_pool)
    b, g = 1, 0
    kc = kp.copy()
    for t in range(4, 20):
        kc[st.block_tables[b][t // 16], g, t % 16, :] = 0.375
    assert np.all(A.segment_mean(kc, st.block_tables[b], g, 4, 20) == 0.375)
    perm = np.random.default_rng(1).permutation(kp.shape[0])
    inv = np.argsort(perm)
    kperm = kp[perm]
    bt = st.block_tables.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    for (s, e) in [(0, 9), (7, 40)]:
        assert np.array_equal(A.segment_mean(kp, st.block_tables[b], g, s, e), A.segment_mean(kperm, bt[b], g, s, e))


def test_planted_mistakes_are_caught():
    """An off-by-one segment end and a sum not divided by the count both disagree with the
    exact rational mean pinned above."""
    st, lt = _layer("f32")
    kp = _np(lt.k_pool)
    b, g, s, e = 0, 1, 2, 21
    good = A.segment_mean(kp, st.block_tables[b], g, s, e)
    assert not np.array_equal(A.segment_mean(kp, st.block_tables[b], g, s, e + 1), good)
    assert not np.allclose(good * (e - s), good)
