"""Pins of the amortisation oracle (``oracle/zoomr_amortise.py``) from outside it.

- With no new tokens the reused step is the full step (same selection, same window).
- The attended tokens after growth match a per-token predicate written from the reading.
- The dense case (window over the whole grown sequence) matches torch's fp64 attention on the logical
  rows plus the summary rows.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from oracle import zoomr_amortise as AM
from oracle import zoomr_oracle as O


def _grown(seed=31, extra=37, **kw):
    """A decode structure at its selection step, the same structure after ``extra`` more tokens per sequence
    (the last segment grows; new blocks come from the spares), and a layer holding the grown cache."""
    base = dict(dtype="f32", head_dim=64, batch=3, num_q_heads=4, num_kv_heads=2, seq_len=None,
                seq_len_range=(60, 150), seg_len_range=(5, 30), topk=2, window=16, seed=seed)
    base.update(kw)
    spec = W.small_spec(**base)
    st0 = W.make_structure(spec, spare_blocks=spec.batch * (extra // 16 + 2))
    Lg = st0.seq_lens.astype(np.int64) + extra
    cols = int(((Lg + 15) // 16).max())
    tables = np.full((st0.batch, cols), -1, np.int32)
    tables[:, :st0.max_blocks_per_seq] = st0.block_tables
    free = [x for x in range(st0.num_blocks) if x not in set(st0.block_tables.ravel().tolist())]
    for b in range(st0.batch):
        for j in range(int((Lg[b] + 15) // 16)):
            if tables[b, j] < 0:
                tables[b, j] = free.pop(0)
    bounds = st0.seg_bounds.copy()
    for b in range(st0.batch):
        bounds[int(st0.seg_ptr[b + 1]) + b] += extra  # the last segment grows
    grown = dataclasses.replace(st0, seq_lens=Lg.astype(np.int32), seg_bounds=bounds, block_tables=tables)
    lt = W.make_layer(grown, 0, "cpu", keep_logical=True)
    return st0, grown, lt


def _unit_inputs(st0, lt, b, g):
    G = st0.spec.num_q_heads // st0.spec.num_kv_heads
    s0, s1 = int(st0.seg_ptr[b]), int(st0.seg_ptr[b + 1])
    q = W.to_numpy32(lt.q)[b, g * G:(g + 1) * G]
    sk = W.to_numpy32(lt.sum_k)
    sv = W.to_numpy32(lt.sum_v)
    return q, st0.bounds(b), sk, sv


def test_no_growth_reuse_is_the_full_step():
    st, _, _ = _grown(extra=0)
    lt = W.make_layer(st, 0, "cpu")
    kp, vp = W.to_numpy32(lt.k_pool), W.to_numpy32(lt.v_pool)
    sk, sv = W.to_numpy32(lt.sum_k), W.to_numpy32(lt.sum_v)
    G = 2
    for b in range(st.batch):
        s0, s1 = int(st.seg_ptr[b]), int(st.seg_ptr[b + 1])
        for g in range(2):
            q = W.to_numpy32(lt.q)[b, g * G:(g + 1) * G]
            full = O.decode_unit(q, kp, vp, st.block_tables[b], g, st.bounds(b), sk[s0:s1, g], sv[s0:s1, g],
                                 int(st.topk[b]), st.window)
            r = AM.reuse_unit(q, kp, vp, st.block_tables[b], g, st.bounds(b), sk[s0:s1, g], sv[s0:s1, g], full.sel,
                              int(st.seq_lens[b]), st.window)
            assert np.array_equal(r.tokens, full.tokens) and np.array_equal(r.summaries, full.summaries)
            assert np.array_equal(r.out, full.out)


@pytest.mark.parametrize("extra,window", [(1, 16), (9, 4), (37, 16), (37, 0), (200, 64)])
def test_grown_token_set_matches_a_per_token_predicate(extra, window):
    st0, grown, lt = _grown(extra=min(extra, 37), window=window)
    rng = np.random.default_rng(extra)
    for b in range(st0.batch):
        n = st0.num_segments(b)
        sel = np.sort(rng.choice(n, size=min(2, n), replace=False))
        L0 = int(st0.seq_lens[b])
        Lnew = L0 + min(extra, 37)
        bnd = [int(x) for x in st0.bounds(b)]
        toks, sums = O.gather_set(st0.bounds(b), sel, Lnew, window)
        want = [t for t in range(Lnew)
                if t >= Lnew - window or any(bnd[i] <= t < bnd[i + 1] for i in sel)]
        assert toks.tolist() == want
        assert sums.tolist() == [i for i in range(n) if i not in set(sel.tolist())]
        q, bounds, sk, sv = _unit_inputs(st0, lt, b, 0)
        s0, s1 = int(st0.seg_ptr[b]), int(st0.seg_ptr[b + 1])
        r = AM.reuse_unit(q, W.to_numpy32(lt.k_pool), W.to_numpy32(lt.v_pool), grown.block_tables[b], 0, bounds,
                          sk[s0:s1, 0], sv[s0:s1, 0], sel, Lnew, window)
        assert r.tokens.tolist() == want


def test_dense_after_growth_matches_library_attention():
    st0, grown, lt = _grown(extra=25, window=10_000)
    G = 2
    kp, vp = W.to_numpy32(lt.k_pool), W.to_numpy32(lt.v_pool)
    for b in range(st0.batch):
        Lnew = int(grown.seq_lens[b])
        s0, s1 = int(st0.seg_ptr[b]), int(st0.seg_ptr[b + 1])
        sel = np.array([0], np.int64)
        q, bounds, sk, sv = _unit_inputs(st0, lt, b, 1)
        r = AM.reuse_unit(q, kp, vp, grown.block_tables[b], 1, bounds, sk[s0:s1, 1], sv[s0:s1, 1], sel, Lnew, 10_000)
        K = torch.cat([lt.logical_k[b][:, 1].double(), torch.from_numpy(sk[s0 + 1:s1, 1]).double()])
        V = torch.cat([lt.logical_v[b][:, 1].double(), torch.from_numpy(sv[s0 + 1:s1, 1]).double()])
        for h in range(G):
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q[h]).double().view(1, 1, 1, -1), K.view(1, 1, *K.shape), V.view(1, 1, *V.shape))
            np.testing.assert_allclose(r.out[h], ref[0, 0, 0].numpy(), rtol=0, atol=1e-12)


def test_consensus_final_set_after_growth_matches_a_predicate():
    st = W.make_consensus_structure(W.consensus_spec())
    b = 0
    bd = [int(x) for x in st.pair_bounds(b)]
    i_c, i_s = np.array([1, 4]), np.array([0, 2, 7])
    L0 = int(st.seq_lens[b])
    for extra, w in [(0, 32), (10, 32), (40, 5), (40, 0)]:
        Lnew = L0 + extra
        got = AM.reuse_final_tokens(np.array(bd), 32, Lnew, w, i_c, i_s).tolist()
        want = [t for t in range(Lnew) if t < 32 or t >= Lnew - w
                or any(bd[2 * i] <= t < bd[2 * i + 1] for i in i_c)
                or any(bd[2 * i + 1] <= t < bd[2 * i + 2] for i in i_s)]
        assert got == want, (extra, w)
