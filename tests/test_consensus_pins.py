"""Pins of the consensus oracle (``oracle/zoomr_consensus.py``) from outside it.

- Votes, I_all, I_c, I_s and I_f against a pure-Python brute force on
  integer-valued queries and mean keys (every fp32 dot is then exact).
- Vote-count invariants and closed forms: k >= n, c = 0, c >= |I_all|.
- The dense case (window over the whole sequence) against a library attention
  routine (torch's scaled_dot_product_attention in fp64) on the logical rows.
- Exact ties in the scores and in the votes go to the lower index.
- Planted mistakes fail the brute-force comparison.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from oracle import zoomr_consensus as OC
from oracle import zoomr_oracle as O


def _structure(**kw):
    return W.make_consensus_structure(W.consensus_spec(**kw))


def _mean_keys_int(st, layers, rng, lo=-3, hi=3):
    """Integer-valued mean keys [seg_ptr[B], Hkv, d] per layer (exact in fp32)."""
    sp = st.spec
    return [rng.integers(lo, hi + 1, size=(st.total_segments, sp.num_kv_heads, sp.head_dim)).astype(np.float32)
            for _ in range(layers)]


def _queries_int(st, layers, rng, lo=-3, hi=3):
    sp = st.spec
    return [rng.integers(lo, hi + 1, size=(st.batch, sp.num_q_heads, sp.head_dim)).astype(np.float32)
            for _ in range(layers)]


def _brute(st, qs, kbars, b, k, c):
    """Python-int scores, per-(layer, head) top-k, votes, consensus and I_f, written from the definitions."""
    sp = st.spec
    G = sp.num_q_heads // sp.num_kv_heads
    s0, s1 = int(st.seg_ptr[b]), int(st.seg_ptr[b + 1])
    n = s1 - s0
    votes = [0] * n
    for l in range(len(qs)):
        for h in range(sp.num_q_heads):
            q = [int(x) for x in qs[l][b, h]]
            scores = [sum(qa * int(ka) for qa, ka in zip(q, kbars[l][s0 + i, h // G])) for i in range(n)]
            ranked = sorted(range(n), key=lambda i: (-scores[i], i))
            for i in ranked[:min(k, n)]:
                votes[i] += 1
    i_all = [i for i in range(n) if votes[i] > 0]
    i_c = sorted(sorted(i_all, key=lambda i: (-votes[i], i))[:min(c, len(i_all))])
    i_s = [i for i in i_all if i not in i_c]
    bd = [int(x) for x in st.pair_bounds(b)]
    L = int(st.seq_lens[b])
    toks = set(range(int(st.prompt_lens[b]))) | set(range(max(0, L - st.window), L))
    for i in i_c:
        toks |= set(range(bd[2 * i], bd[2 * i + 1]))
    for i in i_s:
        toks |= set(range(bd[2 * i + 1], bd[2 * i + 2]))
    return votes, i_all, i_c, i_s, sorted(toks)


def _oracle_selection(st, qs, kbars, lt=None, attend_layers=()):
    pools_k = [W.to_numpy32(lt.k_pool)] * len(qs) if lt is not None else [None] * len(qs)
    pools_v = [W.to_numpy32(lt.v_pool)] * len(qs) if lt is not None else [None] * len(qs)
    return OC.consensus_step(qs, kbars, pools_k, pools_v, st.block_tables, st.seg_ptr, st.seg_bounds,
                             st.prompt_lens, st.seq_lens, st.topk, st.consensus, st.window,
                             attend_layers=list(attend_layers))


def _check_against_brute(st, qs, kbars):
    res = _oracle_selection(st, qs, kbars)
    for b in range(st.batch):
        votes, i_all, i_c, i_s, toks = _brute(st, qs, kbars, b, int(st.topk[b]), int(st.consensus[b]))
        r = res[b]
        assert r.votes.tolist() == votes, b
        assert r.i_all.tolist() == i_all and r.i_c.tolist() == i_c and r.i_s.tolist() == i_s, b
        assert r.tokens.tolist() == toks, b


@pytest.mark.parametrize("k,c,window", [(2, 2, 32), (1, 1, 0), (3, 5, 7), (13, 0, 16), (4, 40, 100)])
def test_selection_matches_integer_brute_force(k, c, window):
    st = _structure(topk=k, consensus=c, window=window, layers=3)
    rng = np.random.default_rng(k * 100 + c)
    _check_against_brute(st, _queries_int(st, 3, rng), _mean_keys_int(st, 3, rng))


def test_vote_invariants_on_real_valued_inputs():
    st = _structure(layers=2)
    sp = st.spec
    lts = [W.make_consensus_layer(st, l, "cpu") for l in range(2)]
    qs = [W.to_numpy32(lt.q) for lt in lts]
    rng = np.random.default_rng(3)
    kbars = [rng.standard_normal((st.total_segments, sp.num_kv_heads, sp.head_dim)).astype(np.float32)
             for _ in range(2)]
    res = _oracle_selection(st, qs, kbars)
    for b, r in enumerate(res):
        n = st.num_segments(b)
        k, c = int(st.topk[b]), int(st.consensus[b])
        assert int(r.votes.sum()) == 2 * sp.num_q_heads * min(k, n)
        assert r.votes.max() <= 2 * sp.num_q_heads
        assert sorted(set(r.i_c.tolist()) | set(r.i_s.tolist())) == r.i_all.tolist()
        assert not set(r.i_c.tolist()) & set(r.i_s.tolist())
        assert len(r.i_c) == min(c, len(r.i_all))
        for i in r.i_c:
            for j in r.i_s:
                assert (r.votes[i], -i) > (r.votes[j], -j)


def test_k_covering_all_segments_gives_every_segment_all_votes():
    st = _structure(topk=100, consensus=3, layers=2)
    sp = st.spec
    rng = np.random.default_rng(4)
    qs = [rng.standard_normal((st.batch, sp.num_q_heads, sp.head_dim)).astype(np.float32) for _ in range(2)]
    kbars = [rng.standard_normal((st.total_segments, sp.num_kv_heads, sp.head_dim)).astype(np.float32)
             for _ in range(2)]
    for b, r in enumerate(_oracle_selection(st, qs, kbars)):
        n = st.num_segments(b)
        assert r.votes.tolist() == [2 * sp.num_q_heads] * n
        assert r.i_c.tolist() == [0, 1, 2]  # all tied: the lowest indices
        bd = st.pair_bounds(b)
        L = int(st.seq_lens[b])
        want = set(range(int(st.prompt_lens[b]))) | set(range(L - st.window, L))
        for i in range(n):
            lo, hi = (bd[2 * i], bd[2 * i + 1]) if i < 3 else (bd[2 * i + 1], bd[2 * i + 2])
            want |= set(range(int(lo), int(hi)))
        assert r.tokens.tolist() == sorted(want)


@pytest.mark.parametrize("c", [0, 10_000])
def test_c_zero_keeps_only_summaries_and_large_c_only_regular_segments(c):
    st = _structure(consensus=c, topk=3, layers=2)
    rng = np.random.default_rng(5 + c)
    qs, kbars = _queries_int(st, 2, rng), _mean_keys_int(st, 2, rng)
    for b, r in enumerate(_oracle_selection(st, qs, kbars)):
        bd = st.pair_bounds(b)
        L = int(st.seq_lens[b])
        want = set(range(int(st.prompt_lens[b]))) | set(range(L - st.window, L))
        for i in r.i_all:
            lo, hi = (bd[2 * i + 1], bd[2 * i + 2]) if c == 0 else (bd[2 * i], bd[2 * i + 1])
            want |= set(range(int(lo), int(hi)))
        assert (len(r.i_c) == 0) if c == 0 else (len(r.i_s) == 0)
        assert r.tokens.tolist() == sorted(want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_window_over_the_whole_sequence_is_dense_attention(dtype):
    st = _structure(dtype=dtype, window=10_000, layers=1)
    sp = st.spec
    G = sp.num_q_heads // sp.num_kv_heads
    lt = W.make_consensus_layer(st, 0, "cpu", keep_logical=True)
    qs = [W.to_numpy32(lt.q)]
    rng = np.random.default_rng(6)
    kbars = [rng.standard_normal((st.total_segments, sp.num_kv_heads, sp.head_dim)).astype(np.float32)]
    res = _oracle_selection(st, qs, kbars, lt, attend_layers=[0])
    for b, r in enumerate(res):
        L = int(st.seq_lens[b])
        assert r.tokens.tolist() == list(range(L))
        for h in range(sp.num_q_heads):
            q = torch.from_numpy(W.to_numpy64(lt.q)[b, h]).view(1, 1, 1, -1)
            K = lt.logical_k[b][:, h // G].to(torch.float64).view(1, 1, L, -1)
            V = lt.logical_v[b][:, h // G].to(torch.float64).view(1, 1, L, -1)
            ref = torch.nn.functional.scaled_dot_product_attention(q, K, V)[0, 0, 0].numpy()
            np.testing.assert_allclose(r.out[0, h], ref, rtol=0, atol=1e-12)


def test_ties_in_scores_and_in_votes_go_to_the_lower_index():
    st = _structure(topk=1, consensus=1, layers=1, batch=1)
    sp = st.spec
    n = st.num_segments(0)
    kbar = np.zeros((st.total_segments, sp.num_kv_heads, sp.head_dim), np.float32)
    kbar[5] = kbar[2] = 1.0   # segments 2 and 5 tie for every head: k = 1 picks 2
    q = np.ones((1, sp.num_q_heads, sp.head_dim), np.float32)
    r = _oracle_selection(st, [q], [kbar])[0]
    assert r.i_all.tolist() == [2] and r.votes[2] == sp.num_q_heads
    # votes tie: half the heads prefer segment 7, half segment 4 (different KV heads) -> I_c = {4}
    kbar[:] = 0.0
    kbar[7, 0] = 1.0
    kbar[4, 1] = 1.0
    r = _oracle_selection(st, [q], [kbar])[0]
    assert r.i_all.tolist() == [4, 7] and r.votes[4] == r.votes[7] and r.i_c.tolist() == [4] and r.i_s.tolist() == [7]
    assert n > 7


def test_planted_mistakes_are_caught(monkeypatch):
    """Ties to the higher index, or summary and regular segments swapped in I_f, fail the brute force."""
    st = _structure(topk=2, consensus=2, layers=2)
    rng = np.random.default_rng(8)
    qs, kbars = _queries_int(st, 2, rng, -1, 1), _mean_keys_int(st, 2, rng, 0, 1)  # many ties
    _check_against_brute(st, qs, kbars)

    def top_k_high_ties(keys, k):
        n = len(keys)
        order = sorted(range(n), key=lambda i: (-float(keys[i]), -i))
        return np.array(sorted(order[:max(0, min(int(k), n))]), dtype=np.int64)

    with monkeypatch.context() as m:
        m.setattr(O, "select_top_k", top_k_high_ties)
        with pytest.raises(AssertionError):
            _check_against_brute(st, qs, kbars)
    real = OC.final_tokens
    with monkeypatch.context() as m:
        m.setattr(OC, "final_tokens", lambda bd, p, L, w, i_c, i_s: real(bd, p, L, w, i_s, i_c))
        with pytest.raises(AssertionError):
            _check_against_brute(st, qs, kbars)
