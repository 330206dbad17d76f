"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a library
routine (torch's scaled_dot_product_attention in fp64) in the special cases
where the step reduces to plain attention, exact rational arithmetic, a
pure-Python brute force with a different membership rule and no paging, hand-
computed rounding cases, and invariants (pool permutation, softmax mass,
convex hull of the attended values).
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from oracle import zoomr_oracle as O
from tests import brute_force as BF
from tests import near_ties as NT
from tests.helpers import oracle_args, unit_args


def _sdpa64(q_group: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """torch's fused attention in fp64 on the CPU: q [G, d], K/V [R, d] -> [G, d]."""
    qt = torch.from_numpy(np.asarray(q_group, np.float64))[None, :, None, :]  # [1, G, 1, d]
    kt = torch.from_numpy(np.asarray(K, np.float64))[None, None].expand(1, qt.shape[1], -1, -1)
    vt = torch.from_numpy(np.asarray(V, np.float64))[None, None].expand(1, qt.shape[1], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0, :, 0, :].numpy()


def _tiny(**kw):
    spec = W.small_spec(**kw)
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cpu", keep_logical=True)
    return st, lt


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("dtype,seed", [("f32", 0), ("bf16", 1), ("f32", 5)])
def test_dense_when_k_covers_all_segments(dtype, seed):
    """k >= n: every segment's tokens are gathered and no summary remains, so the
    step is plain softmax attention over all cached tokens (library routine on
    the logical, unpaged K/V)."""
    st, lt = _tiny(dtype=dtype, seed=seed, topk=1000, window=7, batch=2, num_q_heads=4, num_kv_heads=2)
    res = O.decode_step(**oracle_args(st, lt))
    G = 2
    for b in range(st.batch):
        for g in range(2):
            kl = W.to_numpy64(lt.logical_k[b])[:, g]
            vl = W.to_numpy64(lt.logical_v[b])[:, g]
            ref = _sdpa64(W.to_numpy64(lt.q)[b, g * G:(g + 1) * G], kl, vl)
            np.testing.assert_allclose(res.out[b, g * G:(g + 1) * G], ref, rtol=0, atol=1e-12)
            assert len(res.units[b][g].summaries) == 0
            assert list(res.units[b][g].tokens) == list(range(int(st.seq_lens[b])))


def test_pure_summary_when_k_and_window_are_zero():
    """k = 0 and w = 0 (the ZoomR page's SumR baseline, 4 Experiments): attention
    over the n summary vectors only."""
    st, lt = _tiny(topk=0, window=0, seed=3, num_q_heads=8, num_kv_heads=2)
    res = O.decode_step(**oracle_args(st, lt))
    s0, s1 = int(st.seg_ptr[0]), int(st.seg_ptr[1])
    for g in range(2):
        ref = _sdpa64(W.to_numpy64(lt.q)[0, 4 * g:4 * g + 4], W.to_numpy64(lt.sum_k)[s0:s1, g],
                      W.to_numpy64(lt.sum_v)[s0:s1, g])
        np.testing.assert_allclose(res.out[0, 4 * g:4 * g + 4], ref, rtol=0, atol=1e-12)
        assert len(res.units[0][g].tokens) == 0


def test_window_covering_everything_with_k_zero():
    """w >= L and k = 0: all tokens plus every segment's summary (the spec keeps
    a non-selected segment's summary even when its tokens sit in the window)."""
    st, lt = _tiny(topk=0, window=10_000, seed=4)
    res = O.decode_step(**oracle_args(st, lt))
    s0, s1 = int(st.seg_ptr[0]), int(st.seg_ptr[1])
    K = np.concatenate([W.to_numpy64(lt.logical_k[0])[:, 0], W.to_numpy64(lt.sum_k)[s0:s1, 0]])
    V = np.concatenate([W.to_numpy64(lt.logical_v[0])[:, 0], W.to_numpy64(lt.sum_v)[s0:s1, 0]])
    ref = _sdpa64(W.to_numpy64(lt.q)[0, 0:4], K, V)
    np.testing.assert_allclose(res.out[0, 0:4], ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed,topk,window,dtype", [(0, 2, 16, "f32"), (1, 3, 5, "bf16"), (2, 1, 0, "f32"),
                                                     (7, 4, 33, "bf16")])
def test_matches_pure_python_brute_force(seed, topk, window, dtype):
    st, lt = _tiny(seed=seed, topk=topk, window=window, dtype=dtype, head_dim=16, seq_len=80, seg_len_range=(5, 17),
                   num_q_heads=4, num_kv_heads=2)
    res = O.decode_step(**oracle_args(st, lt))
    for g in range(2):
        q, kl, vl, bounds, sk, sv = unit_args(st, lt, 0, g)
        exact = BF.exact_scores(q, sk)
        ex_sel = BF.dominant_subset(exact, topk)
        assert [Fraction(x) for x in res.units[0][g].keys] == exact
        out, sel, nrows = BF.brute_unit(q, kl, vl, bounds, sk, sv, topk, window, selected=ex_sel)
        u = res.units[0][g]
        assert list(u.sel) == sel
        np.testing.assert_allclose(u.out, np.array(out), rtol=0, atol=1e-12)
        assert u.probs.shape[1] == nrows


def test_gather_set_matches_per_token_predicate():
    rng = np.random.default_rng(11)
    for trial in range(200):
        L = int(rng.integers(1, 200))
        cuts = np.sort(rng.choice(np.arange(1, L), size=min(L - 1, int(rng.integers(0, 12))), replace=False)) \
            if L > 1 else np.array([], dtype=np.int64)
        bounds = np.concatenate([[0], cuts, [L]]).astype(np.int64)
        n = len(bounds) - 1
        sel = np.sort(rng.choice(n, size=int(rng.integers(0, n + 1)), replace=False))
        w = int(rng.integers(0, L + 5))
        tokens, summaries = O.gather_set(bounds, sel, L, w)
        want = [t for t in range(L) if BF.in_gather_set(t, L, w, bounds, set(int(x) for x in sel))]
        assert list(tokens) == want
        assert list(summaries) == [i for i in range(n) if i not in set(sel.tolist())]
        rngs = O.token_ranges(tokens)
        assert sum(int(e - s) for s, e in rngs) == len(tokens)
        assert all(rngs[i + 1, 0] > rngs[i, 1] for i in range(len(rngs) - 1))  # maximal runs


# ---------------------------------------------------------------- selection
def test_top_k_is_the_unique_dominant_subset():
    rng = np.random.default_rng(5)
    for trial in range(300):
        n = int(rng.integers(1, 9))
        keys = rng.integers(-3, 4, size=n).astype(np.float32)  # many exact ties
        k = int(rng.integers(0, n + 2))
        got = O.select_top_k(keys, k)
        assert list(got) == BF.dominant_subset([float(x) for x in keys], k)


def test_ties_go_to_lower_segment_index():
    st, lt = _tiny(seed=9, topk=2, window=0, num_q_heads=2, num_kv_heads=1)
    n = st.num_segments(0)
    assert n >= 5
    sk = lt.sum_k.clone()
    qsum = lt.q[0].to(torch.float64).sum(0)
    v = (qsum / qsum.norm() * 4.0).to(sk.dtype)
    for i in (1, 3, n - 1):  # three segments carry the very same summary key, bit for bit
        sk[i, 0] = v
    lt.sum_k = sk
    res = O.decode_step(**oracle_args(st, lt))
    keys = res.units[0][0].keys
    assert keys[1] == keys[3] == keys[n - 1] == keys.max()
    assert list(res.units[0][0].sel) == [1, 3]


def test_negative_zero_and_positive_zero_keys_tie():
    keys = np.array([0.0, -0.0, 0.0, -1.0], dtype=np.float32)
    assert list(O.select_top_k(keys, 2)) == [0, 1]
    keys = np.array([-0.0, 0.0], dtype=np.float32)
    assert list(O.select_top_k(keys, 1)) == [0]


def test_key_is_exact_where_an_fp32_chain_cancels():
    """Hand cases: 2^24 + 1 - 2^24 is 1 exactly (an fp32 chain in ascending order
    gives 0), in any order of the components; a product is not rounded before the
    add: (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24 exactly."""
    q = np.array([[1.0, 1.0, 1.0, 0.0]], dtype=np.float32)
    for s in ([2.0 ** 24, 1.0, -(2.0 ** 24), 5.0], [1.0, 2.0 ** 24, -(2.0 ** 24), 5.0],
              [2.0 ** 24, -(2.0 ** 24), 1.0, 5.0]):
        assert O.summary_keys(q, np.array([s], dtype=np.float32))[0] == 1
    a = np.float32(1.0 + 2.0 ** -12)
    key = O.summary_keys(np.array([[a]], np.float32), np.array([[a]], np.float32))[0]
    assert Fraction(key) == Fraction(1) + Fraction(1, 2 ** 11) + Fraction(1, 2 ** 24)


def test_inexact_fp64_sum_takes_the_fraction_route():
    """2^60 + 1 - 2^60: the fp64 sum loses the 1 (TwoSum flags it) and the key
    comes from exact rational arithmetic; a clean sum stays on the fp64 route."""
    q = np.array([[1.0, 1.0, 1.0], [0.5, 0.0, 0.0]], dtype=np.float32)
    s = np.array([[2.0 ** 60, 1.0, -(2.0 ** 60)], [3.0, 1.0, 2.0]], dtype=np.float32)
    dots, inexact = O.exact_dots(q, s)
    assert inexact[0, 0] and not inexact[1, 0] and not inexact[0, 1]
    assert isinstance(dots[0, 0], Fraction) and dots[0, 0] == 1
    assert dots[0, 1] == 2.0 ** 59 and dots[1, 0] == 6.0 and dots[1, 1] == 1.5
    assert list(O.summary_keys(q, s)) == [2.0 ** 59, 6.0]


@pytest.mark.parametrize("dtype,scale", [("f32", 1.0), ("bf16", 1.0), ("bf16", 1e-30), ("f32", 1e20)])
def test_keys_equal_the_exact_rational_score(dtype, scale):
    """Full-width (d = 128) random inputs, with a few values planted far below the
    rest (tiny and subnormal magnitudes) so that some fp64 sums are inexact: every
    key equals max over the group of the exact Fraction dot product."""
    rng = np.random.default_rng(31)
    G, n, d = 4, 12, 128
    q = rng.standard_normal((G, d)) * 3.0
    s = rng.standard_normal((n, d)) * 0.12 * scale
    s[2, 5] = 1e-30 * scale
    s[3, 7] = 3e-39  # subnormal in fp32 and bf16
    q[1, 9] = 2.0 ** -70
    s[4, :] = s[5, :]  # an exact tie
    q32 = torch.from_numpy(q).to(torch.float32).to(W.torch_dtype(dtype)).to(torch.float32).numpy()
    s32 = torch.from_numpy(s).to(torch.float32).to(W.torch_dtype(dtype)).to(torch.float32).numpy()
    dots, inexact = O.exact_dots(q32, s32)
    keys = O.summary_keys(q32, s32)
    exact = BF.exact_scores(q32, s32)
    for i in range(n):
        for h in range(G):
            assert Fraction(dots[i, h]) == BF.exact_dot(q32[h], s32[i])
        assert Fraction(keys[i]) == exact[i]
    assert keys[4] == keys[5]


def test_fp32_chain_and_exact_orders_disagree_on_planted_near_ties():
    """bf16 near-ties planted at the top-k boundary (two one-ulp nudges of a
    summary key) where an ascending fp32 chain ranks the pair the other way: the
    oracle's selection follows the exact scores."""
    st, lt = _tiny(seed=17, dtype="bf16", head_dim=128, seq_len=1024, seg_len_range=(32, 64), topk=4, window=0,
                   num_q_heads=8, num_kv_heads=2)
    flips = NT.plant_near_ties(st, lt)
    assert flips, "no near-tie planted"
    res = O.decode_step(**oracle_args(st, lt))
    for (b, g, i, j) in flips:
        q, _, _, _, sk, _ = unit_args(st, lt, b, g)
        exact = BF.exact_scores(q, sk)
        f32 = NT.fp32_chain_keys(q, sk)
        assert (exact[i] > exact[j]) != (f32[i] > f32[j] or (f32[i] == f32[j] and i < j))
        k = int(st.topk[b])
        assert list(res.units[b][g].sel) == sorted(sorted(range(len(exact)), key=lambda m: (-exact[m], m))[:k])
        assert list(res.units[b][g].sel) != list(O.select_top_k(f32, k))


def test_group_of_one_is_per_head_selection_and_mqa_shares_one():
    st, lt = _tiny(seed=13, num_q_heads=3, num_kv_heads=3, topk=2, window=4)  # G = 1
    res = O.decode_step(**oracle_args(st, lt))
    for g in range(3):
        q, _, _, _, sk, _ = unit_args(st, lt, 0, g)
        assert list(res.units[0][g].sel) == BF.dominant_subset(BF.exact_scores(q, sk), 2)
    st, lt = _tiny(seed=14, num_q_heads=6, num_kv_heads=1, topk=3, window=4)  # MQA: one group of all heads
    res = O.decode_step(**oracle_args(st, lt))
    q, _, _, _, sk, _ = unit_args(st, lt, 0, 0)
    per_head_max = [max(BF.exact_dot(q[h], s) for h in range(6)) for s in sk]
    assert list(res.units[0][0].sel) == BF.dominant_subset(per_head_max, 3)


# ---------------------------------------------------------------- invariants
def test_pool_permutation_invariance_bit_identical():
    """Permuting the physical pool and remapping the block tables leaves every
    output bit unchanged (the KV-cache management page: attention reads blocks
    through the table, so placement is invisible)."""
    st, lt = _tiny(seed=21, batch=3, num_q_heads=4, num_kv_heads=2, dtype="bf16", seq_len=120)
    a = oracle_args(st, lt)
    res0 = O.decode_step(**a)
    perm = np.random.default_rng(3).permutation(st.num_blocks)
    inv = np.argsort(perm)
    b = dict(a)
    b["k_pool"] = a["k_pool"][perm]
    b["v_pool"] = a["v_pool"][perm]
    bt = a["block_tables"].copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    b["block_tables"] = bt
    res1 = O.decode_step(**b)
    assert np.array_equal(res0.out, res1.out)
    assert np.array_equal(res0.sel, res1.sel)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_softmax_mass_and_convex_hull(seed):
    st, lt = _tiny(seed=seed, batch=2, num_q_heads=8, num_kv_heads=2, topk=3, window=9)
    res = O.decode_step(**oracle_args(st, lt))
    vp = W.to_numpy64(lt.v_pool)
    svs = W.to_numpy64(lt.sum_v)
    for b in range(2):
        for g in range(2):
            u = res.units[b][g]
            assert np.all(np.abs(u.probs.sum(axis=1) - 1.0) < 1e-12)
            assert np.all(u.probs >= 0)
            s0 = int(st.seg_ptr[b])
            V = np.concatenate([O.paged_rows(vp, st.block_tables[b], g, u.tokens), svs[s0 + u.summaries, g]])
            lo, hi = V.min(axis=0), V.max(axis=0)
            assert np.all(u.out >= lo[None] - 1e-12) and np.all(u.out <= hi[None] + 1e-12)


def test_planted_mistakes_are_caught():
    """Mutations of the oracle that a pin must reject: a dropped 1/sqrt(d), a
    window that is one token short, and ties going to the higher index."""
    st, lt = _tiny(seed=2, topk=2, window=6, num_q_heads=4, num_kv_heads=1, head_dim=16)
    q, kl, vl, bounds, sk, sv = unit_args(st, lt, 0, 0)
    sel = BF.dominant_subset(BF.exact_scores(q, sk), 2)
    ref, _, _ = BF.brute_unit(q, kl, vl, bounds, sk, sv, 2, 6, selected=sel)
    good = O.decode_step(**oracle_args(st, lt)).out[0, 0:4]
    assert np.max(np.abs(good - np.array(ref))) < 1e-12

    orig_attend = O.attend
    try:
        def no_scale(qv, K, V):
            o, p = orig_attend(qv * math.sqrt(len(qv)), K, V)
            return o, p
        O.attend = no_scale
        bad = O.decode_step(**oracle_args(st, lt)).out[0, 0:4]
    finally:
        O.attend = orig_attend
    assert np.max(np.abs(bad - np.array(ref))) > 1e-6

    orig_gather = O.gather_set
    try:
        O.gather_set = lambda bnd, s, L, w: orig_gather(bnd, s, L, max(w - 1, 0))
        bad = O.decode_step(**oracle_args(st, lt)).out[0, 0:4]
    finally:
        O.gather_set = orig_gather
    assert np.max(np.abs(bad - np.array(ref))) > 1e-9

    keys = np.array([1.0, 3.0, 3.0, 0.5], dtype=np.float32)
    wrong = sorted(sorted(range(4), key=lambda i: (-keys[i], -i))[:1])
    assert wrong != list(O.select_top_k(keys, 1)) == BF.dominant_subset(list(keys), 1)

    # a key taken as an ascending fp32 chain (rounded products and adds) picks the wrong segment
    q1 = np.ones((1, 3), np.float32)
    s2 = np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)], [0.5, 0.0, 0.0]], np.float32)
    assert list(O.select_top_k(O.summary_keys(q1, s2), 1)) == [0]
    assert list(O.select_top_k(NT.fp32_chain_keys(q1, s2), 1)) == [1]
