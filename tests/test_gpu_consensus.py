"""GPU parity of ZoomR's consensus path (``zr_consensus_*``) against ``oracle/zoomr_consensus.py``.

Each side computes its own mean summary keys (the device with ``zr_segment_summaries`` over the summary
spans, the oracle with its segment means; the two are checked bit-equal), then the votes, the consensus
set and the final token ranges must match bit for bit, and every layer's outputs within 2e-3 (bf16) /
1e-5 (fp32).
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z
from oracle import zoomr_append as A
from oracle import zoomr_consensus as OC
from oracle import zoomr_oracle as O
from tests.gpu_common import TOL

pytestmark = pytest.mark.gpu


def _np32(t):
    return t.detach().to(torch.float32).cpu().numpy()


def _summary_segs(st):
    return [(b, s, e, int(st.seg_ptr[b]) + i) for b in range(st.batch) for i, (s, e) in enumerate(st.summary_spans(b))]


def _cache_cfg(st):
    sp = st.spec
    return Z.cache_config(batch=st.batch, num_kv_heads=sp.num_kv_heads, head_dim=sp.head_dim,
                          num_blocks=st.num_blocks, max_blocks_per_seq=st.max_blocks_per_seq, dtype=sp.dtype)


def _device_mean_keys(st, lt, bt):
    segs = torch.tensor(_summary_segs(st), dtype=torch.int32, device="cuda")
    sp = st.spec
    mk = torch.empty((st.total_segments, sp.num_kv_heads, sp.head_dim), dtype=W.torch_dtype(sp.dtype), device="cuda")
    mv = torch.empty_like(mk)
    Z.zr_segment_summaries(_cache_cfg(st), segs, bt, lt.k_pool, lt.v_pool, mk, mv)
    return mk


def _oracle_mean_keys(st, kp):
    sp = st.spec
    mk = np.empty((st.total_segments, sp.num_kv_heads, sp.head_dim), np.float32)
    for (b, s, e, r) in _summary_segs(st):
        for g in range(sp.num_kv_heads):
            mk[r, g] = A.round_to_dtype(A.segment_mean(kp, st.block_tables[b], g, s, e), sp.dtype)
    return mk


def _run(st, lts, steps=1):
    """Device: mean keys, votes of every layer, one selection, every layer's attention (``steps`` times)."""
    plan = Z.ConsensusPlan.from_structure(st)
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    sp = st.spec
    mks = [_device_mean_keys(st, lt, bt) for lt in lts]
    outs = []
    for _ in range(steps):
        dbg = plan.new_debug_outputs()
        for l, lt in enumerate(lts):
            plan.vote(lt.q, mks[l])
        plan.select(dbg)
        o = [torch.full((st.batch, sp.num_q_heads, sp.head_dim), float("nan"), device="cuda") for _ in lts]
        for l, lt in enumerate(lts):
            plan.attend(lt.q, lt.k_pool, lt.v_pool, bt, o[l])
        torch.cuda.synchronize()
        outs.append(([x.cpu().numpy() for x in dbg], [x.cpu().numpy() for x in o]))
    err = plan.device_error()
    plan.close()
    return mks, outs, err


def _check(st, lts, steps=1):
    mks, outs, err = _run(st, lts, steps)
    assert err == 0
    sp = st.spec
    kps = [_np32(lt.k_pool) for lt in lts]
    vps = [_np32(lt.v_pool) for lt in lts]
    kbars = [_oracle_mean_keys(st, kp) for kp in kps]
    for l in range(len(lts)):
        assert np.array_equal(_np32(mks[l]).view(np.uint32), kbars[l].view(np.uint32)), l
    res = OC.consensus_step([_np32(lt.q) for lt in lts], kbars, kps, vps, st.block_tables, st.seg_ptr,
                            st.seg_bounds, st.prompt_lens, st.seq_lens, st.topk, st.consensus, st.window)
    worst = 0.0
    for (votes, ic, rng, nr), o in outs:
        for b, r in enumerate(res):
            n = st.num_segments(b)
            assert votes[b, :n].tolist() == r.votes.tolist(), b
            assert np.all(votes[b, n:] == 0)
            assert ic[b, :len(r.i_c)].tolist() == r.i_c.tolist() and np.all(ic[b, len(r.i_c):] == -1), b
            assert np.array_equal(rng[b, :nr[b]], O.token_ranges(r.tokens)), b
            for l in range(len(lts)):
                e = float(np.max(np.abs(o[l][b].astype(np.float64) - r.out[l])))
                assert np.isfinite(e) and e <= TOL[sp.dtype], (b, l, e)
                worst = max(worst, e)
    return res, worst


def _setup(**kw):
    st = W.make_consensus_structure(W.consensus_spec(**kw))
    lts = [W.make_consensus_layer(st, l, "cuda") for l in range(st.spec.layers)]
    return st, lts


@pytest.mark.parametrize("dtype,d,hq,hkv", [("f32", 64, 8, 2), ("bf16", 128, 8, 2), ("bf16", 64, 16, 4),
                                            ("bf16", 128, 32, 2), ("f32", 128, 4, 4)])
def test_consensus_matches_the_oracle(dtype, d, hq, hkv):
    st, lts = _setup(dtype=dtype, head_dim=d, num_q_heads=hq, num_kv_heads=hkv, layers=3)
    _check(st, lts)


@pytest.mark.parametrize("kw", [
    dict(topk=1, consensus=1),
    dict(topk=100, consensus=0),          # every summary voted for; none zoomed: summaries only
    dict(topk=3, consensus=100),          # every candidate zoomed
    dict(prompt_len=0, window=0, topk=2),  # pieces only
    dict(window=10_000),                  # the window covers everything
    dict(prompt_len=0, window=5, topk=0, consensus=3),  # no votes: the window alone
    dict(prompt_len=5, window=0, topk=0),  # no votes: the prompt alone
])
def test_consensus_edge_settings(kw):
    st, lts = _setup(dtype="bf16", head_dim=128, layers=2, **kw)
    _check(st, lts)


def test_repeated_selections_start_from_cleared_votes():
    st, lts = _setup(dtype="bf16", head_dim=128, layers=2)
    _check(st, lts, steps=3)


def test_plan_kinds_are_not_interchangeable():
    st, lts = _setup(dtype="bf16", head_dim=128, layers=1)
    cplan = Z.ConsensusPlan.from_structure(st)
    lib = Z.load()
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    out = torch.empty((st.batch, st.spec.num_q_heads, 128), device="cuda")
    p = Z._dev
    assert lib.zr_decode_attend(cplan.handle, p(cplan.ws), p(lts[0].q), p(lts[0].k_pool), p(lts[0].v_pool), p(bt),
                                p(lts[0].k_pool), p(lts[0].v_pool), p(out), None, None, None, None) == Z.ZR_EINVAL
    k, n = torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32)
    assert lib.zr_plan_dims(cplan.handle, Z._ptr32(k.numpy()), Z._ptr32(n.numpy())) == Z.ZR_EINVAL
    dst = W.make_structure(W.small_spec(dtype="bf16", head_dim=128, num_q_heads=8, num_kv_heads=2))
    dplan = Z.DecodePlan.from_structure(dst)
    assert lib.zr_consensus_vote(dplan.handle, p(dplan.ws), p(lts[0].q), p(lts[0].k_pool), None) == Z.ZR_EINVAL
    assert lib.zr_consensus_select(dplan.handle, p(dplan.ws), None, None, None, None, None) == Z.ZR_EINVAL
    assert lib.zr_consensus_attend(dplan.handle, p(dplan.ws), p(lts[0].q), p(lts[0].k_pool), p(lts[0].v_pool),
                                   p(bt), p(out), None) == Z.ZR_EINVAL
    cplan.close()
    dplan.close()


def test_full_size_votes_and_sampled_attention():
    """The 16K-token, batch-8, 32-layer, 32/8-head bf16 workload: the votes of all 32 layers, the consensus and
    the final ranges of every sequence bit-exact; attention checked on layers 0 and 31 of sequences 0 and 5."""
    st = W.make_consensus_structure(W.CONSENSUS_WORKLOADS[1])
    lts = [W.make_consensus_layer(st, l, "cuda") for l in range(st.spec.layers)]
    mks, outs, err = _run(st, lts)
    assert err == 0
    sp = st.spec
    # the oracle's mean keys, from the blocks that hold summary tokens only (a compact copy of the pool)
    blocks = sorted({int(st.block_tables[b, t // 16]) for (b, s, e, _) in _summary_segs(st) for t in range(s, e)})
    remap = np.full(st.num_blocks, -1, np.int64)
    remap[blocks] = np.arange(len(blocks))
    small_tables = np.where(st.block_tables >= 0, remap[np.maximum(st.block_tables, 0)], -1)
    kbars = []
    for l, lt in enumerate(lts):
        kp_small = _np32(lt.k_pool[torch.tensor(blocks, device="cuda")])
        want = np.empty((st.total_segments, sp.num_kv_heads, sp.head_dim), np.float32)
        for (b, s, e, r) in _summary_segs(st):
            for g in range(sp.num_kv_heads):
                want[r, g] = A.round_to_dtype(A.segment_mean(kp_small, small_tables[b], g, s, e), "bf16")
        assert np.array_equal(_np32(mks[l]).view(np.uint32), want.view(np.uint32)), l
        kbars.append(want)
    layers = [0, 31]
    kp = {l: _np32(lts[l].k_pool) for l in layers}
    vp = {l: _np32(lts[l].v_pool) for l in layers}
    res = OC.consensus_step([_np32(lt.q) for lt in lts], kbars, [kp.get(l) for l in range(sp.layers)],
                            [vp.get(l) for l in range(sp.layers)], st.block_tables, st.seg_ptr, st.seg_bounds,
                            st.prompt_lens, st.seq_lens, st.topk, st.consensus, st.window, attend_layers=[],
                            batch=None)
    (votes, ic, rng, nr), o = outs[0]
    for b, r in enumerate(res):
        n = st.num_segments(b)
        assert votes[b, :n].tolist() == r.votes.tolist(), b
        assert ic[b, :len(r.i_c)].tolist() == r.i_c.tolist(), b
        assert np.array_equal(rng[b, :nr[b]], O.token_ranges(r.tokens)), b
    G = sp.num_q_heads // sp.num_kv_heads
    for b in (0, 5):
        for l in layers:
            want = OC.attend_final(_np32(lts[l].q)[b], kp[l], vp[l], st.block_tables[b], res[b].tokens, G)
            assert np.max(np.abs(o[l][b].astype(np.float64) - want)) <= TOL["bf16"], (b, l)


def test_timed_attend_matches_and_times_the_kernel():
    """zr_consensus_attend_timed: the same outputs as zr_consensus_attend, with events around the
    gather-attention kernel (either one alone works too)."""
    st, lts = _setup(dtype="bf16", head_dim=128, num_q_heads=8, num_kv_heads=2, layers=1)
    plan = Z.ConsensusPlan.from_structure(st).set_deterministic()  # bit-equal outputs across calls
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    sp = st.spec
    mk = _device_mean_keys(st, lts[0], bt)
    plan.vote(lts[0].q, mk)
    plan.select()
    ref = torch.empty((st.batch, sp.num_q_heads, sp.head_dim), device="cuda")
    plan.attend(lts[0].q, lts[0].k_pool, lts[0].v_pool, bt, ref)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for a_, b_ in ((e0, e1), (e0, None), (None, e1)):
        out = torch.full_like(ref, float("nan"))
        plan.attend_timed(lts[0].q, lts[0].k_pool, lts[0].v_pool, bt, out, a_, b_)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    plan.attend_timed(lts[0].q, lts[0].k_pool, lts[0].v_pool, bt, out, e0, e1)
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) > 0
    assert plan.device_error() == 0
    plan.close()


def test_dynamic_split_within_rounding_of_the_even_split():
    """Consensus attention takes the dynamic split by default: ten calls on one workspace (the per-unit batch
    counters return to zero after each) all equal the deterministic plan's output up to the order of the
    sums, at the full 8B shape with 16K generated tokens (two layers)."""
    st = W.make_consensus_structure(dataclasses.replace(W.CONSENSUS_WORKLOADS[1], layers=2))
    lts = [W.make_consensus_layer(st, l, "cuda") for l in range(2)]
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    sp = st.spec
    outs = {}
    for det in (True, False):
        plan = Z.ConsensusPlan.from_structure(st).set_deterministic(det)
        mks = [_device_mean_keys(st, lt, bt) for lt in lts]
        for l, lt in enumerate(lts):
            plan.vote(lt.q, mks[l])
        plan.select()
        got = []
        for _ in range(1 if det else 5):
            for lt in lts:
                out = torch.full((st.batch, sp.num_q_heads, sp.head_dim), float("nan"), device="cuda")
                plan.attend(lt.q, lt.k_pool, lt.v_pool, bt, out)
                got.append(out)
        torch.cuda.synchronize()
        assert plan.device_error() == 0
        outs[det] = got
        plan.close()
    ref = outs[True]
    for i, out in enumerate(outs[False]):
        assert torch.isfinite(out).all()
        torch.testing.assert_close(out, ref[i % len(lts)], rtol=1e-5, atol=1e-5)
