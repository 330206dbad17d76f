"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Selections, gathered token indices and ranges must match bit for bit; outputs
within max-abs 2e-3 (bf16) / 1e-5 (fp32). The five workloads run at their full
sizes; the 16K x 32-layer workload runs all 32 layers back to back with one plan,
as the benchmark does, and is checked on every unit's selection and on sampled
units' outputs.
"""

from __future__ import annotations

import dataclasses
import zlib

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import build as B
from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z
from oracle import zoomr_oracle as O
from tests import gpu_common as C
from tests.helpers import oracle_args

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    Z.load()


def _layer(spec, layer=0, **kw):
    st = W.make_structure(spec, **{k: v for k, v in kw.items() if k in ("spare_blocks", "seq_lens")})
    lt = W.make_layer(st, layer, "cuda", **{k: v for k, v in kw.items() if k in ("poison_unused",)})
    return st, lt


# ------------------------------------------------------------------ the five workloads
@pytest.mark.parametrize("cfg", [0, 1, 3, 4])
def test_workload_parity_full(cfg):
    st, lt = _layer(W.WORKLOADS[cfg])
    r = C.parity(st, lt)
    units = [(b, g) for b in range(st.batch) for g in range(st.spec.num_kv_heads)]
    print(f"cfg{cfg}: max_abs_err={r['max_abs_err']:.3g} "
          f"min_margin={C.min_score_margin(r['oracle'], units, st.topk):.3g}")


def test_headline_workload_32_layers():
    """8 x 16K, 32 layers: the benchmark's plan and launch sequence; every unit's
    selection and ranges bit-exact, sampled units' outputs within tolerance."""
    spec = W.WORKLOADS[2]
    st = W.make_structure(spec)
    plan = Z.DecodePlan.from_structure(st)
    bt = C.device_tables(st)
    layers = [W.make_layer(st, l, "cuda") for l in range(spec.layers)]
    outs, dbgs = [], []
    for lt in layers:
        o, d = C.run_gpu(plan, lt, bt)
        outs.append(o)
        dbgs.append(tuple(x.clone() for x in d))  # the next layer reuses nothing: keep its own copies
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    rng = np.random.default_rng(0)
    all_units = [(b, g) for b in range(st.batch) for g in range(spec.num_kv_heads)]
    worst = 0.0
    for l, lt in enumerate(layers):
        sel, rg, nr = (x.cpu().numpy() for x in dbgs[l])
        args = oracle_args(st, lt) if l in (0, 17, 31) else None
        if args is None:  # selection only: the oracle needs q and the summary keys, not the pool
            q = W.to_numpy32(lt.q)
            sk = W.to_numpy32(lt.sum_k)
            G = spec.num_q_heads // spec.num_kv_heads
            for (b, g) in all_units:
                s0, s1 = int(st.seg_ptr[b]), int(st.seg_ptr[b + 1])
                keys = O.summary_keys(q[b, g * G:(g + 1) * G], sk[s0:s1, g])
                sl = O.select_top_k(keys, int(st.topk[b]))
                toks, _ = O.gather_set(st.bounds(b), sl, int(st.seq_lens[b]), st.window)
                assert list(sel[b, g, :len(sl)]) == list(sl)
                assert np.array_equal(rg[b, g, :nr[b, g]], O.token_ranges(toks))
        else:
            sample = [all_units[i] for i in rng.choice(len(all_units), size=6, replace=False)]
            res = O.decode_step(**args, units=all_units if l == 0 else sample)
            C.check_selection(st, res.units, sel, rg, nr, all_units if l == 0 else sample)
            worst = max(worst, C.check_outputs(res, outs[l].cpu().numpy(), all_units if l == 0 else sample,
                                               spec.num_q_heads // spec.num_kv_heads, C.TOL["bf16"]))
    print(f"cfg2: max_abs_err={worst:.3g}")


# ------------------------------------------------------------------ edge cases
EDGE = {
    "pure_summaries": dict(topk=0, window=0),
    "dense_k_covers_all": dict(topk=10_000, window=3),
    "window_covers_all": dict(topk=0, window=100_000),
    "no_window": dict(topk=3, window=0),
    "one_token": dict(seq_len=1, seg_len_range=(1, 1), topk=1, window=4),
    "one_segment": dict(seq_len=77, seg_len_range=(200, 300), topk=1, window=5),
    "one_segment_k0": dict(seq_len=77, seg_len_range=(200, 300), topk=0, window=5),
    "many_chunks_ragged_tail": dict(seq_len=1001, seg_len_range=(17, 90), topk=10_000, window=7),
    "long_window_many_chunks": dict(seq_len=3000, seg_len_range=(40, 200), topk=4, window=1500),
    "group1": dict(num_q_heads=4, num_kv_heads=4),
    "group2": dict(num_q_heads=8, num_kv_heads=4),
    "group8_mqa": dict(num_q_heads=8, num_kv_heads=1),
    "group16_cuda_cores": dict(num_q_heads=16, num_kv_heads=1),
    "ragged_batch": dict(batch=5, seq_len=None, seq_len_range=(1, 700), topk=None, topk_range=(0, 6)),
    "shared_prefix": dict(batch=4, seq_len=None, seq_len_range=(300, 900), shared_prefix_tokens=256),
    "many_segments": dict(seq_len=3000, seg_len_range=(4, 8), topk=40, window=50),  # n ~ 500 > one per thread
    "very_many_segments": dict(batch=1, seq_len=4000, seg_len_range=(2, 6), topk=300, window=9),  # n ~ 1000
}


@pytest.mark.parametrize("dtype,head_dim", [("bf16", 128), ("bf16", 64), ("f32", 64), ("f32", 128)])
@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(name, dtype, head_dim):
    kw = dict(dtype=dtype, head_dim=head_dim, batch=2, num_q_heads=8, num_kv_heads=2, seq_len=300,
              seg_len_range=(10, 60), topk=3, window=20, seed=zlib.crc32(name.encode()) % 1000)
    kw.update(EDGE[name])
    st, lt = _layer(W.small_spec(**kw))
    C.parity(st, lt)


@pytest.mark.parametrize("merge", ["parts", "comp"])
@pytest.mark.parametrize("name", ["ragged_batch", "many_chunks_ragged_tail", "group8_mqa", "one_token", "shared_prefix"])
def test_both_merge_layouts(name, merge, monkeypatch):
    """The plan picks one of two merge layouts by shape; pin each in turn on the same inputs."""
    monkeypatch.setenv("ZOOMR_MERGE", merge)
    kw = dict(dtype="bf16", head_dim=128, batch=2, num_q_heads=8, num_kv_heads=2, seq_len=300,
              seg_len_range=(10, 60), topk=3, window=20, seed=zlib.crc32(name.encode()) % 1000)
    kw.update(EDGE[name])
    st, lt = _layer(W.small_spec(**kw))
    C.parity(st, lt)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_unowned_pool_rows_are_never_read(dtype):
    """NaN in every pool row no sequence owns (tails of last blocks, spare blocks)."""
    spec = W.small_spec(dtype=dtype, head_dim=128, batch=3, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=(5, 333), seg_len_range=(3, 40), topk=4, window=9, seed=5)
    st, lt = _layer(spec, spare_blocks=7, poison_unused=True)
    C.parity(st, lt)


def test_tied_summary_keys_go_to_the_lower_index():
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=1, num_q_heads=4, num_kv_heads=1, seq_len=400,
                        seg_len_range=(20, 40), topk=2, window=0, seed=9)
    st, lt = _layer(spec)
    n = st.num_segments(0)
    q = lt.q[0].to(torch.float64).sum(0)
    v = (q / q.norm() * 4.0).to(lt.sum_k.dtype)
    for i in (2, 5, n - 1):
        lt.sum_k[i, 0] = v
    r = C.parity(st, lt)
    assert list(r["sel"][0, 0, :2]) == [2, 5]


def test_pool_permutation_gives_identical_bits():
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=3, num_q_heads=8, num_kv_heads=2, seq_len=600,
                        seg_len_range=(10, 80), topk=3, window=33, seed=2)
    st, lt = _layer(spec)
    plan = Z.DecodePlan.from_structure(st).set_deterministic()  # bit-equal outputs across calls
    out0, _ = C.run_gpu(plan, lt, C.device_tables(st))
    perm = torch.randperm(st.num_blocks, generator=torch.Generator().manual_seed(1))
    inv = torch.argsort(perm)
    bt = st.block_tables.copy()
    bt[bt >= 0] = inv.numpy()[bt[bt >= 0]]
    lt.k_pool = lt.k_pool[perm.cuda()].contiguous()
    lt.v_pool = lt.v_pool[perm.cuda()].contiguous()
    out1, _ = C.run_gpu(plan, lt, torch.from_numpy(bt.astype(np.int32)).cuda())
    torch.cuda.synchronize()
    assert torch.equal(out0, out1)


_SMALL_BF16 = W.small_spec(dtype="bf16", head_dim=128, batch=3, num_q_heads=8, num_kv_heads=2, seq_len=300,
                           seg_len_range=(10, 40), topk=3, window=16, seed=5)


@pytest.mark.parametrize("wl", [1, 4, "small"])
def test_dynamic_split_repeated_calls_within_rounding_of_the_static_split(wl):
    """The attend-only calls' default split hands each unit's rows out in 32-row batches from a per-unit
    counter that returns to zero at the end of every call: twelve reuse calls on one workspace (eager, then
    replays of a captured graph) each equal the deterministic split's output up to the order of the sums,
    and that output equals the decode step's."""
    # "small": about one attend warp per 16 rows, so a unit has more home warps than 32-row batches and some
    # warps claim none (their partials are empty)
    st, lt = _layer(_SMALL_BF16 if wl == "small" else W.WORKLOADS[wl])
    plan = Z.DecodePlan.from_structure(st)
    det = Z.DecodePlan.from_structure(st).set_deterministic()
    bt = C.device_tables(st)
    step_out, _ = C.run_gpu(plan, lt, bt, debug=False)  # selects; leaves the ranges in the workspace
    C.run_gpu(det, lt, bt, debug=False)
    ref = torch.empty_like(step_out)
    det.run_reuse(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, ref)
    torch.cuda.synchronize()
    assert torch.equal(ref, step_out)  # the even split in both: the same bits
    outs = []
    for _ in range(4):
        out = torch.full_like(ref, float("nan"))
        plan.run_reuse(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out)
        torch.cuda.synchronize()
        outs.append(out)
    g_out = torch.empty_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            plan.run_reuse(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, g_out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(8):
        g_out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        outs.append(g_out.clone())
    assert plan.device_error() == 0
    for out in outs:
        assert torch.isfinite(out).all()
        torch.testing.assert_close(out, ref, rtol=1e-5, atol=1e-5)
    plan.close()
    det.close()


def test_repeated_calls_are_deterministic_and_graph_capture_replays():
    st, lt = _layer(W.WORKLOADS[1])
    plan = Z.DecodePlan.from_structure(st).set_deterministic()
    bt = C.device_tables(st)
    a, _ = C.run_gpu(plan, lt, bt, debug=False)
    b, _ = C.run_gpu(plan, lt, bt, debug=False)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out, stream=s)  # warm-up on the side stream
        with torch.cuda.graph(g, stream=s):
            plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, out)
    # the timed entry point computes the same thing
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c = torch.empty_like(a)
    plan.run_timed(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, c, e0, e1)
    torch.cuda.synchronize()
    assert torch.equal(a, c) and e0.elapsed_time(e1) > 0
    # either event alone: the one before the attend kernel, or the one after it
    for ev0, ev1 in ((None, e1), (e0, None)):
        c.zero_()
        plan.run_timed(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, c, ev0, ev1)
        torch.cuda.synchronize()
        assert torch.equal(a, c)


def test_out_of_pool_block_id_sets_the_error_word_and_nothing_faults():
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=2, num_q_heads=8, num_kv_heads=2, seq_len=200,
                        seg_len_range=(10, 30), topk=10_000, window=5, seed=3)
    st, lt = _layer(spec)
    plan = Z.DecodePlan.from_structure(st)
    bt = st.block_tables.copy()
    bt[1, 3] = st.num_blocks + 1000  # outside the pool: the kernel must skip the row and flag it
    out, _ = C.run_gpu(plan, lt, torch.from_numpy(bt.astype(np.int32)).cuda(), debug=False)
    torch.cuda.synchronize()
    assert plan.device_error() == 1  # bit 1: a physical block id outside the pool
    assert plan.device_error() == 0  # read-and-clear
    # sequence 0 is untouched by the bad entry and still matches the oracle
    res = O.decode_step(**oracle_args(st, lt), units=[(0, 0), (0, 1)])
    C.check_outputs(res, out.cpu().numpy(), [(0, 0), (0, 1)], 4, C.TOL["bf16"])
    # the library stays usable
    C.parity(st, lt, plan=plan)


def test_exact_key_decides_where_an_fp32_chain_cancels():
    """The ranking key is the exact dot product. Summary keys built so that an fp32 chain in
    ascending order gives different keys and a different top-2: 2^24 + 1 - 2^24 is 1 exactly (0 in
    that chain). Two KV heads, each with one query head of its group carrying the signal, once in
    each half of a packed pair."""
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=1, num_q_heads=8, num_kv_heads=2, seq_len=64,
                        seg_len_range=(16, 16), topk=2, window=0, seed=7)
    st, lt = _layer(spec)
    assert int(st.seg_ptr[1]) == 4
    big = float(2 ** 24)
    rows = [[big, 1.0, -big], [0.5], [1.0, 1.0, -big, big], [-1.0]]  # exact keys 1, 0.5, 2, 0 (max with 0)
    sk = torch.zeros_like(lt.sum_k)
    for i, r in enumerate(rows):
        sk[i, :, :len(r)] = torch.tensor(r, dtype=torch.float32).to(sk.dtype)
    q = torch.zeros_like(lt.q)
    q[0, 1] = 1.0  # KV head 0: the second query head of its group (odd half of the pair)
    q[0, 4] = 1.0  # KV head 1: the first query head of its group (even half)
    lt = dataclasses.replace(lt, sum_k=sk, q=q)
    r = C.parity(st, lt)
    for g in range(2):
        assert list(r["sel"][0, g, :2]) == [0, 2]
        assert list(r["oracle"].units[0][g].sel) == [0, 2]
