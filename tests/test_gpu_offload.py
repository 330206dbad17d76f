"""K/V pools resident in pinned host memory (the pages' offloaded cache, read by the kernels across the
CPU-GPU link): every path gives the same bits as with the pools in HBM, and the decode step matches the
oracle."""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z
from tests import gpu_common as C

pytestmark = pytest.mark.gpu


def _pinned(t: torch.Tensor) -> torch.Tensor:
    return t.cpu().pin_memory()


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.cpu().view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32),
                       b.cpu().view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32))


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_decode_with_host_resident_pools(dtype, d):
    spec = W.small_spec(dtype=dtype, head_dim=d, batch=4, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=(200, 700), seg_len_range=(10, 60), topk=3, window=32, seed=21)
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cuda")
    lt_host = dataclasses.replace(lt, k_pool=_pinned(lt.k_pool), v_pool=_pinned(lt.v_pool))
    plan = Z.DecodePlan.from_structure(st).set_deterministic()  # bit-equal outputs across calls
    bt = C.device_tables(st)
    out_dev, dbg_dev = C.run_gpu(plan, lt, bt)
    out_host, dbg_host = C.run_gpu(plan, lt_host, bt)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    assert torch.equal(out_dev, out_host)
    for a, b in zip(dbg_dev, dbg_host):
        assert torch.equal(a, b)
    C.parity(st, lt_host, plan)
    plan.close()


def test_consensus_with_host_resident_pools():
    st = W.make_consensus_structure(W.consensus_spec(dtype="bf16", head_dim=128, layers=2))
    lts = [W.make_consensus_layer(st, l, "cuda") for l in range(2)]
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    sp = st.spec
    cfg = Z.cache_config(batch=st.batch, num_kv_heads=sp.num_kv_heads, head_dim=sp.head_dim,
                         num_blocks=st.num_blocks, max_blocks_per_seq=st.max_blocks_per_seq, dtype=sp.dtype)
    segs = torch.tensor([(b, s, e, int(st.seg_ptr[b]) + i) for b in range(st.batch)
                         for i, (s, e) in enumerate(st.summary_spans(b))], dtype=torch.int32, device="cuda")
    outs = []
    for host in (False, True):
        pools = [(_pinned(lt.k_pool), _pinned(lt.v_pool)) if host else (lt.k_pool, lt.v_pool) for lt in lts]
        plan = Z.ConsensusPlan.from_structure(st).set_deterministic()  # bit-equal outputs across calls
        mks = []
        for (kp, vp) in pools:
            mk = torch.empty((st.total_segments, sp.num_kv_heads, sp.head_dim), dtype=torch.bfloat16, device="cuda")
            Z.zr_segment_summaries(cfg, segs, bt, kp, vp, mk, torch.empty_like(mk))
            mks.append(mk)
        for l, lt in enumerate(lts):
            plan.vote(lt.q, mks[l])
        dbg = plan.new_debug_outputs()
        plan.select(dbg)
        o = [torch.empty((st.batch, sp.num_q_heads, sp.head_dim), device="cuda") for _ in lts]
        for l, lt in enumerate(lts):
            plan.attend(lt.q, pools[l][0], pools[l][1], bt, o[l])
        torch.cuda.synchronize()
        assert plan.device_error() == 0
        outs.append((mks, dbg, o))
        plan.close()
    (mk0, dbg0, o0), (mk1, dbg1, o1) = outs
    for a, b in zip(mk0, mk1):
        assert _same(a, b)
    for a, b in zip(dbg0, dbg1):
        assert torch.equal(a, b)
    for a, b in zip(o0, o1):
        assert torch.equal(a, b)


def test_append_into_host_resident_pools():
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=3, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=(40, 90), seg_len_range=(8, 30), seed=22)
    st = W.make_structure(spec, spare_blocks=4)
    lt = W.make_layer(st, 0, "cuda")
    cfg = Z.cache_config(batch=st.batch, num_kv_heads=2, head_dim=128, num_blocks=st.num_blocks,
                         max_blocks_per_seq=st.max_blocks_per_seq, dtype="bf16")
    pos = torch.tensor([int(x) - 1 for x in st.seq_lens], dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    kn = torch.randn((st.batch, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    vn = torch.randn((st.batch, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
    kh, vh = _pinned(lt.k_pool), _pinned(lt.v_pool)
    bt = C.device_tables(st)
    Z.zr_append_kv(cfg, pos, kn, vn, bt, lt.k_pool, lt.v_pool)
    Z.zr_append_kv(cfg, pos, kn, vn, bt, kh, vh)
    torch.cuda.synchronize()
    assert _same(lt.k_pool, kh) and _same(lt.v_pool, vh)


# ------------------------------------------------------------------ staged offload (ZoomR 3.4, Decoding Stage)
def _np32(t):
    return t.detach().to(torch.float32).cpu().numpy()


def _touched_blocks(st, tokens_by_seq):
    """Physical blocks the token sets touch, through the block tables (each shared block once)."""
    blocks = set()
    for b, toks in tokens_by_seq.items():
        for lb in sorted(set(int(t) // 16 for t in toks)):
            blocks.add(int(st.block_tables[b, lb]))
    return sorted(blocks)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_staged_consensus_layers_match_the_oracle(dtype, d):
    """Every layer's pools in pinned host memory; per layer the rows of I_f are staged into one of two
    HBM staging pools on a copy stream (the next layer's while the current one attends), and the
    attention runs over the staging pools through the remapped tables. Outputs against the oracle; the
    staging pools start as NaN, so a row that was not staged and were read would show; the rows staged
    are exactly the rows of I_f (every KV head)."""
    from oracle import zoomr_append as OA
    from oracle import zoomr_consensus as OC

    st = W.make_consensus_structure(W.consensus_spec(dtype=dtype, head_dim=d, num_q_heads=8, num_kv_heads=2,
                                                     layers=3, seed=61))
    lts = [W.make_consensus_layer(st, l, "cuda") for l in range(3)]
    sp = st.spec
    G = sp.num_q_heads // sp.num_kv_heads
    kps = [_np32(lt.k_pool) for lt in lts]
    vps = [_np32(lt.v_pool) for lt in lts]
    kbars = []
    for kp in kps:
        mk = np.empty((st.total_segments, sp.num_kv_heads, d), np.float32)
        for b in range(st.batch):
            for i, (s, e) in enumerate(st.summary_spans(b)):
                for g in range(sp.num_kv_heads):
                    mk[int(st.seg_ptr[b]) + i, g] = OA.round_to_dtype(OA.segment_mean(kp, st.block_tables[b], g, s, e),
                                                                     dtype)
        kbars.append(mk)
    tdt = W.torch_dtype(dtype)
    host = [(_pinned(lt.k_pool), _pinned(lt.v_pool)) for lt in lts]
    for lt in lts:  # the cache now lives in host memory only
        lt.k_pool = lt.v_pool = None
    torch.cuda.empty_cache()
    plan = Z.ConsensusPlan.from_structure(st)
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    for l, lt in enumerate(lts):
        plan.vote(lt.q, torch.from_numpy(kbars[l]).to(tdt).cuda())
    dbg = plan.new_debug_outputs()
    plan.select(dbg)
    cap = st.num_blocks
    stage_ids = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    remap = torch.empty_like(bt)
    n_staged = torch.zeros(1, dtype=torch.int32, device="cuda")
    Z.zr_offload_map(plan.handle, plan.ws, bt, cap, stage_ids, remap, n_staged)
    bufs = [(torch.full((cap, sp.num_kv_heads, 16, d), float("nan"), dtype=tdt, device="cuda"),
             torch.full((cap, sp.num_kv_heads, 16, d), float("nan"), dtype=tdt, device="cuda")) for _ in range(2)]
    outs = [torch.full((st.batch, sp.num_q_heads, d), float("nan"), device="cuda") for _ in lts]
    main, copy = torch.cuda.current_stream(), torch.cuda.Stream()
    staged = [torch.cuda.Event() for _ in lts]
    freed = [torch.cuda.Event() for _ in lts]
    copy.wait_stream(main)
    for l, lt in enumerate(lts):  # issued in this order, so every event is recorded before it is waited on
        if l >= 2:
            copy.wait_event(freed[l - 2])  # buffer l % 2 is free once layer l - 2 has attended
        Z.zr_offload_stage(plan.handle, plan.ws, host[l][0], host[l][1], stage_ids, n_staged, cap, bufs[l % 2][0],
                           bufs[l % 2][1], stream=copy)
        staged[l].record(copy)
        main.wait_event(staged[l])
        plan.attend(lt.q, bufs[l % 2][0], bufs[l % 2][1], remap, outs[l])
        freed[l].record(main)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    res = OC.consensus_step([_np32(lt.q) for lt in lts], kbars, kps, vps, st.block_tables, st.seg_ptr,
                            st.seg_bounds, st.prompt_lens, st.seq_lens, st.topk, st.consensus, st.window)
    want_blocks = _touched_blocks(st, {b: r.tokens for b, r in enumerate(res)})
    n = int(n_staged.item())
    assert n == len(want_blocks)
    assert stage_ids[:n].cpu().tolist() == want_blocks
    for b, r in enumerate(res):
        for l in range(len(lts)):
            e = float(np.max(np.abs(outs[l][b].cpu().numpy().astype(np.float64) - r.out[l])))
            assert np.isfinite(e) and e <= C.TOL[dtype], (b, l, e)
    # the staged rows of the last layer's pool: exactly I_f's rows, all KV heads
    slot_of = {blk: i for i, blk in enumerate(want_blocks)}
    want_rows = np.zeros((n, sp.num_kv_heads, 16), bool)
    for b, r in enumerate(res):
        for t in r.tokens:
            want_rows[slot_of[int(st.block_tables[b, int(t) // 16])], :, int(t) % 16] = True
    last = len(lts) - 1
    for pool in bufs[last % 2]:
        got_rows = ~torch.isnan(pool[:n].float()).any(dim=-1).cpu().numpy()
        assert np.array_equal(got_rows, want_rows)
    plan.close()


def test_staged_decode_equals_the_hbm_step_and_overflow_is_reported():
    """A decode plan: after a step over pools in HBM, its blocks staged from the host copies give the same
    bits through zr_decode_attend_reuse; a capacity below the blocks touched sets bit 4 (value 8) of the
    error word and masks the rest, with no fault."""
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=4, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=(300, 900), seg_len_range=(10, 60), topk=3, window=40, seed=62)
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cuda")
    plan = Z.DecodePlan.from_structure(st).set_deterministic()  # bit-equal outputs across calls
    bt = C.device_tables(st)
    ref = torch.empty(lt.q.shape, dtype=torch.float32, device="cuda")
    plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, ref)
    hk, hv = _pinned(lt.k_pool), _pinned(lt.v_pool)
    for cap, want_err in ((st.num_blocks, 0), (8, 8)):
        stage_ids = torch.zeros((cap,), dtype=torch.int32, device="cuda")
        remap = torch.empty_like(bt)
        n_staged = torch.zeros(1, dtype=torch.int32, device="cuda")
        Z.zr_offload_map(plan.handle, plan.ws, bt, cap, stage_ids, remap, n_staged)
        sk = torch.full((cap, 2, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        sv = torch.full_like(sk, float("nan"))
        Z.zr_offload_stage(plan.handle, plan.ws, hk, hv, stage_ids, n_staged, cap, sk, sv)
        out = torch.empty_like(ref)
        plan.run_reuse(lt.q, sk, sv, remap, lt.sum_k, lt.sum_v, out)
        torch.cuda.synchronize()
        err = plan.device_error()
        assert err & 8 == want_err, err
        if not want_err:
            assert torch.equal(out, ref)
            assert int(n_staged.item()) <= st.num_blocks
    plan.close()
