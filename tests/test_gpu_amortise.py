"""GPU parity of the steps between selections (``zr_decode_advance`` + ``zr_decode_attend_reuse``,
``zr_consensus_advance`` + ``zr_consensus_attend``) against ``oracle/zoomr_amortise.py``: after a selection
step, tokens are appended (``zr_append_kv`` on the device, the append oracle on the host), the windows
move, and every step's outputs match the oracle with the selection held fixed."""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z
from oracle import zoomr_amortise as AM
from oracle import zoomr_append as A
from oracle import zoomr_consensus as OC
from oracle import zoomr_oracle as O
from tests.gpu_common import TOL
from tests.helpers import oracle_args

pytestmark = pytest.mark.gpu


def _np32(t):
    return t.detach().to(torch.float32).cpu().numpy()


def _with_room(st, extra):
    """The structure with block-table columns and mapped spare blocks for ``extra`` more tokens."""
    Lg = st.seq_lens.astype(np.int64) + extra
    cols = int(((Lg + 15) // 16).max())
    tables = np.full((st.batch, cols), -1, np.int32)
    tables[:, :st.max_blocks_per_seq] = st.block_tables
    free = [x for x in range(st.num_blocks) if x not in set(st.block_tables.ravel().tolist())]
    for b in range(st.batch):
        for j in range(int((Lg[b] + 15) // 16)):
            if tables[b, j] < 0:
                tables[b, j] = free.pop(0)
    return dataclasses.replace(st, block_tables=tables)


def _new_rows(B, H, d, dt, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn((B, H, d), generator=g, device="cuda").to(dt),
            torch.randn((B, H, d), generator=g, device="cuda").to(dt))


@pytest.mark.parametrize("dtype,d,window,steps", [("bf16", 128, 16, 40), ("f32", 64, 64, 20), ("bf16", 128, 0, 12)])
def test_decode_steps_between_selections(dtype, d, window, steps):
    spec = W.small_spec(dtype=dtype, head_dim=d, batch=3, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=(100, 300), seg_len_range=(5, 40), topk=3, window=window, seed=41)
    st = _with_room(W.make_structure(spec, spare_blocks=3 * (steps // 16 + 2)), steps)
    lt = W.make_layer(st, 0, "cuda")
    plan = Z.DecodePlan.from_structure(st)
    bt = torch.from_numpy(st.block_tables).cuda()
    G, Hq, Hkv = 4, 8, 2
    out = torch.empty((st.batch, Hq, d), device="cuda")
    dbg = plan.new_debug_outputs()
    plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out, dbg)
    torch.cuda.synchronize()
    sel_gpu = dbg[0].cpu().numpy()
    res0 = O.decode_step(**oracle_args(st, lt))
    kp, vp = _np32(lt.k_pool), _np32(lt.v_pool)
    sk, sv = _np32(lt.sum_k), _np32(lt.sum_v)
    cfg = Z.cache_config(batch=st.batch, num_kv_heads=Hkv, head_dim=d, num_blocks=st.num_blocks,
                         max_blocks_per_seq=st.max_blocks_per_seq, dtype=dtype)
    dt = W.torch_dtype(dtype)
    L0 = st.seq_lens.astype(np.int64)
    for s in range(1, steps + 1):
        kn, vn = _new_rows(st.batch, Hkv, d, dt, 1000 + s)
        pos = (L0 + s - 1).astype(np.int32)
        Z.zr_append_kv(cfg, torch.from_numpy(pos).cuda(), kn, vn, bt, lt.k_pool, lt.v_pool)
        kp, vp = A.append_kv(kp, vp, st.block_tables, pos, _np32(kn), _np32(vn))
        g = torch.Generator(device="cuda")
        g.manual_seed(5000 + s)
        q = torch.randn((st.batch, Hq, d), generator=g, device="cuda").to(dt)
        plan.advance(torch.from_numpy((L0 + s).astype(np.int32)).cuda())
        plan.run_reuse(q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out)
        torch.cuda.synchronize()
        o = out.cpu().numpy()
        qh = _np32(q)
        for b in range(st.batch):
            s0, s1 = int(st.seg_ptr[b]), int(st.seg_ptr[b + 1])
            for gg in range(Hkv):
                k_eff = len(res0.units[b][gg].sel)
                assert list(sel_gpu[b, gg, :k_eff]) == list(res0.units[b][gg].sel)
                r = AM.reuse_unit(qh[b, gg * G:(gg + 1) * G], kp, vp, st.block_tables[b], gg, st.bounds(b),
                                  sk[s0:s1, gg], sv[s0:s1, gg], res0.units[b][gg].sel, int(L0[b] + s), window)
                e = float(np.max(np.abs(o[b, gg * G:(gg + 1) * G] - r.out)))
                assert e <= TOL[dtype], (s, b, gg, e)
    assert plan.device_error() == 0
    plan.close()


def test_advance_rejects_shrinking_or_oversized_lengths():
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=2, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=(100, 200), seg_len_range=(5, 40), topk=2, window=16, seed=42)
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cuda")
    plan = Z.DecodePlan.from_structure(st).set_deterministic()  # bit-equal outputs across calls
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    out0 = torch.empty((2, 8, 128), device="cuda")
    out1 = torch.empty_like(out0)
    plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out0)
    L = st.seq_lens.astype(np.int32)
    for bad in ([L[0] - 1, L[1]], [L[0], 16 * st.max_blocks_per_seq + 1]):
        plan.advance(torch.tensor(bad, dtype=torch.int32, device="cuda"))
        plan.run_reuse(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out1)
        torch.cuda.synchronize()
        assert plan.device_error() == 2
    # the lengths that were valid moved nothing: the reused step equals the selection step
    assert torch.equal(out0, out1)
    plan.close()


def test_consensus_steps_between_selections():
    steps = 30
    spec = W.consensus_spec(dtype="bf16", head_dim=128, layers=2, window=12)
    st = _with_room(W.make_consensus_structure(spec, spare_blocks=spec.batch * (steps // 16 + 2)), steps)
    lts = [W.make_consensus_layer(st, l, "cuda") for l in range(2)]
    sp = st.spec
    bt = torch.from_numpy(st.block_tables).cuda()
    cfg = Z.cache_config(batch=st.batch, num_kv_heads=sp.num_kv_heads, head_dim=128, num_blocks=st.num_blocks,
                         max_blocks_per_seq=st.max_blocks_per_seq, dtype="bf16")
    segs = [(b, s, e, int(st.seg_ptr[b]) + i) for b in range(st.batch) for i, (s, e) in enumerate(st.summary_spans(b))]
    segs_d = torch.tensor(segs, dtype=torch.int32, device="cuda")
    plan = Z.ConsensusPlan.from_structure(st)
    mks = []
    for lt in lts:
        mk = torch.empty((st.total_segments, sp.num_kv_heads, 128), dtype=torch.bfloat16, device="cuda")
        Z.zr_segment_summaries(cfg, segs_d, bt, lt.k_pool, lt.v_pool, mk, torch.empty_like(mk))
        mks.append(mk)
        plan.vote(lt.q, mk)
    plan.select()
    kps = [_np32(lt.k_pool) for lt in lts]
    vps = [_np32(lt.v_pool) for lt in lts]
    kbars = []  # the oracle's own mean keys, checked bit-equal to the device's
    for l in range(2):
        kb = np.empty((st.total_segments, sp.num_kv_heads, 128), np.float32)
        for (b, s, e, r) in segs:
            for gg in range(sp.num_kv_heads):
                kb[r, gg] = A.round_to_dtype(A.segment_mean(kps[l], st.block_tables[b], gg, s, e), "bf16")
        assert np.array_equal(_np32(mks[l]).view(np.uint32), kb.view(np.uint32)), l
        kbars.append(kb)
    res0 = OC.consensus_step([_np32(lt.q) for lt in lts], kbars, kps, vps, st.block_tables, st.seg_ptr,
                             st.seg_bounds, st.prompt_lens, st.seq_lens, st.topk, st.consensus, st.window,
                             attend_layers=[])
    L0 = st.seq_lens.astype(np.int64)
    G = sp.num_q_heads // sp.num_kv_heads
    out = torch.empty((st.batch, sp.num_q_heads, 128), device="cuda")
    for s in range(1, steps + 1):
        pos = (L0 + s - 1).astype(np.int32)
        for l, lt in enumerate(lts):
            kn, vn = _new_rows(st.batch, sp.num_kv_heads, 128, torch.bfloat16, 100 * s + l)
            Z.zr_append_kv(cfg, torch.from_numpy(pos).cuda(), kn, vn, bt, lt.k_pool, lt.v_pool)
            kps[l], vps[l] = A.append_kv(kps[l], vps[l], st.block_tables, pos, _np32(kn), _np32(vn))
        plan.advance(torch.from_numpy((L0 + s).astype(np.int32)).cuda())
        for l, lt in enumerate(lts):
            plan.attend(lt.q, lt.k_pool, lt.v_pool, bt, out)
            torch.cuda.synchronize()
            o = out.cpu().numpy()
            for b in range(st.batch):
                r = res0[b]
                toks = AM.reuse_final_tokens(st.pair_bounds(b), int(st.prompt_lens[b]), int(L0[b] + s), st.window,
                                             r.i_c, r.i_s)
                want = OC.attend_final(_np32(lt.q)[b], kps[l], vps[l], st.block_tables[b], toks, G)
                e = float(np.max(np.abs(o[b] - want)))
                assert e <= TOL["bf16"], (s, l, b, e)
    assert plan.device_error() == 0
    plan.close()
