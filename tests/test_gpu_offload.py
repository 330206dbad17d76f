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
    plan = Z.DecodePlan.from_structure(st)
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
        plan = Z.ConsensusPlan.from_structure(st)
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
