"""GPU parity of the decode step with the prompt kept as an attention sink (``zr_plan_sink``) against
``oracle/zoomr_sink.py``: selections and token ranges bit-exact, outputs within 2e-3 (bf16) / 1e-5 (fp32),
also across the select kernel's two range builders (at most and more than 512 segments) and for the steps
between selections."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z
from oracle import zoomr_append as A
from oracle import zoomr_oracle as O
from oracle import zoomr_sink as OS
from tests import gpu_common as C
from tests.gpu_common import TOL
from tests.helpers import oracle_args

pytestmark = pytest.mark.gpu


def _check(st, lt):
    plan = Z.DecodePlan.from_structure(st)
    bt = C.device_tables(st)
    out, dbg = C.run_gpu(plan, lt, bt)
    err, o, sel, rng, nr = C.fetch(out, dbg, plan)
    assert err == 0
    _, res = OS.decode_step_sink(**oracle_args(st, lt), sink_lens=st.sink_lens)
    G = st.spec.num_q_heads // st.spec.num_kv_heads
    for b in range(st.batch):
        for g in range(st.spec.num_kv_heads):
            u = res[b][g]
            assert list(sel[b, g, :len(u.sel)]) == list(u.sel) and np.all(sel[b, g, len(u.sel):] == -1)
            assert np.array_equal(rng[b, g, :nr[b, g]], O.token_ranges(u.tokens)), (b, g)
            e = float(np.max(np.abs(o[b, g * G:(g + 1) * G] - u.out)))
            assert e <= TOL[st.spec.dtype], (b, g, e)
    plan.close()


@pytest.mark.parametrize("dtype,d,sink,window,topk,seg", [
    ("bf16", 128, 16, 12, 2, (5, 30)),
    ("bf16", 128, 33, 0, 1, (5, 30)),
    ("bf16", 128, 8, 1000, 0, (5, 30)),     # the window reaches the prompt: one range
    ("f32", 64, 40, 5, 0, (5, 30)),         # no selection: sink and window only
    ("f32", 64, 24, 16, 100, (5, 30)),      # every segment selected: one range from 0
    ("bf16", 64, 16, 32, 3, (1, 4)),        # short segments, the first one often selected
])
def test_decode_with_a_sink(dtype, d, sink, window, topk, seg):
    spec = W.small_spec(dtype=dtype, head_dim=d, batch=4, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=(120, 400), seg_len_range=seg, topk=topk, window=window, seed=61,
                        sink_tokens=sink)
    st = W.make_structure(spec)
    _check(st, W.make_layer(st, 0, "cuda"))


def test_decode_with_a_sink_and_more_than_512_segments():
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=2, num_q_heads=8, num_kv_heads=2, seq_len=3000,
                        seg_len_range=(1, 6), topk=40, window=20, seed=62, sink_tokens=48)
    st = W.make_structure(spec)
    assert min(st.num_segments(b) for b in range(st.batch)) > 512
    _check(st, W.make_layer(st, 0, "cuda"))


def test_steps_between_selections_keep_the_sink():
    steps = 20
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=3, num_q_heads=8, num_kv_heads=2, seq_len=None,
                        seq_len_range=(120, 300), seg_len_range=(5, 30), topk=2, window=8, seed=63, sink_tokens=20)
    st0 = W.make_structure(spec, spare_blocks=3 * (steps // 16 + 2))
    Lg = st0.seq_lens.astype(np.int64) + steps
    tables = np.full((st0.batch, int(((Lg + 15) // 16).max())), -1, np.int32)
    tables[:, :st0.max_blocks_per_seq] = st0.block_tables
    free = [x for x in range(st0.num_blocks) if x not in set(st0.block_tables.ravel().tolist())]
    for b in range(st0.batch):
        for j in range(int((Lg[b] + 15) // 16)):
            if tables[b, j] < 0:
                tables[b, j] = free.pop(0)
    import dataclasses
    st = dataclasses.replace(st0, block_tables=tables)
    lt = W.make_layer(st, 0, "cuda")
    plan = Z.DecodePlan.from_structure(st)
    bt = torch.from_numpy(tables).cuda()
    out = torch.empty((st.batch, 8, 128), device="cuda")
    plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out)
    _, res0 = OS.decode_step_sink(**oracle_args(st, lt), sink_lens=st.sink_lens)
    kp, vp = W.to_numpy32(lt.k_pool), W.to_numpy32(lt.v_pool)
    sk, sv = W.to_numpy32(lt.sum_k), W.to_numpy32(lt.sum_v)
    cfg = Z.cache_config(batch=st.batch, num_kv_heads=2, head_dim=128, num_blocks=st.num_blocks,
                         max_blocks_per_seq=st.max_blocks_per_seq, dtype="bf16")
    L0 = st.seq_lens.astype(np.int64)
    for s in range(1, steps + 1):
        g = torch.Generator(device="cuda")
        g.manual_seed(700 + s)
        kn = torch.randn((st.batch, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
        vn = torch.randn((st.batch, 2, 128), generator=g, device="cuda").to(torch.bfloat16)
        pos = (L0 + s - 1).astype(np.int32)
        Z.zr_append_kv(cfg, torch.from_numpy(pos).cuda(), kn, vn, bt, lt.k_pool, lt.v_pool)
        kp, vp = A.append_kv(kp, vp, tables, pos, W.to_numpy32(kn), W.to_numpy32(vn))
        plan.advance(torch.from_numpy((L0 + s).astype(np.int32)).cuda())
        plan.run_reuse(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out)
        torch.cuda.synchronize()
        o = out.cpu().numpy()
        q = W.to_numpy32(lt.q)
        for b in range(st.batch):
            s0, s1 = int(st.seg_ptr[b]), int(st.seg_ptr[b + 1])
            for gg in range(2):
                u = res0[b][gg]
                toks, sums = OS.gather_set_sink(st.bounds(b), u.sel, int(L0[b] + s), st.window, 20)
                K = np.concatenate([O.paged_rows(kp, tables[b], gg, toks), sk[s0:s1, gg][sums]])
                V = np.concatenate([O.paged_rows(vp, tables[b], gg, toks), sv[s0:s1, gg][sums]])
                for hh in range(4):
                    want, _ = O.attend(q[b, gg * 4 + hh], K, V)
                    assert np.max(np.abs(o[b, gg * 4 + hh] - want)) <= TOL["bf16"], (s, b, gg, hh)
    assert plan.device_error() == 0
    plan.close()
