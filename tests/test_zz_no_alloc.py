"""The allocation-free entry point, zr_decode_attend_static.

It serves callers that cannot allocate device memory: code handed only its
input and output buffers by a host engine that owns all device allocations, or
a loop that must not call cudaMalloc because it can synchronize the device. The
test checks, through the C ABI, that two calls in a row give the same outputs as
zr_decode_attend with a caller workspace; that an out-of-pool block id is masked
the same way on both paths and that the next clean static call is unaffected
(the error word starts at zero on every call); that a plan too large for the
16 MiB static scratch is refused before anything runs; and, with two GPUs, that
a call with another device current is refused. This file is collected last on
purpose.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import build as B
from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    Z.load()


@pytest.mark.parametrize("cfg", [1, 0])
def test_static_scratch_matches_the_workspace_entry_point_twice(cfg):
    spec = W.WORKLOADS[cfg]
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cuda")
    plan = Z.DecodePlan.from_structure(st).set_deterministic()  # bit-equal outputs across entry points
    assert plan.workspace_bytes <= 16 << 20
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    ref = torch.full(lt.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    Z.zr_decode_attend(plan.handle, plan.ws, lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, ref)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    for _ in range(2):
        out = torch.full(lt.q.shape, float("nan"), dtype=torch.float32, device="cuda")
        Z.zr_decode_attend_static(plan.handle, lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert torch.equal(out, ref)  # same plan, same kernels, same split: the same bits
    plan.close()


def test_plan_over_the_static_limit_is_refused():
    # 32 sequences x 8 KV heads x 4096 two-token segments, all selected: the per-unit range,
    # prefix, selection and summary lists alone take ~21 MB of workspace
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=32, num_q_heads=32, num_kv_heads=8, seq_len=8192,
                        seg_len_range=(2, 2), topk=10_000, window=0)
    st = W.make_structure(spec)
    plan = Z.DecodePlan(batch=st.batch, num_q_heads=32, num_kv_heads=8, head_dim=128, num_blocks=st.num_blocks,
                        max_blocks_per_seq=st.max_blocks_per_seq, window=0, dtype="bf16", seq_lens=st.seq_lens,
                        seg_ptr=st.seg_ptr, seg_bounds=st.seg_bounds, topk=st.topk)
    assert plan.workspace_bytes > 16 << 20
    small = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(64, dtype=torch.int32, device="cuda")
    out = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(Z.ZoomrError) as e:
        Z.zr_decode_attend_static(plan.handle, small, small, small, bt, small, small, out)
    assert e.value.status == Z.ZR_EUNSUPPORTED
    plan.close()


def test_masked_bad_block_then_a_clean_call():
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=2, num_q_heads=8, num_kv_heads=2, seq_len=200,
                        seg_len_range=(10, 30), topk=10_000, window=5, seed=3)
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cuda")
    plan = Z.DecodePlan.from_structure(st).set_deterministic()  # bit-equal outputs across entry points
    good = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    bad_np = st.block_tables.copy()
    bad_np[1, 3] = st.num_blocks + 1000  # outside the pool: masked on both paths
    bad = torch.from_numpy(bad_np.astype(np.int32)).cuda()
    outs = {}
    for name, bt in (("bad", bad), ("good", good)):
        ref = torch.full(lt.q.shape, float("nan"), dtype=torch.float32, device="cuda")
        Z.zr_decode_attend(plan.handle, plan.ws, lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, ref)
        torch.cuda.synchronize()
        assert plan.device_error() == (1 if name == "bad" else 0)
        outs[name] = ref
    for name in ("bad", "good"):  # the masked call, then a clean one on the same static scratch
        out = torch.full(lt.q.shape, float("nan"), dtype=torch.float32, device="cuda")
        Z.zr_decode_attend_static(plan.handle, lt.q, lt.k_pool, lt.v_pool, bad if name == "bad" else good,
                                  lt.sum_k, lt.sum_v, out)
        torch.cuda.synchronize()
        assert torch.equal(out, outs[name]), name
    plan.close()


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs two GPUs")
def test_another_device_current_is_refused():
    st = W.make_structure(W.WORKLOADS[0])
    lt = W.make_layer(st, 0, "cuda:0")
    plan = Z.DecodePlan.from_structure(st, device="cuda:0")
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda(0)
    out = torch.zeros(lt.q.shape, dtype=torch.float32, device="cuda:0")
    with torch.cuda.device(1):
        with pytest.raises(Z.ZoomrError) as e:
            Z.zr_decode_attend_static(plan.handle, lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out)
    assert e.value.status == Z.ZR_EINVAL
    plan.close()
