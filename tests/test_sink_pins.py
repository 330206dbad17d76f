"""Pins of the attention-sink oracle (``oracle/zoomr_sink.py``) from outside it.

- A sink of zero tokens is the decode step itself.
- The attended token set matches a per-token predicate written from the reading.
- With k >= n the step is plain attention over every cached token (torch's fp64 attention on the logical rows).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from oracle import zoomr_oracle as O
from oracle import zoomr_sink as OS
from tests.helpers import oracle_args


def _case(sink, **kw):
    base = dict(dtype="f32", head_dim=64, batch=3, num_q_heads=4, num_kv_heads=2, seq_len=None,
                seq_len_range=(80, 200), seg_len_range=(5, 30), topk=2, window=12, seed=51, sink_tokens=sink)
    base.update(kw)
    st = W.make_structure(W.small_spec(**base))
    return st, W.make_layer(st, 0, "cpu", keep_logical=True)


def test_segments_start_after_the_sink():
    st, _ = _case(24)
    for b in range(st.batch):
        assert int(st.bounds(b)[0]) == 24 and int(st.bounds(b)[-1]) == int(st.seq_lens[b])
    assert st.sink_lens.tolist() == [24] * st.batch


def test_no_sink_is_the_decode_step():
    st, lt = _case(0)
    args = oracle_args(st, lt)
    out, res = OS.decode_step_sink(**args, sink_lens=[0] * st.batch)
    ref = O.decode_step(**args)
    assert np.array_equal(out, ref.out)
    for b in range(st.batch):
        for g in range(2):
            assert np.array_equal(res[b][g].tokens, ref.units[b][g].tokens)


@pytest.mark.parametrize("sink,window,topk", [(16, 12, 2), (33, 0, 1), (8, 1000, 0), (40, 5, 0)])
def test_token_set_matches_a_per_token_predicate(sink, window, topk):
    st, lt = _case(sink, window=window, topk=topk)
    args = oracle_args(st, lt)
    _, res = OS.decode_step_sink(**args, sink_lens=st.sink_lens)
    for b in range(st.batch):
        L = int(st.seq_lens[b])
        bnd = [int(x) for x in st.bounds(b)]
        for g in range(2):
            sel = set(res[b][g].sel.tolist())
            want = [t for t in range(L) if t < sink or t >= L - window
                    or any(bnd[i] <= t < bnd[i + 1] for i in sel)]
            assert res[b][g].tokens.tolist() == want
            assert res[b][g].summaries.tolist() == [i for i in range(len(bnd) - 1) if i not in sel]


def test_k_covering_all_segments_is_dense_attention():
    st, lt = _case(20, topk=1000)
    args = oracle_args(st, lt)
    out, _ = OS.decode_step_sink(**args, sink_lens=st.sink_lens)
    for b in range(st.batch):
        L = int(st.seq_lens[b])
        for h in range(4):
            g = h // 2
            q = torch.from_numpy(W.to_numpy64(lt.q)[b, h]).view(1, 1, 1, -1)
            K = lt.logical_k[b][:, g].double().view(1, 1, L, -1)
            V = lt.logical_v[b][:, g].double().view(1, 1, L, -1)
            ref = torch.nn.functional.scaled_dot_product_attention(q, K, V)[0, 0, 0].numpy()
            np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-12)
