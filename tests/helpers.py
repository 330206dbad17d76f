"""Shared test glue: turn generated inputs into the oracle's host arrays."""

from __future__ import annotations

import numpy as np

from hierarchical_sparse_kv_gb300 import workloads as W


def oracle_args(st: W.Structure, lt: W.LayerTensors) -> dict:
    """Host arrays (exact stored values) for ``oracle.zoomr_oracle.decode_step``."""
    return dict(
        q=W.to_numpy32(lt.q),
        k_pool=W.to_numpy32(lt.k_pool),
        v_pool=W.to_numpy32(lt.v_pool),
        block_tables=st.block_tables.copy(),
        seg_ptr=st.seg_ptr.copy(),
        seg_bounds=st.seg_bounds.copy(),
        sum_k=W.to_numpy32(lt.sum_k),
        sum_v=W.to_numpy32(lt.sum_v),
        topk=st.topk.copy(),
        window=st.window,
    )


def unit_args(st: W.Structure, lt: W.LayerTensors, b: int, g: int):
    """(q_group, logical K, logical V, bounds, sum K rows, sum V rows) of one unit, as float lists/arrays."""
    G = st.spec.num_q_heads // st.spec.num_kv_heads
    s0, s1 = int(st.seg_ptr[b]), int(st.seg_ptr[b + 1])
    q = W.to_numpy32(lt.q)[b, g * G:(g + 1) * G]
    kl = W.to_numpy32(lt.logical_k[b])[:, g]
    vl = W.to_numpy32(lt.logical_v[b])[:, g]
    sk = W.to_numpy32(lt.sum_k)[s0:s1, g]
    sv = W.to_numpy32(lt.sum_v)[s0:s1, g]
    return q, kl, vl, np.asarray(st.bounds(b)), sk, sv
