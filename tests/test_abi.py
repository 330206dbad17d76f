"""The C-ABI library loads, exports every symbol ``include/zoomr.h`` declares,
and rejects bad problem statements on the host (no GPU needed: validation
happens before any CUDA call)."""

from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

from hierarchical_sparse_kv_gb300 import build as B
from hierarchical_sparse_kv_gb300 import zoomr as Z

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "zoomr.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return Z.load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"^ZR_API\s+[\w\s\*]+?\b(zr_\w+)\s*\(", text, flags=re.M)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert set(names) >= {"zr_plan", "zr_decode_attend", "zr_free", "zr_get_device_error", "zr_status_string"}
    for n in names:
        assert hasattr(lib, n), n
    # nothing else leaks out of the library
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read().split("\n")
    exported = sorted(l.split()[-1] for l in out if " T " in l)
    assert exported == sorted(names)


def test_status_strings(lib):
    for s in range(6):
        assert Z.zr_status_string(s).startswith("ZR_")
    assert "unknown" in Z.zr_status_string(42)


def _good():
    # 2 sequences: L = 40 (segments 0,10,25,40) and L = 17 (segments 0,17)
    cfg = Z.zr_config(2, 8, 2, 64, 16, 8, 3, 4, Z.ZR_F32)
    return cfg, [40, 17], [0, 3, 4], [0, 10, 25, 40, 0, 17], [2, 5]


@pytest.mark.parametrize("mutate,want", [
    (lambda c, L, P, Bd, K: setattr(c, "batch", 0), Z.ZR_EINVAL),
    (lambda c, L, P, Bd, K: setattr(c, "num_q_heads", 7), Z.ZR_EINVAL),       # not a multiple of Hkv
    (lambda c, L, P, Bd, K: setattr(c, "block_size", 32), Z.ZR_EINVAL),
    (lambda c, L, P, Bd, K: setattr(c, "window", -1), Z.ZR_EINVAL),
    (lambda c, L, P, Bd, K: setattr(c, "dtype", 7), Z.ZR_EINVAL),
    (lambda c, L, P, Bd, K: setattr(c, "head_dim", 96), Z.ZR_EUNSUPPORTED),
    (lambda c, L, P, Bd, K: setattr(c, "num_q_heads", 34), Z.ZR_EUNSUPPORTED),  # group of 17
    (lambda c, L, P, Bd, K: L.__setitem__(1, 0), Z.ZR_EINVAL),                 # empty sequence
    (lambda c, L, P, Bd, K: L.__setitem__(0, 49), Z.ZR_EINVAL),                # longer than its table
    (lambda c, L, P, Bd, K: K.__setitem__(0, -1), Z.ZR_EINVAL),
    (lambda c, L, P, Bd, K: Bd.__setitem__(1, 25), Z.ZR_EINVAL),               # bounds not ascending
    (lambda c, L, P, Bd, K: Bd.__setitem__(0, 1), Z.ZR_EINVAL),                # first bound not 0
    (lambda c, L, P, Bd, K: Bd.__setitem__(3, 39), Z.ZR_EINVAL),               # last bound not L
    (lambda c, L, P, Bd, K: P.__setitem__(0, 1), Z.ZR_EINVAL),
    (lambda c, L, P, Bd, K: setattr(c, "num_blocks", 0), Z.ZR_EINVAL),
])
def test_plan_rejects_bad_metadata_on_the_host(lib, mutate, want):
    cfg, L, P, Bd, K = _good()
    mutate(cfg, L, P, Bd, K)
    assert Z.zr_plan_status(cfg, L, P, Bd, K) == want


def test_plan_rejects_null_arguments(lib):
    cfg, L, P, Bd, K = _good()
    assert Z.zr_plan_status(None, L, P, Bd, K) == Z.ZR_EINVAL
    st = lib.zr_plan(ctypes.byref(cfg), None, None, None, None, None, None)
    assert st == Z.ZR_EINVAL
    assert lib.zr_decode_attend(*([None] * 13)) == Z.ZR_EINVAL
    lib.zr_free(None)  # no-op


def test_deterministic_setter_checks_its_arguments(lib):
    assert lib.zr_plan_set_deterministic(None, 1) == Z.ZR_EINVAL
    assert lib.zr_plan_set_deterministic(None, 0) == Z.ZR_EINVAL


def test_too_many_segments_is_unsupported(lib):
    n = 4097
    cfg = Z.zr_config(1, 4, 1, 64, 16, 300, 300, 0, Z.ZR_BF16)
    assert Z.zr_plan_status(cfg, [n], [0, n], list(range(n + 1)), [1]) == Z.ZR_EUNSUPPORTED


# ---------------------------------------------------------------- append path
# Fake, 16-byte aligned "device" addresses: every case below is rejected (or is a
# no-op) before any CUDA call, so nothing is dereferenced.
_A = 1 << 20


def _cache_cfg(**kw):
    base = dict(batch=2, num_kv_heads=2, head_dim=64, num_blocks=8, max_blocks_per_seq=3, dtype="bf16")
    base.update(kw)
    return Z.cache_config(**base)


@pytest.mark.parametrize("field,value,want", [
    ("batch", 0, Z.ZR_EINVAL), ("num_kv_heads", 0, Z.ZR_EINVAL), ("block_size", 8, Z.ZR_EINVAL),
    ("num_blocks", 0, Z.ZR_EINVAL), ("max_blocks_per_seq", 0, Z.ZR_EINVAL), ("dtype", 3, Z.ZR_EINVAL),
    ("head_dim", 0, Z.ZR_EINVAL), ("head_dim", 96, Z.ZR_EUNSUPPORTED), ("num_blocks", 1 << 27, Z.ZR_EUNSUPPORTED),
])
def test_append_calls_reject_bad_configs(lib, field, value, want):
    cfg = _cache_cfg()
    setattr(cfg, field, value)
    c = ctypes.byref(cfg)
    assert lib.zr_append_kv(c, _A, _A, _A, _A, _A, _A, None, None) == want
    assert lib.zr_copy_blocks(c, _A, 1, _A, _A, None, None) == want
    assert lib.zr_segment_summaries(c, _A, 1, _A, _A, _A, _A, _A, 4, None, None) == want


def test_append_calls_reject_null_misaligned_and_negative_arguments(lib):
    c = ctypes.byref(_cache_cfg())
    assert lib.zr_append_kv(None, _A, _A, _A, _A, _A, _A, None, None) == Z.ZR_EINVAL
    for i in range(6):
        args = [_A] * 6
        args[i] = None
        assert lib.zr_append_kv(c, *args, None, None) == Z.ZR_EINVAL, i
    for i in (1, 2, 4, 5):  # k_new, v_new, k_pool, v_pool must be 16-byte aligned
        args = [_A] * 6
        args[i] = _A + 8
        assert lib.zr_append_kv(c, *args, None, None) == Z.ZR_EINVAL, i
    assert lib.zr_copy_blocks(c, _A, -1, _A, _A, None, None) == Z.ZR_EINVAL
    assert lib.zr_copy_blocks(c, None, 2, _A, _A, None, None) == Z.ZR_EINVAL
    assert lib.zr_copy_blocks(c, _A, 2, _A + 4, _A, None, None) == Z.ZR_EINVAL
    assert lib.zr_segment_summaries(c, _A, -1, _A, _A, _A, _A, _A, 4, None, None) == Z.ZR_EINVAL
    assert lib.zr_segment_summaries(c, _A, 1, _A, _A, _A, _A, _A, -1, None, None) == Z.ZR_EINVAL
    assert lib.zr_segment_summaries(c, None, 1, _A, _A, _A, _A, _A, 4, None, None) == Z.ZR_EINVAL
    for i in range(5):  # block_tables, k_pool, v_pool, sum_k, sum_v
        args = [_A] * 5
        args[i] = None
        assert lib.zr_segment_summaries(c, _A, 1, *args, 4, None, None) == Z.ZR_EINVAL, i
    assert lib.zr_segment_summaries(c, _A + 4, 1, _A, _A, _A, _A, _A, 4, None, None) == Z.ZR_EINVAL
    assert lib.zr_segment_summaries(c, _A, 1, _A, _A, _A, _A + 2, _A, 4, None, None) == Z.ZR_EINVAL


def test_empty_copy_and_summary_batches_launch_nothing(lib):
    c = ctypes.byref(_cache_cfg())
    assert lib.zr_copy_blocks(c, None, 0, _A, _A, None, None) == Z.ZR_OK
    assert lib.zr_segment_summaries(c, None, 0, _A, _A, _A, _A, _A, 0, None, None) == Z.ZR_OK


# ---------------------------------------------------------------- consensus plan
def _good_consensus():
    # 2 sequences, L = 60 and 40; prompt 4 and 0; pairs (R, S): [4,14),[14,18),[18,30),[30,33) and [0,9),[9,12)
    cfg = Z.zr_config(2, 8, 2, 64, 16, 8, 4, 8, Z.ZR_BF16)
    return cfg, [60, 40], [4, 0], [0, 2, 3], [4, 14, 18, 30, 33, 0, 9, 12], [2, 1], [1, 1]


@pytest.mark.parametrize("mutate,want", [
    (lambda c, L, P, S, Bd, K, C: setattr(c, "batch", 0), Z.ZR_EINVAL),
    (lambda c, L, P, S, Bd, K, C: setattr(c, "head_dim", 96), Z.ZR_EUNSUPPORTED),
    (lambda c, L, P, S, Bd, K, C: setattr(c, "num_q_heads", 34), Z.ZR_EUNSUPPORTED),
    (lambda c, L, P, S, Bd, K, C: L.__setitem__(1, 0), Z.ZR_EINVAL),            # empty sequence
    (lambda c, L, P, S, Bd, K, C: L.__setitem__(0, 65), Z.ZR_EINVAL),           # longer than its table
    (lambda c, L, P, S, Bd, K, C: P.__setitem__(0, 61), Z.ZR_EINVAL),           # prompt longer than L
    (lambda c, L, P, S, Bd, K, C: P.__setitem__(0, 3), Z.ZR_EINVAL),            # bd[0] != prompt length
    (lambda c, L, P, S, Bd, K, C: Bd.__setitem__(2, 14), Z.ZR_EINVAL),          # empty summary segment
    (lambda c, L, P, S, Bd, K, C: Bd.__setitem__(7, 41), Z.ZR_EINVAL),          # pairs past L
    (lambda c, L, P, S, Bd, K, C: S.__setitem__(1, 0), Z.ZR_EINVAL),            # a sequence with no pair
    (lambda c, L, P, S, Bd, K, C: K.__setitem__(0, -1), Z.ZR_EINVAL),
    (lambda c, L, P, S, Bd, K, C: C.__setitem__(1, -1), Z.ZR_EINVAL),
    (lambda c, L, P, S, Bd, K, C: (setattr(c, "window", 0), K.__setitem__(1, 0)), Z.ZR_EINVAL),  # nothing to attend
])
def test_consensus_plan_rejects_bad_metadata_on_the_host(lib, mutate, want):
    cfg, L, P, S, Bd, K, C = _good_consensus()
    mutate(cfg, L, P, S, Bd, K, C)
    assert Z.zr_consensus_plan_status(cfg, L, P, S, Bd, K, C) == want


def test_consensus_entry_points_reject_null_arguments(lib):
    cfg, L, P, S, Bd, K, C = _good_consensus()
    assert Z.zr_consensus_plan_status(None, L, P, S, Bd, K, C) == Z.ZR_EINVAL
    assert lib.zr_consensus_plan(ctypes.byref(cfg), None, None, None, None, None, None, None, None) == Z.ZR_EINVAL
    assert lib.zr_consensus_vote(None, None, None, None, None) == Z.ZR_EINVAL
    assert lib.zr_consensus_select(None, None, None, None, None, None, None) == Z.ZR_EINVAL
    assert lib.zr_consensus_attend(*([None] * 8)) == Z.ZR_EINVAL
    assert lib.zr_consensus_dims(None, None, None) == Z.ZR_EINVAL


def test_steps_between_selections_reject_null_arguments(lib):
    assert lib.zr_decode_advance(None, None, None, None) == Z.ZR_EINVAL
    assert lib.zr_decode_attend_reuse(*([None] * 10)) == Z.ZR_EINVAL
    assert lib.zr_consensus_advance(None, None, None, None) == Z.ZR_EINVAL


def test_sink_plan_checks_the_first_bound_on_the_host(lib):
    cfg, L, P, Bd, K = _good()

    def status(sink, bounds):
        a = [Z._i32(x) for x in (L, sink, P, bounds, K)]
        plan, ws = Z._P(), ctypes.c_size_t()
        return lib.zr_plan_sink(ctypes.byref(cfg), *[Z._ptr32(x) for x in a], ctypes.byref(plan), ctypes.byref(ws))

    assert status([3, 0], Bd) == Z.ZR_EINVAL                       # first bound 0, sink 3
    assert status([-1, 0], Bd) == Z.ZR_EINVAL
    assert status([10, 17], [10, 25, 40, 17, 17]) == Z.ZR_EINVAL   # a sequence with its whole length as sink: empty segment
    assert lib.zr_plan_sink(ctypes.byref(cfg), None, None, None, None, None, None, None) == Z.ZR_EINVAL
