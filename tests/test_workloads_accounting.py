"""Host-side logic: the seeded input generator, the paged block allocator and
the token/byte accounting, pinned to the numbers the pages print."""

from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import accounting as A
from hierarchical_sparse_kv_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- accounting pins
def test_memory_savings_matches_printed_values():
    for c in _golden("memory_savings.json")["cases"]:
        got = A.memory_savings(c["n_prompt"], c["n_gen"], c["n_window"], c["c"], c["mean_regular_len"],
                               c["mean_summary_len"], c["n_candidates"])
        assert round(got, c["printed_digits"]) == c["printed"], (got, c)
    # the reading behind the second case: with 80 candidates the 32K value is not 7.11
    assert round(A.memory_savings(512, 32768, 512, 2, 250, 20, 80), 2) == 10.79


def test_kv_sizing_formula_matches_printed_values():
    llama, opt = _golden("kv_sizing.json")["cases"]
    got = A.dense_kv_bytes(llama["layers"], llama["tokens"], llama["kv_heads"], llama["head_dim"],
                           llama["bytes_per_elem"], llama["sequences"])
    assert got == llama["formula_bytes"] and got > llama["printed_lower_bound_bytes"]
    per_tok = A.dense_kv_bytes(opt["layers"], 1, opt["kv_heads"], opt["head_dim"], opt["bytes_per_elem"])
    assert per_tok == opt["printed_bytes_per_token_kib"] * 1024
    # 2048 tokens: 1.5625 GiB, which the page rounds to 1.6 GB
    assert round(per_tok * 2048 / 2 ** 30, 1) == opt["printed_2048_tokens_gb"]


def test_block_counting():
    assert A.distinct_blocks([0, 1, 15, 16, 40]) == 3
    assert A.ranges_block_count([(0, 16), (16, 17)]) == 2
    assert A.ranges_block_count([(3, 5), (10, 12)]) == 1
    assert A.ranges_block_count([(3, 5), (20, 40), (47, 49)]) == 4
    rng = np.random.default_rng(0)
    for _ in range(100):
        toks = np.unique(rng.integers(0, 300, size=int(rng.integers(1, 80))))
        brk = np.nonzero(np.diff(toks) != 1)[0]
        starts = np.concatenate([[toks[0]], toks[brk + 1]])
        ends = np.concatenate([toks[brk] + 1, [toks[-1] + 1]])
        assert A.ranges_block_count(list(zip(starts, ends))) == A.distinct_blocks(toks) == len(set(toks // 16))
        assert A.ranges_token_count(list(zip(starts, ends))) == len(toks)


def test_full_step_byte_scale_of_the_headline_workload():
    """About 4.9K gathered tokens per unit at 16K context with k=16 of ~57 segments
    (U[64,512] lengths) and a 256-token window: ~160 MB per layer for 64 units."""
    per_unit = A.attend_bytes_per_unit(4864, 41, 310, 4, 128, 2)
    assert 2.4e6 < per_unit < 2.6e6
    assert 150e6 < 64 * per_unit < 170e6


# ---------------------------------------------------------------- allocator
def test_allocator_refcount_fork_free_and_copy_on_write():
    rng = np.random.default_rng(0)
    al = W.PagedBlockAllocator(10, rng)
    a = al.alloc(3)
    assert len(set(a)) == 3 and all(al.ref_count[b] == 1 for b in a)
    child = al.fork(a)
    assert child == a and all(al.ref_count[b] == 2 for b in a)
    copies = al.append_block(child)
    assert len(copies) == 1 and copies[0][0] == a[-1] and child[-1] != a[-1]
    assert al.ref_count[a[-1]] == 1 and al.ref_count[child[-1]] == 1
    assert al.append_block(child) == []  # now private: no copy
    al.free(a)
    assert al.ref_count[a[-1]] == 0 and all(al.ref_count[b] == 1 for b in a[:-1])
    al.free(child)
    assert all(al.ref_count == 0) and sorted(al.free_list) == list(range(10))
    with pytest.raises(MemoryError):
        al.alloc(11)


# ---------------------------------------------------------------- generator
@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_structure_of_each_workload(cfg):
    spec = W.WORKLOADS[cfg]
    st = W.make_structure(spec)
    B = spec.batch
    assert st.batch == B
    used = []
    for b in range(B):
        L = int(st.seq_lens[b])
        bnd = st.bounds(b)
        assert bnd[0] == 0 and bnd[-1] == L and np.all(np.diff(bnd) > 0)
        lens = np.diff(bnd)
        lo, hi = spec.seg_len_range
        assert np.all(lens[:-1] >= lo) and np.all(lens <= hi)
        nblk = (L + 15) // 16
        tb = st.block_tables[b]
        assert np.all(tb[:nblk] >= 0) and np.all(tb[:nblk] < st.num_blocks) and np.all(tb[nblk:] == -1)
        used.append(tb[:nblk])
    P = spec.shared_prefix_tokens // 16
    if P:
        for b in range(1, B):
            assert np.array_equal(used[b][:P], used[0][:P])
        assert np.all(st.ref_count[used[0][:P]] == B)
        own = np.concatenate([u[P:] for u in used] + [used[0][:P]])
    else:
        own = np.concatenate(used)
    assert len(np.unique(own)) == len(own) == st.num_blocks  # every block used once (prefix once)
    if spec.seq_len_range:
        assert np.all(st.seq_lens >= spec.seq_len_range[0]) and np.all(st.seq_lens <= spec.seq_len_range[1])
    if spec.topk_range:
        assert np.all(st.topk >= spec.topk_range[0]) and np.all(st.topk <= spec.topk_range[1])
    # physical placement is shuffled, not the identity
    assert not np.array_equal(np.sort(used[0]), used[0]) or len(used[0]) < 3
    if cfg == 4:
        assert 150 < st.num_segments(0) < 320


def test_layer_tensors_follow_the_recipe():
    spec = W.small_spec(dtype="f32", seq_len=400, seg_len_range=(40, 60), num_q_heads=4, num_kv_heads=2,
                        head_dim=32, batch=2)
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cpu", keep_logical=True)
    for b in range(2):
        L = int(st.seq_lens[b])
        kl = lt.logical_k[b]
        # the pool holds the logical rows at block_table[t // 16], slot t % 16
        for t in (0, 15, 16, 17, L - 1):
            assert torch.equal(lt.k_pool[st.block_tables[b, t // 16], :, t % 16], kl[t])
            assert torch.equal(lt.v_pool[st.block_tables[b, t // 16], :, t % 16], lt.logical_v[b][t])
        bnd = st.bounds(b)
        s0 = int(st.seg_ptr[b])
        noise = []
        for i in range(len(bnd) - 1):
            mean = kl[bnd[i]:bnd[i + 1]].to(torch.float64).mean(0)
            noise.append((lt.sum_k[s0 + i].to(torch.float64) - mean).flatten())
        noise = torch.cat(noise)
        assert abs(noise.std().item() - 0.1) < 0.01 and abs(noise.mean().item()) < 0.01
    # K ~ N(0, 1)
    allk = torch.cat([x.flatten() for x in lt.logical_k])
    assert abs(allk.std().item() - 1) < 0.05


def test_generation_is_deterministic_and_layers_differ():
    spec = W.small_spec(dtype="bf16", seq_len=200)
    st = W.make_structure(spec)
    a = W.make_layer(st, 0, "cpu")
    b = W.make_layer(st, 0, "cpu")
    c = W.make_layer(st, 1, "cpu")
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.q, b.q)
    assert not torch.equal(a.k_pool, c.k_pool)
    st2 = W.make_structure(spec)
    assert np.array_equal(st.block_tables, st2.block_tables) and np.array_equal(st.seg_bounds, st2.seg_bounds)


def test_poisoned_pool_marks_only_unowned_rows():
    spec = W.small_spec(dtype="f32", seq_len=37)
    st = W.make_structure(spec, spare_blocks=2)
    lt = W.make_layer(st, 0, "cpu", poison_unused=True)
    finite_rows = torch.isfinite(lt.k_pool).all(dim=-1)  # [blocks, Hkv, 16]
    assert int(finite_rows.sum()) == 37 * spec.num_kv_heads
