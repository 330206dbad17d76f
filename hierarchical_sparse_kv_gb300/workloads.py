"""Seeded synthetic inputs for one ZoomR decode step over a paged KV cache.

This module draws inputs only. It holds none of the step's own arithmetic: no
summary scoring, no top-k, no gather-set construction and no attention. Both the
CPU oracle's tests and the CUDA path's tests and benchmark take their inputs from
here, so it is the one piece the two sides share.

What is drawn, per workload (the shapes follow the ZoomR page, "1 Introduction"
and "4 Experiments": Llama-3.1-8B attention, 16K generated tokens, batch 8; the
paged layout follows the "KV-cache management" page, "Paged KV cache
(PagedAttention)" and "Block sharing with reference counts and copy-on-write"):

* segment structure: each sequence's cached tokens are cut into consecutive
  "thought" segments whose lengths are uniform integers in a range (the last one
  truncated to fit), which matches the regular segments R_i of ZoomR "3.3 The
  ZoomR Algorithm";
* a physical block pool of 16-token blocks handed out in a shuffled order by a
  host-side reference-counted allocator (``PagedBlockAllocator``), and one block
  table per sequence;
* K and V ~ N(0, 1), rounded to the storage dtype;
* one summary key and one summary value per segment: the fp64 mean of the
  segment's stored K (or V) rows plus N(0, 0.1) noise, rounded to the storage
  dtype (the ZoomR page's "mean summary key", "Representing Context with Mean
  Summary Keys"; the noise stands in for the summary tokens being different
  tokens from the segment);
* queries: 3 x the mean key of one random segment of the sequence, plus N(0, 1)
  (the long single-stream workload instead sums the mean keys of three segments
  taken from different thirds of the sequence, which makes scores peaky).

Randomness: the structure comes from ``numpy.random.default_rng(seed)``; the
per-layer tensors come from a ``torch.Generator`` on the target device seeded
with ``seed * 1000 + layer`` (and the per-layer discrete choices from
``numpy.random.default_rng(seed * 1000 + layer)``). Values drawn on the CPU and
on a GPU differ; each run is deterministic on its own device.
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

BLOCK_SIZE = 16


# --------------------------------------------------------------------------
# host-side paged block allocator
# --------------------------------------------------------------------------
class PagedBlockAllocator:
    """Reference-counted allocator of fixed-size physical KV blocks.

    Follows the "KV-cache management" page, "Paged KV cache (PagedAttention)"
    (one preallocated region carved into blocks; a per-sequence block table
    maps logical to physical blocks; allocation on demand) and "Block sharing
    with reference counts and copy-on-write" (shared blocks carry a count;
    fork raises it, free lowers it and recycles at zero). The free list is
    shuffled so that physical placement is random, as in the workloads.
    """

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.num_blocks = int(num_blocks)
        self.free_list: List[int] = [int(x) for x in rng.permutation(self.num_blocks)]
        self.ref_count = np.zeros(self.num_blocks, dtype=np.int64)

    def alloc(self, n: int) -> List[int]:
        if n > len(self.free_list):
            raise MemoryError(f"pool exhausted: want {n}, have {len(self.free_list)}")
        out = self.free_list[:n]
        del self.free_list[:n]
        for b in out:
            assert self.ref_count[b] == 0
            self.ref_count[b] = 1
        return out

    def fork(self, table: Sequence[int]) -> List[int]:
        """A child that shares every block of ``table`` (refcount + 1 each)."""
        for b in table:
            assert self.ref_count[b] > 0
            self.ref_count[b] += 1
        return list(table)

    def free(self, table: Sequence[int]) -> None:
        for b in table:
            assert self.ref_count[b] > 0
            self.ref_count[b] -= 1
            if self.ref_count[b] == 0:
                self.free_list.append(int(b))

    def append_block(self, table: List[int]) -> List[int]:
        """Copy-on-write rule before writing into the last block of ``table``:
        a shared last block is replaced by a private one. Returns the list of
        (src, dst) copies the caller must perform (empty if none)."""
        last = table[-1]
        if self.ref_count[last] > 1:
            new = self.alloc(1)[0]
            self.ref_count[last] -= 1
            table[-1] = new
            return [(last, new)]
        return []


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    dtype: str  # "f32" or "bf16"
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    seq_len: Optional[int]  # fixed length, or None for seq_len_range
    seq_len_range: Optional[tuple]
    seg_len_range: tuple  # inclusive uniform range of segment lengths
    topk: Optional[int]  # fixed k, or None for topk_range
    topk_range: Optional[tuple]
    window: int
    layers: int = 1
    shared_prefix_tokens: int = 0
    peaky_query: bool = False
    seed: int = 0
    sink_tokens: int = 0  # prompt tokens kept as an attention sink; the segments partition [sink, L)


WORKLOADS: Dict[int, WorkloadSpec] = {
    0: WorkloadSpec("tiny_f32_b1_h8x2_d64_L512", "f32", 1, 8, 2, 64, 512, None, (32, 32), 4, None, 64, seed=0),
    1: WorkloadSpec("llama8b_bf16_b8_L4096", "bf16", 8, 32, 8, 128, 4096, None, (32, 256), 8, None, 128, seed=1),
    2: WorkloadSpec("llama8b_bf16_b8_L16384_32layers", "bf16", 8, 32, 8, 128, 16384, None, (64, 512), 16, None, 256,
                    layers=32, seed=2),
    3: WorkloadSpec("ragged_bf16_b32_L2048-32768_prefix1024", "bf16", 32, 32, 8, 128, None, (2048, 32768), (32, 512),
                    None, (4, 32), 128, shared_prefix_tokens=1024, seed=3),
    4: WorkloadSpec("long_bf16_b1_L131072", "bf16", 1, 32, 8, 128, 131072, None, (128, 1024), 32, None, 512,
                    peaky_query=True, seed=4),
}


@dataclass
class Structure:
    """Everything about a workload that is not a per-layer tensor."""

    spec: WorkloadSpec
    seq_lens: np.ndarray  # int32 [B]
    seg_ptr: np.ndarray  # int32 [B+1]; CSR over segments (n_b = seg_ptr[b+1]-seg_ptr[b])
    seg_bounds: np.ndarray  # int32 [total_segments + B]; sequence b's n_b+1 bounds start at seg_ptr[b]+b
    topk: np.ndarray  # int32 [B] (not clipped)
    window: int
    num_blocks: int
    block_tables: np.ndarray  # int32 [B, max_blocks_per_seq], unused entries -1
    ref_count: np.ndarray  # int64 [num_blocks] after construction
    sink_lens: Optional[np.ndarray] = None  # int32 [B] attention-sink tokens, or None (no sink)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_segments(self) -> int:
        return int(self.seg_ptr[-1])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def bounds(self, b: int) -> np.ndarray:
        n = int(self.seg_ptr[b + 1] - self.seg_ptr[b])
        s = int(self.seg_ptr[b]) + b
        return self.seg_bounds[s:s + n + 1]

    def num_segments(self, b: int) -> int:
        return int(self.seg_ptr[b + 1] - self.seg_ptr[b])


def _draw_segments(rng: np.random.Generator, L: int, lo: int, hi: int) -> np.ndarray:
    """Consecutive segment bounds covering [0, L): lengths ~ U{lo..hi}, last truncated."""
    n_draw = L // lo + 2
    lens = rng.integers(lo, hi + 1, size=n_draw)
    ends = np.cumsum(lens)
    n = int(np.searchsorted(ends, L, side="left")) + 1
    ends = ends[:n].copy()
    ends[-1] = L
    return np.concatenate([[0], ends]).astype(np.int32)


def make_structure(spec: WorkloadSpec, *, seq_lens: Optional[Sequence[int]] = None,
                   spare_blocks: int = 0) -> Structure:
    """Segments, top-k, block pool and block tables for ``spec`` (seeded by spec.seed)."""
    rng = np.random.default_rng(spec.seed)
    B = spec.batch
    if seq_lens is not None:
        lens = np.asarray(seq_lens, dtype=np.int64)
    elif spec.seq_len is not None:
        lens = np.full(B, spec.seq_len, dtype=np.int64)
    else:
        lo, hi = spec.seq_len_range
        lens = rng.integers(lo, hi + 1, size=B)
    lens = np.maximum(lens, spec.shared_prefix_tokens + 1) if spec.shared_prefix_tokens else lens

    bounds_list = []
    sink = int(spec.sink_tokens)
    for b in range(B):
        lo, hi = spec.seg_len_range
        bounds_list.append(_draw_segments(rng, int(lens[b]) - sink, lo, hi) + sink)
    n_seg = np.array([len(x) - 1 for x in bounds_list], dtype=np.int64)
    seg_ptr = np.concatenate([[0], np.cumsum(n_seg)]).astype(np.int32)
    seg_bounds = np.concatenate(bounds_list).astype(np.int32)

    if spec.topk is not None:
        topk = np.full(B, spec.topk, dtype=np.int32)
    else:
        lo, hi = spec.topk_range
        topk = rng.integers(lo, hi + 1, size=B).astype(np.int32)

    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    max_blocks = int(nblk.max())
    P = spec.shared_prefix_tokens // BLOCK_SIZE
    assert spec.shared_prefix_tokens % BLOCK_SIZE == 0
    num_blocks = int(nblk.sum() - (B - 1) * P) + spare_blocks if P else int(nblk.sum()) + spare_blocks
    alloc = PagedBlockAllocator(num_blocks, rng)
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    prefix = alloc.alloc(P) if P else []
    for b in range(B):
        own = alloc.fork(prefix) if P and b > 0 else list(prefix)
        own = own + alloc.alloc(int(nblk[b]) - P)
        tables[b, :len(own)] = own
    return Structure(spec, lens.astype(np.int32), seg_ptr, seg_bounds, topk, spec.window, num_blocks, tables,
                     alloc.ref_count.copy(), np.full(B, sink, np.int32) if sink else None)


# --------------------------------------------------------------------------
# per-layer tensors
# --------------------------------------------------------------------------
def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


@dataclass
class LayerTensors:
    q: torch.Tensor  # [B, Hq, d] dtype
    k_pool: torch.Tensor  # [num_blocks, Hkv, 16, d] dtype
    v_pool: torch.Tensor  # [num_blocks, Hkv, 16, d] dtype
    sum_k: torch.Tensor  # [total_segments, Hkv, d] dtype
    sum_v: torch.Tensor  # [total_segments, Hkv, d] dtype
    logical_k: Optional[List[torch.Tensor]] = field(default=None)  # per seq [L_b, Hkv, d] dtype
    logical_v: Optional[List[torch.Tensor]] = field(default=None)


def _segment_means(x: torch.Tensor, bounds: np.ndarray) -> torch.Tensor:
    """fp64 mean over each segment [bounds[i], bounds[i+1]) of rows of x [L, H, d]."""
    lens = np.diff(bounds)
    seg_id = torch.from_numpy(np.repeat(np.arange(len(lens)), lens)).to(x.device)
    acc = torch.zeros((len(lens),) + tuple(x.shape[1:]), dtype=torch.float64, device=x.device)
    acc.index_add_(0, seg_id, x[int(bounds[0]):int(bounds[-1])].to(torch.float64))
    return acc / torch.from_numpy(lens.astype(np.float64)).to(x.device).view(-1, 1, 1)


def make_layer(st: Structure, layer: int, device: str | torch.device = "cpu", *,
               keep_logical: bool = False, poison_unused: bool = False) -> LayerTensors:
    """Draw one layer's q, paged K/V pool and summary K/V for structure ``st``.

    ``poison_unused`` fills pool rows that no sequence owns (the tail of each
    sequence's last block and any spare block) with NaN, so a kernel that reads
    past the cached tokens shows up as a non-finite output.
    """
    spec = st.spec
    dev = torch.device(device)
    dt = torch_dtype(spec.dtype)
    seed = spec.seed * 1000 + layer
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    nrng = np.random.default_rng(seed)
    B, Hq, Hkv, d = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    G = Hq // Hkv

    fill = float("nan") if poison_unused else 0.0
    k_pool = torch.full((st.num_blocks, Hkv, BLOCK_SIZE, d), fill, dtype=dt, device=dev)
    v_pool = torch.full((st.num_blocks, Hkv, BLOCK_SIZE, d), fill, dtype=dt, device=dev)
    sum_k = torch.empty((st.total_segments, Hkv, d), dtype=dt, device=dev)
    sum_v = torch.empty((st.total_segments, Hkv, d), dtype=dt, device=dev)
    q = torch.empty((B, Hq, d), dtype=dt, device=dev)

    P = spec.shared_prefix_tokens
    if P:
        pk = torch.randn((P, Hkv, d), generator=gen, device=dev).to(dt)
        pv = torch.randn((P, Hkv, d), generator=gen, device=dev).to(dt)
    lk_all, lv_all = [], []
    for b in range(B):
        L = int(st.seq_lens[b])
        own = L - P
        kk = torch.randn((own, Hkv, d), generator=gen, device=dev).to(dt)
        vv = torch.randn((own, Hkv, d), generator=gen, device=dev).to(dt)
        if P:
            kk = torch.cat([pk, kk], 0)
            vv = torch.cat([pv, vv], 0)
        nblk = (L + BLOCK_SIZE - 1) // BLOCK_SIZE
        idx = torch.from_numpy(st.block_tables[b, :nblk].astype(np.int64)).to(dev)
        for src, pool in ((kk, k_pool), (vv, v_pool)):
            pad = torch.full((nblk * BLOCK_SIZE, Hkv, d), fill, dtype=dt, device=dev)
            pad[:L] = src
            pool[idx] = pad.view(nblk, BLOCK_SIZE, Hkv, d).permute(0, 2, 1, 3)
        bnd = st.bounds(b)
        n = len(bnd) - 1
        mk = _segment_means(kk, bnd)
        mv = _segment_means(vv, bnd)
        nk = torch.randn((n, Hkv, d), generator=gen, device=dev).to(torch.float64) * 0.1
        nv = torch.randn((n, Hkv, d), generator=gen, device=dev).to(torch.float64) * 0.1
        s0 = int(st.seg_ptr[b])
        sum_k[s0:s0 + n] = (mk + nk).to(torch.float32).to(dt)
        sum_v[s0:s0 + n] = (mv + nv).to(torch.float32).to(dt)
        # queries
        if spec.peaky_query:
            thirds = [(0, n // 3), (n // 3, 2 * n // 3), (2 * n // 3, n)]
            picks = [int(nrng.integers(lo, max(hi, lo + 1))) for lo, hi in thirds]
            base = mk[picks].sum(0)  # [Hkv, d]
            base = base.repeat_interleave(G, dim=0)  # [Hq, d]
        else:
            picks = nrng.integers(0, n, size=Hq)
            heads = np.arange(Hq) // G
            base = mk[torch.from_numpy(picks).to(dev), torch.from_numpy(heads).to(dev)]  # [Hq, d]
        noise = torch.randn((Hq, d), generator=gen, device=dev).to(torch.float64)
        q[b] = (3.0 * base + noise).to(torch.float32).to(dt)
        if keep_logical:
            lk_all.append(kk)
            lv_all.append(vv)
    return LayerTensors(q, k_pool, v_pool, sum_k, sum_v, lk_all if keep_logical else None,
                        lv_all if keep_logical else None)


def to_numpy64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a stored tensor to a host float64 array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def to_numpy32(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a stored (f32 or bf16) tensor to a host float32 array."""
    return t.detach().to("cpu").to(torch.float32).numpy()


def small_spec(**kw) -> WorkloadSpec:
    """A custom workload for tests (defaults: tiny fp32 shape)."""
    base = dict(name="custom", dtype="f32", batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, seq_len=96,
                seq_len_range=None, seg_len_range=(8, 24), topk=2, topk_range=None, window=16, layers=1,
                shared_prefix_tokens=0, peaky_query=False, seed=0)
    base.update(kw)
    return WorkloadSpec(**base)


# --------------------------------------------------------------------------
# the consensus layout: prompt, then (regular segment, summary segment) pairs
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class ConsensusSpec:
    """A workload of ZoomR's consensus path (3.3 "Global Aggregation and Consensus").

    Every sequence holds ``prompt_len`` prompt tokens and ``gen_len`` generated
    ones. The generated tokens are pairs of a regular segment R_i (length
    U{reg_len_range}) followed by its summary segment S_i (U{sum_len_range}),
    then a tail shorter than the next pair (a paragraph with no summary yet).
    """

    name: str
    dtype: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    prompt_len: int
    gen_len: int
    reg_len_range: tuple
    sum_len_range: tuple
    topk: int
    consensus: int
    window: int
    layers: int = 1
    seed: int = 0


CONSENSUS_WORKLOADS: Dict[int, ConsensusSpec] = {
    # tiny fp32 case the oracle finishes in seconds
    0: ConsensusSpec("consensus_tiny_f32_b2_h8x2_d64_P32_G480", "f32", 2, 8, 2, 64, 32, 480, (16, 48), (4, 8),
                     2, 2, 32, layers=2, seed=10),
    # the ZoomR page's analysis shape (3.5: N_p = 512, N_w = 512, c = 2, mean R 250, mean S 20) at the
    # 8B model's attention shape, 16K generated tokens, batch 8, 32 layers
    1: ConsensusSpec("consensus_llama8b_bf16_b8_P512_G16384_32layers", "bf16", 8, 32, 8, 128, 512, 16384,
                     (200, 300), (10, 30), 4, 2, 512, layers=32, seed=12),
}


@dataclass
class ConsensusStructure:
    spec: ConsensusSpec
    seq_lens: np.ndarray      # int32 [B]
    prompt_lens: np.ndarray   # int32 [B]
    seg_ptr: np.ndarray       # int32 [B+1]; n_b = seg_ptr[b+1] - seg_ptr[b] pairs
    seg_bounds: np.ndarray    # int32; sequence b's 2 n_b + 1 pair bounds start at 2 seg_ptr[b] + b
    topk: np.ndarray          # int32 [B]
    consensus: np.ndarray     # int32 [B]
    window: int
    num_blocks: int
    block_tables: np.ndarray  # int32 [B, max_blocks], unused entries -1

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_segments(self) -> int:
        return int(self.seg_ptr[-1])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def num_segments(self, b: int) -> int:
        return int(self.seg_ptr[b + 1] - self.seg_ptr[b])

    def pair_bounds(self, b: int) -> np.ndarray:
        s = 2 * int(self.seg_ptr[b]) + b
        return self.seg_bounds[s:s + 2 * self.num_segments(b) + 1]

    def summary_spans(self, b: int):
        """(start, end) of every summary segment S_i of sequence b."""
        bd = self.pair_bounds(b)
        return [(int(bd[2 * i + 1]), int(bd[2 * i + 2])) for i in range(self.num_segments(b))]


def make_consensus_structure(spec: ConsensusSpec, *, seq_lens: Optional[Sequence[int]] = None,
                             spare_blocks: int = 0) -> ConsensusStructure:
    """Pairs, block pool and block tables for ``spec`` (seeded by spec.seed)."""
    rng = np.random.default_rng(spec.seed)
    B = spec.batch
    lens = (np.full(B, spec.prompt_len + spec.gen_len, dtype=np.int64) if seq_lens is None
            else np.asarray(seq_lens, dtype=np.int64))
    bounds_list = []
    for b in range(B):
        L = int(lens[b])
        bd = [spec.prompt_len]
        pos = spec.prompt_len
        while True:
            r = int(rng.integers(spec.reg_len_range[0], spec.reg_len_range[1] + 1))
            s = int(rng.integers(spec.sum_len_range[0], spec.sum_len_range[1] + 1))
            if pos + r + s > L:
                break
            bd += [pos + r, pos + r + s]
            pos += r + s
        assert len(bd) >= 3, "sequence too short for one (regular, summary) pair"
        bounds_list.append(np.array(bd, dtype=np.int32))
    n_seg = np.array([(len(x) - 1) // 2 for x in bounds_list], dtype=np.int64)
    seg_ptr = np.concatenate([[0], np.cumsum(n_seg)]).astype(np.int32)
    seg_bounds = np.concatenate(bounds_list).astype(np.int32)
    nblk = (lens + BLOCK_SIZE - 1) // BLOCK_SIZE
    num_blocks = int(nblk.sum()) + spare_blocks
    alloc = PagedBlockAllocator(num_blocks, rng)
    tables = np.full((B, int(nblk.max())), -1, dtype=np.int32)
    for b in range(B):
        own = alloc.alloc(int(nblk[b]))
        tables[b, :len(own)] = own
    return ConsensusStructure(spec, lens.astype(np.int32), np.full(B, spec.prompt_len, np.int32), seg_ptr,
                              seg_bounds, np.full(B, spec.topk, np.int32), np.full(B, spec.consensus, np.int32),
                              spec.window, num_blocks, tables)


@dataclass
class ConsensusLayer:
    q: torch.Tensor        # [B, Hq, d] dtype
    k_pool: torch.Tensor   # [num_blocks, Hkv, 16, d] dtype
    v_pool: torch.Tensor   # [num_blocks, Hkv, 16, d] dtype
    logical_k: Optional[List[torch.Tensor]] = field(default=None)  # per seq [L_b, Hkv, d] dtype
    logical_v: Optional[List[torch.Tensor]] = field(default=None)


def make_consensus_layer(st: ConsensusStructure, layer: int, device: str | torch.device = "cpu", *,
                         keep_logical: bool = False) -> ConsensusLayer:
    """One layer's queries and paged K/V pools: K, V ~ N(0, 1) in the storage dtype; every query head's
    query is 3 x the mean of the stored K rows (its KV head) of one uniformly drawn summary segment, plus
    N(0, 1). Seeded by spec.seed * 1000 + layer (torch generator on the device, numpy for the choices)."""
    spec = st.spec
    dev = torch.device(device)
    dt = torch_dtype(spec.dtype)
    seed = spec.seed * 1000 + layer
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    nrng = np.random.default_rng(seed)
    B, Hq, Hkv, d = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    G = Hq // Hkv
    k_pool = torch.zeros((st.num_blocks, Hkv, BLOCK_SIZE, d), dtype=dt, device=dev)
    v_pool = torch.zeros((st.num_blocks, Hkv, BLOCK_SIZE, d), dtype=dt, device=dev)
    q = torch.empty((B, Hq, d), dtype=dt, device=dev)
    lk_all, lv_all = [], []
    for b in range(B):
        L = int(st.seq_lens[b])
        kk = torch.randn((L, Hkv, d), generator=gen, device=dev).to(dt)
        vv = torch.randn((L, Hkv, d), generator=gen, device=dev).to(dt)
        nblk = (L + BLOCK_SIZE - 1) // BLOCK_SIZE
        idx = torch.from_numpy(st.block_tables[b, :nblk].astype(np.int64)).to(dev)
        for src, pool in ((kk, k_pool), (vv, v_pool)):
            pad = torch.zeros((nblk * BLOCK_SIZE, Hkv, d), dtype=dt, device=dev)
            pad[:L] = src
            pool[idx] = pad.view(nblk, BLOCK_SIZE, Hkv, d).permute(0, 2, 1, 3)
        spans = st.summary_spans(b)
        picks = nrng.integers(0, len(spans), size=Hq)
        for h in range(Hq):
            s, e = spans[int(picks[h])]
            base = kk[s:e, h // G].to(torch.float64).mean(0)
            noise = torch.randn((d,), generator=gen, device=dev).to(torch.float64)
            q[b, h] = (3.0 * base + noise).to(torch.float32).to(dt)
        if keep_logical:
            lk_all.append(kk)
            lv_all.append(vv)
    return ConsensusLayer(q, k_pool, v_pool, lk_all if keep_logical else None, lv_all if keep_logical else None)


def consensus_spec(**kw) -> ConsensusSpec:
    """A custom consensus workload for tests (defaults: the tiny fp32 case)."""
    base = dataclasses.asdict(CONSENSUS_WORKLOADS[0])
    base.update(kw)
    return ConsensusSpec(**base)
