"""Thin ctypes binding of ``libzoomr.so`` (declared in ``include/zoomr.h``).

The functions carry the C names and only marshal arguments: torch tensors are
passed as raw device pointers, host metadata as int32 arrays. Every step of the
decode runs in the library's CUDA kernels; there is no Python or CPU fallback,
and a missing library raises ``ZoomrLibraryMissing``.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzoomr.so")

ZR_OK, ZR_EINVAL, ZR_ENOMEM, ZR_ECUDA, ZR_EUNSUPPORTED, ZR_EDEVICE = range(6)
ZR_F32, ZR_BF16 = 0, 1
DTYPES = {"f32": ZR_F32, "bf16": ZR_BF16}
TORCH_DTYPES = {ZR_F32: torch.float32, ZR_BF16: torch.bfloat16}


class ZoomrLibraryMissing(RuntimeError):
    pass


class ZoomrError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {zr_status_string(status)}")


class zr_config(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("max_blocks_per_seq", ctypes.c_int32), ("window", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lib: Optional[ctypes.CDLL] = None
_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once). Raises ZoomrLibraryMissing if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ZoomrLibraryMissing(f"{path} is missing: build it with `python -m hierarchical_sparse_kv_gb300.build`")
    lib = ctypes.CDLL(path)
    lib.zr_plan.argtypes = [ctypes.POINTER(zr_config), _I32P, _I32P, _I32P, _I32P, ctypes.POINTER(_P),
                            ctypes.POINTER(ctypes.c_size_t)]
    lib.zr_plan.restype = ctypes.c_int
    lib.zr_plan_sink.argtypes = [ctypes.POINTER(zr_config), _I32P, _I32P, _I32P, _I32P, _I32P, ctypes.POINTER(_P),
                                 ctypes.POINTER(ctypes.c_size_t)]
    lib.zr_plan_sink.restype = ctypes.c_int
    lib.zr_plan_dims.argtypes = [_P, _I32P, _I32P]
    lib.zr_plan_dims.restype = ctypes.c_int
    lib.zr_decode_attend.argtypes = [_P] * 13
    lib.zr_decode_attend.restype = ctypes.c_int
    lib.zr_decode_attend_timed.argtypes = [_P] * 12
    lib.zr_decode_attend_timed.restype = ctypes.c_int
    lib.zr_decode_attend_static.argtypes = [_P] * 9
    lib.zr_decode_attend_static.restype = ctypes.c_int
    lib.zr_get_device_error.argtypes = [_P, _P, _P, _I32P]
    lib.zr_get_device_error.restype = ctypes.c_int
    lib.zr_append_kv.argtypes = [ctypes.POINTER(zr_config)] + [_P] * 8
    lib.zr_append_kv.restype = ctypes.c_int
    lib.zr_copy_blocks.argtypes = [ctypes.POINTER(zr_config), _P, ctypes.c_int32, _P, _P, _P, _P]
    lib.zr_copy_blocks.restype = ctypes.c_int
    lib.zr_segment_summaries.argtypes = [ctypes.POINTER(zr_config), _P, ctypes.c_int32] + [_P] * 5 + \
        [ctypes.c_int32, _P, _P]
    lib.zr_segment_summaries.restype = ctypes.c_int
    lib.zr_consensus_plan.argtypes = [ctypes.POINTER(zr_config)] + [_I32P] * 6 + [ctypes.POINTER(_P),
                                                                             ctypes.POINTER(ctypes.c_size_t)]
    lib.zr_consensus_plan.restype = ctypes.c_int
    lib.zr_consensus_dims.argtypes = [_P, _I32P, _I32P]
    lib.zr_consensus_dims.restype = ctypes.c_int
    lib.zr_consensus_vote.argtypes = [_P] * 5
    lib.zr_consensus_vote.restype = ctypes.c_int
    lib.zr_consensus_select.argtypes = [_P] * 7
    lib.zr_consensus_select.restype = ctypes.c_int
    lib.zr_consensus_attend.argtypes = [_P] * 8
    lib.zr_consensus_attend.restype = ctypes.c_int
    lib.zr_consensus_attend_timed.argtypes = [_P] * 10
    lib.zr_consensus_attend_timed.restype = ctypes.c_int
    lib.zr_decode_advance.argtypes = [_P] * 4
    lib.zr_decode_advance.restype = ctypes.c_int
    lib.zr_decode_attend_reuse.argtypes = [_P] * 10
    lib.zr_decode_attend_reuse.restype = ctypes.c_int
    lib.zr_consensus_advance.argtypes = [_P] * 4
    lib.zr_consensus_advance.restype = ctypes.c_int
    lib.zr_offload_map.argtypes = [_P, _P, _P, ctypes.c_int32, _P, _P, _P, _P]
    lib.zr_offload_map.restype = ctypes.c_int
    lib.zr_offload_stage.argtypes = [_P] * 6 + [ctypes.c_int32, _P, _P, _P]
    lib.zr_offload_stage.restype = ctypes.c_int
    lib.zr_plan_set_deterministic.argtypes = [_P, ctypes.c_int32]
    lib.zr_plan_set_deterministic.restype = ctypes.c_int
    lib.zr_free.argtypes = [_P]
    lib.zr_free.restype = None
    lib.zr_status_string.argtypes = [ctypes.c_int]
    lib.zr_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def zr_status_string(status: int) -> str:
    return load().zr_status_string(int(status)).decode()


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr32(a: np.ndarray):
    return a.ctypes.data_as(_I32P)


def _dev(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("zoomr: tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def _pool(t: torch.Tensor) -> int:
    """A K/V pool may live in HBM or in pinned host memory: with unified addressing a pinned host
    allocation is mapped into the device's address space at the same address, and the kernels read
    it across the CPU-GPU link (NVLink-C2C on a Grace system)."""
    if t.is_cuda:
        return _dev(t)
    if t.device.type == "cpu" and t.is_pinned() and t.is_contiguous():
        return t.data_ptr()
    raise ValueError("zoomr: a K/V pool must be a contiguous CUDA tensor or a contiguous pinned host tensor")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def zr_plan(cfg: zr_config, seq_lens, seg_ptr, seg_bounds, topk, sink_lens=None) -> Tuple[int, int]:
    """Returns (plan handle, workspace bytes); with ``sink_lens``, zr_plan_sink. Raises ZoomrError on a
    non-OK status."""
    lib = load()
    a = [_i32(x) for x in (seq_lens, seg_ptr, seg_bounds, topk)]
    plan = _P()
    ws = ctypes.c_size_t()
    if sink_lens is None:
        st = lib.zr_plan(ctypes.byref(cfg), *[_ptr32(x) for x in a], ctypes.byref(plan), ctypes.byref(ws))
    else:
        sk = _i32(sink_lens)
        st = lib.zr_plan_sink(ctypes.byref(cfg), _ptr32(a[0]), _ptr32(sk), *[_ptr32(x) for x in a[1:]],
                              ctypes.byref(plan), ctypes.byref(ws))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_plan_sink" if sink_lens is not None else "zr_plan")
    return plan.value, ws.value


def zr_plan_status(cfg: Optional[zr_config], seq_lens, seg_ptr, seg_bounds, topk) -> int:
    """zr_plan's raw status (any plan created is freed): for error-path tests."""
    lib = load()
    a = [_i32(x) for x in (seq_lens, seg_ptr, seg_bounds, topk)]
    plan = _P()
    ws = ctypes.c_size_t()
    st = lib.zr_plan(ctypes.byref(cfg) if cfg is not None else None, *[_ptr32(x) for x in a], ctypes.byref(plan),
                     ctypes.byref(ws))
    if st == ZR_OK:
        lib.zr_free(plan)
    return st


def zr_plan_dims(plan: int) -> Tuple[int, int]:
    k_max, n_max = ctypes.c_int32(), ctypes.c_int32()
    st = load().zr_plan_dims(plan, ctypes.byref(k_max), ctypes.byref(n_max))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_plan_dims")
    return k_max.value, n_max.value


def zr_decode_attend(plan: int, workspace: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                     v_pool: torch.Tensor, block_tables: torch.Tensor, sum_k: torch.Tensor, sum_v: torch.Tensor,
                     out: torch.Tensor, sel_out: Optional[torch.Tensor] = None,
                     ranges_out: Optional[torch.Tensor] = None, nranges_out: Optional[torch.Tensor] = None,
                     stream=None) -> None:
    st = load().zr_decode_attend(plan, _dev(workspace), _dev(q), _pool(k_pool), _pool(v_pool), _dev(block_tables),
                                 _dev(sum_k), _dev(sum_v), _dev(out), _dev(sel_out), _dev(ranges_out),
                                 _dev(nranges_out), _stream(stream))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_decode_attend")


def _event(ev: Optional[torch.cuda.Event], stream=None) -> Optional[int]:
    """The cudaEvent_t of a torch event (None stays None), created by a first record if needed."""
    if ev is None:
        return None
    if ev.cuda_event == 0:  # torch creates the CUDA event lazily, at its first record
        if torch.cuda.is_current_stream_capturing():
            raise ValueError("zoomr: record timing events once before using them inside a stream capture")
        ev.record(torch.cuda.current_stream() if stream is None or isinstance(stream, int) else stream)
    return ev.cuda_event


def zr_decode_attend_timed(plan: int, workspace: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                           v_pool: torch.Tensor, block_tables: torch.Tensor, sum_k: torch.Tensor,
                           sum_v: torch.Tensor, out: torch.Tensor, ev_start: Optional[torch.cuda.Event],
                           ev_stop: Optional[torch.cuda.Event], stream=None) -> None:
    st = load().zr_decode_attend_timed(plan, _dev(workspace), _dev(q), _pool(k_pool), _pool(v_pool),
                                       _dev(block_tables), _dev(sum_k), _dev(sum_v), _dev(out),
                                       _event(ev_start, stream), _event(ev_stop, stream), _stream(stream))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_decode_attend_timed")


def zr_decode_attend_static(plan: int, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                            block_tables: torch.Tensor, sum_k: torch.Tensor, sum_v: torch.Tensor,
                            out: torch.Tensor, stream=None) -> None:
    """The decode step with the library's static 16 MiB device scratch instead of a
    caller workspace, for callers that cannot allocate device memory."""
    st = load().zr_decode_attend_static(plan, _dev(q), _pool(k_pool), _pool(v_pool), _dev(block_tables), _dev(sum_k),
                                        _dev(sum_v), _dev(out), _stream(stream))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_decode_attend_static")


def zr_get_device_error(plan: int, workspace: torch.Tensor, stream=None) -> int:
    code = ctypes.c_int32()
    st = load().zr_get_device_error(plan, _dev(workspace), _stream(stream), ctypes.byref(code))
    if st not in (ZR_OK, ZR_EDEVICE):
        raise ZoomrError(st, "zr_get_device_error")
    return code.value


def zr_plan_set_deterministic(plan: int, deterministic: bool) -> None:
    """The attend-only calls' even split of the rows (outputs bit-identical across calls) or their default dynamic
    split; the decode step always takes the even split."""
    st = load().zr_plan_set_deterministic(plan, 1 if deterministic else 0)
    if st != ZR_OK:
        raise ZoomrError(st, "zr_plan_set_deterministic")


def zr_free(plan: Optional[int]) -> None:
    if plan:
        load().zr_free(plan)


def cache_config(*, batch: int, num_kv_heads: int, head_dim: int, num_blocks: int, max_blocks_per_seq: int,
                 dtype: str, num_q_heads: int = 0, window: int = 0) -> zr_config:
    """A zr_config for the append-path calls (they ignore num_q_heads and window)."""
    return zr_config(batch, num_q_heads, num_kv_heads, head_dim, 16, num_blocks, max_blocks_per_seq, window,
                     DTYPES[dtype])


def _check_cache(cfg: zr_config, k_pool: torch.Tensor, v_pool: torch.Tensor,
                 block_tables: Optional[torch.Tensor] = None) -> None:
    """The C ABI cannot see buffer sizes: check the tensors against the config here."""
    want = (cfg.num_blocks, cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    dt = TORCH_DTYPES.get(cfg.dtype)
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool)):
        if tuple(t.shape) != want or t.dtype != dt:
            raise ValueError(f"zoomr: {name} must be {want} {dt}, got {tuple(t.shape)} {t.dtype}")
    if block_tables is not None and (tuple(block_tables.shape) != (cfg.batch, cfg.max_blocks_per_seq)
                                     or block_tables.dtype != torch.int32):
        raise ValueError(f"zoomr: block_tables must be int32 {(cfg.batch, cfg.max_blocks_per_seq)}")


def _check_rows(name: str, t: Optional[torch.Tensor], shape: tuple, dtype: torch.dtype) -> None:
    if t is not None and (tuple(t.shape) != shape or t.dtype != dtype):
        raise ValueError(f"zoomr: {name} must be {shape} {dtype}, got {tuple(t.shape)} {t.dtype}")


def zr_append_kv(cfg: zr_config, positions: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                 block_tables: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                 err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Writes k_new/v_new [B, Hkv, d] at token positions[b] (int32, negative: skip) of each sequence."""
    _check_cache(cfg, k_pool, v_pool, block_tables)
    _check_rows("positions", positions, (cfg.batch,), torch.int32)
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _check_rows(name, t, (cfg.batch, cfg.num_kv_heads, cfg.head_dim), TORCH_DTYPES[cfg.dtype])
    st = load().zr_append_kv(ctypes.byref(cfg), _dev(positions), _dev(k_new), _dev(v_new), _dev(block_tables),
                             _pool(k_pool), _pool(v_pool), _dev(err), _stream(stream))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_append_kv")


def zr_copy_blocks(cfg: zr_config, pairs: Optional[torch.Tensor], k_pool: torch.Tensor, v_pool: torch.Tensor,
                   err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copies whole blocks pairs[i, 0] -> pairs[i, 1] (int32 [n, 2]) in both pools."""
    n = 0 if pairs is None else int(pairs.shape[0])
    _check_cache(cfg, k_pool, v_pool)
    _check_rows("pairs", pairs, (n, 2), torch.int32)
    st = load().zr_copy_blocks(ctypes.byref(cfg), _dev(pairs) if n else None, n, _pool(k_pool), _pool(v_pool),
                               _dev(err), _stream(stream))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_copy_blocks")


def zr_segment_summaries(cfg: zr_config, segs: Optional[torch.Tensor], block_tables: torch.Tensor,
                         k_pool: torch.Tensor, v_pool: torch.Tensor, sum_k: torch.Tensor, sum_v: torch.Tensor,
                         err: Optional[torch.Tensor] = None, stream=None) -> None:
    """Mean summary K/V rows of segs[i] = (b, start, end, row) (int32 [n, 4]) into sum_k/sum_v [rows, Hkv, d]."""
    n = 0 if segs is None else int(segs.shape[0])
    _check_cache(cfg, k_pool, v_pool, block_tables)
    _check_rows("segs", segs, (n, 4), torch.int32)
    rows = (int(sum_k.shape[0]), cfg.num_kv_heads, cfg.head_dim)
    _check_rows("sum_k", sum_k, rows, TORCH_DTYPES[cfg.dtype])
    _check_rows("sum_v", sum_v, rows, TORCH_DTYPES[cfg.dtype])
    st = load().zr_segment_summaries(ctypes.byref(cfg), _dev(segs) if n else None, n, _dev(block_tables),
                                     _pool(k_pool), _pool(v_pool), _dev(sum_k), _dev(sum_v), int(sum_k.shape[0]),
                                     _dev(err), _stream(stream))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_segment_summaries")


def zr_offload_map(plan: int, workspace: torch.Tensor, block_tables: torch.Tensor, capacity: int,
                   stage_ids: torch.Tensor, remap_tables: torch.Tensor, n_staged: torch.Tensor, stream=None) -> None:
    """Staging slots for the blocks the workspace's current token ranges touch (ZoomR 3.4, the offloaded
    cache): stage_ids [capacity], remap_tables [B, max_blocks] and n_staged [1], all int32 on the device."""
    for name, t in (("stage_ids", stage_ids), ("remap_tables", remap_tables), ("n_staged", n_staged)):
        if t.dtype != torch.int32 or not t.is_cuda:
            raise ValueError(f"{name} must be an int32 CUDA tensor")
    if stage_ids.numel() < capacity or n_staged.numel() < 1 or remap_tables.shape != block_tables.shape:
        raise ValueError("zr_offload_map: stage_ids holds capacity entries, remap_tables matches block_tables")
    st = load().zr_offload_map(plan, _dev(workspace), _dev(block_tables), int(capacity), _dev(stage_ids),
                               _dev(remap_tables), _dev(n_staged), _stream(stream))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_offload_map")


def zr_offload_stage(plan: int, workspace: torch.Tensor, host_k_pool: torch.Tensor, host_v_pool: torch.Tensor,
                     stage_ids: torch.Tensor, n_staged: torch.Tensor, capacity: int, stage_k: torch.Tensor,
                     stage_v: torch.Tensor, stream=None) -> None:
    """One layer's staging copy: the rows of the mapped blocks that the workspace's ranges cover (the row
    masks zr_offload_map left in the workspace), from the host pools into slots of the staging pools."""
    if stage_k.shape[0] < capacity or stage_v.shape[0] < capacity:
        raise ValueError("zr_offload_stage: the staging pools hold capacity blocks")
    st = load().zr_offload_stage(plan, _dev(workspace), _pool(host_k_pool), _pool(host_v_pool), _dev(stage_ids),
                                 _dev(n_staged), int(capacity), _dev(stage_k), _dev(stage_v), _stream(stream))
    if st != ZR_OK:
        raise ZoomrError(st, "zr_offload_stage")


class DecodePlan:
    """A plan plus its workspace: one ZoomR decode step per call, on the current stream.

    Host metadata follow the C ABI (``include/zoomr.h``): seq_lens [B], seg_ptr
    [B+1] (CSR over segments), seg_bounds (sequence b's n_b + 1 bounds start at
    seg_ptr[b] + b), topk [B]. Tensors passed to ``run`` are the caller's.
    """

    def __init__(self, *, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, num_blocks: int,
                 max_blocks_per_seq: int, window: int, dtype: str, seq_lens: Sequence[int], seg_ptr: Sequence[int],
                 seg_bounds: Sequence[int], topk: Sequence[int], device=None, sink_lens=None):
        self.cfg = zr_config(batch, num_q_heads, num_kv_heads, head_dim, 16, num_blocks, max_blocks_per_seq, window,
                             DTYPES[dtype])
        self.device = torch.device(device if device is not None else "cuda")
        with torch.cuda.device(self.device):
            self.handle, self.workspace_bytes = zr_plan(self.cfg, seq_lens, seg_ptr, seg_bounds, topk, sink_lens)
            self.k_max, self.n_max = zr_plan_dims(self.handle)
            self.workspace = torch.zeros(max(self.workspace_bytes, 256) // 4 + 64, dtype=torch.int32,
                                         device=self.device)
        # 256-byte aligned view of the workspace
        off = (-self.workspace.data_ptr()) % 256
        self.ws = self.workspace[off // 4:]
        assert self.ws.data_ptr() % 256 == 0
        self.batch, self.num_q_heads, self.num_kv_heads, self.head_dim = batch, num_q_heads, num_kv_heads, head_dim

    @classmethod
    def from_structure(cls, st, device=None) -> "DecodePlan":
        """Plan for a ``workloads.Structure`` (any object with the same fields)."""
        sp = st.spec
        return cls(batch=st.batch, num_q_heads=sp.num_q_heads, num_kv_heads=sp.num_kv_heads, head_dim=sp.head_dim,
                   num_blocks=st.num_blocks, max_blocks_per_seq=st.max_blocks_per_seq, window=st.window,
                   dtype=sp.dtype, seq_lens=st.seq_lens, seg_ptr=st.seg_ptr, seg_bounds=st.seg_bounds, topk=st.topk,
                   device=device, sink_lens=getattr(st, "sink_lens", None))

    def new_debug_outputs(self):
        B, H = self.batch, self.num_kv_heads
        sel = torch.full((B, H, self.k_max), -2, dtype=torch.int32, device=self.device)
        rng = torch.full((B, H, self.k_max + 1, 2), -2, dtype=torch.int32, device=self.device)
        nr = torch.full((B, H), -2, dtype=torch.int32, device=self.device)
        return sel, rng, nr

    def run(self, q, k_pool, v_pool, block_tables, sum_k, sum_v, out, debug=None, stream=None) -> None:
        sel, rng, nr = debug if debug is not None else (None, None, None)
        zr_decode_attend(self.handle, self.ws, q, k_pool, v_pool, block_tables, sum_k, sum_v, out, sel, rng, nr,
                         stream)

    def run_timed(self, q, k_pool, v_pool, block_tables, sum_k, sum_v, out, ev_start, ev_stop, stream=None):
        zr_decode_attend_timed(self.handle, self.ws, q, k_pool, v_pool, block_tables, sum_k, sum_v, out, ev_start,
                               ev_stop, stream)

    def advance(self, seq_lens: torch.Tensor, stream=None) -> None:
        """Move every unit's window to the new lengths (device int32 [B]), the selection held fixed."""
        _check_rows("seq_lens", seq_lens, (self.batch,), torch.int32)
        st = load().zr_decode_advance(self.handle, _dev(self.ws), _dev(seq_lens), _stream(stream))
        if st != ZR_OK:
            raise ZoomrError(st, "zr_decode_advance")

    def run_reuse(self, q, k_pool, v_pool, block_tables, sum_k, sum_v, out, stream=None) -> None:
        """Gather-attention and merge over the ranges in the workspace (no scoring or selection)."""
        st = load().zr_decode_attend_reuse(self.handle, _dev(self.ws), _dev(q), _pool(k_pool), _pool(v_pool),
                                           _dev(block_tables), _dev(sum_k), _dev(sum_v), _dev(out), _stream(stream))
        if st != ZR_OK:
            raise ZoomrError(st, "zr_decode_attend_reuse")

    def device_error(self, stream=None) -> int:
        return zr_get_device_error(self.handle, self.ws, stream)

    def set_deterministic(self, deterministic: bool = True):
        """Bit-identical outputs across calls (the even split of the rows in the attend-only calls too) or their
        default dynamic split; returns self."""
        zr_plan_set_deterministic(self.handle, deterministic)
        return self

    def close(self):
        if getattr(self, "handle", None):
            zr_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zr_consensus_plan_status(cfg: Optional[zr_config], seq_lens, prompt_lens, seg_ptr, pair_bounds, topk,
                             consensus) -> int:
    """zr_consensus_plan's raw status (any plan created is freed): for error-path tests."""
    lib = load()
    a = [_i32(x) for x in (seq_lens, prompt_lens, seg_ptr, pair_bounds, topk, consensus)]
    plan = _P()
    ws = ctypes.c_size_t()
    st = lib.zr_consensus_plan(ctypes.byref(cfg) if cfg is not None else None, *[_ptr32(x) for x in a],
                               ctypes.byref(plan), ctypes.byref(ws))
    if st == ZR_OK:
        lib.zr_free(plan)
    return st


class ConsensusPlan:
    """ZoomR's consensus path (``zr_consensus_*``): per-layer votes, one selection, per-layer attention.

    Host metadata follow the C ABI: seq_lens, prompt_lens [B]; seg_ptr [B+1] (CSR over the (regular,
    summary) pairs); pair_bounds (sequence b's 2 n_b + 1 bounds start at 2 seg_ptr[b] + b); topk and
    consensus [B].
    """

    def __init__(self, *, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, num_blocks: int,
                 max_blocks_per_seq: int, window: int, dtype: str, seq_lens, prompt_lens, seg_ptr, pair_bounds,
                 topk, consensus, device=None):
        self.cfg = zr_config(batch, num_q_heads, num_kv_heads, head_dim, 16, num_blocks, max_blocks_per_seq, window,
                             DTYPES[dtype])
        self.device = torch.device(device if device is not None else "cuda")
        lib = load()
        a = [_i32(x) for x in (seq_lens, prompt_lens, seg_ptr, pair_bounds, topk, consensus)]
        plan, ws = _P(), ctypes.c_size_t()
        with torch.cuda.device(self.device):
            st = lib.zr_consensus_plan(ctypes.byref(self.cfg), *[_ptr32(x) for x in a], ctypes.byref(plan),
                                       ctypes.byref(ws))
            if st != ZR_OK:
                raise ZoomrError(st, "zr_consensus_plan")
            self.handle, self.workspace_bytes = plan.value, ws.value
            c_max, n_max = ctypes.c_int32(), ctypes.c_int32()
            st = lib.zr_consensus_dims(self.handle, ctypes.byref(c_max), ctypes.byref(n_max))
            if st != ZR_OK:
                raise ZoomrError(st, "zr_consensus_dims")
            self.c_max, self.n_max = c_max.value, n_max.value
            self.workspace = torch.zeros(max(self.workspace_bytes, 256) // 4 + 64, dtype=torch.int32,
                                         device=self.device)
        off = (-self.workspace.data_ptr()) % 256
        self.ws = self.workspace[off // 4:]
        self.batch, self.num_q_heads, self.num_kv_heads, self.head_dim = batch, num_q_heads, num_kv_heads, head_dim

    @classmethod
    def from_structure(cls, st, device=None) -> "ConsensusPlan":
        """Plan for a ``workloads.ConsensusStructure`` (any object with the same fields)."""
        sp = st.spec
        return cls(batch=st.batch, num_q_heads=sp.num_q_heads, num_kv_heads=sp.num_kv_heads, head_dim=sp.head_dim,
                   num_blocks=st.num_blocks, max_blocks_per_seq=st.max_blocks_per_seq, window=st.window,
                   dtype=sp.dtype, seq_lens=st.seq_lens, prompt_lens=st.prompt_lens, seg_ptr=st.seg_ptr,
                   pair_bounds=st.seg_bounds, topk=st.topk, consensus=st.consensus, device=device)

    def vote(self, q: torch.Tensor, mean_keys: torch.Tensor, stream=None) -> None:
        st = load().zr_consensus_vote(self.handle, _dev(self.ws), _dev(q), _dev(mean_keys), _stream(stream))
        if st != ZR_OK:
            raise ZoomrError(st, "zr_consensus_vote")

    def new_debug_outputs(self):
        B = self.batch
        mk = lambda shape: torch.full(shape, -2, dtype=torch.int32, device=self.device)
        return mk((B, self.n_max)), mk((B, self.c_max)), mk((B, self.n_max + 2, 2)), mk((B,))

    def select(self, debug=None, stream=None) -> None:
        votes, ic, rng, nr = debug if debug is not None else (None, None, None, None)
        st = load().zr_consensus_select(self.handle, _dev(self.ws), _dev(votes), _dev(ic), _dev(rng), _dev(nr),
                                        _stream(stream))
        if st != ZR_OK:
            raise ZoomrError(st, "zr_consensus_select")

    def attend(self, q, k_pool, v_pool, block_tables, out, stream=None) -> None:
        st = load().zr_consensus_attend(self.handle, _dev(self.ws), _dev(q), _pool(k_pool), _pool(v_pool),
                                        _dev(block_tables), _dev(out), _stream(stream))
        if st != ZR_OK:
            raise ZoomrError(st, "zr_consensus_attend")

    def attend_timed(self, q, k_pool, v_pool, block_tables, out, ev_start, ev_stop, stream=None) -> None:
        """attend with CUDA events just before and just after the gather-attention kernel (either may be None)."""
        st = load().zr_consensus_attend_timed(self.handle, _dev(self.ws), _dev(q), _pool(k_pool), _pool(v_pool),
                                              _dev(block_tables), _dev(out), _event(ev_start, stream),
                                              _event(ev_stop, stream), _stream(stream))
        if st != ZR_OK:
            raise ZoomrError(st, "zr_consensus_attend_timed")

    def advance(self, seq_lens: torch.Tensor, stream=None) -> None:
        """Move every sequence's window to the new lengths (device int32 [B]), I_c and I_s held fixed."""
        _check_rows("seq_lens", seq_lens, (self.batch,), torch.int32)
        st = load().zr_consensus_advance(self.handle, _dev(self.ws), _dev(seq_lens), _stream(stream))
        if st != ZR_OK:
            raise ZoomrError(st, "zr_consensus_advance")

    def device_error(self, stream=None) -> int:
        return zr_get_device_error(self.handle, self.ws, stream)

    def set_deterministic(self, deterministic: bool = True):
        """Bit-identical outputs across calls (the even split of the rows in the attend-only calls too) or their
        default dynamic split; returns self."""
        zr_plan_set_deterministic(self.handle, deterministic)
        return self

    def close(self):
        if getattr(self, "handle", None):
            zr_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
