"""GPU-vs-oracle comparison helpers (the GPU side runs only through the C ABI)."""

from __future__ import annotations

from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z
from oracle import zoomr_oracle as O
from tests.helpers import oracle_args

TOL = {"bf16": 2e-3, "f32": 1e-5}


def device_tables(st: W.Structure, device="cuda") -> torch.Tensor:
    return torch.from_numpy(st.block_tables.astype(np.int32)).to(device)


def run_gpu(plan: Z.DecodePlan, lt: W.LayerTensors, bt: torch.Tensor, debug: bool = True):
    B, Hq, d = lt.q.shape
    out = torch.full((B, Hq, d), float("nan"), dtype=torch.float32, device=lt.q.device)
    dbg = plan.new_debug_outputs() if debug else None
    plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out, dbg)
    return out, dbg


def fetch(out, dbg, plan: Z.DecodePlan):
    torch.cuda.synchronize()
    err = plan.device_error()
    o = out.cpu().numpy()
    sel, rng, nr = (x.cpu().numpy() for x in dbg)
    return err, o, sel, rng, nr


def expand_ranges(ranges: np.ndarray) -> np.ndarray:
    if len(ranges) == 0:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([np.arange(int(s), int(e)) for s, e in ranges]).astype(np.int64)


def check_selection(st: W.Structure, res_units, sel, rng, nr, units: Iterable[Tuple[int, int]]):
    """Bit-exact: selected segment indices, -1 padding, gathered token ranges (maximal runs)."""
    for (b, g) in units:
        u = res_units[b][g]
        k_eff = len(u.sel)
        assert list(sel[b, g, :k_eff]) == list(u.sel), (b, g, sel[b, g], u.sel)
        assert np.all(sel[b, g, k_eff:] == -1), (b, g)
        r = rng[b, g, :nr[b, g]]
        assert np.array_equal(r, O.token_ranges(u.tokens)), (b, g, r)
        assert np.array_equal(expand_ranges(r), u.tokens), (b, g)


def check_outputs(res, o: np.ndarray, units: Iterable[Tuple[int, int]], G: int, tol: float) -> float:
    worst = 0.0
    for (b, g) in units:
        got = o[b, g * G:(g + 1) * G].astype(np.float64)
        want = res.units[b][g].out
        assert np.all(np.isfinite(got)), (b, g)
        e = float(np.max(np.abs(got - want)))
        worst = max(worst, e)
        assert e <= tol, (b, g, e)
    return worst


def parity(st: W.Structure, lt: W.LayerTensors, plan: Optional[Z.DecodePlan] = None,
           units: Optional[Sequence[Tuple[int, int]]] = None, tol: Optional[float] = None) -> dict:
    """Run one layer on the GPU and compare it with the oracle on ``units`` (default: all)."""
    plan = plan or Z.DecodePlan.from_structure(st)
    bt = device_tables(st, lt.q.device)
    out, dbg = run_gpu(plan, lt, bt)
    err, o, sel, rng, nr = fetch(out, dbg, plan)
    assert err == 0, f"device error word {err}"
    all_units = [(b, g) for b in range(st.batch) for g in range(st.spec.num_kv_heads)]
    units = list(units) if units is not None else all_units
    res = O.decode_step(**oracle_args(st, lt), units=units)
    check_selection(st, res.units, sel, rng, nr, units)
    G = st.spec.num_q_heads // st.spec.num_kv_heads
    worst = check_outputs(res, o, units, G, tol if tol is not None else TOL[st.spec.dtype])
    return dict(max_abs_err=worst, out=o, sel=sel, ranges=rng, nranges=nr, oracle=res)


def min_score_margin(res, units, topk) -> float:
    """Smallest gap s_(k) - s_(k+1) of the exact keys (as floats) at the top-k boundary over ``units``."""
    m = float("inf")
    for (b, g) in units:
        keys = np.sort(res.units[b][g].keys.astype(np.float64))[::-1]
        k = min(int(topk[b]), len(keys))
        if 0 < k < len(keys):
            m = min(m, keys[k - 1] - keys[k])
    return m
