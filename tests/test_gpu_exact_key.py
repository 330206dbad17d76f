"""The exact ranking key on the GPU (select and vote kernels) against the oracle.

The key is the exact dot product q . s of the stored values (ZoomR page, 3.3 "Per-Head
Importance Scoring and Voting"). These cases are built so that only exact arithmetic gives the
oracle's selection:

* near-ties planted at the top-k boundary where an ascending fp32 chain ranks the pair the
  other way (bf16 on the 8 x 4K workload; fp32 on a small shape; bf16 and fp32 with 64 to 128
  segments per sequence, where the estimate takes 32 elements a lane);
* ties decided by one tiny value: a lower limb (about 2^-30 below the largest), a value below
  the 56-bit frame (the general 640-bit path), a subnormal, and the same on the query side;
* segment counts where the top-k is a radix select (300, 2048 and 4096 segments), with random
  keys and with keys that take only seven distinct values (ties broken by index at full depth);
* the consensus vote kernel with per-head near-ties and a value below the frame;
* a non-finite summary key: bit 3 (value 4) of the error word, no fault.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hierarchical_sparse_kv_gb300 import build as B
from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z
from oracle import zoomr_consensus as OC
from oracle import zoomr_oracle as O
from tests import gpu_common as C
from tests import near_ties as NT
from tests.helpers import oracle_args

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    Z.load()


def _layer(spec, layer=0):
    st = W.make_structure(spec)
    return st, W.make_layer(st, layer, "cuda")


def _fp32_chain_sel(st, lt, b, g):
    G = st.spec.num_q_heads // st.spec.num_kv_heads
    s0, n = int(st.seg_ptr[b]), st.num_segments(b)
    q = W.to_numpy32(lt.q)[b, g * G:(g + 1) * G]
    sk = W.to_numpy32(lt.sum_k)[s0:s0 + n, g]
    return list(O.select_top_k(NT.fp32_chain_keys(q, sk), int(st.topk[b])))


@pytest.mark.parametrize("spec", [W.WORKLOADS[1],
                                  W.small_spec(dtype="f32", head_dim=64, batch=3, num_q_heads=8, num_kv_heads=2,
                                               seq_len=1500, seg_len_range=(20, 60), topk=5, window=32, seed=21),
                                  # 64 < n <= 128 segments: the estimate takes 32 elements a lane (one pass)
                                  W.small_spec(dtype="bf16", head_dim=128, batch=4, num_q_heads=16, num_kv_heads=4,
                                               seq_len=3000, seg_len_range=(20, 40), topk=9, window=40, seed=23),
                                  W.small_spec(dtype="f32", head_dim=128, batch=3, num_q_heads=8, num_kv_heads=2,
                                               seq_len=3000, seg_len_range=(20, 40), topk=9, window=40, seed=24)],
                         ids=["bf16_8x4K", "f32_small", "bf16_n100", "f32_d128_n100"])
def test_planted_near_ties_follow_the_exact_order(spec):
    st, lt = _layer(spec)
    if spec.seg_len_range == (20, 40):
        assert all(64 < st.num_segments(b) <= 128 for b in range(st.batch))
    flips = NT.plant_near_ties(st, lt)
    assert len(flips) >= 4, flips
    r = C.parity(st, lt)
    for (b, g, i, j) in flips:
        got = [int(x) for x in r["sel"][b, g] if x >= 0]
        assert got == list(r["oracle"].units[b][g].sel)
        assert got != _fp32_chain_sel(st, lt, b, g), (b, g, i, j)
    print(f"{len(flips)} planted near-ties, all on the exact side")


def _tie_by_tiny_value(st, lt, b, g, tau: float, side: str):
    """Make the unit's boundary pair equal except in one component t, so that one tiny value decides
    their order in favour of the higher index (where the tie rule alone picks the lower one).

    Both rows become segment i's row with component t zeroed; h* is that row's best head. Side 's': the
    higher-index row gets +-tau at t, signed like q_h*[t]: head h* gains |q_h*[t] tau|, so that row's key
    (a maximum over heads) exceeds the other's, by at most max_h |q_h[t] tau|. Side 'q': q_h*[t] becomes
    tau and the higher-index row gets 0.25 at t, where t is a component whose other group heads are <= 0,
    so only h* gains (tau / 4). Returns (lower index, higher index)."""
    spec = st.spec
    G = spec.num_q_heads // spec.num_kv_heads
    s0, n = int(st.seg_ptr[b]), st.num_segments(b)
    k = min(int(st.topk[b]), n)
    q = W.to_numpy32(lt.q)[b, g * G:(g + 1) * G].copy()
    sk = W.to_numpy32(lt.sum_k)[s0:s0 + n, g].copy()
    i, j = NT.boundary_pair(q, sk, k)
    lo, hi = min(i, j), max(i, j)
    row = sk[i].copy()
    quiet = np.argsort(np.abs(sk[i]) * np.abs(q).max(axis=0))  # components that move keys the least
    if side == "s":
        t = int(next(c for c in quiet if np.all(q[:, c] != 0)))
        row[t] = 0.0
        hs = int(np.argmax(row.astype(np.float64) @ q.astype(np.float64).T))
        sk[lo] = row
        sk[hi] = row
        sk[hi, t] = np.float32(tau if q[hs, t] > 0 else -tau)
    else:
        row0 = row.copy()
        hs = int(np.argmax(row0.astype(np.float64) @ q.astype(np.float64).T))
        t = int(next(c for c in quiet if all(q[h, c] <= 0 for h in range(G) if h != hs)))
        row[t] = 0.0
        hs2 = int(np.argmax(row.astype(np.float64) @ q.astype(np.float64).T))
        assert hs2 == hs
        sk[lo] = row
        sk[hi] = row
        sk[hi, t] = np.float32(0.25)
        q[hs, t] = np.float32(tau)
    dt = lt.sum_k.dtype
    lt.sum_k[s0:s0 + n, g] = torch.from_numpy(sk).to(dt).cuda()
    lt.q[b, g * G:(g + 1) * G] = torch.from_numpy(q).to(dt).cuda()
    return lo, hi


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ties_decided_by_lower_limb_deep_and_subnormal_values(dtype):
    spec = W.small_spec(dtype=dtype, head_dim=128, batch=4, num_q_heads=8, num_kv_heads=2, seq_len=1200,
                        seg_len_range=(20, 60), topk=4, window=16, seed=33)
    st, lt = _layer(spec)
    cases = [(0, 0, 3e-9, "s"),    # a lower limb: about 2^-28 below the row's largest
             (0, 1, 1e-22, "s"),   # below the 56-bit frame: the general path
             (1, 0, 2e-39, "s"),   # a subnormal
             (1, 1, 1e-9, "q"),    # a lower limb on the query side
             (2, 0, 1e-25, "q"),   # below the frame on the query side
             (3, 1, 3e-38, "s")]
    planted = []
    for (b, g, tau, side) in cases:
        lo, hi = _tie_by_tiny_value(st, lt, b, g, tau, side)
        planted.append((b, g, lo, hi))
    r = C.parity(st, lt)
    for (b, g, lo, hi) in planted:
        sel = list(r["oracle"].units[b][g].sel)
        assert hi in sel and lo not in sel, (b, g, sel)  # the tiny value decided it
        assert [int(x) for x in r["sel"][b, g] if x >= 0] == sel


@pytest.mark.parametrize("n,k,distinct", [(300, 40, 0), (2048, 100, 0), (4096, 64, 0), (4096, 1000, 7),
                                          (2048, 2047, 0), (1000, 1, 5)])
def test_radix_select_at_large_segment_counts(n, k, distinct):
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=2, num_q_heads=4, num_kv_heads=1, seq_len=4 * n,
                        seg_len_range=(4, 4), topk=k, window=16, seed=40 + n)
    st, lt = _layer(spec)
    assert st.num_segments(0) == n
    if distinct:
        base = lt.sum_k[:distinct].clone()
        for b in range(st.batch):
            s0 = int(st.seg_ptr[b])
            idx = torch.arange(n, device="cuda") % distinct
            lt.sum_k[s0:s0 + n] = base[idx]
    r = C.parity(st, lt)
    assert np.all(r["sel"][:, :, :k] >= 0)


def test_consensus_votes_exact_with_near_ties_and_a_deep_value():
    st = W.make_consensus_structure(W.consensus_spec(dtype="bf16", head_dim=128, num_q_heads=8, num_kv_heads=2,
                                                     layers=1, topk=3, consensus=2, seed=51))
    lt = W.make_consensus_layer(st, 0, "cuda")
    sp = st.spec
    G = sp.num_q_heads // sp.num_kv_heads
    g = torch.Generator(device="cuda").manual_seed(5)
    mk = (torch.randn((st.total_segments, sp.num_kv_heads, sp.head_dim), generator=g, device="cuda") * 0.2).to(
        torch.bfloat16)
    q = W.to_numpy32(lt.q)
    mkn = W.to_numpy32(mk)
    planted = 0
    for b in range(st.batch):
        s0, n = int(st.seg_ptr[b]), st.num_segments(b)
        for h in range(sp.num_q_heads):
            kv = h // G
            qh = q[b, h:h + 1]
            i, j = NT.boundary_pair(qh, mkn[s0:s0 + n, kv], min(int(st.topk[b]), n))
            row = NT.near_tie_row(qh, mkn[s0:s0 + n, kv], i, j, "bf16")
            if row is not None:
                mkn[s0 + j, kv] = row
                planted += 1
    mkn[0, 0, 3] = 1e-30  # a value below the 56-bit frame: that unit takes the general path
    assert planted >= 3
    mk = torch.from_numpy(mkn).to(torch.bfloat16).cuda()
    plan = Z.ConsensusPlan.from_structure(st)
    plan.vote(lt.q, mk)
    dbg = plan.new_debug_outputs()
    plan.select(dbg)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    votes = dbg[0].cpu().numpy()
    mk32 = W.to_numpy32(mk)
    for b in range(st.batch):
        s0, n = int(st.seg_ptr[b]), st.num_segments(b)
        sets = [OC.head_top_k(q[b, h], mk32[s0:s0 + n, h // G], int(st.topk[b])) for h in range(sp.num_q_heads)]
        want, _, _, _ = OC.consensus(sets, n, int(st.consensus[b]))
        assert votes[b, :n].tolist() == want.tolist(), b
    plan.close()


def test_non_finite_summary_key_sets_bit_3_and_nothing_faults():
    spec = W.small_spec(dtype="bf16", head_dim=128, batch=2, num_q_heads=8, num_kv_heads=2, seq_len=300,
                        seg_len_range=(10, 30), topk=3, window=5, seed=8)
    st, lt = _layer(spec)
    lt.sum_k[int(st.seg_ptr[1]) + 2, 1, 7] = float("nan")
    lt.sum_k[int(st.seg_ptr[1]) + 4, 1, 9] = float("inf")
    plan = Z.DecodePlan.from_structure(st)
    out, _ = C.run_gpu(plan, lt, C.device_tables(st), debug=False)
    torch.cuda.synchronize()
    assert plan.device_error() == 4
    # units without the bad values are unaffected
    res = O.decode_step(**oracle_args(st, lt), units=[(0, 0), (0, 1)])
    C.check_outputs(res, out.cpu().numpy(), [(0, 0), (0, 1)], 4, C.TOL["bf16"])
