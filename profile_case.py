"""Run one layer of a workload through the C ABI a few times (for profilers).

  python profile_case.py --workload 2 --layer 0 --reps 4
  python profile_case.py --path summaries --segments 8 --reps 3

Draws the workload's structure and one layer on cuda:0. The decode path plans
the layer and runs the decode step ``--reps`` times; the summaries path runs
``zr_segment_summaries`` over the layer's first ``--segments`` segments (0: all
of them) ``--reps`` times. Both check the device error word, print what one call
covers and exit 0 on success; they time nothing.
"""

from __future__ import annotations

import argparse
import sys

import numpy as np
import torch

from hierarchical_sparse_kv_gb300 import workloads as W
from hierarchical_sparse_kv_gb300 import zoomr as Z


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--layer", type=int, default=0)
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--path", choices=["decode", "summaries"], default="decode")
    ap.add_argument("--segments", type=int, default=0, help="summaries path: first N segments (0: all)")
    args = ap.parse_args(argv)
    Z.load()
    spec = W.WORKLOADS[args.workload]
    st = W.make_structure(spec)
    lt = W.make_layer(st, args.layer, "cuda")
    if args.path == "summaries":
        return run_summaries(st, lt, args)
    plan = Z.DecodePlan.from_structure(st)
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    out = torch.empty(lt.q.shape, dtype=torch.float32, device="cuda")
    dbg = plan.new_debug_outputs()
    for _ in range(args.reps):
        plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, out, dbg)
    torch.cuda.synchronize()
    err = plan.device_error()
    _, rng, nr = (x.cpu().numpy() for x in dbg)
    rows = sum(int(e - s) for b in range(st.batch) for g in range(spec.num_kv_heads)
               for s, e in rng[b, g, :nr[b, g]])
    print(f"workload {args.workload} ({spec.name}) layer {args.layer}: {args.reps} calls, "
          f"{rows} gathered tokens per call, device error {err}")
    plan.close()
    return 0 if err == 0 else 1


def run_summaries(st: W.Structure, lt: W.LayerTensors, args) -> int:
    spec = st.spec
    segs = []
    for b in range(st.batch):
        bnd = st.bounds(b)
        segs += [(b, int(bnd[i]), int(bnd[i + 1]), int(st.seg_ptr[b]) + i) for i in range(len(bnd) - 1)]
    if args.segments > 0:
        segs = segs[:args.segments]
    cfg = Z.cache_config(batch=st.batch, num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                         num_blocks=st.num_blocks, max_blocks_per_seq=st.max_blocks_per_seq, dtype=spec.dtype)
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).cuda()
    sg = torch.tensor(segs, dtype=torch.int32, device="cuda")
    sk, sv = torch.empty_like(lt.sum_k), torch.empty_like(lt.sum_v)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(args.reps):
        Z.zr_segment_summaries(cfg, sg, bt, lt.k_pool, lt.v_pool, sk, sv, err)
    torch.cuda.synchronize()
    e = int(err.item())
    print(f"workload {args.workload} ({spec.name}) layer {args.layer}: {args.reps} summary calls over "
          f"{len(segs)} segments ({sum(t1 - t0 for _, t0, t1, _ in segs)} tokens), device error {e}")
    return 0 if e == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
