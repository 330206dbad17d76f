"""Run one layer of a workload through the C ABI a few times (for profilers).

  python -m hierarchical_sparse_kv_gb300.profile_case --workload 2 --layer 0 --reps 4

Draws the workload's structure and one layer on cuda:0, plans it, runs the
decode step ``--reps`` times on the current stream and checks the device error
word. It prints the per-call gathered-row count and exits 0; it times nothing.
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
    args = ap.parse_args(argv)
    Z.load()
    spec = W.WORKLOADS[args.workload]
    st = W.make_structure(spec)
    lt = W.make_layer(st, args.layer, "cuda")
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


if __name__ == "__main__":
    sys.exit(main())
