"""Benchmark: ZoomR decode steps/s on the 8B shape at 16K context, batch 8, 32 layers.

One step = the whole hot path (summary score -> top-k -> paged gather ->
attention -> merge) for all 32 layers of one decode step, each layer with its
own K/V pool, summaries and queries (Llama-3.1-8B attention: 32 query / 8 KV
heads, d = 128, bf16; 16-token blocks in a shuffled pool; segments U[64, 512];
top-k 16; window 256). Inputs are seeded synthetic data resident in HBM; one
step reads ~5.1 GB, far more than the 129 MB L2, so no flush is needed between
steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl zoomr|reference]
  python bench.py --path append      # the cache-update path: token appends and segment summaries
  python bench.py --path consensus   # ZoomR's consensus selection and attention over its final set
  python bench.py --path offload     # the consensus decode with the cache in pinned host memory, staged per layer
  python bench.py --path generate    # the consensus path as a decode loop (appends, advance, periodic selection)

Prints one JSON line (rank 0). Under torchrun each rank runs its own replica of
the workload on its own GPU (weak scaling) and the reported time is the max over
ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import statistics
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The CPU oracle legs run single-threaded: cap numpy's BLAS threads before numpy loads.
for _k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_k, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

from hierarchical_sparse_kv_gb300 import accounting as A  # noqa: E402
from hierarchical_sparse_kv_gb300 import workloads as W  # noqa: E402

METRIC = "decode attention steps/s at 8B shape, 16K ctx, batch 8; HBM GB/s vs peak"
WORKLOAD_ID = 2
PEAK_FALLBACK_GBS = 6800.0
KERNEL_SOURCES = ["hierarchical_sparse_kv_gb300/csrc/zoomr_kernels.cu",
                  "hierarchical_sparse_kv_gb300/csrc/zoomr_internal.h"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attend_mma_llama8b_16k_b8.json")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback"


def read_traffic():
    """DRAM bytes per attend launch from the committed ncu summary, if the kernel is unchanged since."""
    try:
        with open(PROFILE_SUMMARY) as f:
            prof = json.load(f)
        if prof.get("kernel_source_hash") == kernel_source_hash():
            return float(prof["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [l.split(",") for l in out.strip().splitlines() if l.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i] and "Not" not in r[5 + i]})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------- inputs
def make_inputs(device, workload=WORKLOAD_ID, layers=None):
    spec = W.WORKLOADS[workload]
    st = W.make_structure(spec)
    nl = spec.layers if layers is None else layers
    lts = [W.make_layer(st, l, device) for l in range(nl)]
    return spec, st, lts


def config_dict(spec, extra=None):
    d = {"workload": spec.name, "batch": spec.batch, "seq_len": spec.seq_len, "layers": spec.layers,
         "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
         "top_k": spec.topk, "window": spec.window, "segment_len": list(spec.seg_len_range), "block_size": 16,
         "l2": "inputs exceed L2 (each step reads ~4.7 GB of K/V; no flush)"}
    if extra:
        d.update(extra)
    return d


# ---------------------------------------------------------------------- oracle timing
def time_oracle(st, lt, budget_s: float, max_units=None):
    """Run the CPU oracle unit by unit on one layer until ``budget_s`` elapses.
    Returns (units done, seconds)."""
    from oracle import zoomr_oracle as O

    q = W.to_numpy32(lt.q)
    kp = W.to_numpy32(lt.k_pool)
    vp = W.to_numpy32(lt.v_pool)
    sk = W.to_numpy32(lt.sum_k)
    sv = W.to_numpy32(lt.sum_v)
    units = [(b, g) for b in range(st.batch) for g in range(st.spec.num_kv_heads)]
    done = 0
    t0 = time.perf_counter()
    while True:  # cycle through the layer's units until the budget (or max_units) is reached
        b, g = units[done % len(units)]
        O.decode_step(q, kp, vp, st.block_tables, st.seg_ptr, st.seg_bounds, sk, sv, st.topk, st.window,
                      units=[(b, g)])
        done += 1
        if (max_units and done >= max_units) or time.perf_counter() - t0 >= budget_s:
            break
    return done, time.perf_counter() - t0


# Worker side of the multi-core oracle timing: the layer's arrays are module globals set before the
# pool forks (copy-on-write), each worker cycles through its own units until the budget is spent.
_ORACLE_ARGS = None


def _oracle_worker(job):
    from oracle import zoomr_oracle as O

    wid, nworkers, budget_s = job
    st, q, kp, vp, sk, sv = _ORACLE_ARGS
    units = [(b, g) for b in range(st.batch) for g in range(st.spec.num_kv_heads)]
    done, t0 = 0, time.perf_counter()
    while True:
        b, g = units[(wid + done * nworkers) % len(units)]
        O.decode_step(q, kp, vp, st.block_tables, st.seg_ptr, st.seg_bounds, sk, sv, st.topk, st.window,
                      units=[(b, g)])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            return done, time.perf_counter() - t0


def cpu_baseline(workload: int, budget_s: float) -> dict:
    """The oracle on the host cores, before any CUDA call (the pool forks): single-threaded for
    ``budget_s`` seconds, then one process per core for ``budget_s`` seconds. Steps/s of each,
    scaled from the (sequence, KV head) units of layer 0 it computed to a full step."""
    global _ORACLE_ARGS
    import multiprocessing as mp

    spec = W.WORKLOADS[workload]
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cpu")
    units_per_step = spec.layers * st.batch * spec.num_kv_heads
    n1, t1 = time_oracle(st, lt, budget_s)
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    _ORACLE_ARGS = (st, W.to_numpy32(lt.q), W.to_numpy32(lt.k_pool), W.to_numpy32(lt.v_pool), W.to_numpy32(lt.sum_k),
                    W.to_numpy32(lt.sum_v))
    with mp.get_context("fork").Pool(ncores) as pool:
        res = pool.map(_oracle_worker, [(i, ncores, budget_s) for i in range(ncores)])
    _ORACLE_ARGS = None
    nn = sum(r[0] for r in res)
    tn = max(r[1] for r in res)
    v1 = n1 / t1 / units_per_step
    vn = nn / tn / units_per_step
    return {"value": vn, "unit": "steps/s", "cores": ncores, "kind": "oracle", "value_1core": v1,
            "sample": f"{nn} (sequence, KV head) unit computations of layer 0 in {tn:.1f} s on {ncores} processes "
                      f"({n1} in {t1:.1f} s on one core), cycling over its {st.batch * spec.num_kv_heads} units; "
                      f"a step is {units_per_step} units"}


def cpu_baseline_accounting(st, lts, G: int, eb: int):
    """Part of the CPU-baseline leg: the oracle's selection steps (summary_keys, select_top_k,
    gather_set) on host copies of the very queries and summary keys the GPU reads, for every unit of
    every layer, outside any timed region. Returns (algorithmic attend bytes per layer, tokens gathered
    per step, {(layer, b, g): token ranges}) for the byte accounting of the roofline."""
    from oracle import zoomr_oracle as O

    spec = st.spec
    per_layer, tok_total, ranges = [], 0, {}
    for l, lt in enumerate(lts):
        q = W.to_numpy32(lt.q)
        sk = W.to_numpy32(lt.sum_k)
        tot = 0
        for b in range(st.batch):
            s0, n = int(st.seg_ptr[b]), st.num_segments(b)
            bounds = np.asarray(st.bounds(b))
            L_b = int(st.seq_lens[b])
            for g in range(spec.num_kv_heads):
                keys = O.summary_keys(q[b, g * G:(g + 1) * G], sk[s0:s0 + n, g])
                sel = O.select_top_k(keys, int(st.topk[b]))
                tokens, summaries = O.gather_set(bounds, sel, L_b, st.window)
                tok_total += len(tokens)
                ranges[(l, b, g)] = O.token_ranges(tokens)
                tot += A.attend_bytes_per_unit(len(tokens), len(summaries), A.distinct_blocks(tokens), G,
                                               spec.head_dim, eb)
        per_layer.append(tot)
    return per_layer, tok_total, ranges


# ---------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------- reference arm
def _oracle_units(job):
    """Reference-arm worker: the oracle on units [i0, i1) of the layer in _ORACLE_ARGS."""
    from oracle import zoomr_oracle as O

    i0, i1 = job
    st, q, kp, vp, sk, sv = _ORACLE_ARGS
    units = [(b, g) for b in range(st.batch) for g in range(st.spec.num_kv_heads)]
    O.decode_step(q, kp, vp, st.block_tables, st.seg_ptr, st.seg_bounds, sk, sv, st.topk, st.window,
                  units=units[i0:i1])
    return i1 - i0


def run_reference(args):
    """The oracle as the reference arm, on the host cores: every timed step is a bounded sample of the
    workload, all (sequence, KV head) units of one layer, computed by one process per core. The layer's
    inputs are drawn on the CPU and the pool forks before any CUDA call. ms_per_step is that sampled
    step's measured time; value scales it to full steps of every layer."""
    global _ORACLE_ARGS
    import multiprocessing as mp

    world, rank, local = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    spec = W.WORKLOADS[args.workload]
    st = W.make_structure(spec)
    lt = W.make_layer(st, 0, "cpu")
    U = st.batch * spec.num_kv_heads
    ncores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    nproc = max(1, min(ncores, U))
    _ORACLE_ARGS = (st, W.to_numpy32(lt.q), W.to_numpy32(lt.k_pool), W.to_numpy32(lt.v_pool),
                    W.to_numpy32(lt.sum_k), W.to_numpy32(lt.sum_v))
    jobs = [(U * i // nproc, U * (i + 1) // nproc) for i in range(nproc)]
    times = []
    with mp.get_context("fork").Pool(nproc) as pool:
        for i in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            done = sum(pool.map(_oracle_units, jobs))
            assert done == U
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
    _ORACLE_ARGS = None
    ms_sample = 1e3 * sum(times) / len(times)
    value = 1e3 / (ms_sample * spec.layers)  # full steps (every layer) per second
    sample = (f"each timed step: the {U} (sequence, KV head) units of one layer (1/{spec.layers} of a full "
              f"step) on {nproc} processes; value = 1 / ({spec.layers} x the measured time of such a step)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_sample,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": config_dict(spec),
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": nproc, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- our arm
def run_zoomr(args):
    # the CPU baseline forks its process pool, so it runs before anything touches CUDA
    solo = int(os.environ.get("WORLD_SIZE", "1")) == 1
    cpu_line = cpu_baseline(args.workload, args.cpu_budget) if solo and not args.no_cpu_baseline else None
    world, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the ZoomR path needs a CUDA GPU")
    from hierarchical_sparse_kv_gb300 import build as B
    from hierarchical_sparse_kv_gb300 import zoomr as Z

    if rank == 0 or world == 1:
        B.build()
    barrier(world)
    Z.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    spec, st, lts = make_inputs(dev, args.workload)
    L = len(lts)
    plan = Z.DecodePlan.from_structure(st, device=dev).set_deterministic(args.deterministic)
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).to(dev)
    # every layer's queries and outputs are slices of one buffer each, so the end-to-end leg moves a
    # step's inputs and results with one copy per direction
    q_all = torch.stack([lt.q for lt in lts])
    for l, lt in enumerate(lts):
        lt.q = q_all[l]
    out_all = torch.empty((len(lts),) + tuple(q_all.shape[1:]), dtype=torch.float32, device=dev)
    outs = [out_all[l] for l in range(len(lts))]
    G = spec.num_q_heads // spec.num_kv_heads

    # Algorithmic bytes of each layer's attend launch. The CPU-baseline leg runs the oracle's selection
    # steps on the very inputs the GPU reads; the kernel's own ranges (debug outputs) must agree with it
    # on every unit, and give the count only when that leg is skipped.
    dbg = plan.new_debug_outputs()
    kern_bytes, select_bytes, kern_tok, kern_ranges = [], 0, 0, {}
    eb = 2 if spec.dtype == "bf16" else 4  # element bytes of q, K/V and summaries
    for l, lt in enumerate(lts):
        plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, outs[l], dbg)
        _, rng, nr = (x.cpu().numpy() for x in dbg)
        tot = 0
        for b in range(st.batch):
            n_b = st.num_segments(b)
            k_b = min(int(st.topk[b]), n_b)
            for g in range(spec.num_kv_heads):
                r = rng[b, g, :nr[b, g]]
                kern_ranges[(l, b, g)] = r
                ntok = A.ranges_token_count(r)
                kern_tok += ntok
                tot += A.attend_bytes_per_unit(ntok, n_b - k_b, A.ranges_block_count(r), G, spec.head_dim, eb)
                select_bytes += A.select_bytes_per_unit(n_b, G, spec.head_dim, eb)
        kern_bytes.append(tot)
    torch.cuda.synchronize()
    assert plan.device_error() == 0
    if cpu_line is not None and not args.no_oracle_accounting:
        t_acc = time.perf_counter()
        attend_bytes, tok_total, oracle_ranges = cpu_baseline_accounting(st, lts, G, eb)
        agree = all(np.array_equal(kern_ranges[key], oracle_ranges[key]) for key in oracle_ranges)
        acct = {"source": "the oracle's selection steps (summary_keys, select_top_k, gather_set) on the GPU's "
                          "inputs, in the CPU-baseline leg", "units": len(oracle_ranges),
                "kernel_ranges_agree": agree, "seconds": round(time.perf_counter() - t_acc, 1)}
    else:
        attend_bytes, tok_total = kern_bytes, kern_tok
        acct = {"source": "the kernel's own token ranges (the CPU-baseline leg was skipped)"}
    out_bytes = L * st.batch * spec.num_q_heads * spec.head_dim * 4
    step_bytes = sum(attend_bytes) + select_bytes + out_bytes

    stream = torch.cuda.Stream(device=dev)

    def step(s, pair=None, sel_att=None, sel_only=None):
        """One decode step over all layers. pair[l]: events around layer l's attend launch; sel_att[l]:
        an event before layer l's call and one after its attend launch; sel_only[l]: an event before the
        call and one after its select launch (the events of a capture become graph nodes)."""
        for l, lt in enumerate(lts):
            if pair is not None:
                plan.run_timed(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, outs[l], pair[l][0], pair[l][1],
                               stream=s)
            elif sel_att is not None:
                sel_att[l][0].record(s)
                plan.run_timed(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, outs[l], None, sel_att[l][1],
                               stream=s)
            elif sel_only is not None:
                sel_only[l][0].record(s)
                plan.run_timed(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, outs[l], sel_only[l][1], None,
                               stream=s)
            else:
                plan.run(lt.q, lt.k_pool, lt.v_pool, bt, lt.sum_k, lt.sum_v, outs[l], stream=s)

    # Events for the measurement steps: plain pairs around each attend launch, and pairs whose first event
    # precedes the call (recorded by us, so inside a capture it must be an "external" event node).
    try:
        ext = lambda: torch.cuda.Event(enable_timing=True, external=True)
        ext()
    except TypeError:
        ext = None
    mk = lambda: torch.cuda.Event(enable_timing=True)
    pair = [(mk(), mk()) for _ in range(L)]
    sel_att = [(ext(), mk()) for _ in range(L)] if ext else None
    sel_only = [(ext(), mk()) for _ in range(L)] if ext else None
    for e_ in [e for p_ in pair + (sel_att or []) + (sel_only or []) for e in p_]:
        e_.record(stream)  # torch creates CUDA events lazily: create them all before any capture
    stream.wait_stream(torch.cuda.current_stream())
    graphs = {}
    with torch.cuda.stream(stream):
        step(stream)  # eager warm-up on the capture stream
        if not args.no_graph:
            for name, kw in (("step", {}), ("pair", {"pair": pair}), ("sel_att", {"sel_att": sel_att}),
                             ("sel_only", {"sel_only": sel_only})):
                if name != "step" and not next(iter(kw.values())):
                    continue
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    step(stream, **kw)
                graphs[name] = g
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()

    def replay(name="step"):
        with torch.cuda.stream(stream):
            if graphs:
                graphs[name].replay()
            else:
                step(stream, **({"pair": pair} if name == "pair" else {"sel_att": sel_att} if name == "sel_att" else
                                {"sel_only": sel_only} if name == "sel_only" else {}))

    for i in range(args.warmup):
        replay()
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.25 if clocks and clocks.proc else 0)
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    t_start.record(stream)
    for i in range(args.steps):
        replay()
    t_stop.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = t_start.elapsed_time(t_stop) / args.steps
    ms = max_over_ranks(ms, world)

    # The attend kernel's duration, after the timed region: an event pair around every layer's attend
    # launch, over `meas_reps` replays of a step (L launches each). Each pair breaks the launch's
    # programmatic overlap with the select kernel and adds the event nodes' latency (an empty kernel
    # between two event nodes measures about 4.4 us), so this direct figure is conservative. Beside it,
    # the kernel's time with the overlap intact: median(select + attend) - median(select), each from an
    # event before the call.
    meas_reps = max(1, -(-args.attend_samples // L))
    pair_ms, pair_bytes, sa, so = [], [], [], []
    for _ in range(meas_reps):
        replay("pair")
        torch.cuda.synchronize()
        pair_ms += [pair[l][0].elapsed_time(pair[l][1]) for l in range(L)]
        pair_bytes += attend_bytes
        if sel_att is not None:
            replay("sel_att")
            torch.cuda.synchronize()
            sa += [sel_att[l][0].elapsed_time(sel_att[l][1]) for l in range(L)]
            replay("sel_only")
            torch.cuda.synchronize()
            so += [sel_only[l][0].elapsed_time(sel_only[l][1]) for l in range(L)]
    attend_ms = sum(pair_ms) / len(pair_ms)  # mean over the sampled launches
    attend_bytes_avg = sum(pair_bytes) / len(pair_bytes)
    in_step = None
    if sa and so:
        in_step_ms = statistics.median(sa) - statistics.median(so)
        mean_bytes = sum(attend_bytes) / L
        in_step = {"attend_us": in_step_ms * 1e3, "achieved": mean_bytes / (in_step_ms * 1e-3) / 1e9,
                   "select_us": statistics.median(so) * 1e3, "select_attend_us": statistics.median(sa) * 1e3,
                   "samples": len(sa)}

    # e2e through the public API with host buffers: one H2D of all layers' queries from pinned
    # memory, the step, one D2H of all layers' outputs into pinned memory.
    host_q = q_all.cpu().pin_memory()
    host_out = torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory()
    h2d = host_q.numel() * host_q.element_size()
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(3, min(args.steps, 50))
    with torch.cuda.stream(stream):
        for _ in range(2):
            q_all.copy_(host_q, non_blocking=True)
            step(stream)
            host_out.copy_(out_all, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            q_all.copy_(host_q, non_blocking=True)
            step(stream)
            host_out.copy_(out_all, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

    peak, peak_kind = read_peak()
    achieved = attend_bytes_avg / (attend_ms * 1e-3) / 1e9
    traffic = read_traffic() if args.workload == WORKLOAD_ID else None
    mma = spec.dtype == "bf16" and G <= 8
    kernel = f"zr_attend_mma_kernel<{spec.head_dim}>" if mma else \
        f"zr_attend_fma_kernel<{'bf16' if spec.dtype == 'bf16' else 'float'}, {spec.head_dim}>"
    l2 = (f"inputs exceed L2 (each step reads ~{step_bytes / 1e9:.2f} GB of K/V; no flush)" if step_bytes > 129e6 else
          f"inputs fit in L2 (each step reads ~{step_bytes / 1e6:.1f} MB; no flush: L2-resident timing)")
    line = {
        "impl": "zoomr", "metric": METRIC, "value": world * 1e3 / ms, "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) K/V, segment-mean summaries + N(0,0.1), queries near segment means)",
        "config": config_dict(spec, {"graph": not args.no_graph, "replicas_per_gpu": 1, "l2": l2,
                                     "split": "even (the decode step always takes the even split of the rows)"}),
        "hbm_gbs": step_bytes / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": traffic,
                     "kernel": kernel, "attend_us": attend_ms * 1e3, "samples": len(pair_ms),
                     "alg_bytes_per_launch": attend_bytes_avg, "alg_bytes": acct,
                     "timing": f"mean over {len(pair_ms)} attend launches ({meas_reps} replays of the step after "
                               "the timed region, every layer), each between two CUDA events on the launching "
                               "stream; the pair breaks the launch's overlap with the select kernel and includes "
                               "the event nodes' latency"},
        "e2e": {"value": world * 1e3 / e2e_ms, "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 3 * L * args.steps,
        "attend_in_step": None if in_step is None else dict(
            in_step, frac=in_step["achieved"] / peak,
            method="median(select+attend) - median(select) over the sampled layers, events before the call and "
                   "after attend or select, launch overlap between the two kernels intact"),
        "timing": "CUDA events on the launching stream around the replays of a captured step (no event nodes "
                  "inside it)",
        "clocks": clk,
        "tokens_gathered_per_step": tok_total,
    }
    if cpu_line is not None:
        line["cpu_baseline"] = cpu_line
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0



def measure_link_gbs(dev) -> float:
    """Pinned-host-to-device copy bandwidth of this machine: a 1 GiB cudaMemcpyAsync, median of 5."""
    src = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dst = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    ts = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    del src, dst
    torch.cuda.empty_cache()
    return (1 << 30) / (float(np.median(ts)) * 1e-3) / 1e9


# ---------------------------------------------------------------------- append path
APPEND_METRIC = ("append-path generation steps/s at 8B shape, 16K ctx, batch 8, 32 layers (every sequence appends "
                 "a token and closes a segment); HBM GB/s of the summary kernel vs peak")


def append_step_plan(st):
    """One generation step of the cache: every sequence appends its next token (a spare block when its last
    one is full) and closes its last segment with it. Returns (block tables with one spare column, positions,
    closing segments as (b, start, end, output row b))."""
    B = st.batch
    tables = np.concatenate([st.block_tables, np.full((B, 1), -1, np.int32)], axis=1)
    used = set(int(x) for x in st.block_tables.ravel() if x >= 0)
    free = [x for x in range(st.num_blocks) if x not in used]
    pos = st.seq_lens.astype(np.int32).copy()
    segs = []
    for b in range(B):
        t = int(pos[b])
        if tables[b, t // 16] < 0:
            tables[b, t // 16] = free.pop(0)
        segs.append((b, int(st.bounds(b)[-2]), t + 1, b))
    return tables, pos, np.array(segs, dtype=np.int32)


def append_cpu_baseline(spec, budget_s: float, layers: int) -> dict:
    """The append-path oracle (one core) on layer 0 of one generation step, repeated for ``budget_s``."""
    from oracle import zoomr_append as OA

    st = W.make_structure(spec, spare_blocks=spec.batch)
    tables, pos, segs = append_step_plan(st)
    lt = W.make_layer(st, 0, "cpu")
    kp, vp = W.to_numpy32(lt.k_pool), W.to_numpy32(lt.v_pool)
    rng = np.random.default_rng(5)
    kn = rng.standard_normal((st.batch, spec.num_kv_heads, spec.head_dim)).astype(np.float32)
    vn = rng.standard_normal((st.batch, spec.num_kv_heads, spec.head_dim)).astype(np.float32)
    done, t0 = 0, time.perf_counter()
    while True:
        k2, v2 = OA.append_kv(kp, vp, tables, pos, kn, vn)
        OA.segment_summaries(k2, v2, tables, [tuple(x) for x in segs], spec.dtype, st.batch)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    t = time.perf_counter() - t0
    return {"value": done / t / layers, "unit": "steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} layer updates (append 8 tokens, 8 closing-segment summaries) of layer 0 in {t:.1f} s, "
                      f"scaled to a {layers}-layer step"}


def run_append(args):
    """Times one generation step of the append path (every layer: zr_append_kv, then zr_segment_summaries of
    the segments the new tokens close), replayed as a CUDA graph; also times the summary kernel alone."""
    spec = W.WORKLOADS[WORKLOAD_ID]
    solo = int(os.environ.get("WORLD_SIZE", "1")) == 1
    layers = spec.layers if args.layers is None else max(1, min(args.layers, spec.layers))
    cpu_line = append_cpu_baseline(spec, args.cpu_budget, layers) if solo and not args.no_cpu_baseline else None
    world, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the append path needs a CUDA GPU")
    from hierarchical_sparse_kv_gb300 import build as B
    from hierarchical_sparse_kv_gb300 import zoomr as Z

    if rank == 0 or world == 1:
        B.build()
    barrier(world)
    Z.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    st = W.make_structure(spec, spare_blocks=spec.batch)
    tables, pos, segs = append_step_plan(st)
    L = spec.layers if args.layers is None else max(1, min(args.layers, spec.layers))
    Bn, H, d = st.batch, spec.num_kv_heads, spec.head_dim
    eb = 2 if spec.dtype == "bf16" else 4
    lts = [W.make_layer(st, l, dev) for l in range(L)]
    cfg = Z.cache_config(batch=Bn, num_kv_heads=H, head_dim=d, num_blocks=st.num_blocks,
                         max_blocks_per_seq=tables.shape[1], dtype=spec.dtype)
    bt = torch.from_numpy(tables).to(dev)
    pos_d = torch.from_numpy(pos).to(dev)
    segs_d = torch.from_numpy(segs).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(spec.seed)
    dt = W.torch_dtype(spec.dtype)
    kn_all = torch.randn((L, Bn, H, d), generator=gen, device=dev).to(dt)
    vn_all = torch.randn((L, Bn, H, d), generator=gen, device=dev).to(dt)
    rows_all = torch.empty((2, L, Bn, H, d), dtype=dt, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(kind, s):
        for l, lt in enumerate(lts):
            if kind in ("full", "append"):
                Z.zr_append_kv(cfg, pos_d, kn_all[l], vn_all[l], bt, lt.k_pool, lt.v_pool, err, stream=s)
            if kind in ("full", "summaries"):
                Z.zr_segment_summaries(cfg, segs_d, bt, lt.k_pool, lt.v_pool, rows_all[0, l], rows_all[1, l], err,
                                       stream=s)

    kinds = ("full", "append", "summaries")
    graphs = {}
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step("full", stream)  # eager warm-up (also sets the summary kernel's shared-memory attribute)
        for k in kinds:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(k, stream)
            graphs[k] = g
    torch.cuda.synchronize()

    def timed(kind, steps, sampler=None):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                graphs[kind].replay()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(steps):
                graphs[kind].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1) / steps, world)

    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.25 if clocks and clocks.proc else 0)
    ms = timed("full", args.steps)
    clk = clocks.stop() if clocks else None
    ms_append = timed("append", args.steps)
    ms_sums = timed("summaries", args.steps)
    assert int(err.item()) == 0, "device error word set"

    # bulk: every segment of layer 0 (the whole 16K-token cache of each sequence)
    segs_all = []
    for b in range(Bn):
        bnd = st.bounds(b)
        segs_all += [(b, int(bnd[i]), int(bnd[i + 1]), int(st.seg_ptr[b]) + i) for i in range(len(bnd) - 1)]
    segs_all_d = torch.tensor(segs_all, dtype=torch.int32, device=dev)
    bulk_k = torch.empty((len(segs_all), H, d), dtype=dt, device=dev)
    bulk_v = torch.empty_like(bulk_k)
    bulk_ms = []
    for i in range(3 + 20):
        l = i % L  # rotate over the layers' pools (each far larger than L2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        Z.zr_segment_summaries(cfg, segs_all_d, bt, lts[l].k_pool, lts[l].v_pool, bulk_k, bulk_v, err, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            bulk_ms.append(e0.elapsed_time(e1))
    bulk_t = float(np.median(bulk_ms))
    bulk_bytes = sum(e - s for _, s, e, _ in segs_all) * H * d * eb * 2 + len(segs_all) * H * d * eb * 2

    # e2e: each step's new K/V rows from pinned host memory, the step, the new summary rows back to the host
    host_new = torch.stack([kn_all, vn_all]).cpu().pin_memory()
    dev_new = torch.stack([kn_all, vn_all])
    host_rows = torch.empty(rows_all.shape, dtype=dt).pin_memory()
    kn_all, vn_all = dev_new[0], dev_new[1]  # the graphs read the old buffers: re-capture on the new ones

    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step("full", stream)
    e2e_steps = max(3, min(args.steps, 50))
    with torch.cuda.stream(stream):
        for _ in range(2):
            dev_new.copy_(host_new, non_blocking=True)
            g.replay()
            host_rows.copy_(rows_all, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            dev_new.copy_(host_new, non_blocking=True)
            g.replay()
            host_rows.copy_(rows_all, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

    peak, peak_kind = read_peak()
    sum_bytes = int(sum(int(e) - int(s) for _, s, e, _ in segs)) * H * d * eb * 2 + Bn * H * d * eb * 2
    sum_us = ms_sums * 1e3 / L
    achieved = sum_bytes / (sum_us * 1e-6) / 1e9
    line = {
        "impl": "zoomr", "path": "append", "metric": APPEND_METRIC, "value": world * 1e3 / ms, "unit": "steps/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) K/V cache, new rows N(0,1))",
        "config": {"workload": spec.name + "_append" + ("" if L == spec.layers else f"_first{L}layers"), "batch": Bn,
                   "seq_len": spec.seq_len, "layers": L,
                   "kv_heads": H, "head_dim": d, "block_size": 16,
                   "closing_segment_tokens": [int(e) - int(s) for _, s, e, _ in segs],
                   "graph": True, "l2": "each step touches 32 layers' pools (far beyond L2); no flush"},
        "append_us_per_layer": ms_append * 1e3 / L, "summaries_us_per_layer": sum_us,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                     "kernel": f"zr_summaries_exact_kernel<{d}>", "alg_bytes_per_launch": sum_bytes,
                     "timing": "summaries-only graph of 32 launches, time / 32 (latency-bound: 8 segments per launch)"},
        "bulk_summaries": {"segments": len(segs_all), "ms": bulk_t, "alg_bytes": bulk_bytes,
                           "achieved_gbs": bulk_bytes / (bulk_t * 1e-3) / 1e9,
                           "frac": bulk_bytes / (bulk_t * 1e-3) / 1e9 / peak,
                           "timing": "median of 20 single launches, event pair, layers rotated"},
        "e2e": {"value": world * 1e3 / e2e_ms, "unit": "steps/s",
                "h2d_bytes_per_step": host_new.numel() * host_new.element_size(),
                "d2h_bytes_per_step": host_rows.numel() * host_rows.element_size()},
        "gpu_launches": 2 * L * args.steps,
        "clocks": clk,
    }
    if cpu_line is not None:
        line["cpu_baseline"] = cpu_line
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------- consensus path
CONSENSUS_METRIC = ("consensus decode steps/s at 8B shape, 512-token prompt + 16K generated, batch 8, 32 layers "
                    "(one selection per 35 steps); HBM GB/s of the gather-attention kernel vs peak")
SELECTION_INTERVAL = 35  # mean tokens between semantic boundaries (ZoomR appendix A.3)


def consensus_cpu_baseline(spec, budget_s: float) -> dict:
    """The consensus oracle (one core) on sequence 0: the votes of every layer and one layer's attention."""
    from oracle import zoomr_append as OA
    from oracle import zoomr_consensus as OC

    st = W.make_consensus_structure(spec)
    lt = W.make_consensus_layer(st, 0, "cpu")
    kp, vp, q = W.to_numpy32(lt.k_pool), W.to_numpy32(lt.v_pool), W.to_numpy32(lt.q)
    s0, s1 = int(st.seg_ptr[0]), int(st.seg_ptr[1])
    kbar = np.zeros((st.total_segments, spec.num_kv_heads, spec.head_dim), np.float32)
    for i, (s, e) in enumerate(st.summary_spans(0)):
        for g in range(spec.num_kv_heads):
            kbar[s0 + i, g] = OA.round_to_dtype(OA.segment_mean(kp, st.block_tables[0], g, s, e), spec.dtype)
    done, t0 = 0, time.perf_counter()
    while True:  # layer 0's inputs stand in for every layer: the work per layer is the same
        OC.consensus_step([q] * spec.layers, [kbar] * spec.layers, [kp], [vp], st.block_tables, st.seg_ptr,
                          st.seg_bounds, st.prompt_lens, st.seq_lens, st.topk, st.consensus, st.window,
                          attend_layers=[0], batch=[0])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    t = time.perf_counter() - t0
    per_seq_step = t / done  # votes of all layers + one layer's attention, one sequence
    # a selection step is that plus (layers - 1) more attention layers; attention dominates the rest
    t_att0 = time.perf_counter()
    OC.consensus_step([q], [kbar], [kp], [vp], st.block_tables, st.seg_ptr, st.seg_bounds, st.prompt_lens,
                      st.seq_lens, st.topk, st.consensus, st.window, attend_layers=[0], batch=[0])
    t_att = time.perf_counter() - t_att0
    step_s = st.batch * (per_seq_step + (spec.layers - 1) * t_att)
    return {"value": 1.0 / step_s, "unit": "steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} runs of sequence 0's votes over {spec.layers} layers and one layer's attention in "
                      f"{t:.1f} s, plus one single-layer run; scaled to {st.batch} sequences and "
                      f"{spec.layers} attention layers (every step treated as a selection step)"}


def run_consensus(args):
    """Times ZoomR's consensus decode on the device: a selection step (votes of every layer, one consensus,
    every layer's attention), an attention-only step (I_f reused between semantic boundaries) and the
    selection part alone, each replayed as a CUDA graph."""
    spec = W.CONSENSUS_WORKLOADS[1]
    solo = int(os.environ.get("WORLD_SIZE", "1")) == 1
    cpu_line = consensus_cpu_baseline(spec, args.cpu_budget) if solo and not args.no_cpu_baseline else None
    world, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the consensus path needs a CUDA GPU")
    from hierarchical_sparse_kv_gb300 import build as B
    from hierarchical_sparse_kv_gb300 import zoomr as Z

    if rank == 0 or world == 1:
        B.build()
    barrier(world)
    Z.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    st = W.make_consensus_structure(spec)
    L = spec.layers if args.layers is None else max(1, min(args.layers, spec.layers))
    Bn, H, Hq, d = st.batch, spec.num_kv_heads, spec.num_q_heads, spec.head_dim
    G = Hq // H
    eb = 2 if spec.dtype == "bf16" else 4
    lts = [W.make_consensus_layer(st, l, dev) for l in range(L)]
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).to(dev)
    # mean summary keys of every layer (zr_segment_summaries over the summary spans)
    cfg = Z.cache_config(batch=Bn, num_kv_heads=H, head_dim=d, num_blocks=st.num_blocks,
                         max_blocks_per_seq=st.max_blocks_per_seq, dtype=spec.dtype)
    segs = torch.tensor([(b, s, e, int(st.seg_ptr[b]) + i) for b in range(Bn)
                         for i, (s, e) in enumerate(st.summary_spans(b))], dtype=torch.int32, device=dev)
    dt = W.torch_dtype(spec.dtype)
    mks = []
    for lt in lts:
        mk = torch.empty((st.total_segments, H, d), dtype=dt, device=dev)
        Z.zr_segment_summaries(cfg, segs, bt, lt.k_pool, lt.v_pool, mk, torch.empty_like(mk))
        mks.append(mk)
    plan = Z.ConsensusPlan.from_structure(st, device=dev).set_deterministic(args.deterministic)
    q_all = torch.stack([lt.q for lt in lts])
    for l, lt in enumerate(lts):
        lt.q = q_all[l]
    out_all = torch.empty((L, Bn, Hq, d), dtype=torch.float32, device=dev)
    dbg = plan.new_debug_outputs()
    for l in range(L):
        plan.vote(lts[l].q, mks[l])
    plan.select(dbg)
    torch.cuda.synchronize()
    _, _, rng, nr = (x.cpu().numpy() for x in dbg)
    tok = [A.ranges_token_count(rng[b, :nr[b]]) for b in range(Bn)]
    attend_bytes = sum(A.attend_bytes_per_unit(tok[b], 0, A.ranges_block_count(rng[b, :nr[b]]), G, d, eb) * H
                       for b in range(Bn)) + Bn * Hq * d * 4
    stream = torch.cuda.Stream(device=dev)
    pair = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
    for e_ in [e for p_ in pair for e in p_]:
        e_.record(stream)  # torch creates CUDA events lazily: create them all before any capture

    def step(kind, s):
        if kind in ("select", "full"):
            for l in range(L):
                plan.vote(lts[l].q, mks[l], stream=s)
            plan.select(stream=s)
        if kind in ("attend", "full"):
            for l in range(L):
                plan.attend(lts[l].q, lts[l].k_pool, lts[l].v_pool, bt, out_all[l], stream=s)
        if kind == "pair":  # an event pair around every layer's gather-attention kernel
            for l in range(L):
                plan.attend_timed(lts[l].q, lts[l].k_pool, lts[l].v_pool, bt, out_all[l], pair[l][0], pair[l][1],
                                  stream=s)

    graphs = {}
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step("full", stream)
        for k in ("full", "attend", "select", "pair"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(k, stream)
            graphs[k] = g
    torch.cuda.synchronize()

    def timed(kind, steps):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                graphs[kind].replay()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(steps):
                graphs[kind].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1) / steps, world)

    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.25 if clocks and clocks.proc else 0)
    ms_attend = timed("attend", args.steps)
    ms_full = timed("full", args.steps)
    clk = clocks.stop() if clocks else None
    ms_select = timed("select", args.steps)
    pair_ms = []
    for _ in range(max(1, -(-args.attend_samples // L))):
        with torch.cuda.stream(stream):
            graphs["pair"].replay()
        torch.cuda.synchronize()
        pair_ms += [pair[l][0].elapsed_time(pair[l][1]) for l in range(L)]
    assert plan.device_error() == 0, "device error word set"
    # one selection step every SELECTION_INTERVAL steps, attention-only steps in between
    ms_mixed = (ms_full + (SELECTION_INTERVAL - 1) * ms_attend) / SELECTION_INTERVAL

    # e2e: every step's queries from pinned host memory, the step, every layer's output back
    host_q = q_all.cpu().pin_memory()
    host_out = torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory()
    e2e_steps = SELECTION_INTERVAL
    with torch.cuda.stream(stream):
        for i in range(2):
            q_all.copy_(host_q, non_blocking=True)
            graphs["full" if i == 0 else "attend"].replay()
            host_out.copy_(out_all, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(e2e_steps):
            q_all.copy_(host_q, non_blocking=True)
            graphs["full" if i == 0 else "attend"].replay()
            host_out.copy_(out_all, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world)

    peak, peak_kind = read_peak()
    layer_us = ms_attend * 1e3 / L  # one layer of the attention-only step: gather-attention + merge + handoffs
    attend_us = sum(pair_ms) / len(pair_ms) * 1e3
    achieved = attend_bytes / (attend_us * 1e-6) / 1e9
    line = {
        "impl": "zoomr", "path": "consensus", "metric": CONSENSUS_METRIC, "value": world * 1e3 / ms_mixed,
        "unit": "steps/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_mixed,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) K/V, queries near one summary segment's mean key)",
        "config": {"split": "even (deterministic plan)" if args.deterministic else "dynamic (attend-only calls)", "workload": spec.name + ("" if L == spec.layers else f"_first{L}layers"), "batch": Bn,
                   "prompt": spec.prompt_len, "generated": spec.gen_len, "layers": L, "q_heads": Hq, "kv_heads": H,
                   "head_dim": d, "top_k": spec.topk, "consensus": spec.consensus, "window": spec.window,
                   "regular_len": list(spec.reg_len_range), "summary_len": list(spec.sum_len_range),
                   "selection_interval": SELECTION_INTERVAL, "graph": True,
                   "l2": "each step reads the 32 layers' final sets (far beyond L2); no flush"},
        "selection_step_ms": ms_full, "attention_step_ms": ms_attend, "selection_part_ms": ms_select,
        "final_set_tokens": tok,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                     "kernel": f"zr_attend_mma_kernel<{d}>", "alg_bytes_per_launch": attend_bytes,
                     "attend_us": attend_us, "samples": len(pair_ms),
                     "timing": f"mean over {len(pair_ms)} gather-attention launches (every layer of replayed "
                               "attention-only steps), each between two CUDA events on the launching stream (the "
                               "pair includes the event nodes' latency)",
                     "per_layer_of_step": {"us": layer_us, "achieved": attend_bytes / (layer_us * 1e-6) / 1e9,
                                           "frac": attend_bytes / (layer_us * 1e-6) / 1e9 / peak,
                                           "timing": "attention-only graph of 32 layers (gather-attention + merge "
                                                     "+ handoffs), time / 32"}},
        "e2e": {"value": world * 1e3 / e2e_ms, "unit": "steps/s", "h2d_bytes_per_step": host_q.numel() * eb,
                "d2h_bytes_per_step": host_out.numel() * 4},
        "gpu_launches": int(round(args.steps * (2 * L + (L + 1) / SELECTION_INTERVAL))),
        "clocks": clk,
    }
    if cpu_line is not None:
        line["cpu_baseline"] = cpu_line
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------- offloaded cache, staged per layer
OFFLOAD_METRIC = ("ZoomR decode steps/s, 512-token prompt + 16K generated, batch 8, 32 layers, every layer's K/V in "
                  "pinned host memory: per layer the final context's rows are staged into HBM over the CPU-GPU link "
                  "(the next layer's while the current one attends); link GB/s vs the measured copy bandwidth")


def run_offload(args):
    """The pages' offloaded decode (ZoomR 3.4, "Decoding Stage"): the cache in host memory; per step the
    blocks of the consensus path's final context I_f are mapped to staging slots once (with the rows each
    KV head needs), and every layer's rows of I_f are staged into one of two HBM staging pools on a copy
    stream while the previous layer attends. Selection held fixed (a step between semantic boundaries)."""
    spec = W.CONSENSUS_WORKLOADS[1]
    world, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the offload path needs a CUDA GPU")
    from hierarchical_sparse_kv_gb300 import build as B
    from hierarchical_sparse_kv_gb300 import zoomr as Z

    if rank == 0 or world == 1:
        B.build()
    barrier(world)
    Z.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    st = W.make_consensus_structure(spec)
    L = spec.layers if args.layers is None else max(1, min(args.layers, spec.layers))
    Bn, H, Hq, d = st.batch, spec.num_kv_heads, spec.num_q_heads, spec.head_dim
    G = Hq // H
    eb = 2 if spec.dtype == "bf16" else 4
    dt = W.torch_dtype(spec.dtype)
    bt = torch.from_numpy(st.block_tables.astype(np.int32)).to(dev)
    cfg = Z.cache_config(batch=Bn, num_kv_heads=H, head_dim=d, num_blocks=st.num_blocks,
                         max_blocks_per_seq=st.max_blocks_per_seq, dtype=spec.dtype)
    segs = torch.tensor([(b, s, e, int(st.seg_ptr[b]) + i) for b in range(Bn)
                         for i, (s, e) in enumerate(st.summary_spans(b))], dtype=torch.int32, device=dev)
    lts, mks, host = [], [], []
    for l in range(L):  # draw on the device, keep the mean keys and queries there, move the pools out
        lt = W.make_consensus_layer(st, l, dev)
        mk = torch.empty((st.total_segments, H, d), dtype=dt, device=dev)
        Z.zr_segment_summaries(cfg, segs, bt, lt.k_pool, lt.v_pool, mk, torch.empty_like(mk))
        mks.append(mk)
        host.append((lt.k_pool.cpu().pin_memory(), lt.v_pool.cpu().pin_memory()))
        lt.k_pool = lt.v_pool = None
        lts.append(lt)
        torch.cuda.empty_cache()
    link_gbs = measure_link_gbs(dev)
    plan = Z.ConsensusPlan.from_structure(st, device=dev).set_deterministic(args.deterministic)
    q_all = torch.stack([lt.q for lt in lts])
    for l, lt in enumerate(lts):
        lt.q = q_all[l]
    out_all = torch.empty((L, Bn, Hq, d), dtype=torch.float32, device=dev)
    dbg = plan.new_debug_outputs()
    for l in range(L):
        plan.vote(lts[l].q, mks[l])
    plan.select(dbg)
    torch.cuda.synchronize()
    _, _, rng, nr = (x.cpu().numpy() for x in dbg)
    need, need_rows = set(), set()
    for b in range(Bn):
        for s_, e_ in rng[b, :nr[b]]:
            need.update(int(st.block_tables[b, j]) for j in range(int(s_) // 16, (int(e_) - 1) // 16 + 1))
            need_rows.update((int(st.block_tables[b, t // 16]), t % 16) for t in range(int(s_), int(e_)))
    cap = len(need)
    stage_ids = torch.zeros(cap, dtype=torch.int32, device=dev)
    remap = torch.empty_like(bt)
    n_staged = torch.zeros(1, dtype=torch.int32, device=dev)
    bufs = [(torch.empty((cap, H, 16, d), dtype=dt, device=dev), torch.empty((cap, H, 16, d), dtype=dt, device=dev))
            for _ in range(2)]
    # K and V of every staged row (the rows of I_f, every KV head: the map's row masks), every layer
    staged_bytes = 2 * len(need_rows) * H * d * eb * L
    tok = [A.ranges_token_count(rng[b, :nr[b]]) for b in range(Bn)]
    attend_bytes = sum(A.attend_bytes_per_unit(tok[b], 0, A.ranges_block_count(rng[b, :nr[b]]), G, d, eb) * H
                       for b in range(Bn)) + Bn * Hq * d * 4
    # the attention on a higher-priority stream: its CTAs are placed before further staging-copy CTAs
    lo_prio, hi_prio = torch.cuda.Stream.priority_range() if hasattr(torch.cuda.Stream, "priority_range") else (0, -1)
    stream, copy = torch.cuda.Stream(device=dev, priority=hi_prio), torch.cuda.Stream(device=dev, priority=lo_prio)
    ev_staged = [torch.cuda.Event() for _ in range(L)]
    ev_freed = [torch.cuda.Event() for _ in range(L)]
    ev_mapped = torch.cuda.Event()

    def step(kind, s):
        """kind: "full" (map, then per layer stage + attend, two streams), "stage" (map + the copies only),
        "attend" (the attention over the staged pools only), "zero_copy" (the attention reading the host
        pools in place, the previous design)."""
        if kind == "zero_copy":
            for l in range(L):
                plan.attend(lts[l].q, host[l][0], host[l][1], bt, out_all[l], stream=s)
            return
        if kind == "attend":
            for l in range(L):
                plan.attend(lts[l].q, bufs[l % 2][0], bufs[l % 2][1], remap, out_all[l], stream=s)
            return
        Z.zr_offload_map(plan.handle, plan.ws, bt, cap, stage_ids, remap, n_staged, stream=s)
        if kind == "stage":
            for l in range(L):
                Z.zr_offload_stage(plan.handle, plan.ws, host[l][0], host[l][1], stage_ids, n_staged, cap, bufs[l % 2][0],
                                   bufs[l % 2][1], stream=s)
            return
        ev_mapped.record(s)
        copy.wait_event(ev_mapped)
        for l in range(L):
            if l >= 2:
                copy.wait_event(ev_freed[l - 2])  # staging pool l % 2 is free once layer l - 2 has attended
            Z.zr_offload_stage(plan.handle, plan.ws, host[l][0], host[l][1], stage_ids, n_staged, cap, bufs[l % 2][0],
                               bufs[l % 2][1], stream=copy)
            ev_staged[l].record(copy)
            s.wait_event(ev_staged[l])
            plan.attend(lts[l].q, bufs[l % 2][0], bufs[l % 2][1], remap, out_all[l], stream=s)
            ev_freed[l].record(s)

    graphs = {}
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        step("full", stream)
        for k in ("full", "stage", "attend", "zero_copy"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(k, stream)
            graphs[k] = g
    torch.cuda.synchronize()
    assert plan.device_error() == 0, "device error word set"

    def timed(kind, steps):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                graphs[kind].replay()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(steps):
                graphs[kind].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1) / steps, world)

    steps = max(3, min(args.steps, 20))  # a step moves ~3 GB over the link: keep the timed work short
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.25 if clocks and clocks.proc else 0)
    ms = timed("full", steps)
    clk = clocks.stop() if clocks else None
    ms_stage = timed("stage", steps)
    ms_attend = timed("attend", steps)
    ms_zero = timed("zero_copy", max(3, steps // 4))
    assert plan.device_error() == 0, "device error word set"

    host_q = q_all.cpu().pin_memory()
    host_out = torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory()
    with torch.cuda.stream(stream):
        q_all.copy_(host_q, non_blocking=True)
        graphs["full"].replay()
        host_out.copy_(out_all, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            q_all.copy_(host_q, non_blocking=True)
            graphs["full"].replay()
            host_out.copy_(out_all, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)

    link_achieved = staged_bytes / (ms * 1e-3) / 1e9
    overlap = (ms_stage + ms_attend - ms) / min(ms_stage, ms_attend) if min(ms_stage, ms_attend) > 0 else None
    line = {
        "impl": "zoomr", "path": "offload", "metric": OFFLOAD_METRIC, "value": world * 1e3 / ms, "unit": "steps/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) K/V, queries near one summary segment's mean key)",
        "config": {"split": "even (deterministic plan)" if args.deterministic else "dynamic (attend-only calls)", "workload": spec.name + "_offload" + ("" if L == spec.layers else f"_first{L}layers"),
                   "batch": Bn, "prompt": spec.prompt_len, "generated": spec.gen_len, "layers": L, "q_heads": Hq,
                   "kv_heads": H, "head_dim": d, "top_k": spec.topk, "consensus": spec.consensus,
                   "window": spec.window, "graph": True, "staging_slots": cap, "staging_pools": 2,
                   "pools": "pinned host memory (every layer's K/V); two HBM staging pools holding the final context's rows"},
        "staged_bytes_per_step": staged_bytes, "final_set_tokens": tok,
        "stage_only_ms": ms_stage, "attend_only_ms": ms_attend, "zero_copy_ms": ms_zero,
        "overlap": overlap,
        "roofline": {"bound": "link", "achieved": link_achieved, "peak": link_gbs, "unit": "GB/s",
                     "frac": link_achieved / link_gbs, "traffic": None, "kernel": "zr_stage_copy_kernel",
                     "peak_kind": "measured pinned-host-to-device copy bandwidth of this box (1 GiB cudaMemcpyAsync, "
                                  "median of 5)",
                     "alg_bytes_per_launch": staged_bytes // L,
                     "timing": "the whole step (map, then every layer's staging copy on a copy stream and its "
                               "attention on the compute stream), captured as one graph; link bytes / step time"},
        "hbm_attend_alg_bytes_per_layer": attend_bytes,
        "e2e": {"value": world * 1e3 / e2e_ms, "unit": "steps/s", "h2d_bytes_per_step": host_q.numel() * eb,
                "d2h_bytes_per_step": host_out.numel() * 4},
        "gpu_launches": (4 + L * 3) * steps,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------- generation loop
GENERATE_METRIC = ("ZoomR generation steps/s at 8B shape, 512-token prompt + 16K generated, batch 8, 32 layers: every "
                   "step appends each layer's K/V and moves the window, every 35th step also votes and selects")


def run_generate(args):
    """The consensus path as a decode loop: each step appends every layer's new K/V row (zr_append_kv), moves
    the windows to the new lengths (zr_consensus_advance) and attends every layer (zr_consensus_attend); every
    35th step first votes in every layer and selects (zr_consensus_vote, zr_consensus_select). The lengths live
    on the device and grow by one per step inside the captured graphs, so consecutive replays are consecutive
    steps."""
    spec = W.CONSENSUS_WORKLOADS[1]
    world, rank, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: the generation loop needs a CUDA GPU")
    from hierarchical_sparse_kv_gb300 import build as B
    from hierarchical_sparse_kv_gb300 import zoomr as Z

    if rank == 0 or world == 1:
        B.build()
    barrier(world)
    Z.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    T = SELECTION_INTERVAL
    rounds_total = args.steps + args.warmup + 2
    room = T * rounds_total + 1
    st0 = W.make_consensus_structure(spec, spare_blocks=spec.batch * (room // 16 + 2))
    Lg = st0.seq_lens.astype(np.int64) + room
    cols = int(((Lg + 15) // 16).max())
    tables = np.full((st0.batch, cols), -1, np.int32)
    tables[:, :st0.max_blocks_per_seq] = st0.block_tables
    used = set(st0.block_tables.ravel().tolist())
    free = [x for x in range(st0.num_blocks) if x not in used]
    for b in range(st0.batch):
        for j in range(int((Lg[b] + 15) // 16)):
            if tables[b, j] < 0:
                tables[b, j] = free.pop(0)
    import dataclasses
    st = dataclasses.replace(st0, block_tables=tables)
    L = spec.layers if args.layers is None else max(1, min(args.layers, spec.layers))
    Bn, H, Hq, d = st.batch, spec.num_kv_heads, spec.num_q_heads, spec.head_dim
    dt = W.torch_dtype(spec.dtype)
    lts = [W.make_consensus_layer(st, l, dev) for l in range(L)]
    bt = torch.from_numpy(st.block_tables).to(dev)
    cfg = Z.cache_config(batch=Bn, num_kv_heads=H, head_dim=d, num_blocks=st.num_blocks,
                         max_blocks_per_seq=st.max_blocks_per_seq, dtype=spec.dtype)
    segs = torch.tensor([(b, s, e, int(st.seg_ptr[b]) + i) for b in range(Bn)
                         for i, (s, e) in enumerate(st.summary_spans(b))], dtype=torch.int32, device=dev)
    mks = []
    for lt in lts:
        mk = torch.empty((st.total_segments, H, d), dtype=dt, device=dev)
        Z.zr_segment_summaries(cfg, segs, bt, lt.k_pool, lt.v_pool, mk, torch.empty_like(mk))
        mks.append(mk)
    plan = Z.ConsensusPlan.from_structure(st, device=dev).set_deterministic(args.deterministic)
    gen = torch.Generator(device=dev)
    gen.manual_seed(spec.seed + 1)
    kn = torch.randn((L, Bn, H, d), generator=gen, device=dev).to(dt)
    vn = torch.randn((L, Bn, H, d), generator=gen, device=dev).to(dt)
    q_all = torch.stack([lt.q for lt in lts])
    out_all = torch.empty((L, Bn, Hq, d), dtype=torch.float32, device=dev)
    lens = torch.from_numpy(st.seq_lens.astype(np.int32)).to(dev)
    pos = torch.empty_like(lens)
    stream = torch.cuda.Stream(device=dev)

    def step(boundary, s):
        lens.add_(1)
        torch.sub(lens, 1, out=pos)
        for l in range(L):
            Z.zr_append_kv(cfg, pos, kn[l], vn[l], bt, lts[l].k_pool, lts[l].v_pool, stream=s)
        if boundary:
            for l in range(L):
                plan.vote(q_all[l], mks[l], stream=s)
            plan.select(stream=s)
        plan.advance(lens, stream=s)
        for l in range(L):
            plan.attend(q_all[l], lts[l].k_pool, lts[l].v_pool, bt, out_all[l], stream=s)

    stream.wait_stream(torch.cuda.current_stream())
    graphs = {}
    with torch.cuda.stream(stream):
        step(True, stream)  # eager: the first selection, and warm-up
        for kind in (True, False):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(kind, stream)
            graphs[kind] = g
    torch.cuda.synchronize()
    # the captures ran nothing: the lengths moved once (the eager step)

    def rounds(n, e2e=False, host_q=None, host_out=None):
        with torch.cuda.stream(stream):
            for _ in range(n):
                for i in range(T):
                    if e2e:
                        q_all.copy_(host_q, non_blocking=True)
                    graphs[i == 0].replay()
                    if e2e:
                        host_out.copy_(out_all, non_blocking=True)

    rounds(args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.25 if clocks and clocks.proc else 0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    rounds(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(e0.elapsed_time(e1) / (args.steps * T), world)
    host_q = q_all.cpu().pin_memory()
    host_out = torch.empty(out_all.shape, dtype=out_all.dtype).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    rounds(1, True, host_q, host_out)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / T, world)
    final_len = lens.cpu().numpy()
    assert int(final_len[0]) <= int(st.seq_lens[0]) + room, "ran past the block tables' room"
    assert plan.device_error() == 0, "device error word set"
    launches_regular = 3 + 3 * L
    launches_boundary = launches_regular + L + 1
    line = {
        "impl": "zoomr", "path": "generate", "metric": GENERATE_METRIC, "value": world * 1e3 / ms, "unit": "steps/s",
        "n_gpus": world, "steps": args.steps * T, "warmup": args.warmup * T, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) K/V and new rows, queries near one summary segment's mean key)",
        "config": {"split": "even (deterministic plan)" if args.deterministic else "dynamic (attend-only calls)", "workload": spec.name + ("" if L == spec.layers else f"_first{L}layers") + "_generate",
                   "batch": Bn, "prompt": spec.prompt_len, "generated_at_start": spec.gen_len, "layers": L,
                   "q_heads": Hq, "kv_heads": H, "head_dim": d, "top_k": spec.topk, "consensus": spec.consensus,
                   "window": spec.window, "selection_interval": T, "graph": True,
                   "tokens_appended": int(final_len[0] - st.seq_lens[0]),
                   "l2": "each step reads the 32 layers' final sets (far beyond L2); no flush"},
        "e2e": {"value": world * 1e3 / e2e_ms, "unit": "steps/s", "h2d_bytes_per_step": host_q.numel() * 2,
                "d2h_bytes_per_step": host_out.numel() * 4},
        "gpu_launches": int(args.steps * ((T - 1) * launches_regular + launches_boundary)),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["zoomr", "reference"], default="zoomr")
    ap.add_argument("--workload", type=int, default=WORKLOAD_ID, choices=sorted(W.WORKLOADS),
                    help="seeded workload (default: the 8 x 16K, 32-layer headline step)")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying CUDA graphs")
    ap.add_argument("--deterministic", action="store_true",
                    help="deterministic plans: the attend-only calls (consensus, generate, offload paths) take the even "
                         "split of the rows instead of the dynamic one; the decode step always takes the even split")
    ap.add_argument("--max-graphs", type=int, default=64, help="distinct captured steps (each with its own events)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-oracle-accounting", action="store_true",
                    help="count algorithmic bytes from the kernel's own ranges instead of the oracle's selection")
    ap.add_argument("--attend-samples", type=int, default=128,
                    help="attend launches timed with an event pair after the timed region")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work for cpu_baseline, once on one core and once on all cores")
    ap.add_argument("--path", choices=["decode", "append", "consensus", "offload", "generate"], default="decode",
                    help="decode: the headline decode step; append: the cache-update path (appends and summaries); "
                         "consensus: ZoomR's own consensus selection and attention over its final set; offload: the "
                         "consensus decode step with every layer's K/V in pinned host memory, the final context "
                         "staged into HBM per layer; generate: the consensus path as a "
                         "decode loop (appends, window advance, a selection every 35 steps)")
    ap.add_argument("--layers", type=int, default=None,
                    help="append, consensus and offload paths only: run the first N layers (a small case for profiling; "
                         "the metrics are defined on all 32)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.path == "append":
        return run_append(args)
    if args.path == "generate":
        return run_generate(args)
    if args.path == "offload":
        return run_offload(args)
    return run_consensus(args) if args.path == "consensus" else run_zoomr(args)


if __name__ == "__main__":
    sys.exit(main())
