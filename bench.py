#!/usr/bin/env python
"""Benchmark: certified decode-attention queries/s at 32K context, and HBM GB/s of the dominant
kernel against the GB300's measured peak.

Workload (the single-layer 32K configuration): n = 32768 tokens, 8 KV heads x 4 query heads,
d = 128, bf16 K/V with outlier channels, importance scores lognormal(0, 1.5) normalised, H = 4
sink + 512 local tokens, eta = 1/16 (6.25 % resident), batch 1, 256 decode queries of which a
quarter are aimed at planted keys PoissonComp did not keep, eps = delta = 0.05.  The layer is
held as 4 independent instances (4 x 73 MiB of resident state > the 129 MB L2) and query t attends
instance t mod 4, so each query streams its sketch from HBM as it would behind 35 other layers.

The default run also records, in the same JSON line, the estimator pass alone (its HBM rate), the
MEMCPY fetch path (copy rate and overlap) and whole decode steps of a 36-layer model at 32K
(batch 8, eta in {1/8, 1/32}) and 128K (batch 4, eps in {0.02, 0.05}) ("model_steps").

One step = PoissonComp over the 4 instances (a1-a3) + 256 decode queries, each through sketch
scoring, the beta solve, the Bernstein certificate, selection, the fetch of selected rows from
page-locked host memory, the shrinkage-estimator attention over the pivotal set and the refine
(a4-a10).  A query is one decode token's attention for all 32 query heads of the layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

# The oracle's matrix products run on numpy's BLAS: one thread each, so that the timed CPU
# baselines use exactly the threads they report (one, or one per core).
for _v in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "certified decode-attention queries/s at 32K ctx; HBM GB/s vs GB300 peak"
UNIT = "queries/s"
LAYERS = 4
QUERIES = 256


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--fetch-mode", choices=["zerocopy", "memcpy"], default="zerocopy")
    p.add_argument("--no-graph", action="store_true", help="launch eagerly instead of graph replay")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--quiet", action="store_true",
                   help="--decode-step / --long128k: no per-call progress on stderr")
    p.add_argument("--no-model-steps", action="store_true",
                   help="skip the 36-layer decode steps (32K batch 8, 128K batch 4) of the default run")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the estimator-pass and MEMCPY-fetch measurements of the default run")
    p.add_argument("--queries", type=int, default=QUERIES)
    p.add_argument("--eps-sweep", action="store_true",
                   help="tolerance sweep: throughput and host-traffic statistics per eps")
    p.add_argument("--shortlist", type=int, default=0,
                   help="shortlist variant: at most this many fetch candidates per KV head (0: off)")
    p.add_argument("--sketch", choices=["exact", "q2"], default="exact",
                   help="token sketch: exact bf16 keys (the headline) or the 2-bit sketch")
    p.add_argument("--long128k", action="store_true",
                   help="the fetch-stressed long-context workload: 128K tokens, --layers layers x "
                        "batch 4 x 8 KV heads, eta = 1/32, needle sets, eps in {0.02, 0.05}")
    p.add_argument("--decode-step", action="store_true",
                   help="the full decode step: --layers layers x batch 8 x 8 KV heads x 4 query "
                        "heads at 32K, eta in {1/8, 1/32}, eps = delta = 0.05")
    p.add_argument("--layers", type=int, default=36,
                   help="layers of the --decode-step and --long128k models")
    p.add_argument("--groups", type=int, default=4,
                   help="--decode-step / --long128k: the batch split over this many contexts, each "
                        "on its own stream (each group's layers run in order; 1: one context)")
    p.add_argument("--pc-sweep", action="store_true",
                   help="PoissonComp throughput: 36 layers x 8 KV heads, n in {32K, 128K}, "
                        "eta in {1/8, 1/16, 1/32}")
    p.add_argument("--pc-n", type=int, nargs="+", default=[32768, 131072],
                   help="context lengths of the PoissonComp sweep")
    p.add_argument("--pc-eta", type=float, nargs="+", default=[1 / 8, 1 / 16, 1 / 32],
                   help="budget fractions of the PoissonComp sweep")
    p.add_argument("--pc-heads", type=int, default=36 * 8,
                   help="heads per PoissonComp call (a multiple of 8: layers x 8 KV heads)")
    p.add_argument("--estimator", action="store_true",
                   help="the shrinkage-estimator pass over the pivotal set alone: batch 32 x 8 KV "
                        "heads x 4 query heads at 32K, eta = 1/16, its HBM rate")
    p.add_argument("--est-batch", type=int, default=32,
                   help="sequences in the --estimator workload (8 KV heads each)")
    p.add_argument("--dense-offload", action="store_true",
                   help="the offloaded-dense baseline alone (every row from the host cache)")
    return p.parse_args()


# ------------------------------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, device=None):
    """The largest value of x over all ranks (x unchanged without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, queries_per_step, steps, max_elapsed_ms):
    """Whole-job queries/s: every rank processed `queries_per_step` per step; the job took as long
    as its slowest rank."""
    return world * queries_per_step * steps / (max_elapsed_ms / 1e3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback 6.8 TB/s"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        # the raw samples stay in a scratch file; the JSON line carries their summary
        self.path = os.path.join(tempfile.gettempdir(), f"verkv_clocks_gpu{device_index}_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200",
                                          "-i", str(self.idx)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
def cpu_baseline(w):
    """Time the oracle, as it stands, on a bounded sample of the workload: on one thread, and on
    every host core (a thread per core: the oracle's C routines run outside the interpreter lock,
    over independent (query, KV head) units and PoissonComp heads).  A quarter of the sampled
    queries are planted, as in the workload.  Scaled to a step of LAYERS layers' PoissonComp +
    QUERIES queries."""
    import concurrent.futures as cf

    import oracle as O

    cores = os.cpu_count() or 1
    planted = [t for t in range(w.queries.shape[0]) if w.planted[t]]
    plain = [t for t in range(w.queries.shape[0]) if not w.planted[t]]
    KV = {(l, h): (O.bf16_to_f64(w.kv[0, l, h, :, 0, :]), O.bf16_to_f64(w.kv[0, l, h, :, 1, :]))
          for l in range(LAYERS) for h in range(w.h_kv)}

    def pc(l, h):
        return O.poissoncomp(w.tau[0, l, h], w.eta, w.n_sink, w.n_local, w.seed, 0, l, h)

    pcs = {}

    def unit(t, h):
        l = int(w.query_layer[t])
        K, V = KV[(l, h)]
        qs = O.bf16_to_f64(w.queries[t, 0, h * w.G:(h + 1) * w.G])
        O.attend_unit(qs, K, K, V, pcs[(l, h)]["r32"], pcs[(l, h)]["resident"], w.eps, w.delta)

    # one thread: PoissonComp of every head; 6 plain and 2 planted queries
    t0 = time.perf_counter()
    for l in range(LAYERS):
        for h in range(w.h_kv):
            pcs[(l, h)] = pc(l, h)
    t_pc1 = time.perf_counter() - t0                            # all heads of LAYERS layers
    sample1 = plain[:6] + planted[:2]
    t0 = time.perf_counter()
    for t in sample1:
        for h in range(w.h_kv):
            unit(t, h)
    t_q1 = (time.perf_counter() - t0) / len(sample1)            # per query
    # every core: PoissonComp of all heads again; 2 x cores queries, a quarter planted
    nq = max(8, 2 * cores)
    sampleN = plain[:nq - nq // 4] + planted[:nq // 4]
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        t0 = time.perf_counter()
        list(ex.map(lambda lh: pc(*lh), [(l, h) for l in range(LAYERS) for h in range(w.h_kv)]))
        t_pcN = time.perf_counter() - t0
        t0 = time.perf_counter()
        list(ex.map(lambda th: unit(*th), [(t, h) for t in sampleN for h in range(w.h_kv)]))
        t_qN = (time.perf_counter() - t0) / len(sampleN)        # per query
    step1 = t_pc1 + QUERIES * t_q1
    stepN = t_pcN + QUERIES * t_qN
    return {"value": QUERIES / stepN, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"all {cores} host cores (a thread each): PoissonComp of {LAYERS} layers x "
                      f"{w.h_kv} heads and {len(sampleN)} queries "
                      f"({sum(1 for t in sampleN if w.planted[t])} planted), 32 query heads each; "
                      f"scaled to a step of {LAYERS} layers' PoissonComp + {QUERIES} queries",
            "seconds": round(t_pcN + t_qN * len(sampleN), 2),
            "single_thread": {"value": QUERIES / step1, "cores": 1,
                              "sample": f"PoissonComp of {LAYERS} layers x {w.h_kv} heads + "
                                        f"{len(sample1)} queries "
                                        f"({sum(1 for t in sample1 if w.planted[t])} planted)",
                              "seconds": round(t_pc1 + t_q1 * len(sample1), 2)}}


def bench_config(args, Q, world):
    """The benchmark workload's description, the same for both arms."""
    return {"workload": "single-layer 32K: n=32768, 8 KV heads x 4 query heads, "
                        "d=128, bf16, eta=1/16, H=4 sink+512 local, batch 1, "
                        f"{Q} decode queries (1/4 aimed at unsampled planted keys), "
                        "eps=delta=0.05; layer held as 4 independent instances, "
                        "query t on instance t mod 4",
            "l2": "inputs larger than L2 (4 x 73 MiB resident state per step)",
            "fetch": args.fetch_mode, "sketch": args.sketch,
            "shortlist": args.shortlist,
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step a bounded sample of the workload."""
    if rank != 0:
        return
    from verified_kv_cache_poissoncomp_gb300 import inputs as I
    import oracle as O

    w = I.single_layer_32k(layers=LAYERS, n_queries=args.queries)
    # Two queries a step, and one PoissonComp head every fourth step: one head per 8 queries, the
    # proportion of the benchmark's step (4 layers x 8 heads per 256 queries); a default run of
    # 43 steps stays within a few minutes.
    per_step = 2
    state = {"q": 0, "head": 0, "step": 0}
    pcs = {}
    for h in range(w.h_kv):
        pcs[h] = O.poissoncomp(w.tau[0, 0, h], w.eta, w.n_sink, w.n_local, w.seed, 0, 0, h)
    layer0 = [t for t in range(w.queries.shape[0]) if w.query_layer[t] == 0]

    def step():
        if state["step"] % 4 == 0:
            h0 = state["head"] % w.h_kv
            O.poissoncomp(w.tau[0, 0, h0], w.eta, w.n_sink, w.n_local, w.seed, 0, 0, h0)
            state["head"] += 1
        state["step"] += 1
        for _ in range(per_step):
            t = layer0[state["q"] % len(layer0)]
            state["q"] += 1
            for h in range(w.h_kv):
                K = O.bf16_to_f64(w.kv[0, 0, h, :, 0, :])
                V = O.bf16_to_f64(w.kv[0, 0, h, :, 1, :])
                qs = O.bf16_to_f64(w.queries[t, 0, h * w.G:(h + 1) * w.G])
                O.attend_unit(qs, K, K, V, pcs[h]["r32"], pcs[h]["resident"], w.eps, w.delta)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": bench_config(args, w.queries.shape[0], world),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": f"each step: {per_step} queries (32 query heads each, "
                                      "from layer instance 0) and, every fourth step, "
                                      "PoissonComp of 1 head: the benchmark's proportion of "
                                      "PoissonComp to queries; single thread"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------------------------------------
def _capture(kernel):
    """This kernel's entry of the committed ncu capture (profiles/traffic.json), or None when
    the kernel's source changed since the capture (the entry stores the source hash)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    ent = table.get(kernel)
    if not ent:
        return None
    src = os.path.join(ROOT, ent["source"])
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != ent["sha256"]:
            return None
    return ent


def traffic_for(kernel):
    """Per-launch DRAM bytes (read + write) from the committed ncu capture, or None."""
    ent = _capture(kernel)
    return ent["dram_bytes_per_launch"] if ent else None


def run_ours(args, world, rank, local):
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B
    from verified_kv_cache_poissoncomp_gb300 import inputs as I
    from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap

    B.lib()  # the CUDA library must be present: no fallback
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = I.single_layer_32k(layers=LAYERS, n_queries=args.queries)
    Q = w.queries.shape[0]
    cap = default_cap(w.n, w.eta)
    stream = torch.cuda.Stream(dev)
    mode = B.VERKV_FETCH_MEMCPY if args.fetch_mode == "memcpy" else B.VERKV_FETCH_ZEROCOPY
    with torch.cuda.stream(stream):
        eng = VerKV(w.B, w.L, w.h_kv, w.G, w.d, w.n, cap, fetch_mode=mode,
                    sketch_format=sketch_format(args))
        eng.load(w.tau.reshape(-1, w.n), w.kv.reshape(-1, w.n, 2, w.d))
        eng.compress(w.eta, w.n_sink, w.n_local, w.seed)   # also builds the sketch
        eng.sync()
        if args.shortlist:
            eng.set_shortlist(args.shortlist)
        q_dev = torch.as_tensor(w.queries.view(np.int16)).to(dev)          # [Q][1][32][128]
        hq = w.B * w.h_kv * w.G
        o_all = torch.empty((Q, hq, w.d), dtype=torch.float32, device=dev)
        lse_all = torch.empty((Q, hq), dtype=torch.float32, device=dev)
        st_all = torch.empty((Q, hq, 16), dtype=torch.int32, device=dev)
        fc_all = torch.zeros((Q, w.B * w.h_kv), dtype=torch.int32, device=dev)  # rows fetched
        tau_dev = eng.tau
        kv_dev = eng.kv

    # The timed steps ask for no fetch ids or counts (the refine reads the selection bitmaps);
    # one untimed pass with counts gives the rows moved per KV head for the statistics.
    def step(counts=False):
        B.verkv_poissoncomp(eng.ctx, tau_dev.data_ptr(), w.eta, B.verkv_hset(w.n_sink, w.n_local),
                            w.seed, kv_dev.data_ptr(), eng.r_full.data_ptr(), eng.pivotal)
        for t in range(Q):
            B.verkv_attend_verified(eng.ctx, int(w.query_layer[t]), q_dev[t].data_ptr(),
                                    eng.pivotal, eng.r_full.data_ptr(), eng.sketch_desc, w.eps,
                                    w.delta, None, fc_all[t].data_ptr() if counts else None)
            B.verkv_fetch_refine(eng.ctx, None, None, eng.host_kv.data_ptr(),
                                 o_all[t].data_ptr(), lse_all[t].data_ptr(), st_all[t].data_ptr())

    # Launches per step, counted by the library over one eager step.
    with torch.cuda.stream(stream):
        before = B.verkv_launch_counts(eng.ctx)
        step()
        B.verkv_sync(eng.ctx)
        after = B.verkv_launch_counts(eng.ctx)
    launches_per_step = int(sum(after[k] - before[k] for k in B.KERNEL_IDS))

    graph = None
    if not args.no_graph and mode == B.VERKV_FETCH_ZEROCOPY:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                step()
        except Exception as e:  # noqa: BLE001 -- fall back to eager launches, reported below
            print(f"graph capture failed, launching eagerly: {e}", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()

    def run_steps(k):
        with torch.cuda.stream(stream):
            for _ in range(k):
                if graph is not None:
                    graph.replay()
                else:
                    step()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # Warm-up, then the timed region (device-resident inputs).
    run_steps(args.warmup)
    barrier()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        run_steps(args.steps)
        ev1.record(stream)
        barrier()
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), dev)
    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(world, Q, args.steps, elapsed_ms)
    B.verkv_sync(eng.ctx)

    # Per-kernel CUDA-event durations over a profiled pass of the same steps (eager launches).
    B.verkv_profile_enable(eng.ctx, 1)
    with torch.cuda.stream(stream):
        for _ in range(max(1, min(args.steps, 10))):
            step()
    launches, total_ms = B.verkv_profile_read(eng.ctx)
    B.verkv_profile_enable(eng.ctx, 0)
    per_kernel = {B.verkv_kernel_name(k): {"launches": int(launches[k]),
                                           "avg_us": 1e3 * total_ms[k] / max(launches[k], 1),
                                           "total_ms": total_ms[k]}
                  for k in range(B.VERKV_K_COUNT) if launches[k] > 0}

    # Host-to-device link: a 256 MiB page-locked cudaMemcpyAsync, best of 5.
    hbuf = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    link = 0.0
    for _ in range(5):
        l0 = torch.cuda.Event(enable_timing=True)
        l1 = torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        with torch.cuda.stream(stream):
            dbuf.copy_(hbuf, non_blocking=True)
        l1.record(stream)
        l1.synchronize()
        link = max(link, hbuf.nbytes / (l0.elapsed_time(l1) * 1e-3) / 1e9)
    del hbuf, dbuf
    peak, peak_src = measured_peaks()
    link_src = "measured: 256 MiB page-locked cudaMemcpyAsync, best of 5"

    # Algorithmic bytes per launch of each kernel of the step; the bound
    # is HBM except for the fetch, which is bound by the host link.
    with torch.cuda.stream(stream):
        step(counts=True)
    B.verkv_sync(eng.ctx)
    counts = eng.p_count.cpu().numpy().astype(np.int64)
    st = st_all.cpu().numpy()
    fetched_rows = fc_all.cpu().numpy().astype(np.int64)          # [Q][units] of the last step
    units_layer = w.B * w.h_kv
    units_all = w.B * w.L * w.h_kv
    sketch_row_bytes = B.verkv_sketch_bytes(eng.shape, eng.sketch_format) // (units_all * w.n)
    fetch_row_bytes = (2 if args.sketch == "exact" else 4) * w.d
    algo = {
        "k_score": ("hbm", units_layer * w.n * sketch_row_bytes),
        # latency- and issue-bound: measured by warp instructions issued, not bytes
        "k_certify": ("alu", units_layer * (w.G * w.n * 4 + w.n * 4)),  # logits + r
        "k_partial(pivotal)": ("hbm", int(counts.mean() * units_layer * (4 * w.d + 8))),
        # with the exact sketch only V rows (2 d bytes) cross the host link, else K|V rows; the
        # zero-copy refine kernel also sums the pivotal rows (HBM) and merges, but the link binds
        "k_refine": ("h2d", int(fetched_rows.sum(1).mean() * fetch_row_bytes)),
        "k_pc_solve": ("hbm", int(units_all * w.n * 8.125 + counts.sum() * 8)),
        "k_pc_gather": ("hbm", int(counts.sum() * 2 * 4 * w.d)),
    }
    # Instruction-issue peak of the part: 152 SMs x 4 schedulers x one warp instruction per clock
    # at the SM clock sampled during the timed region (2070 MHz max).
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk_mhz = (clk.summary() or {}).get("sm_mhz") or 2070.0
    issue_peak = sms * 4 * clk_mhz * 1e6 / 1e9  # G warp-instructions / s
    rooflines = {}
    for k, (bound, nbytes) in algo.items():
        if k in per_kernel and nbytes > 0:
            t_us = per_kernel[k]["avg_us"]
            if bound == "alu":
                ent = _capture(k)
                wi = ent.get("warp_instructions_per_launch") if ent else None
                ach = wi / (t_us * 1e-6) / 1e9 if wi else None
                rooflines[k] = {"bound": "alu", "achieved": round(ach, 1) if ach else None,
                                "peak": round(issue_peak, 1), "unit": "G warp-inst/s",
                                "frac": round(ach / issue_peak, 4) if ach else None,
                                "avg_us": round(t_us, 3), "warp_instructions_per_launch": wi,
                                "algorithmic_bytes_per_launch": int(nbytes),
                                "hbm_GBs": round(nbytes / (t_us * 1e-6) / 1e9, 1),
                                "traffic": traffic_for(k),
                                "peak_source": f"{sms} SMs x 4 schedulers x {clk_mhz:.0f} MHz; "
                                               "instructions from the committed ncu capture"}
                continue
            ach = nbytes / (t_us * 1e-6) / 1e9
            pk = link if bound == "h2d" else peak
            rooflines[k] = {"bound": bound, "achieved": round(ach, 1), "peak": round(pk, 1),
                            "unit": "GB/s", "frac": round(ach / pk, 4), "avg_us": round(t_us, 3),
                            "algorithmic_bytes_per_launch": int(nbytes),
                            "traffic": traffic_for(k),
                            "peak_source": link_src if bound == "h2d" else peak_src}
    # k_score against a bare one-launch read of the same sketch bytes: the library streams each
    # query's layer through the scoring kernel's grid and copy ring with no arithmetic, timed the
    # same way (an event pair per launch) over the same sequence of layer instances.
    if "k_score" in rooflines and args.sketch == "exact":
        pairs = []
        with torch.cuda.stream(stream):
            for t in range(min(Q, 72)):
                e_a = torch.cuda.Event(enable_timing=True)
                e_b = torch.cuda.Event(enable_timing=True)
                e_a.record(stream)
                B.verkv_measure_sketch_stream(eng.ctx, int(w.query_layer[t]), eng.sketch_desc)
                e_b.record(stream)
                if t >= 8:  # the first launches warm up
                    pairs.append((e_a, e_b))
        B.verkv_sync(eng.ctx)
        read_us = 1e3 * sum(a.elapsed_time(b) for a, b in pairs) / len(pairs)
        r = rooflines["k_score"]
        r["one_launch_read_us"] = round(read_us, 3)
        r["one_launch_read_GBs"] = round(r["algorithmic_bytes_per_launch"] / (read_us * 1e-6) / 1e9, 1)
        r["frac_of_one_launch_read"] = round(read_us / r["avg_us"], 4)
    dom = max(per_kernel, key=lambda k: per_kernel[k]["total_ms"])
    roof = dict(rooflines[dom], kernel=dom) if dom in rooflines else None
    # The HBM-bound kernel that moves the most bytes per step (the one whose bandwidth matters).
    hbm = {k: v for k, v in rooflines.items() if v["bound"] == "hbm"}
    dom_hbm = max(hbm, key=lambda k: per_kernel[k]["launches"] * hbm[k]["algorithmic_bytes_per_launch"]) if hbm else None
    roof_hbm = dict(hbm[dom_hbm], kernel=dom_hbm) if dom_hbm else None
    fetch = None
    if "k_refine" in rooflines:
        f = rooflines["k_refine"]
        fetch = {"kernel": "k_refine", "bytes_per_query": f["algorithmic_bytes_per_launch"],
                 "avg_us": f["avg_us"], "achieved_GBs": f["achieved"], "link_peak_GBs": f["peak"],
                 "frac": f["frac"], "link_peak_source": link_src}
    stats_f = st[..., :10].view(np.float32)
    certified = st[..., 10]
    nfetch = st[..., 13]
    fetch_stats = {"certified_frac": float(certified.mean()),
                   "fetched_rows_per_query_head": float(nfetch.mean()),
                   "fetched_frac_of_context": float(nfetch.mean() / w.n),
                   "planted_certified_frac": float(certified[w.planted].mean()),
                   "plain_certified_frac": float(certified[~w.planted].mean())}

    # End to end through the C ABI with host buffers (eager calls): H2D of the step's queries and
    # importance scores, D2H of o, lse and the per-head statistics, inside the timed region.
    e2e = None
    if not args.no_e2e:
        q_host = torch.empty(q_dev.shape, dtype=q_dev.dtype, pin_memory=True)
        q_host.copy_(torch.as_tensor(w.queries.view(np.int16)))
        tau_host = torch.empty(tau_dev.shape, dtype=tau_dev.dtype, pin_memory=True)
        tau_host.copy_(torch.as_tensor(w.tau.reshape(tau_dev.shape)))
        o_host = torch.empty(o_all.shape, dtype=o_all.dtype, pin_memory=True)
        lse_host = torch.empty(lse_all.shape, dtype=lse_all.dtype, pin_memory=True)
        st_host = torch.empty(st_all.shape, dtype=st_all.dtype, pin_memory=True)
        e2e_steps = max(1, min(args.steps, 10))

        def e2e_step():
            q_dev.copy_(q_host, non_blocking=True)
            tau_dev.copy_(tau_host, non_blocking=True)
            step()
            o_host.copy_(o_all, non_blocking=True)
            lse_host.copy_(lse_all, non_blocking=True)
            st_host.copy_(st_all, non_blocking=True)

        with torch.cuda.stream(stream):
            e2e_step()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(e2e_steps):
                e2e_step()
            e1.record(stream)
        barrier()
        e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
        e2e = {"value": job_throughput(world, Q, e2e_steps, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": int(q_host.nbytes + tau_host.nbytes),
               "d2h_bytes_per_step": int(o_host.nbytes + lse_host.nbytes + st_host.nbytes),
               "steps": e2e_steps, "launch": "eager C-ABI calls"}

    # The estimator pass on its own (its HBM fraction at 32K, batch 32) and the MEMCPY fetch path
    # on this workload (copy rate against the link, overlap with the pivotal sums): one GPU only.
    memcpy = None
    if rank == 0 and world == 1 and not args.no_extra:
        est = measure_estimator(32, 10, 3, dev)
        rooflines["k_partial(pivotal)"] = dict(est["roofline"], workload=est["workload"])
        memcpy = measure_memcpy_fetch(w, None, q_dev, 32, dev, link)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    # Whole decode steps of the 36-layer model at 32K (batch 8) and 128K (batch 4), one GPU: a
    # compact record of each, or why it was skipped.
    model = None
    if rank == 0 and world == 1 and not args.no_extra and not args.no_model_steps:
        model = {}
        for kind, host_gb in (("decode-step", 38.7), ("long128k", 77.3)):
            avail = mem_available_gb()
            if avail is not None and avail < 1.5 * host_gb + 8:
                model[kind] = {"skipped": f"{avail:.0f} GB of host memory available, "
                                          f"{host_gb} GB page-locked cache needed"}
                continue
            # In a child process: its page-locked cache and device memory go back when it
            # exits, and a failure there leaves this process's numbers intact.
            cmd = [sys.executable, os.path.join(ROOT, "bench.py"), f"--{kind}", "--layers", "36",
                   "--steps", "3", "--warmup", "2", "--quiet"]
            try:
                p = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
                lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
                if p.returncode == 0 and lines:
                    model[kind] = compact_model_steps(json.loads(lines[-1]))
                else:
                    model[kind] = {"error": f"exit {p.returncode}: " + " | ".join(p.stderr.strip().splitlines()[-2:])}
            except Exception as e:  # noqa: BLE001 -- recorded in the line, the bench goes on
                model[kind] = {"error": f"{type(e).__name__}: {e}"}

    if rank == 0:
        out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
               "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "bf16", "data": "synthetic",
               "config": bench_config(args, Q, world),
               "launch": "CUDA graph replay" if graph is not None else "eager",
               "roofline": roof, "roofline_hbm": roof_hbm, "rooflines": rooflines,
               "per_kernel_us": {
                   k: round(v["avg_us"], 3) for k, v in per_kernel.items()},
               "fetch_stats": fetch_stats, "fetch": fetch, "memcpy_fetch": memcpy,
               "clocks": clk.summary(),
               "gpu_launches": launches_per_step * args.steps,
               "launches_per_step": launches_per_step,
               "e2e": e2e, "cpu_baseline": cpu, "model_steps": model}
        print(json.dumps(out), flush=True)
    if eng is not None:
        eng.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def mem_available_gb():
    """MemAvailable of the host in GB, or None where /proc/meminfo is missing."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 1e6
    except OSError:
        return None
    return None


def compact_model_steps(r):
    """The model-step record without the per-row traffic details."""
    keep = ("eta", "eps", "steps_per_s", "queries_per_s", "ms_per_step", "hbm_GBs",
            "h2d_bytes_per_step", "fetch_GBs_in_k_refine", "fetched_frac_per_kv_head",
            "certified_frac", "decisions_fetching_frac", "overall_read_frac", "clocks")
    rows = []
    for row in r["rows"]:
        c = {k: row[k] for k in keep if k in row}
        c["kernel_ms_per_step"] = {k: v["ms_per_step"] for k, v in row["per_kernel"].items()}
        rows.append(c)
    return {"config": r["config"], "steps": r["steps"], "warmup": r["warmup"],
            "launch": r.get("launch", "CUDA graph of one step, replayed"), "rows": rows,
            **{k: r[k] for k in ("planted_queries", "needle_frac_per_unit") if k in r}}


EPS_SWEEP = [0.01, 0.02, 0.05, 0.1, 0.2, 0.3, 0.5]


def sketch_format(args):
    from verified_kv_cache_poissoncomp_gb300 import binding as B
    return B.VERKV_SKETCH_Q2 if args.sketch == "q2" else B.VERKV_SKETCH_EXACT


def traffic_stats(st, fetched_rows, pivotal_count, n):
    """Host-traffic statistics of one pass over the queries, in the terms of the pages' traffic
    table: a decision is one query head's certificate; it fetches when eps-hat(L) >= eps and then
    moves |F \\ S| rows (the transfer itself is per KV head: the union over its query heads).
      st            int32 [Q][query heads][16]  verkv_head_stats
      fetched_rows  int   [Q][KV heads]         rows moved per KV head
      pivotal_count int   [units]               |H u S| per unit"""
    certified = st[..., 10].astype(bool)
    nfetch = st[..., 13].astype(np.float64)
    fetching = ~certified
    resident = float(pivotal_count.mean()) / n
    return {
        "decisions_fetching_frac": float(fetching.mean()),
        "shortlist_exhausted_frac": float(((st[..., 15] & 4) != 0).mean()),
        "context_frac_per_fetching_decision":
            float((nfetch[fetching] / n).mean()) if fetching.any() else 0.0,
        "overall_read_frac": resident + float((nfetch / n).mean()),
        "resident_frac": resident,
        "kv_head_transfer_frac": float(fetched_rows.mean()) / n,
    }


def time_dense_offload(eng, w, q_dev, stream, steps, warmup):
    """Queries/s of the offloaded-dense baseline on the engine's workload: each query reads every
    K|V row of its layer from the page-locked host cache (graph replay of the query loop)."""
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B

    Q = w.queries.shape[0]
    hq = w.B * w.h_kv * w.G
    o = torch.empty((Q, hq, w.d), dtype=torch.float32, device=q_dev.device)
    lse = torch.empty((Q, hq), dtype=torch.float32, device=q_dev.device)

    def step():
        for t in range(Q):
            B.verkv_attend_dense_host(eng.ctx, int(w.query_layer[t]), q_dev[t].data_ptr(),
                                      eng.host_kv.data_ptr(), o[t].data_ptr(), lse[t].data_ptr())

    with torch.cuda.stream(stream):
        step()
        B.verkv_sync(eng.ctx)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    B.verkv_sync(eng.ctx)
    ms = e0.elapsed_time(e1) / steps
    h2d = w.B * w.h_kv * w.n * 4 * w.d  # every K|V row of the layer, per query
    return {"queries_per_s": round(Q / (ms * 1e-3), 2), "ms_per_step": round(ms, 4),
            "h2d_bytes_per_query": int(h2d), "h2d_GBs": round(h2d * Q / (ms * 1e-3) / 1e9, 1)}


def run_eps_sweep(args, local):
    """One GPU: the bench workload at each tolerance of EPS_SWEEP, graph-replayed like the main
    bench (a step = PoissonComp of the 4 instances + the decode queries)."""
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B
    from verified_kv_cache_poissoncomp_gb300 import inputs as I
    from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap

    B.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = I.single_layer_32k(layers=LAYERS, n_queries=args.queries)
    Q = w.queries.shape[0]
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        eng = VerKV(w.B, w.L, w.h_kv, w.G, w.d, w.n, default_cap(w.n, w.eta),
                    sketch_format=sketch_format(args))
        eng.load(w.tau.reshape(-1, w.n), w.kv.reshape(-1, w.n, 2, w.d))
        eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
        eng.sync()
        if args.shortlist:
            eng.set_shortlist(args.shortlist)
        q_dev = torch.as_tensor(w.queries.view(np.int16)).to(dev)
        hq = w.B * w.h_kv * w.G
        o_all = torch.empty((Q, hq, w.d), dtype=torch.float32, device=dev)
        lse_all = torch.empty((Q, hq), dtype=torch.float32, device=dev)
        st_all = torch.empty((Q, hq, 16), dtype=torch.int32, device=dev)
        fc_all = torch.zeros((Q, w.B * w.h_kv), dtype=torch.int32, device=dev)

    def step(eps, counts=False):  # counts: an untimed pass for the statistics
        B.verkv_poissoncomp(eng.ctx, eng.tau.data_ptr(), w.eta, B.verkv_hset(w.n_sink, w.n_local),
                            w.seed, eng.kv.data_ptr(), eng.r_full.data_ptr(), eng.pivotal)
        for t in range(Q):
            B.verkv_attend_verified(eng.ctx, int(w.query_layer[t]), q_dev[t].data_ptr(),
                                    eng.pivotal, eng.r_full.data_ptr(), eng.sketch_desc, eps,
                                    w.delta, None, fc_all[t].data_ptr() if counts else None)
            B.verkv_fetch_refine(eng.ctx, None, None, eng.host_kv.data_ptr(),
                                 o_all[t].data_ptr(), lse_all[t].data_ptr(), st_all[t].data_ptr())

    rows = []
    counts = None
    for eps in EPS_SWEEP:
        with torch.cuda.stream(stream):
            step(eps)  # eager once: first-use set-up outside the capture
            B.verkv_sync(eng.ctx)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                step(eps)
            for _ in range(args.warmup):
                graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        B.verkv_sync(eng.ctx)
        ms = e0.elapsed_time(e1) / args.steps
        with torch.cuda.stream(stream):
            step(eps, counts=True)
        B.verkv_sync(eng.ctx)
        if counts is None:
            counts = eng.p_count.cpu().numpy().astype(np.int64)
        fr = fc_all.cpu().numpy().astype(np.int64)
        row = {"eps": eps, "queries_per_s": round(Q / (ms * 1e-3), 2), "ms_per_step": round(ms, 4),
               "h2d_bytes_per_query": int(fr.sum(1).mean() * (2 if args.sketch == "exact" else 4) * w.d)}
        row.update({k: round(v, 5) for k, v in
                    traffic_stats(st_all.cpu().numpy(), fr, counts, w.n).items()})
        rows.append(row)
        del graph
    dense = time_dense_offload(eng, w, q_dev, stream, args.steps, args.warmup)
    for row in rows:
        row["speedup_vs_dense_offload"] = round(row["queries_per_s"] / dense["queries_per_s"], 3)
        row["host_bytes_reduction_vs_dense_offload"] = round(
            dense["h2d_bytes_per_query"] / max(row["h2d_bytes_per_query"], 1), 1)
    print(json.dumps({"sweep": "eps", "metric": METRIC, "unit": UNIT, "delta": w.delta,
                      "dense_offload": dense,
                      "steps": args.steps, "warmup": args.warmup, "data": "synthetic",
                      "config": {"workload": "single-layer 32K (the bench workload), "
                                             f"{Q} decode queries per step", "fetch": "zerocopy",
                                 "sketch": args.sketch, "shortlist": args.shortlist,
                                 "graph": True},
                      "rows": rows}), flush=True)
    eng.close()


def run_model_steps(args, local, kind):
    print(json.dumps(measure_model_steps(local, kind, args.layers, args.steps, args.warmup,
                                         verbose=not args.quiet, groups=args.groups)), flush=True)


def measure_model_steps(local, kind, layers, steps, warmup, verbose=True, groups=4):
    """One GPU, a whole decode step of a 36-layer model: every layer's attend_verified +
    fetch_refine for a batch of sequences, the full cache page-locked on the host and the
    pivotal set plus the exact sketch on the device.

    kind "decode-step": n = 32768, batch 8, 8 KV heads x 4 query heads, d = 128, eta in
        {1/8, 1/32}, eps = delta = 0.05; tau, sinks and queries as in the single-layer workload,
        a quarter of the (layer, sequence) queries aimed at unsampled planted keys.
    kind "long128k": n = 131072, batch 4, eta = 1/32, eps in {0.02, 0.05}, delta = 0.05, a needle
        set of U[2 %, 25 %] of the context per KV head that the queries favour.

    The batch is split into `groups` groups of sequences, one context each on its own stream
    (with its sequence offset set, so the Poisson draws are those of the whole-batch context):
    a group runs its layers in order (each layer's call depends on the one before, as in a
    model), and the groups are independent, so one group's host fetch overlaps another's
    scoring and certificate.  A query is one layer of one sequence (32 query heads); a step is
    layers x batch queries.  The first step runs eagerly with a synchronisation and a status
    check after every call; the timed steps replay one CUDA graph of the step (the groups'
    streams forked from and joined into the first); the per-kernel times come from a further
    eager step with the groups run one after another.  One JSON line."""
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B
    from verified_kv_cache_poissoncomp_gb300 import inputs as I
    from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap

    B.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L, KVH, G, D = layers, 8, 4, 128
    if kind == "decode-step":
        Bt, N = 8, 32768
        etas, epss = [1 / 8, 1 / 32], [0.05]
    else:
        Bt, N = 4, 131072
        etas, epss = [1 / 32], [0.02, 0.05]
    if groups < 1 or Bt % groups:
        raise SystemExit(f"--groups must divide the batch ({Bt})")
    bg = Bt // groups           # sequences per group
    ug = bg * L * KVH           # cache units per group (sequence-major: a contiguous slice)
    hg = bg * KVH * G           # query heads per group and layer
    delta = 0.05
    units = Bt * L * KVH
    t0 = time.time()
    if kind == "decode-step":
        tau, kv, queries, planted = I.decode_step_cache_torch(units, N, D, G, L, Bt, KVH, dev)
        extra = {"planted_queries": int(planted.sum())}
    else:
        tau, kv, queries, pfrac = I.long_context_torch(units, N, D, G, L, Bt, KVH, dev)
        extra = {"needle_frac_per_unit": {"mean": round(float(pfrac.mean()), 4),
                                          "min": round(float(pfrac.min()), 4),
                                          "max": round(float(pfrac.max()), 4)}}
    host_kv = torch.empty(kv.shape, dtype=torch.int16, pin_memory=True)
    host_kv.copy_(kv)
    torch.cuda.synchronize()
    gen_s = time.time() - t0
    hq = Bt * KVH * G
    streams = [torch.cuda.Stream(dev) for _ in range(groups)]
    s0 = streams[0]
    rows = []
    for eta in etas:
        engs = []
        for gi in range(groups):
            with torch.cuda.stream(streams[gi]):
                e = VerKV(bg, L, KVH, G, D, N, default_cap(N, eta), seq0=gi * bg)
                e.load_device(tau[gi * ug:(gi + 1) * ug], kv[gi * ug:(gi + 1) * ug],
                              host_kv[gi * ug:(gi + 1) * ug])
                e.compress(eta, 4, 512, 0)
                e.sync()
            engs.append(e)
        o_all = torch.empty((L, hq, D), dtype=torch.float32, device=dev)
        lse_all = torch.empty((L, hq), dtype=torch.float32, device=dev)
        st_all = torch.empty((L, hq, 16), dtype=torch.int32, device=dev)
        fc_all = torch.zeros((L, Bt * KVH), dtype=torch.int32, device=dev)
        # Pivotal counts in the cache's unit order (group by group: the groups are its slices).
        counts = np.concatenate([e.p_count.cpu().numpy() for e in engs]).astype(np.int64)
        for eps in epss:
            def step(check=False, with_counts=False, gis=range(groups)):
                for gi in gis:
                    e, h0, u0 = engs[gi], gi * hg, gi * bg * KVH
                    with torch.cuda.stream(streams[gi]):
                        for l in range(L):
                            if check and verbose:  # where a failing call would stop
                                print(f"checked call: eta={eta:.5f} eps={eps} group={gi} layer={l}",
                                      file=sys.stderr, flush=True)
                            q = queries[l][gi * bg:(gi + 1) * bg]
                            B.verkv_attend_verified(
                                e.ctx, l, q.data_ptr(), e.pivotal, e.r_full.data_ptr(),
                                e.sketch_desc, eps, delta, None,
                                fc_all[l, u0:u0 + bg * KVH].data_ptr() if with_counts else None)
                            if check:
                                B.verkv_sync(e.ctx)
                            B.verkv_fetch_refine(e.ctx, None, None, e.host_kv.data_ptr(),
                                                 o_all[l, h0:h0 + hg].data_ptr(),
                                                 lse_all[l, h0:h0 + hg].data_ptr(),
                                                 st_all[l, h0:h0 + hg].data_ptr())
                            if check:
                                B.verkv_sync(e.ctx)

            step(check=True, with_counts=True)          # checked, and the rows fetched
            torch.cuda.synchronize()
            fr = fc_all.cpu().numpy().astype(np.int64)  # [L][B*KVH]
            st = st_all.cpu().numpy()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s0):
                fork = torch.cuda.Event()
                fork.record(s0)
                for s in streams[1:]:
                    s.wait_event(fork)
                step()
                for s in streams[1:]:
                    join = torch.cuda.Event()
                    join.record(s)
                    s0.wait_event(join)
            with torch.cuda.stream(s0):
                for _ in range(warmup):
                    graph.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with ClockSampler(local) as clk:
                e0.record(s0)
                with torch.cuda.stream(s0):
                    for _ in range(steps):
                        graph.replay()
                e1.record(s0)
                torch.cuda.synchronize()
            for e in engs:
                B.verkv_sync(e.ctx)
            ms = e0.elapsed_time(e1) / steps
            del graph
            launches = np.zeros(B.VERKV_K_COUNT, dtype=np.int64)
            total_ms = np.zeros(B.VERKV_K_COUNT)
            for gi, e in enumerate(engs):  # one group at a time: each kernel's own time
                B.verkv_profile_enable(e.ctx, 1)
                step(gis=[gi])
                torch.cuda.synchronize()
                n_l, t_l = B.verkv_profile_read(e.ctx)
                B.verkv_profile_enable(e.ctx, 0)
                launches += np.asarray(n_l, dtype=np.int64)
                total_ms += np.asarray(t_l, dtype=np.float64)
            # Algorithmic bytes of a step: per layer call the sketch of every unit, the logits
            # written and read once, r, and the pivotal rows (K, V, id and r); host bytes: the V
            # row of every fetched token (the exact sketch holds the keys).
            units_layer = Bt * KVH
            hbm = 0
            for l in range(L):
                cnt_l = sum(int(counts[(b * L + l) * KVH + h]) for b in range(Bt) for h in range(KVH))
                hbm += units_layer * N * D * 2 + 2 * hq * N * 4 + units_layer * N * 4 + \
                    cnt_l * (4 * D + 8)
            h2d = int(fr.sum()) * 2 * D
            nfetch = st[..., 13]
            per_k = {B.verkv_kernel_name(k): {"launches_per_step": int(launches[k]),
                                              "avg_us": round(1e3 * total_ms[k] / launches[k], 2),
                                              "ms_per_step": round(float(total_ms[k]), 3)}
                     for k in range(B.VERKV_K_COUNT) if launches[k] > 0}
            fetch_ms = total_ms[B.VERKV_K_FETCH_HOST]
            rows.append({
                "eta": eta, "eps": eps, "steps_per_s": round(1e3 / ms, 3),
                "queries_per_s": round(L * Bt * 1e3 / ms, 2), "ms_per_step": round(ms, 3),
                "hbm_bytes_per_step": hbm, "hbm_GBs": round(hbm / (ms * 1e-3) / 1e9, 1),
                "h2d_bytes_per_step": h2d,
                "fetch_GBs_in_k_refine": round(h2d / (fetch_ms * 1e-3) / 1e9, 1) if fetch_ms else None,
                "fetched_frac_per_kv_head": {"mean": round(float(fr.mean()) / N, 4),
                                             "min": round(float(fr.min()) / N, 4),
                                             "max": round(float(fr.max()) / N, 4)},
                "certified_frac": round(float(st[..., 10].mean()), 4),
                "fetched_rows_per_query_head": round(float(nfetch.mean()), 1),
                "per_kernel": per_k, "clocks": clk.summary(),
                **traffic_stats(st.reshape(-1, 16), fr.reshape(-1), counts, N)})
        for e in engs:
            e.close()
        del engs, o_all, lse_all, st_all, fc_all
        torch.cuda.empty_cache()
    return {"workload": kind, "metric": METRIC, "unit": UNIT, "steps": steps,
                      "warmup": warmup, "data": "synthetic", "dtype": "bf16",
                      "config": {"layers": L, "batch": Bt, "kv_heads": KVH, "q_per_kv": G,
                                 "head_dim": D, "n": N, "delta": delta,
                                 "host_cache_GB": round(host_kv.nbytes / 1e9, 1),
                                 "sketch": "exact", "fetch": "zerocopy", "graph": True,
                                 "groups": groups, "sequences_per_group": bg},
                      "launch": f"CUDA graph of one step over {groups} contexts on {groups} streams",
                      "input_generation_s": round(gen_s, 1), **extra, "rows": rows}


def run_pc_sweep(args, local):
    """One GPU: verkv_poissoncomp (c solve, Poisson sample, compaction, pivotal K/V gather) over
    every head of a 36-layer x 8-KV-head cache per call (--pc-heads), for n in {32K, 128K}
    (--pc-n) and eta in {1/8, 1/16, 1/32} (--pc-eta); H = 4 sink + 512 local; tau lognormal(0,
    1.5) normalised per head; K/V bytes random on the device.  One JSON line."""
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B
    from verified_kv_cache_poissoncomp_gb300 import inputs as I
    from verified_kv_cache_poissoncomp_gb300.engine import default_cap

    B.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvh, d = 8, 128
    if args.pc_heads < kvh or args.pc_heads % kvh:
        raise SystemExit("--pc-heads must be a positive multiple of 8")
    layers = args.pc_heads // kvh
    units = layers * kvh
    peak, peak_src = measured_peaks()
    stream = torch.cuda.Stream(dev)
    rows = []
    for n in args.pc_n:
        tau = torch.from_numpy(I.pc_sweep_tau(units, n)).to(dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(1240)
        kv = torch.empty((units, n, 2, d), dtype=torch.int16, device=dev)
        kv.random_(-32768, 32767, generator=gen)
        r_full = torch.empty((units, n), dtype=torch.float32, device=dev)
        for eta in args.pc_eta:
            cap = default_cap(n, eta)
            shape = B.verkv_shape(1, layers, kvh, 4, d, n, cap)
            ws_bytes = B.verkv_workspace_size(shape)
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
            ids = torch.empty((units, cap), dtype=torch.int32, device=dev)
            pr = torch.empty((units, cap), dtype=torch.float32, device=dev)
            pkv = torch.empty((units, cap, 2, d), dtype=torch.int16, device=dev)
            cnt = torch.empty((units,), dtype=torch.int32, device=dev)
            res = torch.empty((units, (n + 31) // 32), dtype=torch.int32, device=dev)
            c = torch.empty((units,), dtype=torch.float32, device=dev)
            piv = B.verkv_pivotal(ids.data_ptr(), pr.data_ptr(), pkv.data_ptr(), cnt.data_ptr(),
                                  res.data_ptr(), c.data_ptr())
            ctx = B.verkv_create(local, stream.cuda_stream, shape, ws.data_ptr(), ws_bytes)
            H = B.verkv_hset(4, 512)

            def call():
                B.verkv_poissoncomp(ctx, tau.data_ptr(), eta, H, 0, kv.data_ptr(),
                                    r_full.data_ptr(), piv)

            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    call()
            B.verkv_sync(ctx)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                for _ in range(args.steps):
                    call()
            e1.record(stream)
            torch.cuda.synchronize()
            B.verkv_sync(ctx)
            ms = e0.elapsed_time(e1) / args.steps
            counts = cnt.cpu().numpy().astype(np.int64)
            # algorithmic bytes: tau in, r out, resident bitmap, ids + r of the sample, and the
            # gather's read and write of every pivotal K/V row
            nbytes = units * (8 * n + n // 8) + int(counts.sum()) * (8 + 2 * 4 * d)
            gbs = nbytes / (ms * 1e-3) / 1e9
            rows.append({"n": n, "eta": round(eta, 5), "ms_per_call": round(ms, 4),
                         "heads_per_s": round(units / (ms * 1e-3), 1),
                         "mean_pivotal_rows": round(float(counts.mean()), 1),
                         "algorithmic_bytes_per_call": nbytes, "achieved_GBs": round(gbs, 1),
                         "frac_of_hbm_peak": round(gbs / peak, 4)})
            B.verkv_destroy(ctx)
            del ws, ids, pr, pkv, cnt, res, c
        del kv, tau, r_full
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": "poissoncomp", "unit": "heads/s", "steps": args.steps,
                      "warmup": args.warmup, "data": "synthetic", "hbm_peak_GBs": peak,
                      "peak_source": peak_src,
                      "config": {"workload": f"{layers} layers x 8 KV heads per call, d=128, "
                                             "H=4+512, tau lognormal(0,1.5) normalised per head"},
                      "rows": rows}), flush=True)


def estimator_bytes(count, pivotal_r, d, G, sketch_logits=False):
    """Algorithmic bytes of one pass of the shrinkage estimator over the pivotal set: each
    pivotal row's K and V (4d bytes) and its id and r (8); with a 2-bit sketch (sketch_logits)
    also, for a sampled row (r < 1), the sketch logit of each of its G query heads (lambda's
    w-hat; the exact sketch gives the row's own weight).  count: rows per unit; pivotal_r:
    [units][cap].  Returns (bytes, sampled rows); the queries are negligible."""
    n_l = int(sum(int((pivotal_r[u, :count[u]] < 1.0).sum()) for u in range(len(count))))
    return int(np.sum(count)) * (4 * d + 8) + (n_l * 4 * G if sketch_logits else 0), n_l


def measure_estimator(batch, steps, warmup, dev):
    """The shrinkage-estimator attention over the pivotal set (D-hat, N-hat and the second
    moment), timed alone: in MEMCPY fetch mode the pivotal sums are their own launch,
    k_partial(pivotal) (in zero-copy mode the same stage code runs inside k_refine behind the host
    reads).  Workload: the decode-step cache generator at `batch` sequences x 8 KV heads x 4
    query heads, d = 128, n = 32768, eta = 1/16, H = 4 + 512, eps = delta = 0.05; one layer call
    of batch x 32 query heads per step, eager (the MEMCPY path waits on the host for the
    selection).  The pivotal rows (~270 MB a call at batch 32) are larger than L2, and k_score
    streams the sketch (2 GB at batch 32) before each pass.  Returns a dict."""
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B
    from verified_kv_cache_poissoncomp_gb300 import inputs as I
    from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap

    layers, kvh, G, d, n, eta = 1, 8, 4, 128, 32768, 1 / 16
    units = batch * layers * kvh
    peak, peak_src = measured_peaks()
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        tau, kv, queries, _ = I.decode_step_cache_torch(units, n, d, G, layers, batch, kvh, dev)
        host_kv = torch.empty(kv.shape, dtype=torch.int16, pin_memory=True)
        host_kv.copy_(kv)
        torch.cuda.synchronize()
        eng = VerKV(batch, layers, kvh, G, d, n, default_cap(n, eta),
                    fetch_mode=B.VERKV_FETCH_MEMCPY)
        eng.load_device(tau, kv, host_kv)
        eng.compress(eta, 4, 512, 0)
        eng.sync()
        q = queries[0].contiguous()
        hq = batch * kvh * G
        o = torch.empty((hq, d), dtype=torch.float32, device=dev)
        lse = torch.empty((hq,), dtype=torch.float32, device=dev)
        st = torch.empty((hq, 16), dtype=torch.int32, device=dev)

        def step():
            B.verkv_attend_verified(eng.ctx, 0, q.data_ptr(), eng.pivotal, eng.r_full.data_ptr(),
                                    eng.sketch_desc, 0.05, 0.05, None, None)
            B.verkv_fetch_refine(eng.ctx, None, None, eng.host_kv.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), st.data_ptr())

        for _ in range(warmup):
            step()
        B.verkv_sync(eng.ctx)
        B.verkv_profile_enable(eng.ctx, 1)
        for _ in range(steps):
            step()
        launches, total_ms = B.verkv_profile_read(eng.ctx)
        B.verkv_profile_enable(eng.ctx, 0)
        B.verkv_sync(eng.ctx)
    cnt = eng.p_count.cpu().numpy().astype(np.int64)
    nbytes, n_l = estimator_bytes(cnt, eng.p_r.cpu().numpy(), d, G)
    k = B.VERKV_K_PARTIAL_PIVOTAL
    us = 1e3 * total_ms[k] / max(launches[k], 1)
    gbs = nbytes / (us * 1e-6) / 1e9
    eng.close()
    del eng, tau, kv, host_kv, queries
    torch.cuda.empty_cache()
    return {
        "workload": f"shrinkage-estimator pass over the pivotal set: batch {batch} x 8 KV heads x "
                    "4 query heads, d=128, n=32768, bf16, eta=1/16, H=4+512, eps=delta=0.05, "
                    "MEMCPY fetch mode (the pass is its own launch), eager",
        "l2": "pivotal rows larger than L2; the sketch stream flushes it each pass",
        "kernel": "k_partial(pivotal)", "launches": int(launches[k]), "avg_us": round(us, 3),
        "pivotal_rows_per_call": int(cnt.sum()), "sampled_rows_per_call": n_l,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(gbs / peak, 4), "avg_us": round(us, 3),
                     "algorithmic_bytes_per_launch": nbytes,
                     "traffic": traffic_for("k_partial(pivotal)"), "peak_source": peak_src},
        "per_kernel_us": {B.verkv_kernel_name(j): round(1e3 * total_ms[j] / launches[j], 2)
                          for j in range(B.VERKV_K_COUNT) if launches[j] > 0}}


def measure_memcpy_fetch(w, pcs_unused, queries, steps_q, dev, link):
    """The literal cudaMemcpyAsync fetch path on the benchmark workload: VERKV_FETCH_MEMCPY (the host
    waits for the selection, host threads gather the selected V rows into page-locked staging,
    cudaMemcpyAsync moves them on the side stream, then the staged rows are summed).  Eager calls
    over `steps_q` queries with per-launch events on both streams; per query the pivotal sums
    (main stream) against the gather and the copies (side stream).  Returns a dict."""
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B
    from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap

    stream = torch.cuda.Stream(dev)
    Q = min(steps_q, queries.shape[0])
    hq = w.B * w.h_kv * w.G
    with torch.cuda.stream(stream):
        eng = VerKV(w.B, w.L, w.h_kv, w.G, w.d, w.n, default_cap(w.n, w.eta),
                    fetch_mode=B.VERKV_FETCH_MEMCPY)
        eng.load(w.tau.reshape(-1, w.n), w.kv.reshape(-1, w.n, 2, w.d))
        eng.compress(w.eta, w.n_sink, w.n_local, w.seed)
        eng.sync()
        o = torch.empty((hq, w.d), dtype=torch.float32, device=dev)
        counts = torch.zeros((w.B * w.h_kv,), dtype=torch.int32, device=dev)

        def query(t):
            B.verkv_attend_verified(eng.ctx, int(w.query_layer[t]), queries[t].data_ptr(),
                                    eng.pivotal, eng.r_full.data_ptr(), eng.sketch_desc, w.eps,
                                    w.delta, None, counts.data_ptr())
            B.verkv_fetch_refine(eng.ctx, None, counts.data_ptr(), eng.host_kv.data_ptr(),
                                 o.data_ptr(), None, None)

        for t in range(4):
            query(t)
        B.verkv_sync(eng.ctx)
        torch.cuda.synchronize()
        rows = 0
        piv, gat, cop, call = [], [], [], []
        t0 = time.perf_counter()
        B.verkv_profile_enable(eng.ctx, 1)
        for t in range(Q):
            query(t)
            recs = B.verkv_profile_timeline(eng.ctx)
            rows += int(counts.cpu().numpy().sum())
            by = {}
            for kid, a, b in recs:
                by.setdefault(kid, []).append((a, b))
            piv.append(by[B.VERKV_K_PARTIAL_PIVOTAL][0])
            gat.append(by[B.VERKV_K_FETCH_GATHER][0])
            cop.append(by.get(B.VERKV_K_FETCH_COPY, [(0.0, 0.0)])[0])
            call.append((recs[0][1], recs[-1][2]))
            B.verkv_profile_read(eng.ctx)  # discard the records
        wall = time.perf_counter() - t0
        B.verkv_profile_enable(eng.ctx, 0)
        B.verkv_sync(eng.ctx)
    eng.close()
    row_bytes = 2 * w.d  # V rows: the exact sketch holds the keys
    copy_ms = sum(b - a for a, b in cop)
    gather_ms = sum(b - a for a, b in gat)
    piv_ms = sum(b - a for a, b in piv)
    # the pivotal sums (main stream) overlapped with the fetch: gather start .. copies' end
    overlap_ms = sum(max(0.0, min(pb, cb) - max(pa, ga))
                     for (pa, pb), (ga, _), (_, cb) in zip(piv, gat, cop))
    h2d = rows * row_bytes
    return {
        "workload": "the benchmark workload (single-layer 32K, batch 1) in VERKV_FETCH_MEMCPY mode, "
                    f"{Q} queries, eager calls with events on both streams",
        "h2d_bytes": int(h2d), "copy_ms": round(copy_ms, 3),
        "copy_GBs": round(h2d / (copy_ms * 1e-3) / 1e9, 1) if copy_ms > 0 else None,
        "link_peak_GBs": round(link, 1),
        "copy_frac_of_link": round(h2d / (copy_ms * 1e-3) / 1e9 / link, 4) if copy_ms > 0 else None,
        "gather_ms": round(gather_ms, 3),
        "gather_GBs": round(h2d / (gather_ms * 1e-3) / 1e9, 1) if gather_ms > 0 else None,
        "pivotal_sums_ms": round(piv_ms, 3),
        "pivotal_sums_overlapped_with_fetch_ms": round(overlap_ms, 3),
        "pivotal_sums_overlap_frac": round(overlap_ms / piv_ms, 4) if piv_ms > 0 else None,
        "gpu_ms_per_query": round(sum(b - a for a, b in call) / Q, 4),
        "queries_per_s_eager": round(Q / wall, 1),
        "note": "per query: k_partial(pivotal) on the main stream starts when the selection is done; "
                "the host gather (bracketed by events on the idle side stream) and the side-stream "
                "copies run meanwhile; overlap = time the pivotal sums ran inside [gather start, "
                "copies end]"}


def run_estimator(args, local):
    """One GPU: the shrinkage-estimator pass over the pivotal set alone (measure_estimator at
    --est-batch).  One JSON line."""
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B

    B.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    r = measure_estimator(args.est_batch, args.steps, args.warmup, dev)
    print(json.dumps({"workload": "estimator", "unit": "GB/s", "steps": args.steps,
                      "warmup": args.warmup, "data": "synthetic",
                      "config": {"workload": r["workload"], "l2": r["l2"]}, **{
                          k: v for k, v in r.items() if k not in ("workload", "l2")}}),
          flush=True)


def run_dense_offload(args, local):
    """One GPU: the offloaded-dense baseline on the bench workload, one JSON line."""
    import torch

    from verified_kv_cache_poissoncomp_gb300 import binding as B
    from verified_kv_cache_poissoncomp_gb300 import inputs as I
    from verified_kv_cache_poissoncomp_gb300.engine import VerKV, default_cap

    B.lib()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = I.single_layer_32k(layers=LAYERS, n_queries=args.queries)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        eng = VerKV(w.B, w.L, w.h_kv, w.G, w.d, w.n, default_cap(w.n, w.eta))
        eng.load(w.tau.reshape(-1, w.n), w.kv.reshape(-1, w.n, 2, w.d))
        q_dev = torch.as_tensor(w.queries.view(np.int16)).to(dev)
    r = time_dense_offload(eng, w, q_dev, stream, args.steps, args.warmup)
    print(json.dumps({"baseline": "dense-offload", "metric": METRIC, "unit": UNIT,
                      "value": r["queries_per_s"], "steps": args.steps, "warmup": args.warmup,
                      "data": "synthetic", "dtype": "bf16",
                      "config": {"workload": "single-layer 32K (the bench workload), "
                                             f"{w.queries.shape[0]} decode queries per step; "
                                             "exact attention, every K|V row read from the "
                                             "page-locked host cache", "graph": True},
                      **r}), flush=True)
    eng.close()


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.eps_sweep:
        if rank == 0:
            run_eps_sweep(args, local)
    elif args.dense_offload:
        if rank == 0:
            run_dense_offload(args, local)
    elif args.pc_sweep:
        if rank == 0:
            run_pc_sweep(args, local)
    elif args.long128k:
        if rank == 0:
            run_model_steps(args, local, "long128k")
    elif args.decode_step:
        if rank == 0:
            run_model_steps(args, local, "decode-step")
    elif args.estimator:
        if rank == 0:
            run_estimator(args, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
