#!/usr/bin/env python3
"""Benchmark of the tile-synchronised dependent GEMM chain on GB300.

One step = one run of the whole hot path on one batch of synthetic input: the
chain's semaphores counting up by one run, the producer GEMM with its fused GeLU
epilogue publishing tiles, and the consumer GEMM waiting on them -- one persistent
kernel launch (plus the sentinel fill under the sentinel policy).  The headline
workload is the GPT-3-shaped MLP slice X[256,12288] . W1[12288,6144] -> GeLU ->
. W2[6144,12288] (bf16, fp32 accumulation), timed with CUDA events on the launching
stream for the best tile-synchronisation policy, next to the stream-serialised
two-kernel chain.  The timed runs are replayed from CUDA graphs (captured library
calls) unless --no-graph is given; the end-to-end figure calls the library directly.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead
(on the host cores, a bounded sample of the same workload per step).
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs and TFLOP/s per dependent GEMM chain vs stream-serialised; % of BF16 peak"
UNIT = "TFLOP/s"
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 7900.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Pages' own number for this workload: MLP, batch 256, TileSync, 840 us per chain on a
# Tesla V100 in fp16 ([cuSync] Table tab:waves:mlp).  Context on other hardware.
PAGES_US_B256 = 840.0
# DRAM bytes (read + write) per launch of the fused chain kernel from one ncu capture
# (profiles/chain_kernel_full_<workload>_*.md), valid only for the kernel sources the
# capture was taken on (kernel_source_hash).
NCU_TRAFFIC = {
    # (workload, policy, launch, tile_n, CTAs per tile): (dram__bytes_read.sum +
    # dram__bytes_write.sum per launch of the chain kernel, hash of the kernel sources the
    # capture was taken with)
    ("gpt3_mlp_m256", "ROW", "persistent", 256, 2): (309893632 + 19175936, "0e8c2701ee15b22d"),
    ("gpt3_mlp_m1024", "ROW", "persistent", 256, 2): (554258432 + 31390464, "0e8c2701ee15b22d"),
    ("gpt3_mlp_m1024", "SENTINEL", "persistent", 256, 2): (553572864 + 35731200, "0e8c2701ee15b22d"),
    ("gpt3_mlp_m256", "SENTINEL", "persistent", 256, 2): (313405696 + 20307712, "0e8c2701ee15b22d"),
}

# DRAM bytes (read + write) of one fused RowSync launch with the planner's defaults, per
# workload, from `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum -k regex:chain_kernel
# -s 3 -c 1 python bench.py --workload W --policies ROW --profile-runs 2`, with the hash of the
# kernel sources of the capture (reported in the per-configuration table only while it matches).
NCU_ROW_TRAFFIC = {
    "mlp_tiny_m64": (1212928 + 0, "0e8c2701ee15b22d"),
    "gpt3_mlp_m512": (531374336 + 29944576, "0e8c2701ee15b22d"),
    "gpt3_mlp_m1024": (554258432 + 31390464, "0e8c2701ee15b22d"),
    "gpt3_mlp_m2048": (725913088 + 74533888, "0e8c2701ee15b22d"),
    "gpt3_mlp_m4096": (1035433216 + 153161472, "0e8c2701ee15b22d"),
    "swiglu_m256": (181392640 + 5762304, "0e8c2701ee15b22d"),
    "swiglu_m1024": (307443968 + 14522112, "0e8c2701ee15b22d"),
    "conv_resnet14_n32": (5716992 + 6656, "0e8c2701ee15b22d"),
    "gpt3_attn_m256": (157476352 + 4235008, "0e8c2701ee15b22d"),
    "gpt3_attn_m1024": (295312384 + 36664064, "0e8c2701ee15b22d"),
}


def kernel_source_hash():
    """Hash of the sources that decide what a launch does: the kernels, their geometry and
    the planner and launcher.  The latency model (policy_model.h) only resolves AUTO, which
    the recorded captures do not use, so it is left out."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tile_level_sync_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name == "policy_model.h":
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, policy, launch, tile_n, pair):
    rec = NCU_TRAFFIC.get((workload, policy, launch, tile_n, pair))
    if rec and rec[1] == kernel_source_hash():
        return rec[0]
    return None


def reduce_max(value, device):
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step, world, ms_per_step):
    """Whole-job TFLOP/s: every rank ran the same step; time is the slowest rank's."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="gpt3_mlp_m256")
    p.add_argument("--policies", default="ROW,TILE,STRIDED,SENTINEL")
    p.add_argument("--launch", default="persistent", choices=["persistent", "pdl"])
    p.add_argument("--tile-n", type=int, default=0)
    p.add_argument("--raster", type=int, default=0)
    p.add_argument("--l2-prefetch", type=int, default=0)
    p.add_argument("--cta-pair", type=int, default=0)
    p.add_argument("--ksplit", type=int, default=0, help="producer K split (0 = the planner's choice)")
    p.add_argument("--ksplit-skew", type=int, default=0, help="graded producer K split: k-blocks each unit "
                   "adds to the one before it (0 = the planner's choice, -1 = equal units)")
    p.add_argument("--no-run-overlap", action="store_true", help="launch each run's first kernel in plain "
                   "stream order (CUSYNC_FLAG_NO_RUN_OVERLAP)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true", help="skip the per-configuration table")
    p.add_argument("--no-graph", action="store_true", help="one library call per run in the timed loops "
                   "instead of replaying the runs from CUDA graphs")
    p.add_argument("--sweep-out", default="", help="also time every policy/launch/tile of each workload "
                   "in the comma list --sweep and write the results to this JSON file")
    p.add_argument("--sweep", default="")
    p.add_argument("--trace-out", default="", help="also run STREAM and each listed policy once with the "
                   "in-kernel per-tile trace and write timeline statistics to this JSON file")
    p.add_argument("--profile-runs", type=int, default=0, help="only run the first policy of --policies this many "
                   "times after 3 warm-up runs (for a profiler), then exit without a bench line")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples (every 200 ms) with host timestamps, for the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inwin = [p for (t, p) in self.samples if t0 <= t <= t1]
        used = inwin
        note = "samples inside the timed region"
        if len(inwin) < 1 and self.samples:
            # region shorter than the sampling period: nearest samples around it
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:2]
            used = [p for (_, p) in near]
            note = "timed region shorter than the 200 ms sampling period: nearest samples"
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in used if num(p[1]) is not None]
        smax = [num(p[2]) for p in used if num(p[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in used:
            for name, v in zip(names, p[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(used), "note": note,
                "power_w_max": max([num(p[3]) or 0.0 for p in used])}


# ---------------------------------------------------------------------------- CPU oracle


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count() or 1


def oracle_sample_runner(wl, inputs):
    """Return (fn(rows) -> flops, rows_total): the oracle on a subset of token rows."""
    from oracle import chains
    from tile_level_sync_gb300 import synth

    d = wl.dims
    if wl.kind == "mlp_gelu":
        X, W1, W2 = (synth.f64(t) for t in inputs)

        def fn(rows):
            chains.mlp_gelu_rows(X, W1, W2, rows)
            return 2.0 * len(rows) * d["K"] * d["N1"] + 2.0 * len(rows) * d["N1"] * d["N2"]
        return fn, d["M"]
    if wl.kind == "mlp_swiglu":
        X, Wg, Wu, Wd = (synth.f64(t) for t in inputs)

        def fn(rows):
            chains.mlp_swiglu_rows(X, Wg, Wu, Wd, rows)
            return 2.0 * len(rows) * d["K"] * 2 * d["N1"] + 2.0 * len(rows) * d["N1"] * d["N2"]
        return fn, d["M"]
    if wl.kind == "attention":
        X, Wqkv, W2 = (synth.f64(t) for t in inputs)

        def fn(rows):
            chains.attention_rows(X, Wqkv, W2, rows)
            return 2.0 * len(rows) * d["K"] * 3 * d["N1"] + 2.0 * len(rows) * d["N1"] * d["N2"]
        return fn, d["M"]
    if wl.kind == "conv_stack":
        x, wt = (synth.f64(t) for t in inputs)
        ws = [wt[s] for s in range(d["S"])]

        def fn(rows):  # rows = images
            chains.conv_stack(x[rows], ws)
            return wl.gemm_flops() * len(rows) / d["N"]
        return fn, d["N"]
    x, w1, w2 = (synth.f64(t) for t in inputs)

    def fn(rows):  # rows = images
        chains.conv_relu_chain(x[rows], w1, w2)
        return wl.gemm_flops() * len(rows) / d["N"]
    return fn, d["N"]


def time_oracle(wl, inputs, budget_s=10.0):
    """The oracle on a bounded sample of the workload: evenly spaced token rows (images),
    as many as one pass of about budget_s takes, evaluated in passes until budget_s of CPU
    time has elapsed."""
    fn, total = oracle_sample_runner(wl, inputs)
    import numpy as np
    rows = list(range(total))
    t0 = time.perf_counter()
    fn(rows[:1])
    t1 = time.perf_counter() - t0
    n = int(max(1, min(total, budget_s / max(t1, 1e-6))))
    sel = list(np.linspace(0, total - 1, n).astype(int))
    flops, passes = 0.0, 0
    t0 = time.perf_counter()
    while True:
        flops += fn(sel)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or passes >= 1000:
            break
    unit = "images" if wl.kind in ("conv_relu", "conv_stack") else "token rows"
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{passes} passes over {n} of {total} {unit} of {wl.name}, fp64 numpy oracle, {dt:.2f} s"}


def run_reference(a):
    """The CPU oracle as the reference arm: each step a bounded sample of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from tile_level_sync_gb300 import synth
    import numpy as np
    wl = synth.WORKLOADS[a.workload]
    inputs = synth.workload_inputs(wl, seed=0)
    fn, total = oracle_sample_runner(wl, inputs)
    t0 = time.perf_counter()
    fn([0])
    t_row = max(time.perf_counter() - t0, 1e-6)
    budget = 90.0
    per_step = int(max(1, min(total, budget / ((a.steps + a.warmup) * t_row))))
    sel = list(np.linspace(0, total - 1, per_step).astype(int))
    for _ in range(a.warmup):
        fn(sel)
    t0 = time.perf_counter()
    flops = 0.0
    for _ in range(a.steps):
        flops += fn(sel)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    unit_name = "images" if wl.kind in ("conv_relu", "conv_stack") else "token rows"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": dt / a.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, **wl.dims, "parallelism": "replicas only"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{per_step} of {total} {unit_name} of {wl.name} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- GPU arm


class Setup:
    """Device operands and chains of one workload."""

    def __init__(self, wl, inputs, tile_n, launch, raster=0, l2_prefetch=0, cta_pair=0, ksplit=0, flags=0,
                 ksplit_skew=0):
        import torch
        import tile_level_sync_gb300 as cs
        self.cs = cs
        self.wl = wl
        d = wl.dims
        dev = "cuda"
        if wl.kind == "conv_stack":
            x, wt = inputs
            self.a = x.to(dev)
            self.b0 = wt.contiguous().to(dev)
            self.b1 = None
            self.base = dict(kind=cs.CHAIN_CONV_STACK, n=d["N"], h=d["H"], w=d["W"], c=d["C"], stages=d["S"])
            # a workspace for the largest plan: under the sentinel policy two sets of one
            # buffer per intermediate (cusync_chain_info_t::work_bytes)
            self.h = torch.empty((2 * (d["S"] - 1) * d["N"] * d["H"] * d["W"] * d["C"],), dtype=torch.bfloat16,
                                 device=dev)
            self.y = torch.empty((d["N"], d["H"], d["W"], d["C"]), dtype=torch.bfloat16, device=dev)
            self.x_host = x
        elif wl.kind == "conv_relu":
            x, w1, w2 = inputs
            self.a = x.to(dev)
            self.b0 = w1.contiguous().to(dev)
            self.b1 = w2.contiguous().to(dev)
            self.h = torch.empty((d["N"], d["H"], d["W"], d["K"]), dtype=torch.bfloat16, device=dev)
            self.y = torch.empty_like(self.h)
            self.x_host = x
            self.base = dict(kind=cs.CHAIN_CONV_RELU, n=d["N"], h=d["H"], w=d["W"], c=d["C"], k_out=d["K"])
        elif wl.kind == "attention":
            X, Wqkv, W2 = inputs
            self.a = X.to(dev)
            self.b0 = Wqkv.t().contiguous().to(dev)
            self.b1 = W2.t().contiguous().to(dev)
            self.h = torch.empty((d["M"], 3 * d["N1"]), dtype=torch.bfloat16, device=dev)
            self.h2 = torch.empty((d["M"], d["N1"]), dtype=torch.bfloat16, device=dev)
            self.y = torch.empty((d["M"], d["N2"]), dtype=torch.bfloat16, device=dev)
            self.x_host = X
            self.base = dict(kind=cs.CHAIN_ATTENTION, M=d["M"], K=d["K"], N1=d["N1"], N2=d["N2"])
        else:
            if wl.kind == "mlp_gelu":
                X, W1, W2 = inputs
                W1t = W1.t().contiguous()
                kind = cs.CHAIN_MLP_GELU
            else:
                X, Wg, Wu, W2 = inputs
                W1t = torch.cat([Wg.t(), Wu.t()], 0).contiguous()
                kind = cs.CHAIN_MLP_SWIGLU
            self.a = X.to(dev)
            self.b0 = W1t.to(dev)
            self.b1 = W2.t().contiguous().to(dev)
            self.h = torch.empty((d["M"], d["N1"]), dtype=torch.bfloat16, device=dev)
            self.y = torch.empty((d["M"], d["N2"]), dtype=torch.bfloat16, device=dev)
            self.x_host = X
            self.base = dict(kind=kind, M=d["M"], K=d["K"], N1=d["N1"], N2=d["N2"])
        self.tile_n = tile_n
        self.launch = launch
        self.raster = raster
        self.l2_prefetch = l2_prefetch
        self.cta_pair = cta_pair
        self.ksplit = ksplit
        self.ksplit_skew = ksplit_skew
        self.flags = flags
        self.chains = {}

    def chain(self, policy, launch=None, tile_n=None, raster=None, l2_prefetch=None, cta_pair=None, flags=0):
        cs = self.cs
        launch = self.launch if launch is None else launch
        tile_n = self.tile_n if tile_n is None else tile_n
        raster = self.raster if raster is None else raster
        l2_prefetch = self.l2_prefetch if l2_prefetch is None else l2_prefetch
        cta_pair = self.cta_pair if cta_pair is None else cta_pair
        key = (policy, launch, tile_n, raster, l2_prefetch, cta_pair, flags)
        if key not in self.chains:
            self.chains[key] = cs.Chain(cs.make_desc(policy=policy, launch=launch, tile_n=tile_n, raster_rows=raster,
                                                     l2_prefetch=l2_prefetch, cta_pair=cta_pair,
                                                     flags=flags | self.flags, ksplit=self.ksplit,
                                                     ksplit_skew=self.ksplit_skew, **self.base))
        return self.chains[key]

    def run(self, ch):
        ch.run(self.a, self.b0, self.b1, self.h, self.y, h2=getattr(self, "h2", None))

    def kernels_per_run(self, policy, launch):
        stages = 3 if self.base["kind"] == self.cs.CHAIN_ATTENTION else self.base.get("stages", 2)
        n = stages if (policy == "STREAM" or launch == self.cs.LAUNCH_PDL) else 1
        return n + (1 if policy == "SENTINEL" else 0)


class ChainGraph:
    """n runs of one chain recorded by CUDA stream capture (groups of up to `group` runs
    per graph), so that replaying them costs one graph launch per group instead of one
    library call and two or three kernel launches per run from the host."""

    def __init__(self, torch, setup, ch, n, group=50):
        self.torch = torch
        self.graphs = []
        left = n
        while left > 0:
            k = min(group, left)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(k):
                    setup.run(ch)
            self.graphs.append(g)
            left -= k
        torch.cuda.synchronize()

    def replay(self):
        for g in self.graphs:
            g.replay()


def run_steps(torch, setup, ch, n, graph):
    """Enqueue n runs: from a captured graph, or one library call per run."""
    if graph is not None:
        graph.replay()
    else:
        for _ in range(n):
            setup.run(ch)


def time_runs(torch, setup, ch, n, use_graph=True):
    """Mean ms per run over n back-to-back runs (events on the launching stream)."""
    graph = ChainGraph(torch, setup, ch, n) if use_graph else None
    if graph is not None:
        graph.replay()          # warm the instantiated graphs
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    run_steps(torch, setup, ch, n, graph)
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def per_launch_ms(torch, setup, ch, n):
    """Mean device duration of a single run, each bracketed by its own events."""
    s = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(s)
        setup.run(ch)
        b.record(s)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def trace_stats(torch, setup, policy, launch):
    """One traced run of `policy`: the per-tile timeline (claim, dependencies met, first
    and last MMA, epilogue done) reduced to the figures that explain a chain's time.

    * mainloop ns per k-block (median over tiles) and epilogue us, per stage;
    * consumer wait: dependencies met minus claim, per consumer tile (us);
    * SM activity: SMs with a tile in flight, sampled every 0.5 us over the run, as a
      fraction of the SMs the plan uses; and the same fraction inside the last-wave window,
      from the last tile claim to the end of the run (the tail that wave quantisation
      leaves idle).
    """
    import numpy as np
    cs = setup.cs
    d = cs.make_desc(policy=policy, launch=launch, tile_n=setup.tile_n, raster_rows=setup.raster,
                     l2_prefetch=setup.l2_prefetch, cta_pair=setup.cta_pair, ksplit=setup.ksplit,
                     ksplit_skew=setup.ksplit_skew, flags=cs.FLAG_TRACE, **setup.base)
    ch = cs.Chain(d)
    try:
        for _ in range(3):
            setup.run(ch)
        torch.cuda.synchronize()
        setup.run(ch)
        torch.cuda.synchronize()
        st, code, _ = ch.check()
        if st != cs.OK:
            raise RuntimeError(f"traced {policy}: {cs.status_string(st)} 0x{code:08x}")
        recs = ch.trace()
        info = ch.info()
    finally:
        ch.close()
    stage = np.array([r["stage"] for r in recs])
    t0 = min(r["t_claim"] for r in recs)
    T = {k: (np.array([r[k] for r in recs], dtype=np.float64) - t0) / 1e3
         for k in ("t_claim", "t_ready", "t_mma0", "t_mma1", "t_epi")}
    end = float(T["t_epi"].max())
    sms = int(info.num_sms)
    ts = np.arange(0.0, end, 0.5)
    per_sm = {}
    for r, a, b in zip(recs, T["t_claim"], T["t_epi"]):
        m = per_sm.setdefault(r["smid"], np.zeros(len(ts), dtype=bool))
        m |= (ts >= a) & (ts < b)    # an SM is busy while any of its tiles is in flight
    busy = np.sum(list(per_sm.values()), axis=0).astype(np.float64) if per_sm else np.zeros(len(ts))
    busy *= info.cta_pair            # a pair tile is recorded by its leader and occupies two SMs
    tail = ts >= float(T["t_claim"].max())
    out = {"policy": policy, "launch": "pdl" if launch == cs.LAUNCH_PDL else "persistent", "span_us": end,
           "tiles": [int((stage == 0).sum()), int((stage == 1).sum())], "sms": sms, "cta_pair": int(info.cta_pair),
           "sm_active_frac": float(busy.mean() / sms) if len(ts) else None,
           "last_wave_window_us": float(end - T["t_claim"].max()),
           "sm_active_frac_last_wave": float(busy[tail].mean() / sms) if tail.any() else None}
    for s in (0, 1):
        sel = stage == s
        kb = info.k_blocks[s]
        out[f"stage{s}"] = {"ns_per_kblock": float(np.median((T["t_mma1"] - T["t_mma0"])[sel] / kb * 1e3)),
                            "epilogue_us": float(np.median((T["t_epi"] - T["t_mma1"])[sel]))}
    w = (T["t_ready"] - T["t_claim"])[stage == 1]
    out["consumer_wait_us"] = {"median": float(np.median(w)), "p90": float(np.percentile(w, 90)),
                               "max": float(w.max())}
    # debug counters per consumer tile: semaphore reads of its waits (probes and polls),
    # A k-blocks loaded again under the sentinel check, and the MMA issuer's SM cycles
    # spent waiting for stages (landed, or checked) and the checkers' cycles, per k-block
    cons = [r for r in recs if r["stage"] == 1]
    kb1 = max(1, info.k_blocks[1])
    polls = np.array([r["polls"] for r in cons], dtype=np.float64)
    out["consumer_polls"] = {"median": float(np.median(polls)), "max": float(polls.max())}
    out["sentinel_reloads"] = {"total": int(sum(r["reloads"] for r in cons)),
                               "max_per_tile": int(max(r["reloads"] for r in cons))}
    out["consumer_clk_per_kblock"] = {
        "mma_wait": float(np.median([r["land_clk"] / kb1 for r in cons])),
        "check": float(np.median([r["check_clk"] / kb1 for r in cons]))}
    return out


def algorithmic_bytes(wl):
    d = wl.dims
    if wl.kind == "conv_relu":
        pix = d["N"] * d["H"] * d["W"]
        return 2 * (pix * d["C"] + 9 * d["C"] * d["K"] + 2 * pix * d["K"] + 9 * d["K"] * d["K"] + pix * d["K"])
    if wl.kind == "conv_stack":   # x and y once, each intermediate written once and read once
        act = d["N"] * d["H"] * d["W"] * d["C"]
        return 2 * (2 * act + 2 * (d["S"] - 1) * act + d["S"] * 9 * d["C"] * d["C"])
    if wl.kind == "attention":   # XQKV and XDot each written once and read once
        return 2 * (d["M"] * d["K"] + d["K"] * 3 * d["N1"] + 2 * d["M"] * 3 * d["N1"] + 2 * d["M"] * d["N1"]
                    + d["N1"] * d["N2"] + d["M"] * d["N2"])
    n1w = 2 * d["N1"] if wl.kind == "mlp_swiglu" else d["N1"]
    return 2 * (d["M"] * d["K"] + d["K"] * n1w + 2 * d["M"] * d["N1"] + d["N1"] * d["N2"] + d["M"] * d["N2"])


def check_output(setup, wl, inputs):
    """Sampled rows of the timed workload's output against the oracle."""
    import numpy as np
    from oracle import chains
    from tile_level_sync_gb300 import synth
    d = wl.dims
    Y = setup.y.float().cpu().double().numpy()
    scale = 1.0
    if wl.kind == "conv_stack":
        # end to end through S bf16 roundings: the pair's bound times sqrt(S - 1)
        x, wt = (synth.f64(t) for t in inputs)
        imgs = [0, d["N"] - 1]
        _, ref = chains.conv_stack(x[imgs], [wt[s] for s in range(d["S"])])
        got = Y[imgs]
        scale = float(np.sqrt(d["S"] - 1))
    elif wl.kind == "conv_relu":
        x, w1, w2 = (synth.f64(t) for t in inputs)
        imgs = [0, d["N"] - 1]
        _, ref = chains.conv_relu_chain(x[imgs], w1, w2)
        got = Y[imgs]
    else:
        rows = sorted(set([0, 1, d["M"] // 2, d["M"] - 1]))
        if wl.kind == "mlp_gelu":
            _, ref = chains.mlp_gelu_rows(*(synth.f64(t) for t in inputs), rows)
        elif wl.kind == "attention":
            _, _, ref = chains.attention_rows(*(synth.f64(t) for t in inputs), rows)
        else:
            _, ref = chains.mlp_swiglu_rows(*(synth.f64(t) for t in inputs), rows)
        got = Y[rows]
    bound = scale * 2e-2 * np.maximum(1.0, np.abs(ref))
    return bool(np.all(np.abs(got - ref) <= bound))


# Configurations reported beside the headline, each with its own policies and timing
# (the headline workload is timed in the main region).
PER_CONFIG = ["mlp_tiny_m64", "gpt3_mlp_m512", "gpt3_mlp_m1024", "gpt3_mlp_m2048", "gpt3_mlp_m4096",
              "swiglu_m256", "swiglu_m1024", "conv_resnet14_n32"]


def sampled_rows(M):
    """First and last token row of every 256-row tile."""
    rows = set()
    for t0 in range(0, M, 256):
        rows.update((t0, min(t0 + 255, M - 1)))
    return sorted(rows)


def oracle_parity(setup, wl, inputs):
    """H and Y of the last run against the oracle on sampled rows (convolutions: the first,
    a middle and the last image), |err| <= 2e-2 max(1, |ref|)."""
    import numpy as np
    import torch
    from oracle import chains
    from tile_level_sync_gb300 import synth
    d = wl.dims

    def ok(got, ref):
        got = got.float().cpu().double().numpy()
        return bool(np.all(np.abs(got - ref) <= 2e-2 * np.maximum(1.0, np.abs(ref))))

    if wl.kind == "conv_relu":
        x, w1, w2 = inputs
        imgs = [0, d["N"] // 2, d["N"] - 1]
        h_ref, y_ref = chains.conv_relu_chain(synth.f64(x[imgs]), synth.f64(w1), synth.f64(w2))
        return ok(setup.h[imgs], h_ref) and ok(setup.y[imgs], y_ref), f"images {imgs}"
    rows = sampled_rows(d["M"])
    idx = torch.tensor(rows)
    if wl.kind == "mlp_gelu":
        X, W1, W2 = inputs
        h_ref, y_ref = chains.mlp_gelu(synth.f64(X[idx]), synth.f64(W1), synth.f64(W2))
    else:
        X, Wg, Wu, Wd = inputs
        h_ref, y_ref = chains.mlp_swiglu(synth.f64(X[idx]), synth.f64(Wg), synth.f64(Wu), synth.f64(Wd))
    dev = idx.to(setup.h.device)
    return ok(setup.h[dev], h_ref) and ok(setup.y[dev], y_ref), f"{len(rows)} token rows"


def per_config(torch, cs, synth, peaks):
    """The other benchmarked configurations with the planner's defaults: every
    synchronisation policy under both launch forms and the stream-serialised chain, each
    timed over back-to-back runs replayed from CUDA graphs.  Per configuration: the fastest
    tile-synchronised variant and the stream-serialised chain in us per chain, TFLOP/s and %
    of the measured BF16 peak, the planner's waves on 148 SMs, whether every variant wrote
    the same bytes of H and Y as the stream-serialised chain, and the best variant's H and
    Y against the oracle on sampled rows."""
    out = {}
    for name in PER_CONFIG:
        wl = synth.WORKLOADS[name]
        inputs = synth.workload_inputs(wl, seed=0)
        setup = Setup(wl, inputs, 0, cs.LAUNCH_PERSISTENT)
        flops = wl.gemm_flops()
        n = 40 if flops > 1e11 else 200
        us, identical, ref, graphs = {}, True, None, {}
        for pol in ("STREAM", "ROW", "TILE", "STRIDED", "SENTINEL"):
            for launch in (cs.LAUNCH_PERSISTENT, cs.LAUNCH_PDL):
                if pol == "STREAM" and launch == cs.LAUNCH_PDL:
                    continue
                key = pol + ("/pdl" if launch == cs.LAUNCH_PDL else "")
                try:
                    ch = setup.chain(pol, launch=launch)
                except cs.CusyncError:       # e.g. StridedSync needs n_tiles divisible by G
                    continue
                for _ in range(3):
                    setup.run(ch)
                st, code, _ = ch.check()
                if st != cs.OK:
                    us[key] = f"{cs.status_string(st)} 0x{code:08x}"
                    identical = False
                    continue
                hb, yb = setup.h.view(torch.int16), setup.y.view(torch.int16)
                if ref is None:
                    ref = (hb.clone(), yb.clone())
                elif not (torch.equal(hb, ref[0]) and torch.equal(yb, ref[1])):
                    identical = False
                graphs[key] = ChainGraph(torch, setup, ch, n)
                graphs[key].replay()   # uploads the graph: untimed
        # the variants in turn, several rounds, each variant's median: clock and power
        # state drift between back-to-back measurements would otherwise favour whichever
        # variant runs first
        s = torch.cuda.current_stream()
        samples = {k: [] for k in graphs}
        for _ in range(5):
            for key, g in graphs.items():
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(s)
                g.replay()
                e1.record(s)
                torch.cuda.synchronize()
                samples[key].append(e0.elapsed_time(e1) / n * 1e3)
        for key, v in samples.items():
            us[key] = statistics.median(v)
        del graphs
        timed = {k: v for k, v in us.items() if isinstance(v, float)}
        sync = {k: v for k, v in timed.items() if k != "STREAM"}
        best = min(sync, key=sync.get)
        pol, _, l = best.partition("/")
        ch = setup.chain(pol, launch=cs.LAUNCH_PDL if l == "pdl" else cs.LAUNCH_PERSISTENT)
        setup.run(ch)
        torch.cuda.synchronize()
        parity, sample = oracle_parity(setup, wl, inputs)
        info = ch.info()
        w148 = cs.cusync_plan_waves(cs.make_desc(policy=pol, num_sms=148, **setup.base))
        tflops = flops / (sync[best] * 1e-6) / 1e12
        out[name] = {
            "dims": wl.dims, "gflop": flops / 1e9, "best": best, "best_us": sync[best],
            "stream_us": timed.get("STREAM"), "speedup_vs_stream": timed["STREAM"] / sync[best] if "STREAM" in timed
            else None, "tflops": tflops, "pct_bf16_peak_measured": tflops / peaks["bf16_tflops"] * 100,
            "pct_bf16_sustained_peak_measured": tflops / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * 100,
            "tile": f"{info.tile_m}x{info.tile_n}x{info.tile_k}", "cta_pair": info.cta_pair, "ksplit": info.ksplit,
            "ksplit_skew": info.ksplit_skew, "us": us, "runs_timed": n, "timing": "median of 5 rounds over the variants in turn",
            "bit_identical_all_variants": identical,
            "parity_sampled": parity, "parity_sample": sample,
            "waves_148": {"tbs": list(w148.tbs), "waves": list(w148.waves), "stream_waves": w148.stream_waves,
                          "fused_waves": w148.fused_waves, "last_wave_tbs": w148.last_wave_tbs,
                          "util": list(w148.util)},
            "l2": "operands larger than L2" if algorithmic_bytes(wl) > 129e6 else "operands fit in L2 (not flushed)",
        }
        rec = NCU_ROW_TRAFFIC.get(name)
        if rec and rec[1] == kernel_source_hash():
            alg = algorithmic_bytes(wl)
            out[name]["dram_traffic_row_fused"] = {"bytes": rec[0], "algorithmic_bytes": alg, "ratio": rec[0] / alg,
                                                   "source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one "
                                                             "fused RowSync launch (planner defaults)"}
        for c in setup.chains.values():
            c.close()
        del setup, ref
        torch.cuda.empty_cache()
    return out


def main():
    a = parse()
    if a.impl == "reference":
        return run_reference(a)
    import numpy as np
    import torch
    import torch.distributed as dist
    import tile_level_sync_gb300 as cs
    from tile_level_sync_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    cs.load()

    wl = synth.WORKLOADS[a.workload]
    inputs = synth.workload_inputs(wl, seed=0)
    launch = cs.LAUNCH_PDL if a.launch == "pdl" else cs.LAUNCH_PERSISTENT
    setup = Setup(wl, inputs, a.tile_n, launch, a.raster, a.l2_prefetch, a.cta_pair, a.ksplit,
                  cs.FLAG_NO_RUN_OVERLAP if a.no_run_overlap else 0, a.ksplit_skew)
    flops = wl.gemm_flops()
    peaks, peak_src = load_peaks()

    pols = [p.strip().upper() for p in a.policies.split(",") if p.strip()]
    if a.profile_runs > 0:
        ch = setup.chain(pols[0])
        for _ in range(3 + a.profile_runs):
            setup.run(ch)
        st, code, _ = ch.check()
        ch.close()
        if st != cs.OK:
            raise RuntimeError(f"{pols[0]}: {cs.status_string(st)} 0x{code:08x}")
        return 0

    # warm every policy, then choose the fastest tile-synchronised one
    per_policy = {}
    for pol in pols + ["STREAM"]:
        try:
            ch = setup.chain(pol)
        except cs.CusyncError:        # e.g. StridedSync needs n_tiles divisible by G
            pols = [p for p in pols if p != pol]
            continue
        for _ in range(max(3, a.warmup)):
            setup.run(ch)
        st, code, detail = ch.check()
        if st != cs.OK:
            raise RuntimeError(f"{pol}: {cs.status_string(st)} 0x{code:08x}")
        per_policy[pol] = time_runs(torch, setup, ch, min(200, max(5, a.steps)), not a.no_graph)
    best = min(pols, key=lambda p: per_policy[p])
    ch = setup.chain(best)

    # ---- timed region: exactly K steps, barrier + synchronize on both sides
    graph = None if a.no_graph else ChainGraph(torch, setup, ch, a.steps)
    for _ in range(a.warmup):
        setup.run(ch)
    if graph is not None:
        graph.replay()      # the first launch of an instantiated graph uploads it: untimed
    sampler = ClockSampler(torch.cuda.current_device() if world > 1 else 0)
    sampler.start()
    time.sleep(0.5)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    e0.record(s)
    run_steps(torch, setup, ch, a.steps, graph)
    e1.record(s)
    torch.cuda.synchronize()
    t_host1 = time.time()
    del graph
    if world > 1:
        dist.barrier()
    time.sleep(0.3)
    sampler.stop()
    ms = reduce_max(e0.elapsed_time(e1), "cuda")
    ms_step = ms / a.steps
    st, code, _ = ch.check()
    if st != cs.OK:
        raise RuntimeError(f"timed run reported {cs.status_string(st)} 0x{code:08x}")
    parity_ok = check_output(setup, wl, inputs) if rank == 0 else None

    # ---- stream-serialised baseline, same tiles and k order, same number of steps
    ch_stream = setup.chain("STREAM")
    for _ in range(a.warmup):
        setup.run(ch_stream)
    stream_ms = time_runs(torch, setup, ch_stream, a.steps, not a.no_graph)

    # ---- dominant kernel: the fused chain kernel.  When a step is exactly one launch of it
    # (one persistent kernel, no sentinel fill), the timed region's events give its average
    # launch duration directly; otherwise each run is bracketed by its own events.
    if setup.kernels_per_run(best, launch) == 1:
        kern_ms, kern_src = ms_step, "timed region (one chain-kernel launch per step)"
    else:
        kern_ms, kern_src = per_launch_ms(torch, setup, ch, min(a.steps, 500)), "per-run events"
    alg_bytes = algorithmic_bytes(wl)
    hbm_gbs = alg_bytes / (kern_ms * 1e-3) / 1e9
    tflops_kernel = flops / (kern_ms * 1e-3) / 1e12
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    bound = "hbm" if flops / alg_bytes < ridge else "tensor"
    best_info = setup.chain(best).info()
    traffic = measured_traffic(wl.name, best, a.launch, best_info.tile_n, best_info.cta_pair)
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": hbm_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": hbm_gbs / peaks["hbm_gbs"], "traffic": traffic}
    else:
        roof = {"bound": "tensor", "achieved": tflops_kernel, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": tflops_kernel / peaks["bf16_tflops"], "traffic": traffic}
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["algorithmic_bytes"] = alg_bytes
    roof["kernel_ms"] = kern_ms
    roof["kernel_ms_source"] = kern_src
    roof["tensor_frac_of_measured"] = tflops_kernel / peaks["bf16_tflops"]

    # ---- end to end through the public API: H2D of X, the chain, D2H of Y, every step.
    # Sequential: one stream, copy in -> chain -> copy out.  Pipelined: two buffer sets and
    # two copy streams, so that step k+1's copy in and step k-1's copy out run while step
    # k's chain computes (each step still copies its own input in and its own result out).
    x_pin = setup.x_host.pin_memory()
    y_pin = torch.empty(setup.y.shape, dtype=torch.bfloat16).pin_memory()
    k_e2e = min(a.steps, 2000)
    for _ in range(3):
        setup.a.copy_(x_pin, non_blocking=True)
        setup.run(ch)
        y_pin.copy_(setup.y, non_blocking=True)
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(s)
    for _ in range(k_e2e):
        setup.a.copy_(x_pin, non_blocking=True)
        setup.run(ch)
        y_pin.copy_(setup.y, non_blocking=True)
    e3.record(s)
    torch.cuda.synchronize()
    e2e_seq_ms = e2.elapsed_time(e3) / k_e2e
    xs, ys = [setup.a, torch.empty_like(setup.a)], [setup.y, torch.empty_like(setup.y)]
    x_pins, y_pins = [x_pin, x_pin.clone().pin_memory()], [y_pin, torch.empty_like(y_pin).pin_memory()]
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    landed = [torch.cuda.Event(), torch.cuda.Event()]
    ran = [torch.cuda.Event(), torch.cuda.Event()]
    read = [torch.cuda.Event(), torch.cuda.Event()]

    def pipelined(k_steps):
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_start.record(s)
        cin.wait_stream(s)
        cout.wait_stream(s)
        for k in range(k_steps):
            i = k & 1
            with torch.cuda.stream(cin):
                if k >= 2:
                    cin.wait_event(ran[i])      # step k-2's chain has read xs[i]
                xs[i].copy_(x_pins[i], non_blocking=True)
                landed[i].record(cin)
            s.wait_event(landed[i])
            if k >= 2:
                s.wait_event(read[i])           # step k-2's copy out has read ys[i]
            setup.a, setup.y = xs[i], ys[i]
            setup.run(ch)
            ran[i].record(s)
            with torch.cuda.stream(cout):
                cout.wait_event(ran[i])
                y_pins[i].copy_(ys[i], non_blocking=True)
                read[i].record(cout)
        s.wait_stream(cout)
        s.wait_stream(cin)
        e_end.record(s)
        torch.cuda.synchronize()
        setup.a, setup.y = xs[0], ys[0]
        return e_start.elapsed_time(e_end) / k_steps

    pipelined(4)
    e2e_ms = pipelined(k_e2e)
    h2d = x_pin.numel() * 2
    d2h = y_pin.numel() * 2

    plan = cs.cusync_plan_waves(setup.chain(best).desc)
    plan148 = cs.cusync_plan_waves(cs.make_desc(policy=best, launch=launch, tile_n=a.tile_n, num_sms=148,
                                                cta_pair=a.cta_pair, ksplit=a.ksplit, ksplit_skew=a.ksplit_skew,
                                                **setup.base))
    info = setup.chain(best).info()

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = time_oracle(wl, inputs)

    configs = None
    if rank == 0 and world == 1 and not a.no_per_config:
        sampler2 = ClockSampler(0)
        sampler2.start()
        t_pc0 = time.time()
        configs = per_config(torch, cs, synth, peaks)
        t_pc1 = time.time()
        sampler2.stop()
        configs["clocks"] = sampler2.summary(t_pc0, t_pc1)

    clocks = sampler.summary(t_host0 - 0.05, t_host1 + 0.05)
    value = job_throughput(flops, world, ms_step)
    us = ms_step * 1e3
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": stream_ms / ms_step,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, **wl.dims, "policy": best, "launch": a.launch,
                   "tile": f"{info.tile_m}x{info.tile_n}x{info.tile_k}", "cta_pair": info.cta_pair,
                   "ksplit": info.ksplit, "ksplit_skew": info.ksplit_skew,
                   "parallelism": "replicas only",
                   "enqueue": "library call per run" if a.no_graph else "CUDA-graph replay, up to 50 captured runs (steps) per graph",
                   "l2": f"inputs {alg_bytes / 1e6:.0f} MB of operands > 129 MB L2; no flush between steps"
                   if alg_bytes > 129e6 else "inputs smaller than L2",
                   "vs_baseline_note": "speed-up over the stream-serialised chain (same kernel, tiles and k "
                                       "order, two launches) timed in this run"},
        "context_vs_pages_v100": (value / (flops / (PAGES_US_B256 * 1e-6) / 1e12)
                                  if wl.name == "gpt3_mlp_m256" else None),
        "us_per_chain": us,
        "stream_us_per_chain": stream_ms * 1e3,
        "speedup_vs_stream": stream_ms / ms_step,
        "policies_us": {k: v * 1e3 for k, v in per_policy.items()},
        "pct_bf16_peak": {"measured": value / world / peaks["bf16_tflops"] * 100,
                          "nominal": value / world / NOMINAL_BF16_TFLOPS * 100},
        "hbm_gbs_chain": alg_bytes / (ms_step * 1e-3) / 1e9,
        "waves": {"device_sms": plan.num_sms, "tbs": list(plan.tbs), "stream_waves": plan.stream_waves,
                  "fused_waves": plan.fused_waves, "last_wave_tbs": plan.last_wave_tbs,
                  "util": list(plan.util),
                  "sms148": {"stream_waves": plan148.stream_waves, "fused_waves": plan148.fused_waves,
                             "last_wave_tbs": plan148.last_wave_tbs, "util": list(plan148.util)}},
        "roofline": roof,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "sequential_ms_per_step": e2e_seq_ms,
                "note": "X copied in from pinned host memory and Y read back every step; weights resident; "
                        "two buffer sets, the copies of neighbouring steps overlap the chain (sequential: one "
                        "stream, copy in, chain, copy out)"},
        "gpu_launches": a.steps * setup.kernels_per_run(best, launch),
        "clocks": clocks,
        "parity_sampled_rows": parity_ok,
        "cpu_baseline": cpu,
        "per_config": configs,
    }
    if a.trace_out and rank == 0:
        traces = [trace_stats(torch, setup, "STREAM", cs.LAUNCH_PERSISTENT)]
        for pol in pols:
            traces.append(trace_stats(torch, setup, pol, launch))
        with open(a.trace_out, "w") as f:
            json.dump({"workload": wl.name, "traces": traces}, f, indent=1)
        line["trace_file"] = a.trace_out
    if a.sweep_out and rank == 0:
        line["sweep_file"] = a.sweep_out
        sweep(a, torch, cs, synth, a.sweep_out)
    for c in setup.chains.values():
        c.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def sweep(a, torch, cs, synth, out_path):
    """Every listed workload x tile width x (raster, L2 prefetch) x policy: us per chain.

    Written to a file; not a bench line."""
    names = [n for n in a.sweep.split(",") if n] or list(synth.WORKLOADS)
    results = []
    # (raster rows, L2 prefetch, CTAs per tile; 0 = the planner's choice): every policy and
    # launch mode on the planner's tiling, Stream/Row/Tile on the others
    variants = [(1, 0, 0), (1, 0, 1), (1, 0, 2), (16, 0, 0)]
    for name in names:
        wl = synth.WORKLOADS[name]
        inputs = synth.workload_inputs(wl, seed=0)
        for tile_n in (256, 128):
            setup = Setup(wl, inputs, tile_n, cs.LAUNCH_PERSISTENT)
            row = {"workload": name, "tile_n": tile_n, "gflop": wl.gemm_flops() / 1e9, "us": {}}
            for vi, (raster, pf, pair) in enumerate(variants):
                pols = ["STREAM", "ROW", "TILE", "STRIDED", "SENTINEL"] if vi == 0 else ["STREAM", "ROW", "TILE"]
                if wl.kind == "attention":   # its policies are Row, Tile, Strided+Tile
                    pols = ["STREAM", "ROW", "TILE", "STRIDED"]
                for pol in pols:
                    for launch in (cs.LAUNCH_PERSISTENT, cs.LAUNCH_PDL):
                        if launch == cs.LAUNCH_PDL and (pol == "STREAM" or (vi != 0 and wl.kind != "attention")):
                            continue
                        key = f"{pol}/{'pdl' if launch else 'pers'}/r{raster}/p{pair}"
                        try:
                            ch = setup.chain(pol, launch=launch, raster=raster, l2_prefetch=pf, cta_pair=pair)
                        except cs.CusyncError as e:
                            row["us"][key] = str(e)
                            continue
                        for _ in range(5):
                            setup.run(ch)
                        st, code, _ = ch.check()
                        n = 50 if wl.gemm_flops() > 1e11 else 200
                        ms = time_runs(torch, setup, ch, n, not a.no_graph)
                        row["us"][key] = ms * 1e3 if st == cs.OK else f"status {st}"
                        pk = f"r{raster}/p{pair}"
                        if pk not in row.setdefault("predicted_us", {}):
                            try:
                                pred = cs.cusync_predict_policies(ch.desc)
                                row["predicted_us"][pk] = {n_: pred.us[i] for n_, i in cs.POLICY_NAMES.items()
                                                           if i < 5}
                            except cs.CusyncError:   # the model covers two-stage chains
                                row["predicted_us"][pk] = None
                for c in list(setup.chains.values()):
                    c.close()
                setup.chains = {}
            plan = cs.cusync_plan_waves(setup.chain("ROW").desc)
            row["waves"] = {"tbs": list(plan.tbs), "stream": plan.stream_waves, "fused": plan.fused_waves,
                            "last_wave_tbs": plan.last_wave_tbs, "sms": plan.num_sms}
            for c in setup.chains.values():
                c.close()
            results.append(row)
            print(json.dumps(row), file=sys.stderr, flush=True)
    with open(out_path, "w") as f:
        json.dump(results, f, indent=1)


if __name__ == "__main__":
    sys.exit(main())
