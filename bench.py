"""Benchmark of the ZeRO shard step on GB300: parameters updated per second and achieved
HBM bandwidth against the measured peak, with the parameter gather after it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the shard step over one batch of synthetic input: the rank-order
sum of the Nd fp16 gradient contributions, the overflow flag and exact norm, and the
clipped AdamW update with the fp16 cast. The default workload is the largest one that
fits one GPU: rank 0 of a 13B-parameter, 40-layer ZeRO-3 group of Nd = 64 (a span of
203,125,000 parameters with 64 fp16 contributions, 26 GB per step; two alternating
gradient sets, larger than L2, so no flush), followed in the same line by the gather of
all 64 fp16 shards (rank 0's is the step's output) into the 40 layer buffers, and by a
pass of both together.

For N > 1 (launched with torch.distributed.run, one process per GPU): a workload whose
span is one logical rank gives GPU g the shard of logical rank g (weak scaling); one
whose span covers several logical ranks splits them over the GPUs (strong scaling). The
one exchange step is an NCCL all-reduce of the 64-byte statistics buffer between the two
halves of the step.

``--impl reference`` times the CPU oracle (its C steps partitioned over the host cores) on
a bounded sample of the same workload instead; it needs no GPU.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ZeRO shard-step params/s; achieved HBM GB/s as % of GB300 peak"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300's nominal HBM3e bandwidth (context beside the measured peak)
STEP_INFO_D2H_BYTES = 96  # the device scalars block that zero_step_result copies back


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.windows = []  # (start, end) of each GPU-timed region

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        """Open ("start") or close ("end") a timed window; clocks are summarised over the
        samples taken inside any window (host-bound legs, where the GPU idles, are left
        out)."""
        if which == "start":
            self.windows.append([time.time(), None])
        elif self.windows:
            self.windows[-1][1] = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows
                  if any(a <= r[0] <= (b or 1e18) for a, b in self.windows)]
        used = inside or rows[-3:]
        sm = [float(p[1]) for _, p in used if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in used if p[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in used:
            for name, val in zip(names, p[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None,
               "reasons": sorted(reasons),
               "samples_in_timed_region": len(inside)}
        pw = [float(p[3]) for _, p in used if p[3].replace(".", "").isdigit()]
        if pw:
            out["power_w_max"] = max(pw)
        return out


# ------------------------------------------------------------------------------------
# CPU oracle timing (test infrastructure; the only place the bench runs the oracle)

L2_NOMINAL = 129_000_000  # GB300 L2 bytes
HOLD_CYCLES = 100_000_000  # about 50 ms of SM clock before a flushed timed loop


def l2_bytes(dev) -> int:
    import torch
    got = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 0)
    return max(got, L2_NOMINAL)


def working_set(w) -> int:
    """Bytes one step of the bench touches over its two alternating gradient sets: the
    contributions, master/m/v, the fp16 parameters and the fp32 sums."""
    n_span = w.span()[1]
    return 2 * 2 * w.nd * n_span + 18 * n_span


def l2_flush(w) -> bool:
    """Whether L2 could keep the step's inputs between steps (then it is flushed)."""
    return working_set(w) < 2 * L2_NOMINAL


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


GEN_CHUNK = 1 << 20  # elements per generator call (the counter-based streams split freely)


def _generate(fn, n, pool):
    import numpy as np
    bounds = list(range(0, n, GEN_CHUNK)) + [n]
    parts = list(pool.map(lambda i: fn(bounds[i], bounds[i + 1] - bounds[i]),
                          range(len(bounds) - 1)))
    return np.concatenate(parts) if len(parts) > 1 else parts[0]


def cpu_sample(w, n, threads=None):
    """The first n parameters of the workload's span, generated on the CPU by the seeded
    generator: two gradient sets and the initial master/m/v/param16. Every value depends
    only on its index, so the arrays are generated in chunks on several threads."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import synth
    from synth import workloads as wl
    first = w.span()[0]
    with ThreadPoolExecutor(threads or host_threads()) as pool:
        def f32(kind, sigma, absolute=False):
            return _generate(lambda a, k: synth.values_f32(wl.key(w, kind), sigma, first + a, k,
                                                           absolute=absolute), n, pool)
        master = f32(synth.MASTER, w.master_sigma)
        m = f32(synth.EXP_AVG, w.m_sigma) if w.m_sigma > 0 else np.zeros(n, np.float32)
        v = (f32(synth.EXP_AVG_SQ, w.v_sigma, absolute=True) if w.v_sigma > 0
             else np.zeros(n, np.float32))
        p16 = master.astype(np.float16).view(np.uint16).copy()
        grads = [[_generate(lambda a, k, st=st, r=r: synth.values_f16(
                      wl.key(w, synth.GRAD, st, r), w.grad_sigma * w.loss_scale, first + a, k),
                      n, pool) for r in range(w.nd)] for st in range(2)]
    return grads, master, m, v, p16


class PartitionedOracle:
    """The oracle's shard step run on T host threads over disjoint slices of the span,
    with the same results as one oracle.step over the whole span: each thread sums its
    slice in rank order and takes its slice's non-finite count and exact integer sum of
    squares; the counts and sums are added (exactly, as integers), the step's scalars are
    computed once from the totals, and each thread then updates its own slice. ctypes
    releases the interpreter lock during the oracle's C calls, so the slices run in
    parallel."""

    def __init__(self, n, threads):
        from concurrent.futures import ThreadPoolExecutor
        self.threads = max(1, min(threads, max(1, n // 64)))
        cuts = [(n * i // self.threads) // 64 * 64 for i in range(self.threads)] + [n]
        self.slices = [slice(cuts[i], cuts[i + 1]) for i in range(self.threads)]
        self.pool = ThreadPoolExecutor(self.threads)

    def step(self, grads, master, m, v, p16, loss_scale, clip, hp, t, keep_sums=False):
        """One oracle step over the slices; with keep_sums, self.sums holds each slice's
        fp32 rank-order sums afterwards."""
        import oracle

        def sums(sl):
            gsum = oracle.reduce([c[sl] for c in grads])
            bad, ss = oracle.stats(gsum)
            return gsum, bad, ss

        parts = list(self.pool.map(sums, self.slices))
        self.sums = [p[0] for p in parts] if keep_sums else None
        sc = oracle.scalars(sum(p[1] for p in parts), sum(p[2] for p in parts), loss_scale,
                            clip, hp, t)
        list(self.pool.map(lambda i: oracle.adam(parts[i][0], master[self.slices[i]],
                                                 m[self.slices[i]], v[self.slices[i]],
                                                 p16[self.slices[i]], sc),
                           range(self.threads)))
        return sc

    def close(self):
        self.pool.shutdown()


def oracle_steps(w, n, steps=None, seconds=None, warmup=0, threads=1, sample=None):
    """Run the oracle on a CPU sample of n parameters (single-threaded, or partitioned over
    ``threads`` host threads), either a fixed number of steps or until ``seconds`` pass.
    Returns (params/s, steps, seconds, threads used)."""
    import oracle
    grads, master, m, v, p16 = sample if sample is not None else cpu_sample(w, n)
    if sample is not None:  # the first n parameters of a larger sample
        grads = [[c[:n] for c in g] for g in grads]
        master, m, v, p16 = (x[:n].copy() for x in (master, m, v, p16))
    hp = oracle.Hyper(**w.hparams())
    par = PartitionedOracle(n, threads) if threads > 1 else None

    def one(g, t):
        if par is not None:
            return par.step(g, master, m, v, p16, w.loss_scale, w.clip, hp, t).step
        return oracle.step(g, master, m, v, p16, w.loss_scale, w.clip, hp, t).step

    t = 0
    for i in range(warmup):
        t = one(grads[i % 2], t)
    done = 0
    t0 = time.perf_counter()
    while True:
        t = one(grads[done % 2], t)
        done += 1
        el = time.perf_counter() - t0
        if (steps is not None and done >= steps) or (seconds is not None and el >= seconds):
            break
    used = par.threads if par is not None else 1
    if par is not None:
        par.close()
    return n * done / el, done, el, used


def sample_size(w, max_params):
    n = min(max_params, w.span()[2])
    return max(8, n - n % 8)


SAMPLE_PER_THREAD = 2_000_000  # parameters per host thread in the all-core sample
SAMPLE_BYTES = 4e9             # host memory for the all-core sample at most


def sample_bytes_per_param(w):
    return 2 * 2 * w.nd + 4 * 4 + 2  # two gradient sets, master/m/v + the sum, param16


def all_core_sample_size(w, threads):
    n = min(threads * SAMPLE_PER_THREAD, int(SAMPLE_BYTES / sample_bytes_per_param(w)))
    return sample_size(w, max(8, n))


def oracle_sample_rate(w, seconds: float):
    """The oracle on all host cores (partitioned) and on one core, each for about half of
    ``seconds``, on one sample of the workload. Returns the cpu_baseline object."""
    threads = host_threads()
    n = all_core_sample_size(w, threads)
    sample = cpu_sample(w, n, threads)
    rate, steps, el, used = oracle_steps(w, n, seconds=seconds / 2, threads=threads,
                                         sample=sample)
    n1 = sample_size(w, min(n, 4_000_000))
    rate1, steps1, el1, _ = oracle_steps(w, n1, seconds=seconds / 2, sample=sample)
    return {
        "value": rate, "unit": UNIT, "cores": used, "kind": "oracle",
        "sample": (f"oracle reduce/stats/adam (C, -O2) partitioned over {used} host threads "
                   f"with an exact integer combine of the statistics, on the first {n:,} "
                   f"parameters of the span; {steps} steps in {el:.1f} s; norm and clip taken "
                   f"over the sample"),
        "single_thread": {"value": rate1, "cores": 1,
                          "sample": f"oracle.step on the first {n1:,} parameters, {steps1} "
                                    f"steps in {el1:.1f} s"},
    }


def gather_cpu_rate(w, seconds: float):
    """The oracle's gather timed on the host cores on a scaled-down copy of the workload's
    layout: nd shards of s' elements (s' chosen so the sample has about
    SAMPLE_PER_THREAD parameters per thread) and the layer offsets scaled by s'/s; the
    layers are split into contiguous groups, one oracle.gather call per group and thread.
    Returns the cpu_baseline object (params/s)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    import synth
    from synth import workloads as wl
    threads = host_threads()
    _, s = w.layout()
    s_small = max(8, min(s, threads * SAMPLE_PER_THREAD // w.nd) // 8 * 8)
    layer_offs = [o * s_small // s for o in (w.layers or (0, w.n))]
    n_layers = len(layer_offs) - 1
    # cut points at the layer boundaries and at one slice per thread, so that a layout of
    # few layers (one, for the full-buffer gather) still keeps every thread busy
    span = layer_offs[-1] - layer_offs[0]
    offs = sorted(set(layer_offs) | {layer_offs[0] + span * i // threads
                                     for i in range(threads)})
    n_pieces = len(offs) - 1
    with ThreadPoolExecutor(threads) as pool:
        shards = [_generate(lambda a, k, r=r: synth.values_f16(
                      wl.key(w, synth.SHARD16, 0, r), w.shard_sigma, r * s_small + a, k),
                      s_small, pool) for r in range(w.nd)]
        groups = min(threads, n_pieces)
        cuts = [n_pieces * i // groups for i in range(groups + 1)]
        parts = [offs[cuts[i]:cuts[i + 1] + 1] for i in range(groups)]
        done = 0
        t0 = time.perf_counter()
        while True:
            list(pool.map(lambda o: oracle.gather(shards, s_small, o), parts))
            done += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                break
    moved = offs[-1] - offs[0]
    return {"value": moved * done / el, "unit": "params/s", "cores": groups, "kind": "oracle",
            "sample": (f"oracle.gather (C) over {w.nd} shards of {s_small:,} elements into "
                       f"{n_layers} layers ({moved:,} parameters; the workload's layer "
                       f"offsets scaled by {s_small:,}/{s:,}), cut into {n_pieces} pieces "
                       f"at the layer boundaries and per thread, piece groups on {groups} "
                       f"host threads; {done} passes in {el:.1f} s")}



# ------------------------------------------------------------------------------------
# which logical ranks each process owns

DEFAULT_WORKLOAD = "zero3_13b_rank0_nd64"


def process_span(w0, world: int, rank: int):
    """This process's workload restricted to its logical ranks, and the scaling kind. A
    workload whose span is one logical rank (a device that owns one shard of a ZeRO-2/3
    group) gives process g the shard of logical rank r0 + g, so every process does the
    same work (weak scaling); a workload whose span covers several logical ranks splits
    them into equal contiguous pieces, one per process (strong scaling)."""
    import sharded_emulated_reduce_gb300 as z
    n_ranks = w0.r1 - w0.r0
    if n_ranks == 1:
        if w0.r0 + world > w0.nd:
            raise SystemExit(f"--gpus {world}: the workload has {w0.nd - w0.r0} logical ranks "
                             f"from rank {w0.r0} on")
        g = w0.r0 + rank
        return dataclasses.replace(w0, r0=g, r1=g + 1), "weak"
    if n_ranks % world:
        raise SystemExit(f"--gpus {world} must divide the span's {n_ranks} logical ranks")
    a, b = z.rank_ranges(n_ranks, world)[rank]
    return dataclasses.replace(w0, r0=w0.r0 + a, r1=w0.r0 + b), "strong"


def job_params(w0, world: int) -> int:
    """Real parameters that all processes together update in one step."""
    return sum(process_span(w0, world, g)[0].span()[2] for g in range(world))


def gather_layout(w) -> list:
    """Layer offsets the gather copies: the workload's layer table (ZeRO-3), or one layer
    holding the whole flat parameter vector (the parameter all-gather of ZeRO-1/2)."""
    return list(w.layers) if w.layers else [0, w.n]


def gather_flush(w) -> bool:
    """Whether L2 could keep the gather's shards and layers between calls."""
    return 4 * w.n < 2 * L2_NOMINAL


def config_of(w, n_gpus):
    """The workload as both arms name it (identical objects in the GPU and oracle lines)."""
    first, n_span, n_valid = w.span()
    offs = gather_layout(w)
    weak = (w.r1 - w.r0) == 1
    return {"workload": w.name, "n_params": w.n, "nd": w.nd, "align": w.align,
            "stage": w.stage, "span_ranks": [w.r0, w.r1], "params_in_span": n_valid,
            "loss_scale": w.loss_scale, "clip": w.clip,
            "parallelism": (f"zero{w.stage} nd{w.nd}: each of {n_gpus} gpu steps one logical "
                            f"rank's shard" if weak else
                            f"zero{w.stage} nd{w.nd}: the span's logical ranks split over "
                            f"{n_gpus} gpu"),
            "gather": (f"{w.nd} fp16 shards of {w.layout()[1]:,} into {len(offs) - 1} layer "
                       f"buffers" if w.layers else
                       f"{w.nd} fp16 shards into one flat buffer of {w.n:,} (ZeRO-1/2)"),
            "l2": ("inputs larger than L2 (two alternating gradient sets of "
                   f"{2 * w.nd * n_span / 1e9:.2f} GB each); no flush" if not l2_flush(w)
                   else f"working set {working_set(w) / 1e6:.0f} MB < 2 x L2: L2 flushed (a "
                        f"write of twice the L2 size) before every step, outside the step's "
                        f"events"),
            "io": "fp16 grads in, fp32 master/m/v, fp16 params out",
            "state": "HBM"}


def append_results(path, records) -> None:
    """Append one JSON record per line to `path` (the per-kernel results log)."""
    stamp = time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime())
    with open(path, "a") as f:
        for r in records:
            f.write(json.dumps(dict(r, time=stamp)) + "\n")


def kernel_records(line, kinds, kms, klaunch, traffic_of) -> list:
    """The results-log records of one GPU bench line: one per kernel (its algorithmic and
    moved GB/s and fraction of peak), the whole step, and the gather if it ran."""
    peak = line["roofline"]["peak"]
    base = {"workload": line["config"]["workload"], "impl": "ours", "n_gpus": line["n_gpus"],
            "peak_gbs": peak}
    cpu = line.get("cpu_baseline") or {}
    span_params = line["config"]["params_in_span"]
    out = []
    for k, (name, alg) in kinds.items():
        if not klaunch[k]:
            continue
        ms = kms[k] / klaunch[k]
        traffic = traffic_of(name)
        out.append(dict(base, kernel=name, launches=int(klaunch[k]), avg_ms=ms,
                        alg_bytes_per_launch=alg, alg_gbs=alg / ms / 1e6,
                        frac_of_peak=alg / ms / 1e6 / peak,
                        moved_bytes_per_launch=traffic,
                        moved_gbs=None if traffic is None else traffic / ms / 1e6))
    h = line["step_hbm"]
    out.append(dict(base, kernel="whole step", ms=line["ms_per_step"],
                    params_per_s=line["value"], alg_gbs=h["alg_gbs"], frac_of_peak=h["alg_frac"],
                    min_moved_gbs=h["min_moved_gbs"],
                    oracle_s_per_step=(span_params / cpu["value"]) if cpu else None,
                    oracle_cores=cpu.get("cores")))
    g = line.get("gather")
    if g:
        r = g["roofline"]
        out.append(dict(base, kernel="gather", ms=g["ms_per_call"], params_per_s=g["value"],
                        alg_gbs=r["achieved"], frac_of_peak=r["frac"],
                        moved_bytes_per_launch=r.get("traffic")))
    return out


def run_reference(args, w):
    rank = env_int("RANK", 0)
    if rank != 0:
        return 0
    # size the sample so that warmup + steps take about two minutes at most
    threads = host_threads()
    n_max = all_core_sample_size(w, threads)
    probe = sample_size(w, min(n_max, threads * 65536))
    rate0, _, _, _ = oracle_steps(w, probe, seconds=0.5, threads=threads)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    n = sample_size(w, int(max(8192, min(n_max, rate0 * per_step))))
    value, _, el, used = oracle_steps(w, n, steps=args.steps, warmup=args.warmup,
                                      threads=threads)
    sample = (f"oracle reduce/stats/adam (C) partitioned over {used} host threads, exact "
              f"integer combine, on the first {n:,} of {w.span()[2]:,} parameters per step; "
              f"norm and clip over the sample")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": process_span(w, 1, 0)[1], "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config_of(w, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if not args.no_gather and args.cpu_seconds > 0:
        g = gather_cpu_rate(w, min(args.cpu_seconds, 6.0))
        line["gather"] = {"value": g["value"], "unit": g["unit"], "cpu_baseline": g}
    if args.results:
        append_results(args.results, [{
            "workload": w.name, "impl": "reference", "n_gpus": args.gpus,
            "kernel": "whole step", "ms": line["ms_per_step"], "params_per_s": value,
            "oracle_cores": used, "sample": sample}])
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------------------

def run_ours(args, w0):
    import torch

    import sharded_emulated_reduce_gb300 as z
    from synth import workloads as wl

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local = env_int("LOCAL_RANK", 0)
    dist = None
    if world > 1:
        import torch.distributed as dist
        # one process per GPU; a rehearsal of the multi-process path with more processes
        # than GPUs (ZERO_BENCH_BACKEND=gloo: host-side collectives only, no kernel waits
        # on another process) shares them round robin
        torch.cuda.set_device(local % torch.cuda.device_count())
        dist.init_process_group(os.environ.get("ZERO_BENCH_BACKEND", "nccl"))
    else:
        torch.cuda.set_device(0)
    w, scaling = process_span(w0, world, rank)
    first, n_span, n_valid = w.span()
    dev = torch.device("cuda", torch.cuda.current_device())

    master, m, v, p16, ws = wl.make_state(w, dev)
    if args.state == "host":
        # optimizer state in Grace memory; the fp16 parameters stay in HBM, where the
        # forward pass reads them
        master, m, v = [t.cpu().pin_memory() for t in (master, m, v)]
    gsets = [wl.make_grads(w, s, dev) for s in range(1 if args.one_set else 2)]
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    z.zero_plan_bind(plan, w.r0, w.r1, master, m, v, p16, ws, 0)
    stream = torch.cuda.current_stream()

    def one_step(grads):
        if dist is None:
            z.zero_shard_step(plan, w.r0, w.r1, grads, w.loss_scale, w.clip, stream)
        else:
            z.zero_dist_step(plan, w.r0, w.r1, grads, w.loss_scale, w.clip, stream=stream)

    graphs = None
    if args.graph and dist is None:
        # one captured step per gradient set: a replay launches both kernels at once,
        # which removes the per-launch host cost that dominates small spans
        z.zero_profile_enable(plan, True)
        one_step(gsets[0])
        torch.cuda.synchronize()
        z.zero_profile_enable(plan, False)
        counts = z.zero_profile_read(plan, reset=True)[1]
        launches_per_step = int(counts[0] + counts[1] + counts[2] + counts[4])
        graphs = []
        for gs in gsets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                z.zero_shard_step(plan, w.r0, w.r1, gs, w.loss_scale, w.clip)
            graphs.append(g)
        eager_step = one_step

        def one_step(grads):  # noqa: F811 (graph replay of the same step)
            for gs, g in zip(gsets, graphs):
                if grads is gs:
                    g.replay()
                    return
            eager_step(grads)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def job_max(x: float) -> float:
        """The largest value of x over all processes."""
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        if dist is not None:
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return t.item()

    for i in range(args.warmup):
        one_step(gsets[i % len(gsets)])
    barrier()

    # A working set that L2 could hold between iterations gets an L2 flush before every
    # iteration: a write of twice the L2 size, outside the iteration's own events; the
    # time is then the sum of the per-iteration event intervals.
    flush_buf = (torch.empty(2 * l2_bytes(dev), dtype=torch.uint8, device=dev)
                 if l2_flush(w0) or (not args.no_gather and gather_flush(w0)) else None)

    per_iter = {}  # the last flushed timing's per-iteration event times, by body

    def timed(body, count, flush):
        """`count` iterations of body(i) between events on the launching stream; returns
        milliseconds."""
        barrier()
        if not flush:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(count):
                body(i)
            e1.record(stream)
            barrier()
            return e0.elapsed_time(e1)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(count)]
        # hold the stream for a moment so that the host queues the iterations ahead of the
        # GPU: each iteration's events then bracket device work only, not host waits
        torch.cuda._sleep(HOLD_CYCLES)
        for i in range(count):
            flush_buf.zero_()
            ev[i][0].record(stream)
            body(i)
            ev[i][1].record(stream)
        barrier()
        per_iter[body] = [a.elapsed_time(b) for a, b in ev]
        return sum(per_iter[body])

    def step_body(i):
        one_step(gsets[i % len(gsets)])

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # Timed region 1, the step as a user runs it: the step time and `value`.
    # Timed region 2, the same K steps with the library's per-launch events on: each
    # kernel's average duration (the roofline). The events themselves add a few
    # microseconds per step, which is why the step time is taken without them.
    clocks.mark("start")
    ms_total = timed(step_body, args.steps, l2_flush(w0))
    # with a flush before every step, each step has its own events: their median too
    ms_median = statistics.median(per_iter[step_body]) if l2_flush(w0) else None
    z.zero_profile_read(plan, reset=True)
    z.zero_profile_enable(plan, True)
    ms_profiled = timed(step_body, args.steps, l2_flush(w0)) if graphs is None else None
    clocks.mark("end")
    z.zero_profile_enable(plan, False)
    kms, klaunch = z.zero_profile_read(plan, reset=True)
    info = z.zero_step_result(plan).as_dict()

    ms_per_step = job_max(ms_total) / args.steps
    ms_per_step_median = job_max(ms_median) if ms_median is not None else None
    total_params = job_params(w0, world)
    value = total_params / (ms_per_step / 1e3)

    e2e = run_e2e(args, plan, one_step, gsets, p16, stream, barrier, job_max, world,
                  total_params) if not args.no_e2e else None

    gather = hot = None
    if not args.no_gather:
        # the parameter gather after the step: the span's own shards are the step's fp16
        # output, the other ranks' shards are seeded
        offs = gather_layout(w0)
        shards = wl.span_shards(w, p16, dev)
        dst = [torch.empty(offs[l + 1] - offs[l], dtype=torch.float16, device=dev)
               for l in range(len(offs) - 1)]

        def gather_body(i):
            z.zero_gather_layers(plan, offs, shards, dst, stream)

        for i in range(3):
            gather_body(i)
        barrier()
        z.zero_profile_read(plan, reset=True)
        z.zero_profile_enable(plan, True)
        clocks.mark("start")
        gms = timed(gather_body, args.steps, gather_flush(w0))
        clocks.mark("end")
        z.zero_profile_enable(plan, False)
        gk_ms, gk_n = z.zero_profile_read(plan, reset=True)
        if z.zero_gather_status(plan) != 0:
            raise SystemExit("the gather reported a device failure")
        gather = gather_object(offs, args.steps, job_max(gms) / args.steps,
                               gk_ms[z.PROF_GATHER], gk_n[z.PROF_GATHER], world,
                               traffic=load_traffic("gather", w0))
        if rank == 0 and args.cpu_seconds > 0:
            gather["cpu_baseline"] = gather_cpu_rate(w0, min(args.cpu_seconds, 6.0))

        # one pass of the whole hot path: the step, then the gather of its output
        def pass_body(i):
            step_body(i)
            gather_body(i)

        n_pass = max(3, min(args.steps, 50))
        for i in range(2):
            pass_body(i)
        clocks.mark("start")
        pms = timed(pass_body, n_pass, l2_flush(w0) or gather_flush(w0))
        clocks.mark("end")
        hot = {"ms_per_pass": job_max(pms) / n_pass, "passes": n_pass,
               "what": "one shard step of the span, then the gather of all shards (the "
                       "step's fp16 output among them) into the layer buffers",
               "ms_step_plus_gather_timed_apart": ms_per_step + gather["ms_per_call"]}
        del shards, dst
    clk = clocks.stop()

    peak, peak_kind = load_peaks()
    n_real = n_valid
    kinds = {0: ("reduce", (2 * w.nd + 4) * n_span),
             1: ("update", 30 * n_real),
             2: ("scalars", 0),
             4: ("step", 2 * w.nd * n_span + 26 * n_real)}  # small spans: one launch
    if graphs is None:
        dom = max((k for k in kinds if klaunch[k]), key=lambda k: kms[k])
        name, alg_bytes = kinds[dom]
        avg_ms = kms[dom] / klaunch[dom]
        achieved = alg_bytes / (avg_ms / 1e3) / 1e9
        # the stored captures are of HBM-resident state
        traffic = load_traffic(name, w) if args.state != "host" else None
        roofline = {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                    "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                    "traffic": traffic, "alg_bytes_per_launch": alg_bytes,
                    "avg_launch_ms": avg_ms,
                    "time_share": {kinds[k][0]: kms[k] / sum(kms[j] for j in kinds)
                                   for k in kinds if klaunch[k]},
                    "events": "per-launch events of a second timed pass of the same K steps; "
                              f"that pass took {ms_profiled / args.steps:.4f} ms/step"}
        launches = int(sum(klaunch[k] for k in kinds)) * world
    else:
        # replays carry no per-launch events: the roofline is taken over the whole step
        alg_bytes = (2 * w.nd + 4) * n_span + 30 * n_real
        achieved = alg_bytes / (ms_per_step / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": "reduce+update (graph replay)",
                    "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_kind": peak_kind,
                    "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "traffic": None,
                    "alg_bytes_per_launch": alg_bytes, "avg_launch_ms": ms_per_step}
        launches = launches_per_step * args.steps * world
    step_alg = (2 * w0.nd + 26) * total_params
    step_gbs = step_alg / (ms_per_step / 1e3) / 1e9
    moved = (2 * w0.nd + 34) * total_params / (ms_per_step / 1e3) / 1e9

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        plan.close()
        return 0
    cpu = oracle_sample_rate(w0, args.cpu_seconds) if args.cpu_seconds > 0 else None
    cfg = config_of(w0, world)
    if args.state == "host":
        cfg["state"] = ("master/m/v in pinned Grace memory over NVLink-C2C; fp16 parameters "
                        "in HBM")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_median": ms_per_step_median,
        "higher_is_better": True, "scaling": scaling, "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": cfg,
        "timing": ("K steps between two events on the launching stream, without the "
                   "library's per-launch events (a second pass with them gives the "
                   "per-kernel durations); max over processes"),
        "launch": ("CUDA graph replay (one graph per gradient set)" if graphs is not None
                   else "eager calls through the C ABI"),
        "e2e": e2e,
        "gpu_launches": launches,
        "roofline": roofline,
        "step_hbm": {"alg_bytes_per_param": 2 * w0.nd + 26, "alg_gbs": step_gbs,
                     "alg_frac": step_gbs / peak,
                     "min_moved_bytes_per_param": 2 * w0.nd + 34, "min_moved_gbs": moved,
                     "min_moved_frac": moved / peak, "peak": peak, "peak_kind": peak_kind},
        "gather": gather,
        "hot_path": hot,
        "cpu_baseline": cpu,
        "clocks": clk,
        "last_step": {k: info[k] for k in ("step", "skipped", "global_norm", "clip_coef")},
    }
    if args.results:
        # the stored captures are of HBM-resident state; graph replays carry no per-kernel
        # events, so they give the step and gather records only
        traffic_of = ((lambda name: load_traffic(name, w)) if args.state != "host"
                      else (lambda name: None))
        append_results(args.results, kernel_records(line, kinds if graphs is None else {},
                                                    kms, klaunch, traffic_of))
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    plan.close()
    return 0


E2E_LINK_GBS = 200.0  # host-to-device rate used only to size the end-to-end leg
E2E_SECONDS = 3.0     # about this long per end-to-end mode
E2E_HOST_SHARE = 0.4  # of the host's memory, split over the local processes


def host_memory_bytes() -> int:
    try:
        return os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    except (ValueError, OSError, AttributeError):
        return 0


def run_e2e(args, plan, one_step, gsets, p16, stream, barrier, job_max, world, total_params):
    """The step end to end through the public API from pinned host memory, in the ways a
    user can feed it, each timed over whole steps; every step includes the upload of its
    gradients and the read-back of its result (the step info: flag, skip, norm, counter).
    One pinned gradient set is reused for every step. "copy" stages the gradients into
    HBM with cudaMemcpyAsync and then steps; "copy_overlap" does the same through two
    device buffers, uploading step i+1's gradients on a second stream while step i runs;
    "zero_copy" passes the pinned host pointers to the step, whose reduce kernel reads
    them over NVLink-C2C directly. A fourth leg, "copy" plus a read-back of the fp16
    parameters to pinned host memory each step, is reported beside them."""
    import torch

    import sharded_emulated_reduce_gb300 as z
    # one pinned buffer per logical rank while they fit the process's share of host memory;
    # past it, the buffers are reused cyclically (every step still moves every rank's bytes)
    per_rank = gsets[0][0].numel() * gsets[0][0].element_size()
    local = max(1, env_int("LOCAL_WORLD_SIZE", 1))
    budget = host_memory_bytes() * E2E_HOST_SHARE / local
    distinct = len(gsets[0]) if budget <= 0 else max(1, min(len(gsets[0]), int(budget // per_rank)))
    pinned = [torch.empty(g.numel(), dtype=g.dtype, pin_memory=True) for g in gsets[0][:distinct]]
    for h, g in zip(pinned, gsets[0]):
        h.copy_(g)
    host = [pinned[k % distinct] for k in range(len(gsets[0]))]
    dev_g = [[torch.empty_like(g) for g in gsets[0]] for _ in range(2)]
    p16_host = torch.empty(p16.numel(), dtype=p16.dtype, pin_memory=True)
    h2d_rank = sum(g.numel() * g.element_size() for g in gsets[0])
    est = h2d_rank / (E2E_LINK_GBS * 1e9)
    steps = max(3, min(args.steps, 100, int(E2E_SECONDS / max(est, 1e-6))))
    copy_stream = torch.cuda.Stream()
    uploaded = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def upload(buf):  # the gradients into buf, on the current stream
        for d, h in zip(buf, host):
            d.copy_(h, non_blocking=True)

    def run_mode(mode, n):
        """n steps of `mode`, from the first upload to the last result read."""
        if mode == "copy_overlap":
            # buffer b = i % 2: upload i waits until step i-2 has consumed buffer b
            with torch.cuda.stream(copy_stream):
                upload(dev_g[0])
                uploaded[0].record(copy_stream)
            for i in range(n):
                b = i % 2
                if i + 1 < n:
                    nb = (i + 1) % 2
                    with torch.cuda.stream(copy_stream):
                        if i >= 1:
                            copy_stream.wait_event(consumed[nb])
                        upload(dev_g[nb])
                        uploaded[nb].record(copy_stream)
                stream.wait_event(uploaded[b])
                one_step(dev_g[b])
                consumed[b].record(stream)
                z.zero_step_result(plan)
            return
        for i in range(n):
            if mode == "zero_copy":
                one_step(host)
            else:
                upload(dev_g[0])
                one_step(dev_g[0])
            if mode == "copy_params_to_host":
                p16_host.copy_(p16, non_blocking=True)
            z.zero_step_result(plan)

    rates = {}
    for mode in ("copy", "copy_overlap", "zero_copy", "copy_params_to_host"):
        run_mode(mode, 2)
        barrier()
        t0 = time.perf_counter()
        run_mode(mode, steps)
        barrier()
        rates[mode] = total_params / job_max((time.perf_counter() - t0) / steps)
    del host, pinned, dev_g
    with_params = rates.pop("copy_params_to_host")
    best = max(rates, key=rates.get)
    h2d = h2d_rank * world
    p16_bytes = p16.numel() * p16.element_size() * world
    return {"value": rates[best], "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": STEP_INFO_D2H_BYTES * world, "steps": steps, "mode": best,
            "by_mode": rates,
            "host_buffers": (
                f"{len(gsets[0])} distinct pinned gradient buffers" if distinct == len(gsets[0])
                else f"{distinct} distinct pinned buffers for {len(gsets[0])} ranks, reused "
                     f"cyclically (this process's share of host memory)"),
            "result_read_back": ("the step info (overflow flag, skip, norm, step counter) "
                                 "each step; the fp16 parameters stay in HBM, where the "
                                 "forward pass and the gather read them"),
            "with_params_to_host": {"value": with_params, "unit": UNIT, "mode": "copy",
                                    "h2d_bytes_per_step": h2d,
                                    "d2h_bytes_per_step": p16_bytes + STEP_INFO_D2H_BYTES * world}}


def gather_object(offs, calls, ms_per_call, kernel_ms, launches, world, traffic=None):
    """The gather's figures: parameters moved per second (all processes), and its kernels'
    achieved HBM bandwidth (4 algorithmic bytes per parameter over their summed
    per-launch durations) against the measured peak."""
    peak, peak_kind = load_peaks()
    n_moved = offs[-1] - offs[0]
    alg_total = 4 * n_moved * calls
    achieved = alg_total / (kernel_ms / 1e3) / 1e9
    per_call = launches / calls
    return {"value": world * n_moved / (ms_per_call / 1e3), "unit": "params/s",
            "ms_per_call": ms_per_call, "calls": calls, "params_per_call": n_moved,
            "layers": len(offs) - 1, "gpu_launches": int(launches) * world,
            "roofline": {"bound": "hbm", "kernel": "gather", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_kind": peak_kind,
                         "frac_of_nominal": achieved / NOMINAL_HBM_GBS, "traffic": traffic,
                         "alg_bytes_per_launch": 4 * n_moved / per_call,
                         "avg_launch_ms": kernel_ms / launches}}


KERNEL_SOURCES = ("step_kernels.cu", "gather_kernel.cu", "bulk_async.h", "grid_sync.h",
                  "internal.h", "bounds.h")


def kernel_source_hash() -> str:
    """Short hash of the kernel sources' code (comments and whitespace removed); a
    committed traffic figure is used only if it was captured on exactly this code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "sharded_emulated_reduce_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)                  # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel: str, w):
    """Per-launch DRAM bytes (read + write) of `kernel` on workload `w` from the committed
    ncu summary (profiles/ncu_traffic.json), if it was captured on the current kernel
    sources; None otherwise."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    ent = d.get("workloads", {}).get(w.name, {}).get(kernel)
    return None if not ent else ent.get("dram_bytes_per_launch")


def run_gather(args, w):
    """Time the gather alone: all Nd fp16 shards into the workload's layer buffers
    (ZeRO-3), or, for a workload without a layer table, into one buffer holding the whole
    flat parameter vector (the parameter all-gather of ZeRO-1/2). With --prefetch, layer
    by layer with one completion event per layer."""
    import torch

    import sharded_emulated_reduce_gb300 as z
    from synth import workloads as wl

    if env_int("WORLD_SIZE", 1) > 1 and env_int("RANK", 0) != 0:
        return 0
    torch.cuda.set_device(0)
    _, s = w.layout()
    shard0 = torch.empty(s, dtype=torch.float16, device="cuda")
    shards = wl.make_shards(w, shard0)
    wl.fill(shard0, wl.key(w, wl.SHARD16, 0, 0), w.shard_sigma, start=0, n_valid=w.n)
    offs = gather_layout(w)
    if args.layer_shift:
        # move every interior layer boundary by a few elements: layers then start at
        # addresses misaligned (mod 16 bytes) relative to the shards they copy from
        offs = [offs[0]] + [o + args.layer_shift for o in offs[1:-1]] + [offs[-1]]
    dst = [torch.empty(offs[l + 1] - offs[l], dtype=torch.float16, device="cuda")
           for l in range(len(offs) - 1)]
    plan = z.zero_plan_create(w.n, w.nd, w.stage, w.align, w.hparams())
    stream = torch.cuda.current_stream()
    events = z.make_layer_events(len(offs) - 1) if args.prefetch else None

    def gather():
        if args.prefetch:  # one launch and one event per layer, from one C call
            return z.zero_gather_layers_events(plan, offs, shards, dst, events, stream)
        return z.zero_gather_layers(plan, offs, shards, dst, stream)

    for _ in range(args.warmup):
        gather()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    z.zero_profile_enable(plan, True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark("start")
    e0.record(stream)
    for _ in range(args.steps):
        gather()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark("end")
    kms, kl = z.zero_profile_read(plan, reset=True)  # the timed calls only
    z.zero_profile_enable(plan, False)
    prefetch = None
    if args.prefetch:
        # when each layer is ready, counted from the call (one more call, after the timing)
        timing_events = z.make_layer_events(len(offs) - 1, timing=True)
        t0 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        z.zero_gather_layers_events(plan, offs, shards, dst, timing_events, stream)
        torch.cuda.synchronize()
        ready = [t0.elapsed_time(e) for e in timing_events]
        prefetch = {"layer_ready_ms": ready, "first_layer_ms": ready[0],
                    "all_layers_ms": ready[-1]}
    ms = e0.elapsed_time(e1) / args.steps
    clk = clocks.stop()
    # with --prefetch consecutive layers overlap on two streams, so their per-launch
    # durations overlap too: the bandwidth is taken over whole calls instead
    g = gather_object(offs, args.steps, ms,
                      ms * args.steps if args.prefetch else kms[z.PROF_GATHER],
                      kl[z.PROF_GATHER], 1,
                      traffic=(None if args.layer_shift or args.prefetch
                               else load_traffic("gather", w)))
    if args.prefetch:
        g["roofline"]["timed"] = "whole calls (layers overlap on two streams)"
    line = {
        "metric": "ZeRO-3 gather params/s (fp16 shards to layer buffers); achieved HBM GB/s "
                  "as % of GB300 peak",
        "value": g["value"], "unit": "params/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "f16 (copy)", "data": "synthetic",
        "config": {"workload": w.name, "op": "gather", "n_params": w.n, "nd": w.nd,
                   "layer_shift": args.layer_shift, "prefetch": bool(args.prefetch),
                   "layers": len(offs) - 1, "shard_len": s,
                   "l2": f"inputs larger than L2 ({2 * w.n / 1e9:.1f} GB of shards); no flush"},
        "e2e": None, "gpu_launches": g["gpu_launches"],
        "roofline": g["roofline"],
        "cpu_baseline": (gather_cpu_rate(w, args.cpu_seconds) if args.cpu_seconds > 0
                         else None),
        "clocks": clk,
    }
    if prefetch is not None:
        line["prefetch"] = prefetch
    print(json.dumps(line))
    plan.close()
    return 0


def main(argv=None):
    from synth import workloads as wl
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--op", default="step", choices=["step", "gather"],
                    help="the shard step with the gather after it (default), or the gather "
                         "alone")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU oracle baseline budget (0 skips it)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer e2e leg")
    ap.add_argument("--results", default=None, metavar="PATH",
                    help="append one JSON record per kernel (and the step and gather) to "
                         "this file, as JSON lines")
    ap.add_argument("--no-gather", action="store_true",
                    help="step: leave out the gather and the step + gather pass")
    ap.add_argument("--state", default="device", choices=["device", "host"],
                    help="where master/m/v live: HBM, or pinned Grace memory read and "
                         "written over NVLink-C2C (the fp16 parameters stay in HBM)")
    ap.add_argument("--prefetch", action="store_true",
                    help="gather: one launch and one completion event per layer")
    ap.add_argument("--layer-shift", type=int, default=0,
                    help="gather: shift interior layer boundaries by this many elements")
    ap.add_argument("--graph", action="store_true",
                    help="replay the step from a CUDA graph (one per gradient set)")
    ap.add_argument("--one-set", action="store_true",
                    help="one gradient set instead of two (less device memory)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.op == "gather":
        return run_gather(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
