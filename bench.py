#!/usr/bin/env python3
"""Benchmark: barrier-free AllReduce over N virtual ranks on one GB300.

Workload (one "step"): N=4 virtual ranks, message sizes 128 B .. 1 MiB per
rank in powers of two (14 sizes), binary32 and bfloat16 N(0,1) inputs, all
the automatic algorithm choice; each (dtype, size) replays a CUDA graph of
`--inner` back-to-back calls (the decode-style replay path: no host work per
call), timed with CUDA events on the replay stream.  L2 is flushed (a 256 MiB
write) between steps; the calls inside a step reuse their L2-resident
buffers, the regime the small-message latency floor assumes.  The same calls
launched one by one from Python are reported as stream_launch_us.

value     mean over the 28 (dtype, size) cases of microseconds per call with
          the library's automatic choice (RRA_AUTO), lower is better; every
          algorithm's own figure on every case is reported beside it
e2e       the same metric through the host-buffer call (pinned host buffers
          in and out, synchronised per call), and the host link it runs over:
          the device reading, writing, and copying pinned host memory (GB/s)
roofline  the dominant kernel of the step against the measured HBM peak
floor     measured single-GPU latency floor 2*L2_RTT + L_store->poll and the
          in-kernel time of the 128-byte calls
bandwidth the two-shot kernels at N=8, 4 / 64 / 512 MiB per rank, binary32 and
          binary64, GB/s of compulsory traffic (2*N*M) against the measured HBM
          peak, L2 evicted between calls
configs   N=2 128 B over 1000 back-to-back calls; N=64 1 KiB-256 KiB and an N
          sweep at 16 KiB
barrier_baseline  flag-barrier latency vs N, and the one-shot and two-shot
          barrier baselines beside their barrier-free counterparts (N=4)
collectives ReduceScatter, AllGather, Broadcast, Reduce: N=4 latency (graph
          replay) and N=8 bandwidth of compulsory bytes against the HBM peak
cpu_baseline  the CPU oracle on a bounded sample of the same sweep

Output: the last stdout line is one compact JSON object (well under 4 KB):
the headline, roofline, e2e, cpu_baseline, clocks, the latency floor with
the 128-byte in-kernel times, and the bandwidth fractions.  Every table in
full goes to the JSON file --detail-out (default: bench_detail.json in the
system temp directory), whose path the line names.

--impl reference times the CPU oracle itself on the same sweep.
--case ALGO NRANKS BYTES DTYPE REPS [attr=value ...] runs one configuration
REPS times (a load generator for profiling one kernel): it checks the device
status and that every rank received the same bits, and prints one line.

One GPU only.  The N ranks of an AllReduce are virtual and live on one GPU,
and the library's bulk-copy push (TMA multicast) is for single-GPU processes,
so --gpus N > 1 (or a torchrun launch with WORLD_SIZE > 1) does no GPU work:
rank 0 prints one JSON line with an "unavailable" reason, every rank exits 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

NRANKS = 4
DTYPES = ("fp32", "bf16")
ALGOS = ("oneshot_ll", "oneshot_sentinel", "twoshot_dbuf", "ll128_atomic", "twoshot_direct", "oneshot_cluster",
         "twoshot_cluster")
ELEM = {"fp32": 4, "bf16": 2, "fp64": 8}
METRIC = "AllReduce us/call at 128B-1MB; GB/s vs HBM roofline; N virtual ranks, 1 GB300"
WORKLOAD = "N=4 virtual ranks, 128 B-1 MiB per rank (14 sizes), fp32+bf16 N(0,1), automatic algorithm choice"


# ----------------------------------------------------------------- ranks --
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


MULTI_GPU_REASON = ("one GPU only: the N ranks are virtual ranks on one GPU, and the bulk-copy push "
                    "(TMA multicast) is for single-GPU processes; no multi-GPU run")


def multi_gpu_line(n_gpus):
    """The line printed instead of a measurement when more than one GPU is asked for."""
    return {"metric": METRIC, "n_gpus": n_gpus, "unavailable": MULTI_GPU_REASON}


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_dir=None):
        import tempfile

        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(log_dir or tempfile.gettempdir(), "clocks_rank%d.csv" % gpu_index)

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- helpers ----
def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


# The translation unit of the profiled kernels (cluster_kernel,
# cluster_tma_kernel): cluster.cu and every header it includes.
KERNEL_SOURCES = ("latency_barrier_free_gb300/csrc/cluster.cu", "latency_barrier_free_gb300/csrc/cluster_prims.cuh",
                  "latency_barrier_free_gb300/csrc/prims.cuh", "latency_barrier_free_gb300/csrc/rra_internal.h",
                  "include/rra.h")


def strip_comments(text):
    """C/C++ source without its comments and blank lines (the kernel sources
    hold no comment markers inside string literals)."""
    import re

    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_sha():
    """Hash of the profiled kernels' sources, comments and blank lines left
    out: the source a profile's DRAM traffic belongs to."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(f.encode() + b"\0")
        h.update(strip_comments(open(os.path.join(ROOT, f)).read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(kernel, config):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    except (OSError, ValueError):
        return None
    for e in rec.get("entries", []):
        if e.get("kernel") == kernel and e.get("config") == config and e.get("source_sha") == kernel_source_sha():
            return e.get("dram_bytes_per_launch")
    return None


def to_device(arrs, dtype):
    """Host numpy arrays (bfloat16 as uint16 bit patterns) -> CUDA tensors."""
    import torch

    out = []
    for a in arrs:
        if dtype == "bf16":
            out.append(torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(torch.bfloat16).cuda())
        else:
            out.append(torch.from_numpy(np.ascontiguousarray(a).copy()).cuda())
    return out


def sweep_cases():
    from latency_barrier_free_gb300 import inputs

    return [(dt, size) for dt in DTYPES for size in inputs.W2_SIZES]


# ------------------------------------------------------------ our arm ----
def run_ours(args):
    import torch

    import __graft_entry__
    from latency_barrier_free_gb300 import inputs, measure, rra

    __graft_entry__.build()
    local = 0
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(dev)

    comm = rra.Comm(NRANKS, 1 << 20)
    cases = sweep_cases()
    clocks = ClockSampler(local, args.clock_log_dir)
    clocks.start()
    bufs = {}
    for dt, size in cases:
        sends = to_device(inputs.workload2(size, dt), dt)
        recvs = [torch.empty_like(s) for s in sends]
        bufs[(dt, size)] = ([s.data_ptr() for s in sends], [r.data_ptr() for r in recvs], size // ELEM[dt],
                            sends, recvs)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    inner = args.inner

    # One CUDA graph per case holding `inner` back-to-back calls (decode-style
    # replay: no host work per call).  The calls are prepared with the capture
    # stream so they are recorded into the graph.
    cap = torch.cuda.Stream()

    def make_graph(dt, size, algo):
        sp, rp, count, _, _ = bufs[(dt, size)]
        f = comm.prepare(sp, rp, count, dt, algo, stream=cap)
        f()  # plan/occupancy queries happen outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for _ in range(inner):
                    f()
        return g

    auto_graphs = {(dt, size): make_graph(dt, size, "auto") for dt, size in cases}
    torch.cuda.synchronize()

    def one_step(events):
        for k, (dt, size) in enumerate(cases):
            if events is not None:
                events[k][0].record(stream)
            auto_graphs[(dt, size)].replay()
            if events is not None:
                events[k][1].record(stream)

    for w in range(args.warmup):
        flush.fill_(w & 0xFF)
        one_step(None)
    torch.cuda.synchronize()
    st = comm.status()[0]
    if st != rra.OK:
        raise RuntimeError("device status after warm-up: %s" % rra.STATUS_NAMES.get(st))

    ncase = len(cases)
    per_step_events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                        for _ in range(ncase)] for _ in range(args.steps)]
    step_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
    torch.cuda.synchronize()
    for s in range(args.steps):
        flush.fill_(s & 0xFF)          # evict the previous step's lines from L2
        step_events[s][0].record(stream)
        one_step(per_step_events[s])
        step_events[s][1].record(stream)
    torch.cuda.synchronize()
    st = comm.status()[0]
    if st != rra.OK:
        raise RuntimeError("device status after timed region: %s" % rra.STATUS_NAMES.get(st))

    step_ms = [a.elapsed_time(b) for a, b in step_events]
    auto_us = {}
    for k, (dt, size) in enumerate(cases):
        vals = [per_step_events[s][k][0].elapsed_time(per_step_events[s][k][1]) * 1000.0 / inner
                for s in range(args.steps)]
        auto_us[(dt, size)] = measure.median(vals)
    value = float(np.mean([auto_us[c] for c in cases]))
    auto_pick = {c: rra.select_algo(NRANKS, c[1], c[0]) for c in cases}

    # Every algorithm on every case, measured the same way outside the timed
    # step (context for the automatic choice).
    us_call = {}
    for dt, size in cases:
        for algo in ALGOS:
            g = make_graph(dt, size, algo)
            ts = []
            for _ in range(max(3, args.steps)):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1000.0 / inner)
            us_call[(dt, size, algo)] = measure.median(ts)
            del g
    stream_us = stream_launch_us(comm, bufs, cases, torch, stream)
    best = {(dt, size): min(ALGOS, key=lambda a: us_call[(dt, size, a)]) for dt, size in cases}
    best_us = float(np.mean([us_call[(dt, size, best[(dt, size)])] for dt, size in cases]))
    per_algo_mean = {a: float(np.mean([us_call[(dt, size, a)] for dt, size in cases])) for a in ALGOS}

    # Dominant kernel of the timed step: the kernel (template) whose launches
    # take the most of the step's time; every case launches `inner` calls, so
    # its per-launch average is the sum of the cases' algorithmic bytes over
    # the sum of their per-call times.  The single launch configuration with
    # the largest per-call time is reported beside it.
    # the __global__ function each case launches (as a profiler's launch list
    # names it), from the library's own plan of the call
    launched = {c: comm.plan_kernel(c[1] // ELEM[c[0]], c[0], "auto") for c in cases}
    by_kernel = {}
    for c in cases:
        by_kernel.setdefault(launched[c].split("<")[0], []).append(c)
    kname = max(by_kernel, key=lambda k: sum(auto_us[c] for c in by_kernel[k]))
    kcases = by_kernel[kname]
    peaks = measured_peaks()
    hbm_peak = peaks.get("hbm_gbs")
    peak_src = "measured" if hbm_peak else "fallback"
    hbm_peak = hbm_peak or 6800.0
    k_bytes = float(np.mean([measure.algorithmic_bytes(NRANKS, c[1]) for c in kcases]))
    k_us = float(np.mean([auto_us[c] for c in kcases]))
    achieved = k_bytes / (k_us * 1e-6) / 1e9
    k_cfg = "auto step N=%d fp32+bf16 128B-1MiB, all launches" % NRANKS
    dom_case = max(cases, key=lambda c: auto_us[c])
    dom_dt, dom_size = dom_case
    dom_algo = auto_pick[dom_case]
    dom_cfg = "%s N=%d %s %dB" % (dom_algo, NRANKS, dom_dt, dom_size)
    dom_achieved = measure.algorithmic_bytes(NRANKS, dom_size) / (auto_us[dom_case] * 1e-6) / 1e9
    dom_kernel = launched[dom_case].split("<")[0]
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4), "traffic": committed_traffic(kname, k_cfg),
                "kernel": kname, "config": k_cfg, "launches_per_step": len(kcases) * inner,
                "bytes_per_launch": round(k_bytes, 1), "us_per_launch": round(k_us, 3),
                "share_of_step": round(sum(auto_us[c] for c in kcases) / sum(auto_us.values()), 4),
                "peak_source": peak_src,
                "note": "per-launch average over the step (2*N*M algorithmic bytes, graph-replay time per call); "
                        "at <= 1 MiB per rank the kernel is latency-bound: see latency_floor",
                "launched": {"%s/%d" % c: launched[c] for c in cases},
                "largest_launch": {"config": dom_cfg, "kernel": launched[dom_case],
                                   "achieved": round(dom_achieved, 1), "frac": round(dom_achieved / hbm_peak, 4),
                                   "traffic": committed_traffic(dom_kernel, dom_cfg)}}

    floor = latency_floor(comm, rra, measure, torch, stream)
    clk = clocks.stop()
    bandwidth = bandwidth_end(rra, measure, torch, hbm_peak, args)
    colls = collectives_table(rra, measure, torch, hbm_peak) if args.collectives else None
    barriers = barrier_table(rra, measure, torch) if args.barriers else None
    sweep = scratch_sweep(rra, measure, torch) if args.scratch_sweep else None
    configs = configs_table(rra, measure, torch) if args.configs else None
    e2e = end_to_end(comm, rra, cases, torch, args)
    decode = decode_graph(rra, torch) if args.decode else None

    ms_step = float(np.mean(step_ms))
    launches = args.steps * ncase * inner  # one kernel per call, all ours
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "us/call", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "fp32+bf16",
        "data": "synthetic (seeded N(0,1), no dataset)",
        "config": {"workload": WORKLOAD, "nranks": NRANKS, "sizes_bytes": [c[1] for c in cases if c[0] == "fp32"],
                   "inner_calls": inner, "l2": "flushed (256 MiB write) between steps; calls in a step reuse "
                   "L2-resident buffers", "parallelism": "single GPU",
                   "gpu": props.name, "sms": props.multi_processor_count},
        "gpu_launches": launches,
        "roofline": roofline,
        "latency_floor": floor,
        "bandwidth": bandwidth,
        "e2e": e2e,
        "clocks": clk,
        "auto_us": {"%s/%d" % k: round(v, 3) for k, v in auto_us.items()},
        "auto_algo": {"%s/%d" % k: v for k, v in auto_pick.items()},
        "best_of_algos_mean_us": round(best_us, 3),
        "per_algo_mean_us": {a: round(v, 3) for a, v in per_algo_mean.items()},
        "stream_launch_us": stream_us,
        "per_size_us": {"%s/%d" % (dt, size): {a: round(us_call[(dt, size, a)], 3) for a in ALGOS}
                        for dt, size in cases},
        "best_algo": {"%s/%d" % k: v for k, v in best.items()},
    }
    if decode is not None:
        line["decode_graph"] = decode
    if colls is not None:
        line["collectives"] = colls
    if barriers is not None:
        line["barrier_baseline"] = barriers
    if sweep is not None:
        line["scratch_sweep"] = sweep
    if configs is not None:
        line["configs"] = configs
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    comm.close()
    import tempfile

    path = args.detail_out or os.path.join(tempfile.gettempdir(), "bench_detail.json")
    try:
        with open(path, "w") as f:
            json.dump(line, f, indent=1)
    except OSError as e:
        print("bench: could not write %s: %s" % (path, e), file=sys.stderr)
        path = None
    print(json.dumps(summary_line(line, path)), flush=True)


# the algorithms whose 128-byte in-kernel time the summary line reports
NAMED = ("oneshot_ll", "oneshot_sentinel", "twoshot_dbuf", "ll128_atomic", "oneshot_cluster")
SUMMARY_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "gpu_launches")


def summary_line(d, detail_path):
    """The compact last line (well under 4 KB) from the full result `d`."""
    out = {k: d[k] for k in SUMMARY_KEYS if k in d}
    c = d.get("config", {})
    sizes = c.get("sizes_bytes") or []
    out["config"] = {"workload": c.get("workload"), "nranks": c.get("nranks"),
                     "sizes_bytes": "%d-%d" % (min(sizes), max(sizes)) if sizes else None,
                     "inner_calls": c.get("inner_calls"), "l2": c.get("l2"), "gpu": c.get("gpu"), "sms": c.get("sms")}
    r = d.get("roofline", {})
    out["roofline"] = {k: r.get(k) for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "kernel",
                                             "us_per_launch", "bytes_per_launch", "share_of_step", "peak_source")}
    if "cpu_baseline" in d:
        out["cpu_baseline"] = d["cpu_baseline"]
    e = d.get("e2e", {})
    out["e2e"] = {k: e.get(k) for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "host_link_GBps")}
    out["e2e"]["api"] = "rra_allreduce_mapped on pinned host buffers (zero copy), synchronised per call"
    ck = d.get("clocks", {})
    out["clocks"] = {k: ck.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")}
    f = d.get("latency_floor", {})
    kern = f.get("in_kernel_us_128B", {})
    floors = {"l2": f.get("floor_us"), "dsmem": f.get("floor_dsmem_us")}
    lf = {"floor_us": f.get("floor_us"), "floor_dsmem_us": f.get("floor_dsmem_us"), "in_kernel_us_128B": {},
          "x_floor": {}}
    for key, us in kern.items():
        algo = key.split("/", 1)[1]
        if algo not in NAMED:
            continue
        lf["in_kernel_us_128B"][key] = us
        ref = floors["dsmem"] if algo.endswith("cluster") else floors["l2"]
        if ref:
            lf["x_floor"][key] = round(us / ref, 2)
    out["latency_floor"] = lf
    bw = d.get("bandwidth", {}).get("sizes", {})
    out["bandwidth_hbm_frac"] = {k: v.get("frac") for k, v in bw.items() if "MiB" in k}
    out["detail"] = detail_path
    return out


def run_case(args):
    """--case ALGO NRANKS BYTES DTYPE REPS [attr=value ...]: one configuration
    REPS times, for profiling one kernel (seeded uniform(-1, 1) inputs on the
    device).  Checks the device status and that every rank got the same bits.
    ALGO may also name a collective (reduce_scatter, all_gather, broadcast,
    reduce; root 0), BYTES then being one block; for those the check is the
    device status, plus identical outputs for AllGather and Broadcast."""
    import torch

    import __graft_entry__
    from latency_barrier_free_gb300 import rra

    a = args.case
    if len(a) < 5:
        raise SystemExit("--case needs ALGO NRANKS BYTES DTYPE REPS [attr=value ...]")
    algo, n, size, dtype, reps = a[0], int(a[1]), int(a[2]), a[3], int(a[4])
    attrs = dict(x.split("=", 1) for x in a[5:])
    __graft_entry__.build()
    tdt = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp64": torch.float64}[dtype]
    count = size // ELEM[dtype]
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    if algo in rra.COLLECTIVES:
        blocks_in = n if algo == "reduce_scatter" else 1
        blocks_out = n if algo == "all_gather" else 1
        xs = [(torch.rand(blocks_in * count, device="cuda", generator=g) * 2 - 1).to(tdt) for _ in range(n)]
        ys = [torch.empty(blocks_out * count, dtype=tdt, device="cuda") for _ in range(n)]
        with rra.Comm(n, n * size) as c:
            for k, v in attrs.items():
                c.set_attr(k, int(v))
            sp, rp = [t.data_ptr() for t in xs], [t.data_ptr() for t in ys]
            for _ in range(reps):
                c.collective_ptrs(algo, sp, rp, count, dtype, 0)
            torch.cuda.synchronize()
            st = c.status()[0]
            same = algo in ("reduce_scatter", "reduce") or all(
                torch.equal(ys[0].view(torch.uint8), y.view(torch.uint8)) for y in ys[1:])
            print(json.dumps({"case": a, "kernel": c.last_kernel(), "status": rra.STATUS_NAMES.get(st),
                              "ranks_identical": same}), flush=True)
            return 0 if st == rra.OK and same else 1
    xs = [(torch.rand(count, device="cuda", generator=g) * 2 - 1).to(tdt) for _ in range(n)]
    ys = [torch.empty_like(x) for x in xs]
    with rra.Comm(n, size) as c:
        for k, v in attrs.items():
            c.set_attr(k, int(v))
        grid, steps = c.plan_call(count, dtype, algo)
        for _ in range(reps):
            c.allreduce(xs, ys, algo)
        torch.cuda.synchronize()
        st = c.status()[0]
        same = all(torch.equal(ys[0].view(torch.uint8), y.view(torch.uint8)) for y in ys[1:])
        print(json.dumps({"case": a, "kernel": c.last_kernel(), "grid": grid, "steps": steps,
                          "status": rra.STATUS_NAMES.get(st), "ranks_identical": same}), flush=True)
        return 0 if st == rra.OK and same else 1


def stream_launch_us(comm, bufs, cases, torch, stream, reps=400):
    """The same calls launched one by one from Python on a stream (prepared
    arguments): host-bound, reported next to the graph figure."""
    out = {}
    for dt, size in [c for c in cases if c[1] in (128, 65536, 1 << 20)]:
        sp, rp, count, _, _ = bufs[(dt, size)]
        for algo in ALGOS:
            f = comm.prepare(sp, rp, count, dt, algo)
            for _ in range(20):
                f()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            e0.record(stream)
            for _ in range(reps):
                f()
            e1.record(stream)
            host = (time.perf_counter() - t0) / reps * 1e6
            torch.cuda.synchronize()
            out["%s/%d/%s" % (dt, size, algo)] = {"gpu_us": round(e0.elapsed_time(e1) * 1000.0 / reps, 3),
                                                  "host_us": round(host, 3)}
    return out


def latency_floor(comm, rra, measure, torch, stream):
    """Measured floor 2*L2_RTT + L_store->poll next to the in-kernel time of the
    128-byte calls (N=2 and N=4) and the empty-kernel launch overhead."""
    l2 = [rra.probe_l2_chase(8 << 20, 100000, seed) for seed in (1, 2, 3)]
    sms = rra.probe_sm_count()
    # 32 CTA pairs spread over the grid.  Which SMs a pair lands on changes
    # from launch to launch, and a pair on one die answers in about half the
    # time of a pair across the two dies, so the floor takes the mean over
    # pairs (the expected latency between two ranks placed anywhere).
    pairs = [(0, j) for j in sorted({max(1, (k * sms) // 32) for k in range(32)} | {sms - 1}) if j > 0][:32]
    rtts, sm_pairs = [], []
    for a, b in pairs:
        rtt, sa, sb = rra.probe_pingpong(a, b, 20000)
        rtts.append(rtt)
        sm_pairs.append((sa, sb))
    l2_ns = measure.median(l2)
    store_ns = float(np.mean(rtts)) / 2.0
    floor_ns = measure.sol_floor_ns(l2_ns, store_ns)
    # the floor of the cluster kernels' transport: a bulk copy from an
    # L2-resident input into a peer CTA's shared memory (half a ping-pong
    # round trip inside one cluster) plus the one cluster barrier before it
    ds = [rra.probe_dsmem_pingpong(20000) for _ in range(3)]
    ds_rtt = measure.median([d[0] for d in ds])
    ds_bar = measure.median([d[1] for d in ds])
    dsmem_floor_ns = ds_rtt / 2.0 + ds_bar

    def in_kernel(n, algo, reps=200):
        with rra.Comm(n, 128) as c:
            grid, _ = c.plan_call(32, "fp32", algo)
            buf = torch.zeros(reps, 2 * grid, dtype=torch.int64, device="cuda")
            xs = [torch.randn(32, device="cuda") for _ in range(n)]
            ys = [torch.empty_like(x) for x in xs]
            for i in range(reps):
                c.set_timing(buf[i].data_ptr())
                c.allreduce(xs, ys, algo)
            torch.cuda.synchronize()
            c.set_timing(0)
            t = buf.view(reps, grid, 2).cpu().numpy()
            spans = (t[:, :, 1].max(axis=1) - t[:, :, 0].min(axis=1)) / 1000.0
            return float(np.median(spans[reps // 10:]))

    kern = {}
    for n in (2, 4):
        for algo in ALGOS:
            kern["N%d/%s" % (n, algo)] = round(in_kernel(n, algo), 3)
    best_key = min(kern, key=kern.get)
    # empty-kernel and graph-node overhead, same run
    reps = 2000
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(100):
        rra.probe_empty_kernel()
    e0.record(stream)
    for _ in range(reps):
        rra.probe_empty_kernel()
    e1.record(stream)
    torch.cuda.synchronize()
    empty_us = e0.elapsed_time(e1) * 1000.0 / reps
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(160):
                rra.probe_empty_kernel()
    g.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(20):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    node_us = e0.elapsed_time(e1) * 1000.0 / (20 * 160)

    # the same for an empty kernel launched as the 128-byte cluster AllReduce
    # at N=4 is (4 CTAs of 32 threads, one cluster, programmatic dependent
    # launch): the per-call floor of back-to-back dependent calls of that shape
    def chain_us(cluster, pdl):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            rra.probe_launch_chain(4, 32, cluster, pdl, s)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                for _ in range(160):
                    rra.probe_launch_chain(4, 32, cluster, pdl, s)
        g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(20):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return round(e0.elapsed_time(e1) * 1000.0 / (20 * 160), 3)

    chain = {"cluster4_pdl": chain_us(4, True), "cluster4": chain_us(4, False), "pdl": chain_us(1, True)}

    def over(key):
        ref = dsmem_floor_ns if key.endswith("cluster") else floor_ns
        return round(kern[key] / (ref / 1000.0), 3)

    return {"l2_rtt_ns": round(l2_ns, 1), "store_poll_ns": round(store_ns, 1),
            "pingpong_rtt_ns": [round(x, 1) for x in rtts], "pingpong_sms": sm_pairs,
            "floor_us": round(floor_ns / 1000.0, 3),
            "dsmem_bulk_rtt_ns": round(ds_rtt, 1), "cluster_barrier_ns": round(ds_bar, 1),
            "dsmem_sms": [d[2:] for d in ds], "floor_dsmem_us": round(dsmem_floor_ns / 1000.0, 3),
            "in_kernel_us_128B": kern, "x_floor": {k: over(k) for k in kern}, "best_in_kernel": best_key,
            "best_over_floor": over(best_key),
            "empty_kernel_us": round(empty_us, 3), "graph_node_us": round(node_us, 3),
            "chain_node_us": chain,
            "method": "L2 RTT: dependent ld.global.cg chase, 8 MiB random cycle; store->poll: half the mean RTT "
                      "of a fence-free ping-pong between CTA 0 and 32 CTAs on other SMs (same-die and cross-die "
                      "pairs); floor = 2 L2 RTT + store->poll for the global-memory kernels; floor_dsmem = half "
                      "the RTT of a bulk-copy ping-pong between the 2 CTAs of a cluster (128 B from an "
                      "L2-resident buffer into the peer's shared memory, completing its mbarrier) + one cluster "
                      "barrier, for the cluster kernels; in-kernel: %globaltimer first CTA start to last CTA end, "
                      "median of 180 calls"}


def bandwidth_end(rra, measure, torch, hbm_peak, args):
    """Workload 5: N=8, binary32 and binary64 uniform(-1, 1), 4 / 64 / 512 MiB
    per rank, the two-shot kernels.  Enough buffer sets are rotated that
    each call's working set was evicted from L2 (more than 2x its 129 MB).
    The calls are timed as a CUDA graph replay of the rotation (device time,
    launch gaps included); issued one by one from Python, the marshalling of
    16 tensors per call (about 20 us) would set the pace at 4 MiB per rank,
    so that figure is kept beside it as `eager_ms`."""
    out = {}
    n = 8
    sizes = [4 << 20, 64 << 20] + ([512 << 20] if args.big else [])
    for dtype in ("fp32", "fp64"):
        es = 4 if dtype == "fp32" else 8
        tdt = torch.float32 if dtype == "fp32" else torch.float64
        algos = ("twoshot_dbuf", "twoshot_direct", "twoshot_cluster") if dtype == "fp32" else (
            "twoshot_dbuf", "twoshot_cluster")
        for size in sizes:
            count = size // es
            nsets = max(1, -(-(300 << 20) // (2 * n * size)))
            gen = torch.Generator(device="cuda")
            gen.manual_seed(5000 + size // (1 << 20) + es)
            with rra.Comm(n, size) as c:
                sets = []
                for _ in range(nsets):
                    xs = [(torch.rand(count, device="cuda", generator=gen) * 2 - 1).to(tdt) for _ in range(n)]
                    sets.append((xs, [torch.empty_like(x) for x in xs]))
                for algo in algos:
                    for k in range(2):
                        c.allreduce(*sets[k % nsets], algo)
                    torch.cuda.synchronize()
                    reps = max(5, nsets)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for k in range(reps):
                        c.allreduce(*sets[k % nsets], algo)
                    e1.record()
                    torch.cuda.synchronize()
                    t_eager = e0.elapsed_time(e1) / 1000.0 / reps
                    cap = torch.cuda.Stream()
                    cap.wait_stream(torch.cuda.current_stream())
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=cap):
                        for k in range(reps):
                            c.allreduce(*sets[k % nsets], algo)
                    g.replay()
                    torch.cuda.synchronize()
                    ts = []
                    for _ in range(3):
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record()
                        g.replay()
                        e1.record()
                        torch.cuda.synchronize()
                        ts.append(e0.elapsed_time(e1) / 1000.0 / reps)
                    del g
                    st = c.status()[0]
                    t = measure.median(ts)
                    gbs = measure.hbm_gbs(n, size, t)
                    out["%s/%s/%dMiB" % (algo, dtype, size >> 20)] = {
                        "ms": round(t * 1000, 3), "GB/s": round(gbs, 1), "frac": round(gbs / hbm_peak, 4),
                        "busbw_GB/s": round(measure.busbw_gbs(n, size, t), 1), "eager_ms": round(t_eager * 1000, 3),
                        "status": rra.STATUS_NAMES.get(st)}
                del sets
            torch.cuda.empty_cache()
    return {"nranks": n, "bytes": "2*N*M per call", "sizes": out,
            "note": "L2 evicted between calls (rotating buffer sets, >2x L2); CUDA events around a CUDA-graph "
                    "replay of the rotation (eager_ms: the same calls issued one by one from Python); default chunking"}


def _graph_us(torch, measure, fn, calls=16, reps=20):
    """Median microseconds per call of `fn` replayed `calls` times in a CUDA graph."""
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1000.0 / calls)
    return round(measure.median(ts), 3)


def configs_table(rra, measure, torch):
    """The other configurations' own figures.  Config 1: N=2, 32 binary32
    integers, 1000 back-to-back calls on distinct buffers in one graph.
    Config 4: N=64, binary32, 1 KiB..256 KiB, and an N sweep at 16 KiB, with
    each algorithm's scratch bytes per window (µs per call, graph replay)."""
    from latency_barrier_free_gb300 import inputs

    out = {}
    calls = 1000
    host = np.stack([np.stack(inputs.workload1(i)) for i in range(calls)])
    send = torch.from_numpy(host).cuda()
    recv = torch.empty_like(send)
    c1 = {}
    with rra.Comm(2, 128) as c:
        for algo in ("oneshot_ll", "oneshot_sentinel", "oneshot_cluster", "auto"):
            def step(algo=algo):
                for i in range(calls):
                    c.allreduce_ptrs([send[i, 0].data_ptr(), send[i, 1].data_ptr()],
                                     [recv[i, 0].data_ptr(), recv[i, 1].data_ptr()], 32, "fp32", algo)
            c1[algo] = round(_graph_us(torch, measure, step, calls=1, reps=5) / calls, 3)
        assert c.status()[0] == rra.OK
    exact = host.astype(np.int64).sum(axis=1).astype(np.float32)
    out["config1_N2_128B_us_per_call"] = c1
    out["config1_exact"] = bool(np.array_equal(recv.cpu().numpy()[:, 0], exact))
    algos = ("oneshot_sentinel", "ll128_atomic", "auto")
    c4 = {}
    with rra.Comm(64, 256 << 10) as c:
        lay = c.layout()
        for size in inputs.W4_SIZES:
            count = size // 4
            xs = [torch.randn(count, device="cuda") for _ in range(64)]
            ys = [torch.empty_like(x) for x in xs]
            sp, yp = [t.data_ptr() for t in xs], [t.data_ptr() for t in ys]
            for algo in algos:
                c4["%s/%dB" % (algo, size)] = _graph_us(torch, measure, lambda: c.allreduce_ptrs(sp, yp, count, "fp32", algo))
        assert c.status()[0] == rra.OK
    out["config4_N64_us_per_call"] = c4
    out["config4_scratch_bytes_per_window"] = {"oneshot_sentinel": lay["os_bytes"], "ll128_atomic": lay["la_bytes"],
                                               "max_bytes": 256 << 10}
    sweep = {}
    for n in inputs.W4_NSWEEP:
        count = (16 << 10) // 4
        with rra.Comm(n, 16 << 10) as c:
            xs = [torch.randn(count, device="cuda") for _ in range(n)]
            ys = [torch.empty_like(x) for x in xs]
            sp, yp = [t.data_ptr() for t in xs], [t.data_ptr() for t in ys]
            for algo in algos + (("oneshot_cluster", "twoshot_cluster") if n <= 16 else ()):
                sweep["N%d/%s" % (n, algo)] = _graph_us(torch, measure, lambda: c.allreduce_ptrs(sp, yp, count, "fp32", algo))
            assert c.status()[0] == rra.OK
    out["nsweep_16KiB_us_per_call"] = sweep
    return out


def barrier_table(rra, measure, torch):
    """The design the paper replaces, measured beside the barrier-free one:
    the flag barrier's latency against N (one CTA per rank, back to back),
    and at N=4 binary32 the barrier baselines against their barrier-free
    counterparts (CUDA-graph replay of 16 calls, µs per call)."""
    lat = {}
    for n in (2, 4, 8, 16, 64):
        with rra.Comm(n, 4096) as c:
            lat["N%d" % n] = round(c.barrier_latency(2000) / 1000.0, 3)
    pairs = (("oneshot_barrier", "oneshot_sentinel"), ("twoshot_barrier", "twoshot_dbuf"))
    cap = torch.cuda.Stream()
    us = {}
    n = 4
    for m in (128, 65536, 1 << 20):
        count = m // 4
        with rra.Comm(n, m) as c:
            xs = [torch.randn(count, device="cuda") for _ in range(n)]
            ys = [torch.empty_like(x) for x in xs]
            for pair in pairs:
                for algo in pair:
                    f = c.prepare([t.data_ptr() for t in xs], [t.data_ptr() for t in ys], count, "fp32", algo,
                                  stream=cap)
                    f()
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    cap.wait_stream(torch.cuda.current_stream())
                    with torch.cuda.graph(g, stream=cap):
                        for _ in range(16):
                            f()
                    g.replay()
                    torch.cuda.synchronize()
                    ts = []
                    for _ in range(20):
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record()
                        g.replay()
                        e1.record()
                        torch.cuda.synchronize()
                        ts.append(e0.elapsed_time(e1) * 1000.0 / 16)
                    us["%s/%dB" % (algo, m)] = round(measure.median(ts), 3)
                    del g
            assert c.status()[0] == rra.OK
    return {"barrier_us_vs_N": lat, "N4_fp32_us_per_call": us,
            "pairs": ["%s vs %s" % p for p in pairs]}


# live scratch per window as a function of the per-rank step (chunk) bytes
SCRATCH_OF_CHUNK = {
    "oneshot_sentinel": ("oneshot_chunk", lambda n, ch: 2 * n * ch),      # 2 parities x N slots
    "oneshot_ll": ("oneshot_chunk", lambda n, ch: 4 * n * ch),            # LL doubles every byte
    "twoshot_dbuf": ("twoshot_chunk", lambda n, ch: 4 * ch),              # RS + AG, 2 parities, N parts
    "twoshot_direct": ("twoshot_chunk", lambda n, ch: 2 * ch),            # RS only
    "ll128_atomic": ("ll128_chunk", lambda n, ch: 4 * ch + 4 * ch // n),  # LL AllGather + accumulators
}


def scratch_sweep(rra, measure, torch):
    """Fig. 12 restated: AllReduce latency against the scratch each window
    keeps live, set through the per-step chunk, N=8 binary32, 1 MiB and
    16 MiB per rank (stream-ordered calls, CUDA events, 2 warm-up + 10)."""
    n = 8
    out = {}
    for size in (1 << 20, 16 << 20):
        count = size // 4
        with rra.Comm(n, size) as c:
            xs = [torch.randn(count, device="cuda") for _ in range(n)]
            ys = [torch.empty_like(x) for x in xs]
            for algo, (attr, scratch) in SCRATCH_OF_CHUNK.items():
                if algo.startswith("oneshot") and size > (1 << 20):
                    continue
                for kib in (16, 64, 256, 1024, 4096, 16384, 65536):
                    chunk = kib << 10
                    if chunk > size:
                        continue
                    c.set_attr(attr, chunk)
                    for _ in range(2):
                        c.allreduce(xs, ys, algo)
                    torch.cuda.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    for _ in range(10):
                        c.allreduce(xs, ys, algo)
                    e1.record()
                    torch.cuda.synchronize()
                    out["%s/%dMiB/chunk%dKiB" % (algo, size >> 20, kib)] = {
                        "us": round(e0.elapsed_time(e1) * 100.0, 2),
                        "scratch_KiB": scratch(n, chunk) >> 10}
                c.set_attr(attr, 0)
            assert c.status()[0] == rra.OK
    return out


def collective_bytes(op, n, m):
    """Compulsory HBM bytes of one call: every input read once, every output
    written once (m = bytes of one block of `count` elements)."""
    return {"reduce_scatter": n * n * m + n * m, "all_gather": n * m + n * n * m,
            "broadcast": m + n * m, "reduce": n * m + m}[op]


def collectives_table(rra, measure, torch, hbm_peak):
    """ReduceScatter, AllGather, Broadcast (root 0) and Reduce (root 0):
    latency (CUDA-graph replay of 16 calls, L2-resident buffers) at N=4 with
    128 B, 64 KiB and 1 MiB per block and at N=64 with 1 KiB and 16 KiB, and
    N=8 bandwidth (inputs and outputs far beyond L2) at 16 MiB blocks
    (ReduceScatter, AllGather) / 64 MiB (Broadcast, Reduce), binary32."""
    lat = {4: {}, 64: {}}
    cap = torch.cuda.Stream()
    for n, m in [(4, 128), (4, 65536), (4, 1 << 20), (64, 1024), (64, 16384)]:
        count = m // 4
        with rra.Comm(n, n * m) as c:
            big = [torch.randn(n * count, device="cuda") for _ in range(n)]
            small = [torch.randn(count, device="cuda") for _ in range(n)]
            io = {"reduce_scatter": (big, small), "all_gather": (small, big),
                  "broadcast": (small, [torch.empty_like(t) for t in small]),
                  "reduce": (small, [torch.empty_like(t) for t in small])}
            for op in rra.COLLECTIVES:
                sends, recvs = io[op]
                f = c.prepare_collective(op, [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs],
                                         count, "fp32", 0, stream=cap)
                f()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                cap.wait_stream(torch.cuda.current_stream())
                with torch.cuda.graph(g, stream=cap):
                    for _ in range(16):
                        f()
                g.replay()
                torch.cuda.synchronize()
                ts = []
                for _ in range(20):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    g.replay()
                    e1.record()
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1000.0 / 16)
                lat[n]["%s/%dB" % (op, m)] = round(measure.median(ts), 3)
                del g
            assert c.status()[0] == rra.OK
    bw = {}
    n = 8
    for op in rra.COLLECTIVES:
        m = (16 << 20) if op in ("reduce_scatter", "all_gather") else (64 << 20)
        count = m // 4
        blocks_in = n if op == "reduce_scatter" else 1
        blocks_out = n if op == "all_gather" else 1
        with rra.Comm(n, n * m) as c:
            sends = [torch.rand(blocks_in * count, device="cuda") for _ in range(n)]
            recvs = [torch.empty(blocks_out * count, device="cuda") for _ in range(n)]
            sp, rp = [t.data_ptr() for t in sends], [t.data_ptr() for t in recvs]
            for _ in range(2):
                c.collective_ptrs(op, sp, rp, count, "fp32", 0)
            torch.cuda.synchronize()
            reps = 5
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                c.collective_ptrs(op, sp, rp, count, "fp32", 0)
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) / 1000.0 / reps
            gbs = collective_bytes(op, n, m) / t / 1e9
            bw["%s/%dMiB" % (op, m >> 20)] = {"ms": round(t * 1000, 3), "GB/s": round(gbs, 1),
                                              "frac": round(gbs / hbm_peak, 4),
                                              "status": rra.STATUS_NAMES.get(c.status()[0])}
            del sends, recvs
        torch.cuda.empty_cache()
    return {"latency_us_N4_fp32": lat[4], "latency_us_N64_fp32": lat[64], "bandwidth_N8_fp32": bw,
            "bytes": "compulsory: every input read once, every output written once"}


def end_to_end(comm, rra, cases, torch, args):
    """Host buffers in and out through rra_allreduce_host (pinned memory)."""
    from latency_barrier_free_gb300 import inputs

    reps = max(8, args.inner // 2)
    per = []
    h2d = d2h = 0
    for dt, size in cases:
        count = size // ELEM[dt]
        src = inputs.workload2(size, dt)
        tdt = torch.float32 if dt == "fp32" else torch.bfloat16
        hs = [torch.from_numpy(s.view(np.int16) if dt == "bf16" else s).view(tdt).pin_memory() for s in src]
        hr = [torch.empty_like(h).pin_memory() for h in hs]
        call = comm.prepare_host([h.data_ptr() for h in hs], [h.data_ptr() for h in hr], count, dt, "auto")
        call()
        t0 = time.perf_counter()
        for _ in range(reps):
            call()
        per.append((time.perf_counter() - t0) / reps * 1e6)
        h2d += NRANKS * size
        d2h += NRANKS * size
    # The link these calls run over: the device streaming pinned host memory
    # (32 MiB buffers: the copy's steady rate).  Each case moves N M bytes in
    # and N M bytes out at once, so N M / copy rate is its link-bound time.
    link_r, link_w, link_c = rra.probe_host_link(32 << 20, 10)
    link_us = [round(NRANKS * size / (link_c * 1e3), 2) for _, size in cases]
    return {"value": round(float(np.mean(per)), 3), "unit": "us/call", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "host_link_GBps": {"read": round(link_r, 1), "write": round(link_w, 1), "both": round(link_c, 1)},
            "link_bound_us": link_us,
            "api": "prepared host call (Comm.prepare_host) on pinned host buffers: resolved once by "
                   "rra_host_device_ptrs, then rra_allreduce_mapped per call, synchronised per call; the kernel "
                   "reads the inputs from and writes the outputs to host memory over NVLink-C2C (zero copy)",
            "per_case_us": [round(x, 2) for x in per]}


def decode_graph(rra, torch):
    """N=8, bfloat16 [batch, 8192], 160 AllReduces per token captured in one
    CUDA graph; microseconds per AllReduce = replay time / 160."""
    from latency_barrier_free_gb300 import inputs

    out = {}
    n, calls = 8, inputs.W3_CALLS_PER_TOKEN
    for batch in inputs.W3_BATCHES:
        count = batch * inputs.W3_HIDDEN
        with rra.Comm(n, count * 2) as c:
            xs = [torch.randn(count, device="cuda").to(torch.bfloat16) for _ in range(n)]
            ys = [torch.empty_like(x) for x in xs]
            for algo in ("oneshot_ll", "twoshot_dbuf", "oneshot_cluster", "twoshot_cluster"):
                c.allreduce(xs, ys, algo)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    with torch.cuda.graph(g, stream=s):
                        for _ in range(calls):
                            c.allreduce(xs, ys, algo)
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 10
                e0.record()
                for _ in range(reps):
                    g.replay()
                e1.record()
                torch.cuda.synchronize()
                out["B%d/%s" % (batch, algo)] = round(e0.elapsed_time(e1) * 1000.0 / (reps * calls), 3)
                assert c.status()[0] == rra.OK
            # the layer's AllReduce followed by its residual add: fused into one
            # kernel, against the automatic AllReduce plus a separate add kernel
            # ranks' rows of one [N, count] tensor each, so the unfused add is one kernel
            y_all = torch.empty(n, count, dtype=torch.bfloat16, device="cuda")
            res_all = torch.randn(n, count, device="cuda").to(torch.bfloat16)
            z_all = torch.empty_like(y_all)
            sp = [t.data_ptr() for t in xs]
            qp = [res_all[r].data_ptr() for r in range(n)]
            yp = [y_all[r].data_ptr() for r in range(n)]
            for name in ("fused_residual", "auto+add"):
                def step():
                    if name == "fused_residual":
                        c.allreduce_residual_ptrs(sp, qp, yp, count, "bf16")
                    else:
                        c.allreduce_ptrs(sp, yp, count, "bf16", "auto")
                        torch.add(y_all, res_all, out=z_all)
                step()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    with torch.cuda.graph(g, stream=s):
                        for _ in range(calls):
                            step()
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 10
                e0.record()
                for _ in range(reps):
                    g.replay()
                e1.record()
                torch.cuda.synchronize()
                out["B%d/%s" % (batch, name)] = round(e0.elapsed_time(e1) * 1000.0 / (reps * calls), 3)
                assert c.status()[0] == rra.OK
    return {"us_per_allreduce": out, "calls_per_graph": calls,
            "note": "fused_residual = rra_allreduce_residual; auto+add = rra_allreduce(auto) then one torch add "
                    "kernel over all ranks' rows (the unfused layer epilogue)"}


# ------------------------------------------------------- CPU baseline ----
def cpu_sweep(seconds_budget: float, threads: int):
    """Times the oracle over the sweep cases; returns (mean us/call, reps)."""
    import oracle
    from latency_barrier_free_gb300 import inputs

    cases = sweep_cases()
    data = {c: inputs.workload2(c[1], c[0]) for c in cases}
    outs = {c: [np.empty_like(a) for a in data[c]] for c in cases}
    for c in cases:  # warm-up
        oracle.allreduce_mt(data[c], c[0], threads, recvs=outs[c])
    per = {c: [] for c in cases}
    t_start = time.perf_counter()
    reps = 0
    while True:
        for c in cases:
            t0 = time.perf_counter()
            oracle.allreduce_mt(data[c], c[0], threads, recvs=outs[c])
            per[c].append((time.perf_counter() - t0) * 1e6)
        reps += 1
        if time.perf_counter() - t_start > seconds_budget and reps >= 3:
            break
    us = [float(np.median(per[c])) for c in cases]
    return float(np.mean(us)), reps


def cpu_baseline(seconds_budget: float):
    threads = os.cpu_count() or 1
    v, reps = cpu_sweep(seconds_budget, threads)
    return {"value": round(v, 3), "unit": "us/call", "cores": threads, "kind": "oracle",
            "sample": "the 28-case sweep (N=4, 14 sizes x fp32/bf16), %d repetitions, median per case, "
                      "element range split over %d host threads" % (reps, threads)}


def run_reference(args, world, rank, local):
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    vals = []
    for _ in range(args.warmup):
        cpu_sweep(0.0, threads)
    for _ in range(args.steps):
        v, _ = cpu_sweep(0.0, threads)
        vals.append(v)
    el = time.perf_counter() - t0
    value = float(np.median(vals))
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "us/call", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / max(1, args.steps + args.warmup) * 1000, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "fp32+bf16",
        "data": "synthetic (seeded N(0,1), no dataset)", "impl": "reference",
        "config": {"workload": WORKLOAD, "nranks": NRANKS, "what": "the CPU oracle (no reference code exists)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "us/call", "cores": threads, "kind": "oracle",
                         "sample": "one pass over the 28-case sweep per step"},
        "e2e": {"value": round(value, 3), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--inner", type=int, default=16, help="back-to-back calls per (dtype, size, algo)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-big", dest="big", action="store_false", help="skip the 512 MiB bandwidth case")
    ap.add_argument("--no-decode", dest="decode", action="store_false", help="skip the decode graph case")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-collectives", dest="collectives", action="store_false",
                    help="skip the ReduceScatter/AllGather/Broadcast/Reduce table")
    ap.add_argument("--no-barriers", dest="barriers", action="store_false",
                    help="skip the barrier-baseline table")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the N=2 (1000 calls) and N=64 tables")
    ap.add_argument("--clock-log-dir", default=None,
                    help="directory for the raw nvidia-smi clock samples (default: the system temp directory)")
    ap.add_argument("--scratch-sweep", action="store_true",
                    help="add the latency-vs-scratch sweep of the global-memory kernels (Fig. 12; about a minute)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--detail-out", default=None,
                    help="JSON file for the full result tables (default: bench_detail.json in the temp directory)")
    ap.add_argument("--case", nargs="+", default=None, metavar="ARG",
                    help="ALGO NRANKS BYTES DTYPE REPS [attr=value ...]: run one configuration (profiling)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps, always
    world, rank, local = dist_env()
    if args.case is not None:
        sys.exit(run_case(args))
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    elif args.gpus > 1 or world > 1:
        if rank == 0:
            print(MULTI_GPU_REASON, file=sys.stderr)
            print(json.dumps(multi_gpu_line(max(args.gpus, world))), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
