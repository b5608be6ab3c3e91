"""Benchmark of the emulated ring / double-binary-tree AllReduce.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--sweep]

A step is one ring AllReduce of R=8 virtual ranks x 64 MiB fp32 (16 777 216
elements per rank, values N(0,1), 12 channels, 512 KiB chunks, Sum) through
the C ABI, inputs resident in HBM.  `value` is the HBM throughput of the
whole job: algorithmic bytes (read R*N*4 + write R*N*4 per step) over the
device time of the K timed steps (CUDA events on the launching stream), in
GB/s.  The 512 MiB read + 512 MiB written per step exceed the 129 MB L2,
so no flush is needed between steps.

Rank 0 prints one JSON line.  It also carries algbw/busbw, a roofline object
for the kernel, the CPU oracle timed on the host cores (cpu_baseline), an
end-to-end figure through the same C ABI with the inputs copied in from
pinned host memory and the result (rank 0's copy; every rank holds the same
bits) copied back inside the timed region, pipelined in pieces by
vr_allreduce_host (e2e), SM clocks sampled during the timed region, and the other
workloads (tree bf16 R=8 / R=7, hierarchical fp16 R=64 ring / tree / Sum /
Max, ReduceScatter, AllGather) timed the same way under "workloads".

--gpus N > 1 (under torchrun): N independent replicas, one per GPU; there
is no data-path collective (the emulation does not shard across GPUs); the
job value is the sum of the work over the max time across ranks.

--impl reference times the CPU oracle (the method's plain restatement) on
the same workload, metric and unit, each step a bounded sample.

--sweep prints the ring vs tree sweep (R=4, 8 B .. 256 MiB per rank, fp32,
12 channels, 512 KiB chunks) as JSON lines instead, then the alpha-beta
model fitted to it (vr_fit_cost_model) and its crossover.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

METRIC = "emulated allreduce busbw and HBM GB/s (% of 8 TB/s) vs msg size, ring vs tree"
WORKLOAD = dict(name="ring_allreduce_r8_64mib_fp32", R=8, count=16 * 1024 * 1024, dtype=0, op=0,
                algo=0, n_channels=12, chunk_bytes=512 * 1024, local_ranks=1, dist="normal",
                seed=1)
PROFILE_SUMMARY = os.path.join(HERE, "profiles", "ring_allreduce_r8_64mib_fp32.md")
KERNEL_SOURCES = [os.path.join(HERE, "double_binary_tree_gb300", "csrc", f)
                  for f in ("fold.cuh", "staged.cuh", "kernels_f32.cu", "common.h")]
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
THROTTLE_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
                 0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
                 0x100: "display_clock_setting"}


def max_over_ranks(torch, value, device):
    """The largest of every rank's `value`: the job takes as long as its
    slowest replica.  Identity without an initialised process group."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world, nbytes_per_replica, steps, ms):
    """Whole-job throughput: the work of all `world` replicas over the
    slowest replica's time."""
    return world * nbytes_per_replica * steps / (ms * 1e-3) / 1e9


def elem_size(dtype):
    return 4 if dtype == 0 else 2


def ar_bytes(R, count, dtype):
    return 2 * R * count * elem_size(dtype)


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peak():
    try:
        with open(os.path.join(HERE, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, when it was
    taken on the current kernel sources; else None."""
    try:
        text = open(PROFILE_SUMMARY, encoding="utf-8").read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_sources_sha256_16") != kernel_hash():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples every 100 ms."""

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None

    def __enter__(self):
        cmd = ["nvidia-smi", "-i", str(self.index),
               "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 3:
                try:
                    self.samples.append((time.time(), int(parts[0]), int(parts[1]),
                                         int(parts[2], 16)))
                except ValueError:
                    pass

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 <= s[0] <= t1] or self.samples
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = 0
        for s in win:
            reasons |= s[3]
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": max(s[2] for s in win),
                "reasons": [n for b, n in THROTTLE_BITS.items() if reasons & b and b != 0x1],
                "samples": len(win)}


# ------------------------------------------------------------------ GPU arm
def gpu_arm(args, rank, world, local_rank):
    import torch
    import double_binary_tree_gb300 as vr
    import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    W = WORKLOAD
    R, count, dtype = W["R"], W["count"], W["dtype"]
    inputs = workloads.generate(R, count, dtype, W["dist"], W["seed"])
    src = [t.to(dev) for t in inputs]
    dst = [torch.empty_like(s) for s in src]

    def step():
        vr.vr_allreduce(src, dst, R, count, dtype, W["op"], W["algo"], W["n_channels"],
                        W["chunk_bytes"], stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    if vr.vr_stream_status(stream) != 0:
        raise RuntimeError("device status error during warm-up")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier()
        launches0 = vr.vr_launch_count()
        t_wall0 = time.time()
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        barrier()
        t_wall1 = time.time()
        launches = vr.vr_launch_count() - launches0
    if vr.vr_stream_status(stream) != 0:
        raise RuntimeError("device status error in the timed region")
    ms = max_over_ranks(torch, start.elapsed_time(stop), dev)
    ms_per_step = ms / args.steps
    nbytes = ar_bytes(R, count, dtype)
    value = job_gbs(world, nbytes, args.steps, ms)
    per_gpu = nbytes / (ms_per_step * 1e-3) / 1e9
    S = count * elem_size(dtype)
    algbw = S / (ms_per_step * 1e-3) / 1e9
    busbw = algbw * 2 * (R - 1) / R
    clocks = clk.summary(t_wall0, t_wall1)

    e2e = e2e_arm(args, vr, torch, inputs, dev, stream, world)
    extra = other_workloads(vr, torch, workloads, dev, stream) if not args.quick else {}
    peak, peak_kind = measured_peak()
    traffic = profiled_traffic()
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": W["name"], "R": R, "count_per_rank": count, "bytes_per_rank": S,
                   "algo": "ring", "op": "sum", "n_channels": W["n_channels"],
                   "chunk_bytes": W["chunk_bytes"], "values": "N(0,1) fp32, seed 1",
                   "l2": "inputs larger than L2 (512 MiB read + 512 MiB written per step)",
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "algbw_gbs": round(algbw, 2), "busbw_gbs": round(busbw, 2),
        "frac_of_8tbs": round(per_gpu / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "achieved": round(per_gpu, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(per_gpu / peak, 4), "traffic": traffic,
                     "peak_source": "%s copy bandwidth, burst" % peak_kind,
                     "kernel": "staged_kernel<float, Sum, ring>",
                     "algorithmic_bytes_per_launch": nbytes},
        "e2e": e2e, "gpu_launches": int(launches), "clocks": clocks,
    }
    if extra:
        line["workloads"] = extra
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    return line


def e2e_arm(args, vr, torch, inputs, dev, stream, world):
    """The same AllReduce through the C ABI's host-buffer entry point: each
    step copies the R inputs in from pinned host memory, folds, and copies
    every rank's result back out, pipelined in pieces (vr_allreduce_host)."""
    W = WORKLOAD
    R, count, dtype = W["R"], W["count"], W["dtype"]
    host_in = [t.pin_memory() for t in inputs]
    # The step's result is one vector (every rank receives the same bits):
    # rank 0's copy comes back to the host, the others stay on the device.
    host_out = [torch.empty_like(inputs[0]).pin_memory()] + [None] * (R - 1)
    work = [torch.empty_like(t, device=dev) for t in inputs]

    def step():
        vr.vr_allreduce_host(host_in, host_out, R, count, dtype, W["op"], W["algo"],
                             W["n_channels"], W["chunk_bytes"], W["local_ranks"], work,
                             args.piece_bytes, stream)

    steps = max(1, min(args.steps, args.e2e_steps))
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    if vr.vr_stream_status(stream) != 0:
        raise RuntimeError("device status error in the end-to-end region")
    ms = max_over_ranks(torch, a.elapsed_time(b), dev)
    nbytes = ar_bytes(R, count, dtype)
    S = count * elem_size(dtype)
    return {"value": round(job_gbs(world, nbytes, steps, ms), 1), "unit": "GB/s",
            "h2d_bytes_per_step": R * S, "d2h_bytes_per_step": S, "steps": steps,
            "ms_per_step": round(ms / steps, 4),
            "api": "vr_allreduce_host: R inputs in from pinned host memory, the result "
                   "(rank 0's copy) out, %d MiB per rank per piece" % (
                       (args.piece_bytes or vr.VR_HOST_PIECE_BYTES) >> 20)}


def time_calls(torch, stream, call, sets, iters):
    """Average device time of `call(i)` over iters calls, rotating buffer
    sets i so that L2-sized workloads read from HBM.  The calls are captured
    once into a CUDA graph and replayed, so host-side launch cost does not
    leave the GPU idle between short kernels."""
    for i in range(3):
        call(i % sets, stream)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            cs = torch.cuda.current_stream()
            for i in range(iters):
                call(i % sets, cs)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    graph.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def other_workloads(vr, torch, workloads, dev, stream):
    peak, _ = measured_peak()
    out = {}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def entry(ms, nbytes, S=None, R=None):
        gbs = nbytes / (ms * 1e-3) / 1e9
        e = {"us": round(ms * 1e3, 2), "hbm_gbs": round(gbs, 1),
             "frac_of_measured_peak": round(gbs / peak, 4)}
        if S is not None:
            algbw = S / (ms * 1e-3) / 1e9
            e["algbw_gbs"] = round(algbw, 2)
            e["busbw_gbs"] = round(algbw * 2 * (R - 1) / R, 2)
        return e

    # tree, bf16, R=8 (mirror) and R=7 (shift), 4 MiB per rank, 2 channels
    for name in ("tree_4mib_r8", "tree_4mib_r7"):
        w = workloads.WORKLOADS[name]
        R, count = w["R"], w["count"]
        nbytes = ar_bytes(R, count, w["dtype"])
        sets = max(2, -(-4 * l2 // nbytes))
        base = workloads.generate(R, count, w["dtype"], w["dist"], w["seed"])
        bufs = [([t.to(dev) for t in base], [torch.empty(count, dtype=base[0].dtype, device=dev)
                                             for _ in range(R)]) for _ in range(sets)]
        for nch in (2, 12):
            def call(i, st, nch=nch):
                s, d = bufs[i]
                vr.vr_allreduce(s, d, R, count, w["dtype"], 0, 1, nch, w["chunk_bytes"], st)
            ms = time_calls(torch, stream, call, sets, 200)
            out["%s_tree_%dch" % (name, nch)] = entry(ms, nbytes, count * 2, R)
        del bufs
    # non-fused variants on the bench workload and the tree workload
    W = WORKLOAD
    R8, n8 = W["R"], W["count"]
    g8 = torch.Generator(device=dev)
    g8.manual_seed(W["seed"])
    s8 = [torch.randn(n8, generator=g8, device=dev) for _ in range(R8)]
    d8 = [torch.empty_like(x) for x in s8]
    fifo = torch.empty(vr.vr_ring_stepwise_scratch_bytes(n8, 0), dtype=torch.uint8, device=dev)

    def call_step(i, st):
        vr.vr_allreduce_ring_stepwise(s8, d8, R8, n8, 0, 0, W["n_channels"], W["chunk_bytes"],
                                      fifo, fifo.numel(), st)
    ms = time_calls(torch, stream, call_step, 1, 5)
    out["ring_64mib_fp32_stepwise"] = entry(ms, ar_bytes(R8, n8, 0), n8 * 4, R8)
    out["ring_64mib_fp32_stepwise"]["launches_per_call"] = 1 + 4 * (R8 - 1)

    def call_updown(i, st):
        vr.vr_allreduce_tree_updown(s8, d8, R8, n8, 0, 0, W["n_channels"], W["chunk_bytes"], 1,
                                    st)
    ms = time_calls(torch, stream, call_updown, 1, 20)
    out["tree_64mib_fp32_updown"] = entry(ms, ar_bytes(R8, n8, 0), n8 * 4, R8)

    def call_tree(i, st):
        vr.vr_allreduce(s8, d8, R8, n8, 0, 0, 1, W["n_channels"], W["chunk_bytes"], st)
    ms = time_calls(torch, stream, call_tree, 1, 20)
    out["tree_64mib_fp32_fused"] = entry(ms, ar_bytes(R8, n8, 0), n8 * 4, R8)
    del s8, d8, fifo

    # hierarchical 8 x 8, fp16, 16 MiB per rank
    w = workloads.WORKLOADS["hier_16mib"]
    R, count, L = w["R"], w["count"], w["local_ranks"]
    g = torch.Generator(device=dev)
    g.manual_seed(w["seed"])
    src = [(torch.rand(count, generator=g, device=dev) * 2 - 1).half() for _ in range(R)]
    dst = [torch.empty_like(s) for s in src]
    nbytes = ar_bytes(R, count, 1)
    for algo, aname in ((0, "ring"), (1, "tree")):
        for op, oname in ((0, "sum"), (1, "max")):
            def call(i, st, algo=algo, op=op):
                vr.vr_allreduce_ex(src, dst, R, count, 1, op, algo, 12, 512 * 1024, L, st)
            ms = time_calls(torch, stream, call, 1, 20)
            out["hier_16mib_fp16_%s_%s" % (aname, oname)] = entry(ms, nbytes, count * 2, R)
    rc = count // R
    rs = [torch.empty(rc, dtype=torch.float16, device=dev) for _ in range(R)]

    def call_rs(i, st):
        vr.vr_reduce_scatter(src, rs, R, rc, 1, 0, 0, 12, 512 * 1024, st)
    ms = time_calls(torch, stream, call_rs, 1, 20)
    out["hier_16mib_fp16_reduce_scatter"] = entry(ms, R * count * 2 + R * rc * 2)

    def call_ag(i, st):
        vr.vr_allgather(rs, dst, R, rc, 1, 0, 12, 512 * 1024, st)
    ms = time_calls(torch, stream, call_ag, 1, 20)
    out["hier_16mib_fp16_allgather"] = entry(ms, R * rc * 2 + R * count * 2)
    return out


# ------------------------------------------------------------ CPU oracle
def cpu_baseline(budget_s=10.0):
    """The oracle as it stands (numpy, one thread) on the bench workload,
    repeated for about budget_s seconds."""
    import oracle
    import workloads
    W = WORKLOAD
    inputs = workloads.generate(W["R"], W["count"], W["dtype"], W["dist"], W["seed"])
    raws = [workloads.raw_numpy(t) for t in inputs]
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.allreduce(raws, W["dtype"], W["op"], W["algo"], W["n_channels"], W["chunk_bytes"])
        runs += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    nbytes = ar_bytes(W["R"], W["count"], W["dtype"]) * runs
    return {"value": round(nbytes / dt / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d full AllReduces of the bench workload (R=8 x 16 777 216 fp32), "
                      "%.1f s, numpy literal ring simulation" % (runs, dt)}


def reference_arm(args):
    """The oracle as the reference arm: each step one AllReduce of a bounded
    sample of the bench workload (the first `n` elements of every rank)."""
    import oracle
    import workloads
    W = WORKLOAD
    inputs = workloads.generate(W["R"], W["count"], W["dtype"], W["dist"], W["seed"])
    raws_full = [workloads.raw_numpy(t) for t in inputs]
    t0 = time.perf_counter()
    probe = [x[:1 << 18] for x in raws_full]
    oracle.allreduce(probe, W["dtype"], W["op"], W["algo"], W["n_channels"], W["chunk_bytes"])
    per_elem = (time.perf_counter() - t0) / (1 << 18)
    total = args.steps + args.warmup
    n = int(min(W["count"], max(1 << 16, 90.0 / max(total, 1) / per_elem)))
    raws = [x[:n] for x in raws_full]
    for _ in range(args.warmup):
        oracle.allreduce(raws, W["dtype"], W["op"], W["algo"], W["n_channels"], W["chunk_bytes"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.allreduce(raws, W["dtype"], W["op"], W["algo"], W["n_channels"], W["chunk_bytes"])
    dt = time.perf_counter() - t0
    nbytes = ar_bytes(W["R"], n, W["dtype"])
    value = nbytes * args.steps / dt / 1e9
    sample = "first %d elements of each rank of the bench workload per step" % n
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": W["name"], "R": W["R"], "count_per_rank": W["count"],
                       "algo": "ring", "op": "sum", "n_channels": W["n_channels"],
                       "chunk_bytes": W["chunk_bytes"]},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


PROFILE_CASES = {
    # name: (collective, R, local ranks, dtype, op, algo); counts come from
    # --count (elements per rank for AllReduce, per block for the others)
    "ring_r8_fp32": ("ar", 8, 1, 0, 0, 0),
    "tree_r8_bf16": ("ar", 8, 1, 2, 0, 1),
    "tree_r8_fp32": ("ar", 8, 1, 0, 0, 1),
    "ring_r4_fp32": ("ar", 4, 1, 0, 0, 0),
    "tree_r4_fp32": ("ar", 4, 1, 0, 0, 1),
    "tree_r7_bf16": ("ar", 7, 1, 2, 0, 1),
    "tree_r64_fp16_hier": ("ar", 64, 8, 1, 0, 1),
    "tree_r64_fp16_hier_max": ("ar", 64, 8, 1, 1, 1),
    "ring_r64_fp16": ("ar", 64, 1, 1, 0, 0),
    "ring_r64_fp16_max": ("ar", 64, 1, 1, 1, 0),
    "rs_r64_fp16": ("rs", 64, 1, 1, 0, 0),
    "rs_r8_fp32": ("rs", 8, 1, 0, 0, 0),
    "ag_r64_fp16": ("ag", 64, 1, 1, 0, 0),
}


def profile_case(args):
    """One collective configuration only, W + K plain launches, nothing else
    on the GPU: the command the ncu captures run."""
    import torch
    import double_binary_tree_gb300 as vr
    coll, R, L, dtype, op, algo = PROFILE_CASES[args.profile]
    count = args.count
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[dtype]
    n_in = {"ar": count, "rs": R * count, "ag": count}[coll]
    n_out = {"ar": count, "rs": count, "ag": R * count}[coll]
    src = [torch.randn(n_in, generator=g, device=dev).to(tdt) for _ in range(R)]
    dst = [torch.empty(n_out, dtype=tdt, device=dev) for _ in range(R)]

    def call():
        if coll == "ar":
            vr.vr_allreduce_ex(src, dst, R, count, dtype, op, algo, 12, 512 * 1024, L, stream)
        elif coll == "rs":
            vr.vr_reduce_scatter(src, dst, R, count, dtype, op, 0, 12, 512 * 1024, stream)
        else:
            vr.vr_allgather(src, dst, R, count, dtype, 0, 12, 512 * 1024, stream)

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            torch.cuda.synchronize()
            a.record(stream)
        call()
    b.record(stream)
    torch.cuda.synchronize()
    if vr.vr_stream_status(stream) != 0:
        raise RuntimeError("device status error")
    ms = a.elapsed_time(b) / max(args.steps, 1)
    E = elem_size(dtype)
    nbytes = (n_in + n_out) * R * E
    print(json.dumps({"profile": args.profile, "count": count, "us": round(ms * 1e3, 2),
                      "hbm_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1)}))


def sweep(args):
    """Ring vs tree, R=4 fp32 Sum, 8 B .. 256 MiB per rank, 12 channels,
    512 KiB chunks; L2-sized messages rotate buffer sets."""
    import torch
    import double_binary_tree_gb300 as vr
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, _ = measured_peak()
    R = 4
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    size = 8
    rows = []
    while size <= 256 * 1024 * 1024:
        count = size // 4
        nbytes = ar_bytes(R, count, 0)
        sets = max(1, min(64, -(-4 * l2 // nbytes)))
        bufs = [([torch.rand(count, generator=g, device=dev) * 2 - 1 for _ in range(R)],
                 [torch.empty(count, device=dev) for _ in range(R)]) for _ in range(sets)]
        row = {"bytes_per_rank": size}
        for algo, name in ((0, "ring"), (1, "tree")):
            def call(i, st, algo=algo):
                s, d = bufs[i]
                vr.vr_allreduce(s, d, R, count, 0, 0, algo, 12, 512 * 1024, st)
            iters = 200 if size <= (1 << 24) else 20
            samples = [time_calls(torch, stream, call, sets, iters) for _ in range(5)]
            ms = statistics.median(samples)
            row[name + "_us"] = round(ms * 1e3, 3)
            row[name + "_busbw_gbs"] = round(size / (ms * 1e-3) / 1e9 * 2 * (R - 1) / R, 3)
            row[name + "_hbm_frac"] = round(nbytes / (ms * 1e-3) / 1e9 / peak, 4)
        lo, hi = sorted((row["ring_us"], row["tree_us"]))
        row["winner"] = "tie" if hi / lo - 1 < 0.05 else (
            "ring" if row["ring_us"] < row["tree_us"] else "tree")
        print(json.dumps(row), flush=True)
        rows.append(row)
        del bufs
        size *= 2
    # The pages' alpha-beta model fitted to these times (the library's own
    # relative least squares), its crossover, and how well it predicts.
    n = len(rows)
    sizes = [r["bytes_per_rank"] for r in rows]
    fit = vr.vr_fit_cost_model([R] * n, [1] * n, sizes, [r["ring_us"] for r in rows],
                               [r["tree_us"] for r in rows])
    err = {}
    for algo, name in ((0, "ring"), (1, "tree")):
        rel = [vr.vr_predict_us(algo, R, 1, r["bytes_per_rank"], fit) / r[name + "_us"] - 1
               for r in rows if r["bytes_per_rank"] >= (1 << 20)]
        err[name] = round(max(abs(x) for x in rel), 4)
    print(json.dumps({"fit": {"alpha_us": {"ring": fit[0][0], "tree": fit[0][1]},
                              "us_per_byte": {"ring": fit[1][0], "tree": fit[1][1]}},
                      "crossover_bytes_per_rank": vr.vr_crossover_bytes(R, 1, fit),
                      "max_rel_error_from_1mib": err}), flush=True)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--piece-bytes", type=int, default=0,
                   help="vr_allreduce_host piece size per rank (0: the library default)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--quick", action="store_true", help="skip the other workloads")
    p.add_argument("--sweep", action="store_true")
    p.add_argument("--profile", choices=sorted(PROFILE_CASES),
                   help="run one collective configuration only (for ncu)")
    p.add_argument("--count", type=int, default=8 * 1024 * 1024,
                   help="elements per rank for --profile")
    args = p.parse_args()
    if args.warmup < 3:
        p.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return
    if args.sweep:
        sweep(args)
        return
    if args.profile:
        profile_case(args)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    line = gpu_arm(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
