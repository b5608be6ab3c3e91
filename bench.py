"""Benchmark of the emulated ring / double-binary-tree AllReduce.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--sweep]

A step is one ring AllReduce of R=8 virtual ranks x 64 MiB fp32 (16 777 216
elements per rank, values N(0,1), 12 channels, 512 KiB chunks, Sum) through
the C ABI, inputs resident in HBM.  `value` is the HBM throughput of the
whole job: algorithmic bytes (read R*N*4 + write R*N*4 per step) over the
device time of the K timed steps (CUDA events on the launching stream), in
GB/s.  The 512 MiB read + 512 MiB written per step exceed the 129 MB L2,
so no flush is needed between steps.

Rank 0 prints one JSON line.  Besides the contract's keys it carries:

* step_samples: the same step measured the way the pages measure
  ([Course13] "实验矩阵", "异常样本与定向复测"): 10 samples, each the mean of
  20 launches after 5 warm-up launches; median, P95 and CV; a measurement
  whose CV is above 5 % is taken again once;
* algbw / busbw, a roofline object for the kernel, SM clocks sampled
  during the timed region (NVML, read-only);
* e2e: the same AllReduce through the C ABI's host-buffer entry point
  (vr_allreduce_host), the inputs copied in from pinned host memory and the
  result (rank 0's copy; every rank holds the same bits) copied back inside
  the timed region;
* sweep: ring vs tree on the sweep configuration (R=4 fp32, 12 channels,
  512 KiB chunks) at 8 B, 4 KiB, 256 KiB, 4 MiB, 64 MiB and 256 MiB per
  rank: busbw, HBM GB/s and the winner under the pages' 5 % tie rule
  ([Course13] "性能结果的判定规则"), ring and tree samples taken in mirrored
  order, L2-sized messages timed cold (rotated buffer sets: HBM) and hot
  (L2), only cold counting;
* workloads: the other configurations (tree bf16 R=8 / R=7 with a device
  copy of the same bytes and an empty call beside them, hierarchical fp16
  R=64 ring / tree / Sum / Max, ReduceScatter, AllGather, the non-fused
  variants), each timed as CUDA-graph replays with the same sample rules;
* cpu_baseline: the CPU oracle on the host's cores and on one core.

--gpus N > 1 (under torchrun): N independent replicas, one per GPU; there
is no data-path collective (the emulation does not shard across GPUs); the
job value is the sum of the work over the max time across ranks.

--impl reference times the CPU oracle (the method's plain restatement) on
the same workload, metric and unit, on the host's cores, each step a bounded
sample.

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
                  for f in ("fold.cuh", "staged.cuh", "kernels_f32.cu", "common.h", "bounds.cuh")]
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


class Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes): SM
    clock, its maximum and the active clock-event reasons of one GPU."""

    def __init__(self, local_rank):
        import ctypes
        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return
        c = ctypes
        self.c = c
        if self.lib.nvmlInit_v2() != 0:
            return
        self.handle = c.c_void_p()
        found = False
        uuid = _cuda_uuid(local_rank)
        if uuid:
            found = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), c.byref(self.handle)) == 0
        if not found:
            idx = _nvml_index(local_rank)
            found = self.lib.nvmlDeviceGetHandleByIndex_v2(c.c_uint(idx), c.byref(self.handle)) == 0
        if not found:
            return
        reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = reasons or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.ok = True

    def sample(self):
        c = self.c
        sm, mx, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if (self.lib.nvmlDeviceGetClockInfo(self.handle, 1, c.byref(sm)) != 0 or
                self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, c.byref(mx)) != 0 or
                self.reasons_fn(self.handle, c.byref(rs)) != 0):
            return None
        return int(sm.value), int(mx.value), int(rs.value)


def _cuda_uuid(local_rank):
    """NVML's name ("GPU-<uuid>") of the CUDA device local_rank, or None."""
    try:
        import torch
        u = getattr(torch.cuda.get_device_properties(local_rank), "uuid", None)
        return "GPU-%s" % u if u else None
    except Exception:
        return None


def _nvml_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p.strip() for p in vis.split(",") if p.strip()]
    if local_rank < len(parts) and parts[local_rank].isdigit():
        return int(parts[local_rank])
    return local_rank


class ClockSampler:
    """SM clock and clock-event-reason samples of one GPU, every 2 ms, from a
    thread calling NVML (read-only queries); nvidia-smi's 100 ms loop when
    NVML cannot be opened.  Samples carry host timestamps, so the timed
    window can be picked out afterwards."""

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.stop = threading.Event()
        self.source = None

    def __enter__(self):
        nv = Nvml(self.index)
        if nv.ok and nv.sample() is not None:
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll, args=(nv,), daemon=True)
            self.thread.start()
            return self
        cmd = ["nvidia-smi", "-i", str(_nvml_index(self.index)),
               "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return self
        self.source = "nvidia-smi"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def wait_first(self, timeout=5.0):
        """Block until the first sample arrived (or timeout)."""
        t0 = time.time()
        while not self.samples and time.time() - t0 < timeout and self.source:
            time.sleep(0.01)

    def _poll(self, nv):
        while not self.stop.is_set():
            s = nv.sample()
            if s is not None:
                self.samples.append((time.time(),) + s)
            time.sleep(0.002)

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
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        """Median SM clock, maximum and the union of reasons over [t0, t1];
        over every sample taken when that window holds none."""
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if not win:
            win, window = list(self.samples), "measurement"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": self.source}
        reasons = 0
        for s in win:
            reasons |= s[3]
        return {"sm_mhz": statistics.median(s[1] for s in win),
                "sm_max_mhz": max(s[2] for s in win),
                "reasons": [n for b, n in THROTTLE_BITS.items() if reasons & b and b != 0x1],
                "samples": len(win), "window": window, "source": self.source}


# ------------------------------------------------------------ timing rules
SAMPLES = 10          # samples per measurement
ITERS = 20            # iterations averaged per sample (at least)
WARM = 5              # warm-up iterations before the samples
CV_RERUN = 0.05       # a group whose CV exceeds this is measured once more
TIE = 0.05            # ring and tree within 5 % of each other: a tie


def stats_of(xs):
    """Median, P95 (nearest rank), mean and CV of per-iteration times (ms),
    and the samples themselves (us, in the order taken)."""
    raw = [round(x * 1e3, 3) for x in xs]
    xs = sorted(xs)
    n = len(xs)
    mean = sum(xs) / n
    sd = statistics.pstdev(xs) if n > 1 else 0.0
    return {"median_us": round(statistics.median(xs) * 1e3, 3),
            "p95_us": round(xs[min(n - 1, max(0, -(-95 * n // 100) - 1))] * 1e3, 3),
            "cv": round(sd / mean, 4) if mean > 0 else 0.0, "n": n, "samples_us": raw}


def measure(samplers, samples=SAMPLES):
    """Samples of several measurements taken in mirrored order (A B ... B A,
    repeated), so that drift during the run weighs on all of them alike.
    ``samplers`` maps a name to a function returning one sample (ms per
    iteration).  A measurement whose CV is above CV_RERUN is taken again,
    once, and the second set is kept ("rerun": true)."""
    names = list(samplers)
    got = {k: [] for k in names}
    for i in range(samples):
        for k in (names if i % 2 == 0 else names[::-1]):
            got[k].append(samplers[k]())
    out = {}
    for k in names:
        st = stats_of(got[k])
        if st["cv"] > CV_RERUN:
            st = stats_of([samplers[k]() for _ in range(samples)])
            st["rerun"] = True
        out[k] = st
    return out


def graph_sampler(torch, stream, call, sets, iters=ITERS, warm=WARM):
    """A function returning one sample of ``call``: the mean device time of
    ``iters`` calls (at least ITERS, more for short calls, so that a sample
    spans about a millisecond), rotating buffer sets i so that L2-sized
    workloads read from HBM.  The calls are captured once into a CUDA graph
    (host launch cost does not leave the GPU idle between short kernels);
    ``warm`` calls and one replay run before the first sample."""
    for i in range(warm):
        call(i % sets, stream)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    call(0, stream)
    b.record(stream)
    torch.cuda.synchronize()
    per = max(a.elapsed_time(b), 1e-3)
    n = max(iters, min(2000, int(1.0 / per)))
    n = -(-n // sets) * sets if sets > 1 else n
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            cs = torch.cuda.current_stream()
            for i in range(n):
                call(i % sets, cs)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()

    def sample():
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n
    sample.iters = n
    sample.graph = graph
    return sample


def direct_sampler(torch, stream, call, iters=ITERS):
    """One sample: ``iters`` plain launches of call() between two events (for
    calls long enough that launch cost is hidden)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def sample():
        a.record(stream)
        for _ in range(iters):
            call()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / iters
    return sample


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

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        clk.wait_first()
        # the warm-up steps run right before the timed ones (after the
        # sampler's start-up, which leaves the GPU idle)
        for _ in range(args.warmup):
            step()
        if vr.vr_stream_status(stream) != 0:
            raise RuntimeError("device status error during warm-up")
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
        # The pages' methodology on the same step: SAMPLES samples, each the
        # mean of ITERS launches, after WARM warm-up launches.
        for _ in range(WARM):
            step()
        head_stats = measure({"step": direct_sampler(torch, stream, step)})["step"]
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
    head_stats["hbm_gbs_at_median"] = round(nbytes / (head_stats["median_us"] * 1e-6) / 1e9, 1)

    e2e = e2e_arm(args, vr, torch, inputs, dev, stream, world)
    del src, dst
    extra = other_workloads(vr, torch, workloads, dev, stream) if not args.quick else {}
    sweep_rows = compact_sweep(vr, torch, dev, stream) if not args.quick else []
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
        "step_samples": dict(head_stats, method="%d samples, each the mean of %d launches after "
                             "%d warm-up launches; CV above %.0f%% re-measured once" % (
                                 SAMPLES, ITERS, WARM, CV_RERUN * 100)),
        "e2e": e2e, "gpu_launches": int(launches), "clocks": clocks,
    }
    if sweep_rows:
        line["sweep"] = sweep_rows
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
    """Median device time (ms) of call(i) over SAMPLES graph replays of at
    least ``iters`` calls (graph_sampler)."""
    smp = graph_sampler(torch, stream, call, sets, iters)
    return statistics.median(smp() for _ in range(SAMPLES))


def _entry(st, nbytes, peak, S=None, R=None):
    """One workload's figures from its sample statistics (median time)."""
    ms = st["median_us"] * 1e-3
    gbs = nbytes / (ms * 1e-3) / 1e9
    e = dict(st, us=st["median_us"], hbm_gbs=round(gbs, 1),
             frac_of_measured_peak=round(gbs / peak, 4))
    if S is not None:
        algbw = S / (ms * 1e-3) / 1e9
        e["algbw_gbs"] = round(algbw, 2)
        e["busbw_gbs"] = round(algbw * 2 * (R - 1) / R, 2)
    return e


def _rotation(l2, nbytes):
    """Buffer sets to rotate so that every call reads from HBM (at least 4 x
    L2 of traffic between two uses of a set)."""
    return max(1, min(64, -(-4 * l2 // nbytes)))


def other_workloads(vr, torch, workloads, dev, stream):
    peak, _ = measured_peak()
    out = {}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    # tree, bf16, R=8 (mirror) and R=7 (shift), 4 MiB per rank: 64 / 56 MiB of
    # traffic, L2-sized.  "cold": buffer sets rotated (HBM); "hot": one set
    # (L2); beside them a device copy of the same bytes with the same
    # rotation (the floor of a one-launch HBM pass of this size) and an empty
    # library call (launch floor).
    for name in ("tree_4mib_r8", "tree_4mib_r7"):
        w = workloads.WORKLOADS[name]
        R, count = w["R"], w["count"]
        nbytes = ar_bytes(R, count, w["dtype"])
        sets = max(2, _rotation(l2, nbytes))
        base = workloads.generate(R, count, w["dtype"], w["dist"], w["seed"])
        bufs = [([t.to(dev) for t in base], [torch.empty(count, dtype=base[0].dtype, device=dev)
                                             for _ in range(R)]) for _ in range(sets)]
        flat = [(torch.empty(R * count, dtype=base[0].dtype, device=dev),
                 torch.empty(R * count, dtype=base[0].dtype, device=dev)) for _ in range(sets)]
        for a, _ in flat:
            a.normal_()
        smp = {}
        for nch in (2, 12):
            def call(i, st, nch=nch):
                s, d = bufs[i]
                vr.vr_allreduce(s, d, R, count, w["dtype"], 0, 1, nch, w["chunk_bytes"], st)
            smp["%dch_cold" % nch] = graph_sampler(torch, stream, call, sets)
            smp["%dch_hot" % nch] = graph_sampler(torch, stream, lambda i, st, c=call: c(0, st), 1)

        def copy(i, st):
            a, b = flat[i]
            b.copy_(a)
        smp["copy_cold"] = graph_sampler(torch, stream, copy, sets)
        res = measure(smp)
        for nch in (2, 12):
            key = "%s_tree_%dch" % (name, nch)
            out[key] = _entry(res["%dch_cold" % nch], nbytes, peak, count * 2, R)
            out[key]["rotated_sets"] = sets
            out[key]["hot_l2"] = _entry(res["%dch_hot" % nch], nbytes, peak, count * 2, R)
            out[key]["copy_same_bytes"] = _entry(res["copy_cold"], nbytes, peak)
            out[key]["vs_copy"] = round(res["copy_cold"]["median_us"] /
                                        res["%dch_cold" % nch]["median_us"], 4)
        del bufs, flat, smp
    tiny = [torch.zeros(4, device=dev) for _ in range(2)]

    def empty(i, st):
        vr.vr_allreduce(tiny, tiny, 2, 4, 0, 0, 0, 1, 16, st)
    out["empty_call"] = measure({"e": graph_sampler(torch, stream, empty, 1)})["e"]

    # non-fused variants on the bench workload and the tree workload
    W = WORKLOAD
    R8, n8 = W["R"], W["count"]
    g8 = torch.Generator(device=dev)
    g8.manual_seed(W["seed"])
    s8 = [torch.randn(n8, generator=g8, device=dev) for _ in range(R8)]
    d8 = [torch.empty_like(x) for x in s8]
    fifo = torch.empty(vr.vr_ring_stepwise_scratch_bytes(n8, 0), dtype=torch.uint8, device=dev)
    nb8 = ar_bytes(R8, n8, 0)

    def call_step(i, st):
        vr.vr_allreduce_ring_stepwise(s8, d8, R8, n8, 0, 0, W["n_channels"], W["chunk_bytes"],
                                      fifo, fifo.numel(), st)

    def call_updown(i, st):
        vr.vr_allreduce_tree_updown(s8, d8, R8, n8, 0, 0, W["n_channels"], W["chunk_bytes"], 1,
                                    st)

    def call_tree(i, st):
        vr.vr_allreduce(s8, d8, R8, n8, 0, 0, 1, W["n_channels"], W["chunk_bytes"], st)
    res = measure({"step": graph_sampler(torch, stream, call_step, 1, 5),
                   "updown": graph_sampler(torch, stream, call_updown, 1),
                   "fused": graph_sampler(torch, stream, call_tree, 1)})
    out["ring_64mib_fp32_stepwise"] = _entry(res["step"], nb8, peak, n8 * 4, R8)
    out["ring_64mib_fp32_stepwise"]["launches_per_call"] = 1 + 4 * (R8 - 1)
    out["tree_64mib_fp32_updown"] = _entry(res["updown"], nb8, peak, n8 * 4, R8)
    out["tree_64mib_fp32_fused"] = _entry(res["fused"], nb8, peak, n8 * 4, R8)
    del s8, d8, fifo

    # hierarchical 8 x 8, fp16, 16 MiB per rank
    w = workloads.WORKLOADS["hier_16mib"]
    R, count, L = w["R"], w["count"], w["local_ranks"]
    g = torch.Generator(device=dev)
    g.manual_seed(w["seed"])
    src = [(torch.rand(count, generator=g, device=dev) * 2 - 1).half() for _ in range(R)]
    dst = [torch.empty_like(s) for s in src]
    nbytes = ar_bytes(R, count, 1)
    smp = {}
    for algo, aname in ((0, "ring"), (1, "tree")):
        for op, oname in ((0, "sum"), (1, "max")):
            def call(i, st, algo=algo, op=op):
                vr.vr_allreduce_ex(src, dst, R, count, 1, op, algo, 12, 512 * 1024, L, st)
            smp["%s_%s" % (aname, oname)] = graph_sampler(torch, stream, call, 1)
    rc = count // R
    rs = [torch.empty(rc, dtype=torch.float16, device=dev) for _ in range(R)]

    def call_rs(i, st):
        vr.vr_reduce_scatter(src, rs, R, rc, 1, 0, 0, 12, 512 * 1024, st)

    def call_ag(i, st):
        vr.vr_allgather(rs, dst, R, rc, 1, 0, 12, 512 * 1024, st)
    smp["rs"] = graph_sampler(torch, stream, call_rs, 1)
    smp["ag"] = graph_sampler(torch, stream, call_ag, 1)
    res = measure(smp)
    for k in ("ring_sum", "ring_max", "tree_sum", "tree_max"):
        out["hier_16mib_fp16_" + k] = _entry(res[k], nbytes, peak, count * 2, R)
    out["hier_16mib_fp16_reduce_scatter"] = _entry(res["rs"], R * count * 2 + R * rc * 2, peak)
    out["hier_16mib_fp16_allgather"] = _entry(res["ag"], R * rc * 2 + R * count * 2, peak)
    return out


SWEEP_SIZES = (8, 4096, 256 << 10, 4 << 20, 64 << 20, 256 << 20)


def compact_sweep(vr, torch, dev, stream, sizes=SWEEP_SIZES):
    """Ring vs tree, R=4 fp32 Sum, 12 channels, 512 KiB chunks (the sweep
    configuration) at a few sizes per rank: each size's ring and tree
    samples taken in mirrored order; L2-sized messages timed cold (buffer
    sets rotated: HBM) and hot (one set: L2), only cold counting for the
    roofline and the winner (5 % tie rule)."""
    peak, _ = measured_peak()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = 4
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    rows = []
    for size in sizes:
        count = size // 4
        nbytes = ar_bytes(R, count, 0)
        sets = _rotation(l2, nbytes)
        bufs = [([torch.rand(count, generator=g, device=dev) * 2 - 1 for _ in range(R)],
                 [torch.empty(count, device=dev) for _ in range(R)]) for _ in range(sets)]
        smp = {}
        for algo, name in ((0, "ring"), (1, "tree")):
            def call(i, st, algo=algo):
                s, d = bufs[i]
                vr.vr_allreduce(s, d, R, count, 0, 0, algo, 12, 512 * 1024, st)
            smp[name] = graph_sampler(torch, stream, call, sets)
            if sets > 1:
                smp[name + "_hot"] = graph_sampler(torch, stream, lambda i, st, c=call: c(0, st), 1)
        res = measure(smp)
        row = {"bytes_per_rank": size, "rotated_sets": sets}
        for name in ("ring", "tree"):
            st = res[name]
            ms = st["median_us"] * 1e-3
            row[name] = dict(st, busbw_gbs=round(size / (ms * 1e-3) / 1e9 * 2 * (R - 1) / R, 3),
                             hbm_gbs=round(nbytes / (ms * 1e-3) / 1e9, 1),
                             hbm_frac=round(nbytes / (ms * 1e-3) / 1e9 / peak, 4))
            if name + "_hot" in res:
                row[name]["hot_l2_us"] = res[name + "_hot"]["median_us"]
        lo, hi = sorted((row["ring"]["median_us"], row["tree"]["median_us"]))
        row["winner"] = "tie" if hi / lo - 1 < TIE else (
            "ring" if row["ring"]["median_us"] < row["tree"]["median_us"] else "tree")
        rows.append(row)
        del bufs, smp
    return rows


# ------------------------------------------------------------ CPU oracle
def host_cpu():
    """(usable CPUs, model name) of this host."""
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return int(n or 1), model


def _oracle_channel(task):
    """One channel of the oracle's ring AllReduce (the loop oracle.allreduce
    runs for each channel: its ring loops through the literal simulation),
    on inputs in a file mapped read-only; returns the loops folded."""
    path, R, count, k, nch, cb = task
    import numpy as np
    from oracle import partition, schedules
    xs = np.memmap(path, dtype=np.float32, mode="r", shape=(R, count))
    xs = [xs[r] for r in range(R)]
    cs, cn = partition.channel_ranges(count, 4, nch)[k]
    out = np.empty((R, cn), dtype=np.float32)
    loops = 0
    for loop in partition.ring_blocks(cs, cn, R, cb // 4):
        res = schedules.ring_allreduce_loop(xs, loop, 0)
        for r in range(R):
            for (bs, bn), blk in zip(loop, res[r]):
                out[r, bs - cs:bs - cs + bn] = blk
        loops += 1
    return loops


class OraclePool:
    """The oracle's fp32 ring AllReduce with its channels spread over a pool
    of worker processes (spawn: safe after the GPU was used), one channel
    per task; the channels of the method are independent rings, so this is
    the same computation as oracle.allreduce, on several host cores."""

    def __init__(self, raws, n_channels, chunk_bytes, workers):
        import multiprocessing
        import tempfile
        import numpy as np
        self.dir = tempfile.mkdtemp(prefix="vr_oracle_")
        self.path = os.path.join(self.dir, "inputs.f32")
        R, count = len(raws), int(raws[0].size)
        mm = np.memmap(self.path, dtype=np.float32, mode="w+", shape=(R, count))
        for r in range(R):
            mm[r] = raws[r]
        mm.flush()
        del mm
        self.tasks = [(self.path, R, count, k, n_channels, chunk_bytes)
                      for k in range(n_channels)]
        self.workers = max(1, min(workers, n_channels))
        self.pool = multiprocessing.get_context("spawn").Pool(self.workers)
        self.pool.map(_oracle_channel, self.tasks)          # start-up and first touch

    def allreduce(self):
        self.pool.map(_oracle_channel, self.tasks)

    def close(self):
        self.pool.close()
        self.pool.join()
        os.remove(self.path)
        os.rmdir(self.dir)


def cpu_baseline(budget_s=10.0):
    """The oracle as it stands on the bench workload, on this host's cores
    (channels over a process pool) and on one core (oracle.allreduce), each
    repeated for about budget_s seconds."""
    import oracle
    import workloads
    W = WORKLOAD
    inputs = workloads.generate(W["R"], W["count"], W["dtype"], W["dist"], W["seed"])
    raws = [workloads.raw_numpy(t) for t in inputs]
    nbytes = ar_bytes(W["R"], W["count"], W["dtype"])
    cpus, model = host_cpu()

    def timed(run):
        runs, t0 = 0, time.perf_counter()
        while True:
            run()
            runs += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        dt = time.perf_counter() - t0
        return runs, dt, nbytes * runs / dt / 1e9

    runs1, dt1, v1 = timed(lambda: oracle.allreduce(raws, W["dtype"], W["op"], W["algo"],
                                                    W["n_channels"], W["chunk_bytes"]))
    pool = OraclePool(raws, W["n_channels"], W["chunk_bytes"], cpus)
    try:
        runsn, dtn, vn = timed(pool.allreduce)
    finally:
        pool.close()
    return {"value": round(vn, 3), "unit": "GB/s", "cores": pool.workers, "kind": "oracle",
            "sample": "%d full AllReduces of the bench workload (R=8 x 16 777 216 fp32) in "
                      "%.1f s, the oracle's literal ring simulation with its %d channels over "
                      "%d worker processes" % (runsn, dtn, W["n_channels"], pool.workers),
            "host_cpus": cpus, "cpu_model": model,
            "one_core": {"value": round(v1, 3), "unit": "GB/s", "cores": 1,
                         "sample": "%d full AllReduces in %.1f s, oracle.allreduce" % (
                             runs1, dt1)}}


def reference_arm(args):
    """The oracle as the reference arm, on this host's cores (its channels
    over a process pool): each step one AllReduce of a bounded sample of the
    bench workload (the first `n` elements of every rank)."""
    import oracle
    import workloads
    W = WORKLOAD
    inputs = workloads.generate(W["R"], W["count"], W["dtype"], W["dist"], W["seed"])
    raws_full = [workloads.raw_numpy(t) for t in inputs]
    cpus, model = host_cpu()
    t0 = time.perf_counter()
    probe = [x[:1 << 18] for x in raws_full]
    oracle.allreduce(probe, W["dtype"], W["op"], W["algo"], W["n_channels"], W["chunk_bytes"])
    per_elem = (time.perf_counter() - t0) / (1 << 18)
    total = args.steps + args.warmup
    # about 90 s of one core's work for the whole run, shared by the workers
    n = int(min(W["count"], max(1 << 16, 90.0 * min(cpus, W["n_channels"]) /
                                max(total, 1) / per_elem)))
    raws = [x[:n] for x in raws_full]
    pool = OraclePool(raws, W["n_channels"], W["chunk_bytes"], cpus)
    try:
        for _ in range(args.warmup):
            pool.allreduce()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            pool.allreduce()
        dt = time.perf_counter() - t0
    finally:
        pool.close()
    nbytes = ar_bytes(W["R"], n, W["dtype"])
    value = nbytes * args.steps / dt / 1e9
    sample = ("first %d elements of each rank of the bench workload per step, the oracle's "
              "literal ring simulation with its %d channels over %d worker processes" % (
                  n, W["n_channels"], pool.workers))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": W["name"], "R": W["R"], "count_per_rank": W["count"],
                       "algo": "ring", "op": "sum", "n_channels": W["n_channels"],
                       "chunk_bytes": W["chunk_bytes"]},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": pool.workers,
                             "kind": "oracle", "sample": sample, "host_cpus": cpus,
                             "cpu_model": model},
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
    for opt in args.option:   # library options for the capture, NAME=VALUE
        name, value = opt.split("=", 1)
        vr.vr_set_option(name, int(value))
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
    """Ring vs tree, R=4 fp32 Sum, 8 B .. 256 MiB per rank (every power of
    two), 12 channels, 512 KiB chunks, timed as compact_sweep times its
    sizes."""
    import torch
    import double_binary_tree_gb300 as vr
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    R = 4
    size = 8
    rows = []
    while size <= 256 * 1024 * 1024:
        row = compact_sweep(vr, torch, dev, stream, sizes=(size,))[0]
        row["ring_us"], row["tree_us"] = row["ring"]["median_us"], row["tree"]["median_us"]
        print(json.dumps(row), flush=True)
        rows.append(row)
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
    p.add_argument("--option", action="append", default=[],
                   help="NAME=VALUE library option (vr_set_option) for --profile")
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
