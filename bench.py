"""Benchmark of the low-precision DDA allreduce emulation on one GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
the LP flat allreduce and the LP tree allreduce (quantize, FP32 reduce,
requantize, all-gather) of 8 emulated ranks x 67,108,864 FP32 elements
(256 MiB per rank), the gradient-sized workload. Inputs (2 GiB) are larger
than L2 (129 MB), so no flush is needed between steps.

value        whole-job GB/s: algorithmic bytes of all steps on all ranks /
             max-over-ranks time (CUDA events on the launching stream).
e2e          the same metric through the public API with pinned host
             buffers: per step, host->device copy of the 8 inputs, both
             allreduces, device->host copy of both results.
roofline     the dominant kernel's algorithmic bytes per launch / its average
             launch time against the measured HBM copy bandwidth.
cpu_baseline the CPU oracle on a bounded sample of the same workload.
decode       exact-precision flat allreduce of a decode-size message (8 ranks
             x 32 x 8192 BF16): single-launch and CUDA-graph replay time.
workloads    the other reference workloads, GB/s and us per call.

``--impl reference`` times the CPU oracle (the reference arm of this
benchmark) on a bounded sample of the same workload per step.
Run with torchrun for N > 1: each rank runs an independent replica (the
emulation does not shard across GPUs), rank 0 prints the line.
"""
import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from precision_collective_reduction_gb300 import workloads as W  # noqa: E402

HEADLINE = W.LP_GRAD_N8_256MB_F32
NOMINAL_HBM_GBS = 7900.0
METRIC = "LP allreduce-emulation GB/s"
CPU_SAMPLE_ELEMS = 1 << 23      # cpu_baseline: 8 Mi elements per rank, same recipe
REF_BUDGET_ELEMS = 1 << 25      # reference arm: elements per rank over all steps
E2E_MAX_STEPS = 20
E2E_CHUNK = 1 << 22
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "precision_collective_reduction_gb300", "csrc", f)
                  for f in ("lpcoll_device.cuh", "lpcoll_dda.cuh")]


# -- algorithmic bytes --------------------------------------------------------

def bytes_alg(nranks, n, elem, block, algo):
    """Minimum HBM bytes of one emulated allreduce: inputs read once, each
    rank's FP8 wire (codes + scales) written once, the tree's requantized
    shard wire written once, N outputs written."""
    nb = (n + 127) // 128
    per_rank = n * elem * 2
    if block:
        per_rank += n + 4 * nb
    total = nranks * per_rank
    if block and algo == "tree":
        total += n + 4 * nb
    return total


def step_bytes(w, n=None):
    n = w.n if n is None else n
    return sum(bytes_alg(w.nranks, n, w.elem_bytes, w.block, a) for a in w.algos)


# -- environment ----------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class _StdoutToStderr:
    """Send file descriptor 1 to stderr inside the block, so that libraries
    that print to stdout (NCCL's version banner at communicator creation)
    leave the benchmark's one JSON line alone."""

    def __enter__(self):
        sys.stdout.flush()
        self.saved = os.dup(1)
        os.dup2(2, 1)
        return self

    def __exit__(self, *exc):
        sys.stdout.flush()
        os.dup2(self.saved, 1)
        os.close(self.saved)
        return False


def max_over_ranks(x, dist, device):
    """Largest value of x over all ranks (x itself when not distributed)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(bytes_per_step, steps, world, max_ms):
    """Whole-job throughput: the bytes every rank processed over the slowest
    rank's time."""
    return bytes_per_step * steps * world / (max_ms / 1e3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(kernel_key)
    if not ent or ent.get("source_digest") != kernel_source_digest():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples every 100 ms, from
    construction to stop()."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.monotonic(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1, widen=True):
        """Median SM clock, its maximum and the throttle reasons seen in the
        samples taken between t0 and t1 (window "timed"); with widen, a
        window of fewer than 3 samples is widened to all samples ("run")."""
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed" if widen else "gpu phase"
        if widen and len(inside) < 3:
            inside = [p for _, p in self.samples]
            window = "run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        smax = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[4 + i].lower() == "active"})
        pw = [num(p[2]) for p in inside if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max(pw) if pw else None}


# -- CPU oracle legs ------------------------------------------------------------

def oracle_pass(w, n):
    """One flat + tree pass of the CPU oracle over n elements per rank drawn
    with the workload's recipe and seed; returns seconds."""
    import oracle
    ins = [x[:n].copy() for x in W.draw_all(w, n)]
    t0 = time.perf_counter()
    for algo in w.algos:
        (oracle.tree if algo == "tree" else oracle.flat)(ins, block=w.block)
    return time.perf_counter() - t0


def host_cpu():
    """The host's CPU model (or architecture) and core count."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        # Arm hosts list no model name in /proc/cpuinfo; lscpu has it
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    return {"host_cpu": model or platform.machine(), "host_cores": os.cpu_count()}


def cpu_baseline(w):
    secs = oracle_pass(w, CPU_SAMPLE_ELEMS)
    res = {"value": round(step_bytes(w, CPU_SAMPLE_ELEMS) / secs / 1e9, 4),
           "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": "%d of the workload's %d elements per rank (same recipe and "
                     "seed), %d ranks, one flat + one tree pass, single-threaded C "
                     "oracle (%.1f s)"
                     % (CPU_SAMPLE_ELEMS, w.n, w.nranks, secs)}
    res.update(host_cpu())
    return res


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    w = HEADLINE
    n = REF_BUDGET_ELEMS // (args.steps + args.warmup)
    n = max(64 * 128, min(1 << 20, n // 128 * 128))
    for _ in range(args.warmup):
        oracle_pass(w, n)
    secs = [oracle_pass(w, n) for _ in range(args.steps)]
    total = sum(secs)
    value = step_bytes(w, n) * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "kind": "oracle",
                         "sample": "%d of the workload's %d elements per rank (same "
                                   "recipe and seed), %d ranks, flat + tree per step"
                                   % (n, w.n, w.nranks), **host_cpu()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, world):
    return {"workload": w.name, "nranks_emulated": w.nranks, "elems_per_rank": w.n,
            "dtype": "f32" if w.dtype == W.F32 else "bf16", "block": w.block,
            "algos": list(w.algos), "parallelism": "replicas x%d" % world,
            "l2": "inputs larger than L2 (%d MiB of inputs per step)"
                  % (w.nranks * w.message_bytes >> 20)}


# -- GPU legs -------------------------------------------------------------------

def timed_steps(torch, bufs, w, stream, steps, warmup, dist):
    s = stream.cuda_stream
    for _ in range(warmup):
        for a in w.algos:
            bufs.run(a, s)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(w.algos) + 1)]
          for _ in range(steps)]
    t0 = time.monotonic()
    with torch.cuda.stream(stream):
        for i in range(steps):
            ev[i][0].record(stream)
            for j, a in enumerate(w.algos):
                bufs.run(a, s)
                ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    per_kernel = {a: [ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)]
                  for j, a in enumerate(w.algos)}
    total_ms = ev[0][0].elapsed_time(ev[-1][-1])
    if dist is not None:
        dist.barrier()
    return total_ms, per_kernel, (t0, t1)


def e2e_steps(torch, w, steps, host_in, host_out, chunk):
    """Time `steps` end-to-end allreduces of pinned host buffers through the
    library's host-buffer entry point (lpcoll_host_allreduce, via
    HostAllreduce): per step, the host->device copies of the inputs, both
    allreduces and the device->host copies of both results, overlapped by
    chunk. Each call returns once its results are in host memory; a pair of
    events brackets every call on the first and last stream it uses.
    Returns (total ms, per-step ms list, kernel launches per step)."""
    from precision_collective_reduction_gb300.host import HostAllreduce
    h = HostAllreduce(w.nranks, w.n, w.dtype, w.block, algos=w.algos, chunk=chunk)
    h.run(host_in, host_out)          # warm-up pass
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record(h.streams[0])
        h.run(host_in, host_out)
        b.record(h.streams[2])
    ev[-1][1].synchronize()
    per_step = [a.elapsed_time(b) for a, b in ev]
    total = ev[0][0].elapsed_time(ev[-1][1])
    launches = h.kernel_launches_per_run()
    del h
    return total, per_step, launches


def flush_l2(torch, scratch):
    """Evict L2 by reading a buffer four times its size (a read leaves clean
    lines, so the next kernel pays no write-back of the flush itself)."""
    scratch.sum()


def flushed_median_us(torch, stream, scratch, fn, iters, warmup=3):
    """Median microseconds of fn() over `iters` calls on `stream`, each after
    an L2 flush, timed with CUDA events recorded on that stream; `warmup`
    untimed calls first."""
    for _ in range(warmup):
        fn()
    times = []
    with torch.cuda.stream(stream):
        for _ in range(iters):
            flush_l2(torch, scratch)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
    return statistics.median(times)


def measure_small(torch, w, stream, iters, graph_replays=0):
    """us per call of workload w (median of iters, L2 flushed before each)."""
    from precision_collective_reduction_gb300 import runner
    bufs = runner.RankBuffers(w.nranks, w.n, w.dtype, w.block)
    bufs.load(W.draw_all(w))
    scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    s = stream.cuda_stream
    out = {}
    for algo in w.algos:
        us = flushed_median_us(torch, stream, scratch, lambda: bufs.run(algo, s), iters)
        nbytes = bytes_alg(w.nranks, w.n, w.elem_bytes, w.block, algo)
        res = {"us": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
               "frac_of_peak": round(nbytes / us / 1e3 / measured_peaks()[0], 4),
               "bytes_alg": nbytes, "l2": "flushed"}
        # warm L2: back-to-back calls, no flush (what a chain of calls costs)
        warm_calls = 200
        with torch.cuda.stream(stream):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(warm_calls):
                bufs.run(algo, s)
            b.record(stream)
        torch.cuda.synchronize()
        res["warm_us_per_call"] = round(a.elapsed_time(b) * 1e3 / warm_calls, 3)
        res["warm_calls"] = warm_calls
        if graph_replays:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(graph_replays):
                    bufs.run(algo, stream.cuda_stream)
            g.replay()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                g.replay()
                b.record(stream)
            torch.cuda.synchronize()
            res["graph_us_per_call"] = round(a.elapsed_time(b) * 1e3 / graph_replays, 3)
            res["graph_calls"] = graph_replays
            res["graph_l2"] = "warm (back-to-back replays)"
            del g
        out[algo] = res
    del bufs, scratch
    torch.cuda.empty_cache()
    return out


def collective_bytes(kind, N, count, elem, block):
    """Algorithmic HBM bytes of one reduce-scatter (count = n per rank),
    all-gather (count = m per contribution) or all-to-all (count = c per
    chunk): inputs read once, wires written once, outputs written once."""
    def wire(k):
        return (k + 4 * ((k + 127) // 128)) if block else 0
    if kind == "reduce_scatter":
        return N * count * elem + N * wire(count) + count * elem
    if kind == "all_gather":
        return N * count * elem + N * wire(count) + N * N * count * elem
    return N * N * count * elem + N * N * wire(count) + N * N * count * elem


def measure_collectives(torch, stream, iters=20):
    """ReduceScatter / AllGather / AlltoAll, LP, 8 ranks, 16 MiB BF16 per
    rank (the pages' low-precision threshold), L2 flushed before each call."""
    import precision_collective_reduction_gb300 as pcr
    w = W.LP_FLAT_N8_16MB_BF16
    N, n = w.nranks, w.n
    host = W.draw_all(w)
    ins = []
    for h in host:
        ins.append(torch.from_numpy(h).view(torch.int16).view(torch.bfloat16).cuda())
    nb = pcr.nblocks(n)
    wc = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
    ws = [torch.empty(N * nb, dtype=torch.float32, device="cuda") for _ in range(N)]
    scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    per = pcr.shard_len(n, N)
    rs_out = [torch.empty(max(1, min(per, n - r * per)), dtype=torch.bfloat16,
                          device="cuda") for r in range(N)]
    m = n // N
    ag_in = [t[:m] for t in ins]
    full_out = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
    calls = {
        "reduce_scatter": (lambda s: pcr.reduce_scatter_sim(
            ins, rs_out, wire_codes=wc, wire_scales=ws, stream=s), n),
        "all_gather": (lambda s: pcr.all_gather_sim(
            ag_in, full_out, wire_codes=wc, wire_scales=ws, stream=s), m),
        "all_to_all": (lambda s: pcr.all_to_all_sim(
            ins, full_out, wire_codes=wc, wire_scales=ws, stream=s), n // N),
    }
    out = {}
    for kind, (fn, count) in calls.items():
        us = flushed_median_us(torch, stream, scratch, lambda: fn(stream), iters)
        nbytes = collective_bytes(kind, N, count, 2, 128)
        gus = graph_us(torch, stream, lambda: fn(stream), 50)
        out[kind] = {"us": round(us, 3), "GBps": round(nbytes / us / 1e3, 1),
                     "bytes_alg": nbytes, "count_per_rank": count, "l2": "flushed",
                     "warm_us_per_call": round(back_to_back_us(torch, stream,
                                                               lambda: fn(stream), 100), 3),
                     "graph_us_per_call": round(gus, 3),
                     "graph_GBps": round(nbytes / gus / 1e3, 1),
                     "graph_frac_of_peak": round(nbytes / gus / 1e3 / measured_peaks()[0], 4)}
    del ins, wc, ws, scratch, rs_out, full_out
    torch.cuda.empty_cache()
    return out


def staged_bytes(kind, N, n, elem):
    """Algorithmic bytes of the staged building blocks: lp_quantize of one
    rank (n s read, n q written), lp_dequantize (n q read, n s written),
    lp_reduce of N payloads (N n q read, n s written)."""
    q = n + 4 * ((n + 127) // 128)
    if kind == "lp_quantize":
        return n * elem + q
    if kind == "lp_dequantize":
        return q + n * elem
    return N * q + n * elem


def measure_staged(torch, stream, iters=10):
    """lp_quantize, lp_dequantize and lp_reduce on the headline workload (8 x
    64 Mi FP32) and on 8 x 16 MiB BF16, L2 flushed before each call."""
    import precision_collective_reduction_gb300 as pcr
    scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    res = {}
    for w in (HEADLINE, W.LP_FLAT_N8_16MB_BF16):
        N, n = w.nranks, w.n
        tdt = torch.float32 if w.dtype == W.F32 else torch.bfloat16
        ins = []
        for x in W.draw_all(w):
            t = torch.from_numpy(x)
            ins.append((t.view(torch.int16).view(torch.bfloat16) if w.dtype == W.BF16
                        else t).cuda())
        codes = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
        scales = [torch.empty(pcr.nblocks(n), dtype=torch.float32, device="cuda")
                  for _ in range(N)]
        for r in range(N):
            pcr.lp_quantize(ins[r], codes[r], scales[r], stream=stream)
        out = torch.empty(n, dtype=tdt, device="cuda")
        calls = {
            "lp_quantize": lambda: pcr.lp_quantize(ins[0], codes[0], scales[0], stream=stream),
            "lp_dequantize": lambda: pcr.lp_dequantize(codes[0], scales[0], out, stream=stream),
            "lp_reduce": lambda: pcr.lp_reduce(codes, scales, out, stream=stream),
        }
        row = {}
        small = w.nranks * w.message_bytes < L2_FLUSH_BYTES
        for kind, fn in calls.items():
            us = flushed_median_us(torch, stream, scratch, fn, iters)
            nbytes = staged_bytes(kind, N, n, w.elem_bytes)
            row[kind] = {"us": round(us, 2), "GBps": round(nbytes / us / 1e3, 1),
                         "bytes_alg": nbytes}
            if small:
                # per call without launch gaps: back to back, and replayed
                # from a CUDA graph (both warm: one rank's message fits L2)
                row[kind]["warm_us_per_call"] = round(back_to_back_us(torch, stream, fn, 200), 2)
                row[kind]["graph_us_per_call"] = round(graph_us(torch, stream, fn, 100), 2)
        if small:
            row["chain"] = measure_staged_chain(torch, stream, scratch, ins, codes, scales, out,
                                                iters)
        res[w.name] = row
        del ins, codes, scales, out
        torch.cuda.empty_cache()
    del scratch
    return res


def back_to_back_us(torch, stream, fn, calls):
    """us per call of `calls` calls of fn() enqueued back to back on stream."""
    with torch.cuda.stream(stream):
        fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(calls):
            fn()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / calls


def graph_us(torch, stream, fn, calls):
    """us per call of fn() captured `calls` times into one CUDA graph on
    stream and replayed (median of 5 replays)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    t = []
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        t.append(a.elapsed_time(b) * 1e3 / calls)
    del g
    return statistics.median(t)


def measure_staged_chain(torch, stream, scratch, ins, codes, scales, out, iters):
    """The staged allreduce of N ranks (lp_quantize of every rank's message,
    then lp_reduce of the N payloads): L2-flushed single chains, and per
    chain from a CUDA graph of back-to-back chains, with the N quantize calls
    on the one stream (each waits for the previous kernel) or on N parallel
    graph branches (one stream per rank, as the N ranks quantize at once)."""
    import precision_collective_reduction_gb300 as pcr
    N, n = len(ins), ins[0].numel()
    branches = [torch.cuda.Stream() for _ in range(N)]

    def serial():
        for r in range(N):
            pcr.lp_quantize(ins[r], codes[r], scales[r], stream=stream)
        pcr.lp_reduce(codes, scales, out, stream=stream)

    def branched():
        for r in range(N):
            branches[r].wait_stream(stream)
            pcr.lp_quantize(ins[r], codes[r], scales[r], stream=branches[r])
        for r in range(N):
            stream.wait_stream(branches[r])
        pcr.lp_reduce(codes, scales, out, stream=stream)

    elem = ins[0].element_size()
    nbytes = N * staged_bytes("lp_quantize", N, n, elem) + staged_bytes("lp_reduce", N, n, elem)
    peak, _ = measured_peaks()
    res = {"bytes_alg": nbytes,
           "note": "%d x lp_quantize + lp_reduce; bytes: every quantize's input read and "
                   "payload written, the reduce's %d payloads read and output written" % (N, N)}
    for name, fn in (("serial", serial), ("branched", branched)):
        us = flushed_median_us(torch, stream, scratch, fn, iters)
        gus = graph_us(torch, stream, fn, 20)
        res[name] = {"us": round(us, 2), "graph_us_per_call": round(gus, 2),
                     "graph_GBps": round(nbytes / gus / 1e3, 1),
                     "graph_frac_of_peak": round(nbytes / gus / 1e3 / peak, 4)}
    return res


def measure_variants(torch, stream, n=1 << 22, iters=10):
    """Ablation of the FP8 format and block size (staged path: quantize each
    of 8 ranks, then reduce), on the gradient workload's recipe at n elements
    per rank: error of the FP32 result against the FP64 sum of the inputs,
    compression ratio, and time per allreduce (L2 flushed)."""
    import precision_collective_reduction_gb300 as pcr
    w = W.LP_GRAD_N8_256MB_F32
    N = w.nranks
    ins = [torch.from_numpy(x).cuda() for x in W.draw_all(w, n)]
    exact = torch.zeros(n, dtype=torch.float64, device="cuda")
    for t in ins:
        exact += t.double()
    norm = float(torch.linalg.vector_norm(exact))
    peak = float(exact.abs().max())
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    codes = [torch.empty(n, dtype=torch.uint8, device="cuda") for _ in range(N)]
    scales = [torch.empty(pcr.nblocks(n, 32), dtype=torch.float32, device="cuda")
              for _ in range(N)]
    scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    res = {"workload": "%s recipe, %d elements per rank, FP32" % (w.name, n)}
    for fmt, fname in ((pcr.E4M3, "E4M3"), (pcr.E5M2, "E5M2")):
        for block in pcr.VARIANT_BLOCKS:
            def step():
                for r in range(N):
                    pcr.lp_quantize_fmt(ins[r], codes[r], scales[r], block, fmt,
                                        stream=stream)
                pcr.lp_reduce_fmt(codes, scales, out, block, fmt, stream=stream)
            with torch.cuda.stream(stream):
                step()
            torch.cuda.synchronize()
            err = out.double() - exact
            us = flushed_median_us(torch, stream, scratch, step, iters, warmup=0)
            res["%s/%d" % (fname, block)] = {
                "rel_l2_error": float(torch.linalg.vector_norm(err)) / norm,
                "max_abs_error_over_max": float(err.abs().max()) / peak,
                "compression": round(4 / (1 + 4 / block), 4),
                "us_staged": round(us, 2)}
    del ins, exact, out, codes, scales, scratch
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    dist = None
    if world > 1 or "TORCHELASTIC_RUN_ID" in os.environ:
        # under torchrun (even with one rank) every rank joins the process
        # group: a barrier brackets the timed steps and the slowest rank's
        # time is the job's
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        with _StdoutToStderr():
            tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
            tdist.barrier()
        dist = tdist
    else:
        torch.cuda.set_device(0)
    import __graft_entry__
    __graft_entry__.build()
    from precision_collective_reduction_gb300 import runner

    w = HEADLINE
    stream = torch.cuda.Stream()
    host = W.draw_all(w)
    bufs = runner.RankBuffers(w.nranks, w.n, w.dtype, w.block, separate_tree_out=True)
    bufs.load(host)
    torch.cuda.synchronize()

    # sampled through every GPU leg below; summarized for the timed steps
    # and for the whole GPU phase
    clocks = ClockSampler(local)
    phase_t0 = time.monotonic()
    total_ms, per_kernel, (t0, t1) = timed_steps(torch, bufs, w, stream, args.steps,
                                                 args.warmup, dist)
    total_ms = max_over_ranks(total_ms, dist, "cuda")
    sbytes = step_bytes(w)
    value = whole_job_gbps(sbytes, args.steps, world, total_ms)

    peak, peak_kind = measured_peaks()
    avg = {a: statistics.fmean(v) for a, v in per_kernel.items()}
    dom = max(avg, key=lambda a: avg[a])
    dom_bytes = bytes_alg(w.nranks, w.n, w.elem_bytes, w.block, dom)
    achieved = dom_bytes / (avg[dom] / 1e3) / 1e9
    kernel_key = "dda_kernel<8,f32,%s>" % dom
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": profiled_traffic(kernel_key),
                "kernel": kernel_key, "peak_kind": peak_kind + " hbm_gbs (copy)",
                "bytes_alg_per_launch": dom_bytes,
                "avg_launch_us": round(avg[dom] * 1e3, 2)}
    kernels = {a: {"avg_us": round(avg[a] * 1e3, 2),
                   "GBps": round(bytes_alg(w.nranks, w.n, w.elem_bytes, w.block, a)
                                 / (avg[a] / 1e3) / 1e9, 1),
                   "frac_of_peak": round(bytes_alg(w.nranks, w.n, w.elem_bytes, w.block, a)
                                         / (avg[a] / 1e3) / 1e9 / peak, 4)}
               for a in w.algos}

    # end to end through the public API, pinned host buffers
    del bufs
    torch.cuda.empty_cache()
    host_in = [torch.from_numpy(x).pin_memory() for x in host]
    host_out = {a: [torch.empty(w.n, dtype=torch.float32).pin_memory()
                    for _ in range(w.nranks)] for a in w.algos}
    e2e_n = min(args.steps, E2E_MAX_STEPS)
    e2e_ms, e2e_per_step, e2e_launches = e2e_steps(torch, w, e2e_n, host_in, host_out,
                                                    E2E_CHUNK)
    e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")
    h2d = sum(x.nbytes for x in host)
    d2h = sum(h.numel() * h.element_size() for a in w.algos for h in host_out[a])
    e2e = {"value": round(whole_job_gbps(sbytes, e2e_n, world, e2e_ms), 2),
           "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_ms / e2e_n, 3), "steps": e2e_n,
           "api": "lpcoll_host_allreduce via HostAllreduce.run (chunks of %d "
                  "elements, copies and kernels overlapped on three streams)" % E2E_CHUNK,
           "kernel_launches_per_step": e2e_launches,
           "ms_per_step_median": round(statistics.median(e2e_per_step), 3),
           "ms_per_step_max": round(max(e2e_per_step), 3),
           "note": "mean over the steps; single steps are sometimes delayed "
                   "by host-side stalls of this shared machine (see the max)",
           "transfer_GBps": round((h2d + d2h) / (e2e_ms / e2e_n / 1e3) / 1e9, 1)}
    del host_in, host_out
    torch.cuda.empty_cache()

    extras = {}
    if not args.headline_only:
        extras["decode"] = measure_small(torch, W.DECODE_EXACT_FLAT_N8_BF16, stream,
                                         iters=50, graph_replays=1000)["flat"]
        extras["workloads"] = {
            wl.name: measure_small(torch, wl, stream, iters=20,
                                   graph_replays=200 if wl is W.LP_FLAT_N2_1M_F32 else 0)
            for wl in (W.LP_FLAT_N2_1M_F32, W.LP_FLAT_N8_16MB_BF16,
                       W.LP_TREE_N8_64MB_BF16)}
        extras["collectives_lp_n8_16MiB_bf16"] = measure_collectives(torch, stream)
        extras["ablation_fp8_block"] = measure_variants(torch, stream)
        extras["staged"] = measure_staged(torch, stream)

    clocks.stop()
    clock_info = clocks.summary(t0, t1)
    clock_phase = clocks.summary(phase_t0, time.monotonic(), widen=False)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, world),
        "hbm_frac": round(value / world / peak, 4),
        # the same against GB300's nominal HBM3e bandwidth (7.9 TB/s)
        "hbm_frac_nominal": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": roofline, "kernels": kernels,
        "e2e": e2e, "gpu_launches": len(w.algos) * args.steps,
        "clocks": clock_info, "clocks_gpu_phase": clock_phase,
    }
    line.update(extras)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_crossover(args):
    """Flat vs tree allreduce time across message sizes (8 ranks, BF16, exact
    and low precision, L2 flushed before every call): one JSON line per size."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from precision_collective_reduction_gb300 import runner
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    scratch = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    N = 8
    for kib in (8, 32, 128, 512, 2048, 8192, 32768, 131072, 262144):
        n = kib * 1024 // 2
        row = {"nranks": N, "message_KiB": kib, "dtype": "bf16"}
        for block in (0, 128):
            bufs = runner.RankBuffers(N, n, W.BF16, block, separate_tree_out=True)
            bufs.load(W.random_inputs(N, n, W.BF16, 5, scale_spread=1.0))
            s = stream.cuda_stream
            for algo in ("flat", "tree"):
                us = flushed_median_us(torch, stream, scratch,
                                       lambda: bufs.run(algo, s), args.steps)
                key = "%s_%s_us" % ("lp" if block else "exact", algo)
                row[key] = round(us, 3)
            del bufs
            torch.cuda.empty_cache()
        print(json.dumps(row), flush=True)
    return 0


def _collective_runner(torch, bufs, kind):
    """run(algo, stream) for a reduce-scatter ("rs"), all-gather of the first
    n/N elements of every rank ("ag") or all-to-all with chunks of n/N ("a2a")
    over the buffers of a RankBuffers (low precision, its wires)."""
    import precision_collective_reduction_gb300 as pcr
    N, n = bufs.nranks, bufs.n
    if kind == "rs":
        per = pcr.shard_len(n, N)
        outs = [torch.empty(max(1, min(per, n - r * per)), dtype=bufs.ins[0].dtype,
                            device="cuda") for r in range(N)]
        return lambda a, s: pcr.reduce_scatter_sim(bufs.ins, outs, wire_codes=bufs.wire_codes,
                                                   wire_scales=bufs.wire_scales, stream=s)
    if kind == "ag":
        m = n // N
        return lambda a, s: pcr.all_gather_sim([t[:m] for t in bufs.ins], bufs.outs,
                                               wire_codes=bufs.wire_codes,
                                               wire_scales=bufs.wire_scales, stream=s)
    return lambda a, s: pcr.all_to_all_sim(bufs.ins, bufs.outs, wire_codes=bufs.wire_codes,
                                           wire_scales=bufs.wire_scales, stream=s)


def _staged_runner(torch, bufs, kind):
    """run(algo, stream) for one staged building block over the buffers of a
    RankBuffers (low precision): lp_quantize of rank 0's message, lp_dequantize
    of rank 0's payload, or lp_reduce of all N payloads. The payloads are
    filled once before the first call."""
    import precision_collective_reduction_gb300 as pcr
    s0 = torch.cuda.current_stream().cuda_stream
    for r in range(bufs.nranks):
        pcr.lp_quantize(bufs.ins[r], bufs.wire_codes[r], bufs.wire_scales[r], stream=s0)
    if kind == "quantize":
        return lambda a, s: pcr.lp_quantize(bufs.ins[0], bufs.wire_codes[0],
                                            bufs.wire_scales[0], stream=s)
    if kind == "dequantize":
        return lambda a, s: pcr.lp_dequantize(bufs.wire_codes[0], bufs.wire_scales[0],
                                              bufs.outs[0], stream=s)
    return lambda a, s: pcr.lp_reduce(bufs.wire_codes, bufs.wire_scales, bufs.outs[0],
                                      stream=s)


def run_profile_case(args):
    """A few launches of one workload's kernels, for ncu captures: `warmup`
    untimed launches of each algorithm, then `steps` more."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from precision_collective_reduction_gb300 import runner
    w = W.BY_NAME[args.profile_case]
    n = args.elems or w.n
    algos = [args.algo] if args.algo else list(w.algos)
    bufs = runner.RankBuffers(w.nranks, n, w.dtype, w.block,
                              separate_tree_out="tree" in algos)
    bufs.load(W.draw_all(w, n))
    s = torch.cuda.current_stream().cuda_stream
    run = bufs.run
    if algos[0] in ("rs", "ag", "a2a"):
        run = _collective_runner(torch, bufs, algos[0])
    elif algos[0] in ("quantize", "dequantize", "reduce"):
        run = _staged_runner(torch, bufs, algos[0])
    for _ in range(args.warmup):
        for a in algos:
            run(a, s)
    for _ in range(args.steps):
        for a in algos:
            run(a, s)
    torch.cuda.synchronize()
    print("profile case %s n=%d algos=%s: %d launches" % (
        w.name, n, ",".join(algos), (args.warmup + args.steps) * len(algos)))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the decode and secondary workload measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=sorted(W.BY_NAME),
                    help="only run a few launches of this workload (for ncu)")
    ap.add_argument("--elems", type=int, default=0,
                    help="with --profile-case: elements per rank (default: full)")
    ap.add_argument("--algo", choices=["flat", "tree", "rs", "ag", "a2a", "quantize",
                                       "dequantize", "reduce"], default=None,
                    help="with --profile-case: the operation to run (all but flat and "
                         "tree need a low-precision workload)")
    ap.add_argument("--crossover", action="store_true",
                    help="only time flat vs tree over message sizes")
    args = ap.parse_args()
    if args.profile_case:
        return run_profile_case(args)
    if args.crossover:
        return run_crossover(args)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
