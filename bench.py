"""Benchmark of the fused ZeRO step on one GB300 (N simulated ranks in one HBM).

    python bench.py [--gpus G] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

A step is one fused ZeRO step (reduce-scatter-mean + AdamW + all-gather) over
the whole parameter vector of the workload, with the inputs resident in HBM.
Prints ONE JSON line (rank 0). Under torchrun with G > 1 every rank runs an
independent replica of the workload on its own GPU (weak scaling, no
collective on the data path); the timed region is bracketed by barriers and
the slowest rank's time is reported.

--impl reference times the CPU oracle (fp32-mirror numpy, as it stands) on a
bounded sample of the same workload on the host cores.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from zero_sharded_optimizer_gb300 import inputs  # noqa: E402

METRIC = "ZeRO step params/s at N ranks on 1 GB300; achieved HBM GB/s vs peak"
METRIC_DDP = "DDP all_reduce(mean) params/s at N ranks on 1 GB300; achieved HBM GB/s vs peak"
UNIT = "params/s"
DEFAULT_WORKLOAD = "mixed_1p3b"
KERNEL_SRCS = [os.path.join(ROOT, "zero_sharded_optimizer_gb300", "csrc", name)
               for name in ("zero_kernels.cu", "zero_internal.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
L2_BYTES = 129 * 10 ** 6


def bytes_per_param(wl) -> int:
    """Algorithmic HBM bytes per parameter of one fused step (the mean
    gradient is never stored): fp32 reads N grads + p + m + v and writes m, v
    and N replicas: 8N+20; mixed reads N bf16 grads + master, m, v and writes
    master, m, v and N bf16 replicas: 4N+24."""
    if wl.precision == inputs.BF16_MIXED:
        return 4 * wl.N + 24
    return 8 * wl.N + 20


def dtype_of(wl) -> str:
    """Storage and arithmetic of the workload's step: mixed precision stores
    bf16 replicas and gradients and computes in fp32 on the fp32 master, m, v."""
    if wl.precision == inputs.BF16_MIXED:
        return "bf16 storage (params, grads), f32 arithmetic (master, m, v)"
    return "f32"


def default_steps(wl) -> int:
    # about two seconds of timed work, so the clock sampler sees the load
    per_step_s = wl.n * bytes_per_param(wl) / 6.0e12
    return int(min(20000, max(20, round(2.0 / max(per_step_s, 1e-6)))))


def load_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def code_without_comments(text: str) -> str:
    """C/C++/CUDA source with its // and /* */ comments removed (string and
    character literals kept as they are) and blank lines dropped."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # a literal: copy through its closing quote
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line) + "\n"


def kernel_source_hash() -> str:
    """sha256[:16] over the code of the kernel sources (the kernels and the
    argument structs they are compiled with), in order, comments left out:
    ties a traffic record to the code it was measured on."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, encoding="utf-8") as f:
            h.update(code_without_comments(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(workload: str, elems_per_launch: float):
    """DRAM bytes per launch from the committed ncu summary, or None when absent
    or taken on a different kernel source. A record taken on a launch of another
    size (one full 25 MiB bucket, against the mean bucket of a step whose last
    bucket is short) is scaled to ``elems_per_launch`` by the elements processed."""
    try:
        with open(TRAFFIC_FILE) as f:
            entry = json.load(f).get(workload)
    except Exception:
        return None
    if not entry or entry.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    t = entry.get("dram_bytes_per_launch")
    e = entry.get("elements_per_launch")
    if t is not None and e and e != elems_per_launch:
        t = int(round(t * elems_per_launch / e))
    return t


def config_of(wl, extra=None) -> dict:
    step_bytes = wl.n * bytes_per_param(wl)
    cfg = {
        "workload": wl.name,
        "n_params": wl.n,
        "ranks_simulated": wl.N,
        "state": "bf16 params/grads + fp32 master/m/v" if wl.precision else "fp32 params/grads/m/v",
        "optimizer": f"AdamW lr={wl.lr} betas=({wl.beta1},{wl.beta2}) eps={wl.eps} "
                     f"wd={wl.weight_decay}",
        "shards": "np.array_split",
        "bytes_per_step": step_bytes,
        "l2": f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB touched per step vs 129 MB L2)"
              if step_bytes > L2_BYTES else "L2-resident",
    }
    if wl.bucket_bytes:
        cfg["bucket_bytes"] = wl.bucket_bytes
    if extra:
        cfg.update(extra)
    return cfg


def max_over_ranks(values, device, world: int):
    """Element-wise maximum of `values` over all ranks (the slowest rank decides)."""
    if world <= 1:
        return [float(x) for x in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def host_memory_available() -> int | None:
    """MemAvailable of /proc/meminfo in bytes, or None where it cannot be read."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        return None
    return None


def whole_job_rate(units_per_rank: int, world: int, ms_per_step: float) -> float:
    """Units processed by all ranks per second, over the slowest rank's time."""
    return world * units_per_rank / (ms_per_step / 1e3)


# ------------------------------------------------------------------- clocks --

class _NvmlPoller:
    """Reads the SM clock, its maximum, the power draw and the clock-event
    reasons through NVML (read-only queries) every millisecond on a thread, so
    that a timed region of a few milliseconds still gets samples."""

    REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown",
                   0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, uuid: str):
        import ctypes
        import threading
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
            lib.nvmlShutdown()
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        try:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx))  # 1 = SM clock
        self.max_mhz = float(mx.value)
        # the first queries of a process are slow to answer: make them here,
        # before the timed region, and keep no sample from them
        self._read()
        mw = ctypes.c_uint()
        lib.nvmlDeviceGetPowerUsage(self.dev, ctypes.byref(mw))
        self.samples, self.power = [], []
        self.halt = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _read(self):
        ct = self.ct
        clk, bits = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(clk)) != 0:
            return None
        self.reasons_fn(self.dev, ct.byref(bits))
        return float(clk.value), int(bits.value)

    def _run(self):
        # the clock and its reasons every millisecond; the power reading is
        # slower to answer, so every 50 ms
        next_power = 0.0
        while not self.halt.is_set():
            r = self._read()
            if r is not None:
                self.samples.append(r)
            if time.monotonic() >= next_power:
                mw = self.ct.c_uint()
                if self.lib.nvmlDeviceGetPowerUsage(self.dev, self.ct.byref(mw)) == 0:
                    self.power.append(mw.value / 1000.0)
                next_power = time.monotonic() + 0.05
            self.halt.wait(0.001)

    def stop(self) -> dict:
        self.halt.set()
        self.thread.join(timeout=5)
        self.lib.nvmlShutdown()
        sm = [x[0] for x in self.samples]
        reasons = {name for x in self.samples for bit, name in self.REASON_BITS.items()
                   if x[1] & bit}
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": self.max_mhz,
                "power_w_max": max(self.power) if self.power else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvml, 1 ms"}


def _poller_child(uuid: str) -> None:
    """Body of the clock-poller child process: poll until a line arrives on
    stdin, then print the record as one JSON line. A process of its own, so
    that the benchmark's launch loop, which holds the interpreter lock, does
    not delay the samples."""
    try:
        p = _NvmlPoller(uuid)
    except Exception as e:
        print(f"unavailable {e}", flush=True)
        return
    print("ready", flush=True)
    sys.stdin.readline()
    print(json.dumps(p.stop()), flush=True)


def _readline(proc, timeout_s: float) -> str:
    import select
    ready, _, _ = select.select([proc.stdout], [], [], timeout_s)
    return proc.stdout.readline() if ready else ""


class ClockSampler:
    """Clocks during the timed region: NVML polled every millisecond in a
    child process when the library loads, else nvidia-smi's own 100 ms loop."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.nvml = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
            target = ["-i", uuid]
        except Exception:
            uuid, target = None, []
        if uuid is not None:
            try:
                child = subprocess.Popen(
                    [sys.executable, "-c", f"import sys; sys.path.insert(0, {ROOT!r}); "
                     f"import bench; bench._poller_child({uuid!r})"],
                    stdin=subprocess.PIPE, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                    text=True)
                if _readline(child, 60.0).strip() == "ready":
                    self.nvml = child
                    return
                child.kill()
                child.wait(timeout=5)
            except Exception:
                self.nvml = None
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", *target], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.nvml is not None:
            child, rec = self.nvml, None
            try:
                child.stdin.write("stop\n")
                child.stdin.flush()
                rec = json.loads(_readline(child, 30.0))
            except Exception:
                rec = None
            try:
                child.wait(timeout=5)
            except Exception:
                child.kill()
            return rec or {"sm_mhz": None, "sm_max_mhz": None,
                           "reasons": ["clock poller gave no record"], "samples": 0}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi, 100 ms"}


# ------------------------------------------------------------ cpu baseline --

def oracle_sample_rate(wl, seconds: float, sample_n: int | None = None, steps: int | None = None,
                       op: str = "step"):
    """Time the fp32-mirror oracle's ZeRO step (or, with op "ddp_mean", its DDP
    gradient mean) on a sample of the workload.

    The sample is `sample_n` consecutive parameters with all N ranks (the step
    is elementwise, so any slice is a faithful sub-problem). Returns
    (params per second, steps run, sample size, seconds)."""
    import oracle
    rng = np.random.default_rng(0)
    k = sample_n or min(wl.n, 1 << 20)
    mixed = wl.precision == inputs.BF16_MIXED
    init = rng.normal(0, 0.02 if wl.param_init == "normal" else 0.5, k).astype(np.float32)
    reps = [oracle.f32_to_bf16_rne(init) if mixed else init.copy() for _ in range(wl.N)]
    grads = [rng.normal(0, wl.grad_std, k).astype(np.float32) for _ in range(wl.N)]
    if mixed:
        grads = [oracle.f32_to_bf16_rne(g) for g in grads]
    states = oracle.init_states(k, wl.N, wl.precision, master_init=init, mode="fp32")
    hp = dict(lr=wl.lr, beta1=wl.beta1, beta2=wl.beta2, eps=wl.eps, weight_decay=wl.weight_decay,
              precision=wl.precision, mode="fp32")
    t0 = time.perf_counter()
    t = 0
    while True:
        t += 1
        if op == "ddp_mean":
            oracle.allreduce_mean(grads, wl.precision, mode="fp32")
        else:
            reps, states = oracle.zero_step(reps, grads, states, t, **hp)
        el = time.perf_counter() - t0
        if (steps is not None and t >= steps) or (steps is None and el >= seconds):
            break
    return k * t / el, t, k, el


def cpu_baseline(wl, seconds: float = 12.0, op: str = "step") -> dict:
    rate, steps, k, el = oracle_sample_rate(wl, seconds, op=op)
    what = "DDP means" if op == "ddp_mean" else "steps"
    return {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{steps} oracle {what} (fp32-mirror numpy, one thread) on {k:,} "
                      f"consecutive parameters x {wl.N} ranks of {wl.name}; {el:.1f} s"}


def _oracle_worker(job):
    """One process of the all-cores oracle run: wait for the common start, then
    time the oracle on its own sample for ``seconds``."""
    wl, seconds, op, start_at = job
    while time.time() < start_at:
        time.sleep(0.005)
    rate, steps, k, el = oracle_sample_rate(wl, seconds, op=op)
    return k * steps, el, k


def cpu_baseline_all_cores(wl, seconds: float = 8.0, op: str = "step",
                           procs: int | None = None) -> dict:
    """The same oracle chunked over every core this process may run on: one
    spawned process per core, each stepping its own sample of the workload (the
    step is elementwise, so the samples are independent chunks), all started
    together. Throughput = parameters stepped by all ÷ the longest process's
    time. A pool that breaks or overruns gives a record saying so, not a hang."""
    import concurrent.futures as cf
    import multiprocessing as mp
    cores = procs or len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    ex = cf.ProcessPoolExecutor(max_workers=cores, mp_context=ctx)
    try:
        start_at = time.time() + 5.0  # after every process has imported numpy
        futs = [ex.submit(_oracle_worker, (wl, seconds, op, start_at)) for _ in range(cores)]
        res = [f.result(timeout=seconds + 120.0) for f in futs]
    except Exception as e:  # broken pool, timeout
        ex.shutdown(wait=False, cancel_futures=True)
        return {"value": None, "unit": UNIT, "cores": cores,
                "kind": "oracle, one spawned process per core",
                "unavailable": f"{type(e).__name__}: {e}"[:200]}
    ex.shutdown(wait=True)
    done = sum(r[0] for r in res)
    el = max(r[1] for r in res)
    return {"value": done / el, "unit": UNIT, "cores": cores,
            "kind": "oracle, one spawned process per core",
            "sample": f"{cores} processes x about {seconds:.0f} s, each on {res[0][2]:,} "
                      f"consecutive parameters x {wl.N} ranks of {wl.name} (fp32-mirror numpy)"}


def percentile(sorted_vals, q: float) -> float:
    """Linear-interpolation percentile of an ascending list."""
    if not sorted_vals:
        return float("nan")
    x = (len(sorted_vals) - 1) * q / 100.0
    lo = int(x)
    hi = min(lo + 1, len(sorted_vals) - 1)
    return sorted_vals[lo] + (sorted_vals[hi] - sorted_vals[lo]) * (x - lo)


# --------------------------------------------------------------- GPU arm --

def host_link_timer(dev_in, host_in, host_out, dev_out, stream, chunk: int):
    """A timer of the e2e step's copies alone, in the host-input step's own
    schedule: per chunk of ``chunk`` elements, every host input's piece is
    copied to its device buffer on one stream, then (after an event) the
    output's piece is copied back on another. ``run(k)`` does k such steps back
    to back and returns the milliseconds. Overwrites ``dev_in``."""
    import torch
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    n = dev_out.numel()
    pieces = [(lo, min(n, lo + chunk)) for lo in range(0, n, chunk)]

    def run(k: int) -> float:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        s_in.wait_event(t0)
        s_out.wait_event(t0)
        for _ in range(k):
            for lo, hi in pieces:
                with torch.cuda.stream(s_in):
                    for d, h in zip(dev_in, host_in):
                        d[lo:hi].copy_(h[lo:hi], non_blocking=True)
                    ready = torch.cuda.Event()
                    ready.record(s_in)
                s_out.wait_event(ready)
                with torch.cuda.stream(s_out):
                    host_out[lo:hi].copy_(dev_out[lo:hi], non_blocking=True)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    return run


def producer_report(opt, reps, grads, wl, stream, iters: int, gaps_us=(0, 200)) -> dict:
    """The bucket streamer against a gradient producer, as in a backward pass:
    a producer stream writes each 25 MiB bucket of every rank's gradient in
    reverse index order (a copy from a second set of gradient buffers, 2 bytes
    read and written per element and rank) and records that bucket's ready
    event; the step runs each bucket on a side stream once its event fires.
    ``gap_us`` > 0 puts a bounded single-thread busy wait of that length on the
    producer stream before every bucket, standing in for the backward compute
    that produces it (it uses no memory bandwidth). Reported per mode, in ms
    per step (mean over ``iters`` steps, each bracketed by synchronisation):
      producer_ms   the producer alone;
      overlapped_ms producer start to the last bucket stepped;
      tail_ms       the last bucket's ready event to the last bucket stepped
                    (what of the step is exposed after the gradients are in);
    and once, the bucketed step whose ready events have all fired before it
    is queued (the waits stay on the stream), against the same step with no
    waits: whether the programmatic chaining of bucket launches survives the
    event waits between them."""
    import torch
    ranges = opt.bucket_ranges(wl.bucket_bytes)
    src = [g.clone() for g in grads]
    producer, side = torch.cuda.Stream(), torch.cuda.Stream()
    T = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    # the busy wait counts SM clock cycles: calibrate cycles per microsecond
    a, b = T(), T()
    torch.cuda.synchronize()
    a.record(producer)
    with torch.cuda.stream(producer):
        torch.cuda._sleep(4_000_000)
    b.record(producer)
    torch.cuda.synchronize()
    clock_mhz = 4_000_000 / (a.elapsed_time(b) * 1e3)

    def produce(ready, gap_us):
        with torch.cuda.stream(producer):
            for k, (lo, hi) in enumerate(ranges):
                if gap_us:
                    torch.cuda._sleep(int(gap_us * clock_mhz))
                for d, s_ in zip(grads, src):
                    d[lo:hi].copy_(s_[lo:hi])
                ready[k].record(producer)

    def one(gap_us, with_step):
        ready = [T() for _ in ranges]
        t0, t1, done = T(), T(), T()
        torch.cuda.synchronize()
        t0.record(stream)
        producer.wait_event(t0)
        side.wait_event(t0)
        produce(ready, gap_us)
        if with_step:
            opt.step_bucketed(reps, grads, ready, side, wl.bucket_bytes, done=done)
            stream.wait_event(done)
        stream.wait_stream(producer)
        t1.record(stream)
        torch.cuda.synchronize()
        tail = ready[-1].elapsed_time(done) if with_step else None
        return t0.elapsed_time(t1), tail

    modes = []
    for gap in gaps_us:
        one(gap, True)  # warm-up of this mode
        alone = [one(gap, False)[0] for _ in range(iters)]
        both = [one(gap, True) for _ in range(iters)]
        modes.append({"gap_us_per_bucket": gap,
                      "producer_ms": statistics.mean(alone),
                      "overlapped_ms": statistics.mean(x[0] for x in both),
                      "tail_ms": statistics.mean(x[1] for x in both),
                      "tail_ms_max": max(x[1] for x in both)})

    def bucketed_ms(with_events):
        ready = [T() for _ in ranges]
        if with_events:
            produce(ready, 0)
        torch.cuda.synchronize()
        t0, t1 = T(), T()
        side.wait_stream(stream)
        t0.record(side)
        opt.step_bucketed(reps, grads, ready if with_events else None, side, wl.bucket_bytes)
        t1.record(side)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    bucketed_ms(True)
    fired = statistics.median(bucketed_ms(True) for _ in range(iters))
    no_waits = statistics.median(bucketed_ms(False) for _ in range(iters))
    del src
    full_bucket = max(hi - lo for lo, hi in ranges)
    return {"what": "the bucket streamer against a producer stream writing 25 MiB buckets of "
                    "every rank's gradient in reverse index order (a copy, HBM-bound), optionally "
                    "after a bounded busy wait per bucket standing in for backward compute",
            "buckets": len(ranges), "full_bucket_params": full_bucket,
            "last_bucket_params": ranges[-1][1] - ranges[-1][0],
            "modes": modes,
            "step_with_fired_events_ms": fired,
            "step_without_events_ms": no_waits,
            "busy_wait_cycles_per_us": clock_mhz,
            "iters": iters}


def run_gpu(args, wl, rank: int, world: int, local_rank: int) -> dict | None:
    import torch
    import torch.distributed as dist

    from zero_sharded_optimizer_gb300 import abi
    from zero_sharded_optimizer_gb300.optimizer import BUCKET_BYTES_25MIB, ZeroOptimizer

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    K, W = args.steps, args.warmup
    n, N = wl.n, wl.N
    mixed = wl.precision == inputs.BF16_MIXED
    init = inputs.init_params_fp32(n, wl, seed=rank, device=dev)
    reps = inputs.make_replicas(init, N, wl.precision)
    grads = inputs.make_grads(n, N, wl.precision, device=dev)
    inputs.fill_grads(grads, wl, step=1, seed=rank)
    clip = args.max_grad_norm > 0
    bounds = None
    if args.partition == "tensor":
        # whole-tensor shards over the workload's parameter list
        bounds = abi.zero_tensor_shard_bounds([int(np.prod(s)) for _, s in
                                               inputs.gpt2_small_shapes()], N)
    opt = ZeroOptimizer(n, N, wl.precision, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                        weight_decay=wl.weight_decay, master_init=init if mixed else None,
                        max_grad_norm=args.max_grad_norm, shard_bounds=bounds,
                        stage=args.stage, optimizer=args.optimizer,
                        momentum=0.9 if args.optimizer == "sgd" else 0.0)
    del init
    stage3 = args.stage == 3
    ddp = args.op == "ddp_mean"
    bucketed = wl.bucket_bytes > 0 and not ddp
    launches_per_step = len(opt.bucket_ranges(wl.bucket_bytes)) if bucketed else 1
    if clip:
        launches_per_step = 3       # norm partials, norm total, the clipped step
    if stage3:
        launches_per_step += 1      # the gather after the owner-only step
    stream = torch.cuda.current_stream()

    def one_step(mid=None):
        if ddp:
            abi.ddp_allreduce_mean(grads, wl.precision, n)
        elif bucketed:
            opt.step_bucketed(reps, grads, None, stream, wl.bucket_bytes)
        else:
            opt.step(reps, grads)
            if stage3:
                if mid is not None:  # between the owner-only step and the gather
                    mid.record(stream)
                opt.gather(reps)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(W):
        one_step()
    barrier()

    # The timed region: K steps back to back on the launching stream, one
    # event pair around them (an event between steps delays the next launch
    # by a few microseconds, 1-2 % of a 0.2 ms step). The kernel time is the
    # region's time over the launches in it.
    sampler = ClockSampler(local_rank) if rank == 0 else None
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    t_begin.record(stream)
    for _ in range(K):
        one_step()
    t_end.record(stream)
    barrier()
    clocks = sampler.stop() if sampler else None
    ms_total = t_begin.elapsed_time(t_end)
    ms_step = ms_total / K
    kernel_ms = ms_step

    # After it, untimed for the headline: the same K steps with an event pair
    # around each (the spread of step times) and, at stage 3, one between the
    # owner-only step and the gather.
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(K)] if stage3 else None
    for k in range(K):
        starts[k].record(stream)
        one_step(mids[k] if mids else None)
        ends[k].record(stream)
    barrier()
    step_times = sorted(s.elapsed_time(e) for s, e in zip(starts, ends))
    dist_ms = [percentile(step_times, q) for q in (10, 50, 90)]
    split = None
    if stage3:  # each kernel of the stage-3 step on its own (CUDA events between them)
        es_ = 2 if wl.precision == inputs.BF16_MIXED else 4
        step_part = sum(s.elapsed_time(m) for s, m in zip(starts, mids)) / K
        gather_part = sum(m.elapsed_time(e) for m, e in zip(mids, ends)) / K
        split = {"owner_only_step_ms": step_part, "gather_ms": gather_part,
                 "gather_gbs": n * wl.N * es_ / (gather_part / 1e3) / 1e9,
                 "gather_bytes": "n x N x element size (read the owner's element, write N-1)"}

    ms_step, kernel_ms = max_over_ranks([ms_step, kernel_ms], dev, world)
    producer = None
    if bucketed and args.producer:
        producer = producer_report(opt, reps, grads, wl, stream, iters=10)

    # ---- end to end through the public API: host gradients in, parameters out
    es = 2 if mixed else 4
    h2d_bytes, d2h_bytes = N * n * es, n * es

    def measure_e2e():
        E2E_BLOCK = 5
        K_e = E2E_BLOCK * max(1, min(K, 30) // E2E_BLOCK)
        host_grads = []
        for g in grads:
            h = torch.empty(n, dtype=g.dtype, pin_memory=True)
            h.copy_(g)
            host_grads.append(h)
        host_out = torch.empty(n, dtype=reps[0].dtype, pin_memory=True)
        if ddp:
            host_out = torch.empty(n, dtype=grads[0].dtype, pin_memory=True)

        def e2e_path(o):
            if o.max_grad_norm > 0:
                return ("ZeroOptimizer.step with pinned host gradients -> zero_step_from_host_ex "
                        "with clipping: every 25 MiB chunk copied in on a copy stream, its part of "
                        "the norm summed once it has arrived, the norm's total once all have, then "
                        "the clipped step chunk by chunk, each chunk's "
                        "D2H on a second copy stream while the next is stepped")
            entry = ("zero_step_from_host_ex" if o.stage == 3 or o.optimizer == "sgd"
                     or o.grad_scale != 1.0 else "zero_step_from_host")
            out = ("each shard from its owner's replica" if o.stage == 3
                   else "one updated replica")
            return (f"ZeroOptimizer.step with pinned host gradients -> {entry}: 25 MiB chunks, "
                    "H2D on a copy stream, the step per chunk on the compute stream, D2H of "
                    f"{out} on a second copy stream")

        ddp_h2d, ddp_d2h = (torch.cuda.Stream(), torch.cuda.Stream()) if ddp else (None, None)
        ddp_host = abi.DdpHost() if ddp else None

        def e2e_step():
            if ddp:  # gradients in, the mean gradient out, chunk-pipelined and chained
                ddp_host.mean_from_host(host_grads, grads, wl.precision, n, host_out,
                                        BUCKET_BYTES_25MIB, None, ddp_h2d, ddp_d2h)
            else:
                opt.step(reps, host_grads, host_params_out=host_out)

        # The host link's rate drifts by tens of percent over seconds (the host is
        # shared), so the e2e steps and the copies-alone bound alternate in blocks
        # of E2E_BLOCK back-to-back steps and each side sums its blocks.
        link = host_link_timer(grads, host_grads, host_out, reps[0], stream,
                               BUCKET_BYTES_25MIB // (2 if mixed else 4))

        def e2e_block(k: int) -> float:
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t0.record(stream)
            for _ in range(k):
                e2e_step()
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1)

        for _ in range(2):
            e2e_step()
        link(1)
        barrier()
        e_total = l_total = 0.0
        for _ in range(K_e // E2E_BLOCK):
            e_total += e2e_block(E2E_BLOCK)
            l_total += link(E2E_BLOCK)
        barrier()
        e_ms, link_ms = max_over_ranks([e_total / K_e, l_total / K_e], dev, world)
        e2e = {"value": whole_job_rate(n, world, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "ms_per_step": e_ms, "steps": K_e,
               "host_link_ms": link_ms, "frac_of_host_link": link_ms / e_ms,
               "host_link": f"the same H2D and D2H copies alone in the host-input step's "
                            f"schedule (25 MiB chunks: H2D on one stream, then that chunk's D2H on "
                            f"another), no step: the e2e lower bound on this host link; timed in "
                            f"blocks of {E2E_BLOCK} back-to-back steps alternating with the e2e "
                            f"blocks",
               "path": ("ddp_allreduce_mean_from_host_h with pinned host gradients: 25 MiB "
                        "chunks, H2D on a copy stream, the mean per chunk on the compute stream, "
                        "D2H of the mean on a second copy stream; back-to-back calls on one handle "
                        "chained chunk by chunk") if ddp else
                       e2e_path(opt)}
        return e2e

    # The e2e leg pins the step's host gradients and output (N + 1 vectors per
    # rank). All ranks decide together whether the node's free host memory
    # holds them for every local rank; if not, the leg reports why instead of
    # failing the run.
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", str(world)))
    pinned = h2d_bytes + d2h_bytes
    avail = host_memory_available()
    short = avail is not None and pinned * local_ranks > 0.7 * avail
    short = max_over_ranks([1.0 if short else 0.0], dev, world)[0] > 0
    if short:
        e2e = {"value": None, "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
               "d2h_bytes_per_step": d2h_bytes,
               "unavailable": f"host memory: {local_ranks} local rank(s) x {pinned / 1e9:.1f} GB "
                              f"pinned would exceed 70 % of the node's available "
                              f"{(avail or 0) / 1e9:.1f} GB"}
    else:
        e2e = measure_e2e()

    if rank != 0:
        return None
    peak, peak_kind = load_peaks()
    step_bytes = n * bytes_per_param(wl)
    if ddp:  # read and write every rank's gradient once
        step_bytes = 2 * N * n * (2 if mixed else 4)
    sgd = args.optimizer == "sgd"
    if sgd:  # one fp32 buffer (read + write) instead of m and v
        step_bytes -= n * 8
    if clip:  # the norm pass reads every rank's gradient once more
        step_bytes += n * N * (2 if mixed else 4)
    if stage3:  # the step writes 1 replica, not N; the gather reads 1 and writes N-1
        step_bytes += n * (2 if mixed else 4)
    achieved = step_bytes / (kernel_ms / 1e3) / 1e9
    whole = clip or stage3  # the roofline covers the whole step (several kernels)
    per = 1 if whole else launches_per_step
    # the committed records cover the plain step of each workload (bucketed
    # for the bucket-streamed one) and single variants of it: "<workload>/sgd",
    # "/ddp_mean", and "/clip", "/stage3" (whole steps of several launches);
    # combined variants have none
    variants = [v for v, on in (("sgd", sgd), ("ddp_mean", ddp), ("clip", clip),
                                ("stage3", stage3)) if on]
    key = wl.name + ("/" + "+".join(variants) if variants else "")
    traffic = traffic_per_launch(key, n / per)
    line = {
        "metric": METRIC_DDP if ddp else METRIC,
        "value": whole_job_rate(n, world, ms_step),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_of(wl),
        "data": "synthetic (seeded device draws; inputs resident in HBM)",
        "config": config_of(wl, {"parallelism": f"{N} simulated ranks per GPU; "
                                                f"{world} independent GPU replica(s)",
                                 **({"max_grad_norm": args.max_grad_norm} if clip else {}),
                                 **({"zero_stage": 3} if stage3 else {}),
                                 **({"optimizer": "momentum SGD (0.9)"} if sgd else {}),
                                 **({"op": "ddp_allreduce_mean (no optimizer step)"} if ddp
                                    else {}),
                                 "partition": ("whole tensors (" + ", ".join(
                                     str(int(b2 - b1)) for b1, b2 in zip(bounds, bounds[1:])) +
                                     " params per rank)") if bounds else "np.array_split"}),
        "hbm_gbs": step_bytes / (ms_step / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy "
                                    f"bandwidth)" if peak_kind == "measured" else "fallback",
                     "algorithmic_bytes_per_launch": step_bytes // per,
                     "kernel": "allreduce_mean_kernel" if ddp else
                               ("grad_norm_partials_kernel + grad_norm_total_kernel + "
                                "zero_step_kernel (whole clipped step, chained launches)") if clip else
                               ("zero_step_kernel (owner-only) + gather_kernel "
                                "(whole stage-3 step)") if stage3 else "zero_step_kernel",
                     "kernel_ms": kernel_ms / per,
                     "kernel_ms_source": "the timed region's CUDA events over its launches "
                                         "(K steps back to back)",
                     "step_ms_p10_median_p90": dist_ms,
                     "step_ms_source": "a second pass of K steps, an event pair around each",
                     **({"stage3_split": split} if split else {})},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
        "e2e": e2e,
    }
    if producer is not None:
        line["producer"] = producer
    if args.cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, op=args.op)
        line["cpu_baseline"]["all_cores"] = cpu_baseline_all_cores(wl, op=args.op)
    return line


# ---------------------------------------------------------- reference arm --

def run_reference(args, wl, world: int) -> dict:
    K, W = args.steps, args.warmup
    # calibrate, then size each step's sample so the whole run stays near a minute
    op = args.op
    rate, _, _, _ = oracle_sample_rate(wl, 0.0, sample_n=min(wl.n, 1 << 18), steps=3, op=op)
    budget_s = 60.0
    k = int(min(wl.n, max(4096, rate * budget_s / max(K + W, 1))))
    if W:
        oracle_sample_rate(wl, 0.0, sample_n=k, steps=W, op=op)
    rate, steps, k, el = oracle_sample_rate(wl, 0.0, sample_n=k, steps=K, op=op)
    ms = el / steps * 1e3
    sample = (f"each step: the fp32-mirror oracle (numpy, one thread) on {k:,} consecutive "
              f"parameters x {wl.N} ranks of {wl.name}"
              + ("; the DDP mean only" if op == "ddp_mean" else ""))
    return {
        "impl": "reference",
        "metric": METRIC_DDP if op == "ddp_mean" else METRIC,
        "value": rate,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_of(wl),
        "data": "synthetic (seeded numpy draws)",
        "config": config_of(wl, {"parallelism": f"{wl.N} simulated ranks; host cores"}),
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# -------------------------------------------------------------------- main --

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-producer", dest="producer", action="store_false",
                    help="bucket-streamed workloads: skip the step-against-a-producer report")
    ap.add_argument("--partition", default="array_split", choices=["array_split", "tensor"],
                    help="tensor: shards of whole tensors (workloads with a tensor list)")
    ap.add_argument("--max-grad-norm", type=float, default=0.0,
                    help="> 0: sharded global-norm clipping before every step (norm pass + step)")
    ap.add_argument("--optimizer", default="adamw", choices=["adamw", "sgd"],
                    help="sgd: momentum SGD (momentum 0.9, the workload's lr and decay)")
    ap.add_argument("--op", default="step", choices=["step", "ddp_mean"],
                    help="ddp_mean: time ddp_allreduce_mean on the workload's gradients instead")
    ap.add_argument("--stage", type=int, default=2, choices=[2, 3],
                    help="3: owner-only step, then the gather of the full parameters (2 launches)")
    ap.add_argument("--n", type=int, default=None,
                    help="override the parameter count: a smaller case of the same kernels for "
                         "ncu captures (named <workload>_n<count>; not a bench line)")
    ap.add_argument("--ranks", type=int, default=None,
                    help="override the simulated rank count N (named <workload>_N<ranks>; a "
                         "case for sweeps, not a bench line)")
    args = ap.parse_args(argv)
    wl = inputs.WORKLOADS[args.workload]
    if args.n is not None:
        if args.n <= 0 or args.partition == "tensor":
            ap.error("--n needs a positive count and the np.array_split partition")
        wl = dataclasses.replace(wl, n=args.n, name=f"{wl.name}_n{args.n}")
    if args.ranks is not None:
        if not 1 <= args.ranks <= 64 or args.partition == "tensor":
            ap.error("--ranks needs 1..64 and the np.array_split partition")
        wl = dataclasses.replace(wl, N=args.ranks, name=f"{wl.name}_N{args.ranks}")
    if args.steps is None:
        args.steps = default_steps(wl)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.partition == "tensor" and wl.name != "gpt2_small":
        ap.error("--partition tensor needs a workload with a tensor list (gpt2_small)")
    if args.max_grad_norm > 0 and wl.bucket_bytes:
        ap.error("clipping needs the whole gradient before the step: not with bucket streaming")
    if args.optimizer == "sgd" and wl.bucket_bytes:
        ap.error("bucket streaming runs the AdamW step: not with --optimizer sgd")
    if args.stage == 3 and wl.bucket_bytes:
        ap.error("bucket streaming runs the step with its all-gather: not with --stage 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}; using {world}",
              file=sys.stderr)

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl, world)), flush=True)
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        line = run_gpu(args, wl, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
