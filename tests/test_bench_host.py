"""Host logic of the benchmark, on CPU.

* The clock record, against a fake NVML library. The poller only reads (clock,
  maximum clock, power, clock-event reasons). The fake answers those queries
  and counts them. The record must decode the reason bits that make a timed run
  invalid (hardware and thermal slowdowns) and the one that is only noted
  (software power cap).
* The DRAM traffic records: lookup by kernel-source hash, and scaling from the
  captured launch to the mean launch of the line.
"""

import ctypes
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


class FakeNvml:
    def __init__(self, clocks, reasons):
        self.clocks, self.reasons = clocks, reasons
        self.i = 0
        self.calls = []
        self.uuid = None

    @staticmethod
    def _set(ref, value):
        ref._obj.value = value

    def nvmlInit_v2(self):
        self.calls.append("init")
        return 0

    def nvmlShutdown(self):
        self.calls.append("shutdown")
        return 0

    def nvmlDeviceGetHandleByUUID(self, uuid, ref):
        self.uuid = uuid
        self._set(ref, 1234)
        return 0

    def nvmlDeviceGetMaxClockInfo(self, dev, kind, ref):
        assert kind == 1
        self._set(ref, 2070)
        return 0

    def nvmlDeviceGetClockInfo(self, dev, kind, ref):
        assert kind == 1
        self._set(ref, self.clocks[min(self.i, len(self.clocks) - 1)])
        return 0

    def nvmlDeviceGetPowerUsage(self, dev, ref):
        self._set(ref, 850_000)
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, dev, ref):
        self._set(ref, self.reasons[min(self.i, len(self.reasons) - 1)])
        self.i += 1
        return 0


def run_poller(monkeypatch, clocks, reasons):
    import bench
    fake = FakeNvml(clocks, reasons)
    monkeypatch.setattr(ctypes, "CDLL", lambda name: fake)
    p = bench._NvmlPoller("GPU-0000")
    deadline = time.time() + 5
    while len(p.samples) < len(clocks) and time.time() < deadline:
        time.sleep(0.002)
    rec = p.stop()
    return fake, rec


def test_clock_record_decodes_reasons(monkeypatch):
    fake, rec = run_poller(monkeypatch, [2070, 2070, 1980], [0x0, 0x4, 0x4 | 0x40])
    assert fake.uuid == b"GPU-0000"
    assert fake.calls[0] == "init" and fake.calls[-1] == "shutdown"
    assert rec["samples"] >= 3
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["power_w_max"] == 850.0
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_record_quiet_run(monkeypatch):
    _, rec = run_poller(monkeypatch, [2070] * 4, [0x1] * 4)  # idle bit only: not reported
    assert rec["reasons"] == []
    assert rec["sm_mhz"] == 2070.0


def test_traffic_record_scaled_to_the_mean_launch(monkeypatch, tmp_path):
    """A record taken on one full bucket is scaled to the mean bucket by the
    parameters processed; a stale source hash gives None."""
    import json
    import bench
    path = tmp_path / "traffic.json"
    good = {"dram_bytes_per_launch": 1000, "elements_per_launch": 100,
            "kernel_source_sha256_16": bench.kernel_source_hash()}
    path.write_text(json.dumps({"a": good, "b": dict(good, kernel_source_sha256_16="0" * 16),
                                "c": {k: v for k, v in good.items()
                                      if k != "elements_per_launch"}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.traffic_per_launch("a", 100) == 1000
    assert bench.traffic_per_launch("a", 99.2) == 992
    assert bench.traffic_per_launch("b", 100) is None
    assert bench.traffic_per_launch("c", 50) == 1000
    assert bench.traffic_per_launch("missing", 100) is None


def test_kernel_source_hash_ignores_comments_only(monkeypatch, tmp_path):
    """The traffic record's source hash covers the code: comments and blank
    lines may change, code (including inside a string literal) may not."""
    import bench
    src = tmp_path / "k.cu"
    monkeypatch.setattr(bench, "KERNEL_SRCS", [str(src)])

    def h(text):
        src.write_text(text)
        return bench.kernel_source_hash()

    base = h('int a = 1;\nconst char* s = "x // y";\n')
    assert h('// a note\nint a = 1;  /* two\nlines */\n\nconst char* s = "x // y"; // z\n') == base
    assert h('int a = 2;\nconst char* s = "x // y";\n') != base
    assert h('int a = 1;\nconst char* s = "x // w";\n') != base
    assert bench.code_without_comments("char c = '\"'; // q\n") == "char c = '\"';\n"


def test_committed_traffic_records_cover_the_bench_workloads():
    import json
    import bench
    from zero_sharded_optimizer_gb300 import inputs
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    names = ("fp32_25m", "gpt2_small", "fp32_320m", "mixed_1p3b", "fp32_25m/sgd",
             "gpt2_small/sgd", "fp32_320m/sgd", "fp32_25m/ddp_mean", "gpt2_small/ddp_mean",
             "fp32_25m/clip", "gpt2_small/clip", "fp32_320m/clip", "fp32_25m/stage3",
             "gpt2_small/stage3")
    assert sorted(rec) == sorted(names)
    for name in names:
        assert name.split("/")[0] in inputs.WORKLOADS
        e = rec[name]
        assert e["dram_bytes_per_launch"] == e["dram_bytes_read"] + e["dram_bytes_write"]
        assert os.path.exists(os.path.join(ROOT, e["summary"]))
        # taken on the kernel code as committed: the bench line carries it
        assert e["kernel_source_sha256_16"] == bench.kernel_source_hash(), name


def test_poller_child_protocol(monkeypatch, capsys):
    """The child prints ``ready``, polls until a line arrives on stdin, then
    prints its record as one JSON line; without NVML it says so and stops."""
    import io
    import json
    import bench
    fake = FakeNvml([2070] * 3, [0x0] * 3)
    monkeypatch.setattr(ctypes, "CDLL", lambda name: fake)
    monkeypatch.setattr(sys, "stdin", io.StringIO("stop\n"))
    bench._poller_child("GPU-0000")
    out = capsys.readouterr().out.splitlines()
    assert out[0] == "ready"
    rec = json.loads(out[1])
    assert rec["sm_max_mhz"] == 2070.0 and rec["source"] == "nvml, 1 ms"
    assert fake.calls[-1] == "shutdown"

    def missing(name):
        raise OSError("no such library")
    monkeypatch.setattr(ctypes, "CDLL", missing)
    bench._poller_child("GPU-0000")
    assert capsys.readouterr().out.startswith("unavailable")


def test_step_time_percentiles():
    import numpy as np
    import bench
    v = sorted(np.random.default_rng(3).random(37).tolist())
    for q in (10, 50, 90):
        assert abs(bench.percentile(v, q) - np.percentile(v, q)) < 1e-12
    assert bench.percentile([2.0], 90) == 2.0


def test_all_cores_oracle_baseline_runs_on_spawned_processes():
    """The all-cores oracle leg starts its processes with spawn and adds up
    what they stepped; two processes on the small parity workload."""
    import bench
    from zero_sharded_optimizer_gb300 import inputs
    rec = bench.cpu_baseline_all_cores(inputs.WORKLOADS["tiny_adam"], seconds=0.3, procs=2)
    assert rec["cores"] == 2 and "unavailable" not in rec, rec
    assert rec["value"] > 0


def test_host_memory_available_reads_meminfo():
    """The e2e leg sizes its pinned buffers against MemAvailable: on Linux it
    is a positive byte count below the total memory."""
    import bench
    avail = bench.host_memory_available()
    if not os.path.exists("/proc/meminfo"):
        assert avail is None
        return
    assert avail is not None and avail > 0
    with open("/proc/meminfo") as f:
        total = next(int(l.split()[1]) * 1024 for l in f if l.startswith("MemTotal:"))
    assert avail <= total
