"""bench.py host logic on CPU: rank aggregation over gloo (world size 2), the clock
summary, the traffic record's kernel check and the JSON contract keys of the
reference arm (which needs no GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = 1.0 + rank            # rank 1 is the slow one
    units = 10.0 * (rank + 1)
    bench.barrier(world, rank)
    q.put((rank, bench.aggregate(elapsed, units, world)))
    dist.destroy_process_group()


def test_aggregate_max_time_sum_units_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0] == out[1] == (2.0, 30.0)


def test_aggregate_single_rank_passthrough():
    assert bench.aggregate(1.5, 7.0, 1) == (1.5, 7.0)


def test_clock_summary_window_and_reasons():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [
        (10.0, ["0", "900", "2070", "200", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]),
        (11.0, ["0", "1800", "2070", "1300", "0x4", "Not Active", "Not Active", "Not Active", "Active"]),
        (11.5, ["0", "1700", "2070", "1350", "0x4", "Not Active", "Not Active", "Not Active", "Active"]),
        (13.0, ["0", "1000", "2070", "300", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]),
    ]
    c = s.summary(10.9, 12.0)
    assert c["sm_mhz"] == 1750.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 2 and c["window"] == "timed"
    c2 = s.summary(20.0, 21.0)           # nothing inside: falls back to the whole run
    assert c2["window"] == "whole run" and c2["samples"] == 4


def test_traffic_record_requires_matching_kernel(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    for rel in bench.KERNEL_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        dst.write_bytes(open(os.path.join(ROOT, rel), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"kernel_sha": bench.kernel_source_hash(),
           "workloads": {"w": {"dram_bytes_per_launch": 123}}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic("w") == 123
    assert bench.load_traffic("other") is None
    rec["kernel_sha"] = "stale"
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic("w") is None
    # a workload re-captured later carries its own hash, which wins over the file's
    rec["workloads"]["w"]["kernel_sha"] = bench.kernel_source_hash()
    rec["workloads"]["v"] = {"dram_bytes_per_launch": 7}
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic("w") == 123 and bench.load_traffic("v") is None
    rec["workloads"]["w"]["kernel_sha"] = "stale"
    rec["kernel_sha"] = bench.kernel_source_hash()
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.load_traffic("w") is None and bench.load_traffic("v") == 7


def test_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks["bf16_tflops"] == 1900.0


@pytest.mark.slow
def test_reference_arm_json_line():
    """The reference arm (CPU checker) runs without a GPU and prints the contract keys."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1", "--workload", "gemm256_int_f16",
                        "--ref-seconds", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "impl"):
        assert k in line
    assert line["impl"] == "reference" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0


def test_nvml_reader_rows_with_a_fake_library():
    """The in-process clock sampler's row: SM clock, maximum, power in W and the four
    reasons the bench judges, decoded from NVML's reason bits (read-only queries only)."""
    import ctypes

    class FakeNvml:
        def __init__(self, mhz, mw, reasons):
            self.v = (mhz, mw, reasons)

        def nvmlDeviceGetClockInfo(self, h, which, out):
            out._obj.value = self.v[0]
            return 0

        def nvmlDeviceGetPowerUsage(self, h, out):
            out._obj.value = self.v[1]
            return 0

        def nvmlDeviceGetCurrentClocksEventReasons(self, h, out):
            out._obj.value = self.v[2]
            return 0

    r = bench.NvmlReader.__new__(bench.NvmlReader)
    r.ct, r.h, r.index, r.max_mhz = ctypes, None, 3, 2070
    r.lib = FakeNvml(1850, 1375500, 0x4 | 0x1)
    r.reasons_fn = r.lib.nvmlDeviceGetCurrentClocksEventReasons
    row = r.row()
    assert row[:4] == ["3", "1850", "2070", "1375.50"]
    assert row[5:] == ["Not Active", "Not Active", "Not Active", "Active"]   # power cap only
    r.lib = FakeNvml(900, 200000, 0x8 | 0x40 | 0x20)
    r.reasons_fn = r.lib.nvmlDeviceGetCurrentClocksEventReasons
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [(1.0, r.row())]
    c = s.summary(0.0, 2.0)
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert c["sm_mhz"] == 900.0 and c["sm_max_mhz"] == 2070.0
