"""Throughput of the sm_103a GEMM D = alpha*A*B + beta*C on synthetic operands.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one GEMM over the workload (default: 8192^3 bf16 with C, alpha 1.25,
beta 0.5).  Operands are generated on the host from fixed seeds, copied to the device
once, and stay resident; the timed region holds K back-to-back launches through the C
ABI, bracketed by a barrier and a device synchronise, timed with CUDA events on the
launching stream.  The working set (A, B, C, D) is larger than L2, so no flush is needed
between steps.  Under torchrun every rank runs its own replica (there is no exchange
step in a GEMM), and the slowest rank's time sets the aggregate.

The JSON line carries: value (TFLOP/s, all ranks), e2e (same metric through the public
API with pinned host buffers, copies inside the timed region), roofline (the kernel's
average launch time against the measured tensor peak), clocks sampled during the timed
region, and cpu_baseline (the CPU checker timed on a bounded sample of the same problem).
--impl reference times that CPU checker alone, on rank 0.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/s) at 8192^3 fp16->fp32 acc; % of GB300 dense FP16 peak"
DEFAULT_WORKLOAD = "gemm8192_bf16_c"
METRIC_MX = "GEMM TFLOP/s (2MNK/s) at 8192^3 block-scaled (MX) e4m3 inputs->fp32 acc; % of GB300 dense FP8 peak"
METRIC_FP8 = "GEMM TFLOP/s (2MNK/s) at 8192^3 e4m3 inputs->fp32 acc; % of GB300 dense FP8 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# NVIDIA's published dense FP16/BF16 tensor rate of one GB300 (Blackwell Ultra) GPU: the HGX
# B300 specification lists 36 PFLOPS FP16/BF16 for 8 GPUs, quoted with 2:4 structured
# sparsity, i.e. 2.25 PFLOP/s dense per GPU
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_SOURCE = ("NVIDIA HGX B300 specification: FP16/BF16 tensor 36 PFLOPS per 8 GPUs with 2:4 "
                  "sparsity = 2.25 PFLOP/s dense per GPU")
KERNEL_SOURCES = ["layout_algebra_gb300/csrc/gemm_sm103.cu", "layout_algebra_gb300/csrc/gemm_kernel.cuh",
                  "layout_algebra_gb300/csrc/gemm_launch.cuh", "layout_algebra_gb300/csrc/gemm_inst.cu",
                  "layout_algebra_gb300/csrc/ptx.cuh"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--epilogue", default="plain", choices=["plain", "bias-gelu", "bias-gelu-e4m3"],
                    help="fused epilogue to time (gb_gemm_ex): bias + GELU, optionally with amax "
                         "and a scaled E4M3 output")
    ap.add_argument("--graph", action="store_true",
                    help="launch the timed steps from one captured CUDA graph (for GEMMs shorter "
                         "than the host's per-call work); kernel time = graph time / steps")
    ap.add_argument("--workspace", action="store_true",
                    help="time the workspace entry point (stream-K schedule where it helps)")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="CPU time budget of the whole reference run")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------- helpers


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    w = d.get("workloads", {}).get(workload)
    if w is None:
        return None
    # a workload re-captured on later sources carries its own hash; the others share the file's
    if w.get("kernel_sha", d.get("kernel_sha")) != kernel_source_hash():
        return None
    return w.get("dram_bytes_per_launch")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(elapsed_s, units, world, device=None):
    """(max elapsed over ranks, sum of units over ranks); plain values when world == 1."""
    if world == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), u.item()


def barrier(world, local):
    if world > 1:
        import torch.distributed as dist
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[local])
        else:
            dist.barrier()


class NvmlReader:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes): SM clock, its
    maximum, power draw and the clock event reasons of one GPU.  Nothing is set."""

    SM = 1                          # NVML_CLOCK_SM
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}

    def __init__(self, nvml_index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(nvml_index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for GPU %d" % nvml_index)
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.index = nvml_index
        u = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, ctypes.byref(u))
        self.max_mhz = u.value

    def row(self):
        """One sample in nvidia-smi's field order (see ClockSampler.FIELDS)."""
        ct = self.ct
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, ct.byref(mhz))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reasons_fn(self.h, ct.byref(rs))
        act = lambda bit: "Active" if rs.value & bit else "Not Active"   # noqa: E731
        return [str(self.index), str(mhz.value), str(self.max_mhz), "%.2f" % (mw.value / 1000.0),
                hex(rs.value), act(0x8), act(0x40), act(0x20), act(0x4)]


class ClockSampler:
    """Clock/throttle samples, each stamped with its arrival time: NVML queried in-process
    every 5 ms when the driver's library loads, else nvidia-smi every 100 ms."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    NVML_PERIOD_S = 0.005

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        self.source = None
        self._stop = False
        try:
            self.nvml = NvmlReader(int(gpu_index))
            self.nvml.row()
        except (OSError, ValueError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            self.source = "NVML in-process, every %d ms" % round(self.NVML_PERIOD_S * 1e3)
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            return
        self.source = "nvidia-smi, every 100 ms"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self):
        while not self._stop:
            self.samples.append((time.time(), self.nvml.row()))
            time.sleep(self.NVML_PERIOD_S)

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append((time.time(), parts))

    def stop(self):
        self._stop = True
        if self.nvml is not None:
            self.thread.join(timeout=1)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed"
        if not inside:
            inside = [p for _, p in self.samples]
            window = "whole run"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[5:9]) if v.lower() == "active"})
        power = [num(p[3]) for p in inside if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window,
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max(power) if power else None,
                "source": getattr(self, "source", None)}


def oracle_sample(problem, data, seconds, max_rows=None):
    """Time the CPU checker on whole rows of D until `seconds` elapse (at least one row)."""
    import numpy as np
    from layout_algebra_gb300 import workloads as W
    from oracle import gemm_ref as O
    p = problem
    A, B = W.bits(data["A"]), W.bits(data["B"])
    C = W.bits(data["C"]) if data["C"] is not None else None
    code = O.dtype_code(p.dtype)
    a_code = O.dtype_code(p.a_fmt) if p.a_fmt else code
    b_code = O.dtype_code(p.b_fmt) if p.b_fmt else code
    ma = 0 if p.majorA == "K" else 1
    mb = 0 if p.majorB == "K" else 1
    threads = O.max_threads()
    cols_all = np.arange(p.N, dtype=np.int64)

    def run_rows(r0, nrows, ncols):
        rows = np.repeat(np.arange(r0, r0 + nrows, dtype=np.int64), ncols)
        cols = np.tile(cols_all[:ncols], nrows)
        t = time.perf_counter()
        if p.scale_codes is not None:
            O.gemm_mx(p.M, p.N, p.K, p.alpha, A, data["lda"], a_code, data["SFA"].numpy(), data["ld_sf"],
                      B, data["ldb"], b_code, data["SFB"].numpy(), data["ld_sf"], p.beta, C, p.N, code,
                      rows, cols, threads=threads)
        else:
            O.gemm(p.M, p.N, p.K, p.alpha, A, data["lda"], ma, B, data["ldb"], mb, p.beta, C, p.N,
                   code, rows, cols, threads=threads, a_dtype=a_code, b_dtype=b_code)
        return time.perf_counter() - t

    # probe with a slice of one row, then size the sample to the time budget
    probe_cols = min(p.N, 1024)
    tp = run_rows(0, 1, probe_cols)
    per_entry = max(tp / probe_cols, 1e-9)
    entries = int(seconds / per_entry)
    rows = max(1, min(entries // p.N, p.M if max_rows is None else max_rows))
    if entries < p.N:
        ncols = max(1, min(p.N, entries))
        rows = 1
    else:
        ncols = p.N
    t = run_rows(0, rows, ncols)
    n_out = rows * ncols
    return {"seconds": t, "outputs": n_out, "rows": rows, "cols": ncols, "threads": threads,
            "flops": 2.0 * n_out * p.K}


# ----------------------------------------------------------------------------- arms


def run_reference(args):
    """The CPU checker as it stands, on host cores, over bounded samples of the workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from layout_algebra_gb300 import workloads as W
    p = problem_of(args.workload)
    data = W.make(p)
    total_budget = args.ref_seconds
    per_step = max(0.05, total_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(p, data, per_step)
    flops = secs = 0.0
    last = None
    for _ in range(args.steps):
        last = oracle_sample(p, data, per_step)
        flops += last["flops"]
        secs += last["seconds"]
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": (METRIC_MX if p.scale_codes else METRIC_FP8) if p.a_fmt else METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(p),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["threads"], "kind": "oracle",
                         "sample": "each step: %d row(s) x %d column(s) of D of the %s problem "
                                   "(fp64 triple loop, OpenMP over outputs)"
                                   % (last["rows"], last["cols"], p.name)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def problem_of(name):
    from layout_algebra_gb300 import workloads as W
    if name in W.FP8_WORKLOADS:
        return W.FP8_WORKLOADS[name]
    if name in W.EXTRA_WORKLOADS:
        return W.EXTRA_WORKLOADS[name]
    return W.WORKLOADS[name]


def workload_config(p):
    cfg = {"workload": p.name, "M": p.M, "N": p.N, "K": p.K, "operand_dtype": p.dtype,
            "majorA": p.majorA, "majorB": p.majorB, "alpha": p.alpha, "beta": p.beta,
            "has_C": p.has_c, "values": p.dist, "seed": p.seed,
            "l2": "inputs larger than L2 (no flush between steps)"
            if p.algorithmic_bytes > 256 * 2**20 else "working set may fit in L2",
            "parallelism": "replicas"}
    if p.a_fmt:
        cfg["operand_dtype"] = "%s x %s inputs, %s C and D" % (p.a_fmt, p.b_fmt, p.dtype)
    return cfg


def run_gb300(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from layout_algebra_gb300 import binding as G
    from layout_algebra_gb300 import workloads as W
    p = problem_of(args.workload)
    f8 = p.a_fmt is not None
    mx = p.scale_codes is not None
    out_dt = W.torch_dtype(p.dtype)
    data = W.make(p)
    A, B = data["A"].to(dev), data["B"].to(dev)
    C = data["C"].to(dev) if data["C"] is not None else None
    if mx:   # scales packed once, outside the timed region
        sfa = G.mx_pack_scales(0, p.M, p.K, data["SFA"].to(dev), data["ld_sf"])
        sfb = G.mx_pack_scales(1, p.N, p.K, data["SFB"].to(dev), data["ld_sf"])
    D = torch.empty(p.M * p.N, dtype=out_dt, device=dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    lda, ldb = data["lda"], data["ldb"]
    cptr = C.data_ptr() if C is not None else None
    ws = G.make_workspace(dev) if args.workspace else None
    import ctypes
    epi = None
    if args.epilogue != "plain":
        from layout_algebra_gb300._native import Epilogue
        g = torch.Generator().manual_seed(p.seed + 1)
        bias = torch.randn(p.N, generator=g).to(out_dt).to(dev)
        amax = torch.zeros(1, dtype=torch.float32, device=dev)
        fp8 = args.epilogue.endswith("e4m3")
        if fp8:
            D = torch.empty(p.M * p.N, dtype=torch.float8_e4m3fn, device=dev)
        epi = Epilogue(bias.data_ptr(), 2, amax.data_ptr() if fp8 else None, 1 if fp8 else 0,
                       16.0 if fp8 else 1.0)
    dcode = 1 if out_dt == torch.bfloat16 else 0

    def launch():
        sh = torch.cuda.current_stream().cuda_stream   # the capture stream inside a graph capture
        if mx:
            st = G.lib().gb_gemm_mxfp8(G.fp8_format(p.a_fmt), G.fp8_format(p.b_fmt), dcode, p.M, p.N, p.K,
                                       p.alpha, A.data_ptr(), lda, sfa.data_ptr(), B.data_ptr(), ldb,
                                       sfb.data_ptr(), p.beta, cptr, D.data_ptr(),
                                       ctypes.byref(epi) if epi is not None else None,
                                       ws.data_ptr() if ws is not None else None,
                                       ws.numel() if ws is not None else 0, sh)
        elif f8:
            st = G.lib().gb_gemm_fp8(G.fp8_format(p.a_fmt), G.fp8_format(p.b_fmt), dcode, p.M, p.N,
                                     p.K, p.alpha, A.data_ptr(), lda, B.data_ptr(), ldb, p.beta,
                                     cptr, D.data_ptr(),
                                     ctypes.byref(epi) if epi is not None else None,
                                     ws.data_ptr() if ws is not None else None,
                                     ws.numel() if ws is not None else 0, sh)
        elif epi is not None:
            st = G.lib().gb_gemm_ex(dcode, p.M, p.N, p.K, p.alpha, A.data_ptr(), lda,
                                    G.major_code(p.majorA), B.data_ptr(), ldb, G.major_code(p.majorB),
                                    p.beta, cptr, D.data_ptr(), ctypes.byref(epi),
                                    ws.data_ptr() if ws is not None else None,
                                    ws.numel() if ws is not None else 0, sh)
        elif ws is not None:
            st = G.raw_call_ws(A.dtype, p.M, p.N, p.K, p.alpha, A.data_ptr(), lda, p.majorA,
                               B.data_ptr(), ldb, p.majorB, p.beta, cptr, D.data_ptr(),
                               ws.data_ptr(), ws.numel(), sh)
        else:
            st = G.raw_call(A.dtype, p.M, p.N, p.K, p.alpha, A.data_ptr(), lda, p.majorA,
                            B.data_ptr(), ldb, p.majorB, p.beta, cptr, D.data_ptr(), sh)
        if st != 0:
            raise G.GemmError(st)

    for _ in range(max(3, args.warmup)):
        launch()
    torch.cuda.synchronize()
    st, detail = G.last_device_status()
    if st != 0:
        raise RuntimeError("device status %d (%#x) during warm-up" % (st, detail))

    try:   # NVML's index of this device (CUDA_VISIBLE_DEVICES taken into account)
        phys = torch.cuda._get_nvml_device_index(dev)
    except Exception:   # noqa: BLE001 - any failure: fall back to the variable itself
        phys = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local if world > 1 else 0]
    sampler = ClockSampler(phys)
    time.sleep(0.3)

    graph = None
    if args.graph:
        # the launches of the timed region recorded once; the host's per-call work (planning,
        # tensor maps) happens at capture time, outside the timed region
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                launch()
        torch.cuda.synchronize()
        graph.replay()                      # one untimed replay
        torch.cuda.synchronize()
    # the K launches back to back between one pair of events on the launching stream (an event
    # between two launches would keep a launch's set-up from overlapping the previous one's end,
    # as it does in a user's sequence of GEMMs); kernel time per launch = total / K
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world, local)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    t_start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            launch()
    t_end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world, local)
    time.sleep(0.15)
    sampler.stop()
    st, detail = G.last_device_status()
    if st != 0:
        raise RuntimeError("device status %d (%#x) in the timed region" % (st, detail))
    total_ms = t_start.elapsed_time(t_end)
    kernel_ms = total_ms / args.steps
    # after the timed region: each launch alone between its own events (launch-to-launch overlap
    # lost), for the spread of single launches
    per_launch_ms = []
    if graph is None:
        for _ in range(min(args.steps, 10)):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
            e1.synchronize()
            per_launch_ms.append(e0.elapsed_time(e1))
    launch_stats = {"single_launch_ms_best": min(per_launch_ms) if per_launch_ms else None,
                    "single_launch_ms_median": statistics.median(per_launch_ms) if per_launch_ms else None}
    elapsed_s, total_flops = aggregate(total_ms / 1e3, float(p.flops) * args.steps, world, dev)
    value = total_flops / elapsed_s / 1e12
    clocks = sampler.summary(t_wall0 - 0.05, t_wall1 + 0.05)

    # end to end through the public API with pinned host buffers
    A_h, B_h = data["A"].pin_memory(), data["B"].pin_memory()
    C_h = data["C"].pin_memory() if data["C"] is not None else None
    D_h = torch.empty(p.M * p.N, dtype=D.dtype, pin_memory=True)

    if mx:
        SFA_h, SFB_h = data["SFA"].pin_memory(), data["SFB"].pin_memory()

    def public_call():
        if mx:
            # host operands and plain scales in, D out: copies, packing and the GEMM
            Ad, Bd = A_h.to(dev, non_blocking=True), B_h.to(dev, non_blocking=True)
            Cd = C_h.to(dev, non_blocking=True) if C_h is not None else None
            pa = G.mx_pack_scales(0, p.M, p.K, SFA_h.to(dev, non_blocking=True), data["ld_sf"])
            pb = G.mx_pack_scales(1, p.N, p.K, SFB_h.to(dev, non_blocking=True), data["ld_sf"])
            Dd = G.gemm_mxfp8(Ad, Bd, p.M, p.N, p.K, lda=lda, ldb=ldb, sfa=pa, sfb=pb, a_format=p.a_fmt,
                              b_format=p.b_fmt, out_dtype=out_dt, alpha=p.alpha, beta=p.beta, C=Cd,
                              workspace=ws)
            D_h.copy_(Dd, non_blocking=True)
        elif epi is not None:
            # the fused epilogue has no host-operand form: host copies, gb_gemm_ex, D back
            Ad, Bd = A_h.to(dev, non_blocking=True), B_h.to(dev, non_blocking=True)
            Cd = C_h.to(dev, non_blocking=True) if C_h is not None else None
            Dd = G.gemm_fused(Ad, Bd, p.M, p.N, p.K, lda=lda, ldb=ldb, majorA=p.majorA, majorB=p.majorB,
                              alpha=p.alpha, beta=p.beta, C=Cd, bias=bias, activation="gelu",
                              amax=amax if fp8 else None, out_format="e4m3" if fp8 else "input",
                              out_scale=16.0 if fp8 else 1.0)
            D_h.copy_(Dd, non_blocking=True)
        elif f8:
            # gb_gemm_fp8_host: host buffers in, D out (staging and overlap in the library)
            G.gemm_fp8(A_h, B_h, p.M, p.N, p.K, lda=lda, ldb=ldb, a_format=p.a_fmt,
                       b_format=p.b_fmt, out_dtype=out_dt, alpha=p.alpha, beta=p.beta, C=C_h,
                       D=D_h)
        else:
            # gb_gemm_f16_host / gb_gemm_bf16_host
            G.gemm(A_h, B_h, p.M, p.N, p.K, lda=lda, ldb=ldb, majorA=p.majorA, majorB=p.majorB,
                   alpha=p.alpha, beta=p.beta, C=C_h, D=D_h)

    for _ in range(2):
        public_call()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.e2e_steps, args.steps))
    barrier(world, local)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        public_call()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world, local)
    e2e_s, e2e_flops = aggregate(e0.elapsed_time(e1) / 1e3, float(p.flops) * e2e_steps, world, dev)
    h2d = sum(t.numel() * t.element_size()
              for t in (data["A"], data["B"], data["C"], data.get("SFA"), data.get("SFB")) if t is not None)
    d2h = D_h.numel() * D_h.element_size()
    st, detail = G.last_device_status()
    if st != 0:
        raise RuntimeError("device status %d (%#x) in the end-to-end region" % (st, detail))

    peaks, peak_src = load_peaks()
    # an FP8 contraction runs at twice the 16-bit tensor rate (nominal 4.5 vs 2.25 PFLOP/s
    # dense): its peak is the measured bf16 peak times that ratio
    ratio = 2.0 if f8 else 1.0
    burst = ratio * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = ratio * float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = p.flops / (kernel_ms / 1e3) / 1e12
    traffic = load_traffic(p.name)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # SMs x SM clock under load x the per-SM dense rate behind the nominal figure (8192 16-bit
    # flop per clock per SM: 2.25 PFLOP/s at about 1.8 GHz on 152 SMs)
    clock_peak = ratio * 152 * (clocks.get("sm_mhz") or 2070.0) * 1e6 * 8192 / 1e12
    if p.flops / p.algorithmic_bytes < burst * 1e12 / (hbm * 1e9):
        # below the ridge point the kernel is bound by moving the operands through HBM
        gbs = p.algorithmic_bytes / (kernel_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "traffic": traffic,
                    "peak_source": "%s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_src,
                    "tflops": achieved, "kernel": "gb::gemm_kernel", "kernel_ms": kernel_ms,
                    **launch_stats,
                    "algorithmic_flops_per_launch": p.flops,
                    "algorithmic_bytes_per_launch": p.algorithmic_bytes}
    else:
        # a run that reached the power cap is a long-step measurement: compare it with the
        # sustained peak; otherwise against the burst peak of a kernel timed alone
        capped = "sw_power_cap" in (clocks.get("reasons") or [])
        peak, which = (sustained, "sustained") if capped else (burst, "burst")
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "peak_source": ("%s %s (MEASURED_PEAKS.json bf16_tflops%s) x 2, the nominal FP8:bf16 "
                                    "dense ratio" if f8 else
                                    "%s %s (MEASURED_PEAKS.json bf16_tflops%s); fp16 and bf16 share the rate")
                                   % (peak_src, which, "_sustained" if capped else ""),
                    "frac_of_burst": achieved / burst,
                    "frac_of_sustained": achieved / sustained,
                    "frac_of_nominal": achieved / (NOMINAL_BF16_TFLOPS * ratio),
                    "nominal_source": NOMINAL_SOURCE,
                    "frac_of_clock_peak": achieved / clock_peak, "clock_peak": clock_peak,
                    "kernel": "gb::gemm_kernel", "kernel_ms": kernel_ms,
                    **launch_stats,
                    "algorithmic_flops_per_launch": p.flops,
                    "algorithmic_bytes_per_launch": p.algorithmic_bytes}
    if clocks.get("sm_mhz"):
        # the kernel time in SM clock cycles at the median clock of the timed region: compares
        # runs at different clocks (a short burst at the maximum, a long power-capped run)
        roofline["sm_cycles_per_launch"] = kernel_ms * 1e-3 * clocks["sm_mhz"] * 1e6
        roofline["kernel_ms_at_max_clock"] = roofline["sm_cycles_per_launch"] / (
            (clocks.get("sm_max_mhz") or clocks["sm_mhz"]) * 1e3)

    line = {
        "metric": METRIC_FP8 if f8 else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": p.a_fmt if f8 else p.dtype, "data": "synthetic",
        "config": workload_config(p),
        "e2e": {"value": e2e_flops / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "entry_point": ("host copies + gb_gemm_mxfp8 (no host form)" if mx else
                                "gb_gemm_fp8_host" if f8 else
                                "host copies + gb_gemm_ex (no host form)" if epi is not None else
                                "gb_gemm_%s_host" % p.dtype)},
        "roofline": roofline, "clocks": clocks, "gpu_launches": args.steps,
    }
    # how the timed launches were made (kept out of "config", which names the workload only
    # and is the same in both arms)
    path = {"entry_point": ("gb_gemm_%s_ws (workspace, stream-K where it helps)" % p.dtype
                            if ws is not None else "gb_gemm_%s" % p.dtype)}
    if graph is not None:
        path["launch"] = "one CUDA graph of %d launches" % args.steps
    if mx:
        path["entry_point"] = "gb_gemm_mxfp8" + (" (workspace)" if ws is not None else "")
        path["scales"] = "E8M0 per 32 K elements of each row of A and column of B, codes %d..%d" % p.scale_codes
        line["metric"] = METRIC_MX
    elif f8:
        path["entry_point"] = "gb_gemm_fp8" + (" (workspace)" if ws is not None else "")
    elif epi is not None:
        path["entry_point"] = "gb_gemm_ex"
        path["epilogue"] = args.epilogue
    line["path"] = path
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = oracle_sample(p, data, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": s["flops"] / s["seconds"] / 1e12, "unit": "TFLOP/s", "cores": s["threads"],
            "kind": "oracle",
            "sample": "%d row(s) x %d column(s) of D of the %s problem, fp64 triple loop with "
                      "OpenMP over outputs, %.1f s" % (s["rows"], s["cols"], p.name, s["seconds"])}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
