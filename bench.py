#!/usr/bin/env python3
"""Benchmark of the GB300 FP32 SGEMM (C = A.B, row-major, beta = 0).

Default: the M=N=K=4096 workload (A, B ~ N(0,1) from seed 3) on one GPU; one
JSON line on stdout.  A step is one sgemm_run over the resident inputs.  L2 is
flushed (a 256 MiB write) before every step, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on a bounded sample
  python bench.py --sweep                # one line per named workload

With N > 1 (torchrun) every rank runs its own replica of the workload: the
product has no exchange step, so there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

REPO = os.path.dirname(os.path.abspath(__file__))
if REPO not in sys.path:
    sys.path.insert(0, REPO)

from dense_fp32_gemm_09_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

DEFAULT_WORKLOAD = "sgemm_4096"
METRIC = "SGEMM TFLOP/s (2MNK/t) at M=N=K=4096 FP32; % of GB300 FP32 CUDA-core peak"
FMA_PER_CLK_PER_SM = 128          # FP32 lanes per SM (4 SMSPs x 32)
L2_FLUSH_BYTES = 256 << 20


def describe(w) -> str:
    dist = "N(0,1)" if w.dist == "normal" else f"U[{w.lo:g},{w.hi:g})"
    return f"{w.name}: M={w.M} N={w.N} K={w.K} fp32 row-major, A,B ~ {dist} seed {w.seed}"


# Files whose text is the code of the FFMA kernels, the tile table's template
# parameters included.
KERNEL_SOURCES = ["sgemm_ffma.cuh", "sgemm_sched.cuh", "sgemm_args.h", "sgemm_epilogue.cuh",
                  "sgemm_kernels_main.cu", "sgemm_kernels_small.cu", "sgemm_kernels_any.cu"]


def code_only(text: str) -> str:
    """C++ source text without its comments and with blank space collapsed: what the
    compiler sees, so that editing a comment does not void a recorded capture."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_sources_hash(read=None) -> str:
    """sha256 (first 16 hex digits) of the code of KERNEL_SOURCES.  `read(name)`
    returns a file's text (default: the working tree)."""
    import hashlib
    if read is None:
        def read(name):
            with open(os.path.join(REPO, "dense_fp32_gemm_09_gb300", "csrc", name)) as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(code_only(read(f)).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu capture, or None when there is
    none for this kernel and workload or the kernel sources changed since."""
    try:
        with open(os.path.join(REPO, "profiles", "traffic_per_launch.txt")) as f:
            lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    except OSError:
        return None
    cur = kernel_sources_hash()
    for fields in lines:
        if len(fields) >= 5 and fields[0] == kernel and fields[1] == workload and fields[4] == cur:
            return int(fields[2]) + int(fields[3])
    return None


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over all ranks of the default process group
    (identity when not distributed).  The timed region's length is the slowest
    rank's, so throughput is computed from these maxima."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_tflops(world: int, flops_per_rank: float, ms: float) -> float:
    """Aggregate throughput of `world` replicas that each did `flops_per_rank` in a
    region whose (max over ranks) length is `ms`."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def measured_peaks() -> dict:
    try:
        with open(os.path.join(REPO, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


# ---------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; reading only)
# ---------------------------------------------------------------------------
class ClockSampler:
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, torch_index: int, period_s: float = 0.01):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = ctypes.c_void_p()
            if not self._find_handle(torch_index):
                raise OSError("no NVML handle for this CUDA device")
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
        except OSError as e:
            self.nvml = None
            self.error = str(e)

    def _find_handle(self, torch_index: int) -> bool:
        """NVML handle of the CUDA device torch calls `torch_index` (matched by UUID,
        then PCI address, since NVML numbers every GPU of the node)."""
        import torch
        props = torch.cuda.get_device_properties(torch_index)
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            key = ("GPU-" + str(uuid)).encode()
            if self.nvml.nvmlDeviceGetHandleByUUID(key, ctypes.byref(self.handle)) == 0:
                return True
        if hasattr(props, "pci_bus_id"):
            bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                        getattr(props, "pci_device_id", 0))
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(),
                                                           ctypes.byref(self.handle)) == 0:
                return True
        return self.nvml.nvmlDeviceGetHandleByIndex_v2(torch_index,
                                                       ctypes.byref(self.handle)) == 0

    def _run(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0:
                self.samples.append(int(clk.value))
            if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle,
                                                                ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(self.period)

    def __enter__(self):
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self) -> dict:
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": f"NVML unavailable: {self.error}"}
        reasons = [n for bit, n in self.REASONS.items() if self.reasons & bit]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples)}


# ---------------------------------------------------------------------------
# CPU side: the oracle on a bounded sample (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def oracle_rate(w, A, B, target_s: float = 12.0, max_rows: int | None = None):
    """TFLOP/s of the fp64 oracle on whole rows of C, sized to about target_s."""
    import numpy as np
    import oracle
    oracle.build()
    An, Bn = A.numpy(), B.numpy()
    threads = oracle.default_threads()
    rows = max(1, min(w.M, 16))
    t0 = time.perf_counter()
    oracle.gemm_f64_rows(An, Bn, np.arange(rows, dtype=np.int32), nthreads=threads)
    dt = time.perf_counter() - t0
    per_row = dt / rows
    want = int(max(1, min(w.M if max_rows is None else max_rows,
                          (target_s - dt) / max(per_row, 1e-9))))
    idx = np.linspace(0, w.M - 1, want).astype(np.int32)
    t0 = time.perf_counter()
    oracle.gemm_f64_rows(An, Bn, idx, nthreads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * want * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{want} of {w.M} rows of C (all N={w.N} columns, K={w.K}), "
                      f"fp64 accumulation, {dt:.2f} s wall on {threads} threads",
            "seconds": dt}


L2_NOTE = ("GPU arm: L2 flushed before every step (256 MiB write, outside the timed "
           "events); the oracle arm runs on the host cores")


def workload_config(w, world: int, extra: str = "") -> dict:
    """The `config` of a bench line: the workload and how it is run, the same for
    the GPU arm and the oracle (reference) arm of the same workload."""
    return {"workload": describe(w) + extra, "M": w.M, "N": w.N, "K": w.K, "l2": L2_NOTE,
            "parallelism": "replicas" if world > 1 else "single"}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    A, B = make_inputs(w)
    rates = []
    steps_t = []
    per_step_s = max(1.0, 120.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        r = oracle_rate(w, A, B, target_s=per_step_s)
        if i >= args.warmup:
            rates.append(r["value"])
            steps_t.append(r["seconds"])
    value = statistics.median(rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(steps_t), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "cpu_baseline": {**{k: v for k, v in r.items() if k != "seconds"}, "value": value},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU side
# ---------------------------------------------------------------------------
def bench_gpu(args, w, dist_ctx):
    import torch

    import dense_fp32_gemm_09_gb300 as sg
    from dense_fp32_gemm_09_gb300._abi import check

    rank, world, local = dist_ctx
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = sg.load()
    A, B = make_inputs(w)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.empty(w.M, w.N, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    scaled = args.alpha != 1.0 or args.beta != 0.0
    ta, tb = args.trans[0] == "T", args.trans[1] == "T"
    kid = getattr(args, "kernel_id", None)
    if kid is not None:
        # one forced tile-table entry (--tile-sweep); entries that cannot serve
        # these operands are skipped
        run_fn = lib.sgemm_run_with
        run_args = (w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.N, dC.data_ptr(), w.N,
                    kid, 0, sh)
        if run_fn(*run_args) == sg.SGEMM_ERR_UNSUPPORTED:
            return None
    elif ta or tb:
        # the same logical operands, stored transposed where asked
        sA = A.t().contiguous().to(dev) if ta else dA
        sB = B.t().contiguous().to(dev) if tb else dB
        if scaled:
            dC.normal_()
        run_fn = lib.sgemm_run_op
        run_args = (int(ta), int(tb), w.M, w.N, w.K, args.alpha, sA.data_ptr(),
                    w.M if ta else w.K, sB.data_ptr(), w.K if tb else w.N, args.beta,
                    dC.data_ptr(), w.N, sh)
    elif scaled:
        dC.normal_()
        run_fn = lib.sgemm_run_ex
        run_args = (w.M, w.N, w.K, args.alpha, dA.data_ptr(), w.K, dB.data_ptr(), w.N, args.beta,
                    dC.data_ptr(), w.N, -1, 0, sh)
    else:
        run_fn = lib.sgemm_run
        run_args = (w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.N, dC.data_ptr(), w.N,
                    sh)
    if kid is not None:
        cfg = {k: None for k in ("grid", "tiles", "sk_tiles", "ctas_per_sm", "cluster")}
        cfg["name"] = sg.kernel_table()[kid]["name"]
    elif ta or tb:   # the product runs on 16-byte-aligned transposed copies
        cfg = sg.sgemm_query_config(w.M, w.N, w.K, (w.K + 3) // 4 * 4, (w.N + 3) // 4 * 4, w.N,
                                    None, None, dC.data_ptr())
    else:
        cfg = sg.sgemm_query_config(w.M, w.N, w.K, w.K, w.N, w.N, dA.data_ptr(), dB.data_ptr(),
                                    dC.data_ptr())

    def barrier():
        if world > 1:
            import torch.distributed as tdist
            tdist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        check(run_fn(*run_args), "sgemm_run")
    barrier()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    n_launch0 = lib.sgemm_launch_count()
    with ClockSampler(local) as clocks:
        barrier()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))
            starts[i].record(stream)
            check(run_fn(*run_args), "sgemm_run")
            ends[i].record(stream)
        barrier()
        t_wall = time.perf_counter() - t_wall
    launches = lib.sgemm_launch_count() - n_launch0
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    med_ms = statistics.median(step_ms)
    mean_ms = statistics.fmean(step_ms)
    med_ms, mean_ms = max_over_ranks([med_ms, mean_ms], dev)

    e2e_ms = None
    if kid is None and not (ta or tb):   # the host entry takes row-major operands
        e2e_ms = time_e2e(lib, check, A, B, w, dA, dB, dC, sh, stream, args, barrier, dev)

    if rank != 0:
        return None
    return bench_line(args, w, world, med_ms, mean_ms, t_wall, e2e_ms, clocks, cfg, launches,
                      scaled, dev)


def time_e2e(lib, check, A, B, w, dA, dB, dC, sh, stream, args, barrier, dev):
    """ms per step of the host-buffer entry point: pinned host in, pinned host out."""
    import torch
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.empty(w.M, w.N).pin_memory()
    e2e_args = (w.M, w.N, w.K, hA.data_ptr(), w.K, hB.data_ptr(), w.N, hC.data_ptr(), w.N,
                dA.data_ptr(), dB.data_ptr(), dC.data_ptr(), sh)
    for _ in range(max(1, min(args.warmup, 3))):
        check(lib.sgemm_run_host(*e2e_args), "sgemm_run_host")
    barrier()
    e2e_steps = max(3, min(args.steps, 10))
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(stream)
    for _ in range(e2e_steps):
        check(lib.sgemm_run_host(*e2e_args), "sgemm_run_host")
    ee.record(stream)
    barrier()
    e2e_ms = es.elapsed_time(ee) / e2e_steps
    (e2e_ms,) = max_over_ranks([e2e_ms], dev)
    return e2e_ms


def bench_line(args, w, world, med_ms, mean_ms, t_wall, e2e_ms, clocks, cfg, launches, scaled,
               dev):
    import torch
    peaks = measured_peaks()
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    max_mhz = float(peaks.get("sm_max_mhz") or clocks.summary().get("sm_max_mhz") or 2070.0)
    peak_tflops = sms * FMA_PER_CLK_PER_SM * 2 * max_mhz * 1e6 / 1e12
    flops = float(w.flops)
    value = whole_job_tflops(world, flops, med_ms)
    achieved = flops / (med_ms * 1e-3) / 1e12
    clk = clocks.summary()
    trans = args.trans != "NN"
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": med_ms,
        "ms_per_step_mean": mean_ms, "wall_s_timed_region": t_wall,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": workload_config(
            w, world, (f"; C = {args.alpha:g}*A.B + {args.beta:g}*C" if scaled else "")
            + (f"; operands {args.trans} (T = stored transposed, transposed on the device "
               f"inside the step)" if trans else "")),
        "plan": {"kernel": cfg["name"], "grid": cfg.get("grid"), "tiles": cfg.get("tiles"),
                 "sk_tiles": cfg.get("sk_tiles"), "cluster": cfg.get("cluster"),
                 "ctas_per_sm": cfg.get("ctas_per_sm")},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tflops,
                     "unit": "TFLOP/s", "frac": achieved / peak_tflops,
                     "traffic": None if trans else recorded_traffic(cfg["name"], w.name),
                     "algorithmic_bytes": w.min_bytes,
                     "peak_basis": f"{sms} SMs x {FMA_PER_CLK_PER_SM} FP32 FMA/clk x 2 x "
                                   f"{max_mhz:.0f} MHz (max SM clock)",
                     "frac_at_measured_clock": (
                         achieved / (sms * FMA_PER_CLK_PER_SM * 2 * clk["sm_mhz"] * 1e-6)
                         if clk.get("sm_mhz") else None)},
        "clocks": clk,
        "e2e": None if e2e_ms is None else {
            "value": whole_job_tflops(world, flops, e2e_ms), "unit": "TFLOP/s",
            "ms_per_step": e2e_ms,
            "h2d_bytes_per_step": 4 * (w.M * w.K + w.K * w.N),
            "d2h_bytes_per_step": 4 * w.M * w.N},
        "gpu_launches": int(launches),
    }
    return line


TF32_PER_BF16 = 1.1 / 2.25   # nominal dense TF32 : BF16 tensor rates of the GB300


def tf32x3_summary(args, w, ctx) -> dict:
    """The 3xTF32 tensor-core variant on the same workload, measured in the same run and
    reported beside (never instead of) the FP32 line: its own value and roofline."""
    import argparse
    try:
        sub = argparse.Namespace(**{**vars(args), "steps": min(args.steps, 10),
                                    "warmup": max(3, min(args.warmup, 5))})
        line = bench_tf32x3(sub, w, ctx)
        if line is None:
            return {"error": "not rank 0"}
        keep = ("value", "unit", "ms_per_step", "ms_split", "ms_gemm", "dtype", "roofline",
                "clocks", "gpu_launches")
        return {k: line[k] for k in keep if k in line}
    except Exception as exc:   # noqa: BLE001 - the FP32 line stands on its own
        return {"error": f"{type(exc).__name__}: {exc}"[:300]}


def measured_tf32_peak(dev, n: int = 8192, reps: int = 5):
    """Dense TF32 tensor rate measured here, as the driver measures bf16: cuBLAS
    through torch.matmul on fp32 n^3 operands with TF32 allowed, best of `reps` after
    a warm-up (context only: nothing on the product path calls it).  None if it fails."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    try:
        torch.backends.cuda.matmul.allow_tf32 = True
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        c = torch.empty(n, n, device=dev)
        for _ in range(2):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except Exception:   # noqa: BLE001 - a context figure, never the product
        return None
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def bench_tf32x3(args, w, dist_ctx):
    """The 3xTF32 tensor-core variant: one step = one sgemm_tf32x3_run_ex call
    (operand split + tcgen05 GEMM), inputs resident.  The split and the GEMM are
    also timed apart through the two-step entry points (whose split writes Ahi too,
    as the two-step contract needs); the one-call split is the step less the GEMM."""
    import ctypes as ct

    import torch

    import dense_fp32_gemm_09_gb300 as sg
    from dense_fp32_gemm_09_gb300._abi import check

    rank, world, local = dist_ctx
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = sg.load()
    A, B = make_inputs(w)
    dA, dB = A.to(dev), B.to(dev)
    dC = torch.empty(w.M, w.N, device=dev)
    need = ct.c_size_t(0)
    check(lib.sgemm_tf32x3_workspace_size(w.M, w.N, w.K, ct.byref(need)), "workspace size")
    ws = torch.empty(need.value // 4 + 64, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    prep = (w.M, w.N, w.K, dA.data_ptr(), w.K, dB.data_ptr(), w.N, ws.data_ptr(), need.value, sh)
    mult = (w.M, w.N, w.K, args.alpha, args.beta, dC.data_ptr(), w.N, ws.data_ptr(), need.value,
            sh)

    def barrier():
        if world > 1:
            import torch.distributed as tdist
            tdist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        check(lib.sgemm_tf32x3_prepare(*prep), "prepare")
        check(lib.sgemm_tf32x3_multiply(*mult), "multiply")
    barrier()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        check(lib.sgemm_tf32x3_prepare(*prep), "prepare")
        ev[i][1].record(stream)
        check(lib.sgemm_tf32x3_multiply(*mult), "multiply")
        ev[i][2].record(stream)
    barrier()
    split_full_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    gemm_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)

    # the timed steps: one public call each, inputs resident
    run_dev = (w.M, w.N, w.K, args.alpha, dA.data_ptr(), w.K, dB.data_ptr(), w.N, args.beta,
               dC.data_ptr(), w.N, ws.data_ptr(), need.value, sh)
    for _ in range(args.warmup):
        flush.fill_(1.0)
        check(lib.sgemm_tf32x3_run_ex(*run_dev), "run_ex")
    barrier()
    ev1 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    n0 = lib.sgemm_launch_count()
    with ClockSampler(local) as clocks:
        barrier()
        for i in range(args.steps):
            flush.fill_(float(i))
            ev1[i][0].record(stream)
            check(lib.sgemm_tf32x3_run_ex(*run_dev), "run_ex")
            ev1[i][1].record(stream)
        barrier()
    launches = lib.sgemm_launch_count() - n0
    check(lib.sgemm_device_status(), "device status")
    tcfg = sg.SgemmConfig()
    check(lib.sgemm_tf32x3_query_config(w.M, w.N, w.K, ct.byref(tcfg)), "tf32x3 query")
    step_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev1)
    step_ms, split_full_ms, gemm_ms = max_over_ranks([step_ms, split_full_ms, gemm_ms], dev)
    split_ms = max(step_ms - gemm_ms, 0.0)

    # end to end: pinned host in, pinned host out, through the public entry point
    hA, hB = A.pin_memory(), B.pin_memory()
    hC = torch.empty(w.M, w.N).pin_memory()
    run_ex = (w.M, w.N, w.K, 1.0, dA.data_ptr(), w.K, dB.data_ptr(), w.N, 0.0, dC.data_ptr(),
              w.N, ws.data_ptr(), need.value, sh)
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, min(args.steps, 10))
    es.record(stream)
    for _ in range(e2e_steps):
        dA.copy_(hA, non_blocking=True)
        dB.copy_(hB, non_blocking=True)
        check(lib.sgemm_tf32x3_run_ex(*run_ex), "run_ex")
        hC.copy_(dC, non_blocking=True)
    ee.record(stream)
    barrier()
    (e2e_ms,) = max_over_ranks([es.elapsed_time(ee) / e2e_steps], dev)
    if rank != 0:
        return None
    peaks = measured_peaks()
    bf16 = float(peaks.get("bf16_tflops") or 1900.0)
    tf32 = measured_tf32_peak(dev)
    if tf32 is not None:
        peak = tf32
        basis = (f"measured here: cuBLAS TF32 GEMM 8192^3 {tf32:.1f} TFLOP/s (torch.matmul, "
                 f"TF32 allowed, best of 5); 3 TF32 MMAs per product")
    else:
        peak = bf16 * TF32_PER_BF16
        basis = (f"measured bf16 {bf16:.1f} TFLOP/s x nominal TF32/BF16 ratio "
                 f"{TF32_PER_BF16:.3f}; 3 TF32 MMAs per product")
    flops = float(w.flops)
    clk = clocks.summary()
    return {
        "metric": METRIC, "path": "tf32x3", "value": whole_job_tflops(world, flops, step_ms),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_ms, "ms_split": split_ms, "ms_gemm": gemm_ms,
        "ms_split_two_step": split_full_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "tf32x3",
        "data": "synthetic",
        "config": workload_config(w, world),
        "plan": {"kernel": f"tf32x3_kernel<BN={tcfg.bn}, {tcfg.stages} stages> + split "
                           f"kernels" + (" + sk_reduce_kernel" if tcfg.sk_tiles else ""),
                 "grid": tcfg.grid, "tiles": tcfg.tiles, "sk_tiles": tcfg.sk_tiles},
        "roofline": {"bound": "tensor", "achieved": 3 * flops / (gemm_ms * 1e-3) / 1e12,
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": 3 * flops / (gemm_ms * 1e-3) / 1e12 / peak, "traffic": None,
                     "peak_basis": basis,
                     "peak_derived_from_bf16": bf16 * TF32_PER_BF16,
                     "effective_fp32_tflops_gemm_only": flops / (gemm_ms * 1e-3) / 1e12},
        "clocks": clk,
        "e2e": {"value": whole_job_tflops(world, flops, e2e_ms), "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": 4 * (w.M * w.K + w.K * w.N),
                "d2h_bytes_per_step": 4 * w.M * w.N},
        "gpu_launches": int(launches),
    }


def bench_link(args):
    """Host<->device copy bandwidth from pinned host memory (the bound of the e2e
    lines): each direction alone, both at once, and one copy cut into 4 pieces on 4
    streams.  CUDA events around each copy, median of the steps."""
    import torch
    dev = torch.device("cuda", 0)
    out = []
    for mb in (16, 64, 256):
        n = (mb << 20) // 4
        h_in = torch.empty(n, dtype=torch.float32).pin_memory()
        h_out = torch.empty(n, dtype=torch.float32).pin_memory()
        d_a = torch.empty(n, dtype=torch.float32, device=dev)
        d_b = torch.empty(n, dtype=torch.float32, device=dev)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        split = [torch.cuda.Stream(dev) for _ in range(4)]

        def timed(fn, nbytes):
            ts = []
            for i in range(args.warmup + args.steps):
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                e1.synchronize()
                if i >= args.warmup:
                    ts.append(e0.elapsed_time(e1))
            ms = statistics.median(ts)
            return {"ms": ms, "gb_s": nbytes / (ms * 1e-3) / 1e9}

        def both():
            cur = torch.cuda.current_stream(dev)
            for st in (s_in, s_out):
                st.wait_stream(cur)
            with torch.cuda.stream(s_in):
                d_a.copy_(h_in, non_blocking=True)
            with torch.cuda.stream(s_out):
                h_out.copy_(d_b, non_blocking=True)
            cur.wait_stream(s_in)
            cur.wait_stream(s_out)

        def four():
            cur = torch.cuda.current_stream(dev)
            q = n // 4
            for j, st in enumerate(split):
                st.wait_stream(cur)
                with torch.cuda.stream(st):
                    d_a[j * q:(j + 1) * q].copy_(h_in[j * q:(j + 1) * q], non_blocking=True)
            for st in split:
                cur.wait_stream(st)

        row = {"bytes": 4 * n,
               "h2d": timed(lambda: d_a.copy_(h_in, non_blocking=True), 4 * n),
               "d2h": timed(lambda: h_out.copy_(d_b, non_blocking=True), 4 * n),
               "both_directions": timed(both, 8 * n),
               "h2d_4_streams": timed(four, 4 * n)}
        out.append(row)
        print(json.dumps({"metric": "host<->device copy bandwidth, pinned host memory",
                          "unit": "GB/s", **row}), flush=True)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--sweep", action="store_true", help="one line per named workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["ffma", "tf32x3"], default="ffma",
                    help="ffma: FP32 CUDA-core kernels (the headline); tf32x3: 3xTF32 "
                         "tensor-core variant, reported separately")
    ap.add_argument("--alpha", type=float, default=1.0, help="C = alpha*A.B + beta*C")
    ap.add_argument("--beta", type=float, default=0.0)
    ap.add_argument("--trans", choices=["NN", "NT", "TN", "TT"], default="NN",
                    help="operands stored transposed (T) and multiplied as op(A).op(B)")
    ap.add_argument("--tile-sweep", action="store_true",
                    help="one line per tile-table entry that can serve the workload "
                         "(forced entry, no e2e or CPU baseline)")
    ap.add_argument("--no-variants", action="store_true",
                    help="leave the 3xTF32 variant out of the default line")
    ap.add_argument("--link", action="store_true",
                    help="host<->device copy bandwidth from pinned memory (what bounds "
                         "the e2e lines); no product")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.link:
        bench_link(args)
        return 0

    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
    ctx = (rank, world, local)
    names = sorted(WORKLOADS, key=lambda n: WORKLOADS[n].flops) if args.sweep else [w.name]
    if args.tile_sweep:
        import dense_fp32_gemm_09_gb300 as sg
        for kid in range(len(sg.kernel_table())):
            args.kernel_id = kid
            line = bench_gpu(args, w, ctx)
            if line is not None and rank == 0:
                print(json.dumps(line), flush=True)
        names = []
    for name in names:
        line = (bench_tf32x3 if args.path == "tf32x3" else bench_gpu)(args, WORKLOADS[name], ctx)
        if line is not None and rank == 0:
            if not args.no_cpu_baseline and world == 1 and not args.sweep:
                A, B = make_inputs(WORKLOADS[name])
                cb = oracle_rate(WORKLOADS[name], A, B, target_s=12.0)
                cb.pop("seconds", None)
                line["cpu_baseline"] = cb
            # (one rank only: the variant's timing uses no collective)
            if args.path == "ffma" and not args.sweep and args.trans == "NN" and \
                    args.alpha == 1.0 and args.beta == 0.0 and not args.no_variants and \
                    world == 1:
                line["variants"] = {"tf32x3": tf32x3_summary(args, WORKLOADS[name], ctx)}
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
