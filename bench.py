#!/usr/bin/env python3
"""Benchmark of the cluster GEMM on GB300: GEMM TFLOP/s, % of dense-BF16 peak,
and L2->SM operand bytes against unicast.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline]

One step is one gemm_run over the workload (default: GEMM 4096^3, bf16 in,
bf16 out, 2x1 cluster multicasting A and B). Inputs are seeded synthetic
matrices resident in HBM. Inputs that fit in L2 are rotated through copies
that together exceed twice L2 (so no step finds its operands in L2), or for
tiny problems L2 is flushed (a 512 MB write, then a read) before every step
and each step is timed alone with CUDA events on the launching stream;
otherwise the K steps run back to back between one pair of events.
Prints one JSON line (rank 0).

--impl reference times the CPU oracle (fp64 triple loop, OpenMP) on a bounded
sample of the same workload: the method's plain definition, not a GPU program.
Under torchrun every rank runs the workload on its own GPU (weak scaling, no
collective on the data path; cluster multicast is turned off when more than
one GPU takes part).
"""
from __future__ import annotations

import argparse
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

from dense_gemm_cluster_gb300 import inputs  # noqa: E402
from dense_gemm_cluster_gb300.workloads import (ATTENTION_WORKLOADS, DEFAULT, WORKLOADS,  # noqa: E402
                                                AttentionWorkload, Workload)

METRIC = "GEMM TFLOP/s at 1 GB300 and % of dense-BF16 peak; L2→SM bytes vs unicast"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 129 << 20          # GB300 L2 (126 MiB usable); inputs above this need no flush
MAX_ROTATION = 8              # most copies of a workload's buffers the bench rotates through instead of a flush
KERNEL_SOURCES = ["dense_gemm_cluster_gb300/csrc/gemm_kernel.cuh", "dense_gemm_cluster_gb300/csrc/ptx.cuh",
                  "dense_gemm_cluster_gb300/csrc/gemm_host.cu"]
ATTN_KERNEL_SOURCES = ["dense_gemm_cluster_gb300/csrc/attention.cu", "dense_gemm_cluster_gb300/csrc/ptx.cuh"]


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def aggregate(dist, elapsed_s: float, units: float, device=None):
    """(max elapsed over ranks, sum of units over ranks): the whole-job clock and work."""
    if dist is None:
        return elapsed_s, units
    import torch
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- peaks, clocks, profiles
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


RATED_FLOP_PER_CLK_PER_SM = 8192     # dense bf16 tcgen05 rate of one SM
RATED_SM_MHZ = 2070                  # GB300 maximum SM clock


def rated_tensor_peak(device, clocks) -> dict:
    """The rated dense-bf16 rate: SMs x 8192 FLOP per clock x the maximum SM clock (the
    sampled clocks.max.sm when nvidia-smi answered, else 2070 MHz)."""
    import torch
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    mhz = clocks.get("sm_max_mhz") or RATED_SM_MHZ
    return {"tflops": sms * RATED_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12, "sms": sms, "sm_mhz": mhz}


def in_kernel_clock(probe: dict, launches: int) -> dict:
    """The clock probe's reading of a region: the mean SM clock over the CTAs' lives (SM
    cycle counter over the global nanosecond timer) and the CTAs each launch ran."""
    if not probe or not probe.get("ns"):
        return {"sm_ghz_in_kernel": None}
    return {"sm_ghz_in_kernel": probe["cycles"] / probe["ns"],
            "ctas_per_launch": probe["ctas"] / launches if launches else None,
            "in_kernel_source": "clock64 / %globaltimer over every CTA of every launch (gemm_read_clock)"}


SMEM_PORT_BYTES_PER_CLK = 128   # shared-memory bytes an SM moves per clock (reads and writes together)


def smem_port_bound(block_m: int, block_n: int, cta_group: int) -> dict:
    """Shared-memory traffic per tensor clock of one CTA and the tensor utilisation the port
    allows: per K = 16 step a CTA's MMA reads its A rows (block_m x 16) and its share of B's
    columns (block_n / cta_group x 16) from shared memory, and TMA has written the same bytes
    there; the step takes 2 * block_m * block_n * 16 / 8192 tensor clocks."""
    step_bytes = 2 * 2 * 16 * (block_m + block_n // cta_group)     # (write + read) x bf16 x K16
    clks = 2 * block_m * block_n * 16 / RATED_FLOP_PER_CLK_PER_SM
    per_clk = step_bytes / clks
    return {"bytes_per_tensor_clk": per_clk, "port_bytes_per_clk": SMEM_PORT_BYTES_PER_CLK,
            "tensor_util_bound": min(1.0, SMEM_PORT_BYTES_PER_CLK / per_clk)}


def tensor_peak_at_kernel_clock(tflops: float, clocks: dict, sms: int) -> dict:
    """The dense-bf16 tensor peak at the clock the kernel ran at, for all SMs and for the
    SMs its CTAs occupied (one CTA per SM), and the achieved rate's fraction of each."""
    ghz = (clocks or {}).get("sm_ghz_in_kernel")
    if not ghz:
        return None
    used = (clocks.get("ctas_per_launch") or sms)
    peak_all = sms * RATED_FLOP_PER_CLK_PER_SM * ghz / 1e3
    peak_used = used * RATED_FLOP_PER_CLK_PER_SM * ghz / 1e3
    return {"sm_ghz": ghz, "peak_all_sms": peak_all, "frac_all_sms": tflops / peak_all,
            "sms_used": used, "peak_sms_used": peak_used, "frac_sms_used": tflops / peak_used,
            "unit": "TFLOP/s"}


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, sources=KERNEL_SOURCES):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            recs = json.load(f)
    except (OSError, ValueError):
        return None
    rec = recs.get(workload)
    if not rec or rec.get("kernel_sha") != kernel_source_hash(sources):
        return None
    return rec


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)            # first sample lands before the timed region starts
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.file.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "samples": len(sm), "reasons": sorted(reasons)}


class NvmlClocks:
    """SM clock, power and clock-event reasons of this process's GPU, polled every
    `period_s` on a background thread through NVML's read-only queries (ctypes on
    libnvidia-ml; nothing is set). Samples carry a wall-clock time, so a summary can
    be taken over any window (the timed steps, the sustained region)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, device, period_s: float = 0.0005):
        import ctypes
        import threading
        self.period_s = period_s
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        self._thread = None
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            self.ok = self._find_handle(device)
            self._u = ctypes.c_uint()
            self._ull = ctypes.c_ulonglong()
            self._reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1,
                                                                                 ctypes.byref(mx)) == 0 else None
        except (OSError, AttributeError):
            self.ok = False

    def _find_handle(self, device) -> bool:
        import ctypes
        import torch
        props = torch.cuda.get_device_properties(device)
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            u = str(uuid)
            for cand in (u, "GPU-" + u):
                if self.lib.nvmlDeviceGetHandleByUUID(cand.encode(), ctypes.byref(self.handle)) == 0:
                    return True
        if hasattr(props, "pci_bus_id"):
            bus = f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
            if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.handle)) == 0:
                return True
        return False

    def _poll(self):
        import ctypes
        lib, h, u, ull = self.lib, self.handle, self._u, self._ull
        while not self._stop.is_set():
            t = time.perf_counter()
            mhz = float(u.value) if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(u)) == 0 else None
            mw = float(u.value) if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(u)) == 0 else None
            rs = int(ull.value) if self._reasons_fn(h, ctypes.byref(ull)) == 0 else 0
            if mhz is not None:
                self.samples.append((t, mhz, None if mw is None else mw / 1e3, rs))
            self._stop.wait(self.period_s)

    def __enter__(self):
        import threading
        if self.ok:
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self.ok:
            self.lib.nvmlShutdown()

    def summary(self, t0: float, t1: float) -> dict:
        rows = [r for r in self.samples if t0 <= r[0] <= t1]
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"], "samples": 0}
        sm = [r[1] for r in rows]
        pw = [r[2] for r in rows if r[2] is not None]
        bits = 0
        for r in rows:
            bits |= r[3]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_mhz_min": min(sm) if sm else None,
                "sm_mhz_max_seen": max(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "power_w_max": max(pw) if pw else None, "power_w_median": statistics.median(pw) if pw else None,
                "samples": len(sm), "period_ms": self.period_s * 1e3, "window_s": t1 - t0,
                "reasons": sorted(n for b, n in self.REASONS.items() if bits & b), "source": "nvml, in process"}


# ---------------------------------------------------------------- inputs on the device
class DeviceProblem:
    """The workload's operands, generated on the host from the seed and copied to HBM once."""

    def __init__(self, w: Workload, device, seed: int = 0):
        import numpy as np
        import torch
        self.w = w
        if w.batch > 1:
            A_log = inputs.bf16_matrix(w.batch * w.M, w.K, w.dist, seed + inputs.STREAM_A, w.scale)
            B_log = inputs.bf16_matrix(w.batch * w.N, w.K, w.dist, seed + inputs.STREAM_B, w.scale)
            assert w.layout_a == "row" and w.layout_b == "col" and w.layout_c == "row"
            self.A_host, self.lda, self.sA = A_log, w.K, w.M * w.K
            self.B_host, self.ldb, self.sB = B_log, w.K, w.N * w.K
            self.ldc, self.sC = w.N, w.M * w.N
        else:
            self.A_host, self.lda = inputs.store(inputs.bf16_matrix(w.M, w.K, w.dist, seed + inputs.STREAM_A,
                                                                    w.scale), w.layout_a)
            self.B_host, self.ldb = inputs.store(inputs.bf16_matrix(w.K, w.N, w.dist, seed + inputs.STREAM_B,
                                                                    w.scale), w.layout_b)
            self.sA = self.sB = self.sC = 0
            self.ldc = w.N if w.layout_c == "row" else w.M
        esc = 4 if w.out == "f32" else 2
        c_elems = (w.batch * w.M * w.N)
        if w.beta != 0.0:
            if w.out == "bf16":
                C_log = inputs.bf16_matrix(w.M, w.N, w.c_dist, seed + inputs.STREAM_C)
            else:
                C_log = inputs.f32_matrix(w.M, w.N, w.c_dist, seed + inputs.STREAM_C)
            self.C_host, self.ldc = inputs.store(C_log, w.layout_c)
        else:
            self.C_host = None
        self.A = torch.from_numpy(self.A_host.view(np.int16)).to(device)
        self.B = torch.from_numpy(self.B_host.view(np.int16)).to(device)
        cdt = torch.float32 if w.out == "f32" else torch.int16
        if self.C_host is not None:
            self.C_init = torch.from_numpy(self.C_host.view(np.int16) if w.out == "bf16" else self.C_host).to(device)
            self.C = self.C_init.clone()
        else:
            self.C_init = None
            self.C = torch.empty(c_elems, dtype=cdt, device=device)
        self.c_bytes = c_elems * esc

    def replica(self):
        """Another device copy of the operands and C (same values), for rotating through steps."""
        import copy
        r = copy.copy(self)
        r.A, r.B, r.C = self.A.clone(), self.B.clone(), self.C.clone()
        return r


def run_once(g, p: DeviceProblem, stream):
    w = p.w
    if w.batch > 1:
        g.run_strided_batched(w.M, w.N, w.K, p.A, p.lda, p.sA, p.B, p.ldb, p.sB, p.C, p.ldc, p.sC, w.batch,
                              w.alpha, w.beta, stream)
    else:
        g.run(w.M, w.N, w.K, p.A, p.lda, p.B, p.ldb, p.C, p.ldc, w.alpha, w.beta, stream)


# ---------------------------------------------------------------- CPU oracle sample
def oracle_rate(w: Workload, budget_s: float, seed: int = 0):
    """Times the CPU oracle on the first R output rows of (the first batch of) the workload.

    Returns (TFLOP/s, seconds, rows, threads). R is chosen from a short
    calibration run so the timed sample takes about budget_s seconds.
    """
    import oracle
    assert w.layout_a == "row"
    A_full = inputs.bf16_matrix(w.M, w.K, w.dist, seed + inputs.STREAM_A, w.scale)
    if w.batch > 1:
        B_buf = inputs.bf16_matrix(w.N, w.K, w.dist, seed + inputs.STREAM_B, w.scale)   # K rows = B col-major
        ldb, lb = w.K, "col"
    else:
        B_buf, ldb = inputs.store(inputs.bf16_matrix(w.K, w.N, w.dist, seed + inputs.STREAM_B, w.scale),
                                  w.layout_b)
        lb = w.layout_b
    C_in = None
    ldc = 0
    if w.beta != 0.0:
        C_log = (inputs.bf16_matrix(w.M, w.N, w.c_dist, seed + inputs.STREAM_C) if w.out == "bf16"
                 else inputs.f32_matrix(w.M, w.N, w.c_dist, seed + inputs.STREAM_C))
        C_in, ldc = inputs.store(C_log, "row")

    def timed(rows):
        A = A_full[:rows]
        Cs = C_in[:rows] if C_in is not None else None
        t0 = time.perf_counter()
        oracle.gemm(rows, w.N, w.K, A, w.K, "row", B_buf, ldb, lb, w.alpha, w.beta, Cs, ldc, "row")
        return time.perf_counter() - t0

    per_row_flops = 2.0 * w.N * w.K
    r0 = max(1, min(w.M, int(1e9 / per_row_flops)))
    t0 = timed(r0)
    rate = r0 * per_row_flops / max(t0, 1e-6)
    rows = max(1, min(w.M, int(rate * budget_s / per_row_flops)))
    t = timed(rows)
    return rows * per_row_flops / t / 1e12, t, rows, oracle.num_threads()


def single_core_oracle(name: str) -> dict:
    """The oracle on one host core over a whole small workload (the 256^3 GEMM is quoted as
    "CPU oracle in seconds"): a child process with OMP_NUM_THREADS=1, best of 3 runs."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-core", name], env=env,
                             capture_output=True, text=True, timeout=300, check=True).stdout
        return json.loads(out.strip().splitlines()[-1])
    except (subprocess.SubprocessError, OSError, ValueError, IndexError) as e:
        return {"workload": name, "error": str(e)[:200]}


def oracle_one_core_main(name: str) -> int:
    import oracle
    oracle.build()
    w = WORKLOADS[name]
    assert w.batch == 1 and w.beta == 0.0
    A, lda = inputs.store(inputs.bf16_matrix(w.M, w.K, w.dist, inputs.STREAM_A, w.scale), w.layout_a)
    B, ldb = inputs.store(inputs.bf16_matrix(w.K, w.N, w.dist, inputs.STREAM_B, w.scale), w.layout_b)
    times = []
    for _ in range(3):
        t0 = time.perf_counter()
        oracle.gemm(w.M, w.N, w.K, A, lda, w.layout_a, B, ldb, w.layout_b)
        times.append(time.perf_counter() - t0)
    t = min(times)
    print(json.dumps({"workload": name, "seconds": t, "gflops": w.flops / t / 1e9, "threads": oracle.num_threads(),
                      "runs": 3, "what": "whole product, fp64 oracle, best of 3"}))
    return 0


# ---------------------------------------------------------------- arms
def bench_reference(args, w: Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    per_step = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    # calibrate the per-step sample once (untimed)
    _, _, rows, threads = oracle_rate(w, per_step)
    A_full = inputs.bf16_matrix(rows, w.K, w.dist, inputs.STREAM_A, w.scale)
    if w.batch > 1:
        B_buf, ldb, lb = inputs.bf16_matrix(w.N, w.K, w.dist, inputs.STREAM_B, w.scale), w.K, "col"
    else:
        B_buf, ldb = inputs.store(inputs.bf16_matrix(w.K, w.N, w.dist, inputs.STREAM_B, w.scale), w.layout_b)
        lb = w.layout_b
    C_in, ldc = None, 0
    if w.beta != 0.0:
        C_log = (inputs.bf16_matrix(rows, w.N, w.c_dist, inputs.STREAM_C) if w.out == "bf16"
                 else inputs.f32_matrix(rows, w.N, w.c_dist, inputs.STREAM_C))
        C_in, ldc = inputs.store(C_log, "row")
    for _ in range(args.warmup):
        oracle.gemm(rows, w.N, w.K, A_full, w.K, "row", B_buf, ldb, lb, w.alpha, w.beta, C_in, ldc, "row")
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.gemm(rows, w.N, w.K, A_full, w.K, "row", B_buf, ldb, lb, w.alpha, w.beta, C_in, ldc, "row")
        times.append(time.perf_counter() - t0)
    total = sum(times)
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / total / 1e12
    sample = f"rows 0..{rows - 1} of C ({rows}x{w.N}x{w.K}) per step, of the {w.M}x{w.N}x{w.K}" + \
             (f" x{w.batch} batch" if w.batch > 1 else "") + " workload"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "batch": w.batch,
                   "description": "fp64 CPU oracle (plain triple loop, OpenMP over rows): " + w.description},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_to_sm_report(w: Workload, plan, uni_plan, traffic_rec) -> dict:
    """The multicast evidence: L2 -> SM operand bytes of this launch against the same output
    computed with unicast tiles, analytic (the planner's accounting) and measured (ncu
    lts__t_sectors_srcunit_tex_op_read of both launches, each record taken on the current
    kernel sources; null when either record is missing or stale)."""
    from dense_gemm_cluster_gb300.workloads import UNICAST_TWIN
    twin = UNICAST_TWIN.get(w.name)
    twin_rec = recorded_traffic(twin) if twin else None
    mine = traffic_rec.get("lts_bytes") if traffic_rec else None
    theirs = twin_rec.get("lts_bytes") if twin_rec else None
    return {"analytic": plan.l2_to_sm_operand_bytes,
            "analytic_unicast": uni_plan.l2_to_sm_operand_bytes,
            "reduction_vs_unicast": uni_plan.l2_to_sm_operand_bytes / max(1, plan.l2_to_sm_operand_bytes),
            "measured": mine, "unicast_workload": twin, "measured_unicast": theirs,
            "reduction_measured": (theirs / mine) if (mine and theirs) else None,
            "counter": "ncu lts__t_sectors_srcunit_tex_op_read.sum x 32 B, one launch each (profiles/ncu_traffic.json)"}


def sustained_region(g, copies, stream, steps, region_s, seconds, device, flops_per_step):
    """Repeats the K-step region back to back for about `seconds`, each region between
    its own pair of events on the launching stream. Returns (wall start, wall end,
    summary of the per-region rates)."""
    import math
    import torch
    n = max(2, min(20000, math.ceil(seconds / max(region_s, 1e-6))))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    launches0 = g.launches
    t0 = time.perf_counter()
    for r in range(n):
        evs[r][0].record(stream)
        for i in range(steps):
            run_once(g, copies[i % len(copies)], stream)
        evs[r][1].record(stream)
    torch.cuda.synchronize(device)
    t1 = time.perf_counter()
    ms = [a.elapsed_time(b) for a, b in evs]
    tf = sorted(flops_per_step * steps / (m / 1e3) / 1e12 for m in ms)
    q = lambda f: tf[min(len(tf) - 1, int(f * len(tf)))]
    return t0, t1, {"regions": n, "steps_per_region": steps, "launches": g.launches - launches0,
                    "seconds_gpu": sum(ms) / 1e3, "tflops_median": statistics.median(tf), "tflops_min": tf[0],
                    "tflops_p10": q(0.1), "tflops_p90": q(0.9), "tflops_max": tf[-1],
                    "note": "after the reported steps, not part of value"}


def bench_ours(args, w: Workload):
    import torch
    world, rank, local = dist_env()
    dist = init_dist(world, "nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from dense_gemm_cluster_gb300 import gemm

    opts = dict(w.options)
    if world > 1:
        # Cluster multicast stays off when several GPUs take part. Without it a pair kernel
        # gains nothing from clusters of more than one pair (4-CTA clusters only leave SMs
        # idle: 36 fit on 152 SMs), so the pairs run in 2-CTA clusters.
        opts["mode"] = "unicast"
        if opts.get("cta_group", 1) == 2 and opts.get("cluster_m", 1) > 2 and opts.get("cluster_n", 1) == 1:
            opts["cluster_m"] = 2
    # The clock probe adds each CTA's SM cycles and nanoseconds to handle-owned counters
    # (two timer reads and three atomics per CTA), read between the regions below.
    g = gemm.Gemm(local, layout_a=w.layout_a, layout_b=w.layout_b, layout_c=w.layout_c, out_type=w.out,
                  clock_probe=1, **opts)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    s, plan = gemm.gemm_plan(g.options, w.M, w.N, w.K, w.batch, sms)
    g.check(s)
    uni_opts = gemm.make_options(layout_a=w.layout_a, layout_b=w.layout_b, layout_c=w.layout_c, out_type=w.out,
                                 block_n=plan.block_n)
    _, uni_plan = gemm.gemm_plan(uni_opts, w.M, w.N, w.K, w.batch, sms)

    p = DeviceProblem(w, device)
    stream = torch.cuda.current_stream(device)
    input_bytes = w.min_hbm_bytes()
    # Inputs that fit in L2 must not be served from it: steps rotate through enough
    # copies of the operands and C that the others' traffic between two uses of a
    # copy is more than twice L2; when that takes too many copies, L2 is flushed
    # before every step instead.
    copies = [p]
    needs_flush = False
    if input_bytes <= L2_BYTES:
        rot = -(-2 * L2_BYTES // input_bytes) + 1
        if rot <= MAX_ROTATION:
            copies += [p.replica() for _ in range(rot - 1)]
        else:
            needs_flush = True
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device) if needs_flush else None
    # A read after the write leaves L2 holding clean lines, so the timed kernel
    # does not pay for writing back the flush buffer.
    clean = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.float32, device=device) if needs_flush else None

    for i in range(max(3, args.warmup, len(copies))):
        run_once(g, copies[i % len(copies)], stream)
    g.check(g.query_status(stream))

    # With an L2 flush between steps each step is bracketed by its own events (the
    # flush stays outside the timed region); otherwise one pair of events brackets
    # the K back-to-back steps.
    n_ev = args.steps if needs_flush else 1
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    launches0 = g.launches
    g.read_clock(stream)                               # clears the probe: only timed launches count
    barrier(dist)
    torch.cuda.synchronize(device)
    nv = NvmlClocks(device)
    sustained = None
    with (nv if nv.ok else ClockSampler(local)) as clk:
        wall0 = time.perf_counter()
        if not needs_flush:
            starts[0].record(stream)
        for i in range(args.steps):
            if needs_flush:
                flush.fill_(float(i))                  # evicts the operands from L2
                clean.sum()
                starts[i].record(stream)
            run_once(g, copies[i % len(copies)], stream)
            if needs_flush:
                ends[i].record(stream)
        if not needs_flush:
            ends[0].record(stream)
        torch.cuda.synchronize(device)
        wall1 = time.perf_counter()
        wall = wall1 - wall0
        kclk = g.read_clock(stream)                    # after the timed region, before the sustained one
        barrier(dist)
        launches = g.launches - launches0
        step_ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
        local_s = sum(step_ms) / 1e3
        if args.sustain_s > 0 and not needs_flush:
            # After the reported steps: the same K-step region repeated back to back for
            # about sustain_s, each region between its own events, to see the rate and the
            # clocks under sustained load (power cap) beside the reported burst.
            sustained = sustained_region(g, copies, stream, args.steps, local_s, args.sustain_s, device, w.flops)
            kclk_sus = g.read_clock(stream)
    g.check(g.query_status(stream))
    elapsed, units = aggregate(dist, local_s, float(w.flops) * args.steps, device)
    value = units / elapsed / 1e12
    ms_per_step = 1e3 * elapsed / args.steps

    peaks, peaks_kind = load_peaks()
    tensor_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    avg_launch_s = local_s / args.steps
    traffic_rec = recorded_traffic(w.name)
    intensity = w.flops / w.min_hbm_bytes()
    ridge = tensor_peak * 1e12 / (hbm_peak * 1e9)
    if intensity >= ridge:
        achieved = w.flops / avg_launch_s / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tensor_peak, "unit": "TFLOP/s",
                    "frac": achieved / tensor_peak, "peak_source": f"bf16_tflops (burst) of {peaks_kind}",
                    "algorithmic_flops_per_launch": w.flops}
    else:
        achieved = w.min_hbm_bytes() / avg_launch_s / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "peak_source": f"hbm_gbs (copy) of {peaks_kind}",
                    "algorithmic_bytes_per_launch": w.min_hbm_bytes()}
    clocks = clk.summary(wall0, wall1) if nv.ok else clk.summary()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    clocks.update(in_kernel_clock(kclk, launches))
    if sustained is not None:
        t0, t1, sus = sustained
        sus["clocks"] = nv.summary(t0, t1) if nv.ok else {}
        sus["clocks"].update(in_kernel_clock(kclk_sus, sus["launches"]))
        if roofline["bound"] == "tensor":
            sus_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
            sus.update({"frac_of_sustained_peak": sus["tflops_median"] / sus_peak, "sustained_peak": sus_peak,
                        "frac_of_burst_peak": sus["tflops_median"] / tensor_peak,
                        "peak_source": f"bf16_tflops_sustained and bf16_tflops of {peaks_kind}"})
        else:
            gbs = sus["tflops_median"] * 1e12 / w.flops * w.min_hbm_bytes() / 1e9
            sus.update({"hbm_gbs_median": gbs, "frac_of_hbm_peak": gbs / hbm_peak,
                        "peak_source": f"hbm_gbs of {peaks_kind}"})
        roofline["sustained"] = sus
    if roofline["bound"] == "tensor":
        sus_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        roofline.update({"sustained_peak": sus_peak, "frac_of_sustained_peak": achieved / sus_peak})
    if roofline["bound"] == "tensor":
        roofline["at_kernel_clock"] = tensor_peak_at_kernel_clock(achieved, clocks, sms)
        if roofline["at_kernel_clock"]:
            roofline["at_kernel_clock"]["smem_port"] = smem_port_bound(plan.block_m, plan.block_n, plan.cta_group)
        if sustained is not None:
            roofline["sustained"]["at_kernel_clock"] = tensor_peak_at_kernel_clock(
                roofline["sustained"]["tflops_median"], roofline["sustained"]["clocks"], sms)
        rated = rated_tensor_peak(device, clocks)
        roofline.update({"rated_peak": rated["tflops"], "frac_of_rated": achieved / rated["tflops"],
                         "rated_peak_source": f"{rated['sms']} SMs x {RATED_FLOP_PER_CLK_PER_SM} FLOP/clk x "
                                              f"{rated['sm_mhz']:.0f} MHz"})
    roofline.update({"traffic": traffic_rec["dram_bytes"] if traffic_rec else None,
                     "arithmetic_intensity": intensity, "ridge": ridge,
                     "tflops": w.flops / avg_launch_s / 1e12,
                     "hbm_gbs_at_min_bytes": w.min_hbm_bytes() / avg_launch_s / 1e9})

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "batch": w.batch, "out": w.out,
                   "layouts": f"A {w.layout_a}, B {w.layout_b}, C {w.layout_c}", "alpha": w.alpha,
                   "beta": w.beta, "mode": opts, "cta_group": plan.cta_group, "block": [plan.block_m, plan.block_n,
                                                                                        plan.block_k],
                   "stages": plan.stages, "cluster": [plan.cluster_m, plan.cluster_n],
                   "l2": (f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MB write, then a "
                          f"{L2_FLUSH_BYTES >> 21} MB read), each step between its own pair of events"
                          if needs_flush else
                          (f"no flush: the steps rotate through {len(copies)} copies of the operands and C "
                           f"({(len(copies) * input_bytes) >> 20} MB, more than twice L2 between two uses of a copy); "
                           f"the K steps run back to back between one pair of events" if len(copies) > 1 else
                           f"no flush: the inputs ({input_bytes >> 20} MB) are larger than L2; the K steps run "
                           f"back to back between one pair of events")),
                   "description": w.description},
        "roofline": roofline,
        "l2_to_sm_operand_bytes": l2_to_sm_report(w, plan, uni_plan, traffic_rec),
        "gpu_launches": launches,
        "wall_s_timed_region": wall,
        "clocks": clocks,
    }

    if not args.no_e2e:
        line["e2e"] = e2e_through_host_api(g, p, args, device, stream, dist)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, secs, rows, threads = oracle_rate(w, args.cpu_budget)
        line["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"rows 0..{rows - 1} of C ({rows}x{w.N}x{w.K}"
                                          f"{', first batch' if w.batch > 1 else ''}) in {secs:.1f} s",
                                "single_core_256": single_core_oracle("gemm256_f32_mcastB")}
    g.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def e2e_through_host_api(g, p: DeviceProblem, args, device, stream, dist):
    """The same metric through gemm_run_host (gemm_run_strided_batched_host for a batch):
    pinned host inputs copied in and C copied out every step."""
    import numpy as np
    import torch
    w = p.w
    A_h = torch.from_numpy(p.A_host.view(np.int16)).pin_memory()
    B_h = torch.from_numpy(p.B_host.view(np.int16)).pin_memory()
    esc = 4 if w.out == "f32" else 2
    if p.C_host is not None:
        C_h = torch.from_numpy(p.C_host.view(np.int16) if w.out == "bf16" else p.C_host.copy()).pin_memory()
    else:
        C_h = torch.empty(p.c_bytes // esc, dtype=torch.float32 if w.out == "f32" else torch.int16, pin_memory=True)
    steps = max(1, min(args.steps, args.e2e_steps))
    if w.batch > 1:
        api = "gemm_run_strided_batched_host (C ABI, host buffers)"

        def step():
            g.run_strided_batched_host(w.M, w.N, w.K, A_h, p.lda, p.sA, B_h, p.ldb, p.sB, C_h, p.ldc, p.sC, w.batch,
                                       w.alpha, w.beta, stream)
    else:
        api = "gemm_run_host (C ABI, host buffers)"

        def step():
            g.run_host(w.M, w.N, w.K, A_h, p.lda, B_h, p.ldb, C_h, p.ldc, w.alpha, w.beta, stream)
    for _ in range(2):
        step()
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    local = time.perf_counter() - t0
    elapsed, units = aggregate(dist, local, float(w.flops) * steps, device)
    h2d = A_h.numel() * 2 + B_h.numel() * 2 + (C_h.numel() * esc if w.beta != 0.0 else 0)
    return {"value": units / elapsed / 1e12, "unit": "TFLOP/s", "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(C_h.numel() * esc),
            "ms_per_step": 1e3 * elapsed / steps, "api": api}


# ---------------------------------------------------------------- fused attention workloads
ATTN_METRIC = "attention forward TFLOP/s at 1 GB300 and % of dense-BF16 peak"


def attn_host_inputs(w: AttentionWorkload, seed: int = 0):
    """Q, K, V as bf16 bits, shaped (batch, rows, d); streams 0, 1, 2 of the seed."""
    Q = inputs.bf16_matrix(w.batch * w.sq, w.d, w.dist, seed + inputs.STREAM_A).reshape(w.batch, w.sq, w.d)
    K = inputs.bf16_matrix(w.batch * w.sk, w.d, w.dist, seed + inputs.STREAM_B).reshape(w.batch, w.sk, w.d)
    V = inputs.bf16_matrix(w.batch * w.sk, w.d, w.dist, seed + inputs.STREAM_C).reshape(w.batch, w.sk, w.d)
    return Q, K, V


def attn_oracle_sample(w: AttentionWorkload, budget_s: float, seed: int = 0):
    """Sizes and times an oracle sample: the first H heads, every query row against every key.

    Returns (callable running the sample, TFLOP/s of one run, seconds, heads, threads).
    """
    import oracle
    per_head = 4.0 * w.pairs * w.d

    def head_inputs(h):
        Q = inputs.bf16_matrix(h * w.sq, w.d, w.dist, seed + inputs.STREAM_A).reshape(h, w.sq, w.d)
        K = inputs.bf16_matrix(h * w.sk, w.d, w.dist, seed + inputs.STREAM_B).reshape(h, w.sk, w.d)
        V = inputs.bf16_matrix(h * w.sk, w.d, w.dist, seed + inputs.STREAM_C).reshape(h, w.sk, w.d)
        return Q, K, V

    Q, K, V = head_inputs(1)
    t0 = time.perf_counter()
    oracle.attention_forward(Q, K, V, causal=w.causal)
    rate = per_head / max(time.perf_counter() - t0, 1e-6)
    heads = max(1, min(w.batch, int(rate * budget_s / per_head)))
    Q, K, V = head_inputs(heads)
    t0 = time.perf_counter()
    oracle.attention_forward(Q, K, V, causal=w.causal)
    secs = time.perf_counter() - t0
    return (lambda: oracle.attention_forward(Q, K, V, causal=w.causal)), heads * per_head / secs / 1e12, secs, heads, \
        oracle.num_threads()


def bench_attention_reference(args, w: AttentionWorkload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    per_step = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    run, _, _, heads, threads = attn_oracle_sample(w, per_step)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = 4.0 * heads * w.pairs * w.d * args.steps / total / 1e12
    sample = f"heads 0..{heads - 1} (all {w.sq} query rows against all {w.sk} keys) per step, of the " \
             f"{w.batch}-head workload"
    line = {
        "impl": "reference", "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "sq": w.sq, "sk": w.sk, "d": w.d, "causal": w.causal,
                   "description": "fp64 CPU oracle (softmax of the fp64 scores, OpenMP over rows): " + w.description},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_attention_ours(args, w: AttentionWorkload):
    import numpy as np
    import torch
    world, rank, local = dist_env()
    dist = init_dist(world, "nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from dense_gemm_cluster_gb300 import gemm
    cluster = w.cluster if world == 1 else 1          # multicast stays off when several GPUs take part
    cta_group = w.cta_group if world == 1 else 1
    Qh, Kh, Vh = attn_host_inputs(w)
    Q = torch.from_numpy(Qh.reshape(-1).view(np.int16)).to(device)
    K = torch.from_numpy(Kh.reshape(-1).view(np.int16)).to(device)
    V = torch.from_numpy(Vh.reshape(-1).view(np.int16)).to(device)
    odt = torch.float32 if w.out == "f32" else torch.int16
    O = torch.empty(w.batch * w.sq * w.d, dtype=odt, device=device)
    lse = torch.empty(w.batch * w.sq, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    out_f32 = 1 if w.out == "f32" else 0
    launches = 0

    def run():
        nonlocal launches
        s = gemm.attention_forward_run(Q, K, V, O, lse, w.batch, w.sq, w.sk, w.d, 0.0, out_f32, cluster,
                                       cta_group=cta_group, causal=w.causal, stream=stream)
        if s != gemm.GEMM_OK:
            raise RuntimeError(f"attention_forward_run: status {s}")
        launches += 1

    for _ in range(max(3, args.warmup)):
        run()
    if gemm.attention_forward_query_status(stream) != gemm.GEMM_OK:
        raise RuntimeError("attention kernel reported a device timeout")
    input_bytes = w.min_hbm_bytes()
    # The inputs are larger than L2: one pair of events brackets the K back-to-back steps.
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = launches
    barrier(dist)
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clk:
        wall0 = time.perf_counter()
        start.record(stream)
        for i in range(args.steps):
            run()
        end.record(stream)
        torch.cuda.synchronize(device)
        wall = time.perf_counter() - wall0
    barrier(dist)
    if gemm.attention_forward_query_status(stream) != gemm.GEMM_OK:
        raise RuntimeError("attention kernel reported a device timeout")
    local_s = start.elapsed_time(end) / 1e3
    elapsed, units = aggregate(dist, local_s, float(w.flops) * args.steps, device)
    peaks, peaks_kind = load_peaks()
    tensor_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    avg_launch_s = local_s / args.steps
    achieved = w.flops / avg_launch_s / 1e12
    traffic_rec = recorded_traffic(w.name, ATTN_KERNEL_SOURCES)
    clocks = clk.summary()
    rated = rated_tensor_peak(device, clocks)
    line = {
        "metric": ATTN_METRIC, "value": units / elapsed / 1e12, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "sq": w.sq, "sk": w.sk, "d": w.d, "out": w.out,
                   "cluster": cluster, "cta_group": cta_group, "causal": w.causal,
                   "l2": f"no flush: the inputs ({input_bytes >> 20} MB) are larger than L2; the K steps "
                         f"run back to back between one pair of events",
                   "description": w.description},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tensor_peak, "unit": "TFLOP/s",
                     "frac": achieved / tensor_peak, "peak_source": f"bf16_tflops (burst) of {peaks_kind}",
                     "algorithmic_flops_per_launch": w.flops,
                     "traffic": traffic_rec["dram_bytes"] if traffic_rec else None,
                     "arithmetic_intensity": w.flops / w.min_hbm_bytes(),
                     "ridge": tensor_peak * 1e12 / (hbm_peak * 1e9),
                     "rated_peak": rated["tflops"], "frac_of_rated": achieved / rated["tflops"],
                     "rated_peak_source": f"{rated['sms']} SMs x {RATED_FLOP_PER_CLK_PER_SM} FLOP/clk x "
                                          f"{rated['sm_mhz']:.0f} MHz"},
        "gpu_launches": launches - launches0,
        "wall_s_timed_region": wall,
        "clocks": clocks,
    }
    if not args.no_e2e:
        line["e2e"] = attn_e2e(w, args, device, stream, dist, cluster, cta_group, (Qh, Kh, Vh))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        _, rate, secs, heads, threads = attn_oracle_sample(w, args.cpu_budget)
        line["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"heads 0..{heads - 1} of {w.batch} (all rows and keys) in {secs:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def attn_e2e(w, args, device, stream, dist, cluster, cta_group, host_in):
    """The same metric through attention_forward_run_host: Q, K, V in from pinned host
    memory and O, lse back, every step (the call pipelines the copies over parts of the heads)."""
    import numpy as np
    import torch
    from dense_gemm_cluster_gb300 import gemm
    Qp, Kp, Vp = [torch.from_numpy(a.reshape(-1).view(np.int16)).pin_memory() for a in host_in]
    odt = torch.float32 if w.out == "f32" else torch.int16
    out_f32 = 1 if w.out == "f32" else 0
    O_h = torch.empty(w.batch * w.sq * w.d, dtype=odt).pin_memory()
    lse_h = torch.empty(w.batch * w.sq, dtype=torch.float32).pin_memory()
    ws_bytes = gemm.attention_forward_host_workspace_bytes(w.batch, w.sq, w.sk, w.d, out_f32)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    steps = max(1, min(args.steps, args.e2e_steps))

    def step():
        s = gemm.attention_forward_run_host(Qp, Kp, Vp, O_h, lse_h, w.batch, w.sq, w.sk, w.d, ws, ws_bytes, 0.0,
                                            out_f32, cluster, cta_group, causal=w.causal, stream=stream)
        if s != gemm.GEMM_OK:
            raise RuntimeError(f"attention_forward_run_host: status {s}")

    for _ in range(2):
        step()
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    local = time.perf_counter() - t0
    elapsed, units = aggregate(dist, local, float(w.flops) * steps, device)
    h2d = int((Qp.numel() + Kp.numel() + Vp.numel()) * 2)
    d2h = int(O_h.numel() * O_h.element_size() + lse_h.numel() * 4)
    del ws
    return {"value": units / elapsed / 1e12, "unit": "TFLOP/s", "steps": steps, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * elapsed / steps,
            "api": "attention_forward_run_host (C ABI, host buffers)"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(ATTENTION_WORKLOADS), default=DEFAULT)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back repeats of the timed region after it (rate and clocks under "
                         "sustained load; 0 = none)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch count of a batched workload (smaller profiling captures)")
    ap.add_argument("--oracle-one-core", metavar="WORKLOAD", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.oracle_one_core:
        return oracle_one_core_main(args.oracle_one_core)
    if args.warmup < 3:
        args.warmup = 3
    if args.workload in ATTENTION_WORKLOADS:
        w = ATTENTION_WORKLOADS[args.workload]
        if args.batch:
            import dataclasses
            w = dataclasses.replace(w, batch=args.batch, name=f"{w.name}[batch={args.batch}]")
        if args.impl == "reference":
            return bench_attention_reference(args, w)
        return bench_attention_ours(args, w)
    w = WORKLOADS[args.workload]
    if args.batch:
        import dataclasses
        w = dataclasses.replace(w, batch=args.batch, name=f"{w.name}[batch={args.batch}]")
    if args.impl == "reference":
        return bench_reference(args, w)
    return bench_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
