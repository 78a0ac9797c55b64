"""Benchmark of the packed-Trellis decode-and-multiply on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--entry gemm|decode|gateup|packed] [--rows M]
                    [--bits k] [--window L] [--no-per-config]

One step = one fused decode-and-multiply call (trellis_gemm: code fetch,
window, hash, quotient, scale/bf16 round, the product and the bf16 store) on
the headline workload, the largest of the quantised-linear shapes: M=64
activation rows, K=5120, N=17408, k=4 bits, L=12, T=256 (tensor cores),
seeded synthetic inputs.  Metric: us/call and packed-weight GB/s (code bytes
per second, whole job) with the kernel's roofline fraction.  The same JSON
line carries `per_config`: every quantised-linear workload (M = 5, 8, 15, 1,
64) and the dense decode, each timed in its own region of the same process,
each with its roofline fraction, clocks and the oracle's CPU rate on all host
cores and on one pinned core.

Timing: W warm-up steps, then K steps bracketed by a barrier and
torch.cuda.synchronize(), CUDA events on the launching stream around the K
back-to-back calls, max over ranks.  Between steps the code buffers rotate
through enough independent copies that the set exceeds twice the L2, so every
call streams its codes from HBM.  GPU clocks are sampled with nvidia-smi during
each timed region.  Multi-GPU runs (torchrun) are independent replicas of the
workload, one per rank (weak scaling, no data-path collective).

--impl reference times the CPU oracle (test infrastructure) on the host cores
on a bounded sample of the same workload; it is a deliberately slow baseline.
"""
from __future__ import annotations

import argparse
import dataclasses
import concurrent.futures as cf
import ctypes
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# the largest of the quantised-linear workloads: 64 activation rows (tensor cores)
HEADLINE = "prefill_m64_k5120_n17408_k4"
METRIC = "trellis GEMM us/call & packed-weight GB/s (% of GB300 roofline)"
METRIC_DECODE = "trellis decode packed-weight GB/s"
METRIC_GATEUP = "trellis gate/up GEMM packed-weight GB/s"
METRIC_PACKED = "trellis token-packed GEMM packed-weight GB/s"
DECODE_OPS_PER_WEIGHT = 10        # algorithmic integer/fp32 ops per decoded weight
ALU_LANES_PER_SM = 128            # 4 sub-partitions x 32 lanes, one op per lane per clock


# ----------------------------------------------------------------- helpers --
def max_over_ranks(vals, device="cpu"):
    """Element-wise maximum of `vals` over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def whole_job_gbs(world: int, bytes_per_rank: int, ms_per_step_max: float) -> float:
    """Weak scaling: every rank processes its own copy of the workload, the job
    takes as long as the slowest rank."""
    return world * bytes_per_rank / (ms_per_step_max * 1e-3) / 1e9


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


def _code_only(text: str) -> str:
    """Source text without comments, blank lines or indentation."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.strip() for line in text.splitlines() if line.strip())


# The sources each profiled kernel is built from (plus the shared headers).
KERNEL_SOURCES = {
    "decode": ["decode_kernel.cu"],
    "gemm_smallm": ["gemm_smallm_kernel.cuh", "gemm_smallm.cu", "gemm_smallm_k*.cu"],
    "gemm_tc": ["gemm_tc_kernel.cu"],
}
SHARED_SOURCES = ["trellis_device.cuh"]   # device code shared by all kernels (kernels.h is host plumbing)


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (comments ignored) of one kernel's sources and the
    shared headers: names the kernel an ncu capture in profiles/ was taken on."""
    csrc = os.path.join(ROOT, "trellis_quantized_weight_gb300", "csrc")
    files = set()
    for pat in KERNEL_SOURCES[kernel] + SHARED_SOURCES:
        files.update(glob.glob(os.path.join(csrc, pat)))
    h = hashlib.sha256()
    for f in sorted(files):
        with open(f, encoding="utf-8") as fh:
            h.update(os.path.basename(f).encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/, if the
    capture was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                key, val = line[2:].split(":", 1)
                vals[key.strip()] = val.strip().strip("`")
    if vals.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(self.period_ms / 1000.0 * 2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def to_dev(bits: np.ndarray, torch, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int32)).cuda()


# ---------------------------------------------------------------- our arm --
def path_dtype(entry: str, M: int) -> str:
    """The arithmetic the timed path computes in: the decode and the CUDA-core
    product (M <= 16) multiply bf16-valued operands in fp32; on the tensor
    cores (M > 16) the product is a bf16 MMA with fp32 accumulation."""
    return "bf16" if entry != "decode" and M > 16 else "f32"


def group_rows(M: int, groups: int) -> list[int]:
    """M rows split into `groups` sequences whose sizes differ by at most one."""
    if not 1 <= groups <= M:
        raise ValueError("--groups must be in 1..M")
    return [M // groups + (1 if g < M % groups else 0) for g in range(groups)]


def launches_per_step(entry: str, M: int, groups: int = 1) -> int:
    """Our kernels one step launches: on the tensor cores one launch per matrix
    for M <= 256, else one per 256-row chunk; otherwise one small-M launch; plus
    the gate/up activation, or the packing's gather and scatter."""
    n_mats = 2 if entry == "gateup" else 1
    if entry != "decode" and M > 16:
        n = n_mats * max(1, (M + 255) // 256)
    else:
        n = 1
    if entry == "gateup":
        n += 1
    if entry == "packed" and groups > 1:   # the gather and the scatter, per 64 groups
        n += 2 * ((groups + 63) // 64)
    return n


def roofline(wl, entry: str, kernel_ms: float, num_sms: int):
    """The roofline of one step's kernel(s): time = max(bytes / HBM peak,
    ops / ALU peak[, tensor FLOP / tensor peak]); achieved over peak for the
    binding bound."""
    peaks, peak_src = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz") or 2070.0)
    hbm_peak = float(peaks["hbm_gbs"])
    alu_peak = num_sms * ALU_LANES_PER_SM * sm_max * 1e6 / 1e12   # Tops/s
    tensor_peak = float(peaks.get("bf16_tflops") or 1900.0)
    n_mats = 2 if entry == "gateup" else 1
    t_kernel = kernel_ms * 1e-3
    flops = 0
    if entry in ("gemm", "gateup", "packed") and wl.M > 16:
        # tensor-core path: the decode runs on the ALUs, the M FMAs per weight
        # are a dense bf16 contraction on the tensor cores
        ops = n_mats * wl.weights * DECODE_OPS_PER_WEIGHT
        flops = n_mats * 2 * wl.M * wl.N * wl.K
        hbm_bytes = n_mats * (wl.code_bytes + wl.M * wl.N * 2) + wl.M * wl.K * 2
        kernel_name = "gemm_tc"
    elif entry in ("gemm", "gateup", "packed"):
        # gate/up: both matrices in one launch, plus the elementwise activation
        # (read 2 and write 1 bf16 [M, N]; bytes counted, no ALU ops)
        ops = n_mats * wl.weights * (DECODE_OPS_PER_WEIGHT + wl.M)
        hbm_bytes = n_mats * (wl.code_bytes + wl.M * wl.N * 2) + wl.M * wl.K * 2
        if entry == "gateup":
            hbm_bytes += 3 * wl.M * wl.N * 2
        kernel_name = "gemm_smallm"
    else:
        ops = wl.weights * DECODE_OPS_PER_WEIGHT
        hbm_bytes = wl.code_bytes + wl.weights * 2
        kernel_name = "decode"
    achieved_all = {"alu": ops / t_kernel / 1e12, "hbm": hbm_bytes / t_kernel / 1e9,
                    "tensor": flops / t_kernel / 1e12}
    t_roof = {"alu": ops / (alu_peak * 1e12), "hbm": hbm_bytes / (hbm_peak * 1e9),
              "tensor": flops / (tensor_peak * 1e12)}
    bound = max(t_roof, key=t_roof.get)
    peak = {"alu": alu_peak, "hbm": hbm_peak, "tensor": tensor_peak}[bound]
    achieved = achieved_all[bound]
    return {"bound": bound,
            "achieved": round(achieved, 3),
            "peak": round(peak, 3),
            "unit": {"alu": "Tops/s", "hbm": "GB/s", "tensor": "TFLOP/s"}[bound],
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(kernel_name, wl.name),
            "peak_source": {"alu": f"{peak_src}: {num_sms} SMs x {ALU_LANES_PER_SM} lanes x "
                                   f"{sm_max:.0f} MHz (of measured max clock)",
                            "hbm": f"{peak_src} hbm_gbs (of measured)",
                            "tensor": f"{peak_src} bf16_tflops (of measured)"}[bound],
            "tensor_TFLOPs": round(achieved_all["tensor"], 1) if flops else None,
            "ops_per_launch": ops, "algorithmic_bytes_per_launch": hbm_bytes,
            "hbm_GBps": round(achieved_all["hbm"], 1),
            "hbm_frac": round(achieved_all["hbm"] / hbm_peak, 4),
            "alu_frac": round(achieved_all["alu"] / alu_peak, 4),
            "roofline_us": round(max(t_roof.values()) * 1e6, 2),
            "kernel_us": round(kernel_ms * 1e3, 2)}


class Entry:
    """One workload on one entry point, device-resident and ready to time: the
    codes rotate through enough independent copies (> 2x L2) that every call
    streams them from HBM."""

    def __init__(self, wl, entry: str, lib, torch, stream, groups: int = 4):
        from trellis_quantized_weight_gb300 import binding, synth
        self.wl, self.entry = wl, entry
        self.x, self.codes, self.scales = wl.generate()
        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
        self.n_rot = n_rot = max(2, math.ceil(2 * l2 / wl.code_bytes) + 1)
        self.n_mats = 2 if entry == "gateup" else 1
        self.groups = groups
        self.launches = launches_per_step(entry, wl.M, groups)
        dx = self.dx = to_dev(self.x, torch, "bf16")
        dscales = self.dscales = to_dev(self.scales, torch, "bf16")
        dcodes = self.dcodes = [to_dev(self.codes, torch, "u32") for _ in range(n_rot)]
        s_handle = stream.cuda_stream
        self.codes_u = self.scales_u = None
        if entry == "gateup":
            # the up projection: a second matrix of the same shape, its own seed
            _, self.codes_u, self.scales_u = synth.small(wl.M, wl.K, wl.N, wl.k, seed=wl.seed + 0x1000,
                                                         sigma=wl.sigma).generate()
            dcodes_u = [to_dev(self.codes_u, torch, "u32") for _ in range(n_rot)]
            dscales_u = to_dev(self.scales_u, torch, "bf16")
            outs = [torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
            ws_bytes = binding.gemm_gateup_workspace_bytes(wl.M, wl.K, wl.N, wl.k, wl.L)
            ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")

            def call(i):
                rc = lib.trellis_gemm_gateup(dx.data_ptr(), dcodes[i % n_rot].data_ptr(), dscales.data_ptr(),
                                             dcodes_u[i % n_rot].data_ptr(), dscales_u.data_ptr(), wl.M, wl.K,
                                             wl.N, wl.k, wl.L, wl.T, outs[0].data_ptr(), outs[1].data_ptr(),
                                             outs[2].data_ptr(), ws.data_ptr(), ws.numel(), s_handle)
                if rc != 0:
                    raise RuntimeError(f"trellis_gemm_gateup failed: {binding.status_string(rc)}")
        elif entry == "packed":
            # the workload's M rows as `groups` sequences (sizes as equal as possible),
            # gathered, multiplied once and scattered back by trellis_gemm_packed
            rows = group_rows(wl.M, groups)
            self.offs = offs = np.cumsum([0] + rows)
            out = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda")
            xp = (ctypes.c_void_p * len(rows))(*[dx[a:b].data_ptr() for a, b in zip(offs[:-1], offs[1:])])
            op = (ctypes.c_void_p * len(rows))(*[out[a:b].data_ptr() for a, b in zip(offs[:-1], offs[1:])])
            rp = (ctypes.c_int * len(rows))(*rows)
            ws_bytes = binding.gemm_packed_workspace_bytes(rows, wl.K, wl.N, wl.k, wl.L)
            ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")

            def call(i):
                rc = lib.trellis_gemm_packed(xp, rp, len(rows), dcodes[i % n_rot].data_ptr(), dscales.data_ptr(),
                                             wl.K, wl.N, wl.k, wl.L, wl.T, op, ws.data_ptr(), ws.numel(),
                                             s_handle)
                if rc != 0:
                    raise RuntimeError(f"trellis_gemm_packed failed: {binding.status_string(rc)}")
        elif entry == "gemm":
            # trellis_gemm: the library's own split-K scratch, no workspace argument
            out = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda")

            def call(i):
                rc = lib.trellis_gemm(dx.data_ptr(), dcodes[i % n_rot].data_ptr(), dscales.data_ptr(),
                                      wl.M, wl.K, wl.N, wl.k, wl.L, wl.T, out.data_ptr(), s_handle)
                if rc != 0:
                    raise RuntimeError(f"trellis_gemm failed: {binding.status_string(rc)}")
        else:
            wout = torch.empty((wl.N, wl.K), dtype=torch.bfloat16, device="cuda")

            def call(i):
                rc = lib.trellis_decode(dcodes[i % n_rot].data_ptr(), dscales.data_ptr(), wl.K, wl.N, wl.k,
                                        wl.L, wl.T, wout.data_ptr(), s_handle)
                if rc != 0:
                    raise RuntimeError(f"trellis_decode failed: {binding.status_string(rc)}")
        self.call = call

    def config(self, world: int, graph: bool = False) -> dict:
        wl = self.wl
        return {"workload": wl.name, "entry": "trellis_" + self.entry, "M": wl.M, "K": wl.K, "N": wl.N,
                **({"groups": group_rows(wl.M, self.groups)} if self.entry == "packed" else {}),
                "k": wl.k, "L": wl.L, "T": wl.T, "parallelism": f"replicas{world}",
                "launch": "CUDA graph of the K steps" if graph else "stream, programmatic launches",
                "l2": f"rotating {self.n_rot} code copies ({self.n_rot * wl.code_bytes / 1e6:.0f} MB > 2x L2)"}


def time_steps(ent, steps: int, warmup: int, stream, torch, world: int, gpu_index: int, graph: bool = False):
    """W warm-up calls, then `steps` calls back to back on one stream (as a model
    issues its layers) between one pair of CUDA events, with barriers and
    synchronisation on both sides and nvidia-smi sampling the clocks.  Returns
    (ms per step, clocks, host wall seconds)."""
    import torch.distributed as dist
    with torch.cuda.stream(stream):
        for i in range(warmup):
            ent.call(i)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.15)
    if world > 1:
        dist.barrier()
    g = None
    if graph:
        # the K steps captured once into a CUDA graph (outside the timed region)
        # and replayed inside it: the same launches, no host launch overhead
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(steps):
                ent.call(warmup + i)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    t_host0 = time.perf_counter()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        if g is not None:
            g.replay()
        else:
            for i in range(steps):
                ent.call(warmup + i)
        t_end.record(stream)
    torch.cuda.synchronize()
    t_host = time.perf_counter() - t_host0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    return t_start.elapsed_time(t_end) / steps, clocks, t_host


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def host_cores() -> list[int]:
    """The cores this process may run on."""
    try:
        return sorted(os.sched_getaffinity(0))
    except AttributeError:
        return list(range(os.cpu_count() or 1))


def oracle_rate(wl, x, codes, scales, budget_s: float, threads: int, decode_only: bool = False,
                pin_core: int | None = None):
    """The unchanged oracle (decode + product, or decode alone) over row chunks on
    `threads` host threads for about budget_s seconds.  With pin_core the work
    runs in this thread alone, pinned to that core.  Returns (GB/s of codes,
    microseconds per whole call extrapolated from the rows done, rows, seconds)."""
    import oracle
    o = oracle.get()
    chunk = max(1, min(wl.N, 16 if pin_core is not None else 64))

    def work(r):
        w = o.decode(codes, scales, wl.K, wl.N, wl.k, L=wl.L, rows=r)
        if not decode_only:
            o.gemm_dense(x, w)
        return r[1] - r[0]

    done_rows = 0
    n0 = 0
    if pin_core is not None:
        old = os.sched_getaffinity(0)
        os.sched_setaffinity(0, {pin_core})
        try:
            t0 = time.perf_counter()
            while True:
                n1 = min(wl.N, n0 + chunk)
                done_rows += work((n0, n1))
                n0 = 0 if n1 >= wl.N else n1
                if time.perf_counter() - t0 >= budget_s:
                    break
            dt = time.perf_counter() - t0
        finally:
            os.sched_setaffinity(0, old)
    else:
        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(threads) as ex:
            while True:
                batch = []
                for _ in range(threads):
                    n1 = min(wl.N, n0 + chunk)
                    batch.append((n0, n1))
                    n0 = 0 if n1 >= wl.N else n1
                done_rows += sum(ex.map(work, batch))
                if time.perf_counter() - t0 >= budget_s:
                    break
        dt = time.perf_counter() - t0
    gbs = done_rows * wl.row_words * 4 / dt / 1e9
    us_call = dt / done_rows * wl.N * 1e6
    return gbs, us_call, done_rows, dt


def cpu_baseline_for(wl, x, codes, scales, budget_s: float, decode_only: bool = False) -> dict:
    """The oracle on all host cores and on one pinned core, with the CPU model."""
    cores = host_cores()
    gbs, us, rows, dt = oracle_rate(wl, x, codes, scales, budget_s, len(cores), decode_only)
    gbs1, us1, rows1, dt1 = oracle_rate(wl, x, codes, scales, budget_s, 1, decode_only, pin_core=cores[0])
    what = "decode" if decode_only else "decode + product"
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": len(cores), "kind": "oracle",
            "us_per_call": round(us, 1),
            "sample": f"{rows} rows x K={wl.K} of {wl.name} ({what}) in {dt:.1f} s on {len(cores)} threads",
            "one_core": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1, "us_per_call": round(us1, 1),
                         "sample": f"{rows1} rows ({what}) in {dt1:.1f} s, pinned to core {cores[0]}"},
            "cpu_model": cpu_model()}


# The per-configuration table: every quantised-linear workload through
# trellis_gemm, and the dense decode of the k = 3 and k = 4 weights.
PER_CONFIG = [(name, "gemm") for name in
              ["gemm_m5_k5120_n17408_k2", "gemm_m8_k5120_n17408_k3", "gemm_m15_k5120_n17408_k4",
               "gemv_m1_k17408_n5120_k4", "prefill_m64_k5120_n17408_k4"]] + \
             [("gemm_m8_k5120_n17408_k3", "decode"), ("prefill_m64_k5120_n17408_k4", "decode")]


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")

    from trellis_quantized_weight_gb300 import binding, build, synth
    build.build()
    lib = binding.load()
    props = torch.cuda.get_device_properties(local)
    stream = torch.cuda.Stream()

    ent = Entry(wl, args.entry, lib, torch, stream, args.groups)
    x, codes, scales = ent.x, ent.codes, ent.scales
    torch.cuda.synchronize()
    ms_step, clocks, t_host = time_steps(ent, args.steps, args.warmup, stream, torch, world, local, args.graph)
    kernel_ms = ms_step

    # For context, outside the timed region: one call at a time, each between
    # its own pair of events (adds the launch and drain latency to every call).
    n_iso = min(args.steps, 50)
    iso = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_iso)]
    with torch.cuda.stream(stream):
        for i, (a, b) in enumerate(iso):
            a.record(stream)
            ent.call(args.warmup + args.steps + i)
            b.record(stream)
    torch.cuda.synchronize()
    isolated_ms = statistics.median([a.elapsed_time(b) for a, b in iso])
    ms_step, kernel_ms, isolated_ms = max_over_ranks([ms_step, kernel_ms, isolated_ms], device="cuda")
    n_mats = ent.n_mats

    # ---- end to end through the public API, host buffers in pinned memory ----
    # Every step uploads its inputs from pinned host memory and reads its result
    # back.  Two device buffer sets let step i+1's uploads (two copy streams,
    # each carrying half of the codes) run while step i's product runs; a set is
    # overwritten only after the product that read it has finished.
    e2e = None
    if not args.no_e2e:
        from trellis_quantized_weight_gb300 import gemm as tq_gemm
        hx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
        hc = torch.from_numpy(codes.view(np.int32)).pin_memory()
        hs = torch.from_numpy(scales.view(np.int16)).view(torch.bfloat16).pin_memory()
        hout = torch.empty((wl.M, wl.N), dtype=torch.bfloat16).pin_memory()
        n_e2e = max(3, min(args.steps, args.e2e_steps))
        hcu = hsu = None
        if args.entry == "decode":
            from trellis_quantized_weight_gb300 import decode as tq_decode
            hout = torch.empty((wl.N, wl.K), dtype=torch.bfloat16).pin_memory()
        if args.entry == "packed":
            from trellis_quantized_weight_gb300 import gemm_packed as tq_packed
            ypk = torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device="cuda")
            offs = ent.offs
        if args.entry == "gateup":
            from trellis_quantized_weight_gb300 import gemm_gateup as tq_gateup
            hcu = torch.from_numpy(ent.codes_u.view(np.int32)).pin_memory()
            hsu = torch.from_numpy(ent.scales_u.view(np.int16)).view(torch.bfloat16).pin_memory()
        bufs = []
        for _ in range(2):
            b = {"x": torch.empty_like(ent.dx), "c": torch.empty_like(ent.dcodes[0]),
                 "s": torch.empty_like(ent.dscales)}
            if hcu is not None:
                b["cu"] = torch.empty_like(ent.dcodes[0])
                b["su"] = torch.empty_like(ent.dscales)
            bufs.append(b)
        copy_streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        free = [None, None]            # event: the product that read set b has finished
        half = hc.shape[0] // 2

        def upload(bi, after=None):
            b = bufs[bi]
            done = []
            for j, cs in enumerate(copy_streams):
                if free[bi] is not None:
                    cs.wait_event(free[bi])
                if after is not None:
                    cs.wait_event(after)
                rows = slice(0, half) if j == 0 else slice(half, None)
                with torch.cuda.stream(cs):
                    b["c"][rows].copy_(hc[rows], non_blocking=True)
                    if hcu is not None:
                        b["cu"][rows].copy_(hcu[rows], non_blocking=True)
                    if j == 1:
                        b["s"].copy_(hs, non_blocking=True)
                        if hsu is not None:
                            b["su"].copy_(hsu, non_blocking=True)
                        if args.entry != "decode":
                            b["x"].copy_(hx, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cs)
                    done.append(ev)
            return done

        def compute(bi, ready):
            b = bufs[bi]
            for ev in ready:
                stream.wait_event(ev)
            with torch.cuda.stream(stream):
                if args.entry == "gemm":
                    y = tq_gemm(b["x"], b["c"], b["s"], wl.k, L=wl.L)
                elif args.entry == "packed":
                    tq_packed([b["x"][a:e] for a, e in zip(offs[:-1], offs[1:])], b["c"], b["s"], wl.k, L=wl.L,
                              outs=[ypk[a:e] for a, e in zip(offs[:-1], offs[1:])])
                    y = ypk
                elif args.entry == "gateup":
                    y = tq_gateup(b["x"], b["c"], b["s"], b["cu"], b["su"], wl.k, L=wl.L)[2]   # the activation
                else:
                    y = tq_decode(b["c"], b["s"], wl.K, wl.k, L=wl.L)
                hout.copy_(y, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(stream)
                free[bi] = ev

        def run_steps(n, start=None):
            ready = upload(0, after=start)
            for i in range(n):
                nxt = upload((i + 1) % 2) if i + 1 < n else None
                compute(i % 2, ready)
                ready = nxt

        run_steps(3)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(n_e2e, start=e0)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        (e2e_ms,) = max_over_ranks([e2e_ms], device="cuda")
        h2d = (hx.numel() * 2 if args.entry != "decode" else 0) + n_mats * (hc.numel() * 4 + hs.numel() * 2)
        e2e = {"value": round(whole_job_gbs(world, n_mats * wl.code_bytes, e2e_ms), 2), "unit": "GB/s",
               "us_per_call": round(e2e_ms * 1e3, 2), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": hout.numel() * 2,
               "pipelining": "two buffer sets: step i+1's uploads overlap step i's product"}

    roof = roofline(wl, args.entry, kernel_ms, props.multi_processor_count)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_for(wl, x, codes, scales, args.cpu_budget, decode_only=args.entry == "decode")

    config = ent.config(world, args.graph)

    # ---- every configuration, each in its own timed region ----
    per_config = None
    if not args.no_per_config:
        del ent
        torch.cuda.empty_cache()
        per_config = {}
        for name, entry in PER_CONFIG:
            pwl = synth.WORKLOADS[name]
            pe = Entry(pwl, entry, lib, torch, stream)
            torch.cuda.synchronize()
            p_ms, p_clocks, _ = time_steps(pe, args.per_config_steps, max(3, min(args.warmup, 20)), stream,
                                           torch, world, local)
            (p_ms,) = max_over_ranks([p_ms], device="cuda")
            r = roofline(pwl, entry, p_ms, props.multi_processor_count)
            key = name if entry == "gemm" else f"decode_k{pwl.K}_n{pwl.N}_k{pwl.k}"
            per_config[key] = {
                "entry": "trellis_" + entry, "M": pwl.M, "K": pwl.K, "N": pwl.N, "k": pwl.k,
                "us_per_call": round(p_ms * 1e3, 2),
                "value": round(whole_job_gbs(world, pwl.code_bytes, p_ms), 2), "unit": "GB/s",
                "roofline": {kk: r[kk] for kk in ("bound", "frac", "roofline_us", "achieved", "peak", "unit",
                                                  "hbm_frac", "alu_frac", "traffic")},
                "steps": args.per_config_steps, "clocks": p_clocks,
                "l2": f"rotating {pe.n_rot} code copies",
            }
            if rank == 0 and not args.no_cpu_baseline:
                per_config[key]["cpu_baseline"] = cpu_baseline_for(pwl, pe.x, pe.codes, pe.scales,
                                                                   args.cpu_budget_per_config,
                                                                   decode_only=entry == "decode")
            del pe
            torch.cuda.empty_cache()

    value = whole_job_gbs(world, n_mats * wl.code_bytes, ms_step)
    line = {
        "metric": {"gemm": METRIC, "decode": METRIC_DECODE, "gateup": METRIC_GATEUP,
                   "packed": METRIC_PACKED}[args.entry],
        "value": round(value, 2), "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "us_per_call": round(ms_step * 1e3, 2), "isolated_call_us": round(isolated_ms * 1e3, 2),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": path_dtype(args.entry, wl.M), "data": "synthetic",
        "config": config,
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step(args.entry, wl.M, args.groups),
        "clocks": clocks, "host_wall_s": round(t_host, 3),
        "per_config": per_config,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------- reference arm --
def run_reference(args, wl):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    x, codes, scales = wl.generate()
    threads = len(host_cores())
    # size each step so that warm-up + steps take about args.ref_budget seconds
    per_step = max(0.002, args.ref_budget / max(1, args.steps + args.warmup))
    import oracle
    o = oracle.get()
    t0 = time.perf_counter()
    w = o.decode(codes, scales, wl.K, wl.N, wl.k, rows=(0, 8))
    o.gemm_dense(x, w)
    per_row = (time.perf_counter() - t0) / 8
    rows = max(1, min(wl.N, int(per_step * threads / per_row)))

    def step(i):
        n0 = (i * rows) % wl.N
        n1 = min(wl.N, n0 + rows)
        edges = np.linspace(n0, n1, threads + 1).astype(int)
        parts = [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:]) if b > a]

        def work(r):
            ww = o.decode(codes, scales, wl.K, wl.N, wl.k, L=wl.L, rows=r)
            o.gemm_dense(x, ww)
        list(ex.map(work, parts))
        return n1 - n0

    with cf.ThreadPoolExecutor(threads) as ex:
        for i in range(args.warmup):
            step(i)
        t0 = time.perf_counter()
        done = sum(step(args.warmup + i) for i in range(args.steps))
        dt = time.perf_counter() - t0
    gbs = done * wl.row_words * 4 / dt / 1e9
    ms_step = dt / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "K": wl.K, "N": wl.N, "k": wl.k, "L": wl.L, "T": wl.T,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} rows x K={wl.K} per step (decode + product)",
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--entry", choices=["gemm", "decode", "gateup", "packed"], default="gemm",
                    help="time the fused product (default), the dense decode, the gate/up pair with its "
                         "activation, or the token-packed product of --groups sequences")
    ap.add_argument("--groups", type=int, default=4, help="sequences the M rows are split into (--entry packed)")
    ap.add_argument("--graph", action="store_true",
                    help="capture the K timed steps into one CUDA graph and time its replay")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-budget", type=float, default=5.0,
                    help="seconds of oracle work for cpu_baseline (each of all cores and one core)")
    ap.add_argument("--cpu-budget-per-config", type=float, default=1.0,
                    help="seconds of oracle work per configuration (each of all cores and one core)")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-configuration table")
    ap.add_argument("--per-config-steps", type=int, default=2000)
    ap.add_argument("--ref-budget", type=float, default=60.0, help="seconds for the reference arm's timed run")
    ap.add_argument("--rows", type=int, default=None,
                    help="activation rows M instead of the workload's own (a prefill sweep of the same weights)")
    ap.add_argument("--bits", type=int, default=None, help="bits per weight k instead of the workload's own (1..8)")
    ap.add_argument("--window", type=int, default=None, help="window bits L instead of 12 (k < L <= 24)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from trellis_quantized_weight_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.rows is not None:
        if not 1 <= args.rows <= 65536:
            ap.error("--rows must be in 1..65536")
        kind = "gemv" if args.rows == 1 else ("gemm" if args.rows <= 16 else "prefill")
        wl = dataclasses.replace(wl, M=args.rows, name=f"{kind}_m{args.rows}_k{wl.K}_n{wl.N}_k{wl.k}")
    if args.bits is not None or args.window is not None:
        k = wl.k if args.bits is None else args.bits
        L = wl.L if args.window is None else args.window
        if not (1 <= k <= 8 and k < L <= 24):
            ap.error("need 1 <= k <= 8 and k < L <= 24")
        base = wl.name.rsplit("_k", 1)[0]
        wl = dataclasses.replace(wl, k=k, L=L, name=f"{base}_k{k}" + ("" if L == 12 else f"_L{L}"))
    if args.entry == "packed" and not 1 <= args.groups <= wl.M:
        ap.error("--groups must be in 1..M")
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
