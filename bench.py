#!/usr/bin/env python3
"""Benchmark of the pipelined GEMM library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload f32_4096|f32_1024|f32_256|f32_ragged|bf16_8192]
                    [--fill tma|cpasync|sync] [--stages S] [--tile 64|128]

One step is one GEMM of the chosen workload through the library's C ABI with
inputs resident in device memory; the default is the FP32 GEMM at
M = N = K = 4096 (seeded uniform[-1,1) operands) through the TMA-ring
pipelined fill.  L2 is flushed (a 256 MiB device write) before every timed
step; each step's kernel is timed with CUDA events on the launching stream.

Beside the headline the JSON line carries: the sync / cp.async / TMA fills and
the stage sweep at the same size (TFLOP/s and t_sync / t_fill), the BF16
tensor-core GEMM at 8192^3, an end-to-end number through the public API with
host buffers, the ALU or tensor roofline of the dominant kernel, live clock
samples, and the CPU oracle timed on the host cores on a bounded sample.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent replicas: the GEMM has no exchange step); timing is the max over
ranks and the value sums the ranks' work.

--impl reference times the CPU oracle itself (plain C, float64, all host
cores) on the same workload, each step a bounded sample of output rows.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s and % of FP32-FFMA / BF16-tensor peak, pipelined vs sync fill"
UNIT = "TFLOP/s"
FP32_FMA_PER_SM_PER_CLK = 128        # FP32 lanes per SM on sm_100-family parts
# Dense BF16 tensor-core work per SM per clock on sm_100-family parts
# (tcgen05.mma kind::f16, no 2:4 sparsity): twice Hopper's.  Hopper's figure
# follows from NVIDIA's H100 SXM5 datasheet: 989.4 dense BF16 TFLOP/s at the
# 1830 MHz boost clock on 132 SMs = 4096 FLOP per SM per clock; NVIDIA's
# Blackwell material states the fifth-generation tensor core doubles the
# per-SM FP16/BF16 rate.
BF16_DENSE_FLOP_PER_SM_PER_CLK = 8192
FALLBACK_SM_MAX_MHZ = 2070.0
FALLBACK_BF16_TFLOPS = 1900.0
FLUSH_BYTES = 256 << 20              # > 2x the 126 MiB L2
# BF16: stages 0 and tile 0 take the library's choice for the workload (at
# 8192^3 the 256-row tile with three stages); the plan resolves both before
# anything is timed, so the JSON line names what ran.
DEFAULT_LEG = {"f32": dict(fill="tma", stages=2, tile=128), "bf16": dict(fill="tma", stages=0, tile=0)}


# --------------------------------------------------------------------- dist
class Dist:
    """Rank bookkeeping; torch.distributed only when WORLD_SIZE > 1."""

    def __init__(self, backend: str | None = None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            dist.init_process_group(backend=backend or "nccl")
            self.pg = dist
            self.device = torch.device("cuda", self.local_rank) if (backend or "nccl") == "nccl" else None

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def _reduce(self, x: float, op) -> float:
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=op)
        return float(t.item())

    def max(self, x: float) -> float:
        return self._reduce(x, None if self.pg is None else self.pg.ReduceOp.MAX)

    def sum(self, x: float) -> float:
        return self._reduce(x, None if self.pg is None else self.pg.ReduceOp.SUM)

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


class CudaTimer:
    """Per-step CUDA events on the current stream; read after a sync."""

    def __init__(self):
        import torch
        self.torch = torch
        self.pairs = []

    def begin(self):
        e = self.torch.cuda.Event(enable_timing=True)
        e.record()
        self.pairs.append([e, None])

    def end(self):
        e = self.torch.cuda.Event(enable_timing=True)
        e.record()
        self.pairs[-1][1] = e

    def durations_ms(self):
        return [a.elapsed_time(b) for a, b in self.pairs]


class WallTimer:
    def __init__(self, sync=lambda: None):
        self.sync = sync
        self.t = []

    def begin(self):
        self.sync()
        self.t.append([time.perf_counter(), None])

    def end(self):
        self.sync()
        self.t[-1][1] = time.perf_counter()

    def durations_ms(self):
        return [(b - a) * 1e3 for a, b in self.t]


def timed_loop(dist: Dist, steps: int, warmup: int, step, flush, timer, sync):
    """W untimed steps, then exactly K timed steps bracketed by a barrier and a
    sync on both sides.  Returns (max-over-ranks total ms, local per-step ms)."""
    for _ in range(warmup):
        flush()
        step()
    sync()
    dist.barrier()
    sync()
    for _ in range(steps):
        flush()
        timer.begin()
        step()
        timer.end()
    sync()
    dist.barrier()
    sync()
    per = timer.durations_ms()
    return dist.max(sum(per)), per


# --------------------------------------------------------------------- peaks
def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    return {"_source": "fallback", "sm_max_mhz": FALLBACK_SM_MAX_MHZ, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def fp32_peak_tflops(num_sms: int, mhz: float) -> float:
    return num_sms * FP32_FMA_PER_SM_PER_CLK * 2 * mhz * 1e6 / 1e12


def bf16_derived_peak_tflops(num_sms: int, mhz: float, per_sm_per_clk: float = BF16_DENSE_FLOP_PER_SM_PER_CLK) -> float:
    return num_sms * per_sm_per_clk * mhz * 1e6 / 1e12


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            fields = {}
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
        for key in ("model name", "hardware", "cpu part"):
            if key in fields:
                return fields[key] if key != "cpu part" else f"CPU part {fields[key]}"
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


class DeviceStatusError(RuntimeError):
    pass


def check_status(pg, what: str):
    """A kernel that gave up on a bounded wait leaves C undefined: its timing
    is not a measurement of the GEMM."""
    st, detail = pg.device_status()
    if st != 0:
        raise DeviceStatusError(f"device status {st} ({detail:#x}) after {what}")


# --------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            import atexit
            atexit.register(self.stop)  # never leave the sampler running past an early exit

    def stop(self):
        if self.proc is None or self.proc.returncode is not None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        rows = []
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 11:
                continue
            try:
                rows.append(dict(sm=float(f[2]), smax=float(f[3]), power=float(f[4]) if f[4] not in ("[N/A]", "") else 0.0,
                                 util=float(f[5]) if f[5] not in ("[N/A]", "") else 0.0,
                                 hw=f[7], hwt=f[8], swt=f[9], swp=f[10]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [r for r in rows if r["util"] > 0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded),
                "power_w_max": max(r["power"] for r in loaded)}


# --------------------------------------------------------------------- profiles
def _code_only(src: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed
    (string and character literals are kept as they are)."""
    out, i, n, quote = [], 0, len(src), None
    while i < n:
        c = src[i]
        if quote is None:
            if src.startswith("//", i):
                j = src.find("\n", i)
                i = n if j < 0 else j
                continue
            if src.startswith("/*", i):
                j = src.find("*/", i + 2)
                i = n if j < 0 else j + 2
                out.append(" ")
                continue
            if c in "\"'":
                quote = c
        elif c == "\\" and i + 1 < n:
            out.append(src[i:i + 2])
            i += 2
            continue
        elif c == quote:
            quote = None
        out.append(c)
        i += 1
    return " ".join("".join(out).split())


# Sources that launch no kernel of their own and set no launch parameter:
# the host-buffer executor only sequences copies and library calls.
NON_KERNEL_SOURCES = ("host_exec.cu",)


def kernel_sources_sha() -> str:
    """Hash of the code of the CUDA sources that define the kernels and their
    launches (comments and whitespace ignored); a traffic figure captured
    for other code is stale."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "async_copy_pipelined_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in NON_KERNEL_SOURCES:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode())
                h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was captured
    from the current kernel sources.  Lines read: `source_sha: <hash>` and
    `traffic_bytes_per_launch[<kernel_key>]: <bytes>`."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    sha, traffic = None, None
    with open(path) as f:
        for line in f:
            line = line.strip().strip("-` ")
            if line.startswith("source_sha:"):
                sha = line.split(":", 1)[1].strip()
            if line.startswith(f"traffic_bytes_per_launch[{kernel_key}]:"):
                try:
                    traffic = float(line.rsplit(":", 1)[1].strip())
                except ValueError:
                    traffic = None
    if sha is None or sha != kernel_sources_sha():
        return None
    return traffic


# --------------------------------------------------------------------- workloads
def load_workload(name: str):
    from async_copy_pipelined_gb300 import inputs
    w = dict(inputs.WORKLOADS[name])
    A, B = inputs.workload_operands(name)
    return w, A, B


def to_device(x, cols, dev):
    import numpy as np
    import torch
    if x.dtype == np.uint16:
        t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(x)
    return t.to(dev)[:, :cols]


def f32_kernels_per_call(pg, M, N, K, lda, ldb, fill, stages, tile, workspace="auto") -> int:
    """Kernel launches one device-buffer FP32 call makes.  The TMA fill on
    the 128 tile may first run the wide-row kernel on its top rows
    (plan["wide_rows"]); the rows below it, with a hand-over workspace, split
    the last round of 128 x 128 tiles in K, which takes the one-tile kernel
    for the whole rounds before it (if any) and the persistent kernel for the
    split region.  Every other call is one launch."""
    if fill != "tma" or M == 0 or N == 0 or K == 0:
        return 1
    p = pg.plan_f32(M, N, K, lda=lda, ldb=ldb, fill=fill, stages=stages, block_tile=tile)
    wide = p["wide_rows"]
    n = 1 if wide > 0 else 0
    rows = M - wide
    if rows <= 0:
        return n
    ctas = p["persistent_ctas"]
    if workspace is None or ctas <= 0:
        return n + 1
    tiles = p["grid_x"] * ((rows + p["block_m"] - 1) // p["block_m"])
    return n + (2 if tiles // ctas >= 2 else 1)


class GemmCall:
    """One library call on fixed operands; `kernels` is how many of the
    library's kernels each call launches."""

    def __init__(self, fn, kernels: int):
        self.fn, self.kernels = fn, kernels

    def __call__(self):
        return self.fn()


_LIBRARY_DEFAULT = object()


def gemm_call(pg, name, Ad, Bd, Cd, fill, stages, tile, options=(), workspace=_LIBRARY_DEFAULT):
    """A call of the binding as a user makes it; `workspace` as the binding
    takes it, by default the binding's own default (FP32: "auto", the K
    split; BF16: None, no split)."""
    if name.startswith("bf16"):
        ws = None if workspace is _LIBRARY_DEFAULT else workspace
        return GemmCall(lambda: pg.gemm_bf16(Ad, Bd, Cd, fill=fill, stages=stages, block_m=tile, options=options,
                                             workspace=ws), 1)
    if workspace is _LIBRARY_DEFAULT:
        workspace = "auto"
    k = f32_kernels_per_call(pg, Ad.shape[0], Bd.shape[1], Ad.shape[1], Ad.stride(0), Bd.stride(0), fill, stages,
                             tile, workspace)
    return GemmCall(lambda: pg.gemm_f32(Ad, Bd, Cd, fill=fill, stages=stages, block_tile=tile, options=options,
                                        workspace=workspace), k)


# Library kernel launches made by the measured calls of the side legs
# (time_kernel, clocks_during, the cache-option bit checks).
SIDE_LAUNCHES = {"n": 0}


def _count(call, calls: int):
    SIDE_LAUNCHES["n"] += calls * getattr(call, "kernels", 1)


# The cache qualifiers of the "cp.async" tile-op reference (prefetch size,
# L2 cache policy), each timed beside the default call on the same operands.
CACHE_OPTION_SETS = {"prefetch_128b": ("l2_prefetch_128b",),
                     "a_first_b_last": ("a_evict_first", "b_evict_last"),
                     "a_last_b_last": ("a_evict_last", "b_evict_last")}


def time_cache_options(pg, name, Ad, Bd, Cd, legs, flush, launches, flops):
    """{leg: {option set: TFLOP/s, ...}} for each (fill, stages, tile) leg;
    option sets a fill does not take are skipped.  Bits are checked equal to
    the default call's."""
    import torch
    out, n = {}, 0
    for fill, stages, tile in legs:
        row = {}
        ref = None
        for label, opts in [("default", ())] + list(CACHE_OPTION_SETS.items()):
            if fill == "tma" and "l2_prefetch_128b" in opts:
                continue
            call = gemm_call(pg, name, Ad, Bd, Cd, fill, stages, tile, opts)
            call()
            _count(call, 1)
            torch.cuda.synchronize()
            check_status(pg, f"cache option {label}")
            if ref is None:
                ref = Cd.clone()
            same = bool(torch.equal(Cd.view(torch.int32), ref.view(torch.int32)))
            mean, best, med = time_kernel(pg, call, flush, launches)
            n += launches + 1
            row[label] = {"tflops": flops / (mean / 1e3) / 1e12, "ms": mean, "ms_min": best, "bits_equal_default": same}
        for v in row.values():
            v["vs_default"] = v["tflops"] / row["default"]["tflops"]
        out[f"{fill}/S{stages}/T{tile}"] = row
    return out, n


def time_kernel(pg, call, flush, launches: int, warmup: int = 3):
    """Mean / min / median ms of `launches` calls, each after an L2 flush,
    events on the stream."""
    import torch
    for _ in range(warmup):
        flush()
        call()
    timer = CudaTimer()
    for _ in range(launches):
        flush()
        timer.begin()
        call()
        timer.end()
    torch.cuda.synchronize()
    _count(call, launches)
    check_status(pg, "a timed side leg")
    d = timer.durations_ms()
    return statistics.mean(d), min(d), statistics.median(d)


def clocks_during(call, seconds: float, uuid):
    """Median SM clock (nvidia-smi samples) while `call` runs back to back
    for about `seconds`."""
    import torch
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    t_end = time.perf_counter() + seconds
    launches = 0
    while time.perf_counter() < t_end:
        for _ in range(50):
            call()
        launches += 50
        torch.cuda.synchronize()
    sampler.stop()
    _count(call, launches)
    out = sampler.summary()
    out["calls"] = launches
    return out


# --------------------------------------------------------------------- oracle leg
def oracle_sample(name: str, A, B, w, seconds: float, gpu_rows=None):
    """Time the CPU oracle (float64 definition) on a bounded row sample."""
    import numpy as np
    import oracle
    oracle.build()
    M, N, K = w["M"], w["N"], w["K"]
    fn = oracle.gemm_bf16_f64 if name.startswith("bf16") else oracle.gemm_f64
    cores = oracle.num_threads()
    probe = max(1, min(M, cores))
    t0 = time.perf_counter()
    fn(np.ascontiguousarray(A[:probe]), B, probe, N, K)
    t_probe = time.perf_counter() - t0
    rows = int(max(probe, min(M, probe * seconds / max(t_probe, 1e-6))))
    rows = max(cores, (rows // cores) * cores) if rows >= cores else rows
    rows = min(rows, M)
    t0 = time.perf_counter()
    out = fn(np.ascontiguousarray(A[:rows]), B, rows, N, K)
    t = time.perf_counter() - t0
    res = {"value": 2.0 * rows * N * K / t / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"first {rows} of {M} output rows (all {N} columns, K={K}); {t:.2f} s on the host cores",
           "seconds": t, "rows": rows, "cpu_model": host_cpu_model(), "nproc": os.cpu_count()}
    if gpu_rows is not None:
        g = gpu_rows[:rows].astype(np.float64)
        res["max_abs_diff_vs_gpu"] = float(np.max(np.abs(g - out)))
    return res


def oracle_small_configs():
    """The oracle over the whole output of the two small FP32 workloads, on
    all host cores and on one thread (TFLOP/s and seconds)."""
    import numpy as np
    import oracle
    oracle.build()
    cores = oracle.num_threads()
    out = {}
    try:
        for wname in ("f32_256", "f32_1024"):
            w, A, B = load_workload(wname)
            M, N, K = w["M"], w["N"], w["K"]
            Ac = np.ascontiguousarray(A[:, :K])
            row = {}
            for label, n in (("all_cores", cores), ("one_thread", 1)):
                oracle.set_num_threads(n)
                t0 = time.perf_counter()
                oracle.gemm_f64(Ac, B, M, N, K)
                t = time.perf_counter() - t0
                row[label] = {"threads": n, "seconds": t, "tflops": 2.0 * M * N * K / t / 1e12}
            # The FP32 FMA-chain oracle the parity tests compare bits with;
            # timed for context, not the baseline.
            oracle.set_num_threads(cores)
            t0 = time.perf_counter()
            oracle.gemm_fmaf_chain(Ac, B, M, N, K)
            t = time.perf_counter() - t0
            row["fmaf_chain_all_cores"] = {"threads": cores, "seconds": t, "tflops": 2.0 * M * N * K / t / 1e12}
            out[wname] = row
    finally:
        oracle.set_num_threads(cores)
    return out


def run_reference(args, dist: Dist):
    """--impl reference: the oracle itself, timed on the host cores."""
    if dist.rank != 0:
        return 0
    name = args.workload
    w, A, B = load_workload(name)
    import numpy as np
    import oracle
    oracle.build()
    M, N, K = w["M"], w["N"], w["K"]
    fn = oracle.gemm_bf16_f64 if name.startswith("bf16") else oracle.gemm_f64
    cores = oracle.num_threads()
    t0 = time.perf_counter()
    fn(np.ascontiguousarray(A[:cores]), B, cores, N, K)
    per_row = (time.perf_counter() - t0) / cores
    budget = args.ref_seconds / max(args.steps + args.warmup, 1)
    rows = int(min(M, max(cores, budget / max(per_row, 1e-9))))
    Asub = np.ascontiguousarray(A[:rows])
    for _ in range(args.warmup):
        fn(Asub, B, rows, N, K)
    durs = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        fn(Asub, B, rows, N, K)
        durs.append(time.perf_counter() - t0)
    total = sum(durs)
    value = 2.0 * rows * N * K * args.steps / total / 1e12
    sample = f"first {rows} of {M} output rows per step (all {N} columns, K={K})"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64" if not name.startswith("bf16") else "f64 (bf16 inputs)", "data": "synthetic",
        "config": workload_config(name, w, None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                         "cpu_model": host_cpu_model(), "nproc": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(name, w, leg):
    desc = {
        "f32_256": "fp32 GEMM M=N=K=256, uniform[-1,1) seed 0",
        "f32_1024": "fp32 GEMM M=N=K=1024, uniform[-1,1) seed 1",
        "f32_4096": "fp32 GEMM M=N=K=4096, uniform[-1,1) seed 2",
        "f32_ragged": "fp32 GEMM M=3000 N=5000 K=1000 lda=1003, normal(0,1) seed 3",
        "bf16_8192": "bf16 GEMM (fp32 accumulate/output) M=N=K=8192, normal(0,0.5)->bf16 seed 4",
        "f32_tallk": "fp32 GEMM M=N=32 K=65536 (one CTA), uniform[-1,1) seed 5",
    }[name]
    cfg = {"workload": desc, "M": w["M"], "N": w["N"], "K": w["K"], "lda": w["lda"],
           "l2": "flushed before every timed step (256 MiB device write)"}
    if leg:
        cfg.update(leg)
    return cfg


# --------------------------------------------------------------------- main leg
def run_ours(args, dist: Dist):
    import numpy as np
    import torch
    import async_copy_pipelined_gb300 as pg

    pg.build()
    pg.lib()
    dev = torch.device("cuda", dist.local_rank if dist.world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    num_sms = props.multi_processor_count
    peaks = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz") or FALLBACK_SM_MAX_MHZ)
    fp32_peak = fp32_peak_tflops(num_sms, sm_max)
    bf16_peak = float(peaks.get("bf16_tflops") or FALLBACK_BF16_TFLOPS)

    name = args.workload
    is_bf16 = name.startswith("bf16")
    leg = dict(DEFAULT_LEG["bf16" if is_bf16 else "f32"])
    if args.fill:
        leg["fill"] = args.fill
    if args.stages is not None:
        leg["stages"] = args.stages
    if args.tile is not None:
        leg["tile"] = args.tile
    if leg["fill"] == "sync":
        leg["stages"] = 1
    w, A, B = load_workload(name)
    M, N, K = w["M"], w["N"], w["K"]
    if is_bf16:
        plan = pg.plan_bf16(M, N, K, lda=w["lda"], fill=leg["fill"], stages=leg["stages"], block_m=leg["tile"])
        leg["stages"], leg["tile"] = plan["stages"], plan["block_m"]
    if leg["fill"] == "tma" and not is_bf16 and w["lda"] % 4:
        # TMA cannot describe a row pitch that is not a multiple of 16 bytes;
        # the same logical matrix is repacked at the next legal pitch.
        from async_copy_pipelined_gb300 import inputs
        A = inputs.workload_operands(name, lda=(w["lda"] + 3) // 4 * 4)[0]
    flops = 2.0 * M * N * K
    Ad, Bd = to_device(A, K, dev), to_device(B, N, dev)
    Cd = torch.empty((M, N), dtype=torch.float32, device=dev)
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush = lambda: flush_buf.zero_()  # noqa: E731
    call = gemm_call(pg, name, Ad, Bd, Cd, leg["fill"], leg["stages"], leg["tile"])

    # Correctness gate before any timing (the lesson program's rule): the
    # pipelined result must be bit-identical to the register-path fill (for
    # BF16 on the 128-row tile, so the gate also crosses tile heights).
    call()
    Cs = torch.empty_like(Cd)
    if is_bf16:
        pg.gemm_bf16(Ad, Bd, Cs, fill="sync", block_m=128)
    else:
        pg.gemm_f32(Ad, Bd, Cs, fill="sync", block_tile=leg["tile"])
    torch.cuda.synchronize()
    gate = {"checked": True, "bit_identical_to_sync_fill": bool(torch.equal(Cd.view(torch.int32),
                                                                            Cs.view(torch.int32)))}
    del Cs
    if not gate["bit_identical_to_sync_fill"]:
        print(json.dumps({"error": "pipelined fill differs from the sync fill", "config": leg}), flush=True)
        return 1
    st, detail = pg.device_status()
    if st != 0:
        print(json.dumps({"error": f"device status {st} ({detail:#x})"}), flush=True)
        return 1

    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid else None)
    sampler.start()
    time.sleep(0.3)

    timer = CudaTimer()
    total_ms, per = timed_loop(dist, args.steps, args.warmup, call, flush, timer, torch.cuda.synchronize)
    st, detail = pg.device_status()
    if st != 0:
        sampler.stop()
        print(json.dumps({"error": f"device status {st} ({detail:#x}) after the timed loop"}), flush=True)
        return 1
    launches = args.steps * call.kernels
    SIDE_LAUNCHES["n"] = 0
    ms_step = total_ms / args.steps
    value = dist.world * flops * args.steps / (total_ms / 1e3) / 1e12
    local_mean = statistics.mean(per)
    achieved = flops / (local_mean / 1e3) / 1e12

    extras = {}
    if not args.no_extras and dist.rank == 0:
        if not is_bf16:
            fills = {}
            variants = [("sync", 1, 128), ("sync", 1, 64)]
            variants += [(f, s, 128) for f in ("cpasync", "tma", "cpasync_mbar", "cpasync_ws") for s in (2, 3, 4, 6)]
            variants += [("cpasync", 2, 64), ("tma", 2, 64), ("cpasync_mbar", 2, 64), ("cpasync_ws", 2, 64)]
            if w["lda"] % 4:
                variants = [v for v in variants if v[0] != "tma"]
            for f, s, t in variants:
                c = gemm_call(pg, name, Ad, Bd, Cd, f, s, t)
                mean, best, med = time_kernel(pg, c, flush, args.sweep_launches)
                fills[f"{f}/S{s}/T{t}"] = {"tflops": flops / (mean / 1e3) / 1e12, "ms": mean, "ms_min": best,
                                           "ms_median": med,
                                           "frac_fp32_peak": flops / (mean / 1e3) / 1e12 / fp32_peak}
            # The persistent TMA kernel without its split of the last round
            # of tiles (no hand-over workspace): same bits, SMs idle through
            # the partial last round.
            c = gemm_call(pg, name, Ad, Bd, Cd, "tma", 4, 128, workspace=None)
            mean, best, med = time_kernel(pg, c, flush, args.sweep_launches)
            fills["tma/S4/T128/unsplit"] = {"tflops": flops / (mean / 1e3) / 1e12, "ms": mean, "ms_min": best,
                                            "ms_median": med, "frac_fp32_peak": flops / (mean / 1e3) / 1e12 / fp32_peak}
            # Every row on 128 x 128 tiles (the wide-row kernel switched off
            # for these calls): same bits.
            if w["lda"] % 4 == 0:
                pg.testing_f32_wide(0)
                try:
                    for s in (2, 4):
                        c = gemm_call(pg, name, Ad, Bd, Cd, "tma", s, 128)
                        mean, best, med = time_kernel(pg, c, flush, args.sweep_launches)
                        fills[f"tma/S{s}/T128/no-wide"] = {
                            "tflops": flops / (mean / 1e3) / 1e12, "ms": mean, "ms_min": best, "ms_median": med,
                            "frac_fp32_peak": flops / (mean / 1e3) / 1e12 / fp32_peak}
                finally:
                    pg.testing_f32_wide(-1)
            t_sync = fills["sync/S1/T128"]["ms"]
            for v in fills.values():
                v["t_sync_over_t"] = t_sync / v["ms"]
            extras["fills"] = fills
            # The latency-bound tall-K shape on the one-warp 32x32 tile: one
            # CTA walks 4096 slices, so the fill's latency is the whole story.
            wt, At, Bt = load_workload("f32_tallk")
            Atd, Btd = to_device(At, wt["K"], dev), to_device(Bt, wt["N"], dev)
            Ctd = torch.empty((wt["M"], wt["N"]), dtype=torch.float32, device=dev)
            ft = 2.0 * wt["M"] * wt["N"] * wt["K"]
            tall = {}
            for f, s in (("sync", 1), ("cpasync", 2), ("cpasync", 4), ("cpasync", 6), ("tma", 2), ("tma", 4),
                         ("tma", 6), ("cpasync_mbar", 2), ("cpasync_mbar", 4), ("cpasync_mbar", 6),
                         ("cpasync_ws", 2), ("cpasync_ws", 4), ("cpasync_ws", 6)):
                c = gemm_call(pg, "f32_tallk", Atd, Btd, Ctd, f, s, 32)
                mean, best, med = time_kernel(pg, c, flush, args.sweep_launches)
                tall[f"{f}/S{s}/T32"] = {"us": mean * 1e3, "us_min": best * 1e3, "us_median": med * 1e3,
                                         "gflops": ft / (mean / 1e3) / 1e9}
            for v in tall.values():
                v["t_sync_over_t"] = tall["sync/S1/T32"]["us"] / v["us"]
            extras["tallk_32x32x65536"] = tall
            del Atd, Btd, Ctd
            # Every fill on the other FP32 workloads (the library's automatic
            # tile choice; TMA reads the ragged A repacked at lda = 1004).
            from async_copy_pipelined_gb300 import inputs as _inputs
            per_cfg = {}
            for wname in ("f32_256", "f32_1024", "f32_ragged"):
                wc, Ac, Bc = load_workload(wname)
                Acd, Bcd = to_device(Ac, wc["K"], dev), to_device(Bc, wc["N"], dev)
                A4d = Acd
                if wc["lda"] % 4:
                    A4d = to_device(_inputs.workload_operands(wname, lda=(wc["lda"] + 3) // 4 * 4)[0], wc["K"], dev)
                Ccd = torch.empty((wc["M"], wc["N"]), dtype=torch.float32, device=dev)
                fc = 2.0 * wc["M"] * wc["N"] * wc["K"]
                row = {}
                # The ragged shape is timed on both block tiles; the others on
                # the automatic choice.
                for t in ((128, 64) if wname == "f32_ragged" else (0,)):
                    sfx = f"/T{t}" if t else ""
                    for f, s in (("sync", 1), ("cpasync", 2), ("cpasync_mbar", 2), ("cpasync_ws", 4), ("tma", 2),
                                 ("tma", 4)):
                        c = gemm_call(pg, wname, A4d if f == "tma" else Acd, Bcd, Ccd, f, s, t)
                        mean, best, med = time_kernel(pg, c, flush, args.sweep_launches)
                        row[f"{f}/S{s}{sfx}"] = {"tflops": fc / (mean / 1e3) / 1e12, "us": mean * 1e3,
                                                 "us_min": best * 1e3, "us_median": med * 1e3}
                    for key, v in row.items():
                        if key.endswith(sfx) and (sfx or "/T" not in key):
                            v["t_sync_over_t"] = row[f"sync/S1{sfx}"]["us"] / v["us"]
                per_cfg[wname] = row
                del Acd, Bcd, A4d, Ccd
            extras["fills_per_workload"] = per_cfg
            # Cache qualifiers on the pipelined fills at 4096^3.
            co, n = time_cache_options(pg, name, Ad, Bd, Cd, [("cpasync", 4, 128), ("cpasync_mbar", 4, 128),
                                                               ("cpasync_ws", 4, 128), ("tma", 4, 128)], flush,
                                       args.sweep_launches, flops)
            extras["cache_options_f32_4096"] = co
            # BF16 tensor-core leg at its own full size.
            wb, Ab, Bb = load_workload("bf16_8192")
            Abd, Bbd = to_device(Ab, wb["K"], dev), to_device(Bb, wb["N"], dev)
            Cbd = torch.empty((wb["M"], wb["N"]), dtype=torch.float32, device=dev)
            fb = 2.0 * wb["M"] * wb["N"] * wb["K"]
            pb = pg.plan_bf16(wb["M"], wb["N"], wb["K"], lda=wb["lda"])
            cb = gemm_call(pg, "bf16_8192", Abd, Bbd, Cbd, "tma", pb["stages"], pb["block_m"])
            mean, best, med = time_kernel(pg, cb, flush, args.sweep_launches)
            tf = fb / (mean / 1e3) / 1e12
            roof_b = {"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": UNIT, "frac": tf / bf16_peak,
                      "traffic": profiled_traffic(f"bf16_8192:tma/S{pb['stages']}/T{pb['block_m']}"),
                      "peak_source": f"{peaks['_source']} cuBLAS bf16 burst"}
            if roof_b["traffic"]:
                hbm_b = float(peaks.get("hbm_gbs") or 0.0)
                roof_b["dram_gbs"] = roof_b["traffic"] / (mean / 1e3) / 1e9
                roof_b["dram_frac_of_hbm"] = roof_b["dram_gbs"] / hbm_b if hbm_b else None
            # The chip's dense BF16 peak derived from SM count x per-SM rate x
            # clock, at the maximum SM clock and at the clock sampled while
            # this kernel runs back to back (the tensor cores draw enough power
            # to lower it).
            bclk = clocks_during(cb, 1.0, sampler.uuid)
            bclk.pop("calls", None)
            check_status(pg, "the BF16 clock sample")
            derived = {"per_sm_per_clk": BF16_DENSE_FLOP_PER_SM_PER_CLK, "sms": num_sms,
                       "at_max_clock": {"mhz": sm_max, "tflops": bf16_derived_peak_tflops(num_sms, sm_max)},
                       "clocks_while_running": bclk}
            derived["at_max_clock"]["frac"] = tf / derived["at_max_clock"]["tflops"]
            if bclk.get("sm_mhz"):
                p_obs = bf16_derived_peak_tflops(num_sms, bclk["sm_mhz"])
                derived["at_sampled_clock"] = {"mhz": bclk["sm_mhz"], "tflops": p_obs, "frac": tf / p_obs}
            extras["bf16_8192"] = {"tflops": tf, "ms": mean, "ms_min": best, "ms_median": med,
                                   "stages": pb["stages"], "block_m": pb["block_m"], "roofline": roof_b,
                                   "derived_peak": derived}
            bfills = {}
            for f, s, t in (("tma", 2, 128), ("tma", 3, 128), ("tma", 4, 128), ("cpasync", 2, 128),
                            ("cpasync", 4, 128), ("sync", 1, 128), ("tma", 2, 256), ("tma", 3, 256),
                            ("cpasync", 2, 256), ("cpasync", 3, 256), ("sync", 1, 256)):
                c = gemm_call(pg, "bf16_8192", Abd, Bbd, Cbd, f, s, t)
                m2, b2, md2 = time_kernel(pg, c, flush, args.sweep_launches)
                bfills[f"{f}/S{s}/T{t}"] = {"tflops": fb / (m2 / 1e3) / 1e12, "ms": m2, "ms_min": b2,
                                            "ms_median": md2}
            for v in bfills.values():
                v["t_sync_over_t"] = bfills["sync/S1/T128"]["ms"] / v["ms"]
            extras["bf16_8192"]["fills"] = bfills
            # The TMA fill's opt-in K split of the last round (gemm_bf16_ws)
            # against the default unsplit call, both tiles; bits checked equal.
            bsplit = {}
            for t in (256, 128):
                pb_t = pg.plan_bf16(wb["M"], wb["N"], wb["K"], lda=wb["lda"], fill="tma", block_m=t)
                ref = None
                for label, ws in (("unsplit", None), ("split", "auto")):
                    c = gemm_call(pg, "bf16_8192", Abd, Bbd, Cbd, "tma", pb_t["stages"], t, workspace=ws)
                    c()
                    _count(c, 1)
                    torch.cuda.synchronize()
                    check_status(pg, f"BF16 {label} T{t}")
                    same = True
                    if ref is None:
                        ref = Cbd.clone()
                    else:
                        same = bool(torch.equal(Cbd.view(torch.int32), ref.view(torch.int32)))
                    m2, b2, md2 = time_kernel(pg, c, flush, args.sweep_launches)
                    bsplit[f"tma/S{pb_t['stages']}/T{t}/{label}"] = {"tflops": fb / (m2 / 1e3) / 1e12, "ms": m2,
                                                                    "ms_min": b2, "bits_equal_unsplit": same}
                del ref
            extras["bf16_8192"]["k_split"] = bsplit
            co, n = time_cache_options(pg, "bf16_8192", Abd, Bbd, Cbd, [("tma", 3, 256), ("cpasync", 3, 256)], flush,
                                       args.sweep_launches, fb)
            extras["cache_options_bf16_8192"] = co
            del Abd, Bbd, Cbd
    sampler.stop()
    clocks = sampler.summary()

    # End to end through the public API with host buffers: pinned H2D of A
    # and B, the GEMM, D2H of C, every step.
    e2e = None
    if dist.rank == 0 or dist.world > 1:
        Ah = torch.from_numpy(A if not is_bf16 else A.view(np.int16))
        Bh = torch.from_numpy(B if not is_bf16 else B.view(np.int16))
        if is_bf16:
            Ah, Bh = Ah.view(torch.bfloat16), Bh.view(torch.bfloat16)
        Ah = Ah.pin_memory()[:, :K]
        Bh = Bh.pin_memory()
        Ch = torch.empty((M, N), dtype=torch.float32).pin_memory()
        if is_bf16:
            host_call = lambda: pg.gemm_bf16(Ah, Bh, Ch, stages=leg["stages"], block_m=leg["tile"])  # noqa: E731
        else:
            host_call = lambda: pg.gemm_f32(Ah, Bh, Ch, fill=leg["fill"], stages=leg["stages"],  # noqa: E731
                                            block_tile=leg["tile"])
        e_steps = max(3, min(args.steps, 20))
        wt = WallTimer()
        # With several ranks: barrier + sync around exactly e_steps steps and
        # the max over ranks, like the device-timed leg; whole-job throughput
        # and bytes summed over the ranks.
        e_total, _ = timed_loop(dist if dist.world > 1 else _NoDist(), e_steps, 3, host_call, lambda: None, wt,
                                torch.cuda.synchronize)
        e2e = {"value": dist.world * flops / (e_total / e_steps / 1e3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": dist.world * int(Ah.element_size() * M * K + Bh.element_size() * K * N),
               "d2h_bytes_per_step": dist.world * int(4 * M * N), "ms_per_step": e_total / e_steps}
        # The GEMM launches of the host path, every step: BF16 row chunks; for
        # FP32 the executor's K steps over all rows and the last step's row
        # chunks (device copies at 16-byte row pitches).
        if is_bf16:
            per_step = len(pg.host_row_chunks(M, N, num_sms))
        else:
            kb, rb = pg.host_schedule_f32(M, N, K, num_sms)
            calls = [(M, k1 - k0) for k0, k1 in zip(kb[:-2], kb[1:-1])]
            calls += [(r1 - r0, kb[-1] - kb[-2]) for r0, r1 in zip(rb, rb[1:])]
            lda_d, ldb_d = -(-max(K, 1) // 4) * 4, -(-max(N, 1) // 4) * 4
            per_step = sum(f32_kernels_per_call(pg, m, N, k, lda_d, ldb_d, leg["fill"], leg["stages"], leg["tile"])
                           for m, k in calls)
        launches_e2e = e_steps * per_step

    kernel_key = f"{name}:{leg['fill']}/S{leg['stages']}/T{leg['tile']}"
    if is_bf16:
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": UNIT,
                "frac": achieved / bf16_peak, "traffic": profiled_traffic(kernel_key),
                "peak_source": f"{peaks['_source']} (MEASURED_PEAKS bf16_tflops, cuBLAS burst)",
                "derived_peak_at_max_clock": bf16_derived_peak_tflops(num_sms, sm_max),
                "frac_of_derived_peak_at_max_clock": achieved / bf16_derived_peak_tflops(num_sms, sm_max)}
        if clocks.get("sm_mhz"):
            roof["frac_of_derived_peak_at_observed_clock"] = achieved / bf16_derived_peak_tflops(num_sms,
                                                                                                 clocks["sm_mhz"])
    else:
        roof = {"bound": "alu", "achieved": achieved, "peak": fp32_peak, "unit": UNIT,
                "frac": achieved / fp32_peak, "traffic": profiled_traffic(kernel_key),
                "peak_source": f"{num_sms} SMs x {FP32_FMA_PER_SM_PER_CLK} FP32 FMA/clk x 2 x {sm_max:.0f} MHz "
                               f"({peaks['_source']} max SM clock)"}
        if clocks.get("sm_mhz"):
            roof["frac_at_observed_clock"] = achieved / fp32_peak_tflops(num_sms, clocks["sm_mhz"])
    # Diagnostic, not the bound: the DRAM rate the profiled traffic implies
    # at this launch's mean duration, against the measured copy bandwidth.
    if roof.get("traffic"):
        hbm = float(peaks.get("hbm_gbs") or 0.0)
        dram_gbs = roof["traffic"] / (local_mean / 1e3) / 1e9
        roof["dram_gbs"] = dram_gbs
        roof["dram_frac_of_hbm"] = dram_gbs / hbm if hbm else None

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        gpu_rows = Cd[: min(M, 4096)].cpu().numpy()
        cpu = oracle_sample(name, A, B, w, args.cpu_seconds, gpu_rows=gpu_rows)
        if not is_bf16:
            cpu["small_configs"] = oracle_small_configs()

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step,
        "step_ms": {"mean": local_mean, "median": statistics.median(per), "min": min(per)},
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in, f32 accumulate" if is_bf16 else "f32",
        "data": "synthetic (seeded SplitMix64 operands, see async_copy_pipelined_gb300/inputs.py)",
        "config": workload_config(name, w, {**leg, "gate": gate,
                                            "parallelism": "replicas" if dist.world > 1 else "single GPU"}),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches + SIDE_LAUNCHES["n"] + (launches_e2e if e2e else 0),
        "gpu_launches_breakdown": {"timed_steps": launches, "kernels_per_step": call.kernels,
                                   "sweep_and_bf16_legs": SIDE_LAUNCHES["n"],
                                   "e2e_launches": launches_e2e if e2e else 0},
        "kernel_sources_sha": kernel_sources_sha(),
    }
    line.update(extras)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


class _NoDist(Dist):
    def __init__(self):
        self.world, self.rank, self.local_rank, self.pg, self.device = 1, 0, 0, None, None


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="f32_4096",
                    choices=["f32_256", "f32_1024", "f32_4096", "f32_ragged", "f32_tallk", "bf16_8192"])
    ap.add_argument("--fill", choices=["sync", "cpasync", "tma", "cpasync_mbar", "cpasync_ws"], default=None)
    ap.add_argument("--stages", type=int, default=None)
    ap.add_argument("--tile", type=int, default=None)
    ap.add_argument("--sweep-launches", type=int, default=20)
    ap.add_argument("--no-extras", action="store_true", help="time only the main leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0, help="total oracle time budget for --impl reference")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        if world > 1 and rank != 0:
            return 0
        return run_reference(args, _NoDist())
    dist = Dist()
    try:
        return run_ours(args, dist)
    except DeviceStatusError as e:
        print(json.dumps({"error": str(e)}), flush=True)
        return 1
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
