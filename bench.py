#!/usr/bin/env python3
"""Benchmark of the fused GEMM + bias + ReLU (C = relu(A.B + bias)) on GB300.

One step = one fused GEMM launch over the workload's synthetic inputs, already
resident in HBM.  Prints ONE JSON line (rank 0):

  value        TFLOP/s = 2MNK / (mean device time of the step), summed over ranks
  e2e          the same through tgemm_run_host: host buffers (pinned), host->device
               copies, the GEMM and the device->host copy of C inside the timed region
  roofline     the fused kernel's achieved TFLOP/s (algorithmic 2MNK per launch over
               the CUDA-event launch time) against the measured dense bf16 peak
  cpu_baseline the fp64 CPU oracle on a bounded sample of rows of the same workload
  clocks       SM clocks and throttle reasons sampled during the timed region

--impl reference times the CPU oracle itself as the reference arm.
Multi-GPU (torchrun): every rank runs its own replica of the workload (weak
scaling, no collective on the data path); the timed region is bracketed by a
barrier and the max over ranks is reported.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import seeded_inputs as si  # noqa: E402

METRIC = "fused GEMM+bias+ReLU TFLOP/s (2MNK/t) on 1 GB300; % of dense fp16 tensor peak"
METRIC_GELU = "fused GEMM+bias+GELU TFLOP/s (2MNK/t) on 1 GB300; % of dense fp16 tensor peak"


def metric_for(w):
    return METRIC_GELU if "gelu" in w.epilogue else METRIC
DEFAULT_WORKLOAD = "c2"
FLUSH_BYTES = 256 << 20            # > 2x the 129 MB L2
L2_NOTE = ("flushed between steps (256 MiB written, then read back so that no dirty line of it is "
           "left to write back during the launch; outside the timed launch)")


class L2Flush:
    """Between timed launches: write a 256 MiB buffer (every line of the inputs
    leaves L2), then read it back, so that the lines it leaves are clean.  A
    write alone leaves about 129 MB of dirty lines, whose write-back then runs
    inside the next timed launch (14 us of the HBM-bound skinny workload's 92)."""

    def __init__(self, dev):
        self.buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.zero_()
        torch.sum(self.buf, 0, out=self.sink)
# Sources that decide the device code of each kernel family (the host file
# holds both families' launch code); a recorded DRAM traffic figure stands only
# while these are unchanged.
_CSRC = "gemm_epilogue_02_gb300/csrc/"
KERNEL_SOURCES = {
    "gemm": [_CSRC + f for f in ("gemm_kernel.cuh", "ptx.cuh", "aux_kernels.cuh", "bytes.cuh", "tgemm_api.cu")],
    "attention": [_CSRC + f for f in ("attn_kernel.cuh", "gemm_kernel.cuh", "ptx.cuh", "tgemm_api.cu")],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def kernel_hash(family: str = "gemm") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    """Roofline denominators: the measured dense bf16 burst and sustained
    TFLOP/s and HBM copy GB/s, else the fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"tflops": float(d["bf16_tflops"]), "hbm": float(d["hbm_gbs"]), "kind": "measured",
                "tflops_sustained": float(d["bf16_tflops_sustained"]) if "bf16_tflops_sustained" in d else None}
    except (OSError, KeyError, ValueError):
        return {"tflops": 1900.0, "hbm": 6800.0, "kind": "fallback", "tflops_sustained": 1700.0}


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel is unchanged."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(workload)
        family = "attention" if workload in si.ATTN_WORKLOADS else "gemm"
        if e and e.get("kernel_hash") == kernel_hash(family):
            return float(e["dram_bytes_per_launch"])
    except (OSError, ValueError):
        pass
    return None


class ClockSampler:
    """nvidia-smi sampling (every 20 ms) of SM clocks and throttle reasons.

    Started before the load soak that precedes the timed region; mark() notes
    when the timed region starts and ends, and summary() uses the samples taken
    inside it (or, when the timed region is shorter than a few sampling
    periods, those of the soak + timed window, and says so)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = None
        self.t_start = self.t_end = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def _ts(text):
        from datetime import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10 and parts[2].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if (t := self._ts(r[0])) is not None and self.t_start is not None
                  and self.t_start <= t <= self.t_end]
        window = "timed region"
        if len(inside) < 3:
            inside = [r for r in rows if (t := self._ts(r[0])) is not None and self.t_end is not None
                      and t <= self.t_end] or rows
            window = "load soak + timed region (timed region shorter than 3 samples)"
        sm = [float(r[2]) for r in inside]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        pw = [float(r[4]) for r in inside if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(inside[0][3]),
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max(pw) if pw else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class OracleSample:
    """The fp64 oracle (as it stands) on the first rows of a workload.  Each call
    decodes all of B once (serially) before the rows run in parallel, so a call
    costs a fixed part plus a part per row; `fixed_s` (a one-row call) is
    reported beside every figure so the two CPU legs can be read together."""

    def __init__(self, w):
        import oracle
        self.w = w
        A, B, bias = si.make_workload(w)
        self.args = (si.bits(A), si.bits(B), si.bits(bias) if bias is not None else None)
        self.epi = si.EPILOGUES[w.epilogue]
        self.dt = oracle.dtype_code(w.dtype)
        self.cores = oracle.max_threads()
        self.fixed_s = self.time(1)

    def time(self, rows_n: int) -> float:
        import oracle
        w = self.w
        t0 = time.perf_counter()
        oracle.gemm_epilogue_f64(*self.args, w.M, w.N, w.K, self.dt, self.epi, rows=list(range(rows_n)))
        return time.perf_counter() - t0

    def calibrate(self, target_s: float):
        """Rows for one call of about target_s seconds (or all rows); returns (rows, seconds)."""
        rows_n = min(self.w.M, max(self.cores, 1))
        while True:
            t = self.time(rows_n)
            if t >= 0.5 * target_s or rows_n >= self.w.M:
                return rows_n, t
            var = t - self.fixed_s
            if var < 0.25 * self.fixed_s:      # the per-row part is still lost in the fixed part's noise
                rows_n = min(self.w.M, rows_n * 4)
                continue
            want = int(rows_n * max(target_s - self.fixed_s, var) / var)
            rows_n = int(min(self.w.M, max(rows_n + 1, want)))

    def tflops(self, rows_n: int, t: float) -> float:
        return 2.0 * rows_n * self.w.N * self.w.K / t / 1e12

    def sample_text(self, rows_n: int, per: str = "") -> str:
        w = self.w
        return (f"first {rows_n} of {w.M} rows of {w.name}{per} (all {w.N} columns, K={w.K}), fp64; "
                f"each call first decodes all of B serially ({self.fixed_s:.2f} s, a one-row call)")


def cpu_oracle_sample(w, target_s: float):
    """Time the oracle on a bounded sample of rows (one call of about target_s seconds)."""
    o = OracleSample(w)
    rows_n, t = o.calibrate(target_s)
    return {"value": o.tflops(rows_n, t), "unit": "TFLOP/s", "cores": o.cores, "kind": "oracle",
            "seconds": round(t, 3), "fixed_s": round(o.fixed_s, 3), "sample": o.sample_text(rows_n)}


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle on a bounded sample per step (rank 0 only).
    The sample is sized like the CPU-baseline leg's, capped so that the warm-up
    and timed steps together take about two and a half minutes."""
    if rank != 0:
        return 0
    w = si.WORKLOADS[args.config]
    o = OracleSample(w)
    per_step = min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup))
    rows_n, _ = o.calibrate(per_step)
    for _ in range(args.warmup):
        o.time(rows_n)
    times = [o.time(rows_n) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = o.tflops(rows_n, t)
    line = {"impl": "reference", "metric": metric_for(w), "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": o.cores, "kind": "oracle",
                             "fixed_s": round(o.fixed_s, 3), "sample": o.sample_text(rows_n, " per step")},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


METRIC_ATTN = "attention forward TFLOP/s (4*B*H*S^2*D, half when causal) on 1 GB300; % of dense fp16 tensor peak"


def attn_config(w):
    return {"workload": w.name, "batch": w.B, "seq_len": w.S, "heads": w.H, "head_dim": w.D, "dtype": w.dtype,
            "causal": w.causal, "layout": "[batch, seq, heads, dim]", "inputs": "Q, K, V ~N(0,1)", "seed": w.seed,
            "l2": L2_NOTE}


def attn_oracle_rows(w, q, k, v, nrows):
    import oracle
    total = w.B * w.S * w.H
    rows = [int(r) for r in (np.arange(nrows) * (total // max(nrows, 1))) % total]
    b = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle.attention_f64(b(q), b(k), b(v), w.B, w.S, w.H, w.D, w.causal, oracle.dtype_code(w.dtype), rows=rows)
    return time.perf_counter() - t0, rows


def attn_cpu_sample(w, q, k, v, target_s):
    """The fp64 attention oracle on a bounded, spread sample of query rows,
    growing until one run takes about target_s seconds."""
    import oracle
    total = w.B * w.S * w.H
    n = min(total, 256)
    while True:
        t, rows = attn_oracle_rows(w, q, k, v, n)
        if t >= 0.5 * target_s or n >= total:
            break
        n = int(min(total, max(2 * n, n * target_s / max(t, 1e-6))))
    per_row = 4.0 * w.S * w.D * (0.5 if w.causal else 1.0)   # average flops of one query row
    return {"value": per_row * len(rows) / t / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle", "seconds": round(t, 3),
            "sample": f"{len(rows)} of {total} query rows of {w.name} (spread over batch, heads, positions), fp64"}


def run_attention_bench(args, world, rank, local):
    import gemm_epilogue_02_gb300 as tg
    tg.load()
    w = si.ATTN_WORKLOADS[args.config]
    dev = torch.device("cuda", local)
    q, k, v = si.make_attention_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    od = torch.empty_like(qd)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(dev)

    def step():
        tg.attention(qd, kd, vd, od, causal=w.causal, stream=stream)

    launch_ms, t_wall, clk = timed_steps(step, flush, args, dev, stream, world, local)
    mean_ms, launch_stats = launch_summary(launch_ms, t_wall, args.steps)
    mean_ms_max = max_over_ranks(mean_ms, world)
    value = world * w.flops / (mean_ms_max * 1e-3) / 1e12

    e2e = None
    if not args.no_e2e:
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        oh = torch.empty_like(qh).pin_memory()

        def host_step():
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            tg.attention(qd, kd, vd, od, causal=w.causal, stream=stream)
            oh.copy_(od, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup)):
                host_step()
            torch.cuda.synchronize(dev)
            n_e2e = max(3, min(args.steps, 50))
            es = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
            ee = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
            barrier(world)
            for i in range(n_e2e):
                es[i].record(stream)
                host_step()
                ee[i].record(stream)
            torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(es, ee)) / n_e2e, world)
        e2e = {"value": world * w.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": 3 * qh.numel() * 2, "d2h_bytes_per_step": oh.numel() * 2,
               "ms_per_step": e2e_ms, "steps": n_e2e, "host_memory": "pinned"}

    status = tg.tgemm_last_device_status()
    if rank != 0:
        return 0 if status == 0 else 1
    peaks = measured_peaks()
    peak, peak_kind = peaks["tflops"], peaks["kind"]
    achieved = w.flops / (mean_ms * 1e-3) / 1e12
    line = {"metric": METRIC_ATTN, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup_done, "ms_per_step": mean_ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": attn_config(w),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(args.config),
                         "peak_source": f"{peak_kind} dense bf16 burst (fp16 nominal rate is equal)",
                         "kernel": "attn_fwd_kernel", "algorithmic_flops_per_launch": w.flops,
                         "algorithmic_bytes_per_launch": 4 * w.B * w.S * w.H * w.D * 2},
            "clocks": clk.summary(), "gpu_launches": args.steps, "launch_us": launch_stats,
            "device_status": tg.tgemm_status_string(status), "wall_s_timed_region": t_wall}
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = attn_cpu_sample(w, q, k, v, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0 if status == 0 else 1


def run_attention_reference(args, world, rank):
    """Reference arm for the attention workloads: the fp64 oracle on a bounded
    row sample per step (rank 0 only)."""
    if rank != 0:
        return 0
    import oracle
    w = si.ATTN_WORKLOADS[args.config]
    q, k, v = si.make_attention_inputs(w)
    nrows = max(1, args.ref_rows)
    for _ in range(args.warmup):
        attn_oracle_rows(w, q, k, v, nrows)
    times = [attn_oracle_rows(w, q, k, v, nrows)[0] for _ in range(args.steps)]
    t = sum(times) / len(times)
    per_row = 4.0 * w.S * w.D * (0.5 if w.causal else 1.0)
    value = per_row * nrows / t / 1e12
    sample = f"{nrows} of {w.B * w.S * w.H} query rows of {w.name} per step, fp64"
    line = {"impl": "reference", "metric": METRIC_ATTN, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": attn_config(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dtype": w.dtype,
            "epilogue": w.epilogue, "lda": w.lda or w.K, "ldb": w.ldb or w.N, "ldc": w.ldc or w.N,
            "inputs": {"normal": "A~N(0,1), B~N(0,1)/sqrt(K), bias~N(0,0.1)",
                       "gelu": "A, B ~N(0,1)/K^(1/4), bias~N(0,1)",
                       "int": "uniform integers in {-2..2}"}[w.kind], "seed": w.seed,
            "l2": L2_NOTE}


def timed_steps(step, flush, args, dev, stream, world, local):
    """Warm-up (at least W steps and args.soak seconds), then args.steps timed
    steps bracketed by barriers, each launch timed with CUDA events on `stream`
    and L2 flushed before it.  Returns (launch ms list, wall seconds, clocks)."""
    with torch.cuda.stream(stream), ClockSampler(local) as clk:
        # The first step carries one-time costs (kernel loading, the flush's
        # first reduction): the soak's clock starts once it has finished.
        flush()
        step()
        torch.cuda.synchronize(dev)
        t_soak = time.perf_counter()
        done = 1
        while done < args.warmup or time.perf_counter() - t_soak < args.soak:
            flush()
            step()
            done += 1
            if done % 64 == 0:
                torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        args.warmup_done = done
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        clk.mark_start()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
        clk.mark_end()
        barrier(world)
    return [a.elapsed_time(b) for a, b in zip(starts, ends)], t_wall, clk


def launch_summary(launch_ms, t_wall, steps):
    srt = sorted(launch_ms)
    pct = lambda f: srt[min(len(srt) - 1, int(f * len(srt)))] * 1e3
    mean_ms = sum(launch_ms) / len(launch_ms)
    return mean_ms, {"mean": mean_ms * 1e3, "p10": pct(0.1), "p50": pct(0.5), "p90": pct(0.9),
                     "max": srt[-1] * 1e3, "wall_per_step": t_wall / steps * 1e6}


def gemm_buffers(w, dev):
    """The workload's seeded inputs on the host and their device copies (C with
    the workload's pitch)."""
    A, B, bias = si.make_workload(w)
    ldc = w.ldc or w.N
    Ad = A.to(dev)[:, : w.K]
    Bd = B.to(dev)[:, : w.N]
    bd = bias.to(dev) if bias is not None else None
    Cd = torch.empty((w.M, ldc), dtype=A.dtype, device=dev)[:, : w.N]
    return (A, B, bias), (Ad, Bd, bd, Cd)


def check_rows(M: int) -> list:
    """One row of every 128-row block of C (a different offset in each block),
    plus the first and the last row."""
    rows = {min(M - 1, b * 128 + (b * 37) % 128) for b in range((M + 127) // 128)}
    return sorted(rows | {0, M - 1})


def check_output(w, inputs, Cd):
    """Compare sampled rows of the timed launch's C (every column) with the fp64
    oracle: the method's bounds (relative Frobenius <= 2e-3, per element
    |err| <= 1e-2 + 1e-2 |ref|), bit-exactness for integer inputs."""
    import oracle
    A, B, bias = inputs
    rows = check_rows(w.M)
    got_bits = Cd[rows].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    dt = oracle.dtype_code(w.dtype)
    ref = oracle.gemm_epilogue_f64(si.bits(A), si.bits(B), si.bits(bias) if bias is not None else None,
                                   w.M, w.N, w.K, dt, si.EPILOGUES[w.epilogue], rows=rows)
    got = oracle.decode(got_bits, dt)
    err = np.abs(got - ref)
    frob = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-12))
    elem = float(np.max(err / (1e-2 + 1e-2 * np.abs(ref)))) if err.size else 0.0
    out = {"rows": len(rows), "cols": w.N, "rows_sampled": "one per 128-row block + first + last",
           "max_abs_err": float(err.max()) if err.size else 0.0, "frobenius_rel": frob,
           "max_err_over_elem_bound": elem, "within_bound": bool(frob <= 2e-3 and elem <= 1.0)}
    if w.kind == "int":
        want = oracle.round_to(ref, dt)
        zero = (want & 0x7FFF) == 0          # +-0 compare equal (exact zero sums may carry either sign)
        same = (got_bits == want) | (zero & ((got_bits & 0x7FFF) == 0))
        out["bit_exact"] = bool(same.all())
        out["within_bound"] = out["within_bound"] and out["bit_exact"]
    return out


def gemm_roofline(w, mean_ms, peaks, bound=None):
    """The roofline that bounds a launch: the tensor pipe (2MNK flops at the
    measured dense peak) or HBM (its algorithmic bytes at the measured copy
    bandwidth), whichever takes longer; `bound` forces one.  For the skinny,
    weight-bound shape the algorithmic bytes are B alone (the weight stream)."""
    flops = float(w.flops)
    skinny = w.M <= 256 and w.N * w.K >= 64 * w.M * max(w.N, w.K)
    alg_bytes = w.K * w.N * 2 if skinny else (w.M * w.K + w.K * w.N + w.M * w.N + w.N) * 2
    if bound is None:
        bound = "hbm" if alg_bytes / (peaks["hbm"] * 1e9) > flops / (peaks["tflops"] * 1e12) else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": alg_bytes / (mean_ms * 1e-3) / 1e9, "peak": peaks["hbm"],
                "unit": "GB/s", "peak_source": f"{peaks['kind']} HBM copy bandwidth",
                "algorithmic_bytes": "B (K x N x 2 bytes): the weight stream" if skinny
                else "A + B + C + bias, once each"}
    else:
        roof = {"bound": "tensor", "achieved": flops / (mean_ms * 1e-3) / 1e12, "peak": peaks["tflops"],
                "unit": "TFLOP/s", "peak_source": f"{peaks['kind']} dense bf16 burst (fp16 nominal rate is equal)"}
        if peaks.get("tflops_sustained"):
            roof["peak_sustained"] = peaks["tflops_sustained"]
            roof["frac_sustained"] = roof["achieved"] / peaks["tflops_sustained"]
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof.update(kernel="tgemm_fused_kernel", algorithmic_flops_per_launch=flops,
                algorithmic_bytes_per_launch=alg_bytes)
    return roof


def run_tgemm_bench(args, world, rank, local):
    import gemm_epilogue_02_gb300 as tg
    tg.load()
    w = si.WORKLOADS[args.config]
    dev = torch.device("cuda", local)
    inputs, (Ad, Bd, bd, Cd) = gemm_buffers(w, dev)
    A, B, bias = inputs
    ldc = w.ldc or w.N
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(dev)
    flops = float(w.flops)

    def step():
        tg.run(Ad, Bd, bd, Cd, w.epilogue, stream=stream)

    launch_ms, t_wall, clk = timed_steps(step, flush, args, dev, stream, world, local)
    mean_ms, launch_stats = launch_summary(launch_ms, t_wall, args.steps)
    mean_ms_max = max_over_ranks(mean_ms, world)
    value = world * flops / (mean_ms_max * 1e-3) / 1e12
    torch.cuda.synchronize(dev)
    check = check_output(w, inputs, Cd) if not args.no_check else None

    # End to end through the host-buffer entry point (pinned host memory).
    e2e = None
    if not args.no_e2e:
        Ah, Bh = A.pin_memory(), B.pin_memory()
        bh = bias.pin_memory() if bias is not None else None
        Ch = torch.empty((w.M, ldc), dtype=A.dtype).pin_memory()
        Chv = Ch[:, : w.N]
        Ahv, Bhv = Ah[:, : w.K], Bh[:, : w.N]
        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup)):
                tg.run_host(Ahv, Bhv, bh, Chv, w.epilogue, stream=stream, device=dev)
            torch.cuda.synchronize(dev)
            n_e2e = max(3, min(args.steps, 20))
            es = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
            ee = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
            barrier(world)
            for i in range(n_e2e):
                es[i].record(stream)
                tg.run_host(Ahv, Bhv, bh, Chv, w.epilogue, stream=stream, device=dev)
                ee[i].record(stream)
            torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(es, ee)) / n_e2e, world)
        h2d = (w.M * w.K + w.K * w.N + (w.N if bias is not None else 0)) * 2
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": w.M * w.N * 2,
               "ms_per_step": e2e_ms, "steps": n_e2e, "host_memory": "pinned"}
        del Ah, Bh, bh, Ch

    # The other graded shapes, timed with the same protocol in the same run.
    extras = {}
    if not args.no_extras and args.config == DEFAULT_WORKLOAD:
        extras["skinny"] = sub_record("c3", args, dev, stream, flush, world, local, check=not args.no_check)
        extras["decode"] = sub_record("d16", args, dev, stream, flush, world, local, check=not args.no_check)
        extras["launch_bound"] = launch_bound_record("c0", args, dev, stream)

    status = tg.tgemm_last_device_status()
    if rank != 0:
        return 0 if status == 0 else 1

    peaks = measured_peaks()
    roof = gemm_roofline(w, mean_ms, peaks)
    roof["traffic"] = recorded_traffic(args.config)
    clocks = clk.summary()
    line = {"metric": metric_for(w), "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup_done, "ms_per_step": mean_ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": workload_config(w),
            "roofline": roof,
            "clocks": clocks,
            "gpu_launches": args.steps * launches_per_call(w),
            "launch_us": launch_stats,
            "device_status": tg.tgemm_status_string(status),
            "wall_s_timed_region": t_wall}
    if clocks.get("sm_mhz"):
        # Work per SM clock: the same launch read against the clock it ran at.
        line["tflop_per_ghz"] = roof["achieved"] / (clocks["sm_mhz"] / 1e3) if roof["bound"] == "tensor" else None
    if check is not None:
        line["check"] = check
    if e2e is not None:
        line["e2e"] = e2e
    line.update(extras)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    ok = status == 0 and (check is None or check["within_bound"])
    ok = ok and all(r.get("check", {}).get("within_bound", True) for r in extras.values())
    return 0 if ok else 1


def launches_per_call(w) -> int:
    """Kernels one tgemm_run call of the workload launches: the fused GEMM, plus
    one repack per operand whose pitch is not a multiple of 8 elements."""
    return 1 + (1 if (w.lda or w.K) % 8 else 0) + (1 if (w.ldb or w.N) % 8 else 0)


def sub_record(name, args, dev, stream, flush, world, local, check=True):
    """Another graded workload timed with the main line's protocol (warm-up and
    soak, L2 flushed before each timed launch, CUDA events on the launch stream)."""
    import gemm_epilogue_02_gb300 as tg
    w = si.WORKLOADS[name]
    inputs, (Ad, Bd, bd, Cd) = gemm_buffers(w, dev)

    def step():
        tg.run(Ad, Bd, bd, Cd, w.epilogue, stream=stream)

    sub = argparse.Namespace(**vars(args))
    launch_ms, t_wall, clk = timed_steps(step, flush, sub, dev, stream, world, local)
    mean_ms, stats = launch_summary(launch_ms, t_wall, sub.steps)
    mean_ms = max_over_ranks(mean_ms, world)
    torch.cuda.synchronize(dev)
    peaks = measured_peaks()
    roof = gemm_roofline(w, mean_ms, peaks)
    roof["traffic"] = recorded_traffic(name)
    rec = {"workload": w.name, "config": workload_config(w), "ms_per_step": mean_ms,
           "value": world * w.flops / (mean_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "steps": sub.steps,
           "warmup": sub.warmup_done, "roofline": roof, "clocks": clk.summary(), "launch_us": stats,
           "gpu_launches": sub.steps * launches_per_call(w)}
    if check:
        rec["check"] = check_output(w, inputs, Cd)
    return rec


def launch_bound_record(name, args, dev, stream, reps=1000):
    """The launch-bound workload: `reps` back-to-back calls (no flush; its
    operands are 256 KiB).  Reports the device time per launch (CUDA events
    around the whole burst) and the host time per tgemm_run call."""
    import gemm_epilogue_02_gb300 as tg
    w = si.WORKLOADS[name]
    _, (Ad, Bd, bd, Cd) = gemm_buffers(w, dev)
    with torch.cuda.stream(stream):
        for _ in range(50):
            tg.run(Ad, Bd, bd, Cd, w.epilogue, stream=stream)
        torch.cuda.synchronize(dev)
        # Host cost per call while the GPU keeps up (the queue stays short).
        t_host = []
        for _ in range(reps):
            t0 = time.perf_counter()
            tg.run(Ad, Bd, bd, Cd, w.epilogue, stream=stream)
            t_host.append(time.perf_counter() - t0)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(reps):
            tg.run(Ad, Bd, bd, Cd, w.epilogue, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
    dev_us = e0.elapsed_time(e1) * 1e3 / reps
    t_host.sort()
    return {"workload": w.name, "config": workload_config(w) | {"l2": "not flushed (launch-bound burst)"},
            "reps": reps, "device_us_per_launch": dev_us, "wall_us_per_call": wall / reps * 1e6,
            "host_us_per_call_p50": t_host[len(t_host) // 2] * 1e6,
            "host_us_per_call_p90": t_host[int(0.9 * len(t_host))] * 1e6,
            "value": w.flops / (dev_us * 1e-6) / 1e12, "unit": "TFLOP/s",
            "note": "python binding + C ABI; the library's own host cost is the C part of each call"}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["tgemm", "reference"], default="tgemm")
    ap.add_argument("--config", default=DEFAULT_WORKLOAD, choices=sorted(si.WORKLOADS) + sorted(si.ATTN_WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-check", action="store_true", help="skip the oracle check of the timed output")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the skinny, decode and launch-bound sub-records of the default line")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--soak", type=float, default=1.0, help="minimum seconds of warm-up steps")
    ap.add_argument("--ref-rows", type=int, default=64, help="attention oracle query rows per reference step")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)          # at least 3 untimed warm-up steps
    world, rank, local = dist_setup()
    attn = args.config in si.ATTN_WORKLOADS
    if args.impl == "reference":
        rc = run_attention_reference(args, world, rank) if attn else run_reference(args, world, rank)
    else:
        rc = run_attention_bench(args, world, rank, local) if attn else run_tgemm_bench(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
