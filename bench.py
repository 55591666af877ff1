"""Benchmark of the GB300 SGEMM library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--mode auto|fp32|3xtf32|tf32]
                    [--impl ours|reference] [--no-extra]

One step = one SGEMM C = alpha*A@B + beta*C at M = N = K = 4092 (fp32,
row-major, A and B ~ N(0,1) from seed 2, alpha = 1, beta = 0: the benchmark
shape of "From 1% to 94% of cuBLAS, one kernel at a time") through the C ABI,
inputs resident in HBM.  L2 is flushed (a 2 x L2-sized write) between timed
steps, outside the timed events.  Each rank runs its own replica (weak
scaling; no data-path collective); `value` is the FLOPs of all ranks divided
by the slowest rank's time.

Rank 0 prints one JSON line with the metric, the roofline of the dominant
kernel, the oracle timed on the host cores (cpu_baseline), an end-to-end
figure with host buffers (e2e), the clocks seen during the timed region, and
per-path and batched-GEMM figures.

--impl reference times the CPU oracle (the only reference this library has)
on a bounded row sample of the same workload, on rank 0 only.
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

METRIC = "SGEMM TFLOP/s at M=N=K=4092 fp32 (and % of roofline); BMM TFLOP/s"
UNIT = "TFLOP/s"
WORKLOAD = "sgemm_4092"
# Fallbacks when the driver-written measured peaks are absent.
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}
# Dense tensor-core throughput ratio tf32 : bf16, nominal 1 : 2 (1.125 : 2.25
# PFLOP/s per GPU; tables that print the tf32 figure as 1.1 round it).
TF32_PER_BF16 = 1.0 / 2.0
FP32_LANES_PER_SM = 128


def gemm_flops(M, N, K, Q=1):
    """2*M*N*K*Q: one multiply and one add per term of every dot product
    (the pages' 137 GFLOP for 4092^3)."""
    return 2.0 * M * N * K * Q


def naive_read_bytes(M, N, K):
    """Bytes a kernel with no data reuse reads: two fp32 loads per
    multiply-add (the pages' 548 GB for 4092^3)."""
    return 2.0 * 4 * M * N * K


def compulsory_bytes(M, N, K, Q=1, beta_nonzero=False):
    """Minimum HBM traffic: read A and B once, write C (and read it if beta != 0)."""
    return 4.0 * Q * (M * K + K * N + M * N * (2 if beta_nonzero else 1))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def roofline_peak(mode, num_sms, peaks, source):
    """(bound, peak TFLOP/s, note) of a contraction path."""
    if mode == "fp32":
        mhz = float(peaks.get("sm_max_mhz", FALLBACK_PEAKS["sm_max_mhz"]))
        peak = num_sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
        return "alu", peak, (f"FP32 FFMA peak: {num_sms} SMs x {FP32_LANES_PER_SM} lanes x 2 "
                             f"x {mhz:.0f} MHz max SM clock")
    tf32 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * TF32_PER_BF16
    if mode == "3xtf32":
        return "tensor", tf32 / 3.0, (f"tf32 tensor peak ({source} bf16 burst x the nominal "
                                      f"tf32:bf16 ratio 1/2) / 3 passes; credited 2MNK")
    return "tensor", tf32, f"tf32 tensor peak ({source} bf16 burst x the nominal ratio 1/2)"


# Sources of the kernels a benchmark call runs and of the host code that
# plans them; the probes, the host-buffer entry point and the allocation-free
# entry point are left out (they do not change what the timed kernels do).
TIMED_SOURCES = ("api.cu", "common.cuh", "internal.h", "kernels_simt.cu", "kernels_tc.cu",
                 "kernels_tcp.cu", "params.h", "planes.cu", "raw.cu", "repack.cu",
                 "simt_fp32.cuh", "tc_direct.cuh", "tc_pair.cuh", "tc_ss.cuh", "tc_tf32.cuh",
                 "tune_table.h")


def kernel_source_hash():
    h = hashlib.sha256()
    for name in TIMED_SOURCES:
        with open(os.path.join(ROOT, "dense_fp32_matrix_03_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key):
    """Per-launch DRAM bytes from the committed ncu summary, or None when the
    kernel sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while active."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        for r in rows:
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), r[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


# ------------------------------------------------------------ distributed

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value, world, device=None):
    """Max of a float over ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value, world, device=None):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ oracle

def cpu_baseline(w, target_s=10.0):
    """The oracle, as it stands, on a bounded row sample of workload w on the
    host cores.  Returns the cpu_baseline object (value in TFLOP/s)."""
    import numpy as np
    import oracle
    M, N, K = w["M"], w["N"], w["K"]
    A, B, C0 = w["A"], w["B"], w["C0"]
    beta = w["betas"][0]

    def run(nrows):
        rows = [(0, int(i)) for i in np.linspace(0, M - 1, nrows).astype(int)]
        t0 = time.perf_counter()
        oracle.sgemm_ref(M, N, K, w["alpha"], A, K, B, N, beta, C0, N, rows=rows)
        return time.perf_counter() - t0

    t = run(8)
    rate = 8 / max(t, 1e-6)
    nrows = int(min(M, max(8, rate * target_s)))
    t = run(nrows)
    flops = gemm_flops(nrows, N, K)
    return {"value": flops / t / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(t, 3),
            "sample": f"{nrows} of {M} output rows of the {M}x{N}x{K} problem "
                      f"(fp64 accumulation, {2 * N * K / 1e6:.1f} MFLOP per row)"}


def reference_arm(args, rank, world):
    """--impl reference: the oracle timed per step on the host cores."""
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    import workloads
    oracle.build()
    w = workloads.make(WORKLOAD)
    M, N, K = w["M"], w["N"], w["K"]
    steps, warmup = args.steps, args.warmup
    budget = 150.0  # seconds for the whole run
    per_step = budget / max(1, steps + warmup)
    # calibrate rows per step
    rows8 = [(0, int(i)) for i in range(8)]
    t0 = time.perf_counter()
    oracle.sgemm_ref(M, N, K, w["alpha"], w["A"], K, w["B"], N, 0.0, None, N, rows=rows8)
    rate = 8 / max(time.perf_counter() - t0, 1e-6)
    nrows = int(min(M, max(1, rate * per_step)))
    rng = np.random.default_rng(0)
    times = []
    for s in range(warmup + steps):
        rows = [(0, int(i)) for i in rng.choice(M, nrows, replace=False)]
        t0 = time.perf_counter()
        oracle.sgemm_ref(M, N, K, w["alpha"], w["A"], K, w["B"], N, 0.0, None, N, rows=rows)
        dt = time.perf_counter() - t0
        if s >= warmup:
            times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = gemm_flops(nrows, N, K) / (ms / 1e3) / 1e12
    sample = (f"{nrows} random output rows of the {M}x{N}x{K} problem per step "
              f"(fp64 accumulation)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "alpha": 1.0, "beta": 0.0,
                   "inputs": "normal(0,1) seed 2", "device": "host cores"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- GPU arm

def time_calls(call, steps, warmup, stream, flush, lib=None):
    """Per-step CUDA-event times (ms) on `stream`, L2 flushed before each
    (flush=None: not flushed, the warm-L2 variant);
    with `lib`, also the library's kernel launches during the timed steps."""
    import torch
    for _ in range(warmup):
        if flush is not None:
            flush.zero_()
        call()
    torch.cuda.synchronize()
    evs = []
    n0 = lib.sgemm_kernel_launches() if lib is not None else 0
    for _ in range(steps):
        if flush is not None:
            flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    if lib is None:
        return times
    return times, lib.sgemm_kernel_launches() - n0


# Probe iterations: about a millisecond each on a GB300.
PROBE_ITERS = {"ffma": 2048, "ffma2": 2048, "tf32_ss": 16384, "tf32_ts": 16384,
               "bf16_ss": 16384}
PROBE_FOR = {"fp32": "max(ffma, ffma2)", "3xtf32": "tf32_ts / 3 (three MMAs per k step)",
             "tf32": "tf32_ts"}


def peak_probes(lib, stream, reps=5):
    """Median TFLOP/s of each throughput probe (a path's arithmetic with no
    operand traffic), after one warm-up launch, with CUDA events on `stream`."""
    import torch
    out = {}
    for kind, iters in PROBE_ITERS.items():
        st, flops = lib.sgemm_peak_probe(kind, iters, stream)
        if st != lib.SGEMM_OK:
            out[kind] = None
            continue
        evs = []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            lib.check(lib.sgemm_peak_probe(kind, iters, stream)[0])
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        out[kind] = flops / (ms / 1e3) / 1e12
    lib.check(lib.sgemm_poll_error(stream))
    return out


def probe_peak_for(mode, probes):
    """The probe figure a path's roofline fraction is also set against."""
    if not probes:
        return None
    if mode == "fp32":
        vals = [v for v in (probes.get("ffma"), probes.get("ffma2")) if v]
        return max(vals) if vals else None
    ts = probes.get("tf32_ts")
    if not ts:
        return None
    return ts / 3.0 if mode == "3xtf32" else ts


def resolve_mode(lib, requested):
    if requested != "auto":
        return requested
    import torch
    a = torch.ones(16, 16, device="cuda")
    c = torch.zeros(16, 16, device="cuda")
    st = lib.sgemm_batched_ex("3xtf32", 16, 16, 16, 1.0, a, 16, a, 16, 0.0, c, 16, 0, 0, 0, 0,
                              0, 1)
    torch.cuda.synchronize()
    return "3xtf32" if st == lib.SGEMM_OK else "fp32"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="auto", choices=["auto", "fp32", "3xtf32", "tf32"])
    ap.add_argument("--no-extra", action="store_true", help="skip per-path and BMM figures")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline")
    ap.add_argument("--half-only", action="store_true",
                    help="instead of the benchmark line, print one JSON line with the "
                         "16-bit-input path's figures (bf16 / fp16 at 4092^3 and 8192^3)")
    ap.add_argument("--bmm-only", action="store_true",
                    help="instead of the benchmark line, print one JSON line with the batched "
                         "workload's figures on --mode (3xtf32 for auto), --steps timed calls")
    ap.add_argument("--la-only", action="store_true",
                    help="instead of the benchmark line, print one JSON line with the "
                         "linear-attention kernels' figures (--steps timed calls each)")
    ap.add_argument("--tune", action="store_true",
                    help="instead of the benchmark line, time every kernel route on one shape "
                         "per (mode, size class), print one JSON line per shape, and write "
                         "the table of the fastest routes to --tune-out")
    ap.add_argument("--tune-out", default=os.path.join(ROOT, "dense_fp32_matrix_03_gb300", "csrc",
                                                       "tune_table.h"),
                    help="where --tune writes the table (a C++ header compiled into the "
                         "library; rebuild to use it)")
    ap.add_argument("--all-configs", action="store_true",
                    help="instead of the benchmark line, print one JSON line per workload "
                         "configuration and path (256^3, ragged, size sweep, batched)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = dist_env()

    if args.impl == "reference":
        return reference_arm(args, rank, world)
    if args.all_configs:
        return all_configs(args)
    if args.tune:
        return tune(args)
    if args.la_only:
        return la_only(args.steps)
    if args.half_only:
        return half_only()
    if args.bmm_only:
        return bmm_only(args.mode, args.steps)

    import torch
    import dense_fp32_matrix_03_gb300 as lib
    import workloads

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    lib.load()
    props = torch.cuda.get_device_properties(dev)
    num_sms = props.multi_processor_count
    peaks, peak_src = load_peaks()
    mode = resolve_mode(lib, args.mode)

    w = workloads.make(WORKLOAD)
    M, N, K = w["M"], w["N"], w["K"]
    alpha, beta = w["alpha"], w["betas"][0]
    A = torch.from_numpy(w["A"]).to(dev)
    B = torch.from_numpy(w["B"]).to(dev)
    C = torch.from_numpy(w["C0"]).to(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # split-K workspace (the last, partial wave of tiles is cut along K),
    # allocated once, outside the timed region, like a library handle's
    ws_bytes, ws = workspace(lib, mode, M, N, K, 1, dev)

    def call():
        lib.check(lib.sgemm_batched_ex_ws(mode, M, N, K, alpha, A, K, B, N, beta, C, N, 0, 0, 0,
                                          0, 0, 1, ws, ws_bytes, stream))

    gpu_id = None
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        gpu_id = "GPU-" + str(uuid) if not str(uuid).startswith("GPU-") else str(uuid)

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as clk:
        t_wall0 = time.perf_counter()
        times, launches = time_calls(call, args.steps, args.warmup, stream, flush, lib)
        t_wall = time.perf_counter() - t_wall0
    torch.cuda.synchronize()
    barrier(world)
    lib.check(lib.sgemm_poll_error(stream))
    clocks = clk.summary()

    ms_local = statistics.mean(times)
    ms = reduce_max(ms_local, world, dev)
    # the spread of the timed steps on this rank: the loop runs long enough
    # for the power cap to act, so its later steps are slower than its first
    srt = sorted(times)
    q = max(1, len(times) // 10)
    step_ms = {"min": srt[0], "median": statistics.median(times),
               "p90": srt[min(len(srt) - 1, (9 * len(srt)) // 10)], "max": srt[-1],
               "first_tenth_mean": statistics.mean(times[:q]),
               "last_tenth_mean": statistics.mean(times[-q:])}
    flops_step = gemm_flops(M, N, K)
    total_flops = reduce_sum(flops_step, world, dev)
    value = total_flops / (ms / 1e3) / 1e12

    bound, peak, peak_note = roofline_peak(mode, num_sms, peaks, peak_src)
    achieved = flops_step / (ms_local / 1e3) / 1e12
    kernel_key = f"{mode}:{WORKLOAD}"
    traffic = committed_traffic(kernel_key)
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": UNIT,
                "frac": achieved / peak, "traffic": traffic,
                "kernel": f"sgemm {mode} path ({kernel_key})",
                "timed": ("each call: every kernel it launches -- on the tensor-core paths "
                          "at this size the GEMM kernel (the caller's A and B straight through "
                          "TMA; 3xTF32's lo planes made inside it) and the split-K fix-up; on "
                          "the FP32 path the operand transposition, the GEMM kernel and the "
                          "fix-up (events bracket the whole call; traffic is the GEMM kernel's)"
                          if ws_bytes else "each call: the GEMM kernel"),
                "peak_source": f"{peak_note}; {peak_src} MEASURED_PEAKS.json" if bound != "alu"
                else peak_note,
                "algorithmic_flops_per_launch": flops_step}
    if clocks and clocks.get("sm_mhz") and bound == "alu":
        roofline["frac_at_sampled_clock"] = achieved / (
            num_sms * FP32_LANES_PER_SM * 2 * clocks["sm_mhz"] * 1e6 / 1e12)

    # ---- end to end through the host-buffer entry point (sgemm_host): the
    # operands start in pinned host memory, C ends there; copies inside
    e2e = None
    if rank == 0 or world > 1:
        hA = torch.from_numpy(w["A"]).pin_memory()
        hB = torch.from_numpy(w["B"]).pin_memory()
        hC = torch.from_numpy(w["C0"]).pin_memory()
        dev_bytes = lib.sgemm_host_buffer_size(mode, M, N, K, 0, 0, 0)
        dbuf = torch.empty(dev_bytes, dtype=torch.uint8, device=dev)

        def e2e_call():
            lib.check(lib.sgemm_host(mode, M, N, K, alpha, hA, K, hB, N, beta, hC, N, 0, 0, 0,
                                     dbuf, dev_bytes, stream))
        e_steps = max(3, min(args.steps, 10))
        et, e_launches = time_calls(e2e_call, e_steps, 3, stream, flush, lib)
        e_ms = statistics.mean(et)
        e2e = {"value": flops_step / (e_ms / 1e3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": 4 * (M * K + K * N + (M * N if beta != 0 else 0)),
               "d2h_bytes_per_step": 4 * M * N, "ms_per_step": e_ms,
               "entry": "sgemm_host (pinned host buffers, panels of C overlap copies "
                        "and products)", "gpu_launches": e_launches}
        del dbuf

    probes = None
    if rank == 0:
        probes = peak_probes(lib, stream)
        probe_peak = probe_peak_for(mode, probes)
        if probe_peak:
            roofline["probe_peak"] = probe_peak
            roofline["frac_of_probe"] = achieved / probe_peak
            roofline["probe_note"] = ("the same instructions with no operand traffic, timed "
                                      "here (sgemm_peak_probe): " + PROBE_FOR[mode])

    extra = {}
    if not args.no_extra and rank == 0:
        extra = extra_figures(lib, mode, dev, stream, flush, num_sms, peaks, peak_src)
        extra["configs"] = config_figures(lib, dev, stream, flush, num_sms, peaks, peak_src,
                                          probes)
        extra["linear_attention"] = la_figures(lib, dev, stream, flush, num_sms, peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "step_ms": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "alpha": alpha,
                       "beta": beta, "mode": mode, "inputs": "normal(0,1) seed 2",
                       "entry": "sgemm_batched_ex_ws", "workspace_bytes": ws_bytes,
                       "l2": f"flushed before every timed step ({2 * l2 >> 20} MB write)",
                       "parallelism": f"replicas x{world}"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "peak_probes_tflops": probes,
            "wall_s_timed_loop": t_wall,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def workspace(lib, mode, M, N, K, Q, dev):
    """The split-K workspace the library asks for this call: (bytes, tensor)."""
    import torch
    ws_bytes = lib.sgemm_workspace_size(mode, M, N, K, Q)
    return ws_bytes, torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)


def half_figures(lib, dev, stream, flush, peaks, peak_src):
    """The 16-bit-input path (bf16 / fp16 A and B, fp32 C) at 4092^3 and
    8192^3, A times B-transpose (read directly) and A times B (B copied
    transposed into the workspace first), against the measured bf16 peak."""
    import torch
    out = {}
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    for n in (4092, 8192):
        g = torch.Generator(device=dev).manual_seed(5)
        A = torch.randn(n, n, device=dev, generator=g).to(torch.bfloat16)
        Bt = torch.randn(n, n, device=dev, generator=g).to(torch.bfloat16)
        C = torch.zeros(n, n, device=dev)
        for type_ in ("bf16", "fp16"):
            if type_ == "fp16":
                A, Bt = A.to(torch.float16), Bt.to(torch.float16)
            for tB in (1, 0):
                if n == 8192 and (type_ == "fp16" or tB == 0):
                    continue
                Bd = Bt if tB else Bt.t().contiguous()
                wsb = lib.sgemm_half_workspace_size(type_, n, n, n, 0, tB, n, n, 1)
                ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)

                def call(type_=type_, tB=tB, Bd=Bd, ws=ws, wsb=wsb):
                    lib.check(lib.sgemm_half_batched(type_, n, n, n, 1.0, A, n, Bd, n, 0.0, C, n, 0,
                                                     tB, 0, 0, 0, 1, ws, wsb, stream))
                t = statistics.median(time_calls(call, 10, 3, stream, flush))
                tf = gemm_flops(n, n, n) / (t / 1e3) / 1e12
                out[f"{type_}_{'a_bt' if tB else 'a_b'}_{n}"] = {
                    "tflops": tf, "ms": t, "peak": peak, "frac": tf / peak,
                    "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)"}
        del A, Bt, C
    lib.check(lib.sgemm_poll_error(stream))
    return out


def extra_figures(lib, default_mode, dev, stream, flush, num_sms, peaks, peak_src):
    """Per-path figures at 4092^3 and batched-GEMM figures (fewer steps)."""
    import torch
    import workloads
    out = {"paths": {}, "bmm": {}}
    w = workloads.make(WORKLOAD)
    M, N, K = w["M"], w["N"], w["K"]
    A = torch.from_numpy(w["A"]).to(dev)
    B = torch.from_numpy(w["B"]).to(dev)
    C = torch.zeros(M, N, device=dev)
    for mode in ("fp32", "3xtf32", "tf32"):
        st = lib.sgemm_batched_ex(mode, 16, 16, 16, 1.0, A, K, B, N, 0.0, C, N, 0, 0, 0, 0, 0, 1,
                                  stream)
        if st != lib.SGEMM_OK:
            out["paths"][mode] = {"status": lib.sgemm_status_string(st)}
            continue

        ws_bytes, ws = workspace(lib, mode, M, N, K, 1, dev)

        def call(mode=mode, ws=ws, ws_bytes=ws_bytes):
            lib.check(lib.sgemm_batched_ex_ws(mode, M, N, K, 1.0, A, K, B, N, 0.0, C, N, 0, 0, 0,
                                              0, 0, 1, ws, ws_bytes, stream))
        t = statistics.median(time_calls(call, 10, 3, stream, flush))
        tf = gemm_flops(M, N, K) / (t / 1e3) / 1e12
        bound, peak, note = roofline_peak(mode, num_sms, peaks, peak_src)
        out["paths"][mode] = {"tflops": tf, "ms": t, "bound": bound, "peak": peak,
                              "frac": tf / peak}
    del A, B, C
    out["half"] = half_figures(lib, dev, stream, flush, peaks, peak_src)
    out["bmm"] = bmm_figures(lib, default_mode, dev, stream, flush)
    return out


def graph_device_ms(call_on, steps, flush):
    """Device time of one call: the call captured in a CUDA graph and the
    graph replayed between events (L2 flushed before each replay), so that
    no host work of the library or of this binding is inside the interval
    (median ms)."""
    import torch
    cur = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        call_on(side)  # any first-use set-up outside the capture
    cur.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        call_on(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        g.replay()
        e1.record(cur)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    del g
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def config_figures(lib, dev, stream, flush, num_sms, peaks, peak_src, probes, steps=5):
    """Every workload configuration on every path, through the workspace
    entry point (the library's preferred call, with the workspace it asks
    for): TFLOP/s, the roofline that bounds it -- min(path peak, AI x HBM
    bandwidth), AI over compulsory bytes -- and the fraction of it; beside
    it the fraction of the path's probe-measured rate where the compute roof
    binds.  L2 is flushed before every timed call.  The call is timed with
    events around it, so host work (the library's plan and launches, the
    Python binding) is inside `ms`; for calls under 1e10 FLOP the cell also
    gives `device_ms`, the same call replayed from a CUDA graph (device time
    alone)."""
    import numpy as np
    import torch
    import workloads
    bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])) / 1e3  # TB/s
    cases = [("sgemm_256", 0), ("sgemm_ragged_1000x1500x777", 0),
             ("sgemm_ragged_1000x1500x777", 1)]
    cases += [(f"sweep_{n}", 0) for n in workloads.SWEEP_SIZES]
    cases += [("bmm_q32_1024x1024x512", 0)]
    out = {}
    for name, beta_idx in cases:
        w = workloads.make(name)
        M, N, K, Q = w["M"], w["N"], w["K"], w["Q"]
        beta = w["betas"][beta_idx]
        A = torch.from_numpy(w["A"]).to(dev)
        Bn = torch.from_numpy(w["B"]).to(dev)
        C = torch.from_numpy(w["C0"]).to(dev)
        variants = [(0, Bn, N)]
        if Q > 1:
            Bt = torch.from_numpy(np.ascontiguousarray(np.swapaxes(w["B"], 1, 2))).to(dev)
            variants = [(1, Bt, K), (0, Bn, N)]
        flops = gemm_flops(M, N, K, Q)
        ai = flops / compulsory_bytes(M, N, K, Q, beta != 0)
        for tB, Bd, ldb in variants:
            key = name + (f"_beta={beta:g}" if len(w["betas"]) > 1 else "") + \
                (f"_transB={tB}" if Q > 1 else "")
            row = {}
            for mode in ("fp32", "3xtf32", "tf32"):
                ws_bytes, ws = workspace(lib, mode, M, N, K, Q, dev)

                def call_on(st, mode=mode, Bd=Bd, ldb=ldb, tB=tB, ws=ws, ws_bytes=ws_bytes):
                    lib.check(lib.sgemm_batched_ex_ws(mode, M, N, K, w["alpha"], A, K, Bd, ldb,
                                                      beta, C, N, 0, tB, M * K, K * N, M * N, Q,
                                                      ws, ws_bytes, st))

                def call(call_on=call_on):
                    call_on(stream)
                n_steps = steps if flops < 2e11 else 3
                ms = statistics.median(time_calls(call, n_steps, 3, stream, flush))
                tf = flops / (ms / 1e3) / 1e12
                bound, peak, _ = roofline_peak(mode, num_sms, peaks, peak_src)
                roof = min(peak, ai * bw)
                cell = {"tflops": round(tf, 2), "ms": round(ms, 4), "roof": round(roof, 1),
                        "bound": bound if roof == peak else "hbm", "frac": round(tf / roof, 3)}
                if flops < 1e10:
                    dms = graph_device_ms(call_on, 10, flush)
                    cell["device_ms"] = round(dms, 4)
                    cell["device_tflops"] = round(flops / (dms / 1e3) / 1e12, 2)
                pp = probe_peak_for(mode, probes) if probes else None
                if pp:
                    cell["frac_of_probe_roof"] = round(tf / min(pp, ai * bw), 3)
                row[mode] = cell
                del ws
            out[key] = row
        del A, Bn, C
    lib.check(lib.sgemm_poll_error(stream))
    return out


LA_WORKLOAD = "la_b4h16_t4096_d128"


def la_flops(BH, T, DK, DV, BT=64):
    """Algorithmic FLOPs of the chunked form: per chunk of BT tokens and per
    head, Q K^T (BT x BT x DK), A V (BT x DV x BT), Q h (BT x DV x DK) and the
    state update K^T V (DK x DV x BT), two FLOPs per multiply-add."""
    NT = -(-T // BT)
    return 2.0 * BT * (BT * DK + BT * DV + 2 * DK * DV) * NT * BH


def la_figures(lib, dev, stream, flush, num_sms, peaks, steps=10):
    """The linear-attention building blocks on the benchmark's workload
    (64 heads x 4096 tokens, head dimension 128): the chunked path (state
    pass, then output pass) and the fused pass, L2 flushed before every
    timed call; roofline: the FP32 FFMA peak (the kernels run on the CUDA
    cores) and, beside it, the HBM time of their compulsory bytes."""
    import torch
    import workloads
    q, k, v, g, _, scale = workloads.la_make(LA_WORKLOAD)
    BH, T, DK = q.shape
    DV = v.shape[2]
    NT = -(-T // 64)
    t = lambda x: torch.from_numpy(x).to(dev)
    dq, dk, dv, dg = t(q), t(k), t(v), t(g)
    h = torch.empty(BH, NT, DK, DV, device=dev)
    o = torch.empty(BH, T, DV, device=dev)
    so = torch.empty(BH, DK, DV, device=dev)

    def state():
        lib.check(lib.la_chunk_state(BH, T, DK, DV, dk, dv, dg, None, h, so, stream))

    def output():
        lib.check(lib.la_chunk_output(BH, T, DK, DV, scale, dq, dk, dv, dg, h, o, stream))

    def chunked():
        state()
        output()

    def fused():
        lib.check(lib.la_chunk_fused(BH, T, DK, DV, scale, dq, dk, dv, dg, None, o, so, stream))
    flops = la_flops(BH, T, DK, DV)
    mhz = float(peaks.get("sm_max_mhz", FALLBACK_PEAKS["sm_max_mhz"]))
    peak = num_sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])) / 1e3
    io = 4.0 * BH * T * (2 * DK + 2 * DV)          # q, k, v read; o written
    hb = 4.0 * BH * NT * DK * DV                    # h written and read back
    out = {"workload": LA_WORKLOAD, "BH": BH, "T": T, "DK": DK, "DV": DV, "chunk": 64,
           "algorithmic_gflop": flops / 1e9,
           "roofline": {"bound": "alu", "peak": peak, "unit": "TFLOP/s",
                        "peak_source": f"FP32 FFMA peak: {num_sms} SMs x 128 lanes x 2 x "
                                       f"{mhz:.0f} MHz"}}
    for name, fn, nbytes in (("chunked", chunked, io + 2 * hb), ("fused", fused, io)):
        ms = statistics.median(time_calls(fn, steps, 3, stream, flush))
        tf = flops / (ms / 1e3) / 1e12
        out[name] = {"ms": ms, "tflops": tf, "frac": tf / peak,
                     "hbm_bytes": nbytes, "hbm_floor_ms": nbytes / bw / 1e9}
    out["chunked"]["state_ms"] = statistics.median(time_calls(state, steps, 3, stream, flush))
    out["chunked"]["output_ms"] = statistics.median(time_calls(output, steps, 3, stream, flush))
    lib.check(lib.sgemm_poll_error(stream))
    return out


def bmm_figures(lib, mode, dev, stream, flush, steps=10):
    """The batched workload (Q=32, 1024x1024x512, B stored N x K and K x N)
    through the workspace entry on `mode`: TFLOP/s per layout."""
    import torch
    import workloads
    out = {}
    wb = workloads.make("bmm_q32_1024x1024x512")
    Q, M, N, K = wb["Q"], wb["M"], wb["N"], wb["K"]
    A = torch.from_numpy(wb["A"]).to(dev)
    Bn = torch.from_numpy(wb["B"]).to(dev)                             # Q x K x N
    Bt = torch.from_numpy(wb["B"].transpose(0, 2, 1).copy()).to(dev)   # Q x N x K
    C = torch.from_numpy(wb["C0"]).to(dev)
    ws_bytes, ws = workspace(lib, mode, M, N, K, Q, dev)
    for tB, Bd, ldb in ((1, Bt, K), (0, Bn, N)):
        def call(tB=tB, Bd=Bd, ldb=ldb):
            lib.check(lib.sgemm_batched_ex_ws(mode, M, N, K, wb["alpha"], A, K, Bd, ldb,
                                              wb["betas"][0], C, N, 0, tB, M * K, K * N, M * N, Q,
                                              ws, ws_bytes, stream))
        t = statistics.median(time_calls(call, steps, 3, stream, flush))
        out[f"transB={tB}"] = {"tflops": gemm_flops(M, N, K, Q) / (t / 1e3) / 1e12,
                               "ms": t, "mode": mode}
    return out


def bmm_only(mode, steps):
    """--bmm-only: the batched workload alone (a short command to profile)."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    lib.load()
    if mode == "auto":
        mode = "3xtf32"
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    out = bmm_figures(lib, mode, dev, torch.cuda.current_stream(dev), flush, steps)
    print(json.dumps({"bmm": out, "l2": "flushed before every timed step"}), flush=True)
    return 0


def la_only(steps):
    """--la-only: the linear-attention building blocks alone (a short command
    to profile)."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    lib.load()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    peaks, _ = load_peaks()
    out = la_figures(lib, dev, torch.cuda.current_stream(dev), flush,
                     props.multi_processor_count, peaks, steps)
    print(json.dumps({"linear_attention": out, "l2": "flushed before every timed step"}),
          flush=True)
    return 0


def half_only():
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    lib.load()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    peaks, src = load_peaks()
    out = half_figures(lib, dev, torch.cuda.current_stream(dev), flush, peaks, src)
    print(json.dumps({"half": out, "l2": "flushed before every timed step"}), flush=True)
    return 0


def oracle_timing(w, beta, target_s=2.0):
    """The oracle on a bounded row sample of workload w (rows spread over the
    batch and M), sized for about target_s seconds on the threads it uses
    (OMP_NUM_THREADS, else every core)."""
    import numpy as np
    import oracle
    M, N, K, Q = w["M"], w["N"], w["K"], w["Q"]

    def run(nrows):
        idx = np.linspace(0, Q * M - 1, nrows).astype(np.int64)
        rows = [(int(i // M), int(i % M)) for i in idx]
        t0 = time.perf_counter()
        oracle.sgemm_ref(M, N, K, w["alpha"], w["A"], K, w["B"], N, beta, w["C0"], N,
                         strideA=M * K, strideB=K * N, strideC=M * N, Q=Q, rows=rows)
        return time.perf_counter() - t0

    t = run(4)
    nrows = int(min(Q * M, max(4, 4 / max(t, 1e-6) * target_s)))
    t = run(nrows)
    flops = 2.0 * nrows * N * K
    return {"gflops": round(flops / t / 1e9, 3), "threads": oracle.num_threads(),
            "seconds": round(t, 3), "rows": f"{nrows} of {Q * M}"}


def oracle_timing_single_thread(name, beta_idx):
    """oracle_timing on one thread, in a child process (the oracle's thread
    count is fixed when it loads)."""
    import subprocess
    code = ("import json, bench, workloads; w = workloads.make(%r); "
            "print(json.dumps(bench.oracle_timing(w, w['betas'][%d])))" % (name, beta_idx))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=600)
    if out.returncode != 0:
        return {"error": out.stderr.strip().splitlines()[-1:]}
    return json.loads(out.stdout.strip().splitlines()[-1])


def all_configs(args):
    """One JSON line per (workload, path): TFLOP/s and the roofline it is
    bound by, min(peak, AI * HBM bandwidth) with AI over compulsory bytes;
    for working sets under 2 x L2 also the warm-L2 time.  Then one line per
    workload with the oracle's rate on the host cores (and on one thread for
    the two small configurations)."""
    import numpy as np
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    import workloads
    dev = torch.device("cuda", 0)
    props = torch.cuda.get_device_properties(dev)
    peaks, src = load_peaks()
    bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])) / 1e3  # TB/s
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    cases = [("sgemm_256", 0), ("sgemm_ragged_1000x1500x777", 0),
             ("sgemm_ragged_1000x1500x777", 1)]
    cases += [(f"sweep_{n}", 0) for n in workloads.SWEEP_SIZES]
    cases += [("bmm_q32_1024x1024x512", 0)]
    for name, beta_idx in cases:
        w = workloads.make(name)
        M, N, K, Q = w["M"], w["N"], w["K"], w["Q"]
        beta = w["betas"][beta_idx]
        A = torch.from_numpy(w["A"]).to(dev)
        Bn = torch.from_numpy(w["B"]).to(dev)
        C = torch.from_numpy(w["C0"]).to(dev)
        variants = [(0, Bn, N)]
        if Q > 1:
            Bt = torch.from_numpy(np.ascontiguousarray(np.swapaxes(w["B"], 1, 2))).to(dev)
            variants = [(1, Bt, K), (0, Bn, N)]
        flops = gemm_flops(M, N, K, Q)
        ai = flops / compulsory_bytes(M, N, K, Q, beta != 0)
        for tB, Bd, ldb in variants:
            for mode in ("fp32", "3xtf32", "tf32"):
                ws_bytes = lib.sgemm_workspace_size(mode, M, N, K, Q)
                ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
                for entry in (("plain", "split_k") if ws_bytes else ("plain",)):
                    def call(mode=mode, Bd=Bd, ldb=ldb, tB=tB, entry=entry):
                        if entry == "plain":
                            st = lib.sgemm_batched_ex(mode, M, N, K, w["alpha"], A, K, Bd, ldb,
                                                      beta, C, N, 0, tB, M * K, K * N, M * N, Q,
                                                      stream)
                        else:
                            st = lib.sgemm_batched_ex_ws(mode, M, N, K, w["alpha"], A, K, Bd, ldb,
                                                         beta, C, N, 0, tB, M * K, K * N, M * N,
                                                         Q, ws, ws_bytes, stream)
                        lib.check(st)
                    ms = statistics.median(time_calls(call, args.steps, args.warmup, stream,
                                                      flush))
                    tf = flops / (ms / 1e3) / 1e12
                    bound, peak, _ = roofline_peak(mode, props.multi_processor_count, peaks, src)
                    roof = min(peak, ai * bw)
                    line = {"workload": name, "beta": beta, "transB": tB, "mode": mode,
                            "entry": entry, "ms": round(ms, 4), "tflops": round(tf, 2),
                            "roof_tflops": round(roof, 1),
                            "roof_bound": bound if roof == peak else "hbm",
                            "frac": round(tf / roof, 3)}
                    if compulsory_bytes(M, N, K, Q, beta != 0) + ws_bytes < 2 * l2:
                        msw = statistics.median(time_calls(call, args.steps, args.warmup,
                                                           stream, None))
                        line["ms_warm_l2"] = round(msw, 4)
                        line["tflops_warm_l2"] = round(flops / (msw / 1e3) / 1e12, 2)
                    print(json.dumps(line), flush=True)
    lib.check(lib.sgemm_poll_error(stream))
    for name, beta_idx in cases:
        w = workloads.make(name)
        line = {"workload": name, "beta": w["betas"][beta_idx],
                "oracle": oracle_timing(w, w["betas"][beta_idx])}
        if name in ("sgemm_256", "sgemm_ragged_1000x1500x777"):
            line["oracle_one_thread"] = oracle_timing_single_thread(name, beta_idx)
        print(json.dumps(line), flush=True)
    return 0


# The sweep behind the committed route table (dense_fp32_matrix_03_gb300/
# csrc/tune_table.h).  One representative shape per size class
# (round(log2(M N K Q) / 3)): the square sizes 128 .. 8192 (4092 for class 12,
# the benchmark shape), and the batched workload for the batched class 11.
TUNE_SHAPES = [(128, 128, 128, 1), (256, 256, 256, 1), (512, 512, 512, 1),
               (1024, 1024, 1024, 1), (2048, 2048, 2048, 1), (4092, 4092, 4092, 1),
               (8192, 8192, 8192, 1), (1024, 1024, 512, 32)]
# "models": the cost models' choice with the committed table ignored (the
# baseline; "auto" would replay the table being rewritten)
TUNE_ROUTES = {"fp32": ("models", "small"),
               "3xtf32": ("models", "pair", "direct", "planes", "raw", "inline"),
               "tf32": ("models", "pair", "direct", "planes", "raw")}
TUNE_KEEP_AUTO = 0.02  # a route must beat the cost models' choice by 2% to get an entry


def size_class(M, N, K, Q):
    import math
    c = round(math.log2(max(M * N * K * Q, 1)) / 3.0)
    return min(max(c, 7), 13)


def tune(args):
    """--tune: every route on every representative shape and mode, through
    the workspace entry with the workspace the library asks for under that
    route, L2 flushed before every timed call; the fastest route per (mode,
    class) goes into the table unless the cost models' choice is within
    TUNE_KEEP_AUTO of it."""
    import torch
    import dense_fp32_matrix_03_gb300 as lib
    dev = torch.device("cuda", 0)
    lib.load()
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    entries = []
    try:
        for (M, N, K, Q) in TUNE_SHAPES:
            g = torch.Generator(device=dev).manual_seed(3)
            A = torch.rand(Q, M, K, device=dev, generator=g) * 2 - 1
            B = torch.rand(Q, K, N, device=dev, generator=g) * 2 - 1
            C = torch.zeros(Q, M, N, device=dev)
            flops = gemm_flops(M, N, K, Q)
            steps = 20 if flops < 2e10 else (8 if flops < 3e11 else 3)
            for mode in ("fp32", "3xtf32", "tf32"):
                times = {}
                for route in TUNE_ROUTES[mode]:
                    lib.check(lib.sgemm_tune_force(route))
                    wsb, ws = workspace(lib, mode, M, N, K, Q, dev)

                    def call(mode=mode, ws=ws, wsb=wsb):
                        lib.check(lib.sgemm_batched_ex_ws(mode, M, N, K, 1.0, A, K, B, N, 0.0, C, N,
                                                          0, 0, M * K, K * N, M * N, Q, ws, wsb,
                                                          stream))
                    times[route] = statistics.median(time_calls(call, steps, 3, stream, flush))
                    del ws
                lib.check(lib.sgemm_tune_force("auto"))
                best = min(times, key=times.get)
                cls, batched = size_class(M, N, K, Q), int(Q > 1)
                chosen = best if times[best] < (1 - TUNE_KEEP_AUTO) * times["models"] else "auto"
                line = {"mode": mode, "M": M, "N": N, "K": K, "Q": Q, "size_class": cls,
                        "batched": batched, "us": {r: round(t * 1e3, 1) for r, t in times.items()},
                        "tflops": {r: round(flops / (t / 1e3) / 1e12, 2) for r, t in times.items()},
                        "chosen": chosen}
                print(json.dumps(line), flush=True)
                entries.append(line)
            del A, B, C
        lib.check(lib.sgemm_poll_error(stream))
    finally:
        lib.sgemm_tune_force("auto")
    write_tune_table(entries, args.tune_out, props.name)
    return 0


def write_tune_table(entries, path, gpu):
    """The C++ header the library compiles in: one entry per (mode, class,
    batched) whose fastest route is not the cost models' choice, each with
    the times the sweep measured."""
    import dense_fp32_matrix_03_gb300 as lib
    modes = {"fp32": 0, "3xtf32": 1, "tf32": 2}
    rows = []
    for e in entries:
        if e["chosen"] == "auto":
            continue
        times = ", ".join(f"{r} {t}" for r, t in e["us"].items())
        rows.append(f"    {{{modes[e['mode']]}, {e['size_class']}, {e['batched']}, "
                    f"{lib.ROUTES[e['chosen']]}}},  // {e['mode']} {e['M']}x{e['N']}x{e['K']}"
                    f"{' Q=' + str(e['Q']) if e['Q'] > 1 else ''}: {e['chosen']}; us: {times}")
    kept = [f"//   {e['mode']} {e['M']}x{e['N']}x{e['K']}{' Q=' + str(e['Q']) if e['Q'] > 1 else ''}"
            f" (class {e['size_class']}): us " + ", ".join(f"{r} {t}" for r, t in e["us"].items())
            for e in entries if e["chosen"] == "auto"]
    text = "\n".join([
        "// tune_table.h -- kernel route per (mode, size class, batched) call, as",
        "// measured by the sweep `python bench.py --tune` (which rewrites this file)",
        f"// on {gpu}, L2 flushed before every timed call, through the workspace entry.",
        "// Size class and routes: internal.h (size_class, Route).  A (mode, class)",
        "// without an entry takes the cost models' choice (kRouteAuto), which the",
        f"// sweep keeps unless another route is more than {TUNE_KEEP_AUTO:.0%} faster; the",
        "// shapes where it kept the cost models' choice:",
        *kept,
        "#pragma once",
        "",
        "namespace sg {",
        "",
        "struct TuneEntry {",
        "    int mode, size_class, batched, route;",
        "};",
        "",
        "// {mode (0 FP32, 1 3xTF32, 2 TF32), size class, batched, route}",
        "constexpr TuneEntry kTuneTable[] = {",
        *rows,
        "    {-1, 0, 0, 0},  // end of table",
        "};",
        "",
        "}  // namespace sg",
        "",
    ])
    with open(path, "w") as f:
        f.write(text)


if __name__ == "__main__":
    sys.exit(main())
