"""Benchmark of the GB300 GEMM  C = A . B^T  (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload square_4096|...] [--seconds S]

A step is a batch of R GEMMs over the workload's synthetic seeded operands
(inputs resident in HBM), R chosen after the warm-up so that the K timed steps
last about S seconds (default 12): long enough for clock samplers polling a few
times a second to see the GPU under this load.  By default a 512 MiB buffer is
overwritten before each GEMM to flush the 129 MB L2, outside that GEMM's pair of
CUDA events on the launching stream; a step's time is the sum of its GEMMs'.
`--l2 rotate` instead cycles through copies of A, B and C totalling at least
four times the L2 with the step's R launches back to back between two events
(cold operands in every launch, no launch gap; the GPU then runs at its power
cap throughout).  The decode shapes are always timed the second way.
Secondary sections of the line: `decode` (the four M = 256 shapes), `decode_small_m`
(M = 1..128), `decode_swapped` (shapes the host gives the swapped tiling, with the
plain tiling forced and timed beside them), `fp8` (per-tensor and blockwise scales)
and `grouped` (MoE groups and a group of mixed K).
`value` is TFLOP/s (2MNK per GEMM) over all ranks; `e2e` is the same metric through gemm_run_host with
pinned host buffers (host->device copies of A and B and the device->host copy
of C inside the timed region).  `cpu_baseline` times the CPU oracle on a
bounded sample of the same product (whole rows of C) on the host cores, and
those rows double as a full-size parity check of the GPU result.

Multi-GPU: the GEMM does not exchange data between GPUs; N ranks run N
independent replicas ("weak" scaling, value = all ranks' FLOPs / max time).
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from datetime import datetime

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import seeded_inputs as si  # noqa: E402
from dense_gemm_blackwell_02_gb300 import roofline as rl  # noqa: E402

METRIC = "GEMM TFLOP/s (4096³ fp16) & % of tensor peak; decode-shape HBM GB/s"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20
L2_NOMINAL_BYTES = 129 * 1000 * 1000
# Nominal GB300 figures, reported as context beside the measured peaks.
NOMINAL_TFLOPS = 2250.0   # dense fp16/bf16
# Dense fp16/bf16 tensor work of one SM per clock ("Optimizing GEMMs using tcgen05":
# a 128 x 256 x 16 MMA in 128 cycles); times the SMs and the SM clock observed under
# load, the peak at the clock the kernel actually ran at.
TENSOR_FLOP_PER_SM_CLK = 8192
NOMINAL_HBM_GBS = 7900.0
NOMINAL_FP8_RATIO = 2.0  # dense FP8 / dense bf16 (4.5 / 2.25 PFLOP/s nominal)
# The device code of the kernels (the host-side files -- the C ABI, the launch table --
# do not change what a launch of a given configuration moves).
KERNEL_SOURCES = ("dense_gemm_blackwell_02_gb300/csrc/gemm_kernel.cuh",
                  "dense_gemm_blackwell_02_gb300/csrc/ptx.cuh",
                  "dense_gemm_blackwell_02_gb300/csrc/umma.cuh",
                  "dense_gemm_blackwell_02_gb300/csrc/params.h",
                  "dense_gemm_blackwell_02_gb300/csrc/launch_impl.cuh")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in sorted(os.path.join(ROOT, k) for k in KERNEL_SOURCES):
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    """The job's time is the slowest rank's: max of x over the process group (x itself
    when there is no group).  Replicas exchange nothing else."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, flops_per_step: float, steps: int, slowest_ms: float) -> float:
    """Whole-job TFLOP/s of `world` independent replicas, each running `steps` steps of
    `flops_per_step`, timed by the slowest rank (weak scaling)."""
    return world * flops_per_step * steps / (slowest_ms * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling; statistics are taken over the
    samples inside the timed region (mark() brackets it), and among those over the ones
    with the GPU busy (utilization >= 30%).  The samples go to a temporary file."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.fh = None
        self.window = None

    def start(self):
        try:
            self.fh = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark(self, t0: datetime, t1: datetime):
        """The timed region, in the host's local time (nvidia-smi's timestamps)."""
        self.window = (t0, t1)

    @staticmethod
    def parse(lines, window=None):
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 11:
                continue
            try:
                ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append({"t": ts, "sm": float(parts[2]), "max": float(parts[3]),
                             "power": float(parts[4]), "util": float(parts[5]),
                             "hw": parts[7], "hw_thermal": parts[8], "sw_thermal": parts[9],
                             "sw_power": parts[10]})
            except ValueError:
                continue
        inside = [r for r in rows if window is None or window[0] <= r["t"] <= window[1]]
        loaded = [r for r in inside if r["util"] >= 30]
        use = loaded or inside
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0, "samples_under_load": 0}
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in use):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in use),
                "sm_max_mhz": max(r["max"] for r in use),
                "sm_mhz_min": min(r["sm"] for r in use), "reasons": reasons,
                "power_w_max": max(r["power"] for r in use),
                "samples": len(inside), "samples_under_load": len(loaded),
                "over": "samples inside the timed region with utilization >= 30%"
                        if loaded else "samples inside the timed region (none busy)"}

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.seek(0)
        out = self.parse(self.fh.readlines(), self.window)
        self.fh.close()
        return out


def workload_shape(name: str):
    wl = si.WORKLOADS[name]
    return wl, wl.shapes[0]


def cpu_rows_sample(A, B, din, dout, M, target_s=10.0):
    """Oracle rows timed on the host cores: calibrate on a few rows, then time
    enough rows for ~target_s seconds.  Returns (rows, bits, seconds, threads)."""
    import oracle
    N, K = B.shape[0], B.shape[1]
    # Two probes (32 and 128 rows) separate each call's fixed cost (operand conversion)
    # from the cost per row, so that the sample is sized to the target.
    oracle.gemm_select(A, B, si.sample_indices(M, 2, seed=98), None, din, dout)  # tables, threads
    times = []
    for n in (min(M, 32), min(M, 128)):
        probe = si.sample_indices(M, n, seed=99)
        t0 = time.perf_counter()
        oracle.gemm_select(A, B, probe, None, din, dout)
        times.append((n, time.perf_counter() - t0))
    (n1, t1), (n2, t2) = times
    per_row = max((t2 - t1) / max(n2 - n1, 1), t2 / max(n2, 1) * 0.05, 1e-7)
    fixed = max(t1 - per_row * n1, 0.0)
    nrows = int(min(M, max(32, (target_s - fixed) / per_row)))
    for attempt in range(2):
        # (draws with repeats: every row once the count reaches M)
        rows = (list(range(M)) if nrows >= M else
                si.sample_indices(M, nrows, seed=7, must=(0, 127, 128, 255, 256, -1)))
        t0 = time.perf_counter()
        bits, c64 = oracle.gemm_select(A, B, rows, None, din, dout, want_f64=True)
        dt = time.perf_counter() - t0
        if dt >= 0.5 * target_s or len(rows) >= M:
            break
        # the probes overestimated a row: size once more from this run
        nrows = int(min(M, len(rows) * target_s / max(dt, 1e-3)))
    return rows, bits, c64, dt, os.cpu_count()


def l2_bytes(dev) -> int:
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_NOMINAL_BYTES)


def operand_sets(A, B, C, dev):
    """Copies of (A, B, C) totalling at least 4x the L2, used in turn so that every
    step's operands were evicted by the steps before it."""
    per = A.numel() * A.element_size() + B.numel() * B.element_size() + C.numel() * C.element_size()
    n = max(2, -(-4 * l2_bytes(dev) // per))
    return [(A, B, C)] + [(A.clone(), B.clone(), torch.empty_like(C)) for _ in range(n - 1)], n * per


def time_steps(run, sets, stream, steps, flush=None, per_step=False):
    """ms for `steps` launches: back to back between two events, cycling through
    `sets`; or, with `flush`, one event pair per step after overwriting the flush
    buffer (summed).  With per_step, also the list of per-launch ms (back to back:
    between consecutive events recorded between the launches)."""
    if flush is None:
        # events between the launches only when asked for: a stream event between two
        # launches would also stop the second from starting early (programmatic
        # dependent launch)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record(stream)
        for i in range(steps):
            run(*sets[i % len(sets)])
            if per_step or i == steps - 1:
                ev[i + 1].record(stream)
        torch.cuda.synchronize()
        total = ev[0].elapsed_time(ev[-1])
        if not per_step:
            return total
        return total, [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    ev = []
    for i in range(steps):
        flush.fill_(float(i))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(*sets[0])
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    each = [a.elapsed_time(b) for a, b in ev]
    return (sum(each), each) if per_step else sum(each)


def measure_decode(g, dev, stream, peaks, iters=20, name="decode_m256"):
    """Secondary figures: the decode shapes (fp16 -> fp16, M = 256 or M = 1..128),
    HBM-bound.  Each is timed over `iters` launches back to back, cycling through
    operand copies at least four times the L2 (cold operands in every launch, as when a
    model's layers stream their weights); the figure is the median of five such batches.  Their parity is covered by the full-size
    tests; here only time is taken."""
    flush = None
    wl = si.WORKLOADS[name]
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed)
    for s in wl.shapes:
        A = (torch.rand(s.M, s.K, generator=gen, device=dev) * 2 - 1).half()
        B = (torch.rand(s.N, s.K, generator=gen, device=dev) * 2 - 1).half()
        C = torch.empty(s.M, s.N, dtype=torch.float16, device=dev)
        sets, _ = operand_sets(A, B, C, dev) if flush is None else ([(A, B, C)], 0)

        def run(a, b, c):
            g.run(a, b, c, stream=stream)

        for i in range(3 * len(sets)):
            if flush is not None:
                flush.fill_(0.5)
            run(*sets[i % len(sets)])
        torch.cuda.synchronize()
        # the median of five batches of `iters` launches (one batch alone varied by
        # about 1% from run to run); every batch's mean is kept in the line
        batches = sorted(time_steps(run, sets, stream, iters, flush) / iters for _ in range(5))
        ms = batches[len(batches) // 2]
        gbs = rl.gemm_bytes(s.M, s.N, s.K, 2, 2) / (ms * 1e-3) / 1e9
        out[f"{s.M}x{s.N}x{s.K}"] = {"us": round(ms * 1e3, 2),
                                     "us_batches": [round(b * 1e3, 2) for b in batches],
                                     "GB/s": round(gbs, 1),
                                     "frac_of_hbm": round(gbs / hbm, 4),
                                     "frac_of_nominal_hbm": round(gbs / NOMINAL_HBM_GBS, 4),
                                     "TFLOP/s": round(rl.gemm_flops(s.M, s.N, s.K) / (ms * 1e-3) / 1e12, 1),
                                     "kernel": g.last_config()}
        del A, B, C, sets
    return out


def measure_swapped(g, dev, stream, peaks):
    """The decode shapes on which the library takes the swapped tiling, timed like the
    other decode shapes, with the plain tiling (forced) timed the same way beside them."""
    auto = measure_decode(g, dev, stream, peaks, name="decode_swapped")
    g.set_config(swap_ab=1)
    try:
        plain = measure_decode(g, dev, stream, peaks, name="decode_swapped")
    finally:
        g.reset_config()
    for key, v in auto.items():
        v["plain_us"] = plain[key]["us"]
        v["plain_kernel"] = plain[key]["kernel"]
    return auto


def fp8_peak(peaks):
    """The FP8 dense peak: the measured bf16 peak times the nominal FP8 / bf16 ratio."""
    bf16 = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return bf16 * NOMINAL_FP8_RATIO


def measure_fp8(g, dev, stream, peaks, iters=20):
    """Secondary figures: the FP8 (E4M3 -> bf16) square shapes, tensor-bound, with a
    per-tensor scale pair and with blockwise scales (per row of A and 128 of K; per
    128 x 128 of B).  Each is timed like the main workload, one launch per event pair
    after an L2 flush.  Their parity is covered by the full-size tests; here only time
    is taken."""
    wl = si.WORKLOADS["fp8"]
    peak = fp8_peak(peaks)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed)
    for s in wl.shapes:
        td = si.TORCH_DTYPE[wl.dtype_in]
        A = (torch.rand(s.M, s.K, generator=gen, device=dev) * 2 - 1).to(td)
        B = (torch.rand(s.N, s.K, generator=gen, device=dev) * 2 - 1).to(td)
        C = torch.empty(s.M, s.N, dtype=si.TORCH_DTYPE[wl.dtype_out], device=dev)

        def run(a, b, c):
            g.run(a, b, c, stream=stream)

        # blockwise scales: one per row of A and 128 of K, one per 128 x 128 of B
        nkb = -(-s.K // 128)
        # (stored K-block-major, as the library takes them)
        sfa = torch.exp2(torch.rand(nkb, s.M, generator=gen, device=dev) * 6 - 3)
        sfb = torch.exp2(torch.rand(nkb, -(-s.N // 128), generator=gen, device=dev) * 6 - 3)

        def run_bw(a, b, c):
            g.run_blockwise(a, b, c, sfa, sfb, 1, stream=stream)

        for name, fn in (("per_tensor", run), ("blockwise_1x128_128x128", run_bw)):
            for _ in range(3):
                flush.fill_(0.5)
                fn(A, B, C)
            torch.cuda.synchronize()
            total, each = time_steps(fn, [(A, B, C)], stream, iters, flush, per_step=True)
            ms = total / iters
            tf = rl.gemm_flops(s.M, s.N, s.K) / (ms * 1e-3) / 1e12
            key = f"{s.M}x{s.N}x{s.K}" + ("" if name == "per_tensor" else f" {name}")
            out[key] = {"us": round(ms * 1e3, 2),
                        "median_us": round(1e3 * statistics.median(each), 2),
                        "TFLOP/s": round(tf, 1), "frac_of_peak": round(tf / peak, 4),
                        "peak": round(peak, 1), "scales": name,
                        "dtype_in": si.DTYPE_NAME[wl.dtype_in],
                        "dtype_out": si.DTYPE_NAME[wl.dtype_out],
                        "kernel": g.last_config()}
        del A, B, C, sfa, sfb
    return out


def measure_grouped(g, dev, stream, peaks, iters=10):
    """Secondary figures: the MoE projections as grouped GEMMs (one launch per layer),
    timed like the main workload (one launch per event pair after an L2 flush).  The
    roofline is the larger of the tensor time (2 sum M_e N K FLOPs at the measured peak)
    and the HBM time (every A_e, B_e and C_e moved once, at the measured copy
    bandwidth).  Parity is covered by the full-size tests."""
    tpeak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = {}
    for name, wl in si.MOE_WORKLOADS.items():
        counts = si.moe_counts(wl.experts, wl.rows, wl.seed)
        gen = torch.Generator(device=dev)
        gen.manual_seed(wl.seed)
        td_in, td_out = si.TORCH_DTYPE[wl.dtype_in], si.TORCH_DTYPE[wl.dtype_out]
        probs = [((torch.rand(m, wl.K, generator=gen, device=dev) * 2 - 1).to(td_in),
                  (torch.rand(wl.N, wl.K, generator=gen, device=dev) * 2 - 1).to(td_in),
                  torch.empty(m, wl.N, dtype=td_out, device=dev)) for m in counts]

        def run(*_):
            g.run_grouped(probs, stream=stream)

        for _ in range(3):
            flush.fill_(0.5)
            run()
        torch.cuda.synchronize()
        total, each = time_steps(run, [()], stream, iters, flush, per_step=True)
        us = 1e3 * total / iters
        flops = sum(2.0 * m * wl.N * wl.K for m in counts)
        nbytes = sum(2.0 * (m * wl.K + wl.N * wl.K + m * wl.N) for m in counts)
        tf, gbs = flops / us / 1e6, nbytes / us / 1e3
        t_tensor, t_hbm = flops / (tpeak * 1e6), nbytes / (hbm * 1e3)
        bound = "tensor" if t_tensor >= t_hbm else "hbm"
        out[name] = {"experts": wl.experts, "rows": wl.rows, "N": wl.N, "K": wl.K,
                     "rows_per_expert_min_max": [min(counts), max(counts)],
                     "us": round(us, 2), "median_us": round(1e3 * statistics.median(each), 2),
                     "TFLOP/s": round(tf, 1), "GB/s": round(gbs, 1), "bound": bound,
                     "frac_of_roofline": round(max(t_tensor, t_hbm) / us, 4),
                     "kernel": g.last_config()}
        del probs
    # a group of unequal tile costs (K from 256 to 16384 across its problems), timed with
    # the automatic scheduler (cluster launch control for such a group) and with
    # round-robin over resident CTAs forced, for comparison
    for name, wl in si.MIXED_K_WORKLOADS.items():
        Ks = si.mixed_k_values(wl.problems, wl.seed)
        gen = torch.Generator(device=dev)
        gen.manual_seed(wl.seed)
        td_in, td_out = si.TORCH_DTYPE[wl.dtype_in], si.TORCH_DTYPE[wl.dtype_out]
        probs = [((torch.rand(wl.M, k, generator=gen, device=dev) * 2 - 1).to(td_in),
                  (torch.rand(wl.N, k, generator=gen, device=dev) * 2 - 1).to(td_in),
                  torch.empty(wl.M, wl.N, dtype=td_out, device=dev)) for k in Ks]
        flops = sum(2.0 * wl.M * wl.N * k for k in Ks)
        entry = {"problems": wl.problems, "M": wl.M, "N": wl.N, "K": Ks}
        for key, sched in (("auto", 0), ("round_robin", 1)):
            g.set_config(scheduler=sched)

            def run(*_):
                g.run_grouped(probs, stream=stream)

            for _ in range(3):
                flush.fill_(0.5)
                run()
            torch.cuda.synchronize()
            total, each = time_steps(run, [()], stream, iters, flush, per_step=True)
            us = 1e3 * total / iters
            entry[key] = {"us": round(us, 2), "median_us": round(1e3 * statistics.median(each), 2),
                          "TFLOP/s": round(flops / us / 1e6, 1),
                          "frac_of_tensor_peak": round(flops / us / 1e6 / tpeak, 4),
                          "kernel": g.last_config()}
            g.reset_config()
        out[name] = entry
        del probs
    return out


def run_reference(args):
    """The oracle as it stands, timed on the host cores on bounded samples."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    wl, s = workload_shape(args.workload)
    A, B = si.make_operands(s.M, s.N, s.K, wl.dtype_in, wl.dist, wl.seed)
    rows_per_step = max(1, int(os.environ.get("GEMM_REF_ROWS", "64")))
    times = []
    for step in range(args.warmup + args.steps):
        rows = si.sample_indices(s.M, rows_per_step, seed=1000 + step)
        t0 = time.perf_counter()
        oracle.gemm_select(A, B, rows, None, wl.dtype_in, wl.dtype_out)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append((len(rows), dt))
    flops = sum(2.0 * r * s.N * s.K for r, _ in times)
    secs = sum(t for _, t in times)
    value = flops / secs / 1e12
    sample = (f"{rows_per_step} seeded rows of C per step ({2.0 * rows_per_step * s.N * s.K / 1e9:.2f}"
              f" GFLOP), binary64 accumulation, all host threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / max(len(times), 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "M": s.M, "N": s.N, "K": s.K,
                       "dtype_in": si.DTYPE_NAME[wl.dtype_in], "dtype_out": si.DTYPE_NAME[wl.dtype_out],
                       "dist": wl.dist, "seed": wl.seed},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_ours(args):
    from dense_gemm_blackwell_02_gb300.binding import Gemm

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", rank=rank, world_size=ws)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    wl, s = workload_shape(args.workload)
    M, N, K = s.M, s.N, s.K
    din, dout = wl.dtype_in, wl.dtype_out
    A_cpu, B_cpu = si.make_operands(M, N, K, din, wl.dist, wl.seed)
    A, B = A_cpu.to(dev), B_cpu.to(dev)
    C = torch.empty(M, N, dtype=si.TORCH_DTYPE[dout], device=dev)
    flush = (torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
             if args.l2 == "flush" else None)
    if flush is None:
        sets, set_bytes = operand_sets(A, B, C, dev)
        l2_note = (f"inputs larger than L2: {len(sets)} copies of A, B, C ({set_bytes >> 20} MiB in all,"
                   f" L2 {l2_bytes(dev) / 1e6:.0f} MB) used in turn, launches back to back")
    else:
        sets = [(A, B, C)]
        l2_note = "flushed (512 MiB write before each step, outside its events)"
    stream = torch.cuda.current_stream(dev)
    g = Gemm()
    if args.config:
        g.set_config(**json.loads(args.config))

    def run(a, b, c):
        g.run(a, b, c, stream=stream)

    for i in range(max(args.warmup, 3, len(sets))):
        if flush is not None:
            flush.fill_(1.0)
        run(*sets[i % len(sets)])
    torch.cuda.synchronize()
    code, word = g.device_status(stream)
    if code != 0:
        raise RuntimeError(f"device status after warm-up: {code} ({word:#x})")

    # R GEMMs per step, so that the K timed steps last about args.seconds: calibrated on
    # the wall time of a few warm-up steps of the same form.
    t0 = time.perf_counter()
    for i in range(16):
        if flush is not None:
            flush.fill_(1.0)
        run(*sets[i % len(sets)])
    torch.cuda.synchronize()
    per_launch_s = (time.perf_counter() - t0) / 16
    reps = max(1, int(round(args.seconds / max(args.steps, 1) / max(per_launch_s, 1e-6))))
    if args.reps:
        reps = args.reps
    if ws > 1:
        # every rank runs the same R (rank 0's)
        r = torch.tensor([reps], dtype=torch.int64, device=dev)
        torch.distributed.broadcast(r, 0)
        reps = int(r.item())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps if flush is not None else 1)]

    def step(i0):
        """One step: R GEMMs; returns (ms of the step's GEMMs, per-launch ms list)."""
        if flush is not None:
            for j in range(reps):
                flush.fill_(float(j & 7))
                ev[j][0].record(stream)
                run(*sets[0])
                ev[j][1].record(stream)
            torch.cuda.synchronize()
            each = [a.elapsed_time(b) for a, b in ev]
            return sum(each), each
        # back to back between one event pair (events between the launches would stop
        # each from starting early: programmatic dependent launch)
        ev[0][0].record(stream)
        for j in range(reps):
            run(*sets[(i0 + j) % len(sets)])
        ev[0][1].record(stream)
        torch.cuda.synchronize()
        t = ev[0][0].elapsed_time(ev[0][1])
        return t, [t / reps]

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)  # let the sampler take its first reading
    for i in range(args.warmup):
        step(i * reps)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = datetime.now()
    step_ms, each_ms = [], []
    for i in range(args.steps):
        t, each = step(i * reps)
        step_ms.append(t)
        each_ms += each
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall1 = datetime.now()
    local_ms = sum(step_ms)
    time.sleep(0.1)
    sampler.mark(wall0, wall1)
    clocks = sampler.stop()
    total_ms = max_over_ranks(local_ms, dev)
    code, word = g.device_status(stream)
    if code != 0:
        raise RuntimeError(f"device status after timing: {code} ({word:#x})")
    cfg = g.last_config()
    # The same workload timed the other way (compute-bound shapes are reported both
    # ways): back to back over operand copies larger than L2, or flushed per step.
    if flush is not None:
        other_sets, _ = operand_sets(A, B, C, dev)
        other_flush, other_how = None, "back to back over operand copies >= 4x L2"
    else:
        other_sets = [(A, B, C)]
        other_flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        other_how = "L2 flushed before each step"
    for i in range(2 * len(other_sets)):
        run(*other_sets[i % len(other_sets)])
    other_steps = min(args.steps, 20)
    other_ms = time_steps(run, other_sets, stream, other_steps, other_flush) / other_steps
    del other_sets, other_flush
    decode = measure_decode(g, dev, stream, peaks) if args.decode else None
    decode_small = (measure_decode(g, dev, stream, peaks, name="decode_small_m")
                    if args.decode > 1 else None)
    decode_swapped = measure_swapped(g, dev, stream, peaks) if args.decode > 1 else None
    fp8 = measure_fp8(g, dev, stream, peaks) if args.fp8 else None
    grouped = measure_grouped(g, dev, stream, peaks) if args.grouped else None
    flops = rl.gemm_flops(M, N, K)
    ms_per_step = total_ms / args.steps
    value = replica_throughput(ws, flops * reps, args.steps, total_ms)
    ms_per_launch = total_ms / (args.steps * reps)
    kernel_tflops = flops / (ms_per_launch * 1e-3) / 1e12

    # ---- end to end through the C ABI with pinned host buffers
    A_h = A_cpu.pin_memory()
    B_h = B_cpu.pin_memory()
    C_h = torch.empty(M, N, dtype=si.TORCH_DTYPE[dout]).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    g.run_host(A_h, B_h, C_h, din, dout, stream=stream)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        g.run_host(A_h, B_h, C_h, din, dout, stream=stream)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    out_b = 4 if dout == si.F32 else 2
    in_b = 1 if din in (si.E4M3, si.E5M2) else 2
    e2e = {"value": flops / e2e_s / 1e12, "unit": UNIT,
           "h2d_bytes_per_step": in_b * (M * K + N * K), "d2h_bytes_per_step": out_b * M * N}

    line = None
    if rank == 0:
        # ---- CPU oracle on whole rows: the cpu_baseline, and a full-size parity check
        import numpy as np
        from tests import parity as par
        rows, want, c64, cpu_s, threads = cpu_rows_sample(A_cpu, B_cpu, din, dout, M,
                                                           target_s=args.cpu_seconds)
        got = par.bits_of(C[rows])
        metrics = par.check(got, want, dout, what="bench rows", c64=c64,
                            sigma=par.sigma_of(A_cpu, B_cpu, rows), K=K)
        e2e_rows = par.bits_of(C_h[rows])
        assert np.array_equal(e2e_rows, got), "gemm_run_host disagrees with gemm_run"
        cpu_value = 2.0 * len(rows) * N * K / cpu_s / 1e12

        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        peak_note = f"{peak_src} bf16_tflops (burst; fp16 has the same dense rate)"
        ratio = 1.0
        if in_b == 1:
            ratio = NOMINAL_FP8_RATIO
            peak = fp8_peak(peaks)
            peak_sus *= ratio
            peak_note = (f"{peak_src} bf16_tflops (burst) x {NOMINAL_FP8_RATIO:g}, the nominal "
                         f"FP8 / bf16 dense ratio")
        # the tensor peak at the SM clock observed under load during the timed region
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        clock_peak = None
        if clocks.get("sm_mhz"):
            clock_peak = sms * TENSOR_FLOP_PER_SM_CLK * ratio * clocks["sm_mhz"] * 1e6 / 1e12
        traffic = None
        tf_path = os.path.join(ROOT, "profiles", "traffic.json")
        if os.path.exists(tf_path):
            rec = json.load(open(tf_path)).get(args.workload)
            # valid only for the same kernel source and the same launch configuration
            if (rec and rec.get("source_hash") == kernel_source_hash()
                    and rec.get("config") == cfg):
                traffic = rec.get("bytes_per_launch")
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": si.DTYPE_NAME[din], "data": "synthetic",
            "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                       "dtype_in": si.DTYPE_NAME[din], "dtype_out": si.DTYPE_NAME[dout],
                       "dist": wl.dist, "seed": wl.seed, "l2": l2_note,
                       "kernel": cfg, "parallelism": "replicas" if ws > 1 else "single-gpu"},
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": args.steps * reps,
            "roofline": {"bound": "tensor", "achieved": kernel_tflops, "peak": peak,
                         "unit": "TFLOP/s", "frac": kernel_tflops / peak, "traffic": traffic,
                         "peak_source": peak_note,
                         "frac_of_sustained": kernel_tflops / peak_sus,
                         "sustained_peak": peak_sus,
                         "clock_peak": clock_peak,
                         "frac_of_clock_peak": (kernel_tflops / clock_peak) if clock_peak else None,
                         "clock_peak_source": (f"{sms} SMs x {TENSOR_FLOP_PER_SM_CLK * ratio:g} "
                                               f"FLOP/clk x the median SM clock under load"),
                         "kernel_mcycles": (ms_per_launch * 1e-3 * clocks["sm_mhz"])
                                           if clocks.get("sm_mhz") else None,
                         "algorithmic_flops_per_launch": flops},
            "gemms_per_step": reps,
            "per_launch_us": {"median": 1e3 * statistics.median(each_ms), "best": 1e3 * min(each_ms),
                              "mean": 1e3 * ms_per_launch},
            "timed_region_s": (wall1 - wall0).total_seconds(),
            "timed_other_way": {"how": other_how, "us": 1e3 * other_ms,
                                "TFLOP/s": flops / (other_ms * 1e-3) / 1e12},
            "nominal_context": {"tensor_tflops": NOMINAL_TFLOPS, "hbm_gbs": NOMINAL_HBM_GBS,
                                "frac_of_nominal_tensor": kernel_tflops / NOMINAL_TFLOPS},
            "cpu_baseline": {"value": cpu_value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{len(rows)} whole rows of C ({2.0 * len(rows) * N * K / 1e9:.1f}"
                                       f" GFLOP) in {cpu_s:.1f} s"},
            "parity": {"rows_checked": len(rows), **metrics},
        }
        if decode is not None:
            line["decode"] = decode
        if decode_small is not None:
            line["decode_small_m"] = decode_small
        if decode_swapped:
            line["decode_swapped"] = decode_swapped
        if fp8 is not None:
            line["fp8"] = fp8
        if grouped is not None:
            line["grouped"] = grouped
        print(json.dumps(line))
    g.close()
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="square_4096", choices=sorted(si.WORKLOADS))
    ap.add_argument("--config", default=None, help="JSON gemm_config_t override (sweeps)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--seconds", type=float, default=12.0,
                    help="target length of the timed region (sets the GEMMs per step)")
    ap.add_argument("--reps", type=int, default=0, help="GEMMs per step (0: from --seconds)")
    ap.add_argument("--decode", type=int, default=2,
                    help="also time the M=256 decode shapes (HBM GB/s) into the line; "
                         "2 adds the M=1..128 decode shapes")
    ap.add_argument("--fp8", type=int, default=1,
                    help="also time the FP8 (E4M3 -> bf16) square shapes into the line")
    ap.add_argument("--grouped", type=int, default=1,
                    help="also time the MoE projections as grouped GEMMs into the line")
    ap.add_argument("--l2", default="flush", choices=["rotate", "flush"],
                    help="main workload: flush L2 before each separately timed step (default), "
                         "or cycle operand copies larger than L2 with launches back to back")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
