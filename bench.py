"""Benchmark of the fused GEMM + epilogue engine on GB300.

One step = one pass of the whole hot path (TMA-fed tcgen05 main loop plus the
on-chip epilogue program) over one batch of the synthetic workload, with its
inputs resident in HBM.  The default workload is the MLP up-projection with
the interleaved SwiGLU epilogue (A 8192x4096, B 4096x28672 -> 8192x14336).

Prints ONE JSON line (rank 0).  Metric: fused GEMM+epilogue TFLOP/s
(2*M*N*K per step), with the roofline fraction, the bare-GEMM time (same main
loop, store-only epilogue) and the resulting epilogue overhead, an unfused
two-pass time, an end-to-end number through the C ABI from pinned host
buffers, and the CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle as the reference arm)
"""
from __future__ import annotations

import argparse
import gc
import glob
import hashlib
import json
import os
import random
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused GEMM+epilogue TFLOP/s and % of GB300 BF16 roofline; overhead vs bare GEMM"
# A step whose roofline time (the slower of its FLOPs at the bf16 peak and
# its bytes at the copy bandwidth) is below this is timed as a CUDA-graph
# replay, so that the host's launch cost cannot hide GPU time.
LATENCY_BOUND_SECONDS = 200e-6
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_NAME = "fused_gemm_epilogue_kernel"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="swiglu")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip bare / unfused comparison runs")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--per-config", default=None,
                    help="comma-separated workloads measured after the headline, each at full size with its "
                         "bare and unfused comparison (default: fp8,downproj,backward with the swiglu headline, "
                         "none otherwise; 'none' to skip)")
    return ap.parse_args()


# The benchmark configurations measured beside the SwiGLU headline: the FP8-
# training epilogue, the down-projection with residual and row RMS, and the
# GELU backward with column sums.
DEFAULT_PER_CONFIG = ("fp8", "downproj", "backward")


def per_config_names(args):
    if args.per_config is None:
        return list(DEFAULT_PER_CONFIG) if args.workload == "swiglu" else []
    if args.per_config.strip().lower() in ("", "none"):
        return []
    return [n.strip() for n in args.per_config.split(",") if n.strip()]


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "gemm_epilogue_transformer_smem_gb300", "csrc", "*"))):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from a committed ncu summary of this kernel and
    workload, if it was taken on the current kernel source (else None)."""
    cur = kernel_source_hash()
    for f in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(f).read()
        m = re.search(r"bench-traffic:\s*workload=(\S+)\s+source=(\S+)\s+bytes_per_launch=(\d+)", text)
        if m and m.group(1) == workload and m.group(2) == cur:
            return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.05 <= r[0] <= (self.t1 or 1e18) + 0.05]
        use = inside or rows[-3:]
        sm = [float(p[1]) for _, p in use if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in use if p[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in use:
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max((float(p[3]) for _, p in use
                                    if re.match(r"^[0-9.]+$", p[3])), default=None)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of x over all ranks (x itself at world size 1)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ oracle leg

def oracle_problem(w, inp):
    """The workload as the CPU oracle takes it: host copies of the same bf16
    bit patterns or FP8 codes, the same scalars."""
    import oracle
    from gemm_epilogue_transformer_smem_gb300 import synth

    def operand(t):
        if t is None:
            return None
        return synth.bf16_bits(t) if w.in_type == "bf16" else t.contiguous().cpu().numpy()

    def scalar(t):
        return 1.0 if t is None else float(t.item())

    first = (lambda t: None if t is None else t[0]) if w.batch > 1 else (lambda t: t)  # batch 0
    aux = synth.bf16_bits(first(inp.aux)) if inp.aux is not None else None
    row_scale = None if inp.row_scale is None else inp.row_scale.cpu().numpy()[:w.M]
    return oracle.Problem(operand(first(inp.A)), operand(first(inp.B)), list(w.program), b_is_nk=(w.b_layout == "nk"),
                          alpha=inp.alpha, bias=None if inp.bias is None else inp.bias.cpu().numpy(),
                          residual=aux if w.aux == "residual" else None,
                          preact=aux if w.aux == "preact" else None, fp8_scale=inp.fp8_scale,
                          B2=operand(inp.B2), a_type=w.in_type, b_type=w.in_type,
                          a_scale_inv=scalar(inp.a_scale_inv), b_scale_inv=scalar(inp.b_scale_inv),
                          col_scale=None if inp.col_scale is None else inp.col_scale.cpu().numpy(),
                          row_scale=row_scale)


def oracle_step(w, inp, prob, rows):
    """One bounded sample of the oracle's step: the listed rows of the GEMM
    + epilogue, then the workload's second pass on those rows."""
    import oracle
    from gemm_epilogue_transformer_smem_gb300 import synth
    ref = prob.rows(rows)
    if w.finish == "rmsnorm_backward":
        idx = rows
        oracle.rmsnorm_backward(ref["c_bf16"], synth.bf16_bits(inp.aux)[idx], inp.row_stat.cpu().numpy()[idx],
                                ref["row_stat"], w=inp.col_scale.cpu().numpy())
    return ref


def oracle_rows_sample(w, inp, seconds: float):
    """Times the CPU oracle on leading rows of the workload, growing the row
    count until about `seconds` of work.  Returns (tflops, rows, threads)."""
    import oracle

    prob = oracle_problem(w, inp)
    threads = oracle.cpu_threads()
    rows = max(1, min(w.M, threads))
    while True:
        t0 = time.perf_counter()
        oracle_step(w, inp, prob, list(range(rows)))
        dt = time.perf_counter() - t0
        if dt >= seconds * 0.5 or rows >= w.M:
            break
        rows = min(w.M, max(rows + 1, int(rows * min(8.0, seconds / max(dt, 1e-3)))))
    flops = 2.0 * rows * w.N * w.K
    return flops / dt / 1e12, rows, threads, dt


def host_inputs(w, seed=None):
    from gemm_epilogue_transformer_smem_gb300 import synth
    return synth.make_inputs(w, "cpu", seed=seed)


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on bounded samples."""
    from gemm_epilogue_transformer_smem_gb300 import synth
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    inp = host_inputs(w)
    # about 150 s of oracle work over the whole run, whatever the step count
    per_step = max(0.05, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    # size one step once, then run warmup + steps of that size
    _, rows, threads, _ = oracle_rows_sample(w, inp, per_step)
    prob = oracle_problem(w, inp)
    for _ in range(args.warmup):
        oracle_step(w, inp, prob, list(range(rows)))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, inp, prob, list(range(rows)))
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / dt / 1e12
    sample = "%d of %d rows%s (all %d columns, K=%d) per step" % (
        rows, w.M, " of the first of %d problems" % w.batch if w.batch > 1 else "", w.n_out, w.K)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "batch": w.batch, "program": list(w.program)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def time_steps(fn, steps, stream):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3  # seconds


def run_ours(args, world, rank, local):
    import torch

    from gemm_epilogue_transformer_smem_gb300 import api, build, synth

    build.build()
    dev = torch.device("cuda", local)
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w, dev)
    types = dict(a_type=w.in_type, b_type=w.in_type)
    plan = api.Plan(w.M, w.N, w.K, w.program, b_layout=w.b_layout, dual=w.dual, batch=w.batch, **types)
    out = api.allocate_outputs(plan, dev)
    stream = torch.cuda.current_stream(dev)
    kw = dict(alpha=inp.alpha, fp8_scale=inp.fp8_scale, bias=inp.bias, aux=inp.aux, B2=inp.B2,
              col_scale=inp.col_scale, row_scale=inp.row_scale, a_scale_inv=inp.a_scale_inv,
              b_scale_inv=inp.b_scale_inv)
    fin = make_finish(w, inp, out, dev)
    launches_per_step = 2 if fin else 1

    def gemm():
        api.run_program(plan, inp.A, inp.B, out, **kw)

    def step():
        gemm()
        if fin:
            fin()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    status = plan.query_status(out.workspace)
    if status != 0:
        raise RuntimeError("fused kernel reported status %d" % status)

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("begin")
    graph = None
    if fin:
        # The GEMM's own launch time (the roofline's kernel) from events
        # around each GEMM launch inside the timed loop.
        seconds, gemm_seconds, fin_seconds = time_steps_split(gemm, fin, args.steps, stream)
    elif roofline_seconds(w) < LATENCY_BOUND_SECONDS:
        # A short step (launch bound, or a skinny GEMM of a few tens of
        # microseconds): the K steps are captured once in a CUDA graph and
        # the replay is timed, so host launch cost is excluded.
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(args.steps):
                step()
        stream.wait_stream(cap)
        graph.replay()
        torch.cuda.synchronize()
        seconds = time_steps(graph.replay, 1, stream)
        gemm_seconds = None
    else:
        seconds = time_steps(step, args.steps, stream)
        gemm_seconds = None
    torch.cuda.synchronize()
    clocks.mark("end")
    barrier(world)
    seconds = max_over_ranks(seconds, world)
    clk = clocks.stop() if rank == 0 else None
    flops = float(w.flops)
    value = aggregate_value(flops * args.steps, world, seconds) / 1e12
    ms_per_step = seconds / args.steps * 1e3
    fused_tflops = flops / ((gemm_seconds if gemm_seconds is not None else seconds) / args.steps) / 1e12

    extras = {}
    if not args.no_extras:
        extras = compare_variants(w, plan, inp, out, kw, fin, step, dev, stream, args.steps)

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(plan, w, inp, out, kw, dev, max(3, min(args.steps, 20)), world, fin)

    l2_note = "no flush: inputs + output (%d MB) exceed the 129 MB L2" % (
        sum(t.numel() * t.element_size() for t in (inp.A, inp.B, inp.B2, inp.aux, inp.bias)
            if t is not None) // 2 ** 20 + plan.M * plan.n_out * 2 // 2 ** 20)
    has_fin = fin is not None
    per_config = {}
    names = per_config_names(args)
    if names:
        # The headline's buffers are released first: each configuration
        # allocates its own full-size inputs and outputs.
        del inp, out, plan, kw, fin, gemm, step
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        for name in names:
            per_config[name] = measure_config(name, args, dev, stream, local, world, rank)
            torch.cuda.empty_cache()

    if rank != 0:
        return
    peaks, src = load_peaks()
    roofline = roofline_entry(w, fused_tflops)
    second_pass = None
    if has_fin:
        # The memory-bound second pass, against the measured copy bandwidth
        # (its time includes the clearing of dw that precedes each launch).
        t_fin = fin_seconds / args.steps
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        nbytes = finish_bytes(w)
        second_pass = {"kernel": "rmsnorm_bwd_kernel", "bound": "hbm", "us_per_launch": t_fin * 1e6,
                       "achieved": nbytes / t_fin / 1e9, "peak": hbm, "unit": "GB/s",
                       "frac": nbytes / t_fin / 1e9 / hbm, "algorithmic_bytes_per_launch": nbytes,
                       "traffic": profiled_traffic(w.name + ":second_pass"),
                       "peak_source": "%s HBM copy" % src}
    cpu = None
    if not args.no_cpu and world == 1:  # the oracle baseline is timed at N = 1 only
        host = synth.make_inputs(w, "cpu")
        tf, rows, threads, dt = oracle_rows_sample(w, host, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": "%d of %d rows%s x all %d output columns, K=%d (%.1f s)" % (
                   rows, w.M, " of the first of %d problems" % w.batch if w.batch > 1 else "", w.n_out, w.K, dt)}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.in_type == "bf16" else w.in_type,
        "data": "synthetic",
        "timing": "CUDA-graph replay of the %d steps" % args.steps if graph is not None else "stream launches",
        "us_per_step": seconds / args.steps * 1e6,
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "batch": w.batch, "b_layout": w.b_layout,
                   "program": list(w.program), "parallelism": "replicas" if world > 1 else "single",
                   "l2": l2_note},
        "roofline": roofline,
        **({"second_pass": second_pass} if second_pass else {}),
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk,
        **extras,
    }
    if per_config:
        line["per_config"] = per_config
    print(json.dumps(line), flush=True)


def compare_variants(w, plan, inp, out, kw, fin, step, dev, stream, steps):
    """Fused, bare GEMM (same main loop, store-only program) and unfused (bare
    GEMM + separate epilogue pass) timed in interleaved rounds so that all
    three see the same clock and power state; medians."""
    from gemm_epilogue_transformer_smem_gb300 import api, native
    types = dict(a_type=w.in_type, b_type=w.in_type)
    scales = dict(a_scale_inv=kw.get("a_scale_inv"), b_scale_inv=kw.get("b_scale_inv"))
    flops = float(w.flops)
    bare = api.Plan(w.M, w.N, w.K, ["store_bf16"], b_layout=w.b_layout, dual=w.dual, batch=w.batch, **types)
    bare_out = api.allocate_outputs(bare, dev)

    def bare_step():
        bare.run(inp.A, inp.B, C=bare_out.C, workspace=bare_out.workspace, B2=inp.B2, **scales)

    scratch = bare_out.C

    def unfused_step():
        api.run_program(plan, inp.A, inp.B, out, unfused_scratch=scratch, **kw)
        if fin:
            fin()

    fns = [("fused", step), ("bare", bare_step)]
    if w.batch == 1:  # the separate pass runs single problems
        try:
            unfused_step()
            fns.append(("unfused", unfused_step))
        except native.GemmEpiError:  # a program the separate pass does not cover
            pass
    for _, f in fns[1:]:
        for _ in range(3):
            f()
    n = max(3, min(steps // 4, 10))
    t = {name: [] for name, _ in fns}
    rng = random.Random(0)
    for _ in range(15):
        rng.shuffle(fns)  # no variant keeps a fixed place in the power-cap cycle
        for name, fn in fns:
            t[name].append(time_steps(fn, n, stream) / n)
    med = {k: statistics.median(v) for k, v in t.items()}
    # The floor of any two-pass design: the bare GEMM plus a separate pass
    # (and the second pass, where the step has one) moving only its
    # algorithmic bytes at the measured HBM copy bandwidth.
    hbm_gbs = float(load_peaks()[0].get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ideal = med["bare"] + (separate_pass_bytes(w) + (finish_bytes(w) if fin else 0)) / (hbm_gbs * 1e9)
    return {
        "bare_gemm_ms": med["bare"] * 1e3, "bare_gemm_tflops": flops / med["bare"] / 1e12,
        "unfused_ideal_ms": ideal * 1e3, "fused_vs_unfused_ideal": ideal / med["fused"],
        "unfused_ms": med["unfused"] * 1e3 if "unfused" in med else None,
        "unfused_tflops": flops / med["unfused"] / 1e12 if "unfused" in med else None,
        "fused_ms_interleaved": med["fused"] * 1e3,
        "overhead_vs_bare": med["fused"] / med["bare"] - 1.0,
        "comparison": "15 rounds of %d launches each, order shuffled per round, medians" % n,
    }


def roofline_entry(w, fused_tflops):
    """The roofline object of one fused launch: tensor bound against the
    measured bf16 burst peak (x 2 for 8-bit operands), or HBM bound against
    the measured copy bandwidth when the operand bytes take longer."""
    peaks, src = load_peaks()
    flops = float(w.flops)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_source = "%s burst bf16 (cuBLAS)" % src
    if w.in_type != "bf16":
        # FP8 operands: the measured bf16 peak times the nominal dense
        # FP8 / BF16 ratio (4.5 / 2.25 PFLOP/s).
        peak *= 2.0
        peak_source = "%s burst bf16 (cuBLAS) x 2, the nominal dense fp8/bf16 ratio" % src
    traffic = profiled_traffic(w.name)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    nbytes = fused_bytes(w)
    if nbytes / (hbm * 1e9) > flops / (peak * 1e12):
        # Reading the operands takes longer at HBM speed than the FLOPs at
        # tensor speed (a skinny GEMM): the HBM roofline binds.
        t_launch = flops / (fused_tflops * 1e12)
        roofline = {"bound": "hbm", "achieved": nbytes / t_launch / 1e9, "peak": hbm, "unit": "GB/s",
                    "frac": nbytes / t_launch / 1e9 / hbm, "traffic": traffic,
                    "peak_source": "%s HBM copy" % src, "algorithmic_bytes_per_launch": nbytes,
                    "tflops": fused_tflops}
    else:
        roofline = {"bound": "tensor", "achieved": fused_tflops, "peak": peak, "unit": "TFLOP/s",
                    "frac": fused_tflops / peak, "traffic": traffic, "peak_source": peak_source,
                    "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes}
    if "bf16_tflops_sustained" in peaks and roofline["bound"] == "tensor":
        # For context: the same against the power-capped sustained figure
        # (a seconds-long loop), the regime long timed regions run in.
        sustained = float(peaks["bf16_tflops_sustained"]) * (2.0 if w.in_type != "bf16" else 1.0)
        roofline["frac_of_sustained"] = fused_tflops / sustained
    return roofline


def measure_config(name, args, dev, stream, local, world, rank):
    """One more benchmark configuration at full size, measured the way the
    headline is: a burst of fused launches with CUDA events, then the
    interleaved fused / bare / unfused rounds, with the clocks sampled over
    both.  Returns the config's entry of the line's per_config object."""
    import torch
    from gemm_epilogue_transformer_smem_gb300 import api, synth
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w, dev)
    types = dict(a_type=w.in_type, b_type=w.in_type)
    plan = api.Plan(w.M, w.N, w.K, w.program, b_layout=w.b_layout, dual=w.dual, batch=w.batch, **types)
    out = api.allocate_outputs(plan, dev)
    kw = dict(alpha=inp.alpha, fp8_scale=inp.fp8_scale, bias=inp.bias, aux=inp.aux, B2=inp.B2,
              col_scale=inp.col_scale, row_scale=inp.row_scale, a_scale_inv=inp.a_scale_inv,
              b_scale_inv=inp.b_scale_inv)
    fin = make_finish(w, inp, out, dev)

    def gemm():
        api.run_program(plan, inp.A, inp.B, out, **kw)

    def step():
        gemm()
        if fin:
            fin()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    status = plan.query_status(out.workspace)
    if status != 0:
        raise RuntimeError("fused kernel reported status %d on %s" % (status, name))
    steps = max(20, min(args.steps, 100))
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("begin")
    if fin:
        seconds, gemm_seconds, _ = time_steps_split(gemm, fin, steps, stream)
    else:
        seconds = gemm_seconds = time_steps(step, steps, stream)
    seconds = max_over_ranks(seconds, world)
    gemm_seconds = max_over_ranks(gemm_seconds, world)
    fused_tflops = float(w.flops) / (gemm_seconds / steps) / 1e12
    extras = {} if args.no_extras else compare_variants(w, plan, inp, out, kw, fin, step, dev, stream, steps)
    torch.cuda.synchronize()
    clocks.mark("end")
    clk = clocks.stop() if rank == 0 else None
    entry = {"M": w.M, "N": w.N, "K": w.K, "program": list(w.program), "b_layout": w.b_layout,
             "steps": steps, "ms_per_step": seconds / steps * 1e3,
             "value": aggregate_value(float(w.flops) * steps, world, seconds) / 1e12,
             "fused_tflops": fused_tflops, "roofline": roofline_entry(w, fused_tflops), "clocks": clk}
    if fin:
        entry["gemm_ms"] = gemm_seconds / steps * 1e3
    entry.update(extras)
    del inp, out, plan
    return entry


def roofline_seconds(w):
    """The slower of the step's FLOPs at the measured bf16 (or 2x for 8-bit)
    peak and its algorithmic bytes at the measured copy bandwidth."""
    peaks, _ = load_peaks()
    tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * (2.0 if w.in_type != "bf16" else 1.0)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return max(w.flops / (tf * 1e12), fused_bytes(w) / (hbm * 1e9))


def fused_bytes(w):
    """Algorithmic bytes of one fused launch: A and B (and B2) read once,
    any auxiliary tensor read, the program's outputs written (vectors and
    reductions ignored)."""
    prog = [op.partition(":")[0] for op in w.program]
    esz = 1 if w.in_type != "bf16" else 2
    b = w.batch * (w.M * w.K + w.K * w.N) * esz
    if w.aux:
        b += w.batch * w.M * w.n_out * 2
    if "store_bf16" in prog:
        b += w.batch * w.M * w.n_out * 2
    if "store_e4m3" in prog:
        b += w.batch * w.M * w.n_out
    return b


def separate_pass_bytes(w):
    """Algorithmic bytes of the epilogue as its own pass after a bare GEMM
    that stored the bf16 accumulator: that accumulator and any auxiliary
    tensor read, the program's outputs written (reduction vectors ignored)."""
    prog = [op.partition(":")[0] for op in w.program]
    rows = w.batch * w.M
    b = rows * w.N * 2
    if w.aux:
        b += rows * w.n_out * 2
    if "store_bf16" in prog:
        b += rows * w.n_out * 2
    if "store_e4m3" in prog:
        b += rows * w.n_out
    return b


def finish_bytes(w):
    """Algorithmic bytes of one RMSNorm-backward second pass: dy and x read
    and dx written (bf16), w, S and r read and dw written (fp32)."""
    return 3 * w.M * w.n_out * 2 + 4 * (2 * w.n_out + 2 * w.M)


def make_finish(w, inp, out, dev):
    """The workload's second pass as a callable (None without one): the
    RMSNorm backward from the GEMM's stored dy and row reduction."""
    if w.finish != "rmsnorm_backward":
        return None
    import torch
    from gemm_epilogue_transformer_smem_gb300 import api
    dx = torch.empty(out.C.shape, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(out.C.shape[1], dtype=torch.float32, device=dev)

    def fin(aux=None, C=None, row_out=None, w_=None, s_=None):
        api.rmsnorm_backward(out.C if C is None else C, inp.aux if aux is None else aux,
                             inp.row_stat if s_ is None else s_, out.row_out if row_out is None else row_out,
                             w=inp.col_scale if w_ is None else w_, dx=dx, dw=dw)

    fin.outputs = (dx, dw)
    return fin


def time_steps_split(first, second, steps, stream):
    """Times `steps` of first(); second() with events around the whole loop
    and around each call; returns (total seconds, seconds in first(),
    seconds in second())."""
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    marks = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    start.record(stream)
    for a, b, c in marks:
        a.record(stream)
        first()
        b.record(stream)
        second()
        c.record(stream)
    end.record(stream)
    end.synchronize()
    return (start.elapsed_time(end) / 1e3, sum(a.elapsed_time(b) for a, b, _ in marks) / 1e3,
            sum(b.elapsed_time(c) for _, b, c in marks) / 1e3)


def measure_e2e(plan, w, inp, out, kw, dev, steps, world, fin=None):
    """Same metric through the C ABI with host buffers: every step copies its
    inputs from pinned host memory, runs, and reads its outputs back.

    Pipelined (the reported value): step i's host-to-device copy, compute and
    device-to-host copy run on three streams over two device buffer sets, so
    one step's transfers overlap its neighbours' kernels; events guard each
    buffer's reuse.  The serial figure (copy in, run, copy out, one stream)
    is reported beside it."""
    import torch
    from gemm_epilogue_transformer_smem_gb300 import api

    names = ("A", "B", "bias", "aux", "B2", "a_scale_inv", "b_scale_inv", "col_scale", "row_stat", "row_scale")
    src = dict(zip(names, (inp.A, inp.B, inp.bias, inp.aux, inp.B2, inp.a_scale_inv, inp.b_scale_inv,
                           inp.col_scale, inp.row_stat, inp.row_scale)))
    h = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in src.items()}

    def buffers():
        d = {k: (torch.empty_like(v, device=dev) if v is not None else None) for k, v in h.items()}
        o = api.allocate_outputs(plan, dev)
        f = make_finish(w, inp, o, dev) if fin else None
        outs = [t for t in (o.C, o.C8, o.amax, o.row_out, o.col_out) if t is not None]
        if f:
            outs += list(f.outputs)
        ho = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        return {"d": d, "o": o, "f": f, "outs": outs, "ho": ho}

    sets = [buffers(), buffers()]
    h2d = sum(v.numel() * v.element_size() for v in h.values() if v is not None)
    d2h = sum(t.numel() * t.element_size() for t in sets[0]["outs"])

    def copy_in(b):
        for k, v in h.items():
            if v is not None:
                b["d"][k].copy_(v, non_blocking=True)

    def compute(b, stream=None):
        d = b["d"]
        api.run_program(plan, d["A"], d["B"], b["o"], alpha=kw["alpha"], fp8_scale=kw["fp8_scale"],
                        bias=d["bias"], aux=d["aux"], B2=d["B2"], a_scale_inv=d["a_scale_inv"],
                        b_scale_inv=d["b_scale_inv"], col_scale=d["col_scale"], row_scale=d["row_scale"],
                        stream=stream)
        if b["f"]:
            b["f"](aux=d["aux"], w_=d["col_scale"], s_=d["row_stat"])

    def copy_out(b):
        for t, ht in zip(b["outs"], b["ho"]):
            ht.copy_(t, non_blocking=True)

    # Serial: one stream, one buffer set.
    stream = torch.cuda.current_stream(dev)

    def serial_step():
        copy_in(sets[0])
        compute(sets[0])
        copy_out(sets[0])

    for _ in range(2):
        serial_step()
    torch.cuda.synchronize()
    barrier(world)
    serial_s = max_over_ranks(time_steps(serial_step, steps, stream), world)

    # Pipelined: three streams, two buffer sets.
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, run_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def pipelined(n):
        for i in range(n):
            k = i % 2
            b = sets[k]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(run_done[k])      # step i-2's kernel has read these inputs
                copy_in(b)
                in_ready[k].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(in_ready[k])
                if i >= 2:
                    s_run.wait_event(out_done[k])     # step i-2's outputs have been read back
                compute(b, stream=s_run)
                run_done[k].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(run_done[k])
                copy_out(b)
                out_done[k].record(s_out)

    pipelined(4)
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    pipelined(steps)
    s_in.wait_stream(s_out)
    end.record(s_in)
    end.synchronize()
    seconds = max_over_ranks(start.elapsed_time(end) / 1e3, world)
    value = aggregate_value(float(w.flops) * steps, world, seconds) / 1e12
    return {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": seconds / steps * 1e3,
            "mode": "pipelined: copy-in, compute and copy-out of consecutive steps on three streams, "
                    "two device buffer sets",
            "serial_value": aggregate_value(float(w.flops) * steps, world, serial_s) / 1e12,
            "serial_ms_per_step": serial_s / steps * 1e3}


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
