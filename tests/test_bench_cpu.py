"""bench.py on the CPU: the reference arm's JSON line (the oracle, timed on
the host), and the algorithmic byte counts behind the two-pass floor and the
second pass's roofline."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gemm_epilogue_transformer_smem_gb300 import synth  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                          "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600, check=True)
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and "rows" in d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["gpu_launches"] == 0 and d["config"]["workload"] == "tiny"


def test_separate_pass_bytes():
    w = synth.WORKLOADS
    # swiglu: the stored 8192 x 28672 accumulator read, 8192 x 14336 written
    assert bench.separate_pass_bytes(w["swiglu"]) == 8192 * 28672 * 2 + 8192 * 14336 * 2
    # fp8: accumulator read, bf16 and e4m3 outputs written
    assert bench.separate_pass_bytes(w["fp8"]) == 8192 * 8192 * (2 + 2 + 1)
    # backward: accumulator and pre-activation read, output written
    assert bench.separate_pass_bytes(w["backward"]) == 8192 * 16384 * (2 + 2 + 2)
    # dswiglu: 8192 x 14336 accumulator, 8192 x 28672 pre-activations read and outputs written
    assert bench.separate_pass_bytes(w["dswiglu"]) == 8192 * 14336 * 2 + 8192 * 28672 * (2 + 2)


def test_second_pass_bytes():
    w = synth.WORKLOADS["drmsnorm"]
    # dy and x read, dx written (bf16); w, S, r read and dw written (fp32)
    assert bench.finish_bytes(w) == 3 * 16384 * 4096 * 2 + 4 * (2 * 4096 + 2 * 16384)
    assert bench.finish_bytes(w) / 1e6 == pytest.approx(402.8, abs=0.1)


def test_fused_bytes_and_binding_roofline():
    w = synth.WORKLOADS
    # swiglu: A 8192 x 4096 and B 4096 x 28672 read, C 8192 x 14336 written (bf16)
    assert bench.fused_bytes(w["swiglu"]) == (8192 * 4096 + 4096 * 28672 + 8192 * 14336) * 2
    # e4m3 operands are one byte each; the outputs stay bf16 + e4m3
    assert bench.fused_bytes(w["fp8in"]) == 2 * 8192 * 8192 + 8192 * 8192 * (2 + 1)
    # batched: every problem's operands and outputs
    assert bench.fused_bytes(w["moe8"]) == 8 * ((2048 * 4096 + 4096 * 28672) * 2 + 2048 * 14336 * 2)
    # the prefill-sized GEMMs are tensor bound, the 64-token decode step HBM bound
    for name in ("swiglu", "fp8", "downproj", "backward", "dswiglu", "moe8"):
        wl = w[name]
        peaks, _ = bench.load_peaks()
        tf = float(peaks.get("bf16_tflops", bench.FALLBACK_PEAKS["bf16_tflops"]))
        assert bench.roofline_seconds(wl) == pytest.approx(wl.flops / (tf * 1e12)), name
    assert bench.roofline_seconds(w["decode"]) < bench.LATENCY_BOUND_SECONDS  # timed as a graph replay
    assert bench.roofline_seconds(w["swiglu"]) > bench.LATENCY_BOUND_SECONDS


def test_per_config_defaults_to_the_other_benchmark_configs():
    """The default (SwiGLU) line also measures the FP8, down-projection and
    backward configurations; other workloads measure none unless asked."""
    class A:
        workload, per_config = "swiglu", None
    assert bench.per_config_names(A) == ["fp8", "downproj", "backward"]
    A.workload = "fp8"
    assert bench.per_config_names(A) == []
    A.per_config = "backward, dswiglu"
    assert bench.per_config_names(A) == ["backward", "dswiglu"]
    A.per_config = "none"
    assert bench.per_config_names(A) == []
    for name in bench.DEFAULT_PER_CONFIG:
        assert name in synth.WORKLOADS
