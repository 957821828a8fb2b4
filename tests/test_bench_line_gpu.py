"""bench.py on the GPU prints one JSON line with every key of the benchmark contract: the
metric, the device-timed value, the roofline object of the dominant kernel, the CPU-oracle
baseline, the end-to-end figure with its host-device bytes, the launch count and the clock
record, and the side workloads' figures (the tiny workload with one small side workload,
so that it runs in seconds)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_carries_the_contract(gpu_lib):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny", "--steps", "3",
                        "--warmup", "3", "--cpu-seconds", "1", "--side-workloads", "small_vocab",
                        "--side-seconds", "0.2"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches",
                "clocks"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3 and d["dtype"] == "bf16"
    roof = d["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    # the roofline is the GEMM kind with the most device time, timed live per launch
    kinds = d["roofline_kernels"]
    assert set(kinds) == {"forward", "gradient", "dW", "dX"}
    top = max(kinds, key=lambda k: kinds[k]["ms_per_step"])
    assert roof["kernel"] == kinds[top]["kernel"] and roof["achieved"] == kinds[top]["achieved"]
    assert kinds["forward"]["launches_per_step"] == 1 and kinds["dX"]["launches_per_step"] >= 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 3 * d["gpu_launches_per_step_expected"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    # one GPU; a figure of another system is context, not a baseline
    assert d["n_gpus"] == 1 and d["vs_baseline"] is None and "liger_cutedsl_flce_b200" in d["context"]
    side = d["workloads"]["results"]["small_vocab"]
    assert side["N"] == 4096 and side["D"] == 2048 and side["V"] == 32000 and side["steps"] >= 5
    assert side["tokens_per_s"] > 0 and abs(side["tokens_per_s"] * side["ms_per_step_median"] / 1000 - 4096) < 1e-3
    # no N x V buffer: at this small N the gradient band spans half the vocabulary
    assert 0 < side["peak_mb"]["extra"] < side["peak_mb"]["logits_bf16_would_be"]
    # a step this short is also timed as a replayed CUDA graph of the same calls
    g = side["graph"]
    assert g["replays"] == side["steps"] and 0 < g["ms_per_step"] < 10 * side["ms_per_step_median"]
