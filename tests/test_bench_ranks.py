"""The benchmark's process logic on CPU. The GPU arm is single-GPU by design (its GEMMs
share operand tiles inside a cluster with TMA multicast, kept to one-GPU processes): a
launch of several processes or GPUs is refused before the library is loaded. The
reference arm (the CPU oracle) runs on rank 0 only; other ranks exit 0 without work."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(args, **env):
    e = dict(os.environ)
    e.update({k: str(v) for k, v in env.items()})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=300, cwd=ROOT, env=e)


@pytest.mark.parametrize("args,env", [
    (["--workload", "tiny"], {"WORLD_SIZE": 2, "RANK": 0, "LOCAL_RANK": 0}),
    (["--workload", "tiny", "--gpus", "2"], {}),
], ids=["torchrun_world_2", "gpus_2"])
def test_gpu_arm_refuses_more_than_one_gpu(args, env):
    r = _bench(args, **env)
    assert r.returncode == 2, (r.returncode, r.stderr[-2000:])
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "ours" and d["n_gpus"] == 2 and "one GPU" in d["unavailable"]
    # refused before the library was loaded or a kernel was built
    assert "libflce" not in r.stderr and "Traceback" not in r.stderr


def test_gpu_arm_refusal_is_quiet_on_other_ranks():
    r = _bench(["--workload", "tiny"], WORLD_SIZE=2, RANK=1, LOCAL_RANK=1)
    assert r.returncode == 2 and not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_reference_arm_other_ranks_exit_without_work():
    r = _bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0"], WORLD_SIZE=2,
               RANK=1, LOCAL_RANK=1)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_bench_makes_no_process_group():
    """No collective, no NCCL: bench.py never creates a process group."""
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert "init_process_group" not in src and "torch.distributed" not in src


def test_launch_count_matches_the_band_schedule():
    import bench
    # forward: valid-row list + gather + GEMM + finalize + loss reduction
    total, bands, vc = bench.kernel_launches_per_step(65536, 4096, 128256, "mean")
    assert (bands, vc) == (21, 6144) and total == 5 + 4 + 3 * 21 + 1   # the workspace's capacity
    total, bands, vc = bench.kernel_launches_per_step(65536, 4096, 128256, "mean", 4608)
    assert bands == 28 and total == 5 + 4 + 3 * 28 + 1                  # a narrower band chosen on the device
    total, _, _ = bench.kernel_launches_per_step(65536, 4096, 128256, "mean", 4608, compact=False, compact_fwd=False)
    assert total == 3 + 2 + 3 * 28 + 1                                  # no valid-row compaction
    total, bands, vc = bench.kernel_launches_per_step(65536, 4096, 128256, "mean", row_band=16384,
                                                      compact_fwd=False)
    assert (bands, vc) == (8, 16384) and total == 3 + 1 + 4 * (1 + 2 + 3 * 8 + 1)   # four row bands


def test_clock_record_decides_a_remeasurement():
    """Thermal or hardware slowdown, or clocks held far below maximum with no reason,
    make the bench measure once more; the power cap alone does not."""
    import bench
    c = bench.ClockSampler(0)
    row = "0, {mhz}, 2070, 1300, 0x0, {hw}, Not Active, Not Active, {cap}"
    c.lines = [row.format(mhz=1600, hw="Not Active", cap="Active")] * 3
    assert c.summary()["reasons"] == ["sw_power_cap"] and not c.throttled()
    c.lines = [row.format(mhz=1600, hw="Active", cap="Active")] * 3
    assert c.throttled()
    c.lines = [row.format(mhz=900, hw="Not Active", cap="Not Active")] * 3
    assert c.throttled()
    c.lines = []
    assert c.summary()["samples"] == 0 and not c.throttled()


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference (the fp64 oracle on the host cores) prints one JSON line
    with the contract's keys, its cpu_baseline describing the same run, and an e2e with no
    host-device bytes."""
    r = _bench(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    # the time per step is the time of what ran: rows_per_step rows at the line's rate
    rows = d["config"]["rows_per_step"]
    assert abs(d["ms_per_step"] * d["value"] / 1000.0 - rows) <= 1e-6 * rows
