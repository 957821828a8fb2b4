"""The benchmark's multi-rank plumbing on CPU: two gloo ranks agree on the maximum
elapsed time and pass the barrier (each rank runs its own replica; there is no
collective on the data path)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(10.0 * (rank + 1), w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_launch_count_matches_the_band_schedule():
    import bench
    total, bands, vc = bench.kernel_launches_per_step(65536, 4096, 128256, "mean")
    assert (bands, vc) == (21, 6144) and total == 3 + 4 + 3 * 21 + 1   # the workspace's capacity
    total, bands, vc = bench.kernel_launches_per_step(65536, 4096, 128256, "mean", 4608)
    assert bands == 28 and total == 3 + 4 + 3 * 28 + 1                  # a narrower band chosen on the device
    total, _, _ = bench.kernel_launches_per_step(65536, 4096, 128256, "mean", 4608, compact=False)
    assert total == 3 + 2 + 3 * 28 + 1                                  # no valid-row compaction
    total, bands, vc = bench.kernel_launches_per_step(65536, 4096, 128256, "mean", row_band=16384)
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
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=root)
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
