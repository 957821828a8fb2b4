"""Benchmark: fused linear cross-entropy forward + backward tokens/s on GB300.

One step = flce_forward + flce_backward (grad_out = 1.0) over one batch of the
headline workload, N=65536 tokens (batch 8 x 8192), D=4096, V=128256, bf16, 5%
ignored rows, mean reduction -- the Llama-3-8B language-model head of "Cutting LLM
Memory by 84%: A Deep Dive into Fused Kernels" ("The Logit Bottleneck") and of the
Liger-Kernel PR #1291 BT sweep. Inputs are synthetic (seeded, see workloads).

Prints ONE JSON line. The GPU arm runs on one GPU in one process: its GEMMs share
operand tiles between the CTAs of a cluster with TMA multicast, which this library
keeps to single-GPU processes, so a launch with WORLD_SIZE > 1 or --gpus > 1 is
refused before the library is loaded. Beside the headline figure the line carries the
other four workloads and the memory-benchmark shape ("workloads"), each timed for a
fraction of a second.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle on bounded samples of the same workload
(the reference arm); under torchrun only rank 0 runs it, the other ranks exit 0.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "FLCE fwd+bwd tokens/s at N=65536,D=4096,V=128256 bf16; % of bf16 TC peak; peak MB"
UNIT = "tokens/s"
# Liger-Kernel PR #1291: CuTe-DSL FLCE fwd+bwd p50 = 194 ms at BT=65536, V=128256, H=4096, bf16, on B200.
PAGES_TOKENS_PER_S = 65536 / 0.194


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    def throttled(self) -> bool:
        """Hardware or thermal slowdown seen, or the median clock far below the maximum
        with no reason given."""
        s = self.summary()
        if set(s["reasons"]) & {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}:
            return True
        return bool(s["sm_mhz"] is not None and s["sm_max_mhz"] and not s["reasons"]
                    and s["sm_mhz"] < 0.6 * s["sm_max_mhz"])

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        power = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                power.append(float(f[3]))
            except (IndexError, ValueError):
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
               "samples": len(sm), "power_w": statistics.median(power) if power else None}
        if getattr(self, "remeasured", False):
            out["remeasured"] = True
        return out


def launch_env():
    """(world size, rank) of a torchrun launch, or (1, 0) for a plain process. No process
    group is ever created: the GPU arm refuses a world size above one, and the reference
    arm runs on rank 0 alone."""
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))


ONE_GPU_ONLY = ("one GPU per process only: the GEMMs share each operand tile among the CTAs of a "
                "cluster with TMA multicast, which this library keeps to single-GPU processes; "
                "run bench.py without torchrun and with --gpus 1")


def refuse_multi_gpu(args, world: int, rank: int) -> int:
    """The GPU arm in a launch of several processes or GPUs: print why (rank 0) and return
    the exit status, before the library is loaded or a device is touched."""
    if rank == 0:
        print(json.dumps({"impl": "ours", "n_gpus": max(args.gpus, world), "unavailable": ONE_GPU_ONLY}), flush=True)
    print(f"bench.py: {ONE_GPU_ONLY}", file=sys.stderr, flush=True)
    return 2


L2_BYTES = 129e6  # GB300's L2


def data_recipe(wl) -> str:
    """The synthetic input recipe of a workload, for the JSON line's `data`."""
    ign = f"{wl.ignore_frac:.0%} ignore_index" if wl.ignore_frac else "no ignored rows"
    return f"synthetic (seeded; X~N(0,1), W~N(0,1/D) in bf16, {wl.target_dist} targets, {ign})"


def l2_note(wl) -> str:
    """Whether the inputs outsize the L2 (then no flush is needed between steps)."""
    x, w = wl.N * wl.D * 2, wl.D * wl.V * 2
    if min(x, w) > L2_BYTES:
        return f"inputs larger than L2 (X {x / 1e9:.2f} GB, W {w / 1e9:.2f} GB > 129 MB); no flush"
    if x + w > L2_BYTES:
        return (f"inputs larger than L2 together (X {x / 1e6:.1f} MB + W {w / 1e6:.1f} MB > 129 MB); "
                f"no flush")
    return (f"inputs fit in the 129 MB L2 (X {x / 1e6:.2f} MB + W {w / 1e6:.2f} MB) and stay there between "
            f"steps; no flush (a latency-bound size)")


def kernel_launches_per_step(N, D, V, reduction, vc=None, compact=True, row_band=0, compact_fwd=True):
    """Kernels the library launches per step: (the forward's valid-row list and gather, with
    a workspace that has room for them) forward GEMM + finalize (+ loss reduction),
    backward denominator, then per row band (one, or ceil(N / row_band)) row coefficients
    (+ valid-row compaction and gather) + 3 GEMMs per vocabulary band + the dX cast. vc is
    the band width (flce_backward_band_width on the device); without it, the workspace's
    band capacity. compact: the backward compacts the valid rows (a 16-bit dX)."""
    rows = row_band if 0 < row_band < N else N
    if vc is None:
        unit = 512  # one cluster's vocabulary tiles: 2 CTA pairs x 256
        vc = max(unit, min(16384, ((3 << 28) // (2 * rows)) // unit * unit))
        half = (((V + 1) // 2) + unit - 1) // unit * unit
        vc = min(vc, half)
    bands = -(-V // vc)
    fwd = (2 if compact_fwd else 0) + 1 + 1 + (0 if reduction == "none" else 1)
    bwd = 1 + -(-N // rows) * (1 + (2 if compact else 0) + 3 * bands + 1)
    return fwd + bwd, bands, vc


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_sample_rate(wl, X, W, y, rows: int):
    """fp64 oracle fwd+bwd on the first `rows` rows with the full vocabulary; returns (tokens/s, seconds)."""
    import oracle
    t0 = time.perf_counter()
    oracle.forward_backward(X[:rows], W, y[:rows], wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                            wl.reduction)
    dt = time.perf_counter() - t0
    return rows / dt, dt


def oracle_sample_for(wl, X, W, y, seconds: float, chunk: int = 256):
    """fp64 oracle fwd+bwd over successive chunks of rows (full vocabulary) until `seconds`
    of CPU time have passed or every row is done; returns (tokens/s, rows, seconds)."""
    rows, dt = 0, 0.0
    while rows < X.shape[0] and (rows == 0 or dt < seconds):
        n = min(chunk, X.shape[0] - rows)
        sl = slice(rows, rows + n)
        r, t = oracle_sample_rate(wl, X[sl], W, y[sl], n)
        rows += n
        dt += t
    return rows / dt, rows, dt


def pipeline_waits(ws, phase):
    """Shares of the MMA thread's cycles spent waiting, read from the workspace header of
    the last call, which a library built with -DFLCE_WAIT_STATS=1 fills: per GEMM kind,
    cycles the MMA thread waited for operands (full stages) and for a drained accumulator,
    and cycles the producer waited for a free stage, over the MMA thread's total."""
    h = ws[:256].cpu().view(torch.int64).tolist()
    kinds = {"forward": -1} if phase == "fwd" else {"gradient": 0, "dW": 1, "dX": 2}
    out = {}
    for name, k in kinds.items():
        base = (32 + 32 * (k + 1)) // 8
        full, tempty, empty, total = h[base:base + 4]
        if total > 0:
            out[name] = {"mma_waits_operands": full / total, "mma_waits_epilogue": tempty / total,
                         "producer_waits_free_stage": empty / total}
    return out


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, wl):
    X, W, y = make_inputs(wl)
    rows = min(args.oracle_rows, wl.N)
    rates, times = [], []
    for _ in range(args.warmup):
        oracle_sample_rate(wl, X, W, y, rows)
    for _ in range(args.steps):
        r, dt = oracle_sample_rate(wl, X, W, y, rows)
        rates.append(r)
        times.append(dt)
    ms_step = 1000.0 * statistics.median(times)
    value = rows / (ms_step / 1000.0)
    sample = (f"fp64 oracle fwd+bwd of {rows} rows x full V={wl.V} (D={wl.D}) per step; "
              f"tokens/s = rows / time; {args.steps} steps after {args.warmup} warm-up")
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": data_recipe(wl),
        "config": {"workload": wl.name, "N": wl.N, "D": wl.D, "V": wl.V, "reduction": wl.reduction,
                   "ignore_frac": wl.ignore_frac, "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------- GPU arm

class Problem:
    """Device buffers of one workload and its forward / backward calls on one stream."""

    def __init__(self, flce, wl, dev, stream, X, W, y, row_band=0):
        self.flce, self.wl, self.dev, self.stream = flce, wl, dev, stream
        N, D, V = wl.N, wl.D, wl.V
        self.X, self.W, self.y = X, W, y
        self.ws_f = flce.flce_workspace_size(N, D, V, False)
        self.row_band = row_band if 0 < row_band < N else 0
        self.opt_b = flce.make_options(row_band=self.row_band) if self.row_band else None
        self.ws_b = flce.flce_workspace_size(self.row_band or N, D, V, True)
        self.loss = torch.empty(1, dtype=torch.float32, device=dev)
        self.lse = torch.empty(N, dtype=torch.float32, device=dev)
        self.g = torch.ones(1, dtype=torch.float32, device=dev)
        self.dX = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty(D, V, dtype=torch.float32, device=dev)
        self.opts = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
        self.ws = None

    def io_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.X, self.W, self.y, self.loss, self.lse, self.dX,
                                                           self.dW))

    def alloc_workspace(self, with_bwd=True):
        self.ws = torch.empty(max(self.ws_f, self.ws_b) if with_bwd else self.ws_f, dtype=torch.uint8,
                              device=self.dev)

    def fwd(self):
        self.flce.flce_forward(self.X, self.W, self.y, self.loss, self.lse, self.ws, *self.opts, stream=self.stream)

    def bwd(self):
        if self.opt_b is None:
            self.flce.flce_backward(self.X, self.W, self.y, self.lse, self.g, self.dX, self.dW, self.ws, *self.opts,
                                    stream=self.stream)
        else:
            self.flce.flce_backward_ex(self.X, self.W, self.y, self.lse, self.g, self.dX, self.dW, self.ws,
                                       *self.opts, options=self.opt_b, stream=self.stream)

    def check(self, where):
        st = self.flce.flce_check_device_error(self.ws, self.stream)
        if st != 0:
            raise RuntimeError(f"device error {where}: {self.flce.flce_status_string(st)}")

    def timed_steps(self, steps, gpu_index, kernel_timing=False):
        """`steps` forward + backward steps on the stream, each bracketed by CUDA events;
        returns (total ms, per-step forward ms, per-step backward ms, launches, clocks,
        per-GEMM-kind timing). With kernel_timing the library also brackets every GEMM
        launch of these steps with CUDA events on the stream (flce_profile_gemms), so each
        GEMM kind's device time is measured over this same region."""
        flce = self.flce
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize(self.dev)
        if kernel_timing:
            flce.flce_profile_read()  # nothing pending
        launches_before = flce.flce_kernel_launches()
        with ClockSampler(gpu_index) as clk:
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            if kernel_timing:
                flce.flce_profile_gemms(True)
            try:
                start.record(self.stream)
                for i in range(steps):
                    ev[i][0].record(self.stream)
                    self.fwd()
                    ev[i][1].record(self.stream)
                    self.bwd()
                    ev[i][2].record(self.stream)
                end.record(self.stream)
            finally:
                if kernel_timing:
                    flce.flce_profile_gemms(False)
            launches = flce.flce_kernel_launches() - launches_before
            torch.cuda.synchronize(self.dev)
        self.check("in the timed region")
        kinds = None
        if kernel_timing:
            kinds = {}
            for kind, (ms, n) in flce.flce_profile_read().items():
                if n:
                    kinds[kind] = {"ms_per_step": ms / steps, "launches_per_step": n / steps, "avg_launch_ms": ms / n}
            kinds = {"kinds": kinds, "steps": steps}
        return (start.elapsed_time(end), [a.elapsed_time(b) for a, b, _ in ev],
                [b.elapsed_time(c) for _, b, c in ev], launches, clk, kinds)


def run_ours(args, wl):
    import linear_cross_entropy_tcgen05_gb300 as flce
    flce.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    N, D, V = wl.N, wl.D, wl.V
    X, W, y = make_inputs(wl)
    stream = torch.cuda.current_stream(dev)
    pb = Problem(flce, wl, dev, stream, X.to(dev), W.to(dev), y.to(dev), row_band=args.row_band)
    with_bwd = args.only != "fwd"
    torch.cuda.synchronize(dev)
    base_alloc = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    pb.alloc_workspace(with_bwd)

    if args.only is not None:
        # profiling driver: warm-up + steps of one phase, nothing else on the device
        if args.only == "bwd":
            pb.fwd()
        step = pb.fwd if args.only == "fwd" else pb.bwd
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        # each call timed with CUDA events on the stream, clocks sampled meanwhile
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        with ClockSampler(0) as clk:
            for a, b in ev:
                a.record(stream)
                step()
                b.record(stream)
            torch.cuda.synchronize(dev)
        ms = [a.elapsed_time(b) for a, b in ev]
        c = clk.summary()
        line = {"only": args.only, "workload": wl.name, "steps": args.steps, "ms_mean": statistics.mean(ms),
                "ms_median": statistics.median(ms), "clocks": c}
        if c["sm_mhz"]:
            # time x clock: the work in SM cycles, comparable across boxes and power states
            line["mcycles_median"] = statistics.median(ms) * c["sm_mhz"] / 1000.0
        if args.wait_stats:
            line["pipeline_waits"] = pipeline_waits(pb.ws, args.only)
        st = flce.flce_check_device_error(pb.ws, stream)
        line["status"] = flce.flce_status_string(st)
        print(json.dumps(line))
        if st != 0:
            raise SystemExit(1)
        return

    for _ in range(args.warmup):
        pb.fwd()
        pb.bwd()
    torch.cuda.synchronize(dev)
    pb.check("after warm-up")
    peak_alloc = torch.cuda.max_memory_allocated(dev)
    extra_bytes = peak_alloc - base_alloc

    timing = not args.no_kernel_timing
    total_ms, fwd_ms, bwd_ms, launches_timed, clk, kernels = pb.timed_steps(args.steps, 0, timing)
    # a run that saw thermal or hardware slowdown, or clocks held far below maximum with no
    # reason given (a leftover clock lock), is measured once more
    if clk.throttled():
        total_ms, fwd_ms, bwd_ms, launches_timed, clk, kernels = pb.timed_steps(args.steps, 0, timing)
        clk.remeasured = True
    ms_step = total_ms / args.steps
    value = N / (ms_step / 1000.0)
    band_width = flce.flce_backward_band_width(N, D, V, pb.opt_b) or None

    # end to end through the public API: pinned host inputs -> device, fwd+bwd, loss/dX/dW -> host
    e2e_value, e2e_ms, h2d, d2h = run_e2e(args, dev, stream, X, W, y, pb)
    del pb
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    side = run_side_workloads(args, flce, dev, stream) if args.side_workloads else None
    return finish(args, wl, N, D, V, X, W, y, ms_step, value, fwd_ms, bwd_ms, peak_alloc, extra_bytes,
                  e2e_value, e2e_ms, h2d, d2h, clk, launches_timed, band_width, side, kernels,
                  flce.flce_workspace_size(N, D, V, False),
                  flce.flce_workspace_size(args.row_band if 0 < args.row_band < N else N, D, V, True),
                  flce.flce_workspace_size(N, D, V, "forward_valid_rows"))


KERNEL_NAMES = {"forward": "flce_forward_gemm_kernel (forward GEMM + online softmax)",
                "gradient": "flce_walk_gemm_kernel (gradient GEMM: recomputed logits -> G band)",
                "dW": "flce_walk_gemm_kernel (dW GEMM: X^T G, K = valid rows)",
                "dX": "flce_walk_gemm_kernel (dX GEMM: G W^T, fp32 accumulate)"}


def recorded_traffic(kind):
    """A one-pass ncu capture of this GEMM kind's DRAM bytes per launch at the headline
    shape, recorded under profiles/ with the hash of the kernel source it was taken on;
    None unless that hash matches the source."""
    p = os.path.join(ROOT, "profiles", "gemm_traffic_headline.json")
    if not os.path.exists(p):
        return None, None
    rec = json.load(open(p))
    if rec.get("kernel_source_hash") != _kernel_hash() or kind not in rec.get("kinds", {}):
        return None, None
    k = rec["kinds"][kind]
    return k["bytes_per_launch"], {"kind": "recorded ncu capture of this kernel source, not measured in this run",
                                   "captured": rec.get("captured"), "case": k.get("launch"),
                                   "record": "profiles/gemm_traffic_headline.json"}


def run_e2e(args, dev, stream, X, W, y, pb):
    """End to end through the public API: every step copies X, W and targets from pinned
    host memory to the device and loss, dX and dW back. Copies run on their own streams
    with three buffer sets, so step i's compute overlaps the input copy of step i+1 and the
    result copy of step i-1, and a copy slowed by the shared host link has two steps of
    slack before compute waits for it (what a training loop feeding this op would do)."""
    if args.no_e2e:
        return None, None, 0, 0
    flce = pb.flce
    N, D = X.shape
    V = W.shape[1]
    Xh, Wh, yh = X.pin_memory(), W.pin_memory(), y.pin_memory()
    loss_h = torch.empty(1, dtype=torch.float32).pin_memory()
    dX_h = torch.empty(N, D, dtype=torch.bfloat16).pin_memory()
    dW_h = torch.empty(D, V, dtype=torch.float32).pin_memory()
    h2d = Xh.numel() * 2 + Wh.numel() * 2 + yh.numel() * 4
    d2h = 4 + dX_h.numel() * 2 + dW_h.numel() * 4
    # buffer sets: set 0 reuses the resident buffers, the others are copies
    nbuf = 3
    bufs = [(pb.X, pb.W, pb.y, pb.loss, pb.dX, pb.dW)] + [
        (torch.empty_like(pb.X), torch.empty_like(pb.W), torch.empty_like(pb.y), torch.empty_like(pb.loss),
         torch.empty_like(pb.dX), torch.empty_like(pb.dW)) for _ in range(nbuf - 1)]
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    inputs_free = [torch.cuda.Event() for _ in range(nbuf)]
    inputs_ready = [torch.cuda.Event() for _ in range(nbuf)]
    outputs_ready = [torch.cuda.Event() for _ in range(nbuf)]
    outputs_free = [torch.cuda.Event() for _ in range(nbuf)]
    steps = max(1, args.steps)
    warm = nbuf
    for ev in inputs_free + outputs_free:
        ev.record(stream)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    for it in range(warm + steps):
        if it == warm:
            torch.cuda.synchronize(dev)
            t0.record(stream)
        b = it % nbuf
        Xb, Wb, yb, lb, dXb, dWb = bufs[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(inputs_free[b])
            Xb.copy_(Xh, non_blocking=True)
            Wb.copy_(Wh, non_blocking=True)
            yb.copy_(yh, non_blocking=True)
            inputs_ready[b].record(s_in)
        stream.wait_event(inputs_ready[b])
        stream.wait_event(outputs_free[b])
        # compute is serialised on one stream, so every buffer set shares the workspace
        flce.flce_forward(Xb, Wb, yb, lb, lse, pb.ws, *pb.opts, stream=stream)
        if pb.opt_b is not None:
            flce.flce_backward_ex(Xb, Wb, yb, lse, pb.g, dXb, dWb, pb.ws, *pb.opts, options=pb.opt_b,
                                  stream=stream)
        else:
            flce.flce_backward(Xb, Wb, yb, lse, pb.g, dXb, dWb, pb.ws, *pb.opts, stream=stream)
        inputs_free[b].record(stream)
        outputs_ready[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(outputs_ready[b])
            loss_h.copy_(lb, non_blocking=True)
            dX_h.copy_(dXb, non_blocking=True)
            dW_h.copy_(dWb, non_blocking=True)
            outputs_free[b].record(s_out)
    stream.wait_stream(s_out)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    pb.check("in the end-to-end region")
    e2e_ms = t0.elapsed_time(t1) / steps
    e2e_value = N / (e2e_ms / 1000.0)
    del bufs
    return e2e_value, e2e_ms, h2d, d2h


def device_inputs(wl, dev):
    """Inputs of a side workload drawn on the device: X ~ N(0,1) and W ~ N(0,1/D) from
    torch's seeded device generator, rounded to bf16 (the recipe's distributions, drawn in
    a fraction of a second where the host recipe takes seconds per gigabyte), and the
    recipe's own targets and ignored rows."""
    from workloads import make_targets_of
    gen = torch.Generator(device=dev)
    gen.manual_seed(wl.seed)
    X = torch.randn(wl.N, wl.D, generator=gen, device=dev).to(torch.bfloat16)
    W = torch.randn(wl.D, wl.V, generator=gen, device=dev).mul_(1.0 / math.sqrt(wl.D)).to(torch.bfloat16)
    y = make_targets_of(wl).to(dev)
    return X, W, y


GRAPH_BELOW_MS = 5.0  # side workloads whose step is this short are also timed as a replayed CUDA graph


def graph_replay(pb, steps):
    """One forward + backward step captured into a CUDA graph (the calls issue only stream
    work, so they capture as they are) and replayed `steps` times back to back: the step
    without the host's per-call cost, which is most of a small problem's time."""
    graph = torch.cuda.CUDAGraph()
    launch_stream = pb.stream
    try:
        with torch.cuda.graph(graph):
            pb.stream = torch.cuda.current_stream(pb.dev)  # the capture stream
            pb.fwd()
            pb.bwd()
    finally:
        pb.stream = launch_stream
    with torch.cuda.stream(launch_stream):
        for _ in range(3):
            graph.replay()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(launch_stream)
        for _ in range(steps):
            graph.replay()
        end.record(launch_stream)
    torch.cuda.synchronize(pb.dev)
    pb.check("in the graph replays")
    ms = start.elapsed_time(end) / steps
    return {"ms_per_step": ms, "tokens_per_s": pb.wl.N / (ms / 1000.0), "replays": steps}


def run_side_workloads(args, flce, dev, stream):
    """The other workloads and the memory-benchmark shape, each warmed up and then timed
    for about `args.side_seconds` (at least 5 steps): median fwd+bwd step, tokens/s, the
    fraction of the sustained bf16 peak for 8*N*D*V flops, and peak device memory (total
    for inputs, outputs and workspace; extra = beyond the inputs and outputs)."""
    from workloads import MEMORY_BENCHMARK
    peaks, peak_kind = measured_peaks()
    sustained = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    out = {}
    chosen = [w for w in args.side_workloads.split(",") if w and w != args.workload]
    for name in chosen:
        wl = MEMORY_BENCHMARK if name == MEMORY_BENCHMARK.name else WORKLOADS[name]
        torch.cuda.synchronize(dev)
        base = torch.cuda.memory_allocated(dev)
        X, W, y = device_inputs(wl, dev)
        pb = Problem(flce, wl, dev, stream, X, W, y)
        torch.cuda.synchronize(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        io = torch.cuda.memory_allocated(dev)
        pb.alloc_workspace(True)
        for _ in range(3):
            pb.fwd()
            pb.bwd()
        torch.cuda.synchronize(dev)
        pb.check(f"after the warm-up of {name}")
        peak = torch.cuda.max_memory_allocated(dev)
        # a short probe sets the step count for about side_seconds of timed work
        t_probe = pb.timed_steps(2, 0)[0]
        steps = int(min(400, max(5, math.ceil(args.side_seconds * 1000.0 / max(t_probe / 2, 1e-3)))))
        total, f_ms, b_ms, launches, clk, _ = pb.timed_steps(steps, 0)
        step_ms = [f + b for f, b in zip(f_ms, b_ms)]
        med = statistics.median(step_ms)
        N, D, V = wl.N, wl.D, wl.V
        tf = 8.0 * N * D * V / (med / 1000.0) / 1e12
        out[name] = {
            "N": N, "D": D, "V": V, "options": wl.describe(), "steps": steps,
            "ms_per_step_median": med, "fwd_ms_median": statistics.median(f_ms),
            "bwd_ms_median": statistics.median(b_ms), "ms_per_step_mean": total / steps,
            "tokens_per_s": N / (med / 1000.0), "tflops": tf,
            "frac_of_sustained_bf16": tf / sustained,
            "peak_kind": f"{peak_kind} sustained cuBLAS bf16 ({sustained} TF/s)",
            "peak_mb": {"total": (peak - base) / 2**20, "extra": (peak - io) / 2**20,
                        "workspace": pb.ws.numel() / 2**20, "logits_bf16_would_be": N * V * 2 / 2**20},
            "launches_per_step": launches / steps,
            "clocks": clk.summary(),
        }
        if med < GRAPH_BELOW_MS:
            out[name]["graph"] = graph_replay(pb, steps)
        if name == "llama8k":
            out[name]["context"] = ("Liger-Kernel PR #1291, Benchmarks: CuTe-DSL FLCE fwd+bwd 25.7 ms at BT=8192, "
                                    "V=128256, H=4096, bf16, on B200 (another system and GPU)")
        if name == MEMORY_BENCHMARK.name:
            out[name]["context"] = ("Cutting LLM Memory by 84%, Memory Benchmark: peak 36.02 GB eager PyTorch, "
                                    "5.04 GB Triton FLCE, at S=16384, D=4096, V=128256 on A100 (another system)")
        del pb, X, W, y
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    return {"inputs": "X, W drawn on the device (torch's seeded generator, the recipe's distributions); "
                      "targets and ignored rows from the recipe", "results": out}


def finish(args, wl, N, D, V, X, W, y, ms_step, value, fwd_ms, bwd_ms, peak_alloc, extra_bytes, e2e_value, e2e_ms,
           h2d, d2h, clk, launches_timed, band_width, side, kernels, ws_f, ws_b, ws_fc):
    peaks, peak_kind = measured_peaks()
    flops_step = 8.0 * N * D * V
    fwd_avg = statistics.mean(fwd_ms)
    fwd_gemm_tf = 2.0 * N * D * V / (fwd_avg / 1000.0) / 1e12
    step_tf = flops_step / (ms_step / 1000.0) / 1e12
    bwd_tf = 6.0 * N * D * V / (statistics.mean(bwd_ms) / 1000.0) / 1e12
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    launches, bands, vc = kernel_launches_per_step(N, D, V, wl.reduction, band_width,
                                                   row_band=args.row_band if 0 < args.row_band < N else 0,
                                                   compact_fwd=max(ws_f, ws_b) >= ws_fc and N >= 2048)
    cpu = None
    if not args.no_cpu_baseline:
        rate, rows, dt = oracle_sample_for(wl, X, W, y, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"fp64 oracle fwd+bwd of the first {rows} rows x full V in chunks of 256 "
                         f"({dt:.1f} s); tokens/s = rows/time"}
    # every GEMM kind does 2*N*D*V algorithmic flops per step (all rows, as counted for the
    # step), spread over its launches; the roofline object is the kind with the most time
    valid_rows = int((y != wl.ignore_index).sum())
    per_kind = {}
    dominant = None
    if kernels:
        for kind, k in kernels["kinds"].items():
            tf = 2.0 * N * D * V / (k["ms_per_step"] / 1000.0) / 1e12
            traffic, source = recorded_traffic(kind)
            per_kind[kind] = {"kernel": KERNEL_NAMES.get(kind, kind), "ms_per_step": k["ms_per_step"],
                              "launches_per_step": k["launches_per_step"], "avg_launch_ms": k["avg_launch_ms"],
                              "achieved": tf, "frac": tf / sustained,
                              "achieved_valid_rows": tf * valid_rows / N,
                              "traffic": traffic, "traffic_source": source}
        dominant = max(per_kind, key=lambda kd: per_kind[kd]["ms_per_step"])
    if dominant is not None:
        dk = per_kind[dominant]
        roofline = {"kernel": dk["kernel"], "bound": "tensor", "achieved": dk["achieved"], "peak": sustained,
                    "unit": "TFLOP/s", "frac": dk["frac"], "traffic": dk["traffic"],
                    "traffic_source": dk["traffic_source"],
                    "peak_kind": f"{peak_kind} sustained cuBLAS bf16 (kernels timed inside a seconds-long loop)",
                    "frac_of_burst": dk["achieved"] / burst,
                    "algorithmic": "2*N*D*V flops per step over the kind's launches (all rows counted)",
                    "avg_launch_ms": dk["avg_launch_ms"], "launches_per_step": dk["launches_per_step"],
                    "share_of_gemm_time": dk["ms_per_step"] / sum(v["ms_per_step"] for v in per_kind.values()),
                    "frac_valid_rows": dk["achieved_valid_rows"] / sustained,
                    "measured": (f"CUDA events around every launch of the kind on its stream "
                                 f"(flce_profile_gemms), over the {kernels['steps']} steps of the timed region")}
    else:
        roofline = {"kernel": "flce_forward_gemm_kernel", "bound": "tensor", "achieved": fwd_gemm_tf,
                    "peak": sustained, "unit": "TFLOP/s", "frac": fwd_gemm_tf / sustained, "traffic": None,
                    "traffic_source": None}
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": data_recipe(wl),
        "config": {"workload": wl.name, "N": N, "D": D, "V": V, "reduction": wl.reduction,
                   "ignore_frac": wl.ignore_frac, "label_smoothing": wl.label_smoothing,
                   "zloss_scale": wl.zloss_scale, "grad_out": 1.0,
                   "l2": l2_note(wl),
                   "parallelism": "one GPU", "vocab_band": vc, "bands": bands,
                   **({"row_band": args.row_band} if 0 < args.row_band < N else {})},
        # another system on another GPU: context, not a baseline
        "context": {"liger_cutedsl_flce_b200": {
            "tokens_per_s": PAGES_TOKENS_PER_S,
            # a ratio only where the figure's shape is the one measured here
            "ratio": value / PAGES_TOKENS_PER_S if (N, D, V) == (65536, 4096, 128256) else None,
            "source": "Liger-Kernel PR #1291, Benchmarks: 194 ms fwd+bwd at BT=65536, V=128256, H=4096, bf16, B200"}},
        "pct_bf16_peak": 100.0 * step_tf / burst,
        "tflops": step_tf,
        "fwd_ms": fwd_avg, "bwd_ms": statistics.mean(bwd_ms),
        "peak_mb": {"total": peak_alloc / 2**20, "extra": extra_bytes / 2**20,
                    "workspace": max(ws_f, ws_b) / 2**20,
                    "logits_bf16_would_be": N * V * 2 / 2**20},
        # the kernels run inside a seconds-long fwd+bwd loop at the board's power limit, so
        # their peak is the sustained cuBLAS figure; the burst fraction is given beside it
        "roofline": roofline,
        "roofline_kernels": per_kind,
        "roofline_forward_call": {"achieved": fwd_gemm_tf, "frac": fwd_gemm_tf / sustained, "unit": "TFLOP/s",
                                  "algorithmic": "2*N*D*V flops over the forward call (GEMM + finalize), "
                                                 "timed in the timed region"},
        "roofline_step": {"bound": "tensor", "achieved": step_tf, "peak": sustained, "unit": "TFLOP/s",
                          "frac": step_tf / sustained, "peak_kind": f"{peak_kind} sustained cuBLAS bf16",
                          "algorithmic": "8*N*D*V flops per step"},
        "roofline_backward": {"achieved": bwd_tf, "unit": "TFLOP/s", "frac": bwd_tf / sustained},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        # counted by the library (flce_kernel_launches) over the timed region; the band
        # schedule predicts launches_per_step x steps
        "gpu_launches": launches_timed,
        "gpu_launches_per_step_expected": launches,
        "clocks": clk.summary(),
    }
    # the step in SM cycles (time x median clock): comparable across boxes whose
    # power-capped clocks differ
    if out["clocks"].get("sm_mhz"):
        out["mcycles_per_step"] = ms_step * out["clocks"]["sm_mhz"] / 1000.0
    if side is not None:
        out["workloads"] = side
    print(json.dumps(out), flush=True)


def _kernel_hash() -> str:
    """Hash of the GEMM kernels' source code with comments and blank space removed, so
    that a recorded ncu traffic figure stays attached to the code it was measured on."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("flce_gemm.cu", "sm103_ptx.cuh", "flce_internal.h"):
        p = os.path.join(ROOT, "linear_cross_entropy_tcgen05_gb300", "csrc", f)
        if os.path.exists(p):
            src = open(p).read()
            src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
            src = re.sub(r"//[^\n]*", " ", src)
            h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


SIDE_DEFAULT = "tiny,small_vocab,llama8k,large_vocab,memory_benchmark"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="headline", choices=sorted(WORKLOADS))
    ap.add_argument("--oracle-rows", type=int, default=512, help="rows per step of the reference arm")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU time of the cpu_baseline sample")
    ap.add_argument("--shape", default=None, help="N,D,V override of the workload's shape (profiling cases)")
    ap.add_argument("--row-band", type=int, default=0,
                    help="memory-lean backward: rows per band (0: the whole batch at once)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--side-workloads", default=SIDE_DEFAULT,
                    help="comma-separated workloads timed after the main one ('' for none)")
    ap.add_argument("--side-seconds", type=float, default=0.5, help="timed seconds per side workload")
    ap.add_argument("--no-kernel-timing", action="store_true",
                    help="time the region without the per-GEMM-kind events (the roofline then falls back to "
                         "the forward call)")
    ap.add_argument("--wait-stats", action="store_true",
                    help="with --only and a library built with -DFLCE_WAIT_STATS=1: print pipeline wait shares")
    ap.add_argument("--only", choices=["fwd", "bwd"], default=None,
                    help="profiling driver: run only this phase (warm-up + steps), print a status line")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]
    if args.shape:
        import dataclasses
        n, d, v = (int(x) for x in args.shape.split(","))
        wl = dataclasses.replace(wl, name=f"{wl.name}@{n}x{d}x{v}", N=n, D=d, V=v)
    world, rank = launch_env()
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, wl)
        return 0
    if world > 1 or args.gpus > 1:
        return refuse_multi_gpu(args, world, rank)
    run_ours(args, wl)
    return 0


if __name__ == "__main__":
    sys.exit(main())
