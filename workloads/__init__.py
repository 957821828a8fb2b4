"""Seeded synthetic inputs for fused linear cross-entropy (FLCE).

This module only draws inputs. It holds none of the loss arithmetic, so both the
CUDA path and the fp64 oracle can take their inputs from it without sharing any
of the method's code.

Shapes and distributions follow the workloads of the source pages:

* "Cutting LLM Memory by 84%: A Deep Dive into Fused Kernels", section "The Logit
  Bottleneck": a Llama-3-8B language-model head, hidden size D=4096, vocabulary
  V=128,256, N = batch 8 x 8192 tokens = 65,536 rows; section "Memory Benchmark"
  uses the same D and V.
* Liger-Kernel pull request #1291 ("[CuteDSL] FLCE: 2-SM online-softmax fast
  path"), section "Benchmarks": H=4096, V=128256, BT from 8192 to 65536, plus the
  V=32000 production vocabulary of its "Correctness" section.

No dataset or trained weights are used: hidden states X ~ N(0,1), the vocabulary
projection W ~ N(0, 1/D), both rounded to bf16 (round-to-nearest-even), targets
uniform (or Zipf(1.1)-distributed ranks mapped through a seeded permutation, as a
stand-in for natural token frequencies), and an exact count of rows set to the
ignore index at seeded random positions.

Random draws use numpy's Generator, one child stream per fixed-size block of the
output (``SeedSequence.spawn``), filled by a thread pool. The values therefore
depend only on the seed and the shape, not on the number of threads.
"""
from __future__ import annotations

import concurrent.futures as _cf
import math
import os
from dataclasses import dataclass, field

import numpy as np
import torch

IGNORE_INDEX = -100  # the pages' default ignore index (page 1, "Setup and Target Logit Pre-computation")

_BLOCK = 1 << 22  # elements per independent child stream


@dataclass(frozen=True)
class Workload:
    """One FLCE problem: shapes, loss options and the input recipe."""

    name: str
    N: int
    D: int
    V: int
    seed: int
    ignore_frac: float = 0.0
    target_dist: str = "uniform"  # "uniform" or "zipf"
    zipf_s: float = 1.1
    label_smoothing: float = 0.0
    zloss_scale: float = 0.0
    reduction: str = "mean"
    ignore_index: int = IGNORE_INDEX
    note: str = field(default="", compare=False)

    def describe(self) -> str:
        return (f"N={self.N},D={self.D},V={self.V},eps={self.label_smoothing},"
                f"zloss={self.zloss_scale},{self.reduction},ignore={self.ignore_frac},"
                f"targets={self.target_dist},seed={self.seed}")


# The five workloads, smallest first. Seeds 1-4 are ours; seed 0 is given for the tiny case.
WORKLOADS = {
    "tiny": Workload("tiny", 256, 128, 1024, seed=0,
                     note="tiny FLCE, no ignored rows, mean"),
    "small_vocab": Workload("small_vocab", 4096, 2048, 32000, seed=1, ignore_frac=0.10,
                            note="V=32000 production vocabulary, 10% ignored rows"),
    "llama8k": Workload("llama8k", 8192, 4096, 128256, seed=2, target_dist="zipf",
                        note="Llama-3-8B LM head, one 8192-token sequence, Zipf(1.1) targets"),
    "headline": Workload("headline", 65536, 4096, 128256, seed=3, ignore_frac=0.05,
                         note="batch 8 x 8192 tokens, Llama-3-8B LM head, 5% ignored rows"),
    "large_vocab": Workload("large_vocab", 16384, 2304, 256000, seed=4, ignore_frac=0.05,
                            label_smoothing=0.1, zloss_scale=1e-4, reduction="sum",
                            note="V=256000, label smoothing 0.1, z-loss 1e-4, sum"),
}


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _fill_normal(out: np.ndarray, seed_seq: np.random.SeedSequence, scale: float) -> None:
    """Fill a flat float32 array with N(0, scale^2), one child stream per block."""
    n = out.size
    nblocks = (n + _BLOCK - 1) // _BLOCK
    children = seed_seq.spawn(nblocks)

    def work(b: int) -> None:
        lo = b * _BLOCK
        hi = min(n, lo + _BLOCK)
        g = np.random.Generator(np.random.Philox(children[b]))
        g.standard_normal(out=out[lo:hi], dtype=np.float32)
        if scale != 1.0:
            out[lo:hi] *= np.float32(scale)

    if nblocks == 1:
        work(0)
        return
    with _cf.ThreadPoolExecutor(max_workers=min(_threads(), nblocks)) as ex:
        list(ex.map(work, range(nblocks)))


def normal_bf16(shape, seed_seq: np.random.SeedSequence, scale: float = 1.0,
                dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """A bf16 (or f16) tensor of N(0, scale^2) draws, rounded to nearest even."""
    buf = np.empty(int(np.prod(shape)), dtype=np.float32)
    _fill_normal(buf, seed_seq, scale)
    return torch.from_numpy(buf).view(*shape).to(dtype)


def _zipf_ranks(g: np.random.Generator, n: int, V: int, s: float) -> np.ndarray:
    """Ranks 0..V-1 drawn with P(rank k) proportional to (k+1)^-s (inverse CDF on a table)."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = g.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1)


def make_targets(wl: Workload, seed_seq: np.random.SeedSequence) -> torch.Tensor:
    g = np.random.Generator(np.random.Philox(seed_seq))
    if wl.target_dist == "uniform":
        y = g.integers(0, wl.V, size=wl.N, dtype=np.int64)
    elif wl.target_dist == "zipf":
        ranks = _zipf_ranks(g, wl.N, wl.V, wl.zipf_s)
        perm = g.permutation(wl.V)
        y = perm[ranks]
    else:
        raise ValueError(f"unknown target distribution {wl.target_dist!r}")
    n_ign = int(round(wl.ignore_frac * wl.N))
    if n_ign:
        rows = g.permutation(wl.N)[:n_ign]
        y[rows] = wl.ignore_index
    return torch.from_numpy(y.astype(np.int32))


def make_inputs(wl: Workload, seed: int | None = None, dtype: torch.dtype = torch.bfloat16):
    """Draw (X [N,D], W [D,V], targets int32 [N]) on the CPU; X and W in bf16 (or f16,
    rounded from the same fp32 draws).

    Draw order: X, W, targets (with the ignore mask). ``seed`` overrides the
    workload's own seed.
    """
    root = np.random.SeedSequence(wl.seed if seed is None else seed)
    sx, sw, sy = root.spawn(3)
    X = normal_bf16((wl.N, wl.D), sx, 1.0, dtype)
    W = normal_bf16((wl.D, wl.V), sw, 1.0 / math.sqrt(wl.D), dtype)
    y = make_targets(wl, sy)
    return X, W, y


def make_targets_of(wl: Workload, seed: int | None = None) -> torch.Tensor:
    """The targets (with the ignore mask) that make_inputs draws for this workload and
    seed, without drawing X and W."""
    root = np.random.SeedSequence(wl.seed if seed is None else seed)
    _, _, sy = root.spawn(3)
    return make_targets(wl, sy)


# The shape of the peak-memory comparison in "Cutting LLM Memory by 84%: A Deep Dive into
# Fused Kernels", section "Memory Benchmark": one 16,384-token sequence through the
# Llama-3-8B head (D=4096, V=128,256). The page used real text; uniform targets stand in.
MEMORY_BENCHMARK = Workload("memory_benchmark", 16384, 4096, 128256, seed=5,
                            note="peak-memory shape of the Memory Benchmark section, uniform targets, mean")


def custom(name: str, N: int, D: int, V: int, seed: int = 0, **kw) -> Workload:
    """A workload with the same recipe and other shapes (parity edge cases)."""
    return Workload(name, N, D, V, seed=seed, **kw)


def sample_indices(n_total: int, k: int, seed: int) -> np.ndarray:
    """k distinct sorted indices in [0, n_total), seeded (rows or columns to compare)."""
    g = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, 7919])))
    k = min(k, n_total)
    return np.sort(g.choice(n_total, size=k, replace=False))
