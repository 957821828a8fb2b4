"""Data-parallel use over rows on two gloo ranks (CPU): each rank takes half of the rows,
computes its sum-reduced gradients, and the ranks all-reduce n_valid and dW. Scaled by
1 / (global n_valid) -- which is what passing reduction='sum' and grad_out = 1 / n_valid to
the library does -- the result equals the mean-reduced gradient of the whole batch. The
per-rank arithmetic here is the fp64 oracle's; the library's sum reduction and grad_out
scaling are covered by the GPU parity tests."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import oracle
    from workloads import IGNORE_INDEX, custom, make_inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = custom("dp", 96, 16, 64, seed=91, ignore_frac=0.2, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y = make_inputs(wl)
    rows = slice(rank * wl.N // world, (rank + 1) * wl.N // world)
    Xr, yr = X[rows], y[rows]
    n_valid = torch.tensor([float((yr != IGNORE_INDEX).sum())], dtype=torch.float64)
    dist.all_reduce(n_valid)
    loss_r, _, _, dW_r = oracle.forward_backward(Xr, W, yr, IGNORE_INDEX, 0.1, 1e-3, "sum",
                                                 grad_out=1.0 / float(n_valid))
    dW = torch.from_numpy(np.ascontiguousarray(dW_r))
    loss = torch.tensor([loss_r / float(n_valid)], dtype=torch.float64)
    dist.all_reduce(dW)
    dist.all_reduce(loss)
    if rank == 0:
        ref_loss, _, _, ref_dW = oracle.forward_backward(X, W, y, IGNORE_INDEX, 0.1, 1e-3, "mean")
        out["loss_err"] = abs(float(loss) - ref_loss)
        out["dW_err"] = float(np.max(np.abs(dW.numpy() - ref_dW)))
    dist.destroy_process_group()


def test_row_parallel_mean_equals_the_whole_batch():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out["loss_err"] < 1e-12 and out["dW_err"] < 1e-12
