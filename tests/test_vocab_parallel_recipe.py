"""Vocabulary-parallel use on two gloo ranks (CPU): each rank holds a block of W's columns,
computes the per-row statistics of its shard (lse over the shard, logit sum, target logit
if it owns the target), and the ranks exchange them with one all-gather of 4 numbers per
row. Combined, they give the whole problem's lse and loss; each rank's gradient columns,
formed with the combined lse, give its block of dW exactly and, after one all-reduce of
the dX partials, the whole dX. This is the exchange that sits beside the library's
flce_shard_stats / flce_combine_shards / flce_backward_ex(v_offset, v_total), whose
arithmetic the GPU shard tests check against the same oracle functions; the per-rank
arithmetic here is the fp64 oracle's."""
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


# uneven shards: the first rank holds 40 columns, the second 56
CUTS = (0, 40, 96)


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import oracle
    from workloads import IGNORE_INDEX, custom, make_inputs

    dist.init_process_group("gloo", rank=rank, world_size=world)
    eps, s = 0.1, 1e-3
    wl = custom("tp", 80, 16, CUTS[-1], seed=92, ignore_frac=0.2, label_smoothing=eps, zloss_scale=s)
    X, W, y = make_inputs(wl)
    a, b = CUTS[rank], CUTS[rank + 1]
    W_r = W[:, a:b]                          # all this rank holds of W

    # forward: the shard's statistics, gathered from every rank (4 x N per rank)
    mine = torch.from_numpy(np.stack(oracle.shard_stats(X, W_r, y, a, IGNORE_INDEX)))
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine)
    stats = [tuple(t.numpy()) for t in gathered]
    loss, lse = oracle.combine_shard_stats(stats, wl.V, y, IGNORE_INDEX, eps, s, "mean")

    # backward: this rank's gradient columns with the combined lse; dW stays local,
    # the dX partials are summed over ranks
    n_valid = int((y != IGNORE_INDEX).sum())
    g = oracle.grad_scale(1.0, n_valid, "mean")
    z_r = oracle.logits(oracle.widen(X), oracle.widen(W_r))
    dz_r = oracle.grad_logits(z_r, lse, y, wl.V, IGNORE_INDEX, eps, s, g, cols=np.arange(a, b))
    dW_r = oracle.widen(X).T @ dz_r
    dX = torch.from_numpy(np.ascontiguousarray(dz_r @ oracle.widen(W_r).T))
    dist.all_reduce(dX)

    ref_loss, ref_lse, ref_dX, ref_dW = oracle.forward_backward(X, W, y, IGNORE_INDEX, eps, s, "mean")
    valid = y.numpy() != IGNORE_INDEX
    out[rank] = dict(loss=abs(loss - ref_loss), lse=float(np.max(np.abs(lse[valid] - ref_lse[valid]))),
                     dW=float(np.max(np.abs(dW_r - ref_dW[:, a:b]))),
                     dX=float(np.max(np.abs(dX.numpy() - ref_dX))),
                     exchanged=int(mine.numel()))
    dist.destroy_process_group()


def test_vocab_parallel_equals_the_whole_vocabulary():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        res = out[r]
        assert res["loss"] < 1e-12 and res["lse"] < 1e-12, res
        assert res["dW"] < 1e-12 and res["dX"] < 1e-12, res
        assert res["exchanged"] == 4 * 80       # 4 statistics per row, nothing of size V
