"""The forward on the valid rows only. With a workspace of flce_workspace_size(..., 3)
bytes (every backward workspace has that room) the forward gathers the valid rows of X
and runs its GEMM on them alone; with the forward's own, smaller workspace it runs on every
row (the valid-row path needs 2048 rows or more, so every case here has them). The
results must be the same bit for bit (each valid row's logits are the same dot
products in the same order), the lse of an ignored row is exactly 0 either way, and both
agree with the fp64 oracle on the valid rows."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
import oracle
from tests.flce_cases import TOL_LOSS_REL, TOL_LSE_ABS
from workloads import custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _forward(X, W, y, wl, kind, reduction=None):
    red = wl.reduction if reduction is None else reduction
    N, D, V = wl.N, wl.D, wl.V
    ws = torch.empty(flce.flce_workspace_size(N, D, V, kind), dtype=torch.uint8, device=DEV)
    loss = torch.full((N if red == "none" else 1,), float("nan"), device=DEV)
    lse = torch.full((N,), float("nan"), device=DEV)
    flce.flce_forward(X, W, y, loss, lse, ws, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, red)
    assert flce.flce_check_device_error(ws) == 0
    return loss, lse


CASES = [
    custom("fc1", 2100, 136, 4104, seed=301, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-4),
    custom("fc2", 2048, 256, 8200, seed=302, ignore_frac=0.9, reduction="sum"),
    custom("fc3", 2777, 64, 1000, seed=303, ignore_frac=0.5),
    custom("fc4", 2561, 128, 2048, seed=304, ignore_frac=0.3, reduction="none"),
]


@pytest.mark.parametrize("wl", CASES, ids=[c.name for c in CASES])
def test_valid_rows_forward_is_bitwise_the_full_forward(gpu_lib, wl):
    assert wl.N >= 2048
    X, W, y = make_inputs(wl)
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    full = _forward(Xd, Wd, yd, wl, "forward")
    valid_only = _forward(Xd, Wd, yd, wl, "forward_valid_rows")
    torch.cuda.synchronize()
    for a, b in zip(full, valid_only):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    ign = (y == wl.ignore_index).numpy()
    lse = valid_only[1].cpu().double().numpy()
    assert np.all(lse[ign] == 0.0)
    ref_loss, ref_lse = oracle.forward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    assert np.max(np.abs(lse[~ign] - ref_lse[~ign])) <= TOL_LSE_ABS
    got = valid_only[0].cpu().double().numpy()
    ref = np.atleast_1d(np.asarray(ref_loss, dtype=np.float64))
    scale = np.maximum(np.abs(ref), 1.0) if wl.reduction == "none" else np.abs(ref)
    assert np.all(np.abs(got - ref) <= TOL_LOSS_REL * scale)


def test_valid_rows_forward_with_every_row_ignored(gpu_lib):
    wl = custom("fc_all", 2100, 64, 1024, seed=305, ignore_frac=1.0)
    X, W, y = make_inputs(wl)
    for kind in ("forward", "forward_valid_rows"):
        loss, lse = _forward(X.to(DEV), W.to(DEV), y.to(DEV), wl, kind)
        torch.cuda.synchronize()
        assert loss.item() == 0.0 and torch.all(lse == 0.0)


def test_valid_rows_forward_then_backward_matches_the_oracle(gpu_lib):
    """The backward takes the lse the valid-row forward wrote (0 on ignored rows, which
    the backward never reads) and gives the oracle's gradients."""
    from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, CudaRun, rel_fro
    wl = custom("fc_bwd", 2500, 200, 3000, seed=306, ignore_frac=0.6, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y = make_inputs(wl)
    run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    assert run.ws.numel() >= flce.flce_workspace_size(wl.N, wl.D, wl.V, "forward_valid_rows")
    assert run.forward() == 0 and run.backward() == 0
    got = run.host()
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                                                wl.reduction)
    valid = y.numpy() != wl.ignore_index
    assert abs(got["loss"][0] - loss) <= TOL_LOSS_REL * abs(loss)
    assert np.max(np.abs(got["lse"][valid] - lse[valid])) <= TOL_LSE_ABS
    assert np.all(got["lse"][~valid] == 0.0)
    assert rel_fro(got["dX"], dX) <= TOL_DX_REL and rel_fro(got["dW"], dW) <= TOL_DW_REL


def _random_case(i):
    g = np.random.default_rng(7000 + i)
    return dict(N=int(g.integers(2048, 5000)), D=8 * int(g.integers(1, 40)), V=8 * int(g.integers(1, 600)),
                seed=7100 + i, ignore_frac=float(g.choice([0.0, 0.1, 0.5, 0.9])),
                eps=float(g.choice([0.0, 0.1])), s=float(g.choice([0.0, 1e-3])),
                red=str(g.choice(["mean", "sum", "none"])), layout=str(g.choice(["dv", "vd"])),
                dtype=str(g.choice(["bf16", "f16"])))


RANDOM = [_random_case(i) for i in range(8)]


@pytest.mark.parametrize("c", RANDOM, ids=[f"{c['N']}x{c['D']}x{c['V']}-{c['layout']}-{c['dtype']}-{c['red']}"
                                           for c in RANDOM])
def test_valid_rows_forward_random_shapes(gpu_lib, c):
    """Seeded random shapes and options on the valid-row path (both weight layouts, bf16
    and f16): bit for bit the all-rows forward, and the oracle on the valid rows."""
    dt = torch.float16 if c["dtype"] == "f16" else torch.bfloat16
    wl = custom("fcr", c["N"], c["D"], c["V"], seed=c["seed"], ignore_frac=c["ignore_frac"],
                label_smoothing=c["eps"], zloss_scale=c["s"], reduction=c["red"])
    X, W, y = make_inputs(wl, dtype=dt)
    N, D, V = wl.N, wl.D, wl.V
    Wdev = (W.t().contiguous() if c["layout"] == "vd" else W).to(DEV)
    Xd, yd = X.to(DEV), y.to(DEV)
    opt = flce.make_options(weight_layout=c["layout"], input_dtype=dt)
    outs = []
    for kind in ("forward", "forward_valid_rows"):
        ws = torch.empty(flce.flce_workspace_size(N, D, V, kind), dtype=torch.uint8, device=DEV)
        loss = torch.full((N if c["red"] == "none" else 1,), float("nan"), device=DEV)
        lse = torch.full((N,), float("nan"), device=DEV)
        flce.flce_forward_ex(Xd, Wdev, yd, loss, lse, ws, wl.ignore_index, c["eps"], c["s"], c["red"], options=opt)
        assert flce.flce_check_device_error(ws) == 0
        outs.append((loss, lse))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    ref_loss, ref_lse = oracle.forward(X, W, y, wl.ignore_index, c["eps"], c["s"], c["red"])
    ign = (y == wl.ignore_index).numpy()
    lse = outs[1][1].cpu().double().numpy()
    assert np.all(lse[ign] == 0.0)
    if (~ign).any():
        assert np.max(np.abs(lse[~ign] - ref_lse[~ign])) <= TOL_LSE_ABS
    got = outs[1][0].cpu().double().numpy()
    ref = np.atleast_1d(np.asarray(ref_loss, dtype=np.float64))
    scale = np.maximum(np.abs(ref), 1.0) if c["red"] == "none" else np.maximum(np.abs(ref), 1e-30)
    assert np.all(np.abs(got - ref) <= TOL_LOSS_REL * scale)
