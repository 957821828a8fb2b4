"""Seeded random sweep over shapes and options, each case compared with the fp64 oracle:
ragged N, D and V, every reduction, smoothing and z-loss, ignored rows, the [V, D] layout,
f16 inputs, softcap, bias and class weights, row bands. Shapes and options come from one
seeded generator, so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, TOL_LOSS_REL, TOL_LSE_ABS, rel_fro
from workloads import IGNORE_INDEX, custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _case(i):
    g = np.random.default_rng(1000 + i)
    N = int(g.integers(1, 1500))
    D = 8 * int(g.integers(1, 80))
    V = 8 * int(g.integers(1, 1200))
    return dict(
        N=N, D=D, V=V, seed=2000 + i,
        ignore_frac=float(g.choice([0.0, 0.1, 0.5])),
        eps=float(g.choice([0.0, 0.0, 0.1, 0.3])),
        s=float(g.choice([0.0, 1e-4, 1e-2])),
        red=str(g.choice(["mean", "sum"])),
        layout=str(g.choice(["dv", "vd"])),
        dtype=str(g.choice(["bf16", "bf16", "f16"])),
        softcap=float(g.choice([0.0, 0.0, 20.0])),
        bias=bool(g.random() < 0.3),
        cw=bool(g.random() < 0.3),
        row_band=int(g.choice([0, 0, max(1, N // 3)])),
        grad_out=float(g.choice([1.0, 0.5, -2.0])),
    )


CASES = [_case(i) for i in range(24)] + [
    # f16 with heavy smoothing and a small grad_out: dX entries near 1e-6, below f16's
    # normal range, so the f16 output itself carries percent-level rounding error
    dict(N=972, D=1720, V=4432, seed=60021, ignore_frac=0.05, eps=0.9, s=0.0, red="mean", layout="vd",
         dtype="f16", softcap=5.0, bias=False, cw=True, row_band=0, grad_out=-0.25),
    dict(N=2994, D=408, V=5944, seed=60068, ignore_frac=0.0, eps=0.9, s=0.1, red="mean", layout="dv",
         dtype="f16", softcap=0.0, bias=False, cw=False, row_band=0, grad_out=-0.25),
]


@pytest.mark.parametrize("c", CASES, ids=[f"{c['N']}x{c['D']}x{c['V']}-{c['layout']}-{c['dtype']}" for c in CASES])
def test_random_case_matches_the_oracle(gpu_lib, c):
    dt = torch.float16 if c["dtype"] == "f16" else torch.bfloat16
    wl = custom("rand", c["N"], c["D"], c["V"], seed=c["seed"], ignore_frac=c["ignore_frac"],
                label_smoothing=c["eps"], zloss_scale=c["s"], reduction=c["red"])
    X, W, y = make_inputs(wl, dtype=dt)
    g = np.random.default_rng(c["seed"])
    bias = torch.tensor(g.standard_normal(wl.V) * 0.5, dtype=torch.float32) if c["bias"] else None
    cw = torch.tensor(g.uniform(0.25, 2.0, size=wl.V), dtype=torch.float32) if c["cw"] else None
    N, D, V = wl.N, wl.D, wl.V
    Wdev = (W.t().contiguous() if c["layout"] == "vd" else W).to(DEV)
    Xd, yd = X.to(DEV), y.to(DEV)
    bd = bias.to(DEV) if bias is not None else None
    wd = cw.to(DEV) if cw is not None else None
    common = (wl.ignore_index, c["eps"], c["s"], c["red"])
    fopt = flce.make_options(softcap=c["softcap"], bias=bd, class_weight=wd, weight_layout=c["layout"],
                             input_dtype=dt)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    ws_f = torch.empty(flce.flce_workspace_size(N, D, V, 0), dtype=torch.uint8, device=DEV)
    flce.flce_forward_ex(Xd, Wdev, yd, loss, lse, ws_f, *common, options=fopt)
    assert flce.flce_check_device_error(ws_f) == 0
    rows = c["row_band"] if c["row_band"] else N
    ws_b = torch.empty(flce.flce_workspace_size(rows, D, V, 1), dtype=torch.uint8, device=DEV)
    dX = torch.full((N, D), float("nan"), dtype=dt, device=DEV)
    dW = torch.full(tuple(Wdev.shape), float("nan"), device=DEV)
    db = torch.full((V,), float("nan"), device=DEV) if bias is not None else None
    bopt = flce.make_options(softcap=c["softcap"], bias=bd, class_weight=wd, dbias=db, row_band=c["row_band"],
                             weight_layout=c["layout"], input_dtype=dt)
    flce.flce_backward_ex(Xd, Wdev, yd, lse, torch.tensor([c["grad_out"]], device=DEV), dX, dW, ws_b, *common,
                          options=bopt)
    assert flce.flce_check_device_error(ws_b) == 0
    torch.cuda.synchronize()
    ref_loss, ref_lse, ref_dX, ref_dW, ref_db = oracle.forward_backward_ext(
        X, W, y, *common, grad_out=c["grad_out"], softcap=c["softcap"], bias=bias, class_weight=cw)
    valid = y.numpy() != IGNORE_INDEX
    if abs(ref_loss) > 0:
        assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss) + 1e-6
    else:
        assert loss.item() == 0.0
    if valid.any():
        assert np.max(np.abs(lse.cpu().double().numpy()[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    dWn = dW.cpu().numpy()
    # dX is rounded once to X's type; its own rounding of the exact dX (large where entries
    # fall below f16's normal range, 6.1e-5) is added to the tolerance
    fmt_err = rel_fro(torch.from_numpy(ref_dX).to(dt).double().numpy(), ref_dX)
    assert rel_fro(dX.float().cpu().numpy(), ref_dX) <= TOL_DX_REL + fmt_err
    assert rel_fro(dWn.T if c["layout"] == "vd" else dWn, ref_dW) <= TOL_DW_REL
    if bias is not None:
        assert rel_fro(db.cpu().numpy(), ref_db) <= TOL_DW_REL
    assert np.all(dX.float().cpu().numpy()[~valid] == 0.0)


def _shard_case(i):
    g = np.random.default_rng(90000 + i)
    N = int(g.integers(1, 1200))
    D = 8 * int(g.integers(1, 100))
    V = 8 * int(g.integers(2, 1500))
    K = int(g.integers(1, 4))
    cuts = sorted(set([0, V] + [8 * int(x) for x in g.integers(1, V // 8, size=K - 1)]))
    return dict(N=N, D=D, V=V, cuts=cuts, seed=91000 + i, ignore_frac=float(g.choice([0.0, 0.2])),
                eps=float(g.choice([0.0, 0.1])), s=float(g.choice([0.0, 1e-3])), red=str(g.choice(["mean", "sum"])),
                layout=str(g.choice(["dv", "vd"])), dtype="f16" if g.random() < 0.3 else "bf16")


SHARD_CASES = [_shard_case(i) for i in range(8)]


@pytest.mark.parametrize("c", SHARD_CASES, ids=[f"{c['N']}x{c['D']}x{c['V']}-{len(c['cuts']) - 1}shards"
                                                for c in SHARD_CASES])
def test_random_vocabulary_shards(gpu_lib, c):
    """Random splits of the vocabulary: shard statistics, their combination and the shard
    backward reproduce the whole-vocabulary oracle."""
    dt = torch.float16 if c["dtype"] == "f16" else torch.bfloat16
    wl = custom("sh", c["N"], c["D"], c["V"], seed=c["seed"], ignore_frac=c["ignore_frac"])
    X, W, y = make_inputs(wl, dtype=dt)
    N, D, V = wl.N, wl.D, wl.V
    Xd, yd = X.to(DEV), y.to(DEV)

    def ws(n, d, v, which):
        return torch.empty(flce.flce_workspace_size(n, d, v, which), dtype=torch.uint8, device=DEV)

    opt = flce.make_options(weight_layout=c["layout"], input_dtype=dt)
    cuts = c["cuts"]
    stats = torch.empty(len(cuts) - 1, 4, N, device=DEV)
    shards = []
    for k, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        Wk = (W[:, a:b].t() if c["layout"] == "vd" else W[:, a:b]).contiguous().to(DEV)
        shards.append((a, b, Wk))
        w_ = ws(N, D, b - a, 0)
        flce.flce_shard_stats(Xd, Wk, yd, a, stats[k], w_, options=opt)
        assert flce.flce_check_device_error(w_) == 0
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    wc = ws(N, 8, 8, 0)
    flce.flce_combine_shards(stats, yd, V, loss, lse, wc, label_smoothing=c["eps"], zloss_scale=c["s"],
                             reduction=c["red"])
    assert flce.flce_check_device_error(wc) == 0
    dX = torch.zeros(N, D, device=DEV)
    dW = torch.empty(D, V, device=DEV)
    for a, b, Wk in shards:
        part = torch.empty(N, D, device=DEV)
        dWk = torch.empty(tuple(Wk.shape), device=DEV)
        w_ = ws(N, D, b - a, 1)
        flce.flce_backward_ex(Xd, Wk, yd, lse, torch.ones(1, device=DEV), None, dWk, w_,
                              label_smoothing=c["eps"], zloss_scale=c["s"], reduction=c["red"],
                              options=flce.make_options(dX_f32=part, v_offset=a, v_total=V,
                                                        weight_layout=c["layout"], input_dtype=dt))
        assert flce.flce_check_device_error(w_) == 0
        dX += part
        dW[:, a:b] = dWk.t() if c["layout"] == "vd" else dWk
    torch.cuda.synchronize()
    ref_loss, ref_lse, ref_dX, ref_dW = oracle.forward_backward(X, W, y, IGNORE_INDEX, c["eps"], c["s"], c["red"])
    valid = y.numpy() != IGNORE_INDEX
    if abs(ref_loss) > 0:
        assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss) + 1e-6
    if valid.any():
        assert np.max(np.abs(lse.cpu().double().numpy()[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(dX.cpu().numpy(), ref_dX) <= 5e-3
    assert rel_fro(dW.cpu().numpy(), ref_dW) <= TOL_DW_REL
