"""The backward's valid-row compaction: with a 16-bit dX, the GEMMs run on the valid rows
only (gathered into the dX buffer, per row band when there are row bands) and dX is cast
back to the original rows. Results equal the uncompacted path's (taken with the fp32 dX output, which
keeps rows in place): dX bit for bit, dW to fp32 rounding (its sum over rows runs in
another order); the oracle checks both. Edge cases: no valid row, one valid row, a batch
that is mostly ignored, a dX buffer that aliases X (no scratch: no compaction), and dbias
summed over the compacted band; row bands."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, rel_fro
from workloads import IGNORE_INDEX, custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _ws(N, D, V):
    return torch.empty(flce.flce_workspace_size(N, D, V, 2), dtype=torch.uint8, device=DEV)


def _both_paths(X, W, y, common, row_band=0):
    """(dX bf16, dW) compacted, and (dX fp32, dW) uncompacted, on the same inputs."""
    N, D = X.shape
    V = W.shape[1]
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    ws = _ws(N, D, V)
    flce.flce_forward(Xd, Wd, yd, loss, lse, ws, *common)
    g = torch.ones(1, device=DEV)
    dX = torch.full((N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    dW = torch.full((D, V), float("nan"), device=DEV)
    flce.flce_backward_ex(Xd, Wd, yd, lse, g, dX, dW, ws, *common, options=flce.make_options(row_band=row_band))
    assert flce.flce_check_device_error(ws) == 0
    dX32 = torch.full((N, D), float("nan"), device=DEV)
    dW2 = torch.full((D, V), float("nan"), device=DEV)
    flce.flce_backward_ex(Xd, Wd, yd, lse, g, None, dW2, ws, *common,
                          options=flce.make_options(dX_f32=dX32, row_band=row_band))
    assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    return dX.cpu(), dW.cpu().numpy(), dX32.cpu(), dW2.cpu().numpy()


@pytest.mark.parametrize("N,D,V,ignore_frac", [(1000, 136, 4104, 0.1), (2048, 256, 3000, 0.9),
                                               (777, 200, 1544, 0.5), (4100, 128, 2056, 0.05)])
def test_compacted_backward_equals_the_uncompacted_one(gpu_lib, N, D, V, ignore_frac):
    wl = custom("compact", N, D, V, seed=81, ignore_frac=ignore_frac, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y = make_inputs(wl)
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    dX, dW, dX32, dW2 = _both_paths(X, W, y, common)
    assert torch.equal(dX, dX32.to(torch.bfloat16))
    assert rel_fro(dW, dW2) <= 1e-5
    _, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y, *common)
    assert rel_fro(dX.float().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(dW, ref_dW) <= TOL_DW_REL
    ignored = y.numpy() == IGNORE_INDEX
    assert torch.all(dX[torch.from_numpy(ignored)] == 0)


@pytest.mark.parametrize("n_valid", [0, 1, 513])
def test_few_valid_rows(gpu_lib, n_valid):
    """No valid row (every gradient is zero), one, and one past a row-tile group."""
    wl = custom("fewvalid", 1500, 136, 2056, seed=82, label_smoothing=0.1, zloss_scale=1e-3, reduction="sum")
    X, W, y = make_inputs(wl)
    keep = np.random.default_rng(83).permutation(wl.N)[:n_valid]
    y2 = torch.full_like(y, IGNORE_INDEX)
    y2[torch.from_numpy(keep)] = y[torch.from_numpy(keep)]
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "sum")
    dX, dW, dX32, dW2 = _both_paths(X, W, y2, common)
    assert torch.equal(dX, dX32.to(torch.bfloat16))
    if n_valid == 0:
        assert torch.all(dX == 0) and np.all(dW == 0)
        return
    assert rel_fro(dW, dW2) <= 1e-5
    _, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y2, *common)
    assert rel_fro(dX.float().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(dW, ref_dW) <= TOL_DW_REL


def test_dx_aliasing_x_is_computed_in_place(gpu_lib):
    """dX given as X's own buffer: nothing may be staged there, so the backward runs
    uncompacted, reads X throughout and writes dX over it at the end."""
    wl = custom("alias", 1000, 136, 2056, seed=84, ignore_frac=0.2, label_smoothing=0.1)
    X, W, y = make_inputs(wl)
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    N, D, V = wl.N, wl.D, wl.V
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    ws = _ws(N, D, V)
    flce.flce_forward(Xd, Wd, yd, loss, lse, ws, *common)
    dW = torch.empty(D, V, device=DEV)
    flce.flce_backward(Xd, Wd, yd, lse, torch.ones(1, device=DEV), Xd, dW, ws, *common)
    assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    _, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y, *common)
    assert rel_fro(Xd.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(dW.cpu().numpy(), ref_dW) <= TOL_DW_REL


def test_compacted_dbias(gpu_lib):
    """With a bias, the dbias column sums stop at the valid-row count of the compacted band."""
    wl = custom("compact_bias", 1300, 136, 3000, seed=85, ignore_frac=0.3, label_smoothing=0.1)
    X, W, y = make_inputs(wl)
    bias = torch.tensor(np.random.default_rng(86).standard_normal(wl.V) * 0.5, dtype=torch.float32)
    N, D, V = wl.N, wl.D, wl.V
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    Xd, Wd, yd, bd = X.to(DEV), W.to(DEV), y.to(DEV), bias.to(DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    ws = _ws(N, D, V)
    flce.flce_forward_ex(Xd, Wd, yd, loss, lse, ws, *common, options=flce.make_options(bias=bd))
    g = torch.ones(1, device=DEV)
    outs = []
    for f32 in (False, True):
        dX = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
        dX32 = torch.empty(N, D, device=DEV) if f32 else None
        dW = torch.empty(D, V, device=DEV)
        db = torch.full((V,), float("nan"), device=DEV)
        flce.flce_backward_ex(Xd, Wd, yd, lse, g, None if f32 else dX, dW, ws, *common,
                              options=flce.make_options(bias=bd, dbias=db, dX_f32=dX32))
        assert flce.flce_check_device_error(ws) == 0
        outs.append(db.cpu().numpy())
    torch.cuda.synchronize()
    assert rel_fro(outs[0], outs[1]) <= 1e-5
    _, _, _, _, ref_db = oracle.forward_backward_ext(X, W, y, *common, bias=bias)
    assert rel_fro(outs[0], ref_db) <= TOL_DW_REL


@pytest.mark.parametrize("row_band", [384, 1000])
def test_compaction_per_row_band(gpu_lib, row_band):
    """Row bands: each band's valid rows are compacted into that band's rows of dX."""
    wl = custom("compact_band", 2500, 136, 3000, seed=87, ignore_frac=0.3, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y = make_inputs(wl)
    y[:400] = IGNORE_INDEX  # a whole band (or most of one) without a valid row
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    dX, dW, dX32, dW2 = _both_paths(X, W, y, common, row_band)
    assert torch.equal(dX, dX32.to(torch.bfloat16))
    assert rel_fro(dW, dW2) <= 1e-5
    _, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y, *common)
    assert rel_fro(dX.float().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(dW, ref_dW) <= TOL_DW_REL
