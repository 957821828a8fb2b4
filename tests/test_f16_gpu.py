"""GPU parity of f16 inputs (X and W f16, dX f16, dW fp32) against the fp64 oracle on
the same f16-rounded inputs. The f16 gradient band is stored as G/g scaled by 2^10;
these cases check that the scale is undone exactly where it must be (dX, dW, dbias) and
that g = 0 (every row ignored) still gives zero gradients."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, TOL_LOSS_REL, TOL_LSE_ABS, rel_fro
from workloads import IGNORE_INDEX, custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
F16 = torch.float16


def _ws(N, D, V, which):
    return torch.empty(flce.flce_workspace_size(N, D, V, which), dtype=torch.uint8, device=DEV)


def _run(X, W, y, common, opts, grad_out=1.0, vd=False):
    N, D = X.shape
    V = W.shape[1]
    Wd = (W.t().contiguous() if vd else W).to(DEV)
    Xd, yd = X.to(DEV), y.to(DEV)
    ws = _ws(N, D, V, 2)
    loss = torch.empty(N if common[3] == "none" else 1, device=DEV)
    lse = torch.empty(N, device=DEV)
    flce.flce_forward_ex(Xd, Wd, yd, loss, lse, ws, *common, options=opts)
    assert flce.flce_check_device_error(ws) == 0
    if common[3] == "none":
        return loss.cpu().double().numpy(), lse.cpu().double().numpy(), None, None
    g = torch.tensor([grad_out], device=DEV)
    dX = torch.full((N, D), float("nan"), dtype=F16, device=DEV)
    dW = torch.full(tuple(Wd.shape), float("nan"), device=DEV)
    flce.flce_backward_ex(Xd, Wd, yd, lse, g, dX, dW, ws, *common, options=opts)
    assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    dWn = dW.cpu().numpy()
    return loss.item(), lse.cpu().double().numpy(), dX.float().cpu().numpy(), (dWn.T if vd else dWn)


CASES = [
    # (N, D, V, eps, s, reduction, grad_out)
    (1, 8, 8, 0.0, 0.0, "mean", 1.0),
    (300, 128, 1000, 0.0, 0.0, "mean", 1.0),
    (1000, 136, 4104, 0.1, 1e-3, "sum", 0.5),
    (777, 264, 8200, 0.0, 1e-4, "mean", 2.0),
    (4096, 2048, 32000, 0.0, 0.0, "mean", 1.0),
]


@pytest.mark.parametrize("N,D,V,eps,s,red,go", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}" for c in CASES])
def test_f16_matches_the_oracle(gpu_lib, N, D, V, eps, s, red, go):
    wl = custom("f16", N, D, V, seed=61, ignore_frac=0.1 if N > 1 else 0.0, label_smoothing=eps,
                zloss_scale=s, reduction=red)
    X, W, y = make_inputs(wl, dtype=F16)
    common = (wl.ignore_index, eps, s, red)
    loss, lse, dX, dW = _run(X, W, y, common, flce.make_options(input_dtype="f16"), grad_out=go)
    ref_loss, ref_lse, ref_dX, ref_dW = oracle.forward_backward(X, W, y, *common, grad_out=go)
    valid = y.numpy() != IGNORE_INDEX
    assert abs(loss - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert np.max(np.abs(lse[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(dX, ref_dX) <= TOL_DX_REL
    assert rel_fro(dW, ref_dW) <= TOL_DW_REL


def test_f16_with_options_layout_and_row_bands(gpu_lib):
    wl = custom("f16_opts", 1000, 136, 4104, seed=62, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y = make_inputs(wl, dtype=F16)
    g = np.random.default_rng(6262)
    bias = torch.tensor(g.standard_normal(wl.V) * 0.5, dtype=torch.float32)
    cw = torch.tensor(g.uniform(0.25, 2.0, size=wl.V), dtype=torch.float32)
    N, D, V = wl.N, wl.D, wl.V
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean")
    Xd, yd, Wvd = X.to(DEV), y.to(DEV), W.t().contiguous().to(DEV)
    bd, wd = bias.to(DEV), cw.to(DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    fopt = flce.make_options(softcap=6.0, bias=bd, class_weight=wd, weight_layout="vd", input_dtype="f16")
    flce.flce_forward_ex(Xd, Wvd, yd, loss, lse, _ws(N, D, V, 0), *common, options=fopt)
    band = 384
    ws = _ws(band, D, V, 1)
    dX = torch.empty(N, D, dtype=F16, device=DEV)
    dW = torch.full((V, D), float("nan"), device=DEV)
    dbias = torch.empty(V, device=DEV)
    flce.flce_backward_ex(Xd, Wvd, yd, lse, torch.tensor([1.5], device=DEV), dX, dW, ws, *common,
                          options=flce.make_options(softcap=6.0, bias=bd, class_weight=wd, dbias=dbias,
                                                    row_band=band, weight_layout="vd", input_dtype="f16"))
    assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    ref_loss, ref_lse, ref_dX, ref_dW, ref_db = oracle.forward_backward_ext(
        X, W, y, *common, softcap=6.0, bias=bias, class_weight=cw, grad_out=1.5)
    valid = y.numpy() != IGNORE_INDEX
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert np.max(np.abs(lse.cpu().double().numpy()[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(dX.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(dW.cpu().numpy().T, ref_dW) <= TOL_DW_REL
    assert rel_fro(dbias.cpu().numpy(), ref_db) <= TOL_DW_REL


def test_f16_all_rows_ignored_gives_zero_gradients(gpu_lib):
    wl = custom("f16_ign", 300, 128, 1000, seed=63, ignore_frac=1.0)
    X, W, y = make_inputs(wl, dtype=F16)
    loss, _, dX, dW = _run(X, W, y, (IGNORE_INDEX, 0.0, 0.0, "mean"), flce.make_options(input_dtype="f16"))
    assert loss == 0.0
    assert np.all(dX == 0.0) and np.all(dW == 0.0)


def test_f16_reduction_none_forward(gpu_lib):
    wl = custom("f16_none", 500, 128, 2048, seed=64, ignore_frac=0.1)
    X, W, y = make_inputs(wl, dtype=F16)
    loss, lse, _, _ = _run(X, W, y, (IGNORE_INDEX, 0.0, 0.0, "none"), flce.make_options(input_dtype="f16"))
    ref_loss, ref_lse = oracle.forward(X, W, y, IGNORE_INDEX, 0.0, 0.0, "none")
    assert np.max(np.abs(loss - ref_loss)) <= 2e-3
    valid = y.numpy() != IGNORE_INDEX
    assert np.max(np.abs(lse[valid] - ref_lse[valid])) <= TOL_LSE_ABS


def test_f16_through_autograd(gpu_lib):
    wl = custom("f16_autograd", 512, 256, 3000, seed=65, ignore_frac=0.05)
    X, W, y = make_inputs(wl, dtype=F16)
    Xa = X.to(DEV).requires_grad_()
    Wa = W.to(DEV).requires_grad_()
    loss = flce.linear_cross_entropy(Xa, Wa, y.to(DEV))
    loss.backward()
    torch.cuda.synchronize()
    ref_loss, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y)
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert Xa.grad.dtype == F16 and Wa.grad.dtype == F16
    assert rel_fro(Xa.grad.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(Wa.grad.float().cpu().numpy(), ref_dW) <= 1e-2


def test_f16_gradient_range_is_reported(gpu_lib):
    """A class weight too large for the scaled f16 gradient band is reported, not hidden."""
    wl = custom("f16_range", 256, 128, 1024, seed=66)
    X, W, y = make_inputs(wl, dtype=F16)
    cw = torch.ones(wl.V, device=DEV)
    cw[int(y[0])] = 100.0  # (1 - eps) w_y = 100 > 64
    N, D, V = wl.N, wl.D, wl.V
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    ws = _ws(N, D, V, 2)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    opts = flce.make_options(class_weight=cw, input_dtype="f16")
    flce.flce_forward_ex(Xd, Wd, yd, loss, lse, ws, options=opts)
    assert flce.flce_check_device_error(ws) == 0
    dX = torch.empty(N, D, dtype=F16, device=DEV)
    dW = torch.empty(D, V, device=DEV)
    flce.flce_backward_ex(Xd, Wd, yd, lse, torch.ones(1, device=DEV), dX, dW, ws, options=opts)
    assert flce.STATUS[flce.flce_check_device_error(ws)] == "FLCE_ERR_F16_RANGE"
    # weights in range pass
    cw[int(y[0])] = 50.0
    flce.flce_backward_ex(Xd, Wd, yd, lse, torch.ones(1, device=DEV), dX, dW, ws, options=opts)
    assert flce.flce_check_device_error(ws) == 0
