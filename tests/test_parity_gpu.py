"""GPU parity on small problems: every output compared element by element with the
fp64 oracle (sizes that span several tiles and ragged tails), plus edge cases."""
import numpy as np
import pytest
import torch

import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, TOL_LOSS_REL, TOL_LSE_ABS, CudaRun, rel_fro
from workloads import IGNORE_INDEX, WORKLOADS, custom, make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # name, N, D, V, options
    ("tiny", WORKLOADS["tiny"]),
    ("ragged_rows_cols", custom("ragged", 1000, 136, 1000, seed=5, ignore_frac=0.1)),
    ("ragged_all_terms_sum", custom("ragged2", 777, 200, 4104, seed=6, ignore_frac=0.05, label_smoothing=0.1,
                                    zloss_scale=1e-4, reduction="sum")),
    ("one_tile_plus_one", custom("t129", 129, 64, 264, seed=7)),
    ("minimal", custom("min", 1, 8, 8, seed=8)),
    ("vocab_32008", custom("v32008", 300, 64, 32008, seed=9, ignore_frac=0.2, label_smoothing=0.05)),
    ("zloss_mean", custom("zl", 512, 256, 2048, seed=10, zloss_scale=0.01, ignore_frac=0.3)),
    ("deep_k", custom("deepk", 256, 1032, 768, seed=11, reduction="sum")),
    # ignore_index that is also a class id, near-total smoothing, a strong z-loss
    ("unusual_options", custom("odd", 333, 72, 1544, seed=22, ignore_frac=0.1, ignore_index=0,
                               label_smoothing=0.999, zloss_scale=1.0)),
    # a vocabulary of 8 or 16 with heavy smoothing: each non-target column gets eps/V of the
    # target mass, so spreading it over V-1 columns instead is ~7% of a gradient entry
    ("small_vocab_smoothing_mean", custom("v8s", 512, 64, 8, seed=23, ignore_frac=0.1, label_smoothing=0.5)),
    ("small_vocab_smoothing_sum", custom("v16s", 512, 64, 16, seed=24, ignore_frac=0.1, label_smoothing=0.9,
                                         reduction="sum")),
]


def _check(wl, grad_out=1.0):
    X, W, y = make_inputs(wl)
    run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    assert run.forward() == 0
    assert run.backward(grad_out) == 0
    got = run.host()
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                                                wl.reduction, grad_out=grad_out)
    valid = y.numpy() != wl.ignore_index
    assert abs(got["loss"][0] - loss) <= TOL_LOSS_REL * abs(loss)
    assert np.max(np.abs(got["lse"][valid] - lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(got["dX"], dX) <= TOL_DX_REL
    assert rel_fro(got["dW"], dW) <= TOL_DW_REL
    assert np.all(got["dX"][~valid] == 0.0), "ignored rows must have exactly zero dX"
    return got


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_parity_small(gpu_lib, name, wl):
    _check(wl)


def test_scalar_upstream_gradient(gpu_lib):
    """A loss that is not the last layer: grad_out != 1 scales dX and dW."""
    _check(custom("g25", 300, 128, 1024, seed=12, ignore_frac=0.1), grad_out=2.5)
    _check(custom("gneg", 300, 128, 1024, seed=13, reduction="sum"), grad_out=-0.75)


def test_reduction_none_forward(gpu_lib):
    wl = custom("none", 600, 128, 3000, seed=14, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-3,
                reduction="none")
    X, W, y = make_inputs(wl)
    run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "none")
    assert run.forward() == 0
    got = run.host()
    ell, lse = oracle.forward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "none")
    assert np.max(np.abs(got["loss"] - ell) / np.maximum(1.0, np.abs(ell))) <= TOL_LOSS_REL
    ign = y.numpy() == wl.ignore_index
    assert np.all(got["loss"][ign] == 0.0)
    # the backward refuses 'none'
    import linear_cross_entropy_tcgen05_gb300 as flce
    g = torch.ones(1, device="cuda")
    st = flce.flce_backward(run.X, run.W, run.y, run.lse, g, torch.empty_like(run.X),
                            torch.empty(wl.D, wl.V, device="cuda"), run.ws, *run.opts, raise_on_error=False)
    assert st == 5


def test_all_rows_ignored_mean_is_zero(gpu_lib):
    wl = custom("allign", 200, 64, 512, seed=15, ignore_frac=1.0)
    X, W, y = make_inputs(wl)
    run = CudaRun(X, W, y)
    assert run.forward() == 0
    assert run.backward() == 0
    got = run.host()
    assert got["loss"][0] == 0.0
    assert np.all(got["dX"] == 0.0) and np.all(got["dW"] == 0.0)


def test_bad_target_sets_the_error_word_and_poisons_its_row(gpu_lib):
    wl = custom("bad", 256, 64, 512, seed=16)
    X, W, y = make_inputs(wl)
    y[5] = wl.V + 3
    y[9] = -7
    run = CudaRun(X, W, y, reduction="none")
    assert run.forward() == 7  # FLCE_ERR_BAD_TARGET
    got = run.host()
    assert np.isnan(got["loss"][5]) and np.isnan(got["loss"][9])
    ok = np.ones(wl.N, bool)
    ok[[5, 9]] = False
    assert np.all(np.isfinite(got["loss"][ok]))
    # the error word is cleared by reading it
    import linear_cross_entropy_tcgen05_gb300 as flce
    assert flce.flce_check_device_error(run.ws) == 0
    run2 = CudaRun(X, W, y, reduction="sum")
    assert run2.forward() == 7
    assert run2.backward() == 7
    g = run2.host()
    assert np.isnan(g["loss"][0])
    assert np.all(np.isnan(g["dX"][5])) and np.all(np.isfinite(g["dX"][ok]))


def test_bitwise_deterministic(gpu_lib):
    wl = custom("det", 700, 256, 5000, seed=17, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-4)
    X, W, y = make_inputs(wl)
    outs = []
    for _ in range(2):
        run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
        assert run.forward() == 0 and run.backward() == 0
        outs.append(run.host())
    for k in ("loss", "lse", "dX", "dW"):
        assert np.array_equal(outs[0][k], outs[1][k]), k


def test_ignored_rows_do_not_change_dw(gpu_lib):
    """Changing the hidden state of ignored rows leaves the loss and dW bit-identical."""
    wl = custom("ignx", 512, 128, 2048, seed=18, ignore_frac=0.25)
    X, W, y = make_inputs(wl)
    r1 = CudaRun(X, W, y)
    assert r1.forward() == 0 and r1.backward() == 0
    a = r1.host()
    X2 = X.clone()
    ign = (y == IGNORE_INDEX)
    X2[ign] = (X2[ign].float() * -3.0 + 1.0).bfloat16()
    r2 = CudaRun(X2, W, y)
    assert r2.forward() == 0 and r2.backward() == 0
    b = r2.host()
    assert np.array_equal(a["loss"], b["loss"])
    assert np.array_equal(a["dW"], b["dW"])


@pytest.mark.parametrize("N", [384, 2300], ids=["small", "valid_row_forward"])
def test_autograd_wrapper(gpu_lib, N):
    """Through torch.autograd; from 2048 rows a training forward runs on the valid rows."""
    import linear_cross_entropy_tcgen05_gb300 as flce
    wl = custom("ag", N, 128, 1024, seed=19, ignore_frac=0.1)
    X, W, y = make_inputs(wl)
    Xd = X.cuda().requires_grad_(True)
    Wd = W.cuda().requires_grad_(True)
    loss = flce.linear_cross_entropy(Xd, Wd, y.cuda())
    (2.0 * loss).backward()
    ref_loss, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y, grad_out=2.0)
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert rel_fro(Xd.grad.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(Wd.grad.float().cpu().numpy(), ref_dW) <= 1e-2  # dW returned in bf16 through autograd


def test_zero_weights_give_the_closed_form(gpu_lib):
    """W = 0: every logit is 0, lse = ln V (0 on an ignored row, whose lse the forward
    does not compute), loss = ln V + s (ln V)^2, dX = 0 and
    dZ = g (p (1 + 2 s lse) - (1 - eps) onehot - eps/V) with p = 1/V (the oracle's own pin,
    here on the GPU)."""
    import math
    wl = custom("w0", 300, 128, 1000, seed=20, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y = make_inputs(wl)
    W = torch.zeros_like(W)
    run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean")
    assert run.forward() == 0
    assert run.backward() == 0
    got = run.host()
    lnV = math.log(wl.V)
    valid = y.numpy() != wl.ignore_index
    assert np.max(np.abs(got["lse"][valid] - lnV)) <= 1e-5
    assert np.all(got["lse"][~valid] == 0.0)
    assert abs(got["loss"][0] - (lnV + 1e-3 * lnV * lnV)) <= 1e-5
    assert np.all(got["dX"] == 0.0)
    _, _, _, ref_dW = oracle.forward_backward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean")
    assert rel_fro(got["dW"], ref_dW) <= TOL_DW_REL
    assert valid.sum() > 0


def test_large_logits_stay_finite(gpu_lib):
    """Logits in the hundreds (X scaled by 64): the online softmax keeps every exponent
    <= 0, so nothing overflows, and the results still match the oracle. Ignored rows must
    give exact zeros here too (their coefficient has an exponent of -inf, not 0: with 0,
    exp2 of a logit above ~88 overflows and 0 * inf poisons dW with NaN)."""
    wl = custom("big", 512, 256, 4104, seed=21, ignore_frac=0.05, label_smoothing=0.1, zloss_scale=1e-4)
    X, W, y = make_inputs(wl)
    X = (X.float() * 64).bfloat16()
    run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean")
    assert run.forward() == 0
    assert run.backward() == 0
    got = run.host()
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                                                "mean")
    valid = y.numpy() != wl.ignore_index
    assert np.isfinite(got["loss"]).all() and np.isfinite(got["dW"]).all() and np.isfinite(got["dX"]).all()
    assert abs(got["loss"][0] - loss) <= TOL_LOSS_REL * abs(loss)
    assert np.max(np.abs(got["lse"][valid] - lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(got["dX"], dX) <= TOL_DX_REL
    assert rel_fro(got["dW"], dW) <= TOL_DW_REL


@pytest.mark.parametrize("where", ["first", "last"])
def test_targets_at_the_vocabulary_edges(gpu_lib, where):
    """Every target in column 0, or in column V-1 (inside the last, partly masked tile):
    the one tile that holds the target captures its logit."""
    wl = custom("edge", 300, 128, 1000, seed=23, label_smoothing=0.1)
    X, W, y = make_inputs(wl)
    y = torch.full_like(y, 0 if where == "first" else wl.V - 1)
    y[::7] = IGNORE_INDEX
    run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing)
    assert run.forward() == 0
    assert run.backward() == 0
    got = run.host()
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, wl.ignore_index, wl.label_smoothing)
    assert abs(got["loss"][0] - loss) <= TOL_LOSS_REL * abs(loss)
    assert rel_fro(got["dX"], dX) <= TOL_DX_REL
    assert rel_fro(got["dW"], dW) <= TOL_DW_REL
