"""GPU parity on the five named workloads, in the launch configuration the benchmark
times. The small-vocabulary workload is compared in full; the three large ones on the
full loss (every row through the oracle), 512 seeded rows of lse and dX, and 512
seeded vocabulary columns of dW (all D entries)."""
import time

import numpy as np
import pytest

import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, TOL_LOSS_REL, TOL_LSE_ABS, CudaRun, rel_fro
from workloads import WORKLOADS, make_inputs, sample_indices

pytestmark = pytest.mark.gpu


def _gpu(wl, X, W, y):
    run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    assert run.forward() == 0
    assert run.backward() == 0
    return run.host()


@pytest.mark.parametrize("name", ["tiny", "small_vocab"])
def test_workload_full(gpu_lib, name):
    wl = WORKLOADS[name]
    X, W, y = make_inputs(wl)
    got = _gpu(wl, X, W, y)
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                                                wl.reduction)
    valid = y.numpy() != wl.ignore_index
    errs = {"loss": abs(got["loss"][0] - loss) / abs(loss),
            "lse": float(np.max(np.abs(got["lse"][valid] - lse[valid]))),
            "dX": rel_fro(got["dX"], dX), "dW": rel_fro(got["dW"], dW)}
    print(name, errs)
    assert errs["loss"] <= TOL_LOSS_REL and errs["lse"] <= TOL_LSE_ABS
    assert errs["dX"] <= TOL_DX_REL and errs["dW"] <= TOL_DW_REL


@pytest.mark.parametrize("name", ["llama8k", "large_vocab", "headline"])
def test_workload_sampled(gpu_lib, name):
    wl = WORKLOADS[name]
    t0 = time.time()
    X, W, y = make_inputs(wl)
    got = _gpu(wl, X, W, y)
    t1 = time.time()
    W64 = oracle.widen(W)
    lse_all, ell_all = oracle.full_row_stats(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                                             W64=W64)
    yv = y.numpy()
    valid = yv != wl.ignore_index
    loss = oracle.reduce_loss(ell_all, valid, wl.reduction)
    g = oracle.grad_scale(1.0, int(valid.sum()), wl.reduction)
    rows = sample_indices(wl.N, 512, seed=wl.seed)
    cols = sample_indices(wl.V, 512, seed=wl.seed + 1)
    dX_rows = oracle.grad_x_rows(X, W, y, rows, lse_all[rows], g, wl.ignore_index, wl.label_smoothing,
                                 wl.zloss_scale, W64=W64)
    del W64
    dW_cols = oracle.grad_w_cols(X, W, y, cols, lse_all, g, wl.ignore_index, wl.label_smoothing, wl.zloss_scale)
    t2 = time.time()
    vr = valid[rows]
    errs = {"loss": abs(got["loss"][0] - loss) / abs(loss),
            "lse_rows": float(np.max(np.abs(got["lse"][rows][vr] - lse_all[rows][vr]))),
            "lse_all": float(np.max(np.abs(got["lse"][valid] - lse_all[valid]))),
            "dX_rows": rel_fro(got["dX"][rows], dX_rows),
            "dW_cols": rel_fro(got["dW"][:, cols], dW_cols)}
    print(name, errs, f"gpu+inputs {t1 - t0:.1f}s oracle {t2 - t1:.1f}s")
    assert errs["loss"] <= TOL_LOSS_REL
    assert errs["lse_rows"] <= TOL_LSE_ABS and errs["lse_all"] <= TOL_LSE_ABS
    assert errs["dX_rows"] <= TOL_DX_REL
    assert errs["dW_cols"] <= TOL_DW_REL
    # ignored rows: exactly zero dX at full size
    assert np.all(got["dX"][~valid] == 0.0)
