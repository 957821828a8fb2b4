"""Non-finite inputs propagate as in IEEE arithmetic, and only where the mathematics sends
them: a row of X that holds NaN gives that row a NaN lse and a NaN loss, a NaN mean loss,
a NaN row of dX and (since every element of dW sums over every row) a NaN dW; every other
row's lse and dX is bit-for-bit what the same inputs without the NaN give. Nothing hangs,
and the device error word stays clear (a NaN is data, not a fault)."""
import numpy as np
import pytest
import torch

from tests.flce_cases import CudaRun
from workloads import IGNORE_INDEX, custom, make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bad", ["nan", "inf"])
def test_a_non_finite_row_stays_in_its_row(gpu_lib, bad):
    wl = custom("nonfinite", 700, 136, 4104, seed=71, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y = make_inputs(wl)
    r = int(np.nonzero(y.numpy() != IGNORE_INDEX)[0][5])  # a valid row
    Xb = X.clone()
    Xb[r] = float(bad)
    runs = []
    for Xi in (X, Xb):
        run = CudaRun(Xi, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
        assert run.forward() == 0
        assert run.backward() == 0
        runs.append(run.host())
    clean, dirty = runs
    others = np.arange(wl.N) != r
    assert np.isnan(dirty["loss"][0]) and np.isfinite(clean["loss"][0])
    assert not np.isfinite(dirty["lse"][r])
    assert np.array_equal(dirty["lse"][others], clean["lse"][others])
    assert np.all(np.isnan(dirty["dX"][r]))
    assert np.array_equal(dirty["dX"][others], clean["dX"][others])
    assert np.all(np.isnan(dirty["dW"]))
