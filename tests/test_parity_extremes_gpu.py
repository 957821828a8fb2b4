"""GPU parity at the edges of the shape space, compared in full with the fp64 oracle:
a hidden size of 16384 (256 K blocks per tile), a vocabulary of half a million
(many bands, the split count at its cap) and a quarter of a million rows with a
one-block hidden size (many row blocks per cluster)."""
import numpy as np
import pytest

import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, TOL_LOSS_REL, TOL_LSE_ABS, CudaRun, rel_fro
from workloads import custom, make_inputs

pytestmark = pytest.mark.gpu

EXTREMES = [
    ("wide_hidden", custom("d16k", 512, 16384, 4104, seed=81, ignore_frac=0.05, label_smoothing=0.1)),
    ("half_million_vocab", custom("v512k", 256, 128, 524296, seed=82, ignore_frac=0.1, zloss_scale=1e-4)),
    ("quarter_million_rows", custom("n256k", 262144, 64, 520, seed=83, ignore_frac=0.05, reduction="sum")),
]


@pytest.mark.parametrize("name,wl", EXTREMES, ids=[c[0] for c in EXTREMES])
def test_parity_at_extreme_shapes(gpu_lib, name, wl):
    X, W, y = make_inputs(wl)
    run = CudaRun(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    assert run.forward() == 0
    assert run.backward(1.0) == 0
    got = run.host()
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                                                wl.reduction)
    valid = y.numpy() != wl.ignore_index
    assert abs(got["loss"][0] - loss) <= TOL_LOSS_REL * abs(loss)
    assert np.max(np.abs(got["lse"][valid] - lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(got["dX"], dX) <= TOL_DX_REL
    assert rel_fro(got["dW"], dW) <= TOL_DW_REL
