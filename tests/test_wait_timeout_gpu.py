"""Failure detection on the GPU without a fault: a kernel whose pipeline wait (the
bounded mbarrier wait of the GEMMs) waits for an arrival that never comes gives up
after the wait limit, reports FLCE_ERR_TIMEOUT through the workspace, and leaves the
context usable for the next call."""
import time

import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
import oracle
from tests.flce_cases import TOL_LOSS_REL, CudaRun
from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_a_wait_that_runs_out_reports_a_timeout_and_the_context_survives(gpu_lib):
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    t0 = time.perf_counter()
    assert flce.flce_selftest_wait_timeout(ws) == 0
    st = flce.flce_check_device_error(ws)
    elapsed = time.perf_counter() - t0
    assert flce.STATUS[st] == "FLCE_ERR_TIMEOUT"
    assert 1.5 < elapsed < 60.0, elapsed          # the 2 s limit, not a hang
    assert flce.flce_check_device_error(ws) == 0   # the word was read and cleared
    # the next call on the same context works and is correct
    wl = WORKLOADS["tiny"]
    X, W, y = make_inputs(wl)
    run = CudaRun(X, W, y)
    assert run.forward() == 0
    assert run.backward() == 0
    loss, _, _, _ = oracle.forward_backward(X, W, y)
    got = run.host()
    assert abs(got["loss"][0] - loss) <= TOL_LOSS_REL * abs(loss)
    assert np.isfinite(got["dW"]).all()
