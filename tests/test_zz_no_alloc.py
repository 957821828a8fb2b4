"""flce_forward_noalloc: the forward pass for callers that cannot allocate device
memory (allocator or memory-pool callbacks, fixed device arenas). Its scratch is a
static device array inside the library, so the caller passes only inputs and
outputs. It must agree with flce_forward (which takes a caller-owned workspace)
within the parity tolerances, call after call, since every call reuses the array.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
from tests.flce_cases import TOL_LOSS_REL, TOL_LSE_ABS
from workloads import custom, make_inputs

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    fn = lib.flce_forward_noalloc
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    fn.argtypes = [vp, vp, vp, i64, i64, i64, i32, f32, f32, ctypes.c_int, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def _run_both(fn, wl):
    X, W, y = make_inputs(wl)
    dev = torch.device("cuda:0")
    Xd, Wd, yd = X.to(dev), W.to(dev), y.to(dev)
    n_loss = wl.N if wl.reduction == "none" else 1
    red = flce.REDUCTIONS[wl.reduction]
    stream = torch.cuda.current_stream(dev).cuda_stream
    # existing entry point, caller-owned workspace
    ws = torch.empty(flce.flce_workspace_size(wl.N, wl.D, wl.V, False), dtype=torch.uint8, device=dev)
    loss_ref = torch.full((n_loss,), float("nan"), device=dev)
    lse_ref = torch.full((wl.N,), float("nan"), device=dev)
    flce.flce_forward(Xd, Wd, yd, loss_ref, lse_ref, ws, wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                      wl.reduction)
    # the entry point without a workspace
    loss = torch.full((n_loss,), float("nan"), device=dev)
    lse = torch.full((wl.N,), float("nan"), device=dev)
    st = fn(Xd.data_ptr(), Wd.data_ptr(), yd.data_ptr(), wl.N, wl.D, wl.V, wl.ignore_index, wl.label_smoothing,
            wl.zloss_scale, red, loss.data_ptr(), lse.data_ptr(), stream)
    assert st == 0, flce.flce_status_string(st)
    torch.cuda.synchronize(dev)
    valid = (y != wl.ignore_index).numpy()
    a, b = loss.cpu().double().numpy(), loss_ref.cpu().double().numpy()
    assert np.all(np.abs(a - b) <= TOL_LOSS_REL * np.maximum(np.abs(b), 1e-30))
    la, lb = lse.cpu().double().numpy(), lse_ref.cpu().double().numpy()
    assert np.max(np.abs(la[valid] - lb[valid])) <= TOL_LSE_ABS


def test_noalloc_forward_matches_workspace_forward(gpu_lib):
    fn = _noalloc(flce.load_library())
    # two calls in a row on the shared scratch, with different shapes and options
    _run_both(fn, custom("na1", 1000, 136, 4104, seed=201, ignore_frac=0.1, label_smoothing=0.1,
                         zloss_scale=1e-4, reduction="mean"))
    _run_both(fn, custom("na2", 700, 256, 2048, seed=202, ignore_frac=0.05, reduction="sum"))
    _run_both(fn, custom("na3", 300, 64, 1024, seed=203, reduction="none"))


def test_noalloc_refuses_shapes_beyond_its_scratch(gpu_lib):
    fn = _noalloc(flce.load_library())
    N, D, V = 262144, 8, 128256  # forward scratch ~200 MB > 64 MiB
    assert flce.flce_workspace_size(N, D, V, False) > (64 << 20)
    dev = torch.device("cuda:0")
    X = torch.zeros(N, D, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(D, V, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(N, dtype=torch.int32, device=dev)
    loss = torch.zeros(1, device=dev)
    lse = torch.zeros(N, device=dev)
    st = fn(X.data_ptr(), W.data_ptr(), y.data_ptr(), N, D, V, -100, 0.0, 0.0, 0, loss.data_ptr(), lse.data_ptr(),
            torch.cuda.current_stream(dev).cuda_stream)
    assert st == 4  # FLCE_ERR_WORKSPACE_TOO_SMALL
