"""flce_forward_noalloc: the forward pass for callers that cannot allocate device
memory (allocator or memory-pool callbacks, fixed device arenas). Its scratch is a
static device array inside the library, so the caller passes only inputs and
outputs. Every call reuses the array, so it is checked call after call: against
flce_forward (which takes a caller-owned workspace and runs the same kernels, so the
results must be identical bit for bit), against the fp64 oracle within the parity
tolerances, for allocating nothing, and for its error behaviour.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
import oracle
from tests.flce_cases import TOL_LOSS_REL, TOL_LSE_ABS
from workloads import WORKLOADS, custom, make_inputs, sample_indices

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20


def _noalloc(lib):
    fn = lib.flce_forward_noalloc
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    fn.argtypes = [vp, vp, vp, i64, i64, i64, i32, f32, f32, ctypes.c_int, vp, vp, vp]
    fn.restype = ctypes.c_int
    return fn


class _Both:
    """One problem on the device, run through flce_forward (caller workspace) and
    through flce_forward_noalloc (library scratch)."""

    def __init__(self, fn, wl, X, W, y, reduction=None):
        self.fn, self.wl = fn, wl
        self.red = wl.reduction if reduction is None else reduction
        self.dev = torch.device("cuda:0")
        self.X, self.W, self.y = X.to(self.dev), W.to(self.dev), y.to(self.dev)
        self.n_loss = wl.N if self.red == "none" else 1
        self.stream = torch.cuda.current_stream(self.dev).cuda_stream
        self.ws = torch.empty(flce.flce_workspace_size(wl.N, wl.D, wl.V, False), dtype=torch.uint8, device=self.dev)
        self.opts = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale)

    def workspace_call(self):
        loss = torch.full((self.n_loss,), float("nan"), device=self.dev)
        lse = torch.full((self.wl.N,), float("nan"), device=self.dev)
        flce.flce_forward(self.X, self.W, self.y, loss, lse, self.ws, *self.opts, self.red)
        return loss, lse

    def noalloc_call(self, loss=None, lse=None):
        wl = self.wl
        if loss is None:
            loss = torch.full((self.n_loss,), float("nan"), device=self.dev)
            lse = torch.full((wl.N,), float("nan"), device=self.dev)
        st = self.fn(self.X.data_ptr(), self.W.data_ptr(), self.y.data_ptr(), wl.N, wl.D, wl.V, wl.ignore_index,
                     wl.label_smoothing, wl.zloss_scale, flce.REDUCTIONS[self.red], loss.data_ptr(), lse.data_ptr(),
                     self.stream)
        assert st == 0, flce.flce_status_string(st)
        return loss, lse


def _bitwise(a, b):
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def _check_full(fn, wl):
    """Both entry points bit for bit, and the oracle over every row."""
    X, W, y = make_inputs(wl)
    both = _Both(fn, wl, X, W, y)
    loss_ws, lse_ws = both.workspace_call()
    loss, lse = both.noalloc_call()
    torch.cuda.synchronize()
    assert _bitwise(loss, loss_ws) and _bitwise(lse, lse_ws)
    ref_loss, ref_lse = oracle.forward(X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    valid = y.numpy() != wl.ignore_index
    got_loss = loss.cpu().double().numpy()
    got_lse = lse.cpu().double().numpy()
    ref_loss = np.atleast_1d(np.asarray(ref_loss, dtype=np.float64))
    assert np.all(np.abs(got_loss - ref_loss) <= TOL_LOSS_REL * np.maximum(np.abs(ref_loss), 1.0 if
                                                                           wl.reduction == "none" else 1e-30))
    assert np.max(np.abs(got_lse[valid] - ref_lse[valid])) <= TOL_LSE_ABS


def test_noalloc_forward_matches_workspace_forward_and_oracle(gpu_lib):
    fn = _noalloc(flce.load_library())
    # calls in a row on the shared scratch, with different shapes and options
    _check_full(fn, custom("na1", 1000, 136, 4104, seed=201, ignore_frac=0.1, label_smoothing=0.1,
                           zloss_scale=1e-4, reduction="mean"))
    _check_full(fn, custom("na2", 700, 256, 2048, seed=202, ignore_frac=0.05, reduction="sum"))
    _check_full(fn, custom("na3", 300, 64, 1024, seed=203, reduction="none"))
    # room in the scratch for the forward on the valid rows (the workspace call above it
    # runs on every row): the two must still agree bit for bit
    big = custom("na6", 4096, 256, 8200, seed=206, ignore_frac=0.3, label_smoothing=0.05)
    assert flce.flce_workspace_size(big.N, big.D, big.V, "forward_valid_rows") <= SCRATCH_BYTES
    _check_full(fn, big)
    _check_full(fn, custom("na1", 1000, 136, 4104, seed=201, ignore_frac=0.1, label_smoothing=0.1,
                           zloss_scale=1e-4, reduction="mean"))


def test_noalloc_llama8k_shape(gpu_lib):
    """The Llama-3-8B head on one 8192-token sequence (N=8192, D=4096, V=128256): its
    forward scratch (64 vocabulary splits) fits the array. Bit for bit against
    flce_forward with the workload's mean reduction and with per-row losses, and the
    per-row losses and lse of 512 seeded rows against the oracle."""
    fn = _noalloc(flce.load_library())
    wl = WORKLOADS["llama8k"]
    assert flce.flce_workspace_size(wl.N, wl.D, wl.V, False) <= SCRATCH_BYTES
    X, W, y = make_inputs(wl)
    for red in ("mean", "none"):
        both = _Both(fn, wl, X, W, y, reduction=red)
        loss_ws, lse_ws = both.workspace_call()
        loss, lse = both.noalloc_call()
        loss2, lse2 = both.noalloc_call()  # a second call on the same scratch
        torch.cuda.synchronize()
        assert _bitwise(loss, loss_ws) and _bitwise(lse, lse_ws), red
        assert _bitwise(loss2, loss) and _bitwise(lse2, lse), red
    rows = sample_indices(wl.N, 512, seed=wl.seed + 11)
    idx = torch.from_numpy(rows)
    ref_ell, ref_lse = oracle.forward(X[idx], W, y[idx], wl.ignore_index, wl.label_smoothing, wl.zloss_scale,
                                      "none")
    got_ell = loss.cpu().double().numpy()[rows]
    got_lse = lse.cpu().double().numpy()[rows]
    valid = y.numpy()[rows] != wl.ignore_index
    assert np.max(np.abs(got_lse[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert np.all(np.abs(got_ell - ref_ell) <= TOL_LOSS_REL * np.maximum(np.abs(ref_ell), 1.0))


def test_noalloc_allocates_nothing(gpu_lib):
    """A warm call changes neither torch's allocator count nor the device's free memory
    (an allocation would take at least one 2 MiB page)."""
    fn = _noalloc(flce.load_library())
    wl = custom("na4", 2048, 512, 8192, seed=204, ignore_frac=0.1)
    X, W, y = make_inputs(wl)
    both = _Both(fn, wl, X, W, y)
    loss = torch.empty(1, device=both.dev)
    lse = torch.empty(wl.N, device=both.dev)
    both.noalloc_call(loss, lse)  # first call on this device: module load and address look-up
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        both.noalloc_call(loss, lse)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_before - free_after < (2 << 20), (free_before, free_after)


def test_noalloc_bad_target_poisons_the_loss(gpu_lib):
    """The error word is internal, so a target outside [0, V) shows as NaN: in its row's
    loss and in the reduced loss; the other rows stay finite."""
    fn = _noalloc(flce.load_library())
    wl = custom("na5", 256, 64, 512, seed=205)
    X, W, y = make_inputs(wl)
    y[17] = wl.V + 5
    for red in ("mean", "none"):
        loss, lse = _Both(fn, wl, X, W, y, reduction=red).noalloc_call()
        torch.cuda.synchronize()
        got = loss.cpu().numpy()
        if red == "mean":
            assert np.isnan(got[0])
        else:
            ok = np.ones(wl.N, bool)
            ok[17] = False
            assert np.isnan(got[17]) and np.all(np.isfinite(got[ok]))
    # the next call with valid targets is clean again
    y[17] = 3
    loss, _ = _Both(fn, wl, X, W, y).noalloc_call()
    torch.cuda.synchronize()
    assert np.isfinite(loss.item())


def test_noalloc_refuses_shapes_beyond_its_scratch(gpu_lib):
    fn = _noalloc(flce.load_library())
    N, D, V = 262144, 8, 128256  # forward scratch ~200 MB > 64 MiB
    assert flce.flce_workspace_size(N, D, V, False) > SCRATCH_BYTES
    dev = torch.device("cuda:0")
    X = torch.zeros(N, D, dtype=torch.bfloat16, device=dev)
    W = torch.zeros(D, V, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(N, dtype=torch.int32, device=dev)
    loss = torch.zeros(1, device=dev)
    lse = torch.zeros(N, device=dev)
    st = fn(X.data_ptr(), W.data_ptr(), y.data_ptr(), N, D, V, -100, 0.0, 0.0, 0, loss.data_ptr(), lse.data_ptr(),
            torch.cuda.current_stream(dev).cuda_stream)
    assert st == 4  # FLCE_ERR_WORKSPACE_TOO_SMALL
