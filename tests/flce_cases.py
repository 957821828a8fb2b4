"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI and
compare with the fp64 oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import linear_cross_entropy_tcgen05_gb300 as flce

# Tolerances: loss relative error, per-row LSE absolute error (valid rows),
# dX relative Frobenius error, dW relative Frobenius error (fp32 accumulation).
TOL_LOSS_REL = 1e-4
TOL_LSE_ABS = 2e-3
TOL_DX_REL = 1e-2
TOL_DW_REL = 5e-3


def rel_fro(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    return float(num / den) if den > 0 else float(num)


class CudaRun:
    """Device buffers and one forward (+ backward) of the CUDA path."""

    def __init__(self, X, W, y, ignore_index=-100, label_smoothing=0.0, zloss_scale=0.0, reduction="mean",
                 device="cuda:0"):
        self.dev = torch.device(device)
        self.N, self.D = X.shape
        self.V = W.shape[1]
        self.X = X.to(self.dev)
        self.W = W.to(self.dev)
        self.y = y.to(self.dev)
        self.opts = (ignore_index, label_smoothing, zloss_scale, reduction)
        self.reduction = reduction
        N, D, V = self.N, self.D, self.V
        self.ws = torch.empty(max(flce.flce_workspace_size(N, D, V, False), flce.flce_workspace_size(N, D, V, True)),
                              dtype=torch.uint8, device=self.dev)
        self.loss = torch.full((N if reduction == "none" else 1,), float("nan"), dtype=torch.float32, device=self.dev)
        self.lse = torch.full((N,), float("nan"), dtype=torch.float32, device=self.dev)
        self.dX = None
        self.dW = None

    def forward(self):
        flce.flce_forward(self.X, self.W, self.y, self.loss, self.lse, self.ws, *self.opts)
        return flce.flce_check_device_error(self.ws)

    def backward(self, grad_out=1.0):
        g = torch.tensor([grad_out], dtype=torch.float32, device=self.dev)
        self.dX = torch.full((self.N, self.D), float("nan"), dtype=torch.bfloat16, device=self.dev)
        self.dW = torch.full((self.D, self.V), float("nan"), dtype=torch.float32, device=self.dev)
        flce.flce_backward(self.X, self.W, self.y, self.lse, g, self.dX, self.dW, self.ws, *self.opts)
        return flce.flce_check_device_error(self.ws)

    def host(self):
        torch.cuda.synchronize(self.dev)
        out = {"loss": self.loss.cpu().double().numpy(), "lse": self.lse.cpu().double().numpy()}
        if self.dX is not None:
            out["dX"] = self.dX.float().cpu().double().numpy()
            out["dW"] = self.dW.cpu().double().numpy()
        return out
