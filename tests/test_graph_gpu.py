"""The forward and backward calls captured into a CUDA graph and replayed on new
inputs give the same bits as eager calls: every entry point is stream-ordered, and
after a first eager call it makes no allocation, synchronisation or attribute call."""
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
from workloads import custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_forward_backward_replayed_from_a_cuda_graph(gpu_lib):
    wl = custom("graph", 1000, 136, 4104, seed=71, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-4)
    X1, W, y1 = make_inputs(wl)
    X2, _, y2 = make_inputs(wl, seed=72)  # a second batch for the same W
    N, D, V = wl.N, wl.D, wl.V
    Xd = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    yd = torch.empty(N, dtype=torch.int32, device=DEV)
    Wd = W.to(DEV)
    ws = torch.empty(flce.flce_workspace_size(N, D, V, 2), dtype=torch.uint8, device=DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    dX = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = torch.empty(D, V, device=DEV)
    g = torch.tensor([0.5], device=DEV)
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean")

    def step():
        flce.flce_forward(Xd, Wd, yd, loss, lse, ws, *common)
        flce.flce_backward(Xd, Wd, yd, lse, g, dX, dW, ws, *common)

    eager = []
    for Xh, yh in ((X1, y1), (X2, y2)):
        Xd.copy_(Xh)
        yd.copy_(yh)
        step()
        assert flce.flce_check_device_error(ws) == 0
        eager.append([t.clone() for t in (loss, lse, dX, dW)])

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for (Xh, yh), want in zip(((X2, y2), (X1, y1)), (eager[1], eager[0])):
        Xd.copy_(Xh)
        yd.copy_(yh)
        graph.replay()
        torch.cuda.synchronize()
        for name, a, b in zip(("loss", "lse", "dX", "dW"), (loss, lse, dX, dW), want):
            assert torch.equal(a, b), name
    assert flce.flce_check_device_error(ws) == 0
