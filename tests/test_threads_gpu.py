"""Entry points called from a thread that has made no CUDA call of its own (as a
framework's autograd worker does): the library binds the device's primary context
before it encodes tensor maps, and the results equal those of the main thread."""
import threading

import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
from workloads import custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _buffers(N, D, V):
    return dict(loss=torch.empty(1, device=DEV), lse=torch.empty(N, device=DEV),
                dX=torch.empty(N, D, dtype=torch.bfloat16, device=DEV), dW=torch.empty(D, V, device=DEV),
                ws=torch.empty(flce.flce_workspace_size(N, D, V, 2), dtype=torch.uint8, device=DEV))


def _step(X, W, y, g, b, stream):
    st_f = flce.flce_forward(X, W, y, b["loss"], b["lse"], b["ws"], stream=stream, raise_on_error=False)
    st_b = flce.flce_backward(X, W, y, b["lse"], g, b["dX"], b["dW"], b["ws"], stream=stream,
                              raise_on_error=False)
    return st_f, st_b


def test_first_call_on_a_fresh_thread(gpu_lib):
    wl = custom("thread", 640, 256, 3000, seed=51, ignore_frac=0.05)
    X, W, y = make_inputs(wl)
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    g = torch.ones(1, device=DEV)
    stream = torch.cuda.current_stream(DEV).cuda_stream  # taken here, so the thread makes no torch CUDA call
    main = _buffers(wl.N, wl.D, wl.V)
    assert _step(Xd, Wd, yd, g, main, stream) == (0, 0)
    torch.cuda.synchronize()

    other = _buffers(wl.N, wl.D, wl.V)
    torch.cuda.synchronize()
    result = {}

    def work():
        result["status"] = _step(Xd, Wd, yd, g, other, stream)
        result["detail"] = flce.flce_last_error_detail()

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert result["status"] == (0, 0), result["detail"]
    torch.cuda.synchronize()
    for k in ("loss", "lse", "dX", "dW"):
        assert torch.equal(main[k], other[k]), k


def test_two_threads_on_two_streams(gpu_lib):
    """Two threads, each with its own stream and workspace, run forward + backward at the
    same time; each result equals the one-thread result bit for bit."""
    wl = custom("thread2", 768, 256, 4104, seed=52, ignore_frac=0.1, label_smoothing=0.1)
    X, W, y = make_inputs(wl)
    X2, _, y2 = make_inputs(wl, seed=53)
    Wd = W.to(DEV)
    g = torch.ones(1, device=DEV)
    inputs = [(X.to(DEV), y.to(DEV)), (X2.to(DEV), y2.to(DEV))]
    want = []
    for Xd, yd in inputs:
        b = _buffers(wl.N, wl.D, wl.V)
        assert _step(Xd, Wd, yd, g, b, torch.cuda.current_stream(DEV).cuda_stream) == (0, 0)
        torch.cuda.synchronize()
        want.append(b)
    streams = [torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)]
    got = [_buffers(wl.N, wl.D, wl.V) for _ in inputs]
    torch.cuda.synchronize()
    status = [None, None]

    def work(i):
        for _ in range(3):
            status[i] = _step(inputs[i][0], Wd, inputs[i][1], g, got[i], streams[i].cuda_stream)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert status == [(0, 0), (0, 0)]
    for i in range(2):
        assert flce.flce_check_device_error(got[i]["ws"]) == 0
        for k in ("loss", "lse", "dX", "dW"):
            assert torch.equal(got[i][k], want[i][k]), (i, k)
