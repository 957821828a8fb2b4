"""Which memory the entry points accept: device memory of the current device, from the
default caching allocator or from PyTorch's expandable segments (virtual-memory
mappings); host memory is refused before anything is launched. Host buffers used here are
pinned, so that even a call that slipped through would only read host memory over the
link, never fault."""
import os
import subprocess
import sys

import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
from workloads import custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _problem():
    wl = custom("memkind", 384, 128, 1024, seed=61, ignore_frac=0.1)
    X, W, y = make_inputs(wl)
    return wl, X, W, y


def _device_buffers(N, D, V):
    return dict(loss=torch.empty(1, device=DEV), lse=torch.empty(N, device=DEV),
                dX=torch.empty(N, D, dtype=torch.bfloat16, device=DEV), dW=torch.empty(D, V, device=DEV),
                g=torch.ones(1, device=DEV),
                ws=torch.empty(flce.flce_workspace_size(N, D, V, 2), dtype=torch.uint8, device=DEV))


@pytest.mark.parametrize("which", ["X", "W", "targets", "workspace", "loss", "lse"])
def test_forward_refuses_host_memory(gpu_lib, which):
    wl, X, W, y = _problem()
    b = _device_buffers(wl.N, wl.D, wl.V)
    args = dict(X=X.to(DEV), W=W.to(DEV), targets=y.to(DEV), workspace=b["ws"], loss=b["loss"], lse=b["lse"])
    args[which] = args[which].cpu().pin_memory()
    torch.cuda.synchronize()
    before = flce.flce_kernel_launches()
    st = flce.flce_forward(args["X"], args["W"], args["targets"], args["loss"], args["lse"], args["workspace"],
                           raise_on_error=False)
    assert st == 1, flce.flce_status_string(st)  # FLCE_ERR_INVALID_ARG
    assert flce.flce_kernel_launches() == before
    assert flce.flce_last_error_detail() == f"{which}: is host memory, not device memory"


@pytest.mark.parametrize("which", ["dX", "dW", "g", "lse"])
def test_backward_refuses_host_memory(gpu_lib, which):
    wl, X, W, y = _problem()
    b = _device_buffers(wl.N, wl.D, wl.V)
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    assert flce.flce_forward(Xd, Wd, yd, b["loss"], b["lse"], b["ws"]) == 0
    b[which] = b[which].cpu().pin_memory()
    torch.cuda.synchronize()
    before = flce.flce_kernel_launches()
    st = flce.flce_backward(Xd, Wd, yd, b["lse"], b["g"], b["dX"], b["dW"], b["ws"], raise_on_error=False)
    assert st == 1, flce.flce_status_string(st)
    assert flce.flce_kernel_launches() == before
    name = "grad_out" if which == "g" else which
    assert flce.flce_last_error_detail() == f"{name}: is host memory, not device memory"


def test_option_arrays_refuse_host_memory(gpu_lib):
    wl, X, W, y = _problem()
    b = _device_buffers(wl.N, wl.D, wl.V)
    bias = torch.zeros(wl.V).pin_memory()
    before = flce.flce_kernel_launches()
    st = flce.flce_forward_ex(X.to(DEV), W.to(DEV), y.to(DEV), b["loss"], b["lse"], b["ws"],
                              options=flce.make_options(bias=bias), raise_on_error=False)
    assert st == 1
    assert flce.flce_kernel_launches() == before
    assert flce.flce_last_error_detail() == "options.bias: is host memory, not device memory"


_CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import linear_cross_entropy_tcgen05_gb300 as flce
from workloads import custom, make_inputs
dev = torch.device("cuda:0")
wl = custom("memkind", 384, 128, 1024, seed=61, ignore_frac=0.1)
X, W, y = make_inputs(wl)
Xd, Wd, yd = X.to(dev), W.to(dev), y.to(dev)
N, D, V = wl.N, wl.D, wl.V
loss, lse = torch.empty(1, device=dev), torch.empty(N, device=dev)
dX, dW = torch.empty(N, D, dtype=torch.bfloat16, device=dev), torch.empty(D, V, device=dev)
ws = torch.empty(flce.flce_workspace_size(N, D, V, 2), dtype=torch.uint8, device=dev)
flce.flce_forward(Xd, Wd, yd, loss, lse, ws)
flce.flce_backward(Xd, Wd, yd, lse, torch.ones(1, device=dev), dX, dW, ws)
assert flce.flce_check_device_error(ws) == 0
torch.save({"loss": loss.cpu(), "lse": lse.cpu(), "dX": dX.cpu(), "dW": dW.cpu()}, sys.argv[2])
"""


def test_expandable_segments_are_device_memory(gpu_lib, tmp_path):
    """Tensors from PyTorch's expandable segments (virtual-memory mappings) are accepted,
    and the results equal those from the default allocator bit for bit."""
    out = {}
    for conf in ("expandable_segments:False", "expandable_segments:True"):
        path = str(tmp_path / (conf.replace(":", "_") + ".pt"))
        env = dict(os.environ, PYTORCH_CUDA_ALLOC_CONF=conf)
        r = subprocess.run([sys.executable, "-c", _CHILD, ROOT, path], env=env, capture_output=True, text=True,
                           timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        out[conf] = torch.load(path)
    a, b = out.values()
    for k in a:
        assert torch.equal(a[k], b[k]), k
