"""Host-side checks of the C ABI: the library loads, exports every declared entry
point, sizes its workspace, and refuses bad arguments before launching anything.

No test here launches a kernel: the argument checks run before the device check.
"""
import ctypes
import json
import os
import re
import shutil
import subprocess

import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
from linear_cross_entropy_tcgen05_gb300 import build as flce_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(flce.library_path()):
        flce_build.build()
    return flce.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(flce_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    fns = declared_functions()
    for name in ("flce_forward", "flce_backward", "flce_workspace_size", "flce_check_device_error",
                 "flce_status_string", "flce_version"):
        assert name in fns
    assert set(fns) == set(flce.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", flce.library_path()], capture_output=True, text=True).stdout
        exported = set(re.findall(r"\bT\s+(flce_\w+)", out))
        assert set(declared_functions()) <= exported


def test_version_and_status_strings(lib):
    assert flce.flce_version() == 300
    for code, name in flce.STATUS.items():
        assert flce.flce_status_string(code).startswith(name)
    assert "unknown" in flce.flce_status_string(99)


def test_workspace_sizes(lib):
    # forward: header + 3 partial arrays [S,N] + target logits + block sums; S = min(64, V/256 tiles)
    ws = flce.flce_workspace_size(256, 128, 1024, False)
    assert ws >= 3 * 4 * 256 * 4 + 256 * 4
    assert flce.flce_workspace_size(0, 128, 1024, False) == 0
    assert flce.flce_workspace_size(16, -1, 1024, True) == 0
    # backward at the headline shape: a bf16 band of Vc < V columns plus the fp32 dX accumulator
    N, D, V = 65536, 4096, 128256
    wb = flce.flce_workspace_size(N, D, V, True)
    logits_bf16 = flce.logits_bytes(N, V, 2)
    assert wb < logits_bf16 / 8, "the backward workspace must stay under an eighth of an N x V bf16 buffer"
    assert wb >= N * D * 4  # holds the fp32 dX accumulator
    # every band is narrower than the vocabulary once V exceeds one 256-column tile
    for (n, d, v) in [(256, 128, 1024), (4096, 2048, 32000), (8192, 4096, 128256), (16384, 2304, 256000)]:
        band = flce.flce_workspace_size(n, d, v, True) - n * d * 4 - n * 16 - 256
        assert band < n * v * 2
        # the forward on the valid rows only: its own workspace plus the row list and the
        # gathered rows of X; every backward workspace has that room
        f, fc = flce.flce_workspace_size(n, d, v, "forward"), flce.flce_workspace_size(n, d, v, "forward_valid_rows")
        assert fc >= f + n * d * 2 + 2 * n * 4
        assert flce.flce_workspace_size(n, d, v, "backward") >= fc
        assert flce.flce_workspace_size(n, d, v, "both") >= fc


def test_logit_bottleneck_arithmetic():
    """The page's sizes: 65,536 x 128,256 logits are ~8.4 B values, 16.8 GB bf16, 33.6 GB fp32."""
    g = json.load(open(os.path.join(GOLDEN, "logit_bottleneck.json")))
    n = g["N"] * g["V"]
    assert round(n / 1e9, 1) == g["elements_billions"]
    assert round(flce.logits_bytes(g["N"], g["V"], 2) / 1e9, 1) == g["bf16_GB"]
    assert round(flce.logits_bytes(g["N"], g["V"], 4) / 1e9, 1) == g["fp32_GB"]


class _Fake:
    """A stand-in address with a chosen alignment; never dereferenced (checks fail first)."""

    def __init__(self, addr):
        self.addr = addr


def _fwd(lib, X=0x10000, W=0x20000, y=0x30000, N=256, D=128, V=1024, eps=0.0, s=0.0, red=0, loss=0x40000,
         lse=0x50000, ws=0x60000, wsb=None):
    wsb = flce.flce_workspace_size(256, 128, 1024, False) if wsb is None else wsb
    return lib.flce_forward(X, W, y, N, D, V, -100, eps, s, red, loss, lse, ws, wsb, None)


def _bwd(lib, red=0, D=128, V=1024, grad=0x70000, wsb=None, X=0x10000):
    wsb = flce.flce_workspace_size(256, D, V, True) if wsb is None else wsb
    return lib.flce_backward(X, 0x20000, 0x30000, 0x50000, 256, D, V, -100, 0.0, 0.0, red, grad, 0x80000,
                             0x90000, 0x60000, wsb, None)


def test_forward_argument_checks(lib):
    assert _fwd(lib, X=None) == 1
    assert _fwd(lib, N=0) == 1
    assert _fwd(lib, eps=1.0) == 1
    assert _fwd(lib, eps=-0.1) == 1
    assert _fwd(lib, eps=float("nan")) == 1
    assert _fwd(lib, s=-1.0) == 1
    assert _fwd(lib, s=float("inf")) == 1
    assert _fwd(lib, red=3) == 1
    assert _fwd(lib, loss=None) == 1
    assert _fwd(lib, D=130) == 2      # D % 8
    assert _fwd(lib, V=1001) == 2     # V % 8
    assert _fwd(lib, X=0x10008) == 2  # 16-byte alignment
    assert _fwd(lib, y=0x30002) == 2
    assert _fwd(lib, N=1 << 31) == 9
    assert _fwd(lib, wsb=16) == 4


def test_backward_argument_checks(lib):
    assert _bwd(lib, red=2) == 5      # reduction 'none' with a gradient is refused
    assert _bwd(lib, grad=None) == 1
    assert _bwd(lib, V=1004) == 2
    assert _bwd(lib, X=0x10004) == 2
    assert _bwd(lib, wsb=1024) == 4


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the refusal on a machine without a GB300")
def test_refuses_without_a_supported_device(lib):
    assert _fwd(lib) == 3
    assert _bwd(lib) == 3
    assert lib.flce_selftest_wait_timeout(0x60000, 4096, None) == 3
    assert lib.flce_selftest_wait_timeout(None, 4096, None) == 1
    assert lib.flce_selftest_wait_timeout(0x60000, 16, None) == 4
    assert flce.flce_backward_band_width(65536, 4096, 128256) == 0   # depends on the device


def test_options_struct_matches_the_header():
    """Field order and offsets of flce_options as declared in flce.h (the ctypes mirror)."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct flce_options \{(.*?)\} flce_options;", text, flags=re.S).group(1)
    names = re.findall(r"(\w+);", body)
    assert names == [f[0] for f in flce.FlceOptions._fields_]
    assert flce.make_options(weight_layout="vd").weight_layout == 1
    assert flce.make_options().weight_layout == 0


def test_python_wrapper_checks_the_weight_layout_shape():
    X = torch.zeros(4, 8, dtype=torch.bfloat16)
    Wvd = torch.zeros(16, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match=r"W \[D,V\]"):
        flce.linear_cross_entropy(X, Wvd, y)                       # [V, D] passed as [D, V]
    with pytest.raises(ValueError, match="CUDA"):
        flce.linear_cross_entropy(X, Wvd, y, weight_layout="vd")  # shapes fine, CPU tensors refused


def test_python_wrapper_names_the_input_dtype():
    """The library cannot see an element type: the wrappers refuse f16 tensors unless the
    options say f16, and bf16 ones if they do (checked before any library call)."""
    X16 = torch.zeros(4, 8, dtype=torch.float16)
    W16 = torch.zeros(8, 16, dtype=torch.float16)
    y = torch.zeros(4, dtype=torch.int32)
    out = torch.zeros(4)
    with pytest.raises(TypeError, match="input_dtype"):
        flce.flce_forward(X16, W16, y, out, out, out)
    with pytest.raises(TypeError, match="input_dtype"):
        flce.flce_forward_ex(X16, W16, y, out, out, out, options=flce.make_options())
    with pytest.raises(TypeError, match="input_dtype"):
        flce.flce_backward_ex(X16.bfloat16(), W16, y, out, out, out, out, out,
                              options=flce.make_options(input_dtype="f16"))
    assert flce.make_options(input_dtype=torch.float16).input_dtype == 1
    with pytest.raises(TypeError, match="both"):
        flce.linear_cross_entropy(X16, W16.bfloat16(), y)
    with pytest.raises(ValueError, match="CUDA"):
        flce.linear_cross_entropy(X16, W16, y)                     # f16 accepted, CPU tensors refused


def test_python_wrapper_validates_dtypes():
    X = torch.zeros(4, 8, dtype=torch.float32)
    W = torch.zeros(8, 16, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(TypeError):
        flce.linear_cross_entropy(X, W, y)
    with pytest.raises(ValueError):
        flce.linear_cross_entropy(X.bfloat16(), W, y)  # CPU tensors are refused, never computed on the host


def _opts(**kw):
    return flce.make_options(**kw)


def _fwd_ex(lib, opts, V=1024):
    return lib.flce_forward_ex(0x10000, 0x20000, 0x30000, 256, 128, V, -100, 0.0, 0.0, 0, ctypes.byref(opts),
                               0x40000, 0x50000, 0x60000, flce.flce_workspace_size(256, 128, V, 0), None)


def _bwd_ex(lib, opts, V=1024):
    return lib.flce_backward_ex(0x10000, 0x20000, 0x30000, 0x50000, 256, 128, V, -100, 0.0, 0.0, 0,
                                ctypes.byref(opts), 0x70000, 0x80000, 0x90000, 0x60000,
                                flce.flce_workspace_size(256, 128, V, 1), None)


def test_option_checks(lib):
    assert _fwd_ex(lib, _opts(softcap=-1.0)) == 1
    assert _fwd_ex(lib, _opts(softcap=float("inf"))) == 1
    assert _fwd_ex(lib, _opts(v_total=2048)) == 1          # forward shards go through flce_shard_stats
    assert _fwd_ex(lib, _opts(v_offset=8)) == 1
    assert _fwd_ex(lib, _opts(bias=0x1002)) == 2            # misaligned
    assert _bwd_ex(lib, _opts(dbias=0xA0000)) == 1          # dbias needs a bias
    assert _bwd_ex(lib, _opts(v_offset=1000, v_total=1500)) == 1  # shard beyond the vocabulary
    assert _bwd_ex(lib, _opts(bias=0xA0000, v_offset=0, v_total=4096)) == 1  # shards take no bias
    assert _bwd_ex(lib, _opts(dX_f32=0xA0008)) == 2         # fp32 dX needs 16-byte alignment
    assert _fwd_ex(lib, _opts(weight_layout=2)) == 1        # not a flce_weight_layout
    assert _bwd_ex(lib, _opts(weight_layout=-1)) == 1
    assert _fwd_ex(lib, _opts(input_dtype=2)) == 1          # not a flce_input_dtype
    assert _bwd_ex(lib, flce.FlceOptions(accumulate_grads=2)) == 1  # not 0 or 1
    for bad in (_opts(softcap=2.0), _opts(row_band=64), _opts(weight_layout=3)):  # storage options only
        assert lib.flce_shard_stats_ex(0x10000, 0x20000, 0x30000, 256, 128, 1024, 0, -100, ctypes.byref(bad),
                                       0x40000, 0x60000, 1 << 20, None) == 1
    assert lib.flce_combine_shards(0x10000, 0, 0x30000, 256, 1024, -100, 0.0, 0.0, 0, 0x40000, 0x50000,
                                   0x60000, 1 << 20, None) == 1   # K >= 1
    assert lib.flce_shard_stats(0x10000, 0x20000, 0x30000, 256, 128, 1024, -8, -100, 0x40000, 0x60000,
                                1 << 20, None) == 1         # negative offset


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the refusal on a machine without a GB300")
def test_extended_entry_points_refuse_without_a_device(lib):
    assert _fwd_ex(lib, _opts(softcap=30.0)) == 3
    assert _bwd_ex(lib, _opts(v_offset=0, v_total=2048)) == 3


def test_fused_workspace_is_the_larger_of_the_two():
    for (n, d, v) in [(256, 128, 1024), (4096, 2048, 32000), (16, 8, 65536)]:
        f = flce.flce_workspace_size(n, d, v, 0)
        b = flce.flce_workspace_size(n, d, v, 1)
        assert flce.flce_workspace_size(n, d, v, 2) == max(f, b)


def test_loss_module_checks_its_arguments():
    with pytest.raises(ValueError, match="reduction"):
        flce.FusedLinearCrossEntropyLoss(reduction="avg")
    crit = flce.FusedLinearCrossEntropyLoss(return_predicted_tokens=True)
    weight = torch.zeros(16, 8, dtype=torch.bfloat16)     # [V, D]
    hidden = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        crit(weight, hidden, torch.zeros(4, dtype=torch.int64))   # shapes fine, CPU tensors refused
    with pytest.raises(ValueError, match=r"W \[V,D\]"):
        crit(weight.t().contiguous(), hidden, torch.zeros(4, dtype=torch.int64))


def test_header_compiles_as_c_and_links(lib, tmp_path):
    """include/flce.h is plain C: a C99 client builds with -Wall -Wextra -pedantic, links
    against libflce.so and gets answers that need no device."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "flce_c_client")
    libdir = os.path.dirname(flce.library_path())
    src = os.path.join(ROOT, "tests", "c", "flce_c_client.c")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        src, "-L", libdir, "-lflce", "-Wl,-rpath," + libdir, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    version, ws, status = out[0].split()
    assert int(version) == flce.flce_version()
    assert int(ws) == flce.flce_workspace_size(256, 128, 1024, True)
    assert int(status) == 1                    # FLCE_ERR_INVALID_ARG
    assert out[1].startswith("FLCE_ERR_F16_RANGE")
