"""GPU parity of the [V, D] weight layout (the weight of an nn.Linear(D, V) head)
against the fp64 oracle, which works on W [D, V]: the same inputs go in transposed, and
dW comes back in the [V, D] layout."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, TOL_LOSS_REL, TOL_LSE_ABS, rel_fro
from workloads import IGNORE_INDEX, custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _ws(N, D, V, which):
    return torch.empty(flce.flce_workspace_size(N, D, V, which), dtype=torch.uint8, device=DEV)


def _run(X, W_dev, y, V, common, options, grad_out=1.0):
    N, D = X.shape
    Xd, yd = X.to(DEV), y.to(DEV)
    ws = _ws(N, D, V, 2)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    g = torch.tensor([grad_out], device=DEV)
    dX = torch.full((N, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    dW = torch.full(tuple(W_dev.shape), float("nan"), device=DEV)
    flce.flce_forward_ex(Xd, W_dev, yd, loss, lse, ws, *common, options=options)
    assert flce.flce_check_device_error(ws) == 0
    flce.flce_backward_ex(Xd, W_dev, yd, lse, g, dX, dW, ws, *common, options=options)
    assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    return loss.item(), lse.cpu().double().numpy(), dX.float().cpu().numpy(), dW.cpu().numpy()


# (N, D, V): one vocabulary band; two bands with an odd tile count in the last one; D a
# multiple of 256 with several dW column tiles.
SHAPES = [(300, 128, 1000), (1000, 136, 4104), (2048, 1024, 8200)]


@pytest.mark.parametrize("N,D,V", SHAPES, ids=[f"{n}x{d}x{v}" for n, d, v in SHAPES])
@pytest.mark.parametrize("eps,s,red", [(0.0, 0.0, "mean"), (0.1, 1e-3, "sum")])
def test_vd_layout_matches_the_oracle(gpu_lib, N, D, V, eps, s, red):
    wl = custom("vd", N, D, V, seed=41, ignore_frac=0.1, label_smoothing=eps, zloss_scale=s, reduction=red)
    X, W, y = make_inputs(wl)
    common = (wl.ignore_index, eps, s, red)
    Wvd = W.t().contiguous().to(DEV)
    loss, lse, dX, dWvd = _run(X, Wvd, y, V, common, flce.make_options(weight_layout="vd"), grad_out=0.75)
    ref_loss, ref_lse, ref_dX, ref_dW = oracle.forward_backward(X, W, y, *common, grad_out=0.75)
    valid = y.numpy() != IGNORE_INDEX
    assert abs(loss - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert np.max(np.abs(lse[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(dX, ref_dX) <= TOL_DX_REL
    assert dWvd.shape == (V, D)
    assert rel_fro(dWvd.T, ref_dW) <= TOL_DW_REL
    # the [D, V] path on the same inputs agrees to rounding
    loss2, lse2, dX2, dW2 = _run(X, W.to(DEV), y, V, common, None, grad_out=0.75)
    assert abs(loss - loss2) <= 1e-6 * abs(loss2)
    assert np.max(np.abs(lse - lse2)) <= 1e-5
    assert rel_fro(dWvd.T, dW2) <= 1e-3


def test_vd_layout_with_options_and_row_bands(gpu_lib):
    wl = custom("vd_opts", 1000, 136, 4104, seed=42, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y = make_inputs(wl)
    g = np.random.default_rng(4242)
    bias = torch.tensor(g.standard_normal(wl.V) * 0.5, dtype=torch.float32)
    cw = torch.tensor(g.uniform(0.25, 2.0, size=wl.V), dtype=torch.float32)
    N, D, V = wl.N, wl.D, wl.V
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean")
    Xd, yd, Wvd = X.to(DEV), y.to(DEV), W.t().contiguous().to(DEV)
    bd, wd = bias.to(DEV), cw.to(DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    flce.flce_forward_ex(Xd, Wvd, yd, loss, lse, _ws(N, D, V, 0), *common,
                         options=flce.make_options(softcap=6.0, bias=bd, class_weight=wd, weight_layout="vd"))
    band = 384
    ws = _ws(band, D, V, 1)
    dX = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = torch.full((V, D), float("nan"), device=DEV)
    dbias = torch.empty(V, device=DEV)
    flce.flce_backward_ex(Xd, Wvd, yd, lse, torch.ones(1, device=DEV), dX, dW, ws, *common,
                          options=flce.make_options(softcap=6.0, bias=bd, class_weight=wd, dbias=dbias,
                                                    row_band=band, weight_layout="vd"))
    assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    ref_loss, ref_lse, ref_dX, ref_dW, ref_db = oracle.forward_backward_ext(X, W, y, *common, softcap=6.0,
                                                                            bias=bias, class_weight=cw)
    valid = y.numpy() != IGNORE_INDEX
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert np.max(np.abs(lse.cpu().double().numpy()[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(dX.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(dW.cpu().numpy().T, ref_dW) <= TOL_DW_REL
    assert rel_fro(dbias.cpu().numpy(), ref_db) <= TOL_DW_REL


def test_vd_layout_vocabulary_shard_backward(gpu_lib):
    """A [V, D] shard is a block of rows; its backward takes the combined lse."""
    wl = custom("vd_shard", 700, 136, 4104, seed=43, ignore_frac=0.1)
    X, W, y = make_inputs(wl)
    N, D, V = wl.N, wl.D, wl.V
    Xd, yd = X.to(DEV), y.to(DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    flce.flce_forward(Xd, W.to(DEV), yd, loss, lse, _ws(N, D, V, 0))
    g = torch.ones(1, device=DEV)
    dX = torch.zeros(N, D, device=DEV)
    dW = torch.empty(V, D, device=DEV)
    for a, b in [(0, 1544), (1544, 4104)]:
        Wk = W[:, a:b].t().contiguous().to(DEV)
        part = torch.empty(N, D, device=DEV)
        dWk = torch.empty(b - a, D, device=DEV)
        ws = _ws(N, D, b - a, 1)
        flce.flce_backward_ex(Xd, Wk, yd, lse, g, None, dWk, ws,
                              options=flce.make_options(dX_f32=part, v_offset=a, v_total=V, weight_layout="vd"))
        assert flce.flce_check_device_error(ws) == 0
        dX += part
        dW[a:b] = dWk
    torch.cuda.synchronize()
    _, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y)
    assert rel_fro(dX.cpu().numpy(), ref_dX) <= 5e-3
    assert rel_fro(dW.cpu().numpy().T, ref_dW) <= TOL_DW_REL


def test_vd_layout_through_autograd(gpu_lib):
    wl = custom("vd_autograd", 512, 256, 3000, seed=44, ignore_frac=0.05)
    X, W, y = make_inputs(wl)
    Xa = X.to(DEV).requires_grad_()
    Wa = W.t().contiguous().to(DEV).requires_grad_()  # nn.Linear(D, V).weight layout
    loss = flce.linear_cross_entropy(Xa, Wa, y.to(DEV), weight_layout="vd")
    loss.backward()
    torch.cuda.synchronize()
    ref_loss, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y)
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert Wa.grad.shape == (wl.V, wl.D)
    assert rel_fro(Xa.grad.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    # the autograd path returns dW in W's dtype (bf16): compare at bf16 resolution
    assert rel_fro(Wa.grad.float().cpu().numpy().T, ref_dW) <= 1e-2


def test_vd_f16_shards_end_to_end(gpu_lib):
    """Vocabulary shards of an f16 [V, D] weight: statistics, combination and backward."""
    from workloads import make_inputs as mk
    wl = custom("vd_f16_shard", 640, 136, 4104, seed=45, ignore_frac=0.1, label_smoothing=0.1)
    X, W, y = mk(wl, dtype=torch.float16)
    N, D, V = wl.N, wl.D, wl.V
    Xd, yd = X.to(DEV), y.to(DEV)
    cuts = [0, 1544, 4104]
    K = len(cuts) - 1
    stats = torch.empty(K, 4, N, device=DEV)
    opt = flce.make_options(weight_layout="vd", input_dtype="f16")
    shards = []
    for k, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        Wk = W[:, a:b].t().contiguous().to(DEV)
        shards.append((a, Wk))
        ws = _ws(N, D, b - a, 0)
        flce.flce_shard_stats(Xd, Wk, yd, a, stats[k], ws, options=opt)
        assert flce.flce_check_device_error(ws) == 0
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    wsc = _ws(N, 8, 8, 0)
    flce.flce_combine_shards(stats, yd, V, loss, lse, wsc, label_smoothing=0.1)
    assert flce.flce_check_device_error(wsc) == 0
    g = torch.ones(1, device=DEV)
    dX = torch.zeros(N, D, device=DEV)
    dW = torch.empty(V, D, device=DEV)
    for a, Wk in shards:
        Vk = Wk.shape[0]
        part = torch.empty(N, D, device=DEV)
        dWk = torch.empty(Vk, D, device=DEV)
        ws = _ws(N, D, Vk, 1)
        flce.flce_backward_ex(Xd, Wk, yd, lse, g, None, dWk, ws, label_smoothing=0.1,
                              options=flce.make_options(dX_f32=part, v_offset=a, v_total=V, weight_layout="vd",
                                                        input_dtype="f16"))
        assert flce.flce_check_device_error(ws) == 0
        dX += part
        dW[a:a + Vk] = dWk
    torch.cuda.synchronize()
    ref_loss, ref_lse, ref_dX, ref_dW = oracle.forward_backward(X, W, y, label_smoothing=0.1)
    valid = y.numpy() != IGNORE_INDEX
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert np.max(np.abs(lse.cpu().double().numpy()[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(dX.cpu().numpy(), ref_dX) <= 5e-3
    assert rel_fro(dW.cpu().numpy().T, ref_dW) <= TOL_DW_REL
