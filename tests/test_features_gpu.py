"""GPU parity of the extended options against the fp64 oracle: logit softcap, bias
(and its gradient), per-class weights, argmax metrics, the fused forward+backward
call, fp32 dX, and vocabulary-parallel shards combined on one GPU."""
import numpy as np
import pytest
import torch

import linear_cross_entropy_tcgen05_gb300 as flce
import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, TOL_LOSS_REL, TOL_LSE_ABS, rel_fro
from workloads import IGNORE_INDEX, custom, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(wl, seed_extra=0):
    X, W, y = make_inputs(wl)
    g = np.random.default_rng(wl.seed + 1000 + seed_extra)
    bias = torch.tensor(g.standard_normal(wl.V) * 0.5, dtype=torch.float32)
    cw = torch.tensor(g.uniform(0.25, 2.0, size=wl.V), dtype=torch.float32)
    return X, W, y, bias, cw


def _ws(N, D, V, which):
    return torch.empty(flce.flce_workspace_size(N, D, V, which), dtype=torch.uint8, device=DEV)


def _check_argmax(pred_gpu, X, W, y, bias, softcap, valid, acc_gpu):
    """Compare what is unique (the argmax where the top two logits are well separated);
    elsewhere check that the GPU's choice is a maximum within rounding."""
    _, u = oracle.ext_logits(oracle.widen(X), oracle.widen(W), bias, softcap)
    ref = oracle.argmax_first(u)
    top = u[np.arange(u.shape[0]), ref]
    picked = u[np.arange(u.shape[0]), pred_gpu]
    clear = ref == pred_gpu
    assert np.all(clear | (top - picked <= 1e-4 * np.maximum(1.0, np.abs(top)))), "argmax far from the maximum"
    assert np.mean(clear) > 0.99
    n_valid = valid.sum()
    want = ((pred_gpu == y) & valid).sum() / n_valid
    assert abs(acc_gpu - want) < 1e-6


FEATURE_CASES = [
    ("softcap", dict(softcap=30.0), "mean"),
    ("softcap_small", dict(softcap=2.0), "sum"),
    ("bias", dict(bias=True), "mean"),
    ("weights", dict(cw=True), "mean"),
    ("weights_sum", dict(cw=True), "sum"),
    ("everything", dict(softcap=5.0, bias=True, cw=True), "mean"),
]


@pytest.mark.parametrize("name,feat,red", FEATURE_CASES, ids=[c[0] for c in FEATURE_CASES])
def test_extended_options_forward_backward(gpu_lib, name, feat, red):
    wl = custom("feat_" + name, 777, 200, 4104, seed=31, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-3,
                reduction=red)
    X, W, y, bias, cw = _inputs(wl)
    softcap = feat.get("softcap", 0.0)
    b = bias if feat.get("bias") else None
    w = cw if feat.get("cw") else None
    N, D, V = wl.N, wl.D, wl.V
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    bd = b.to(DEV) if b is not None else None
    wd = w.to(DEV) if w is not None else None
    pred = torch.full((N,), -7, dtype=torch.int32, device=DEV)
    acc = torch.full((1,), -1.0, device=DEV)
    dbias = torch.full((V,), float("nan"), device=DEV) if b is not None else None
    opts = flce.make_options(softcap=softcap, bias=bd, class_weight=wd, predicted=pred, accuracy=acc, dbias=dbias)
    ws = _ws(N, D, V, 2)
    loss = torch.empty(1, device=DEV)
    lse = torch.empty(N, device=DEV)
    g = torch.ones(1, device=DEV)
    dX = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = torch.empty(D, V, device=DEV)
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, red)
    flce.flce_forward_ex(Xd, Wd, yd, loss, lse, ws, *common, options=opts)
    assert flce.flce_check_device_error(ws) == 0
    flce.flce_backward_ex(Xd, Wd, yd, lse, g, dX, dW, ws, *common, options=opts)
    assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    ref_loss, ref_lse, ref_dX, ref_dW, ref_db = oracle.forward_backward_ext(
        X, W, y, *common, softcap=softcap, bias=b, class_weight=w)
    valid = y.numpy() != IGNORE_INDEX
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert np.max(np.abs(lse.cpu().double().numpy()[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(dX.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(dW.cpu().numpy(), ref_dW) <= TOL_DW_REL
    if b is not None:
        assert rel_fro(dbias.cpu().numpy(), ref_db) <= TOL_DW_REL
    _check_argmax(pred.cpu().numpy(), X, W, y.numpy(), b, softcap, valid, acc.item())


def test_accuracy_without_predicted_output(gpu_lib):
    wl = custom("acc_only", 512, 128, 2048, seed=32, ignore_frac=0.2)
    X, W, y, _, _ = _inputs(wl)
    # make half of the targets the argmax so that accuracy is far from 0
    z = X.float() @ W.float()
    am = z.argmax(1).int()
    y2 = torch.where(torch.arange(wl.N) % 2 == 0, am, y)
    y2[y == IGNORE_INDEX] = IGNORE_INDEX
    acc = torch.zeros(1, device=DEV)
    ws = _ws(wl.N, wl.D, wl.V, 0)
    loss, lse = torch.empty(1, device=DEV), torch.empty(wl.N, device=DEV)
    flce.flce_forward_ex(X.to(DEV), W.to(DEV), y2.to(DEV), loss, lse, ws,
                         options=flce.make_options(accuracy=acc))
    torch.cuda.synchronize()
    _, _, _, ref_acc = oracle.forward_ext(X, W, y2)
    assert abs(acc.item() - ref_acc) <= 2.0 / wl.N  # at most a near-tie row or two


def test_fused_call_equals_separate_calls(gpu_lib):
    wl = custom("fused", 1000, 136, 5000, seed=33, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-4)
    X, W, y, _, _ = _inputs(wl)
    N, D, V = wl.N, wl.D, wl.V
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean")
    g = torch.tensor([1.5], device=DEV)
    out = []
    for fused in (True, False):
        ws = _ws(N, D, V, 2)
        loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
        dX = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
        dW = torch.empty(D, V, device=DEV)
        if fused:
            flce.flce_forward_backward(Xd, Wd, yd, g, loss, lse, dX, dW, ws, *common)
        else:
            flce.flce_forward(Xd, Wd, yd, loss, lse, ws, *common)
            flce.flce_backward(Xd, Wd, yd, lse, g, dX, dW, ws, *common)
        assert flce.flce_check_device_error(ws) == 0
        out.append([t.cpu() for t in (loss, lse, dX, dW)])
    for a, b in zip(*out):
        assert torch.equal(a, b)
    ref_loss, _, ref_dX, ref_dW = oracle.forward_backward(X, W, y, *common, grad_out=1.5)
    assert abs(out[0][0].item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert rel_fro(out[0][2].float().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(out[0][3].numpy(), ref_dW) <= TOL_DW_REL


def test_fp32_dx_output(gpu_lib):
    wl = custom("dx32", 600, 256, 3000, seed=34, ignore_frac=0.1)
    X, W, y, _, _ = _inputs(wl)
    N, D, V = wl.N, wl.D, wl.V
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    ws = _ws(N, D, V, 2)
    loss, lse, g = torch.empty(1, device=DEV), torch.empty(N, device=DEV), torch.ones(1, device=DEV)
    flce.flce_forward(Xd, Wd, yd, loss, lse, ws)
    dX16 = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = torch.empty(D, V, device=DEV)
    flce.flce_backward(Xd, Wd, yd, lse, g, dX16, dW, ws)
    dX32 = torch.full((N, D), float("nan"), device=DEV)
    dW2 = torch.empty(D, V, device=DEV)
    flce.flce_backward_ex(Xd, Wd, yd, lse, g, None, dW2, ws, options=flce.make_options(dX_f32=dX32))
    torch.cuda.synchronize()
    assert torch.equal(dX32.bfloat16(), dX16), "bf16 dX is the fp32 accumulator rounded once"
    # the bf16-dX call compacts the valid rows, so dW sums its rows in another order
    assert rel_fro(dW.cpu().numpy(), dW2.cpu().numpy()) <= 1e-5
    _, _, ref_dX, _ = oracle.forward_backward(X, W, y)
    assert rel_fro(dX32.cpu().numpy(), ref_dX) <= 5e-3


@pytest.mark.parametrize("cuts", [[0, 1000, 2048, 4104], [0, 264, 4104], [0, 4104], [0, 8, 4096, 4104]])
@pytest.mark.parametrize("eps,s,red", [(0.0, 0.0, "mean"), (0.1, 1e-3, "sum")])
def test_vocabulary_shards_match_the_whole(gpu_lib, cuts, eps, s, red):
    wl = custom("shards", 700, 136, 4104, seed=35, ignore_frac=0.1)
    X, W, y, _, _ = _inputs(wl)
    N, D, V = wl.N, wl.D, wl.V
    Xd, yd = X.to(DEV), y.to(DEV)
    K = len(cuts) - 1
    stats = torch.empty(K, 4, N, device=DEV)
    shards = []
    for k, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        Wk = W[:, a:b].contiguous().to(DEV)
        shards.append((a, Wk))
        ws = _ws(N, D, b - a, 0)
        flce.flce_shard_stats(Xd, Wk, yd, a, stats[k], ws)
        assert flce.flce_check_device_error(ws) == 0
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    wsc = _ws(N, 8, 8, 0)
    flce.flce_combine_shards(stats, yd, V, loss, lse, wsc, label_smoothing=eps, zloss_scale=s, reduction=red)
    assert flce.flce_check_device_error(wsc) == 0
    # backward per shard with the combined lse: partial fp32 dX summed over shards, dW blocks side by side
    g = torch.ones(1, device=DEV)
    dX = torch.zeros(N, D, device=DEV)
    dW = torch.empty(D, V, device=DEV)
    for a, Wk in shards:
        Vk = Wk.shape[1]
        part = torch.empty(N, D, device=DEV)
        dWk = torch.empty(D, Vk, device=DEV)
        ws = _ws(N, D, Vk, 1)
        flce.flce_backward_ex(Xd, Wk, yd, lse, g, None, dWk, ws, label_smoothing=eps, zloss_scale=s,
                              reduction=red, options=flce.make_options(dX_f32=part, v_offset=a, v_total=V))
        assert flce.flce_check_device_error(ws) == 0
        dX += part
        dW[:, a:a + Vk] = dWk
    torch.cuda.synchronize()
    ref_loss, ref_lse, ref_dX, ref_dW = oracle.forward_backward(X, W, y, label_smoothing=eps, zloss_scale=s,
                                                                reduction=red)
    valid = y.numpy() != IGNORE_INDEX
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert np.max(np.abs(lse.cpu().double().numpy()[valid] - ref_lse[valid])) <= TOL_LSE_ABS
    assert rel_fro(dX.cpu().numpy(), ref_dX) <= 5e-3
    assert rel_fro(dW.cpu().numpy(), ref_dW) <= TOL_DW_REL
    # the shard statistics themselves
    for k, (a, Wk) in enumerate(shards):
        lse_k, sz_k, zy_k, own_k = oracle.shard_stats(X, W[:, a:a + Wk.shape[1]], y, a)
        st = stats[k].cpu().double().numpy()
        assert np.max(np.abs(st[0] - lse_k)) <= TOL_LSE_ABS
        assert np.array_equal(st[3], own_k)
        assert np.max(np.abs(st[2] - zy_k)) <= 1e-3


@pytest.mark.parametrize("row_band,opts", [(300, {}), (256, {"cw": True}), (512, {"bias": True, "softcap": 8.0}),
                                            (999, {})])  # the last band holds one row
def test_row_band_backward_matches_the_oracle(gpu_lib, row_band, opts):
    """Micro-batching along N: the backward in bands of rows, with a workspace sized for one band."""
    wl = custom("bands", 1000, 136, 4104, seed=36, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-3)
    X, W, y, bias, cw = _inputs(wl)
    N, D, V = wl.N, wl.D, wl.V
    b = bias if opts.get("bias") else None
    w = cw if opts.get("cw") else None
    softcap = opts.get("softcap", 0.0)
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    bd = b.to(DEV) if b is not None else None
    wd = w.to(DEV) if w is not None else None
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean")
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    flce.flce_forward_ex(Xd, Wd, yd, loss, lse, _ws(N, D, V, 0), *common,
                         options=flce.make_options(softcap=softcap, bias=bd, class_weight=wd))
    ws = _ws(row_band, D, V, 1)  # one band's workspace
    assert ws.numel() < flce.flce_workspace_size(N, D, V, 1)
    dX = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = torch.empty(D, V, device=DEV)
    dbias = torch.empty(V, device=DEV) if b is not None else None
    g = torch.ones(1, device=DEV)
    flce.flce_backward_ex(Xd, Wd, yd, lse, g, dX, dW, ws, *common,
                          options=flce.make_options(softcap=softcap, bias=bd, class_weight=wd, dbias=dbias,
                                                    row_band=row_band))
    assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    _, _, ref_dX, ref_dW, ref_db = oracle.forward_backward_ext(X, W, y, *common, softcap=softcap, bias=b,
                                                               class_weight=w)
    assert rel_fro(dX.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(dW.cpu().numpy(), ref_dW) <= TOL_DW_REL
    if b is not None:
        assert rel_fro(dbias.cpu().numpy(), ref_db) <= TOL_DW_REL
    # too small a workspace for the band is refused
    small = _ws(row_band // 2, D, V, 1)
    st = flce.flce_backward_ex(Xd, Wd, yd, lse, g, dX, dW, small, *common, raise_on_error=False,
                               options=flce.make_options(row_band=row_band))
    assert st == 4


@pytest.mark.parametrize("N", [1000, 2500], ids=["forward_all_rows", "forward_valid_rows"])
def test_launch_counter_matches_the_band_schedule(gpu_lib, N):
    """flce_kernel_launches counts what the bench reports as gpu_launches; one forward
    plus backward launches what the band schedule predicts (from 2048 rows the forward
    adds its valid-row list and gather)."""
    import bench
    wl = custom("count", N, 136, 4104, seed=37, ignore_frac=0.1)
    X, W, y, _, _ = _inputs(wl)
    N, D, V = wl.N, wl.D, wl.V
    Xd, Wd, yd = X.to(DEV), W.to(DEV), y.to(DEV)
    ws = _ws(N, D, V, 2)
    loss, lse, g = torch.empty(1, device=DEV), torch.empty(N, device=DEV), torch.ones(1, device=DEV)
    dX = torch.empty(N, D, dtype=torch.bfloat16, device=DEV)
    dW = torch.empty(D, V, device=DEV)
    before = flce.flce_kernel_launches()
    flce.flce_forward(Xd, Wd, yd, loss, lse, ws)
    flce.flce_backward(Xd, Wd, yd, lse, g, dX, dW, ws)
    counted = flce.flce_kernel_launches() - before
    assert flce.flce_check_device_error(ws) == 0
    vc = flce.flce_backward_band_width(N, D, V)
    assert vc > 0 and vc % 512 == 0
    assert ws.numel() >= flce.flce_workspace_size(N, D, V, "forward_valid_rows")
    expected, bands, _ = bench.kernel_launches_per_step(N, D, V, "mean", vc, compact_fwd=N >= 2048)
    assert bands == -(-V // vc) and counted == expected


def test_gradient_accumulation_over_micro_batches(gpu_lib):
    """accumulate_grads: dW and dbias of two micro-batches (sum reduction) added into the
    same buffers equal one call over the whole batch (to fp32 rounding) and the oracle."""
    wl = custom("accum", 1000, 136, 4104, seed=38, ignore_frac=0.1, label_smoothing=0.1, zloss_scale=1e-3,
                reduction="sum")
    X, W, y, bias, _ = _inputs(wl)
    N, D, V = wl.N, wl.D, wl.V
    Wd, bd = W.to(DEV), bias.to(DEV)
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "sum")
    g = torch.ones(1, device=DEV)
    dW = torch.full((D, V), float("nan"), device=DEV)
    db = torch.full((V,), float("nan"), device=DEV)
    for i, (a, b) in enumerate([(0, 600), (600, N)]):
        Xm, ym = X[a:b].contiguous().to(DEV), y[a:b].contiguous().to(DEV)
        n = b - a
        ws = _ws(n, D, V, 2)
        loss, lse = torch.empty(1, device=DEV), torch.empty(n, device=DEV)
        dX = torch.empty(n, D, dtype=torch.bfloat16, device=DEV)
        opts = flce.make_options(bias=bd, dbias=db, accumulate_grads=i > 0)
        flce.flce_forward_backward(Xm, Wd, ym, g, loss, lse, dX, dW, ws, *common, options=opts)
        assert flce.flce_check_device_error(ws) == 0
    torch.cuda.synchronize()
    _, _, _, ref_dW, ref_db = oracle.forward_backward_ext(X, W, y, *common, bias=bias)
    assert rel_fro(dW.cpu().numpy(), ref_dW) <= TOL_DW_REL
    assert rel_fro(db.cpu().numpy(), ref_db) <= TOL_DW_REL
    # one call over the whole batch gives the same dW up to the order of fp32 additions
    ws = _ws(N, D, V, 2)
    dW1 = torch.empty(D, V, device=DEV)
    db1 = torch.empty(V, device=DEV)
    loss, lse = torch.empty(1, device=DEV), torch.empty(N, device=DEV)
    flce.flce_forward_backward(X.to(DEV), Wd, y.to(DEV), g, loss, lse, torch.empty(N, D, dtype=torch.bfloat16,
                               device=DEV), dW1, ws, *common, options=flce.make_options(bias=bd, dbias=db1))
    torch.cuda.synchronize()
    assert rel_fro(dW.cpu().numpy(), dW1.cpu().numpy()) <= 1e-5
    assert rel_fro(db.cpu().numpy(), db1.cpu().numpy()) <= 1e-5


def test_loss_module_with_metrics(gpu_lib):
    """FusedLinearCrossEntropyLoss on an nn.Linear-layout weight: the loss and gradients of
    the autograd path, plus token accuracy and predictions from the same forward."""
    wl = custom("module", 640, 136, 3000, seed=39, ignore_frac=0.1, label_smoothing=0.05, zloss_scale=1e-4)
    X, W, y, bias, cw = _inputs(wl)
    head = W.t().contiguous().to(DEV).requires_grad_()   # [V, D]
    hidden = X.to(DEV).requires_grad_()
    b = bias.to(DEV).requires_grad_()
    crit = flce.FusedLinearCrossEntropyLoss(ce_weight=cw.to(DEV), ignore_index=wl.ignore_index,
                                            lse_square_scale=wl.zloss_scale, label_smoothing=wl.label_smoothing,
                                            softcap=12.0, return_token_accuracy=True, return_predicted_tokens=True)
    loss, acc, pred = crit(head, hidden, y.to(DEV).long(), b)
    loss.backward()
    torch.cuda.synchronize()
    ref_loss, _, ref_dX, ref_dW, ref_db = oracle.forward_backward_ext(
        X, W, y, wl.ignore_index, wl.label_smoothing, wl.zloss_scale, "mean", softcap=12.0, bias=bias,
        class_weight=cw)
    assert abs(loss.item() - ref_loss) <= TOL_LOSS_REL * abs(ref_loss)
    assert rel_fro(hidden.grad.float().cpu().numpy(), ref_dX) <= TOL_DX_REL
    assert rel_fro(head.grad.float().cpu().numpy().T, ref_dW) <= 1e-2   # returned in bf16
    assert rel_fro(b.grad.float().cpu().numpy(), ref_db) <= TOL_DW_REL
    valid = y.numpy() != IGNORE_INDEX
    _check_argmax(pred.cpu().numpy(), X, W, y.numpy(), bias, 12.0, valid, acc.item())
