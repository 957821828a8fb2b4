"""Pins for the fp64 oracle: results fixed by the pages and by mathematics.

None of these re-types the oracle's own formulas. Each one checks the oracle
against something independent of it: a closed form, an invariant, pure-Python
brute force, torch's fp64 cross-entropy, central finite differences, or the
label-smoothing rule printed in the TransformerEngine review thread.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import IGNORE_INDEX, WORKLOADS, custom, make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_problem(N, D, V, seed, ignored=(), scale=1.0):
    r = np.random.default_rng(seed)
    X = r.standard_normal((N, D))
    W = r.standard_normal((D, V)) * scale / math.sqrt(D)
    y = r.integers(0, V, size=N)
    for i in ignored:
        y[i] = IGNORE_INDEX
    return X, W, y


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("s", [0.0, 1e-4, 0.3])
@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_w_zero_closed_form(eps, s, reduction):
    """W = 0: every logit is 0, so lse = ln V and each valid row's loss is ln V + s (ln V)^2."""
    N, D, V = 6, 5, 37
    X, _, y = _rand_problem(N, D, V, 1, ignored=(2,))
    W = np.zeros((D, V))
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, label_smoothing=eps, zloss_scale=s,
                                                reduction=reduction, grad_out=1.0)
    lnV = math.log(V)
    assert np.all(np.abs(lse - lnV) < 1e-14)
    n_valid = N - 1
    per_row = lnV + s * lnV * lnV
    want = per_row if reduction == "mean" else n_valid * per_row
    assert abs(loss - want) < 1e-12 * max(1.0, abs(want))
    assert np.all(dX == 0.0)
    # dW_kj = g * sum_i X_ik * (p_ij (1 + 2 s lnV) - (1-eps) [j == y_i] - eps/V), p = 1/V
    g = 1.0 / n_valid if reduction == "mean" else 1.0
    want_dW = np.zeros((D, V))
    for i in range(N):
        if y[i] == IGNORE_INDEX:
            continue
        for j in range(V):
            dz = (1.0 / V) * (1 + 2 * s * lnV) - eps / V - ((1 - eps) if j == y[i] else 0.0)
            for k in range(D):
                want_dW[k, j] += g * X[i, k] * dz
    assert np.max(np.abs(dW - want_dW)) < 1e-13


def test_w_zero_loss_is_ln_v_for_any_smoothing():
    X, _, y = _rand_problem(4, 3, 1000, 2)
    for eps in (0.0, 0.05, 0.5, 0.9):
        loss, _ = oracle.forward(X, np.zeros((3, 1000)), y, label_smoothing=eps)
        assert abs(loss - math.log(1000)) < 1e-13


# --------------------------------------------------------------------------- invariants

@pytest.mark.parametrize("s", [0.0, 1e-4, 0.2])
@pytest.mark.parametrize("eps", [0.0, 0.1])
def test_gradient_rows_sum_to_zlosss_term(s, eps):
    """sum_j dZ_ij = g * 2 s lse_i: zero without z-loss (softmax and targets both sum to 1)."""
    N, D, V = 7, 6, 50
    X, W, y = _rand_problem(N, D, V, 3, ignored=(4,), scale=3.0)
    Xf = oracle.widen(X)
    z = oracle.logits(Xf, W)
    lse = oracle.logsumexp_rows(z)
    g = 0.37
    dz = oracle.grad_logits(z, lse, y, V, IGNORE_INDEX, eps, s, g)
    want = np.where(y != IGNORE_INDEX, g * 2 * s * lse, 0.0)
    assert np.max(np.abs(dz.sum(axis=1) - want)) < 1e-14
    # the same through dW: each row of dW sums to g * sum_i X_ik * 2 s lse_i
    _, _, _, dW = oracle.forward_backward(X, W, y, label_smoothing=eps, zloss_scale=s,
                                          reduction="sum", grad_out=g)
    want_rows = (Xf * want[:, None]).sum(axis=0)
    assert np.max(np.abs(dW.sum(axis=1) - want_rows)) < 1e-12


def test_ignored_rows_contribute_nothing():
    N, D, V = 8, 6, 40
    X, W, y = _rand_problem(N, D, V, 4, ignored=(1, 5))
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, reduction="sum")
    ell = oracle.forward(X, W, y, reduction="none")[0]
    assert ell[1] == 0.0 and ell[5] == 0.0 and np.all(ell[[0, 2, 3, 4, 6, 7]] > 0)
    assert np.all(dX[1] == 0.0) and np.all(dX[5] == 0.0)
    # changing the hidden state of an ignored row changes neither the loss nor dW
    X2 = X.copy()
    X2[1] += 10.0
    X2[5] *= -3.0
    loss2, _, _, dW2 = oracle.forward_backward(X2, W, y, reduction="sum")
    assert loss2 == loss
    assert np.max(np.abs(dW2 - dW)) < 1e-15


def test_mean_with_no_valid_rows_is_zero():
    N, D, V = 3, 4, 9
    X, W, y = _rand_problem(N, D, V, 5, ignored=(0, 1, 2))
    loss, _, dX, dW = oracle.forward_backward(X, W, y, reduction="mean")
    assert loss == 0.0 and np.all(dX == 0) and np.all(dW == 0)


def test_out_of_range_target_poisons_its_row():
    N, D, V = 4, 3, 10
    X, W, y = _rand_problem(N, D, V, 6)
    y[2] = V  # neither a class nor the ignore index
    ell = oracle.forward(X, W, y, reduction="none")[0]
    assert np.isnan(ell[2]) and np.all(np.isfinite(ell[[0, 1, 3]]))
    _, _, dX, _ = oracle.forward_backward(X, W, y, reduction="sum")
    assert np.all(np.isnan(dX[2])) and np.all(np.isfinite(dX[[0, 1, 3]]))


def test_shift_invariance_without_zloss():
    """Adding the same vector to every column of W shifts row i's logits by a constant."""
    N, D, V = 5, 4, 30
    X, W, y = _rand_problem(N, D, V, 7)
    u = np.random.default_rng(8).standard_normal(D)
    for eps in (0.0, 0.1):
        l0, _ = oracle.forward(X, W, y, label_smoothing=eps)
        l1, _ = oracle.forward(X, W + u[:, None], y, label_smoothing=eps)
        assert abs(l0 - l1) < 1e-12


# --------------------------------------------------------------------------- brute force

def _brute_force_loss(X, W, y, eps, s, reduction):
    """Pure-Python cross-entropy H(q, softmax(z)) without any max-shift."""
    N, D = len(X), len(X[0])
    V = len(W[0])
    total, n_valid, rows = 0.0, 0, []
    for i in range(N):
        if y[i] == IGNORE_INDEX:
            rows.append(0.0)
            continue
        z = [sum(X[i][k] * W[k][j] for k in range(D)) for j in range(V)]
        e = [math.exp(v) for v in z]
        den = sum(e)
        q = [(1 - eps) * (1.0 if j == y[i] else 0.0) + eps / V for j in range(V)]
        ell = -sum(q[j] * math.log(e[j] / den) for j in range(V)) + s * math.log(den) ** 2
        rows.append(ell)
        total += ell
        n_valid += 1
    if reduction == "none":
        return rows
    return total / n_valid if reduction == "mean" else total


@pytest.mark.parametrize("eps,s,reduction", [(0.0, 0.0, "mean"), (0.1, 0.0, "sum"),
                                             (0.0, 0.01, "mean"), (0.2, 0.05, "none")])
def test_brute_force_tiny(eps, s, reduction):
    N, D, V = 5, 4, 7
    X, W, y = _rand_problem(N, D, V, 9, ignored=(3,), scale=2.0)
    want = _brute_force_loss(X.tolist(), W.tolist(), y.tolist(), eps, s, reduction)
    got, _ = oracle.forward(X, W, y, label_smoothing=eps, zloss_scale=s, reduction=reduction)
    assert np.max(np.abs(np.asarray(got) - np.asarray(want))) < 1e-13


# --------------------------------------------------------------------------- torch fp64

@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("s", [0.0, 1e-3])
def test_matches_torch_cross_entropy_fp64(eps, reduction, s):
    """torch's F.cross_entropy (fp64, CPU) plus the z-loss term, with autograd gradients."""
    N, D, V = 33, 24, 301
    X, W, y = _rand_problem(N, D, V, 10, ignored=(0, 7, 30), scale=4.0)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    yt = torch.tensor(y)
    z = Xt @ Wt
    ce = F.cross_entropy(z, yt, ignore_index=IGNORE_INDEX, label_smoothing=eps, reduction=reduction)
    valid = (yt != IGNORE_INDEX).double()
    zl = s * torch.logsumexp(z, dim=1) ** 2 * valid
    if reduction == "mean":
        ref = ce + zl.sum() / valid.sum()
    elif reduction == "sum":
        ref = ce + zl.sum()
    else:
        ref = ce + zl
    got, _ = oracle.forward(X, W, y, label_smoothing=eps, zloss_scale=s, reduction=reduction)
    assert np.max(np.abs(np.asarray(got) - ref.detach().numpy())) < 1e-12
    if reduction == "none":
        return
    ref.backward()
    _, _, dX, dW = oracle.forward_backward(X, W, y, label_smoothing=eps, zloss_scale=s,
                                           reduction=reduction)
    assert np.max(np.abs(dX - Xt.grad.numpy())) < 1e-13
    assert np.max(np.abs(dW - Wt.grad.numpy())) < 1e-13
    dX2, dW2 = oracle.backward(X, W, y, label_smoothing=eps, zloss_scale=s, reduction=reduction)
    assert np.max(np.abs(dX2 - Xt.grad.numpy())) < 1e-13
    assert np.max(np.abs(dW2 - Wt.grad.numpy())) < 1e-13


# --------------------------------------------------------------------------- finite differences

@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("s", [0.0, 1e-4, 0.5])
@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_central_finite_differences(eps, s, reduction):
    """N=4, D=8, V=16 with one ignored row; h = 1e-6 in fp64."""
    N, D, V = 4, 8, 16
    X, W, y = _rand_problem(N, D, V, 11, ignored=(2,), scale=2.0)
    grad_out = 1.7
    _, _, dX, dW = oracle.forward_backward(X, W, y, label_smoothing=eps, zloss_scale=s,
                                           reduction=reduction, grad_out=grad_out)

    def f(Xv, Wv):
        return grad_out * oracle.forward(Xv, Wv, y, label_smoothing=eps, zloss_scale=s,
                                         reduction=reduction)[0]

    h = 1e-6
    fdX = np.zeros_like(X)
    for i in range(N):
        for k in range(D):
            Xp, Xm = X.copy(), X.copy()
            Xp[i, k] += h
            Xm[i, k] -= h
            fdX[i, k] = (f(Xp, W) - f(Xm, W)) / (2 * h)
    fdW = np.zeros_like(W)
    for k in range(D):
        for j in range(V):
            Wp, Wm = W.copy(), W.copy()
            Wp[k, j] += h
            Wm[k, j] -= h
            fdW[k, j] = (f(X, Wp) - f(X, Wm)) / (2 * h)
    assert np.linalg.norm(dX - fdX) <= 1e-6 * np.linalg.norm(fdX)
    assert np.linalg.norm(dW - fdW) <= 1e-6 * np.linalg.norm(fdW)
    assert np.all(dX[2] == 0.0)


# --------------------------------------------------------------------------- TE smoothing rule

@pytest.mark.parametrize("alpha,V", [(0.1, 16), (0.1, 1024), (0.3, 7)])
def test_transformer_engine_smoothing_rule(alpha, V):
    """TE/Megatron: smoothing = alpha V/(V-1); the target keeps 1 - alpha, others alpha/(V-1).

    The TransformerEngine review thread prints the conversion
    ``smoothing = label_smoothing * vocab_size / (vocab_size - 1)`` and a backward
    that subtracts (1 - smoothing) at the target and smoothing/V everywhere. With
    eps = smoothing the oracle must equal the cross-entropy against the target
    distribution q (1 - alpha on the label, alpha/(V-1) elsewhere), and its logit
    gradient must be softmax - q.
    """
    N, D = 6, 5
    X, W, y = _rand_problem(N, D, V, 12, scale=2.0)
    smoothing = alpha * V / (V - 1)
    z = X @ W
    p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
    q = np.full((N, V), alpha / (V - 1))
    q[np.arange(N), y] = 1 - alpha
    want_rows = -(q * np.log(p)).sum(axis=1)
    got_rows, lse = oracle.forward(X, W, y, label_smoothing=smoothing, reduction="none")
    assert np.max(np.abs(got_rows - want_rows)) < 1e-12
    dz = oracle.grad_logits(oracle.logits(X, W), lse, y, V, IGNORE_INDEX, smoothing, 0.0, 1.0)
    assert np.max(np.abs(dz - (p - q))) < 1e-14


# --------------------------------------------------------------------------- batched helpers

@pytest.mark.parametrize("eps,s", [(0.0, 0.0), (0.1, 1e-2)])
def test_batched_helpers_match_dense(eps, s):
    wl = custom("helpers", 300, 40, 257, seed=13, ignore_frac=0.1)
    X, W, y = make_inputs(wl)
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, label_smoothing=eps, zloss_scale=s,
                                                reduction="mean")
    lse_b, ell_b = oracle.full_row_stats(X, W, y, label_smoothing=eps, zloss_scale=s, row_batch=64)
    assert np.max(np.abs(lse_b - lse)) < 1e-12
    n_valid = int((y != IGNORE_INDEX).sum())
    assert abs(ell_b.sum() / n_valid - loss) < 1e-12
    g = 1.0 / n_valid
    rows = np.array([0, 5, 77, 299])
    dXr = oracle.grad_x_rows(X, W, y, rows, lse[rows], g, label_smoothing=eps, zloss_scale=s)
    assert np.max(np.abs(dXr - dX[rows])) < 1e-14
    cols = np.array([0, 3, int(y[9]) if y[9] >= 0 else 1, 256])
    dWc = oracle.grad_w_cols(X, W, y, cols, lse, g, label_smoothing=eps, zloss_scale=s,
                             row_batch=100)
    assert np.max(np.abs(dWc - dW[:, cols])) < 1e-14


# --------------------------------------------------------------------------- statistical sanity

def test_tiny_workload_loss_near_ln_v_plus_half():
    """With X~N(0,1) and W~N(0,1/D) the logits are ~N(0,1), so the mean loss is ~ ln V + 1/2."""
    wl = WORKLOADS["tiny"]
    X, W, y = make_inputs(wl)
    loss, lse = oracle.forward(X, W, y)
    assert abs(loss - (math.log(wl.V) + 0.5)) < 0.15
    assert np.all(np.isfinite(lse))
