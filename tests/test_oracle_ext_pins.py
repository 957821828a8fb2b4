"""Pins for the oracle's extended options (logit softcap, vocabulary bias, per-class
weights, argmax metrics, vocabulary-parallel combination)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import IGNORE_INDEX

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _problem(N, D, V, seed, ignored=(), scale=2.0):
    r = np.random.default_rng(seed)
    X = r.standard_normal((N, D))
    W = r.standard_normal((D, V)) * scale / math.sqrt(D)
    y = r.integers(0, V, size=N)
    for i in ignored:
        y[i] = IGNORE_INDEX
    b = r.standard_normal(V) * 0.5
    w = r.uniform(0.2, 2.0, size=V)
    return X, W, y, b, w


def test_defaults_reduce_to_the_base_definitions():
    X, W, y, _, _ = _problem(9, 7, 40, 1, ignored=(3,))
    for red in ("mean", "sum"):
        a = oracle.forward_backward_ext(X, W, y, label_smoothing=0.1, zloss_scale=1e-3, reduction=red)
        b = oracle.forward_backward(X, W, y, label_smoothing=0.1, zloss_scale=1e-3, reduction=red)
        assert abs(a[0] - b[0]) < 1e-13
        for i in (1, 2, 3):
            assert np.max(np.abs(a[i] - b[i])) < 1e-14
        assert a[4] is None


@pytest.mark.parametrize("eps", [0.0, 0.1])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("softcap", [0.0, 3.0])
@pytest.mark.parametrize("use_bias,use_w", [(False, True), (True, False), (True, True)])
def test_matches_torch_weighted_smoothed_capped(eps, reduction, softcap, use_bias, use_w):
    """torch fp64: F.cross_entropy(softcap(X W + b), y, weight, label_smoothing) and autograd."""
    N, D, V = 21, 12, 97
    X, W, y, b, w = _problem(N, D, V, 2, ignored=(0, 5))
    bias = b if use_bias else None
    cw = w if use_w else None
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    z = Xt @ Wt + (bt if use_bias else 0.0)
    u = softcap * torch.tanh(z / softcap) if softcap else z
    ref = F.cross_entropy(u, torch.tensor(y), weight=torch.tensor(w) if use_w else None,
                          ignore_index=IGNORE_INDEX, label_smoothing=eps, reduction=reduction)
    loss, lse, pred, acc = oracle.forward_ext(X, W, y, label_smoothing=eps, reduction=reduction,
                                              softcap=softcap, bias=bias, class_weight=cw)
    assert np.max(np.abs(np.asarray(loss) - ref.detach().numpy())) < 1e-12
    assert np.max(np.abs(lse - torch.logsumexp(u, 1).detach().numpy())) < 1e-12
    if reduction == "none":
        return
    ref.backward()
    _, _, dX, dW, db = oracle.forward_backward_ext(X, W, y, label_smoothing=eps, reduction=reduction,
                                                   softcap=softcap, bias=bias, class_weight=cw)
    assert np.max(np.abs(dX - Xt.grad.numpy())) < 1e-12
    assert np.max(np.abs(dW - Wt.grad.numpy())) < 1e-12
    if use_bias:
        assert np.max(np.abs(db - bt.grad.numpy())) < 1e-12


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_central_finite_differences_all_options(reduction):
    """N=4, D=8, V=16, every option on (softcap, bias, weights, smoothing, z-loss), h=1e-6."""
    N, D, V = 4, 8, 16
    X, W, y, b, w = _problem(N, D, V, 3, ignored=(1,))
    kw = dict(label_smoothing=0.1, zloss_scale=0.05, reduction=reduction, softcap=2.5, class_weight=w)
    go = 1.3
    _, _, dX, dW, db = oracle.forward_backward_ext(X, W, y, grad_out=go, bias=b, **kw)

    def f(Xv, Wv, bv):
        return go * oracle.forward_ext(Xv, Wv, y, bias=bv, **kw)[0]

    h = 1e-6
    for arr, grad, which in ((X, dX, 0), (W, dW, 1), (b, db, 2)):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            ap, am = arr.copy(), arr.copy()
            ap[idx] += h
            am[idx] -= h
            args_p = [X, W, b]
            args_m = [X, W, b]
            args_p[which] = ap
            args_m[which] = am
            fd[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
        assert np.linalg.norm(grad - fd) <= 1e-6 * np.linalg.norm(fd)


def test_uniform_class_weights_cancel_in_the_mean():
    X, W, y, _, _ = _problem(10, 6, 30, 4, ignored=(2,))
    a = oracle.forward_ext(X, W, y, label_smoothing=0.1, class_weight=np.full(30, 2.5))[0]
    b = oracle.forward_ext(X, W, y, label_smoothing=0.1)[0]
    assert abs(a - b) < 1e-13


def test_softcap_closed_form_constant_logits():
    """W = 0 and a constant bias: every capped logit is c tanh(b/c), so lse = that + ln V."""
    N, D, V, c, bval = 3, 4, 50, 4.0, 7.0
    X = np.random.default_rng(5).standard_normal((N, D))
    _, lse, _, _ = oracle.forward_ext(X, np.zeros((D, V)), np.zeros(N, int), softcap=c, bias=np.full(V, bval))
    assert np.max(np.abs(lse - (c * math.tanh(bval / c) + math.log(V)))) < 1e-13


def test_argmax_first_index_on_ties_and_accuracy():
    """Duplicated columns give exact ties; torch.argmax convention: the first index wins."""
    r = np.random.default_rng(6)
    N, D, V = 30, 5, 12
    X = r.standard_normal((N, D))
    W = r.standard_normal((D, V))
    W[:, 7] = W[:, 2]  # column 7 ties column 2 exactly
    W[:, 9] = W[:, 4]
    y = r.integers(0, V, size=N)
    y[[3, 4]] = IGNORE_INDEX
    _, _, pred, acc = oracle.forward_ext(X, W, y)
    z = X @ W
    for i in range(N):
        best, arg = -np.inf, -1
        for j in range(V):
            if z[i, j] > best:
                best, arg = z[i, j], j
        assert pred[i] == arg and arg not in (7, 9)
    valid = y != IGNORE_INDEX
    want = sum(1 for i in range(N) if valid[i] and pred[i] == y[i]) / valid.sum()
    assert acc == want


@pytest.mark.parametrize("cuts", [[0, 40, 100], [0, 8, 64, 65, 100], [0, 100]])
@pytest.mark.parametrize("eps,s", [(0.0, 0.0), (0.1, 1e-3)])
def test_vocabulary_shards_combine_to_the_full_loss(cuts, eps, s):
    """log-sum-exp over a partition of the vocabulary is the log-sum-exp of the parts."""
    X, W, y, _, _ = _problem(17, 9, 100, 7, ignored=(4,))
    stats = [oracle.shard_stats(X, W[:, a:b], y, a) for a, b in zip(cuts[:-1], cuts[1:])]
    loss, lse = oracle.combine_shard_stats(stats, 100, y, label_smoothing=eps, zloss_scale=s)
    ref_loss, ref_lse = oracle.forward(X, W, y, label_smoothing=eps, zloss_scale=s)
    assert np.max(np.abs(lse - ref_lse)) < 1e-12
    assert abs(loss - ref_loss) < 1e-12
    # every valid row's target is owned by exactly one shard
    owned = sum(st[3] for st in stats)
    assert np.all(owned[y != IGNORE_INDEX] == 1.0) and np.all(owned[y == IGNORE_INDEX] == 0.0)


def test_targets_on_shard_boundaries():
    """Targets in the first and the last column of every shard: each is owned by exactly one
    shard, whose target logit it carries, and the combination equals the full loss."""
    cuts = [0, 8, 64, 65, 100]
    X, W, _, _, _ = _problem(12, 9, 100, 8)
    y = np.array([a for a in cuts[:-1]] + [b - 1 for b in cuts[1:]] + [IGNORE_INDEX, 50, 99, 0])
    stats = [oracle.shard_stats(X, W[:, a:b], y, a) for a, b in zip(cuts[:-1], cuts[1:])]
    z = X @ W
    for k, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        mine = (y >= a) & (y < b)
        assert np.all(stats[k][3] == mine.astype(float))
        assert np.max(np.abs(stats[k][2][mine] - z[mine, y[mine]])) < 1e-13
        assert np.all(stats[k][2][~mine] == 0.0)
    loss, lse = oracle.combine_shard_stats(stats, 100, y, label_smoothing=0.1)
    ref_loss, ref_lse = oracle.forward(X, W, y, label_smoothing=0.1)
    assert abs(loss - ref_loss) < 1e-12 and np.max(np.abs(lse - ref_lse)) < 1e-12
