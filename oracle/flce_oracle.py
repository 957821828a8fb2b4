"""Plain, slow fp64 CPU oracle for fused linear cross-entropy (FLCE).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module. The CUDA library never does, and the two share no code: the oracle
takes its inputs as plain arrays from the seeded generators in ``workloads``.

It works on the same bf16-rounded (or f16-rounded) inputs as the GPU path, widened
exactly to float64, and computes everything in float64 with numpy. Matrix products use
numpy's ``@`` as a library step; there is no blocking or fusion beyond splitting
independent rows into batches to bound memory.

Sources (cited by page title and section):

[P1] "Cutting LLM Memory by 84%: A Deep Dive into Fused Kernels" (blog post).
[P3] NVIDIA TransformerEngine pull request #995, "Add efficient Cross-Entropy by
     cuda kernel ..." (the review thread on label smoothing in the backward kernel).
[P4] Liger-Kernel pull request #1291, "[CuteDSL] FLCE: 2-SM online-softmax fast
     path (Blackwell)", section "Summary" (feature list).

Notation: X [N,D], W [D,V], targets y [N]; z = X @ W; eps = label smoothing
(torch convention: the target keeps 1 - eps + eps/V of the mass, every other
class eps/V); s = z-loss scale ("lse_square_scale" in [P4]); valid(i) iff
y_i != ignore_index; g = grad_out (divided by the number of valid rows under
"mean").

Readings where the pages are silent or garbled (each is also listed in the
design notes):

* label smoothing: the only printed formula is [P3]'s
  ``smoothing = label_smoothing * vocab_size / (vocab_size - 1)``, after which the
  backward subtracts ``1 - smoothing`` at the target and ``smoothing / V``
  everywhere. That is the torch-convention loss below with eps = smoothing; the
  tests pin the identity.
* z-loss: [P4] only names it; we read it as ``s * lse_i^2`` per valid row, added
  to the row loss and reduced with it, whose gradient adds ``2 s lse_i p_ij``.
* mean: divides by the number of valid rows; with no valid row the loss and the
  gradients are 0.
* a target outside [0, V) that is not the ignore index has no defined loss: that
  row's loss and gradient are NaN.

Every function here has a pin in ``tests/test_oracle_pins.py`` or, for the
extended options and shards, ``tests/test_oracle_ext_pins.py`` (closed forms,
invariants, brute force, a torch fp64 library routine and central finite
differences); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "widen", "logits", "logsumexp_rows", "row_losses", "reduce_loss", "grad_scale",
    "grad_logits", "forward", "backward", "forward_backward", "full_row_stats",
    "grad_x_rows", "grad_w_cols", "REDUCTIONS", "ext_logits", "ext_row_losses", "ext_denominator",
    "ext_grad_u", "argmax_first", "forward_ext", "forward_backward_ext", "shard_stats", "combine_shard_stats",
]

REDUCTIONS = ("mean", "sum", "none")


def widen(a) -> np.ndarray:
    """Exact widening of a torch tensor (any dtype, e.g. bf16) or array to float64."""
    if hasattr(a, "detach"):
        import torch  # only for tensors handed in by the tests
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def _int_targets(y) -> np.ndarray:
    if hasattr(y, "detach"):
        y = y.detach().cpu().numpy()
    return np.asarray(y, dtype=np.int64)


def logits(X: np.ndarray, W: np.ndarray) -> np.ndarray:
    """z = X @ W, [N,V], in float64.

    [P1] "The Logit Bottleneck": the logit matrix is Y = X @ W with X [N x D] and
    W [D x V].
    """
    return X @ W


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    """lse_i = m_i + log sum_j exp(z_ij - m_i), with m_i = max_j z_ij.

    [P1] "Definition and Forward Pass": the numerically stable softmax subtracts
    the global maximum logit; the forward pass reduces to the target logit, the
    log-sum-exp and that maximum.
    """
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def _valid_and_bad(y: np.ndarray, V: int, ignore_index: int):
    valid = y != ignore_index
    bad = valid & ((y < 0) | (y >= V))
    return valid, bad


def row_losses(z: np.ndarray, lse: np.ndarray, y, V: int, ignore_index: int,
               label_smoothing: float, zloss_scale: float) -> np.ndarray:
    """Per-row loss l_i (0 for ignored rows, NaN for out-of-range targets).

    l_i = (1 - eps) (lse_i - z_{i,y_i}) + eps (lse_i - (1/V) sum_j z_ij) + s lse_i^2

    [P1] "Definition and Forward Pass": with a one-hot target the cross-entropy
    collapses to lse - z_y. The eps term is the same cross-entropy against the
    uniform distribution (the mean log-probability of [P3]'s forward kernel), the
    s term the z-loss of [P4]. [P1] "Setup and Target Logit Pre-computation": a
    row whose label is the ignore index has loss 0.
    """
    y = _int_targets(y)
    valid, bad = _valid_and_bad(y, V, ignore_index)
    safe_y = np.where(valid & ~bad, y, 0)
    z_y = z[np.arange(z.shape[0]), safe_y]
    mean_z = z.mean(axis=1)
    eps = float(label_smoothing)
    ell = (1.0 - eps) * (lse - z_y) + eps * (lse - mean_z) + float(zloss_scale) * lse * lse
    ell = np.where(valid, ell, 0.0)
    ell = np.where(bad, np.nan, ell)
    return ell


def reduce_loss(ell: np.ndarray, valid: np.ndarray, reduction: str):
    """Sum, mean over valid rows, or the per-row vector.

    [P1] "Fused Linear Cross-Entropy": in a batch the loss (and the W gradient)
    is reduced over rows with a sum or a mean. Mean divides by the number of
    valid rows; with none it is 0.
    """
    if reduction == "none":
        return ell.copy()
    total = float(ell.sum())
    if reduction == "sum":
        return total
    if reduction == "mean":
        n_valid = int(valid.sum())
        return total / n_valid if n_valid else 0.0
    raise ValueError(f"reduction must be one of {REDUCTIONS}")


def grad_scale(grad_out: float, n_valid: int, reduction: str) -> float:
    """g: the upstream gradient, divided by the number of valid rows under mean."""
    if reduction == "mean":
        return float(grad_out) / n_valid if n_valid else 0.0
    if reduction == "sum":
        return float(grad_out)
    raise ValueError("the backward pass needs reduction 'mean' or 'sum'")


def grad_logits(z: np.ndarray, lse: np.ndarray, y, V: int, ignore_index: int,
                label_smoothing: float, zloss_scale: float, g: float,
                cols: np.ndarray | None = None) -> np.ndarray:
    """dZ_ij = g [p_ij (1 + 2 s lse_i) - (1 - eps) delta_{j,y_i} - eps/V].

    p_ij = exp(z_ij - lse_i). [P1] "Cross-Entropy" (backward): the gradient of the
    loss with respect to the logits is the prediction minus the ground truth,
    softmax(z) - onehot(y). [P3] backward kernel review: with smoothing the target
    entry loses (1 - smoothing) and every entry loses smoothing / V. The z-loss
    term s lse^2 adds 2 s lse p. Ignored rows get 0; out-of-range targets NaN.

    ``cols`` names the vocabulary columns that the columns of ``z`` hold (default:
    all V in order), so that selected columns of dZ can be formed alone.
    """
    y = _int_targets(y)
    valid, bad = _valid_and_bad(y, V, ignore_index)
    eps = float(label_smoothing)
    cols = np.arange(V) if cols is None else np.asarray(cols)
    p = np.exp(z - lse[:, None])
    dz = p * (1.0 + 2.0 * float(zloss_scale) * lse)[:, None] - eps / V
    hit = (y[:, None] == cols[None, :]) & (valid & ~bad)[:, None]
    dz -= (1.0 - eps) * hit
    dz *= g
    dz[~valid] = 0.0
    dz[bad] = np.nan
    return dz


def forward(X, W, y, ignore_index: int = -100, label_smoothing: float = 0.0,
            zloss_scale: float = 0.0, reduction: str = "mean"):
    """Loss (scalar, or [N] for 'none') and lse [N] of softmax(X @ W)."""
    X, W = widen(X), widen(W)
    y = _int_targets(y)
    V = W.shape[1]
    z = logits(X, W)
    lse = logsumexp_rows(z)
    ell = row_losses(z, lse, y, V, ignore_index, label_smoothing, zloss_scale)
    valid, _ = _valid_and_bad(y, V, ignore_index)
    return reduce_loss(ell, valid, reduction), lse


def backward(X, W, y, ignore_index: int = -100, label_smoothing: float = 0.0,
             zloss_scale: float = 0.0, reduction: str = "mean", grad_out: float = 1.0):
    """(dX [N,D], dW [D,V]) of the reduced loss.

    [P1] "Matrix Multiplication" (backward): for Y = X @ W with upstream gradient
    dY, dX = dY @ W^T and dW = X^T @ dY. [P1] "Fused Linear Cross-Entropy": the
    FLCE gradient chains the logit gradient through the linear layer.
    """
    X, W = widen(X), widen(W)
    y = _int_targets(y)
    V = W.shape[1]
    valid, _ = _valid_and_bad(y, V, ignore_index)
    g = grad_scale(grad_out, int(valid.sum()), reduction)
    z = logits(X, W)
    lse = logsumexp_rows(z)
    dz = grad_logits(z, lse, y, V, ignore_index, label_smoothing, zloss_scale, g)
    return dz @ W.T, X.T @ dz


def forward_backward(X, W, y, ignore_index: int = -100, label_smoothing: float = 0.0,
                     zloss_scale: float = 0.0, reduction: str = "mean", grad_out: float = 1.0):
    """Loss, lse, dX, dW in one pass over the logits (same definitions as above)."""
    X, W = widen(X), widen(W)
    y = _int_targets(y)
    V = W.shape[1]
    valid, _ = _valid_and_bad(y, V, ignore_index)
    z = logits(X, W)
    lse = logsumexp_rows(z)
    ell = row_losses(z, lse, y, V, ignore_index, label_smoothing, zloss_scale)
    loss = reduce_loss(ell, valid, reduction)
    if reduction == "none":
        return loss, lse, None, None
    g = grad_scale(grad_out, int(valid.sum()), reduction)
    dz = grad_logits(z, lse, y, V, ignore_index, label_smoothing, zloss_scale, g)
    return loss, lse, dz @ W.T, X.T @ dz


# ---------------------------------------------------------------------------
# Large problems: the same definitions evaluated on row batches (rows are
# independent) or on selected rows / columns of the outputs.
# ---------------------------------------------------------------------------

def full_row_stats(X, W, y, ignore_index: int = -100, label_smoothing: float = 0.0,
                   zloss_scale: float = 0.0, row_batch: int = 256, W64: np.ndarray | None = None):
    """lse [N] and per-row loss [N] for every row, batching rows to bound memory.

    Same definitions as ``logsumexp_rows`` and ``row_losses``; rows are
    independent, so the batches change nothing but peak memory.
    """
    W64 = widen(W) if W64 is None else W64
    y = _int_targets(y)
    N, V = y.shape[0], W64.shape[1]
    lse = np.empty(N)
    ell = np.empty(N)
    for lo in range(0, N, row_batch):
        hi = min(N, lo + row_batch)
        z = logits(widen(X[lo:hi]), W64)
        lse[lo:hi] = logsumexp_rows(z)
        ell[lo:hi] = row_losses(z, lse[lo:hi], y[lo:hi], V, ignore_index,
                                label_smoothing, zloss_scale)
    return lse, ell


def grad_x_rows(X, W, y, rows, lse_rows: np.ndarray, g: float, ignore_index: int = -100,
                label_smoothing: float = 0.0, zloss_scale: float = 0.0,
                W64: np.ndarray | None = None) -> np.ndarray:
    """dX[rows, :] = dZ[rows, :] @ W^T, with dZ from ``grad_logits``."""
    W64 = widen(W) if W64 is None else W64
    y = _int_targets(y)
    rows = np.asarray(rows)
    z = logits(widen(X[rows]), W64)
    dz = grad_logits(z, lse_rows, y[rows], W64.shape[1], ignore_index, label_smoothing,
                     zloss_scale, g)
    return dz @ W64.T


def grad_w_cols(X, W, y, cols, lse: np.ndarray, g: float, ignore_index: int = -100,
                label_smoothing: float = 0.0, zloss_scale: float = 0.0,
                row_batch: int = 8192) -> np.ndarray:
    """dW[:, cols] = X^T @ dZ[:, cols] for selected vocabulary columns.

    dZ[i, j] needs only z_ij, lse_i and y_i (``grad_logits`` restricted to the
    selected columns, with the full-vocabulary lse of every row).
    """
    y = _int_targets(y)
    cols = np.asarray(cols)
    V = W.shape[1]
    Wc = widen(W[:, cols])
    N = y.shape[0]
    out = np.zeros((Wc.shape[0], cols.shape[0]))
    for lo in range(0, N, row_batch):
        hi = min(N, lo + row_batch)
        Xb = widen(X[lo:hi])
        dz = grad_logits(Xb @ Wc, lse[lo:hi], y[lo:hi], V, ignore_index, label_smoothing,
                         zloss_scale, g, cols=cols)
        out += Xb.T @ dz
    return out


# ---------------------------------------------------------------------------
# Extended options (Liger-Kernel PR #1291 "Summary" feature list): logit
# softcap, a vocabulary bias, per-class weights, argmax metrics, and the
# vocabulary-parallel split of the reduction. The pages name these features
# without defining them; the readings below are torch's conventions (the PR
# claims parity with torch) and are listed in the design notes.
# ---------------------------------------------------------------------------

def ext_logits(X: np.ndarray, W: np.ndarray, bias=None, softcap: float = 0.0):
    """(z, u): z = X @ W (+ bias broadcast over rows); u = softcap * tanh(z / softcap) if softcap > 0."""
    z = logits(X, W)
    if bias is not None:
        z = z + widen(bias)[None, :]
    if softcap and softcap > 0:
        u = float(softcap) * np.tanh(z / float(softcap))
    else:
        u = z
    return z, u


def ext_row_losses(u, lse, y, V, ignore_index, label_smoothing, zloss_scale, class_weight=None):
    """l_i = (1-eps) w_{y_i} (lse_i - u_{i,y_i}) + (eps/V) sum_j w_j (lse_i - u_ij) + s lse_i^2.

    torch's weighted, label-smoothed cross-entropy per row plus the z-loss; w = 1 gives
    ``row_losses``. Ignored rows 0, out-of-range targets NaN.
    """
    y = _int_targets(y)
    valid, bad = _valid_and_bad(y, V, ignore_index)
    w = np.ones(V) if class_weight is None else widen(class_weight)
    safe_y = np.where(valid & ~bad, y, 0)
    u_y = u[np.arange(u.shape[0]), safe_y]
    eps = float(label_smoothing)
    smooth = (lse * w.sum() - u @ w) / V
    ell = (1.0 - eps) * w[safe_y] * (lse - u_y) + eps * smooth + float(zloss_scale) * lse * lse
    ell = np.where(valid, ell, 0.0)
    return np.where(bad, np.nan, ell)


def ext_denominator(y, V, ignore_index, class_weight=None) -> float:
    """Mean denominator: the number of valid rows, or the sum of their target weights."""
    y = _int_targets(y)
    valid, bad = _valid_and_bad(y, V, ignore_index)
    ok = valid & ~bad
    if class_weight is None:
        return float(valid.sum())
    w = widen(class_weight)
    return float(w[y[ok]].sum())


def ext_grad_u(u, lse, y, V, ignore_index, label_smoothing, zloss_scale, g, class_weight=None):
    """dU_ij = g [p_ij ((1-eps) w_y + (eps/V) W + 2 s lse_i) - (eps/V) w_j - (1-eps) w_y delta_{j,y}].

    The gradient of ``ext_row_losses`` with respect to u (W = sum_j w_j); w = 1 gives
    ``grad_logits``.
    """
    y = _int_targets(y)
    valid, bad = _valid_and_bad(y, V, ignore_index)
    w = np.ones(V) if class_weight is None else widen(class_weight)
    eps = float(label_smoothing)
    ok = valid & ~bad
    safe_y = np.where(ok, y, 0)
    wy = w[safe_y]
    p = np.exp(u - lse[:, None])
    a = (1.0 - eps) * wy + eps / V * w.sum() + 2.0 * float(zloss_scale) * lse
    du = p * a[:, None] - (eps / V) * w[None, :]
    rows = np.nonzero(ok)[0]
    du[rows, y[rows]] -= (1.0 - eps) * wy[rows]
    du *= g
    du[~valid] = 0.0
    du[bad] = np.nan
    return du


def argmax_first(u: np.ndarray) -> np.ndarray:
    """Index of each row's largest value, the smallest such index on ties (torch.argmax)."""
    return np.argmax(u, axis=1)


def forward_ext(X, W, y, ignore_index=-100, label_smoothing=0.0, zloss_scale=0.0, reduction="mean",
                softcap=0.0, bias=None, class_weight=None):
    """Loss, lse, predicted [N] and accuracy of the extended options.

    accuracy = (valid rows whose argmax equals the target) / (valid rows), 0 if none.
    """
    X, W = widen(X), widen(W)
    y = _int_targets(y)
    V = W.shape[1]
    _, u = ext_logits(X, W, bias, softcap)
    lse = logsumexp_rows(u)
    ell = ext_row_losses(u, lse, y, V, ignore_index, label_smoothing, zloss_scale, class_weight)
    valid, _ = _valid_and_bad(y, V, ignore_index)
    if reduction == "none":
        loss = ell
    elif reduction == "sum":
        loss = float(ell.sum())
    else:
        den = ext_denominator(y, V, ignore_index, class_weight)
        loss = float(ell.sum()) / den if den else 0.0
    pred = argmax_first(u)
    n_valid = int(valid.sum())
    acc = float((pred[valid] == y[valid]).sum()) / n_valid if n_valid else 0.0
    return loss, lse, pred, acc


def forward_backward_ext(X, W, y, ignore_index=-100, label_smoothing=0.0, zloss_scale=0.0, reduction="mean",
                         grad_out=1.0, softcap=0.0, bias=None, class_weight=None):
    """Loss, lse, dX, dW, dbias of the extended options (dbias None without a bias).

    dZ = dU * (1 - (u / softcap)^2) with a softcap (the derivative of c tanh(z / c)),
    dX = dZ W^T, dW = X^T dZ, dbias = sum over rows of dZ.
    """
    X, W = widen(X), widen(W)
    y = _int_targets(y)
    V = W.shape[1]
    z, u = ext_logits(X, W, bias, softcap)
    lse = logsumexp_rows(u)
    loss = forward_ext(X, W, y, ignore_index, label_smoothing, zloss_scale, reduction, softcap, bias,
                       class_weight)[0]
    if reduction == "sum":
        g = float(grad_out)
    elif reduction == "mean":
        den = ext_denominator(y, V, ignore_index, class_weight)
        g = float(grad_out) / den if den else 0.0
    else:
        raise ValueError("the backward pass needs reduction 'mean' or 'sum'")
    du = ext_grad_u(u, lse, y, V, ignore_index, label_smoothing, zloss_scale, g, class_weight)
    dz = du * (1.0 - (u / float(softcap)) ** 2) if softcap and softcap > 0 else du
    dbias = dz.sum(axis=0) if bias is not None else None
    return loss, lse, dz @ W.T, X.T @ dz, dbias


def shard_stats(X, W_shard, y, v_offset: int, ignore_index=-100):
    """Per-row statistics of one vocabulary shard: (lse over the shard, sum of its logits,
    target logit if the target falls in the shard else 0, 1.0 if it does else 0.0)."""
    X, Ws = widen(X), widen(W_shard)
    y = _int_targets(y)
    z = logits(X, Ws)
    lse_k = logsumexp_rows(z)
    rel = y - int(v_offset)
    own = (y != ignore_index) & (rel >= 0) & (rel < Ws.shape[1])
    zy = np.where(own, z[np.arange(z.shape[0]), np.where(own, rel, 0)], 0.0)
    return lse_k, z.sum(axis=1), zy, own.astype(np.float64)


def combine_shard_stats(stats, V_total, y, ignore_index=-100, label_smoothing=0.0, zloss_scale=0.0,
                        reduction="mean"):
    """lse and loss from the shards' statistics: lse = log sum_k exp(lse_k), the target logit
    and the logit sum are sums over shards; then the row loss of ``row_losses``."""
    y = _int_targets(y)
    lse_k = np.stack([s[0] for s in stats])
    m = lse_k.max(axis=0)
    lse = m + np.log(np.exp(lse_k - m[None, :]).sum(axis=0))
    sum_z = sum(s[1] for s in stats)
    zy = sum(s[2] for s in stats)
    valid, bad = _valid_and_bad(y, V_total, ignore_index)
    eps = float(label_smoothing)
    ell = (1.0 - eps) * (lse - zy) + eps * (lse - sum_z / V_total) + float(zloss_scale) * lse * lse
    ell = np.where(valid, ell, 0.0)
    ell = np.where(bad, np.nan, ell)
    return reduce_loss(ell, valid, reduction), lse
