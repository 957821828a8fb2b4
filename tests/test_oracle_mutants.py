"""The oracle's pins catch plausible mistakes.

Each mutant below plants one mistake in the oracle, on the CPU: a dropped term, a wrong
sign, an off-by-one index, a scrambled operand, a wrong denominator. It does so by
replacing one oracle function for the duration of a check (the mutants are small
restatements of those functions with the mistake in them). With the mutant in place, at
least one pin of ``test_oracle_pins.py`` or ``test_oracle_ext_pins.py`` must fail; a mutant
that every pin lets through marks a gap in the pins. Without a mutant every pin passes.
"""
import contextlib

import numpy as np
import pytest

import oracle
from oracle import flce_oracle as O
from tests import test_oracle_ext_pins as E
from tests import test_oracle_pins as P

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

# ---------------------------------------------------------------------------- the pins

PINS = [
    ("W=0 closed form (eps, s, mean)", lambda: P.test_w_zero_closed_form(0.1, 1e-4, "mean")),
    ("W=0 closed form (s, sum)", lambda: P.test_w_zero_closed_form(0.0, 0.3, "sum")),
    ("W=0 loss is ln V", P.test_w_zero_loss_is_ln_v_for_any_smoothing),
    ("gradient rows sum", lambda: P.test_gradient_rows_sum_to_zlosss_term(0.2, 0.1)),
    ("ignored rows", P.test_ignored_rows_contribute_nothing),
    ("no valid rows", P.test_mean_with_no_valid_rows_is_zero),
    ("out-of-range target", P.test_out_of_range_target_poisons_its_row),
    ("shift invariance", P.test_shift_invariance_without_zloss),
    ("brute force (eps, sum)", lambda: P.test_brute_force_tiny(0.1, 0.0, "sum")),
    ("brute force (s, mean)", lambda: P.test_brute_force_tiny(0.0, 0.01, "mean")),
    ("brute force (none)", lambda: P.test_brute_force_tiny(0.2, 0.05, "none")),
    ("torch fp64 (eps, s, mean)", lambda: P.test_matches_torch_cross_entropy_fp64(0.1, "mean", 1e-3)),
    ("torch fp64 (sum)", lambda: P.test_matches_torch_cross_entropy_fp64(0.0, "sum", 0.0)),
    ("finite differences", lambda: P.test_central_finite_differences(0.1, 0.5, "mean")),
    ("TE smoothing rule", lambda: P.test_transformer_engine_smoothing_rule(0.1, 16)),
    ("batched helpers", lambda: P.test_batched_helpers_match_dense(0.1, 1e-2)),
    ("defaults reduce to base", E.test_defaults_reduce_to_the_base_definitions),
    ("torch weighted smoothed capped (mean)",
     lambda: E.test_matches_torch_weighted_smoothed_capped(0.1, "mean", 3.0, True, True)),
    ("torch weighted smoothed (sum)",
     lambda: E.test_matches_torch_weighted_smoothed_capped(0.1, "sum", 0.0, False, True)),
    ("torch capped bias (mean)",
     lambda: E.test_matches_torch_weighted_smoothed_capped(0.0, "mean", 3.0, True, False)),
    ("finite differences, all options", lambda: E.test_central_finite_differences_all_options("mean")),
    ("uniform class weights", E.test_uniform_class_weights_cancel_in_the_mean),
    ("softcap closed form", E.test_softcap_closed_form_constant_logits),
    ("argmax ties and accuracy", E.test_argmax_first_index_on_ties_and_accuracy),
    ("shards combine",
     lambda: E.test_vocabulary_shards_combine_to_the_full_loss([0, 8, 64, 65, 100], 0.1, 1e-3)),
    ("shard boundary targets", E.test_targets_on_shard_boundaries),
]


def _failing_pins():
    failed = []
    for name, pin in PINS:
        try:
            pin()
        except Exception:  # an assertion, or a shape or index error the mistake provokes
            failed.append(name)
    return failed


@contextlib.contextmanager
def _planted(name, fn):
    """Replace oracle function ``name`` (in the module and in the package namespace)."""
    saved = getattr(O, name)
    exported = hasattr(oracle, name)
    setattr(O, name, fn)
    if exported:
        setattr(oracle, name, fn)
    try:
        yield
    finally:
        setattr(O, name, saved)
        if exported:
            setattr(oracle, name, saved)


# ---------------------------------------------------------------------------- the mutants
# Gradient of the loss with respect to the logits, with one mistake switched on.

def _grad(z, lse, y, V, ignore_index, eps, s, g, cols=None, *, zloss=2.0, spread=None, sign=-1.0,
          zero_ignored=True, shift=0):
    y = O._int_targets(y)
    valid, bad = O._valid_and_bad(y, V, ignore_index)
    cols = np.arange(V) if cols is None else np.asarray(cols)
    p = np.exp(z - lse[:, None])
    dz = p * (1.0 + zloss * s * lse)[:, None] - eps / (V if spread is None else spread)
    hit = ((y[:, None] + shift) == cols[None, :]) & (valid & ~bad)[:, None]
    dz = dz + sign * (1.0 - eps) * hit
    dz = dz * g
    if zero_ignored:
        dz[~valid] = 0.0
    dz[bad] = np.nan
    return dz


def _losses(z, lse, y, V, ignore_index, eps, s, *, smooth=True, zpow=2, zero_ignored=True, ref="mean"):
    y = O._int_targets(y)
    valid, bad = O._valid_and_bad(y, V, ignore_index)
    z_y = z[np.arange(z.shape[0]), np.where(valid & ~bad, y, 0)]
    ref_z = z.mean(axis=1) if ref == "mean" else z.max(axis=1)
    ell = (1.0 - eps) * (lse - z_y) + (eps * (lse - ref_z) if smooth else 0.0) + s * lse ** zpow
    if zero_ignored:
        ell = np.where(valid, ell, 0.0)
    return np.where(bad, np.nan, ell)


def _forward_backward_shifted_dW(X, W, y, ignore_index=-100, label_smoothing=0.0, zloss_scale=0.0,
                                 reduction="mean", grad_out=1.0):
    """dW = X^T dZ with row i of X paired with row i - 1 of dZ."""
    loss, lse, dX, dW = _ORIG["forward_backward"](X, W, y, ignore_index, label_smoothing, zloss_scale,
                                                  reduction, grad_out)
    if dW is None:
        return loss, lse, dX, dW
    Xw, Ww, yv = O.widen(X), O.widen(W), O._int_targets(y)
    valid, _ = O._valid_and_bad(yv, Ww.shape[1], ignore_index)
    g = O.grad_scale(grad_out, int(valid.sum()), reduction)
    dz = O.grad_logits(O.logits(Xw, Ww), lse, yv, Ww.shape[1], ignore_index, label_smoothing, zloss_scale, g)
    return loss, lse, dX, np.roll(Xw, 1, axis=0).T @ dz


_ORIG = {n: getattr(O, n) for n in ("forward_backward", "logits", "logsumexp_rows", "reduce_loss",
                                   "grad_scale", "_valid_and_bad", "ext_logits", "ext_denominator",
                                   "ext_row_losses", "ext_grad_u", "argmax_first", "combine_shard_stats",
                                   "shard_stats")}


def _ext_denominator_rows(y, V, ignore_index, class_weight=None):
    return _ORIG["ext_denominator"](y, V, ignore_index, None)


def _ext_logits_clip(X, W, bias=None, softcap=0.0):
    z = O.logits(X, W)
    if bias is not None:
        z = z + O.widen(bias)[None, :]
    u = np.clip(z, -softcap, softcap) if softcap and softcap > 0 else z
    return z, u


def _ext_row_losses_unweighted_smoothing(u, lse, y, V, ignore_index, eps, s, class_weight=None):
    ell = _ORIG["ext_row_losses"](u, lse, y, V, ignore_index, eps, s, class_weight)
    if class_weight is None or not eps:
        return ell
    w = O.widen(class_weight)
    weighted = eps * (lse * w.sum() - u @ w) / V
    plain = eps * (lse * V - u.sum(axis=1)) / V
    return np.where(np.isfinite(ell) & (ell != 0.0), ell - weighted + plain, ell)


def _ext_grad_u_no_target_weight(u, lse, y, V, ignore_index, eps, s, g, class_weight=None):
    if class_weight is None:
        return _ORIG["ext_grad_u"](u, lse, y, V, ignore_index, eps, s, g, None)
    yv = O._int_targets(y)
    w = O.widen(class_weight)
    ok = yv != ignore_index
    # the target weight w_y replaced by 1 in both places it enters
    du = _ORIG["ext_grad_u"](u, lse, yv, V, ignore_index, eps, s, g, class_weight)
    wy = np.where(ok, w[np.where(ok, yv, 0)], 1.0)
    p = np.exp(u - lse[:, None])
    corr = (1.0 - eps) * (1.0 - wy)
    du = du + g * p * corr[:, None]
    rows = np.nonzero(ok)[0]
    du[rows, yv[rows]] -= g * corr[rows]
    du[~ok] = 0.0
    return du


def _argmax_last(u):
    return u.shape[1] - 1 - np.argmax(u[:, ::-1], axis=1)


def _combine_summing_lse(stats, V_total, y, ignore_index=-100, label_smoothing=0.0, zloss_scale=0.0,
                         reduction="mean"):
    """The shards' log-sum-exps added, instead of combined by a log-sum-exp."""
    merged = [tuple(sum(st[k] for st in stats) for k in range(4))]
    return _ORIG["combine_shard_stats"](merged, V_total, y, ignore_index, label_smoothing, zloss_scale,
                                        reduction)


def _shard_stats_first_column_not_owned(X, W_shard, y, v_offset, ignore_index=-100):
    lse_k, sz, zy, own = _ORIG["shard_stats"](X, W_shard, y, v_offset, ignore_index)
    first = O._int_targets(y) == int(v_offset)
    return lse_k, sz, np.where(first, 0.0, zy), np.where(first, 0.0, own)


MUTANTS = [
    ("gradient: z-loss term dropped", "grad_logits",
     lambda z, lse, y, V, ii, e, s, g, cols=None: _grad(z, lse, y, V, ii, e, s, g, cols, zloss=0.0)),
    ("gradient: z-loss factor s instead of 2 s", "grad_logits",
     lambda z, lse, y, V, ii, e, s, g, cols=None: _grad(z, lse, y, V, ii, e, s, g, cols, zloss=1.0)),
    ("gradient: smoothing spread as eps/(V-1)", "grad_logits",
     lambda z, lse, y, V, ii, e, s, g, cols=None: _grad(z, lse, y, V, ii, e, s, g, cols, spread=V - 1)),
    ("gradient: target term with the wrong sign", "grad_logits",
     lambda z, lse, y, V, ii, e, s, g, cols=None: _grad(z, lse, y, V, ii, e, s, g, cols, sign=1.0)),
    ("gradient: ignored rows not zeroed", "grad_logits",
     lambda z, lse, y, V, ii, e, s, g, cols=None: _grad(z, lse, y, V, ii, e, s, g, cols,
                                                        zero_ignored=False)),
    ("gradient: target column off by one", "grad_logits",
     lambda z, lse, y, V, ii, e, s, g, cols=None: _grad(z, lse, y, V, ii, e, s, g, cols, shift=1)),
    ("loss: smoothing term dropped", "row_losses",
     lambda z, lse, y, V, ii, e, s: _losses(z, lse, y, V, ii, e, s, smooth=False)),
    ("loss: smoothing against the max logit", "row_losses",
     lambda z, lse, y, V, ii, e, s: _losses(z, lse, y, V, ii, e, s, ref="max")),
    ("loss: z-loss s lse instead of s lse^2", "row_losses",
     lambda z, lse, y, V, ii, e, s: _losses(z, lse, y, V, ii, e, s, zpow=1)),
    ("loss: ignored rows not zeroed", "row_losses",
     lambda z, lse, y, V, ii, e, s: _losses(z, lse, y, V, ii, e, s, zero_ignored=False)),
    ("lse: the max not added back", "logsumexp_rows",
     lambda z: _ORIG["logsumexp_rows"](z) - z.max(axis=1)),
    ("lse: log of the mean instead of the sum", "logsumexp_rows",
     lambda z: _ORIG["logsumexp_rows"](z) - np.log(z.shape[1])),
    ("logits: the [D,V] buffer read as [V,D]", "logits",
     lambda X, W: _ORIG["logits"](X, np.ascontiguousarray(W).reshape(W.shape[1], W.shape[0]).T)),
    ("mean: divided by all rows", "reduce_loss",
     lambda ell, valid, red: _ORIG["reduce_loss"](ell, np.ones_like(valid), red)),
    ("backward: 1/n_valid missing under mean", "grad_scale",
     lambda go, n, red: _ORIG["grad_scale"](go, 1 if n else 0, "mean" if red == "mean" else red)),
    ("targets: out-of-range test off by one", "_valid_and_bad",
     lambda y, V, ii: _ORIG["_valid_and_bad"](y, V + 1, ii)),
    ("dW: rows of X paired with the wrong rows of dZ", "forward_backward", _forward_backward_shifted_dW),
    ("softcap: tanh replaced by a hard clip", "ext_logits", _ext_logits_clip),
    ("class weights: mean denominator counts rows", "ext_denominator", _ext_denominator_rows),
    ("class weights: smoothing term unweighted", "ext_row_losses", _ext_row_losses_unweighted_smoothing),
    ("class weights: gradient ignores the target weight", "ext_grad_u", _ext_grad_u_no_target_weight),
    ("argmax: ties go to the last index", "argmax_first", _argmax_last),
    ("shards: log-sum-exps added instead of combined", "combine_shard_stats", _combine_summing_lse),
    ("shards: a target in a shard's first column is not owned", "shard_stats",
     _shard_stats_first_column_not_owned),
]


def test_every_pin_passes_on_the_unmutated_oracle():
    assert _failing_pins() == []


@pytest.mark.parametrize("what,name,fn", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_some_pin_catches_the_mutant(what, name, fn):
    with _planted(name, fn):
        failed = _failing_pins()
    assert failed, f"no pin catches the planted mistake: {what}"
