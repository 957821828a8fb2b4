"""What the GPU parity tests can see: how far each planted oracle mistake moves the results,
in units of the parity tolerances, on the small cases of the GPU parity suite (their
shapes, inputs and options). A kernel that made the same mistake would sit that far from
the oracle. The GPU results sit within 0.003 tolerance of the oracle in loss and lse, 0.26
in dX and 0.56 in dW (the largest errors the parity suite has measured), so a mistake two
tolerances away in some output of some case cannot pass the suite. Every mistake on the
base path must reach that line in some case. CPU only: the mutants are planted in the
oracle, never in the CUDA path."""
import numpy as np
import pytest

import oracle
from tests.flce_cases import TOL_DW_REL, TOL_DX_REL, TOL_LOSS_REL, TOL_LSE_ABS, rel_fro
from tests.test_oracle_mutants import MUTANTS, _planted
from tests.test_parity_gpu import CASES
from workloads import make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

# mistakes these cases cannot show (no out-of-range targets, no extended options or shards;
# the GPU suite's own tests of those features carry them)
NOT_EXERCISED = {
    "targets: out-of-range test off by one",
    "softcap: tanh replaced by a hard clip",
    "class weights: mean denominator counts rows",
    "class weights: smoothing term unweighted",
    "class weights: gradient ignores the target weight",
    "argmax: ties go to the last index",
    "shards: log-sum-exps added instead of combined",
    "shards: a target in a shard's first column is not owned",
}


def _distances(X, W, y, wl, truth):
    common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
    loss, lse, dX, dW = oracle.forward_backward(X, W, y, *common)
    valid = y.numpy() != wl.ignore_index
    return {
        "loss": abs(loss - truth[0]) / (TOL_LOSS_REL * abs(truth[0])),
        "lse": float(np.max(np.abs(lse[valid] - truth[1][valid]))) / TOL_LSE_ABS,
        "dX": rel_fro(dX, truth[2]) / TOL_DX_REL,
        "dW": rel_fro(dW, truth[3]) / TOL_DW_REL,
    }


class _Cases:
    """The parity cases, cheapest first, with the oracle's results computed on first use.
    The 32008-column case is left out: its oracle run takes longest and it adds no option
    the others lack."""

    def __init__(self):
        self.specs = sorted(((name, wl) for name, wl in CASES if name != "vocab_32008"),
                            key=lambda c: c[1].N * c[1].V * (c[1].D + 8))
        self.done = {}

    def __iter__(self):
        for name, wl in self.specs:
            if name not in self.done:
                X, W, y = make_inputs(wl)
                common = (wl.ignore_index, wl.label_smoothing, wl.zloss_scale, wl.reduction)
                self.done[name] = (X, W, y, oracle.forward_backward(X, W, y, *common))
            yield (name, wl) + self.done[name]


@pytest.fixture(scope="module")
def cases():
    return _Cases()


@pytest.mark.parametrize("what,name,fn", [m for m in MUTANTS if m[0] not in NOT_EXERCISED],
                         ids=[m[0] for m in MUTANTS if m[0] not in NOT_EXERCISED])
def test_gpu_parity_sees_the_mistake(cases, what, name, fn):
    worst = {}
    for case, wl, X, W, y, truth in cases:  # the unmutated results are taken outside the mutant
        with _planted(name, fn):
            worst[case] = max(_distances(X, W, y, wl, truth).values())
        if worst[case] >= 2.0:
            break  # one case that fails parity is enough
    assert max(worst.values()) >= 2.0, (what, worst)
