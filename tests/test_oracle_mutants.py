"""Controls: every planted mistake must be caught by the parity suite in the same run.

The mistakes are planted in the ORACLE (a `mutant` switch of the C struct, CPU only).  The
suite is the one the GPU tests use: router logits within 1e-5 relative, ids exact except at
near-ties (exact ties to the lowest index), routing weights within 1e-5, outputs within
max|err| <= 2e-2 max|y| and relative L2 <= 5e-3, the combine in slot order, and the dispatch
arrays exact.  The clean oracle must pass the same suite (against itself on another thread
count), so the suite is not vacuous either way.
"""
import numpy as np
import pytest

from gen import moegen as g
from oracle import oracle as o
from tests import parity


def _tie_layer():
    """Small FP8 layer whose router has exact ties: expert 2j+1 is a copy of expert 2j."""
    w = g.make_layer(21, 128, 64, 384, fp8=True, bias_var=0.5)
    w.Wr[1::2] = w.Wr[0::2]
    w.bias[1::2] = w.bias[0::2]
    return w


def suite(w, x, mut_layer, clean_layer):
    ref = o.layer_forward(clean_layer, x, want_probs=True)
    got = o.layer_forward(mut_layer, x, want_probs=True, nthreads=3)
    fails = []
    xf = g.bf16_bits_to_f32(x) if x.dtype == np.uint16 else x
    for t in range(0, x.shape[0], 5):
        a, b = o.router_logits(mut_layer, xf[t]), o.router_logits(clean_layer, xf[t])
        if np.max(np.abs(a - b)) > 1e-5 * np.max(np.abs(b)):
            fails.append("logits")
            break
    ok, bad, _ = parity.ids_ok(got["ids"], ref["ids"], ref["p"], w.E)
    if not ok:
        fails.append(f"ids {bad[:1]}")
    same = np.all(got["ids"] == ref["ids"], axis=1)
    if same.any():
        okw, msg = parity.weights_ok(got["w"][same], ref["w"][same])
        if not okw:
            fails.append("weights " + msg)
        oky, msg = parity.outputs_ok(got["y"][same], ref["y"][same])
        if not oky:
            fails.append("outputs " + msg)
    # combine in slot order, bit for bit, from the layer's own expert outputs
    for t in range(min(3, x.shape[0])):
        acc = o.expert(mut_layer, w.E, xf[t])
        for i in range(6):
            acc = (acc + np.float32(got["w"][t, i]) * o.expert(mut_layer, int(got["ids"][t, i]), xf[t])).astype(np.float32)
        if not np.array_equal(acc.view(np.uint32), got["y"][t].view(np.uint32)):
            fails.append("combine order")
            break
    dm = o.dispatch(got["ids"], w.E, mutant=mut_layer.s.mutant)
    dr = o.dispatch(got["ids"], w.E)
    if not all(np.array_equal(dm[key], dr[key]) for key in dr):
        fails.append("dispatch")
    return fails


@pytest.fixture(scope="module")
def data():
    w = _tie_layer()
    x = g.make_x(22, 40, w.d, bf16=True)
    return w, x


def test_clean_oracle_passes_the_suite(data):
    w, x = data
    assert suite(w, x, o.Layer(w), o.Layer(w)) == []


# a mistake that only exists in one bias mode is planted in that mode (both layers)
MUTANT_BIAS_MODE = {"biased_weights": o.BIAS_SELECT}


@pytest.mark.parametrize("name", sorted(o.MUTANTS))
def test_each_planted_mistake_is_caught(data, name):
    w, x = data
    bm = MUTANT_BIAS_MODE.get(name, o.BIAS_SCORE)
    fails = suite(w, x, o.Layer(w, mutant=o.MUTANTS[name], bias_mode=bm), o.Layer(w, bias_mode=bm))
    assert fails, f"mutant {name} passed every check"


def test_clean_oracle_passes_the_suite_in_the_selection_only_bias_mode(data):
    w, x = data
    assert suite(w, x, o.Layer(w, bias_mode=o.BIAS_SELECT), o.Layer(w, bias_mode=o.BIAS_SELECT)) == []
