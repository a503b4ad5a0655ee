"""Routing diagnostics (the router comparison the pages make): the GPU routers against the
oracle's fp32 router, next to a bf16-emulated router as the calibrator ("We Ported Aleph
Alpha's Kolibri to a MacBook. Our Own Gate Said No.", section "Taking it apart": a bf16
router is the planted bug their gate catches).  Reported for the decode router (64 tokens)
and the tensor-core router (2048 tokens); the GPU must sit orders of magnitude closer to the
fp32 reference than the calibrator does (measured at 2048 tokens: max 2.9e-5 of a row
standard deviation and no disagreement, against 1.5e-2 and 4.9 % of tokens for bf16).
"""
import numpy as np
import pytest

from gen import moegen as g
from oracle import oracle as o
from tests import parity
from tests.gpu_helpers import to_dev_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import routed_expert_layer_fp32_gb300 as m
    return m


@pytest.mark.parametrize("T", [64, 2048])
def test_router_diagnostics_against_fp32_and_a_bf16_calibrator(moe, T):
    w = g.make_layer(71, 2048, 64, 384, fp8=True, bias_var=0.5)
    L = moe.Layer.from_host(w)
    x = g.make_x(72, T, 2048, bf16=True)
    ws = moe.workspace(L, T)
    ids, _, lg = moe.route(to_dev_x(x), L, ws, logits=True)
    nt = o.default_threads()
    ref = o.layer_forward(o.Layer(w), x, want_probs=True, nthreads=nt)
    cal = o.layer_forward(o.Layer(w, mutant=o.MUTANTS["bf16_router"]), x, want_probs=True, nthreads=nt)
    gpu = parity.routing_diagnostics(lg.cpu().numpy(), ids.cpu().numpy(), ref["logits"], ref["ids"])
    bf16 = parity.routing_diagnostics(cal["logits"], cal["ids"], ref["logits"], ref["ids"])
    print(f"T={T} GPU: {gpu}\nT={T} bf16 calibrator: {bf16}")
    assert gpu["sigma_err_max"] < 1e-2 * bf16["sigma_err_max"]  # measured: 2e-5 vs 1.5e-2 of a row std
    assert bf16["token_set_disagreement"] > 0.0
    assert gpu["token_set_disagreement"] <= 0.01
    assert moe.get_status(ws) == 0
