"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against a closed form, a brute-force search, an independent
library routine (torch float64 / torch's float8 and bf16 conversions / numpy's stable sort)
or an invariant the definition of the layer fixes.  A plausible slip in the oracle (a dropped
term, a wrong sign or index, a swapped operand, a wrong tie rule, a wrong summation order)
fails at least one of them; test_oracle_mutants.py checks that claim for planted slips.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

from gen import moegen as g
from oracle import oracle as o
from tests import parity

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kolibri_layer_facts.json")


@pytest.fixture(scope="module")
def tiny():
    w = g.tiny_layer()
    x = g.make_x(g.SEED_TINY, 32, w.d, bf16=False)
    return w, x


# ------------------------------------------------------------------ number formats --------

def test_e4m3_decode_matches_torch_float8_and_format():
    dec = o.e4m3_decode_all()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(dec), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(dec[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # format facts: max 448, smallest subnormal 2^-9, smallest normal 2^-6, one = 0x38
    assert dec[0x7E] == 448.0 and dec[0x01] == 2.0 ** -9 and dec[0x08] == 2.0 ** -6 and dec[0x38] == 1.0
    assert np.all(np.diff(dec[:0x7F]) > 0)  # monotone over the non-negative finite codes


def _all_e4m3_midpoints():
    dec = o.e4m3_decode_all()[:0x7F].astype(np.float64)
    mids = (dec[:-1] + dec[1:]) / 2  # exact in fp32 (at most 5 significant bits)
    return dec, mids.astype(np.float32)


def test_e4m3_encode_ties_to_even_and_neighbours():
    dec, mids = _all_e4m3_midpoints()
    codes = o.e4m3_encode(mids)
    lo = np.arange(0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(codes, expect)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    assert np.array_equal(o.e4m3_encode(up), lo + 1)
    assert np.array_equal(o.e4m3_encode(dn), lo)
    # negatives mirror positives with the sign bit
    assert np.array_equal(o.e4m3_encode(-up), (lo + 1) | 0x80)


def test_e4m3_encode_matches_torch_in_range_and_saturates():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(200_000) * s for s in (1e-3, 0.1, 1, 10, 100)]).astype(np.float32)
    v = v[np.abs(v) < 464]
    ours = o.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    big = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e4, 3e38], np.float32)
    assert np.all(o.e4m3_encode(big) == 0x7E)
    assert np.all(o.e4m3_encode(-big) == 0xFE)


# The OCP Microscaling Formats specification v1.0 (section 5.3.3) lists the E2M1 element
# format by its representable values: sign bit 3; magnitudes 0 and 0.5 (subnormal), 1, 1.5,
# 2, 3, 4, 6 (max normal 6.0, min normal 1.0, min subnormal 0.5); no infinities or NaN.
E2M1_SPEC = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], np.float64)


def test_e2m1_decode_matches_the_format():
    dec = o.e2m1_decode_all().astype(np.float64)
    assert np.array_equal(dec[:8], E2M1_SPEC)
    assert np.array_equal(dec[8:], -E2M1_SPEC) and np.signbit(dec[8])


def test_generator_e2m1_quantiser_rounds_to_nearest_even():
    """The 4-bit checkpoint's encoder (the generator's, input preparation): every midpoint
    goes to the even code, its neighbours to the nearest, beyond 6 saturates."""
    mids = (E2M1_SPEC[:-1] + E2M1_SPEC[1:]) / 2
    v = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(9)),
                        np.nextafter(mids.astype(np.float32), np.float32(-1)), E2M1_SPEC, [7.0, 1e9]]).astype(np.float32)
    got = g.quant_e2m1(v)
    want = []
    for x in v.astype(np.float64):
        dist = np.abs(E2M1_SPEC - x)
        best = np.flatnonzero(dist == dist.min())
        want.append(best[0] if len(best) == 1 else best[best % 2 == 0][0])
    assert np.array_equal(got, np.array(want, np.uint8))
    assert np.array_equal(g.quant_e2m1(-v), np.array(want, np.uint8) | 8)


def _dec4(packed):
    """Packed E2M1 rows (two codes per byte, element 2i in the low nibble) as float64 values,
    decoded with the specification's table."""
    codes = np.stack([packed & 15, packed >> 4], axis=-1).reshape(*packed.shape[:-1], -1)
    return np.where(codes & 8, -1.0, 1.0) * E2M1_SPEC[codes & 7]


def test_w4a8_expert_matches_float64_with_torch_quantiser():
    """The expert with 4-bit weights: E2M1 codes times their row scales, per-row E4M3
    activations (torch's conversion), float64 products, as the W8A8 pin above."""
    w = g.make_layer(17, 256, 128, 8, fp8=False, bias_var=0.5, fp4=True)
    x = g.make_x(18, 64, w.d, bf16=True)
    xf = g.bf16_bits_to_f32(x)
    L = o.Layer(w)

    def q(v):
        s = np.float32(np.max(np.abs(v)) / np.float32(448.0))
        codes = torch.from_numpy((v / s).astype(np.float32)).to(torch.float8_e4m3fn)
        return codes.double().numpy(), float(s)

    errs = []
    for t in range(64):
        e = t % 8
        qx, sx = q(xf[t])
        gg = (_dec4(w.Wgu[e, 0]) @ qx) * sx * w.sgu[e, 0].astype(np.float64)
        uu = (_dec4(w.Wgu[e, 1]) @ qx) * sx * w.sgu[e, 1].astype(np.float64)
        h = (gg / (1 + np.exp(-gg)) * uu).astype(np.float32)
        qh, sh = q(h)
        y = (_dec4(w.Wd[e]) @ qh) * sh * w.sd[e].astype(np.float64)
        errs.append(parity.rel_l2(o.expert(L, e, xf[t]), y))
    errs = np.array(errs)
    assert np.mean(errs < 1e-5) >= 0.9, errs
    assert errs.max() < 1e-3, errs


def test_one_hot_route_is_the_dense_ffn_w4a16():
    """4-bit weights, forced_w = (1,0,0,0,0,0), shared expert zeroed: y = the dense FFN of that
    expert on fp32 activations and the spec-decoded weights (float64)."""
    w = g.make_layer(19, 128, 128, 16, fp8=False, bias_var=0.5, fp4=True)
    w.sh_sgu[:] = 0
    w.sh_sd[:] = 0
    x = g.make_x(20, 6, w.d, bf16=True)
    xf = g.bf16_bits_to_f32(x).astype(np.float64)
    L = o.Layer(w, act_mode=o.ACT_W8A16)
    ids = np.array([[e, (e + 3) % 16, (e + 5) % 16, (e + 7) % 16, (e + 9) % 16, (e + 11) % 16] for e in range(6)],
                   np.int32)
    fw = np.zeros((6, 6), np.float32)
    fw[:, 0] = 1
    out = o.layer_forward(L, x, forced_ids=ids, forced_w=fw)
    for t in range(6):
        e = ids[t, 0]
        Wg = _dec4(w.Wgu[e, 0]) * w.sgu[e, 0][:, None]
        Wu = _dec4(w.Wgu[e, 1]) * w.sgu[e, 1][:, None]
        Wd = _dec4(w.Wd[e]) * w.sd[e][:, None]
        gg, uu = Wg @ xf[t], Wu @ xf[t]
        y = Wd @ (gg / (1 + np.exp(-gg)) * uu)
        assert parity.rel_l2(out["y"][t], y) < 2e-6


def test_4bit_checkpoint_is_a_coarser_copy_of_the_same_weights():
    """The 4-bit and the FP8 checkpoints of one seed decode to the same Gaussian weights within
    each format's rounding (E2M1 keeps one mantissa bit), so their layers agree loosely."""
    w8 = g.make_layer(21, 256, 128, 8, fp8=True, bias_var=0.5)
    w4 = g.make_layer(21, 256, 128, 8, fp8=False, bias_var=0.5, fp4=True)
    a = _dec4(w4.Wgu) * w4.sgu[..., None]
    b = _dec(w8.Wgu) * w8.sgu[..., None]
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 0.05 < rel < 0.2, rel
    x = g.make_x(22, 16, 256, bf16=True)
    y8 = o.layer_forward(o.Layer(w8), x)
    y4 = o.layer_forward(o.Layer(w4), x, forced_ids=y8["ids"])
    assert 0.03 < parity.rel_l2(y4["y"], y8["y"]) < 0.3


def test_bf16_rne_matches_definition_and_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, (rng.integers(0, 2 ** 16, 100_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000])
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    ours = o.bf16_rne(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # torch overflows to inf where RNE carries past the largest finite bf16; so does the definition
    assert np.array_equal(ours, ref)
    # two-candidate definition: truncate or truncate + 1 ulp, the nearer one, ties to even
    u = f.view(np.uint32)
    trunc = (u >> 16).astype(np.uint32)
    lo = (trunc << 16).view(np.float32).astype(np.float64)
    hi = ((trunc + 1) << 16).view(np.float32).astype(np.float64)
    x = f.astype(np.float64)
    dlo, dhi = np.abs(x - lo), np.abs(hi - x)
    pick = np.where(dlo < dhi, trunc, np.where(dhi < dlo, trunc + 1, np.where(trunc % 2 == 0, trunc, trunc + 1)))
    fin = np.isfinite(hi)
    assert np.array_equal(ours[fin], pick[fin].astype(np.uint16))


# ------------------------------------------------------------------------- routing --------

def _ref_topk(p, k):
    # full stable sort by (-p, index): the lowest index comes first among equal p
    order = np.lexsort((np.arange(p.shape[0]), -p.astype(np.float64)))
    return order[:k].astype(np.int32)


def test_topk_matches_full_stable_sort_E384():
    rng = np.random.default_rng(2)
    for trial in range(200):
        logits = rng.standard_normal(384).astype(np.float32)
        if trial % 4 == 0:  # planted exact ties
            dup = rng.choice(384, 40, replace=False)
            logits[dup[20:]] = logits[dup[:20]]
        p = o.softmax(logits)
        assert np.array_equal(o.topk(p, 6), _ref_topk(p, 6))


def test_topk_matches_subset_enumeration_E12():
    rng = np.random.default_rng(3)
    for _ in range(50):
        p = rng.permutation(np.arange(1, 13)).astype(np.float32) / 78.0
        best = None
        for s in itertools.combinations(range(12), 6):
            rest = [i for i in range(12) if i not in s]
            if min(p[list(s)]) > max(p[rest]):
                best = set(s)
        ids = o.topk(p, 6)
        assert set(ids.tolist()) == best
        assert np.all(np.diff(p[ids]) < 0)  # descending probability order


def test_exact_ties_go_to_lowest_index():
    p = np.full(384, 1.0 / 384, np.float32)
    assert np.array_equal(o.topk(p, 6), np.arange(6))
    p[[10, 20, 30, 40, 50, 60, 70]] = 0.01
    assert np.array_equal(o.topk(p, 6), [10, 20, 30, 40, 50, 60])


def test_renormalisation_sums_to_one_and_is_shift_invariant():
    rng = np.random.default_rng(4)
    for _ in range(100):
        logits = (np.round(rng.standard_normal(384) * 1024) / 1024).astype(np.float32)
        p = o.softmax(logits)
        ids = o.topk(p, 6)
        w = o.renorm(p, ids)
        assert abs(float(w.astype(np.float64).sum()) - 1.0) <= 1e-6
        p2 = o.softmax(logits + np.float32(3.0))  # exact shift (multiples of 2^-10)
        assert np.array_equal(o.topk(p2, 6), ids)
        assert np.array_equal(o.renorm(p2, ids), w)


def test_softmax_matches_torch_float64():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((64, 384)).astype(np.float32) * 3
    ref = torch.softmax(torch.from_numpy(logits).double(), dim=-1).numpy()
    for t in range(64):
        assert np.max(np.abs(o.softmax(logits[t]) - ref[t]) / ref[t]) < 1e-5


# ------------------------------------------------------------- the layer, fp32 ------------

def _torch_f64_layer(w, x, ids=None):
    """The tiny all-fp32 layer in torch float64 (independent library evaluation)."""
    X = torch.from_numpy(np.asarray(x, np.float32)).double()
    Wr = torch.from_numpy(w.Wr).double()
    logits = X @ Wr.T + (torch.from_numpy(w.bias).double() if w.bias is not None else 0)
    p = torch.softmax(logits, -1)
    if ids is None:
        ids = torch.topk(p, 6, dim=-1, sorted=True).indices.numpy().astype(np.int32)
    ids_t = torch.from_numpy(np.asarray(ids)).long()
    pw = torch.gather(p, 1, ids_t)
    wts = pw / pw.sum(1, keepdim=True)

    def ffn(Wgu, Wd, xx):
        gg = xx @ torch.from_numpy(Wgu[0]).double().T
        uu = xx @ torch.from_numpy(Wgu[1]).double().T
        return (gg * torch.sigmoid(gg) * uu) @ torch.from_numpy(Wd).double().T

    y = ffn(w.sh_Wgu, w.sh_Wd, X)
    for t in range(X.shape[0]):
        for i in range(6):
            e = int(ids_t[t, i])
            y[t] += wts[t, i] * ffn(w.Wgu[e], w.Wd[e], X[t:t + 1])[0]
    return ids, p.numpy(), wts.numpy(), y.numpy()


def test_tiny_fp32_layer_matches_torch_float64(tiny):
    w, x = tiny
    L = o.Layer(w)
    out = o.layer_forward(L, x, want_probs=True)
    ids_ref, p_ref, w_ref, _ = _torch_f64_layer(w, x)
    ok, bad, _ = parity.ids_ok(out["ids"], ids_ref, p_ref, w.E)
    assert ok, bad
    # evaluate the float64 layer on the oracle's ids (identical unless a near-tie flipped)
    _, _, w_ref, y_ref = _torch_f64_layer(w, x, ids=out["ids"])
    assert np.max(np.abs(out["w"] - w_ref)) < 1e-6
    assert parity.rel_l2(out["y"], y_ref) < 1e-5
    assert np.max(np.abs(out["y"] - y_ref)) < 1e-5 * np.max(np.abs(y_ref)) * 10


def test_forced_equals_free_bit_exact(tiny):
    w, x = tiny
    L = o.Layer(w)
    free = o.layer_forward(L, x)
    forced = o.layer_forward(L, x, forced_ids=free["ids"])
    assert np.array_equal(forced["ids"], free["ids"])
    assert np.array_equal(forced["w"].view(np.uint32), free["w"].view(np.uint32))
    assert np.array_equal(forced["y"].view(np.uint32), free["y"].view(np.uint32))


def test_selection_only_bias_against_float64_definition():
    """Selection-only bias mode (the per-expert bias ranks the experts, the weights come from
    the unbiased softmax), against float64 numpy: logits = x Wr^T without the bias; ids = the
    six largest logits + b (lowest index first on ties); w = softmax of the unbiased logits
    over those six.  A large bias on one expert forces it into every token's set while its
    weight stays what its own logit gives."""
    w = g.make_layer(51, 256, 128, 384, fp8=True, bias_var=0.5)
    w.bias[7] = 50.0  # expert 7 always selected, first
    x = g.make_x(52, 24, 256, bf16=True)
    xf = g.bf16_bits_to_f32(x).astype(np.float64)
    L = o.Layer(w, bias_mode=o.BIAS_SELECT)
    out = o.layer_forward(L, x, want_probs=True)
    raw = xf @ w.Wr.astype(np.float64).T
    for t in range(x.shape[0]):
        assert np.max(np.abs(out["logits"][t] - raw[t])) < 1e-5 * np.max(np.abs(raw[t]))
        score = raw[t] + w.bias.astype(np.float64)
        order = np.lexsort((np.arange(384), -score))[:6]
        assert np.array_equal(out["ids"][t], order)
        assert out["ids"][t][0] == 7
        e = np.exp(raw[t][order] - raw[t][order].max())
        np.testing.assert_allclose(out["w"][t], e / e.sum(), rtol=2e-6, atol=1e-7)
    # the same ids under the score mode carry different weights (the bias changes them there)
    s_out = o.layer_forward(o.Layer(w), x, forced_ids=out["ids"])
    assert not np.allclose(s_out["w"], out["w"], atol=1e-3)


def test_score_mode_bias_against_float64_definition():
    """Score-mode bias (the routing of every Kolibri-shaped workload: the per-expert bias is
    added to the router score, "We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate
    Said No.", section 1), against float64 numpy: logits = x Wr^T + b; p = softmax over all
    experts; ids = the six largest p (lowest index first on ties); w = p over those six,
    renormalised.  A large positive bias on one expert puts it first in every token's set
    with most of the weight; a large negative one keeps another out of every set.  A slip in
    the sign or the scale of b moves the logits by |b| (about 0.7 here) and fails the logit
    check by five orders of magnitude."""
    w = g.make_layer(55, 256, 128, 384, fp8=True, bias_var=0.5)
    w.bias[11] = 12.0   # always selected, and dominant in the weights
    w.bias[3] = -40.0   # never selected
    x = g.make_x(56, 24, 256, bf16=True)
    xf = g.bf16_bits_to_f32(x).astype(np.float64)
    out = o.layer_forward(o.Layer(w), x, want_probs=True)
    lg = xf @ w.Wr.astype(np.float64).T + w.bias.astype(np.float64)
    for t in range(x.shape[0]):
        assert np.max(np.abs(out["logits"][t] - lg[t])) < 1e-5 * np.max(np.abs(lg[t]))
        e = np.exp(lg[t] - lg[t].max())
        p = e / e.sum()
        np.testing.assert_allclose(out["p"][t], p, rtol=1e-5, atol=1e-9)
        order = np.lexsort((np.arange(384), -p))[:6]
        assert np.array_equal(out["ids"][t], order)
        assert out["ids"][t][0] == 11 and 3 not in out["ids"][t]
        np.testing.assert_allclose(out["w"][t], p[order] / p[order].sum(), rtol=1e-5, atol=1e-7)
        assert out["w"][t][0] > 0.99


def test_stack_is_layers_with_a_bf16_residual_update():
    """The stack (50 layers in Kolibri-1: "We Ported Aleph Alpha's Kolibri to a MacBook. Our Own
    Gate Said No.", section "The gate") is, layer after layer, r <- bf16(r + layer(r)): the
    oracle's stack against three separate layer calls with the residual update done by torch
    (fp32 add, then torch's round-to-nearest-even conversion to bf16), bit-exact, free routing
    and forced.  A stack that rounded y alone, skipped the rounding or fed a layer the
    unrounded sum differs in the bits."""
    ws = [g.make_layer(57 + l, 128, 64, 16, fp8=True, bias_var=0.5) for l in range(3)]
    Ls = [o.Layer(w) for w in ws]
    r0 = g.make_x(60, 20, 128, bf16=True)
    r = torch.from_numpy(r0.view(np.int16).copy()).view(torch.bfloat16)
    ids_ref = []
    for L in Ls:
        out = o.layer_forward(L, r.view(torch.int16).numpy().view(np.uint16))
        r = (r.float() + torch.from_numpy(out["y"])).to(torch.bfloat16)
        ids_ref.append(out["ids"])
    r_ref = r.view(torch.int16).numpy().view(np.uint16)
    got, ids = o.stack_forward(Ls, r0)
    assert np.array_equal(ids, np.stack(ids_ref))
    assert np.array_equal(got, r_ref)
    forced, ids_f = o.stack_forward(Ls, r0, forced_ids=ids)
    assert np.array_equal(ids_f, ids) and np.array_equal(forced, r_ref)
    # the update is not a no-op and not y alone
    assert not np.array_equal(got, r0)
    y_only = torch.from_numpy(o.layer_forward(Ls[0], r0)["y"]).to(torch.bfloat16).view(torch.int16).numpy()
    assert not np.array_equal(o.stack_forward(Ls[:1], r0)[0], y_only.view(np.uint16))


def test_selection_only_bias_with_zero_bias_equals_score_mode():
    w = g.make_layer(53, 256, 128, 384, fp8=True, bias_var=None)
    x = g.make_x(54, 16, 256, bf16=True)
    a = o.layer_forward(o.Layer(w, bias_mode=o.BIAS_SELECT), x)
    b = o.layer_forward(o.Layer(w), x)
    for key in ("ids", "w", "y"):
        assert np.array_equal(a[key].view(np.uint32), b[key].view(np.uint32))


def test_combine_is_in_slot_order(tiny):
    """y is bit-identical to y_shared + w_0 y_0 + ... + w_5 y_5 accumulated left to right in
    fp32 (numpy float32 ops, no fused multiply-add), from the oracle's own expert outputs."""
    w, x = tiny
    L = o.Layer(w)
    out = o.layer_forward(L, x[:4])
    for t in range(4):
        acc = o.expert(L, w.E, x[t])
        for i in range(6):
            prod = np.float32(out["w"][t, i]) * o.expert(L, int(out["ids"][t, i]), x[t])
            acc = (acc + prod).astype(np.float32)
        assert np.array_equal(acc.view(np.uint32), out["y"][t].view(np.uint32))


def test_zero_weights_give_shared_expert_alone(tiny):
    w, x = tiny
    L = o.Layer(w)
    free = o.layer_forward(L, x)
    zero = o.layer_forward(L, x, forced_ids=free["ids"], forced_w=np.zeros((32, 6), np.float32))
    for t in range(0, 32, 7):
        assert np.array_equal(zero["y"][t].view(np.uint32), o.expert(L, w.E, x[t]).view(np.uint32))


def test_permutation_equivariance_and_chunk_invariance(tiny):
    w, x = tiny
    L = o.Layer(w)
    full = o.layer_forward(L, x)
    perm = np.random.default_rng(6).permutation(32)
    pe = o.layer_forward(L, x[perm])
    assert np.array_equal(pe["y"].view(np.uint32), full["y"][perm].view(np.uint32))
    assert np.array_equal(pe["ids"], full["ids"][perm])
    parts = [o.layer_forward(L, x[i:i + 8]) for i in range(0, 32, 8)]
    assert np.array_equal(np.concatenate([p["y"] for p in parts]).view(np.uint32), full["y"].view(np.uint32))
    mt = o.layer_forward(L, x, nthreads=4)
    assert np.array_equal(mt["y"].view(np.uint32), full["y"].view(np.uint32))


# ------------------------------------------------------------- the layer, FP8 -------------

def _small_fp8_layer(seed=11, d=128, ffn=64, E=16, bias=0.5):
    return g.make_layer(seed, d, ffn, E, fp8=True, bias_var=bias)


def _dec(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def test_one_hot_route_is_the_dense_ffn_w8a16():
    """forced_w = (1,0,0,0,0,0) with the shared expert zeroed: y = dense FFN of that expert on
    fp32 activations and decoded weights (torch float64, torch's own FP8 decoding)."""
    w = _small_fp8_layer()
    w.sh_sgu[:] = 0
    w.sh_sd[:] = 0
    x = g.make_x(12, 8, w.d, bf16=True)
    xf = g.bf16_bits_to_f32(x).astype(np.float64)
    L = o.Layer(w, act_mode=o.ACT_W8A16)
    ids = np.array([[e, (e + 1) % 16, (e + 2) % 16, (e + 3) % 16, (e + 4) % 16, (e + 5) % 16] for e in range(8)], np.int32)
    fw = np.zeros((8, 6), np.float32)
    fw[:, 0] = 1
    out = o.layer_forward(L, x, forced_ids=ids, forced_w=fw)
    for t in range(8):
        e = ids[t, 0]
        Wg = _dec(w.Wgu[e, 0]) * w.sgu[e, 0][:, None]
        Wu = _dec(w.Wgu[e, 1]) * w.sgu[e, 1][:, None]
        Wd = _dec(w.Wd[e]) * w.sd[e][:, None]
        gg, uu = Wg @ xf[t], Wu @ xf[t]
        y = Wd @ (gg / (1 + np.exp(-gg)) * uu)
        assert parity.rel_l2(out["y"][t], y) < 2e-6


def test_w8a8_expert_matches_float64_with_torch_quantiser():
    """The W8A8 expert: per-row activation quantisation with scale max|v|/448, E4M3 codes from
    torch's conversion, float64 products.  Quantisation codes are a rounding decision, so a code
    can flip where fp32 and fp64 disagree near a rounding boundary: almost all tokens must
    agree to 1e-5 and all within 1e-3."""
    w = _small_fp8_layer(seed=13, d=256, ffn=128, E=8)
    x = g.make_x(14, 64, w.d, bf16=True)
    xf = g.bf16_bits_to_f32(x)
    L = o.Layer(w)

    def q(v):
        s = np.float32(np.max(np.abs(v)) / np.float32(448.0))
        codes = torch.from_numpy((v / s).astype(np.float32)).to(torch.float8_e4m3fn)
        return codes.double().numpy(), float(s)

    errs = []
    for t in range(64):
        e = t % 8
        qx, sx = q(xf[t])
        gg = (_dec(w.Wgu[e, 0]) @ qx) * sx * w.sgu[e, 0].astype(np.float64)
        uu = (_dec(w.Wgu[e, 1]) @ qx) * sx * w.sgu[e, 1].astype(np.float64)
        h = (gg / (1 + np.exp(-gg)) * uu).astype(np.float32)
        qh, sh = q(h)
        y = (_dec(w.Wd[e]) @ qh) * sh * w.sd[e].astype(np.float64)
        errs.append(parity.rel_l2(o.expert(L, e, xf[t]), y))
    errs = np.array(errs)
    assert np.mean(errs < 1e-5) >= 0.9, errs
    assert errs.max() < 1e-3, errs


def test_w8a8_vs_w8a16_gap_is_the_size_of_e4m3_rounding():
    w = _small_fp8_layer(seed=15, d=256, ffn=128, E=16)
    x = g.make_x(16, 32, w.d, bf16=True)
    a = o.layer_forward(o.Layer(w, act_mode=o.ACT_W8A8), x)
    b = o.layer_forward(o.Layer(w, act_mode=o.ACT_W8A16), x, forced_ids=a["ids"])
    gap = parity.rel_l2(a["y"], b["y"])
    # E4M3 keeps 3 mantissa bits: relative rounding error ~ 2^-4/sqrt(3) per element, and the
    # two activation quantisations add up to a few per cent on the output
    assert 0.005 < gap < 0.08, gap


# ----------------------------------------------------------------------- dispatch --------

def _np_dispatch(ids, E):
    T, k = ids.shape
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")  # by expert, then (t, i) row-major = ascending t
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    counts = np.append(counts, T).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    perm = np.concatenate([order // k, np.arange(T)]).astype(np.int32)
    pos = np.empty(T * k, np.int32)
    pos[order] = np.arange(T * k)
    return counts, offsets, perm, pos.reshape(T, k)


@pytest.mark.parametrize("T", [0, 1, 5, 64, 333])
def test_dispatch_matches_numpy_stable_sort(T):
    rng = np.random.default_rng(T)
    ids = np.array([rng.choice(384, 6, replace=False) for _ in range(T)], np.int32).reshape(T, 6)
    d = o.dispatch(ids, 384)
    c, off, perm, pos = _np_dispatch(ids, 384)
    assert np.array_equal(d["counts"], c) and np.array_equal(d["offsets"], off)
    assert np.array_equal(d["perm"], perm) and np.array_equal(d["pos"], pos)
    assert d["counts"][:384].sum() == 6 * T
    rows = d["pos"].reshape(-1)
    assert np.array_equal(np.sort(rows), np.arange(6 * T))  # bijection
    for e in range(384):
        seg = d["perm"][d["offsets"][e]:d["offsets"][e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_dispatch_single_expert_holds_every_row():
    T = 100
    ids = np.tile(np.arange(6, dtype=np.int32), (T, 1))
    d = o.dispatch(ids, 384)
    assert np.array_equal(d["counts"][:6], [T] * 6) and d["counts"][6:384].sum() == 0


def test_golden_facts_match_the_workloads():
    facts = json.load(open(GOLDEN))
    assert g.KOLIBRI["E"] == facts["n_routed_experts"]["value"]
    assert g.KOLIBRI["k"] == facts["top_k"]["value"]
    fw = facts["first_wave_rows"]["value"]
    assert fw["prompts"] * fw["padded_len"] * fw["top_k"] == fw["rows"]
    gw = facts["gemma_first_wave_rows"]["value"]
    assert gw["prompts"] * gw["padded_len"] * gw["top_k"] == gw["rows"] and gw["rows"] % 64 == 0
    assert all(r % 64 for r in facts["gather_rowcounts_wrong_on_m5"]["value"])


def test_routing_diagnostics_on_constructed_rows():
    """The diagnostics helper on rows whose answers are known by construction."""
    ref = np.array([[0.0, 1.0, 2.0, 3.0], [1.0, 1.0, 3.0, 3.0]], np.float32)  # stds 1.118..., 1.0
    got = ref.copy()
    got[1, 2] += 0.5
    d = parity.routing_diagnostics(got, np.array([[3, 2], [2, 3]]), ref, np.array([[3, 2], [3, 1]]))
    assert d["sigma_err_max"] == pytest.approx(0.5)
    assert d["sigma_err_mean"] == pytest.approx(0.25)
    assert d["token_set_disagreement"] == pytest.approx(0.5)  # {2,3} vs {1,3} in the second token
    assert d["slot_disagreement"] == pytest.approx(0.5)       # slots differ in the second token only
