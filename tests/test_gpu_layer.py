"""GPU parity: libmoe through its C ABI against the CPU oracle on the same seeded inputs.

Acceptance (the layer's stated tolerances): forced ids bit-exact; free ids exact except at
near-ties (reference probabilities within 1e-4, exact ties to the lowest index); outputs
within max|err| <= 2e-2 max|y_ref| and relative L2 <= 5e-3 of the oracle.  Where free
routing flips a near-tie, the outputs are compared with the oracle run on the GPU's ids.
"""
import numpy as np
import pytest
import torch

from gen import moegen as g
from oracle import oracle as o
from tests import parity
from tests.gpu_helpers import check_forced_layer, check_free_layer, oracle_route, to_dev_x, to_host_bf16_bits

pytestmark = pytest.mark.gpu

# expert kernels: weight-streaming warp-MMA path, or the tcgen05 grouped GEMM
PATHS = {"stream": 1, "tc": 2}


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import routed_expert_layer_fp32_gb300 as m
    assert torch.cuda.is_available()
    return m


class KolibriLayers:
    """The Kolibri-shaped layer's host weights and the device layer in both weight layouts:
    tiled (tcgen05 expert kernels, the default) and rows (weight-streaming kernels).
    Unpacks as (weights, tiled layer)."""

    def __init__(self, w, tiled, rows):
        self.w, self.tiled, self.rows = w, tiled, rows

    def __iter__(self):
        return iter((self.w, self.tiled))

    def for_path(self, path):
        return self.rows if path == "stream" else self.tiled


@pytest.fixture(scope="module")
def kolibri(moe):
    w = g.kolibri_layer(g.SEED_DECODE)
    return KolibriLayers(w, moe.Layer.from_host(w), moe.Layer.from_host(w, tiled=False))


@pytest.fixture(scope="module")
def tiny(moe):
    w = g.tiny_layer()
    return w, moe.Layer.from_host(w)


# ------------------------------------------------------------------------ codec ----------

def test_device_e4m3_encoder_matches_oracle(moe):
    dec = o.e4m3_decode_all()[:0x7F].astype(np.float64)
    mids = ((dec[:-1] + dec[1:]) / 2).astype(np.float32)
    rng = np.random.default_rng(0)
    v = np.concatenate([mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(0)),
                        -mids, np.array([0, 448, 449, 464, 480, 1e6, 3e38, 1e-30, 2 ** -10, 2 ** -11], np.float32),
                        (rng.standard_normal(2_000_000) * rng.choice([1e-3, 1, 100, 1000], 2_000_000)).astype(np.float32)])
    v = np.concatenate([v, -v]).astype(np.float32)
    got = moe.e4m3_encode(torch.from_numpy(v).cuda()).cpu().numpy()
    ref = o.e4m3_encode(v)
    # -0 and +0 are the same value; compare codes after folding the zero codes
    got0 = np.where(got == 0x80, 0, got)
    ref0 = np.where(ref == 0x80, 0, ref)
    bad = np.nonzero(got0 != ref0)[0]
    assert bad.size == 0, [(float(v[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def _tiled_reference(rows: np.ndarray, block_rows: int, gate_up: bool, F: int) -> np.ndarray:
    """The tiled layout as include/libmoe.h states it, built with numpy from the row layout:
    16 KB tiles of 128 rows x 128 bytes, 16-byte chunk c of row r stored at chunk c ^ (r % 8)."""
    E, R, K = rows.shape
    tiles = []
    for e in range(E):
        for n in range((F if gate_up else R) // 128):
            for j in range(K // 128):
                for half in ((0, 1) if gate_up else (None,)):
                    r0 = (half * F if gate_up else 0) + n * 128
                    tile = rows[e, r0:r0 + 128, j * 128:(j + 1) * 128].reshape(128, 8, 16)
                    out = np.empty_like(tile)
                    for r in range(128):
                        out[r, np.arange(8) ^ (r % 8)] = tile[r]
                    tiles.append(out.reshape(-1))
    return np.concatenate(tiles)


def test_pack_weights_matches_the_documented_tiled_layout(moe):
    """moe_pack_weights against a numpy construction of the layout the header documents, on
    a small E4M3 layer (3 experts, d = 384, ffn = 256), byte for byte."""
    w = g.make_layer(41, 384, 256, 8, fp8=True, bias_var=None)
    rows = moe.Layer.from_host(w, tiled=False)
    tiled = rows.tiled()
    torch.cuda.synchronize()
    E, d, F = 8, 384, 256
    got = tiled.tensors["w_gate_up"].cpu().numpy().reshape(-1)
    want = _tiled_reference(w.Wgu.reshape(E, 2 * F, d), 128, True, F)
    assert np.array_equal(got, want)
    got = tiled.tensors["w_down"].cpu().numpy().reshape(-1)
    assert np.array_equal(got, _tiled_reference(w.Wd.reshape(E, d, F), 128, False, F))
    got = tiled.tensors["sh_gate_up"].cpu().numpy().reshape(-1)
    assert np.array_equal(got, _tiled_reference(w.sh_Wgu.reshape(1, 2 * F, d), 128, True, F))
    got = tiled.tensors["sh_down"].cpu().numpy().reshape(-1)
    assert np.array_equal(got, _tiled_reference(w.sh_Wd.reshape(1, d, F), 128, False, F))


def test_layouts_and_paths(moe, kolibri):
    """The tiled layer runs on the tcgen05 kernels (AUTO and TC), the row layer on the
    streaming kernels (AUTO and STREAM); asking for the other path is MOE_ERR_UNSUPPORTED."""
    x = to_dev_x(g.make_x(g.SEED_DECODE, 8, 2048, bf16=True))
    ws = moe.workspace(kolibri.tiled, 8)
    y_t, _, _ = moe.forward(x, kolibri.tiled, ws)
    y_r, _, _ = moe.forward(x, kolibri.rows, ws)
    assert torch.isfinite(y_t).all() and torch.isfinite(y_r).all()
    for L, flags in ((kolibri.tiled, 1), (kolibri.rows, 2)):
        with pytest.raises(moe.binding.MoeError) as err:
            moe.forward(x, L, ws, flags=flags)
        assert err.value.status == -2


# ------------------------------------------------------------------------ router ---------

@pytest.mark.parametrize("T", [1, 8, 33, 64, 129, 300, 2048])
def test_router_logits_ids_weights(moe, kolibri, T):
    w, L = kolibri
    x = g.make_x(g.SEED_DECODE, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    ids, wt, lg = moe.route(to_dev_x(x), L, ws, logits=True)
    ref = oracle_route(w, x)
    lg = lg.cpu().numpy()
    # fp32 logits: both sides accumulate in fp32 in different orders (the prefill router sums
    # three bf16 weight terms on the tensor cores); the bound is far below what moves a
    # routing decision (near-ties within 1e-4 in probability)
    err = np.max(np.abs(lg - ref["logits"]), axis=1) / np.max(np.abs(ref["logits"]), axis=1)
    assert err.max() < 3e-5, err.max()
    ok, bad, ndiff = parity.ids_ok(ids.cpu().numpy(), ref["ids"], ref["p"], w.E)
    assert ok, bad
    same = np.all(ids.cpu().numpy() == ref["ids"], axis=1)
    assert np.max(np.abs(wt.cpu().numpy()[same] - ref["w"][same])) < 1e-5
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("d,E,T", [(2048, 384, 600), (2048, 384, 2048), (2048, 384, 4096), (2048, 384, 9000),
                                   (2048, 384, 12000), (1024, 512, 1024), (1024, 480, 1024), (1024, 256, 1024),
                                   (1024, 224, 1024)])
def test_prefill_router_cluster_sizes(moe, d, E, T):
    """The tensor-core prefill router at every way it spreads the tiles: a cluster of P = 4 or
    2 CTAs per 128-token tile, each CTA E / P experts (600, 2048 and 4096 tokens: P = 4; 9000:
    P = 2; 12,000: one CTA per tile, all experts), 256 experts split 4 x 64 and 224 experts
    only 2 x 112 (224 is not a multiple of 4 x 16), and 480 and 512 experts at d = 1024, where
    two halves' weight stages do not fit in shared memory and the SIMT router with the
    selection kernel runs instead.  Logits, ids and weights against
    the oracle on every token up to 2048 and on 256 sampled tokens above (each token's routing
    is independent of the others)."""
    w = g.make_layer(61 + E, d, 64, E, fp8=True, bias_var=0.5)
    L = moe.Layer.from_host(w)
    x = g.make_x(62 + T, T, d, bf16=True)
    ws = moe.workspace(L, T)
    ids, wt, lg = moe.route(to_dev_x(x), L, ws, logits=True)
    rows = np.arange(T) if T <= 2048 else np.sort(np.random.default_rng(T).choice(T, 256, replace=False))
    ref = oracle_route(w, x[rows])
    lg = lg.cpu().numpy()[rows]
    err = np.max(np.abs(lg - ref["logits"]), axis=1) / np.max(np.abs(ref["logits"]), axis=1)
    assert err.max() < 3e-5, err.max()
    ids_h, wt_h = ids.cpu().numpy()[rows], wt.cpu().numpy()[rows]
    ok, bad, _ = parity.ids_ok(ids_h, ref["ids"], ref["p"], E)
    assert ok, bad
    same = np.all(ids_h == ref["ids"], axis=1)
    assert np.max(np.abs(wt_h[same] - ref["w"][same])) < 1e-5
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("d,E,T,bf16", [(256, 200, 128, True), (512, 200, 65, True), (768, 384, 17, False),
                                        (1280, 100, 128, True), (2048, 384, 100, False), (512, 512, 64, True),
                                        (256, 1000, 40, True), (512, 1000, 300, True), (512, 480, 200, True)])
def test_router_shapes(moe, d, E, T, bf16):
    """The decode router at every cluster size it takes (d / 256 = 1..8 k-slices), expert counts
    that leave a ragged expert group or need every lane-register count of the warp selection
    (E up to 128, 256, 384, 512, 1024), one and two token blocks, bf16 and fp32 x; the prefill
    routers beside them (tensor-core with fused selection for E <= 512, SIMT + select kernel
    above); each twice in a row on one workspace, so a selection ticket left behind would show
    in the second call."""
    w = g.make_layer(31 + d, d, 64, E, fp8=True, bias_var=0.5)
    L = moe.Layer.from_host(w)
    x = g.make_x(32 + d, T, d, bf16=bf16)
    ws = moe.workspace(L, T)
    ref = oracle_route(w, x)
    first = None
    for _ in range(2):
        ids, wt, lg = moe.route(to_dev_x(x), L, ws, logits=True)
        lg = lg.cpu().numpy()
        err = np.max(np.abs(lg - ref["logits"]), axis=1) / np.max(np.abs(ref["logits"]), axis=1)
        assert err.max() < 3e-5, err.max()
        ok, bad, _ = parity.ids_ok(ids.cpu().numpy(), ref["ids"], ref["p"], E)
        assert ok, bad
        same = np.all(ids.cpu().numpy() == ref["ids"], axis=1)
        assert np.max(np.abs(wt.cpu().numpy()[same] - ref["w"][same])) < 1e-5
        if first is None:
            first = (ids.clone(), wt.clone())
        else:
            assert torch.equal(ids, first[0]) and torch.equal(wt, first[1])
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("T,E,d", [(64, 384, 2048), (100, 384, 1024), (300, 384, 2048), (40, 1000, 256),
                                   (300, 1000, 512)])
def test_selection_only_bias_routing(moe, T, E, d):
    """MOE_BIAS_SELECT on every router: the decode router (mma.sync, ticketed selection), the
    tensor-core router with its epilogue selection, and the SIMT router + selection kernel
    (E = 1000).  Logits carry no bias; ids pass the near-tie rule on the oracle's selection
    probabilities (softmax of logits + bias); weights are the renormalised unbiased softmax."""
    w = g.make_layer(61 + d, d, 64, E, fp8=True, bias_var=0.5)
    L = moe.Layer.from_host(w, bias_mode=moe.binding.BIAS_SELECT)
    x = g.make_x(62 + d, T, d, bf16=True)
    ws = moe.workspace(L, T)
    ids, wt, lg = moe.route(to_dev_x(x), L, ws, logits=True)
    ref = o.layer_forward(o.Layer(w, bias_mode=o.BIAS_SELECT), x, want_probs=True, nthreads=o.default_threads())
    lg = lg.cpu().numpy()
    err = np.max(np.abs(lg - ref["logits"]), axis=1) / np.max(np.abs(ref["logits"]), axis=1)
    assert err.max() < 3e-5, err.max()
    ids = ids.cpu().numpy()
    ok, bad, _ = parity.ids_ok(ids, ref["ids"], ref["p"], E)
    assert ok, bad
    same = np.all(ids == ref["ids"], axis=1)
    assert same.mean() > 0.9
    assert np.max(np.abs(wt.cpu().numpy()[same] - ref["w"][same])) < 1e-5
    # both modes rank on logits + bias, so they pick the same experts; only the weights differ
    score = o.layer_forward(o.Layer(w), x)
    assert np.array_equal(score["ids"], ref["ids"])
    assert np.max(np.abs(score["w"] - ref["w"])) > 1e-2
    assert moe.get_status(ws) == 0


def test_selection_only_bias_layer_free_and_forced(moe, kolibri):
    """A full decode layer (tiled weights, tcgen05 experts) in MOE_BIAS_SELECT: free routing
    against the oracle in that mode, then forced ids with the weights left to the router
    (the unbiased softmax), then the planted 'biased weights' mistake must fail."""
    w = kolibri.w
    L = moe.Layer.from_host(w, bias_mode=moe.binding.BIAS_SELECT)
    T = 64
    x = g.make_x(63, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws)
    check_free_layer(w, x, y, ids, wt, where="select-only free", bias_mode=o.BIAS_SELECT)
    fid = ids.cpu().numpy()
    y2, ids2, _ = moe.forward(to_dev_x(x), L, ws, forced_ids=ids)
    check_forced_layer(w, x, fid, None, y2, ids2, where="select-only forced", bias_mode=o.BIAS_SELECT)
    mut = o.layer_forward(o.Layer(w, bias_mode=o.BIAS_SELECT, mutant=o.MUTANTS["biased_weights"]), x,
                          nthreads=o.default_threads())
    same = np.all(mut["ids"] == fid, axis=1)
    assert same.any() and not parity.weights_ok(wt.cpu().numpy()[same], mut["w"][same])[0]
    assert moe.get_status(ws) == 0


def test_router_fp32_tiny(moe, tiny):
    w, L = tiny
    x = g.make_x(g.SEED_TINY, 32, w.d, bf16=False)
    ws = moe.workspace(L, 32)
    ids, wt, lg = moe.route(to_dev_x(x), L, ws, logits=True)
    ref = o.layer_forward(o.Layer(w), x, want_probs=True)
    assert np.max(np.abs(lg.cpu().numpy() - ref["logits"])) < 1e-5 * np.max(np.abs(ref["logits"]))
    ok, bad, _ = parity.ids_ok(ids.cpu().numpy(), ref["ids"], ref["p"], w.E)
    assert ok, bad


def test_exact_ties_pick_lowest_index(moe):
    w = g.make_layer(21, 256, 64, 384, fp8=True, bias_var=0.5)
    w.Wr[1::2] = w.Wr[0::2]
    w.bias[1::2] = w.bias[0::2]
    L = moe.Layer.from_host(w)
    x = g.make_x(22, 64, 256, bf16=True)
    ws = moe.workspace(L, 64)
    ids, _, _ = moe.route(to_dev_x(x), L, ws)
    ids = ids.cpu().numpy()
    ref = o.layer_forward(o.Layer(w), x, want_probs=True)
    ok, bad, _ = parity.ids_ok(ids, ref["ids"], ref["p"], w.E)
    assert ok, bad
    # wherever both members of a tied pair are chosen, the even (lower) one comes first
    for t in range(64):
        for i in range(6):
            e = ids[t, i]
            if e % 2 == 1 and e - 1 in ids[t]:
                assert list(ids[t]).index(e - 1) < i


# ----------------------------------------------------------------------- dispatch --------

@pytest.fixture(scope="module")
def shape_layer(moe):
    return moe.Layer.from_host(g.make_layer(1, 256, 64, 384, fp8=True, bias_var=None))


@pytest.mark.parametrize("T,mode", [(1, "rand"), (5, "rand"), (64, "rand"), (1023, "rand"), (1024, "rand"),
                                    (1025, "rand"), (5462, "rand"), (8792, "rand"), (8792, "one_expert_set"),
                                    (32769, "one_expert_set")])
def test_dispatch_exact(moe, shape_layer, T, mode):
    rng = np.random.default_rng(T)
    if mode == "rand":
        ids = np.argsort(rng.random((T, 384)), axis=1)[:, :6].astype(np.int32)
    else:
        ids = np.tile(np.array([5, 17, 3, 200, 383, 0], np.int32), (T, 1))
    ref = o.dispatch(ids, 384)
    ws = moe.workspace(shape_layer, T)
    got = moe.dispatch(torch.from_numpy(ids).cuda(), 384, ws)
    for key in ("counts", "offsets", "perm", "pos"):
        assert np.array_equal(got[key].cpu().numpy().reshape(ref[key].shape), ref[key]), key


@pytest.mark.parametrize("T", [1, 700, 5000])
def test_dispatch_exact_many_experts(moe, T):
    """E = 1000 (>= 512): the multi-CTA dispatch at every size, bit-exact against the oracle."""
    E = 1000
    layer = moe.Layer.from_host(g.make_layer(1, 256, 64, E, fp8=True, bias_var=None))
    ids = np.argsort(np.random.default_rng(T + 7).random((T, E)), axis=1)[:, :6].astype(np.int32)
    ref = o.dispatch(ids, E)
    got = moe.dispatch(torch.from_numpy(ids).cuda(), E, moe.workspace(layer, T))
    for key in ("counts", "offsets", "perm", "pos"):
        assert np.array_equal(got[key].cpu().numpy().reshape(ref[key].shape), ref[key]), key


# ------------------------------------------------------------------------- layer ---------

def test_tiny_fp32_layer_free_then_forced(moe, tiny):
    w, L = tiny
    x = g.make_x(g.SEED_TINY, 32, w.d, bf16=False)
    ws = moe.workspace(L, 32)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws)
    _, msg, _ = check_free_layer(w, x, y, ids, wt, where="tiny free")
    y2, ids2, _ = moe.forward(to_dev_x(x), L, ws, forced_ids=ids)
    check_forced_layer(w, x, ids.cpu().numpy(), None, y2, ids2, where="tiny forced")
    assert torch.equal(y2, y), "forced with the recorded ids must reproduce the free run bit for bit"
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("T", [1, 8, 64])
def test_decode_layer(moe, kolibri, T, path):
    w, L = kolibri.w, kolibri.for_path(path)
    x = g.make_x(g.SEED_DECODE, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws, flags=PATHS[path])
    _, msg, _ = check_free_layer(w, x, y, ids, wt, where=f"decode T={T} {path}")
    print(f"T={T} {path}: {msg}")
    y_bf, _, _ = moe.forward(to_dev_x(x), L, ws, y_dtype=torch.bfloat16, flags=PATHS[path])
    assert torch.allclose(y_bf.float(), y, rtol=1e-2, atol=1e-2 * y.abs().max().item())
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("select_only", [False, True])
def test_decode_around_the_one_rank_limit(moe, kolibri, select_only):
    """Free-routing decode at 2, 5, 8, 9, 3, 9 and 1 tokens in turn on one workspace, checked
    against the oracle.  Up to 8 tokens the decode router's rank 0 takes every token and one
    CTA selects and dispatches them from shared memory; at 9 the selection is spread over the
    ranks and a second ticket picks the dispatching CTA.  Switching between the two must leave
    every ticket at zero for the other (a stale ticket would skip or repeat a selection)."""
    w = kolibri.w
    bias_mode = o.BIAS_SELECT if select_only else o.BIAS_SCORE
    L = moe.Layer.from_host(w, bias_mode=moe.binding.BIAS_SELECT) if select_only else kolibri.for_path("tc")
    ws = moe.workspace(L, 9)
    for i, T in enumerate((2, 5, 8, 9, 3, 9, 1)):
        x = g.make_x(g.SEED_DECODE + 300 + i, T, w.d, bf16=True)
        y, ids, wt = moe.forward(to_dev_x(x), L, ws)
        check_free_layer(w, x, y, ids, wt, where=f"T={T} (call {i}, select_only={select_only})", bias_mode=bias_mode)
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("T", [1, 8, 64])
def test_back_to_back_forwards_see_their_own_routing(moe, kolibri, T):
    """Forwards on one workspace with different inputs, launched back to back without a host
    synchronisation: each must use its own routing (tile list, permutation) and its own
    quantised activations, not the previous call's.  At decode the router writes both, and
    the expert kernel that follows overlaps it (programmatic dependent launch)."""
    w, L = kolibri
    ws = moe.workspace(L, T)
    xs = [g.make_x(200 + i, T, w.d, bf16=True) for i in range(3)]
    outs = [moe.forward(to_dev_x(x), L, ws) for x in xs]
    for i, (x, (y, ids, wt)) in enumerate(zip(xs, outs)):
        check_free_layer(w, x, y, ids, wt, where=f"T={T} call {i}")
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("path", sorted(PATHS))
def test_prefill_2048_free_then_4x512_forced(moe, kolibri, path):
    w, L = kolibri.w, kolibri.for_path(path)
    T = 2048
    x = g.make_x(g.SEED_PREFILL, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws, flags=PATHS[path])
    check_free_layer(w, x, y, ids, wt, where=f"prefill 2048 free {path}")
    ys = []
    for c in range(4):
        sl = slice(512 * c, 512 * (c + 1))
        yc, idc, _ = moe.forward(to_dev_x(x[sl]), L, ws, forced_ids=ids[sl].contiguous(), flags=PATHS[path])
        assert torch.equal(idc, ids[sl]), "forced ids must be used bit-exactly"
        ys.append(yc)
    ych = torch.cat(ys)
    ok, msg = parity.outputs_ok(ych.cpu().numpy(), y.cpu().numpy())
    assert ok, f"4x512 forced vs 2048 free: {msg}"
    check_forced_layer(w, x, ids.cpu().numpy(), None, ych, ids, where="prefill 4x512 forced")


@pytest.mark.parametrize("T", [1, 64])
def test_graphed_forward_matches_the_call(moe, kolibri, T):
    """GraphedForward replays (pinned host x -> device, the layer, y -> pinned host) and gives
    what the plain call gives, bit for bit, for new inputs written between replays."""
    w, L = kolibri
    ws = moe.workspace(L, T)
    x_pin = torch.empty((T, w.d), dtype=torch.bfloat16).pin_memory()
    y_pin = torch.empty((T, w.d), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty((T, w.d), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, w.d), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((T, 6), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, 6), dtype=torch.float32, device="cuda")
    step = moe.GraphedForward(xd, L, ws, y, ids, wt, x_host=x_pin, y_host=y_pin)
    for seed in (401, 402):
        x = g.make_x(seed, T, w.d, bf16=True)
        x_pin.copy_(torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16))
        step.replay()
        torch.cuda.synchronize()
        y_ref, ids_ref, w_ref = moe.forward(to_dev_x(x), L, moe.workspace(L, T), y_dtype=torch.bfloat16)
        assert torch.equal(ids, ids_ref) and torch.equal(wt, w_ref)
        assert torch.equal(y_pin.view(torch.int16), y_ref.cpu().view(torch.int16))
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("T", [1, 32])
def test_graphed_stack_matches_the_call(moe, T):
    """GraphedStack replays (input -> residual, a four-layer stack) and gives what the plain
    moe_forward_stack call gives, bit for bit (residual and every layer's ids), for new inputs
    written between replays."""
    layers_w = [g.make_layer(700 + l, 512, 128, 64, fp8=True, bias_var=0.5) for l in range(4)]
    layers = [moe.Layer.from_host(lw) for lw in layers_w]
    ws = moe.workspace(layers[0], T)
    x = torch.empty((T, 512), dtype=torch.bfloat16, device="cuda")
    r = torch.empty_like(x)
    ids = torch.empty((4, T, 6), dtype=torch.int32, device="cuda")
    step = moe.GraphedStack(layers, r, ws, x=x, ids_out=ids)
    for seed in (711, 712):
        xh = to_dev_x(g.make_x(seed, T, 512, bf16=True))
        x.copy_(xh)
        step.replay()
        torch.cuda.synchronize()
        r_ref = xh.clone()
        ids_ref = torch.empty_like(ids)
        moe.forward_stack(layers, r_ref, moe.workspace(layers[0], T), ids_out=ids_ref)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_ref)
        assert torch.equal(r.view(torch.int16), r_ref.view(torch.int16))
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("T", [8192, 9001])
def test_large_prefill_sampled_rows(moe, kolibri, T):
    """Large prefill (128-token tiles, ragged at T = 9001): free routing, 64 sampled rows
    against the oracle run with the GPU's ids forced (every token is independent, so a row
    sample is exact for those rows)."""
    w, L = kolibri
    x = g.make_x(300 + T, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws)
    rows = np.sort(np.random.default_rng(T).choice(T, 64, replace=False))
    ref = o.layer_forward(o.Layer(w), x[rows], forced_ids=ids.cpu().numpy()[rows], nthreads=o.default_threads())
    ok, msg = parity.outputs_ok(y.cpu().numpy()[rows], ref["y"])
    assert ok, f"T={T}: {msg}"
    assert moe.get_status(ws) == 0


def _edge_ids(counts, T, E=384, first_filler=100):
    """Forced ids for T tokens in which edge expert j (ids 10 + j) holds exactly counts[j] rows
    (tokens 0 .. counts[j] - 1); each token's remaining slots take filler experts
    first_filler, first_filler + 1, ... in turn (never an edge expert)."""
    ids = np.zeros((T, 6), np.int32)
    nxt = 0
    n_fill = E - first_filler
    for t in range(T):
        row = [10 + j for j, c in enumerate(counts) if t < c]
        while len(row) < 6:
            row.append(first_filler + nxt % n_fill)
            nxt += 1
        ids[t] = row
    return ids


def _check_sampled_forced(w, x, fid, y, ids, extra_rows, where, n=40):
    """Forced ids bit-exact; outputs of a seeded row sample plus the given rows against the
    oracle (every token is independent, so a row sample is exact for those rows)."""
    assert np.array_equal(ids.cpu().numpy(), fid), f"{where}: forced ids not bit-exact"
    T = x.shape[0]
    rows = np.unique(np.concatenate([np.random.default_rng(T).choice(T, n, replace=False),
                                     np.array([r for r in extra_rows if 0 <= r < T], np.int64)]))
    ref = o.layer_forward(o.Layer(w), x[rows], forced_ids=fid[rows], nthreads=o.default_threads())
    ok, msg = parity.outputs_ok(y.float().cpu().numpy()[rows], ref["y"])
    assert ok, f"{where}: {msg}"


@pytest.mark.parametrize("path", sorted(PATHS))
def test_one_expert_set_holds_every_row(moe, kolibri, path):
    """The pages' first wave, 8 x 1,099 x 6 = 52,752 routed rows ("We Ported Aleph Alpha's
    Kolibri to a MacBook. Our Own Gate Said No.", section 3, update of 5 October), all on one
    set of six experts: 8,792 tokens forced to the same experts, so six groups of 8,792 rows and
    the shared expert's 8,792 (long runs of full tiles of one expert; 8,792 is not a multiple of
    the tile height)."""
    w, L = kolibri.w, kolibri.for_path(path)
    T = 8 * 1099
    fid = np.tile(np.array([[200, 3, 377, 41, 96, 250]], np.int32), (T, 1))
    assert fid.size == 52752
    x = g.make_x(401, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, _ = moe.forward(to_dev_x(x), L, ws, forced_ids=torch.from_numpy(fid).cuda(), flags=PATHS[path])
    _check_sampled_forced(w, x, fid, y, ids, [0, 127, 128, T - 1], f"52,752 rows, {path}")
    assert moe.get_status(ws) == 0


def test_grouped_gemm_row_count_edges(moe, kolibri):
    """Groups of exactly 32,767, 32,768, 32,769, 32,832, 33,000 and 34,000 rows in one call: the
    row counts around 2^15 at which the pages' sorted grouped GEMM went wrong (32,769, 33,000,
    34,000) or stayed right (32,768, 32,832) ("We Ported Aleph Alpha's Kolibri to a MacBook. Our
    Own Gate Said No.", section 3, update of 5 October), 34,000 tokens forced so that six experts
    hold those counts, on the tcgen05 grouped GEMMs.  Rows at every group boundary are among the
    sampled rows."""
    w, L = kolibri.w, kolibri.tiled
    counts = [32767, 32768, 32769, 32832, 33000, 34000]
    T = max(counts)
    fid = _edge_ids(counts, T)
    per_expert = np.bincount(fid.ravel(), minlength=384)
    assert [int(per_expert[10 + j]) for j in range(6)] == counts
    x = g.make_x(402, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, _ = moe.forward(to_dev_x(x), L, ws, forced_ids=torch.from_numpy(fid).cuda(), flags=PATHS["tc"])
    edges = [c + dd for c in counts for dd in (-1, 0)]
    _check_sampled_forced(w, x, fid, y, ids, edges, "row-count edges")
    assert moe.get_status(ws) == 0


@pytest.mark.parametrize("path", sorted(PATHS))
def test_batched_decode_zipf_forced(moe, kolibri, path):
    w, L = kolibri.w, kolibri.for_path(path)
    T = 128
    x = g.make_x(g.SEED_ZIPF, T, w.d, bf16=True)
    fid = g.zipf_ids(g.SEED_ZIPF, 0, T, 384, 6, 1.1)
    fw = g.dirichlet_w(g.SEED_ZIPF, 0, T, 6)
    ws = moe.workspace(L, T)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws, forced_ids=torch.from_numpy(fid).cuda(),
                             forced_w=torch.from_numpy(fw).cuda(), flags=PATHS[path])
    assert np.array_equal(wt.cpu().numpy(), fw)
    _, msg = check_forced_layer(w, x, fid, fw, y, ids, where="zipf T=128")
    print(msg)


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("T", [0, 37, 333, 1500])
def test_ragged_token_counts(moe, kolibri, T, path):
    w, L = kolibri.w, kolibri.for_path(path)
    x = g.make_x(77, max(T, 1), w.d, bf16=True)[:T]
    ws = moe.workspace(L, max(T, 1))
    y, ids, wt = moe.forward(to_dev_x(x), L, ws, flags=PATHS[path])
    if T == 0:
        assert y.shape == (0, w.d)
        return
    check_free_layer(w, x, y, ids, wt, where=f"ragged T={T}")


def test_bad_forced_ids_are_reported_and_skipped(moe, kolibri):
    w, L = kolibri
    T = 4
    x = g.make_x(78, T, w.d, bf16=True)
    fid = np.array([[1, 2, 3, 4, 5, 6], [1, 1, 3, 4, 5, 6], [1, 2, 3, 4, 5, 999], [7, 8, 9, 10, 11, -3]], np.int32)
    fw = np.full((T, 6), 1 / 6, np.float32)
    ws = moe.workspace(L, T)
    y, ids, _ = moe.forward(to_dev_x(x), L, ws, forced_ids=torch.from_numpy(fid).cuda(),
                            forced_w=torch.from_numpy(fw).cuda())
    assert moe.get_status(ws) == -4
    assert moe.get_status(ws) == 0  # cleared
    ids = ids.cpu().numpy()
    assert ids[1, 1] == -1 and ids[2, 5] == -1 and ids[3, 5] == -1 and np.all(ids[0] == fid[0])
    # a rejected slot contributes nothing: compare with the oracle on zero weight there
    fw2 = fw.copy()
    fid2 = fid.copy()
    for t, i in ((1, 1), (2, 5), (3, 5)):
        fw2[t, i] = 0
        fid2[t, i] = 100 + t  # any valid unused id with weight 0
    ref = o.layer_forward(o.Layer(w), x, forced_ids=fid2, forced_w=fw2)
    ok, msg = parity.outputs_ok(y.cpu().numpy(), ref["y"])
    assert ok, msg


def test_device_wait_timeout_is_reported_and_context_survives(moe, kolibri):
    """A wait that can never complete gives up after its limit, reports MOE_ERR_TIMEOUT
    through the status record, and the next forward on the same context is correct."""
    w, L = kolibri
    ws = moe.workspace(L, 8)
    assert moe.get_status(ws) == 0
    moe.binding.selftest_wait_timeout(ws, 10000)
    assert moe.get_status(ws) == -5
    assert moe.get_status(ws) == 0  # cleared
    x = g.make_x(81, 8, w.d, bf16=True)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws)
    check_free_layer(w, x, y, ids, wt, where="after timeout self-test")
    assert moe.get_status(ws) == 0


def test_rows_do_not_depend_on_other_rows(moe, kolibri):
    """Batch parity: a token's output is the same alone, in a batch, and in a permuted batch
    (the batched expert layer on the pages returned wrong rows depending on the batch)."""
    w, L = kolibri
    T = 96
    x = g.make_x(79, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, _ = moe.forward(to_dev_x(x), L, ws)
    perm = np.random.default_rng(0).permutation(T)
    yp, idp, _ = moe.forward(to_dev_x(x[perm]), L, ws)
    assert torch.equal(idp, ids[perm])
    ok, msg = parity.outputs_ok(yp.cpu().numpy(), y[perm].cpu().numpy(), max_frac=1e-4, rl2=1e-5)
    assert ok, msg
    for t in (0, 50, 95):
        y1, id1, _ = moe.forward(to_dev_x(x[t:t + 1]), L, ws)
        assert torch.equal(id1[0], ids[t])
        ok, msg = parity.outputs_ok(y1.cpu().numpy(), y[t:t + 1].cpu().numpy(), max_frac=1e-4, rl2=1e-5)
        assert ok, msg


@pytest.mark.parametrize("name", ["unbiased_select", "no_renorm", "no_shared", "swap_gate_up", "scale_axis",
                                  "bf16_router"])
def test_planted_oracle_mistakes_fail_against_the_gpu(moe, kolibri, name):
    """Controls: the GPU result must FAIL parity against an oracle with a planted mistake."""
    w, L = kolibri
    T = 64
    x = g.make_x(80, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws)
    _, _, lg = moe.route(to_dev_x(x), L, ws, logits=True)
    mut = o.Layer(w, mutant=o.MUTANTS[name])
    ref = o.layer_forward(mut, x, want_probs=True, nthreads=o.default_threads())
    fails = []
    if np.max(np.abs(lg.cpu().numpy() - ref["logits"])) > 1e-5 * np.max(np.abs(ref["logits"])):
        fails.append("logits")
    ok, _, _ = parity.ids_ok(ids.cpu().numpy(), ref["ids"], ref["p"], w.E)
    if not ok:
        fails.append("ids")
    same = np.all(ids.cpu().numpy() == ref["ids"], axis=1)
    if same.any():
        if not parity.weights_ok(wt.cpu().numpy()[same], ref["w"][same])[0]:
            fails.append("weights")
        if not parity.outputs_ok(y.cpu().numpy()[same], ref["y"][same])[0]:
            fails.append("outputs")
    assert fails, f"planted mistake {name} went unnoticed"
