"""4-bit expert weights (E2M1 codes with per-row fp32 scales, the library's reading of the K4
builds of "We Stopped the Kolibri Benchmark Before Scoring One Answer", section "What this
means if you want Kolibri on a Mac") through the C ABI against the CPU oracle in its E2M1
mode, on the Kolibri-shaped layer (d = 2048, ffn = 640, 384 experts + 1 shared, bias
N(0, 0.5)).  The codes enter tcgen05.mma kind::f8f6f4 as the A operand beside E4M3
activations.  Tolerances as for the FP8 layer: forced ids bit-exact, free ids within the
near-tie rule, outputs max|err| <= 2e-2 max|y_ref| and relative L2 <= 5e-3."""
import numpy as np
import pytest
import torch

from gen import moegen as g
from oracle import oracle as o
from tests import parity
from tests.gpu_helpers import check_forced_layer, check_free_layer, to_dev_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import routed_expert_layer_fp32_gb300 as m
    return m


@pytest.fixture(scope="module")
def w4(moe):
    w = g.kolibri_layer(g.SEED_DECODE, fp4=True)
    return w, moe.Layer.from_host(w)


def test_pack_matches_the_documented_4bit_tiled_layout(moe):
    """moe_pack_weights on E2M1 rows against the layout include/libmoe.h states, built with
    numpy: 8 KB tiles of 128 rows x 64 bytes, rows in order, the 8-bit layout's tile order."""
    w = g.make_layer(41, 256, 128, 3, fp8=False, bias_var=None, fp4=True)
    L = moe.Layer.from_host(w)
    got = L.tensors["w_gate_up"].cpu().numpy().reshape(-1)
    E, F, d = 3, 128, 256
    KT, NB = d // 128, F // 128
    want = np.empty_like(got)
    t = 0
    for e in range(E):
        for n in range(NB):
            for j in range(KT):
                for half in range(2):
                    rows = w.Wgu[e, half, n * 128:(n + 1) * 128, j * 64:(j + 1) * 64]
                    want[t * 8192:(t + 1) * 8192] = rows.reshape(-1)
                    t += 1
    assert np.array_equal(got, want)
    got_d = L.tensors["w_down"].cpu().numpy().reshape(-1)
    want_d = np.concatenate([w.Wd[e, m * 128:(m + 1) * 128, j * 64:(j + 1) * 64].reshape(-1)
                             for e in range(E) for m in range(d // 128) for j in range(F // 128)])
    assert np.array_equal(got_d, want_d)


@pytest.mark.parametrize("T", [1, 8, 64])
def test_w4_decode_layer_free_then_forced(moe, w4, T):
    w, L = w4
    x = g.make_x(g.SEED_DECODE + 100, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws, y_dtype=torch.float32)
    _, msg, _ = check_free_layer(w, x, y, ids, wt, where=f"w4 T={T}")
    y2, ids2, _ = moe.forward(to_dev_x(x), L, ws, forced_ids=ids, y_dtype=torch.float32)
    check_forced_layer(w, x, ids.cpu().numpy(), None, y2, ids2, where=f"w4 forced T={T}")
    assert moe.get_status(ws) == 0
    print(msg)


def test_w4_zipf_forced_batched_decode(moe, w4):
    w, L = w4
    T = 128
    x = g.make_x(g.SEED_ZIPF, T, w.d, bf16=True)
    fid = g.zipf_ids(g.SEED_ZIPF, 0, T, 384, 6, 1.1)
    fw = g.dirichlet_w(g.SEED_ZIPF, 0, T, 6)
    ws = moe.workspace(L, T)
    y, ids, _ = moe.forward(to_dev_x(x), L, ws, forced_ids=torch.from_numpy(fid).cuda(),
                            forced_w=torch.from_numpy(fw).cuda(), y_dtype=torch.float32)
    check_forced_layer(w, x, fid, fw, y, ids, where="w4 zipf T=128")


@pytest.mark.parametrize("T", [333, 2048])
def test_w4_prefill_sampled_rows(moe, w4, T):
    """Prefill-sized calls (64- and 128-token tiles): free routing, sampled rows against the
    oracle run with the GPU's ids forced (every token is independent)."""
    w, L = w4
    x = g.make_x(g.SEED_PREFILL + 100, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, _ = moe.forward(to_dev_x(x), L, ws, y_dtype=torch.float32)
    rows = np.sort(np.random.default_rng(T).choice(T, 48, replace=False))
    ref = o.layer_forward(o.Layer(w), x[rows], forced_ids=ids.cpu().numpy()[rows], nthreads=o.default_threads())
    ok, msg = parity.outputs_ok(y.cpu().numpy()[rows], ref["y"])
    assert ok, f"w4 T={T}: {msg}"
    assert moe.get_status(ws) == 0


def test_w4_layer_differs_from_the_fp8_layer_by_the_coarser_rounding(moe, w4):
    """The 4-bit layer and the FP8 layer of the same seed agree loosely (both quantise the same
    Gaussian weights): a mix-up of the two formats' scales or codes on the GPU would be far off."""
    w, L = w4
    w8 = g.kolibri_layer(g.SEED_DECODE)
    L8 = moe.Layer.from_host(w8)
    T = 16
    x = to_dev_x(g.make_x(g.SEED_DECODE + 200, T, w.d, bf16=True))
    ws = moe.workspace(L8, T)
    y8, ids8, _ = moe.forward(x, L8, ws, y_dtype=torch.float32)
    y4, _, _ = moe.forward(x, L, ws, forced_ids=ids8, y_dtype=torch.float32)
    rel = parity.rel_l2(y4.cpu().numpy(), y8.cpu().numpy())
    assert 0.03 < rel < 0.3, rel
