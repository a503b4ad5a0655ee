"""Prefill-sized calls through the tcgen05 grouped GEMMs against the CPU oracle, on the
Kolibri-shaped layer (d = 2048, ffn = 640, 384 experts + 1 shared, bias N(0, 0.5)), at the
tile shapes where the kernels change behaviour: each MMA's N is a tile's row count rounded up
to 16 (tiles of up to 128 token rows from 1025 tokens), and rows past a tile's end are not
gathered.  Every token is independent, so sampled rows checked against the oracle run with the
same (forced) ids are exact for those rows.  Tolerances as for every layer test: forced ids
bit-exact, outputs max|err| <= 2e-2 max|y_ref| and relative L2 <= 5e-3."""
import numpy as np
import pytest
import torch

from gen import moegen as g
from oracle import oracle as o
from tests import parity
from tests.gpu_helpers import to_dev_x

pytestmark = pytest.mark.gpu

WIDE_TILE_MIN_T = 1025  # from this many tokens the GEMM tiles hold up to 128 token rows


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import routed_expert_layer_fp32_gb300 as m
    return m


@pytest.fixture(scope="module")
def layer(moe):
    w = g.kolibri_layer(g.SEED_PREFILL)
    return w, moe.Layer.from_host(w)


def _sampled(w, x, fid, fw, y, rows, where):
    ref = o.layer_forward(o.Layer(w), x[rows], forced_ids=fid[rows], forced_w=None if fw is None else fw[rows],
                          nthreads=o.default_threads())
    ok, msg = parity.outputs_ok(y.float().cpu().numpy()[rows], ref["y"])
    assert ok, f"{where}: {msg}"


@pytest.mark.parametrize("T", [WIDE_TILE_MIN_T - 1, WIDE_TILE_MIN_T, 5000])
def test_threshold_free_routing_sampled_rows(moe, layer, T):
    """Either side of the change from 64- to 128-row tiles, and a call of 5000 tokens: free
    routing, then 48 sampled rows against the oracle with the GPU's ids forced."""
    w, L = layer
    x = g.make_x(g.SEED_PREFILL + 500 + T, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, _ = moe.forward(to_dev_x(x), L, ws, y_dtype=torch.float32)
    rows = np.sort(np.random.default_rng(T).choice(T, 48, replace=False))
    _sampled(w, x, ids.cpu().numpy(), None, y, rows, f"T={T}")
    assert moe.get_status(ws) == 0


def _edge_ids(counts, T, E=384, first_filler=100):
    """Forced ids in which edge expert j (id 10 + j) holds exactly counts[j] rows (tokens
    0 .. counts[j] - 1); the other slots cycle through filler experts 100 .. E - 1."""
    ids = np.zeros((T, 6), np.int32)
    nxt = 0
    n_fill = E - first_filler
    for t in range(T):
        row = [10 + j for j, c in enumerate(counts) if t < c][:6]
        while len(row) < 6:
            row.append(first_filler + nxt % n_fill)
            nxt += 1
        ids[t] = row
    return ids


@pytest.mark.parametrize("counts", [[1, 15, 16, 17, 127, 128], [129, 255, 256, 257, 511, 513]])
def test_tile_heights_around_the_mma_width(moe, layer, counts):
    """Groups of 1, 15, 16, 17, 127, 128, 129, 255, 256, 257, 511 and 513 rows: tiles of 128
    rows and ragged last tiles whose MMA width rounds their rows up to 16 (a last tile of 17
    rows: 32 columns, 15 of them padding).  Every row of the small groups and every tile
    boundary is among the checked rows."""
    w, L = layer
    T = 4096
    fid = _edge_ids(counts, T)
    per_expert = np.bincount(fid.ravel(), minlength=384)
    assert [int(per_expert[10 + j]) for j in range(len(counts))] == counts
    x = g.make_x(g.SEED_PREFILL + 600 + counts[0], T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, _ = moe.forward(to_dev_x(x), L, ws, forced_ids=torch.from_numpy(fid).cuda(), y_dtype=torch.float32)
    assert np.array_equal(ids.cpu().numpy(), fid)
    edges = {r for c in counts for r in (c - 2, c - 1, c) if 0 <= r < T}
    edges |= {r for b in (7, 8, 15, 16, 63, 64, 127, 128, 255, 256) for r in (b - 1, b) if 0 <= r < T}
    rows = np.array(sorted(edges | set(np.random.default_rng(counts[0]).choice(T, 16, replace=False).tolist())))
    _sampled(w, x, fid, None, y, rows, f"tile heights {counts}")
    assert moe.get_status(ws) == 0


def test_zipf_forced_prefill(moe, layer):
    """Zipf(1.1) expert popularity over 384 experts with Dirichlet routing weights at 8192
    tokens: a few experts fill many full tiles, most hold a ragged handful of rows."""
    w, L = layer
    T = 8192
    fid = g.zipf_ids(g.SEED_ZIPF, 7, T, 384, 6, 1.1)
    fw = g.dirichlet_w(g.SEED_ZIPF, 7, T, 6)
    x = g.make_x(g.SEED_ZIPF + 700, T, w.d, bf16=True)
    ws = moe.workspace(L, T)
    y, ids, wt = moe.forward(to_dev_x(x), L, ws, forced_ids=torch.from_numpy(fid).cuda(),
                             forced_w=torch.from_numpy(fw).cuda(), y_dtype=torch.float32)
    assert np.array_equal(ids.cpu().numpy(), fid)
    assert np.array_equal(wt.cpu().numpy(), fw)
    counts = np.bincount(fid.ravel(), minlength=384)
    assert counts.max() > 6 * 128  # the most popular expert spans several full tiles
    rows = np.sort(np.random.default_rng(8).choice(T, 64, replace=False))
    _sampled(w, x, fid, fw, y, rows, "zipf prefill")
    assert moe.get_status(ws) == 0


def test_prefill_repeats_bit_exactly(moe, layer):
    """Two calls on the same input give the same bits: every sum is taken in a fixed order
    whatever the timing of the CTAs."""
    w, L = layer
    T = 4096 + 123
    x = to_dev_x(g.make_x(g.SEED_PREFILL + 800, T, w.d, bf16=True))
    ws = moe.workspace(L, T)
    y1, ids1, _ = moe.forward(x, L, ws)
    y2, ids2, _ = moe.forward(x, L, ws)
    assert torch.equal(ids1, ids2)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert moe.get_status(ws) == 0
