"""The MOE_DEBUG build of libmoe (every kernel checks the indices it reads from the tile list,
perm and pos, records MOE_ERR_INDEX on a bad one and keeps the access inside its buffer): on
small layers it must run clean (no index check fires) and agree with the oracle like the
release build, on both expert paths, with free and forced routing, ragged token counts, and
forced ids that the layer drops (slots marked -1, which the checks must not mistake for bad
rows)."""
import numpy as np
import pytest
import torch

from gen import moegen as g
from tests.gpu_helpers import check_forced_layer, check_free_layer, to_dev_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_moe():
    import __graft_entry__
    __graft_entry__.build()
    from routed_expert_layer_fp32_gb300 import _build, binding
    path = _build.build(debug=True)
    binding.use_library(path)
    import routed_expert_layer_fp32_gb300 as moe
    try:
        yield moe
    finally:
        binding.use_library(None)


@pytest.fixture(scope="module")
def small(debug_moe):
    w = g.make_layer(71, 512, 128, 64, fp8=True, bias_var=0.5)
    return w, debug_moe.Layer.from_host(w), debug_moe.Layer.from_host(w, tiled=False)


@pytest.mark.parametrize("T", [1, 37, 300])
@pytest.mark.parametrize("path", ["tc", "stream"])
def test_debug_build_runs_clean_and_matches_oracle(debug_moe, small, T, path):
    w, tiled, rows = small
    L = tiled if path == "tc" else rows
    x = g.make_x(72 + T, T, w.d, bf16=True)
    ws = debug_moe.workspace(L, T)
    y, ids, wt = debug_moe.forward(to_dev_x(x), L, ws, y_dtype=torch.float32, flags=1 if path == "stream" else 2)
    assert debug_moe.get_status(ws) == 0, "an index check fired"
    check_free_layer(w, x, y, ids, wt, where=f"debug build T={T} {path}")
    y2, ids2, _ = debug_moe.forward(to_dev_x(x), L, ws, forced_ids=ids, y_dtype=torch.float32,
                                    flags=1 if path == "stream" else 2)
    assert debug_moe.get_status(ws) == 0, "an index check fired (forced)"
    check_forced_layer(w, x, ids.cpu().numpy(), None, y2, ids2, where=f"debug build forced T={T} {path}")


def test_debug_build_dropped_forced_slots_are_not_index_errors(debug_moe, small):
    w, tiled, _ = small
    T = 16
    x = g.make_x(80, T, w.d, bf16=True)
    fid = np.tile(np.arange(6, dtype=np.int32), (T, 1))
    fid[3, 2] = 999   # out of range
    fid[5, 4] = fid[5, 1]  # repeated within the token
    ws = debug_moe.workspace(tiled, T)
    debug_moe.forward(to_dev_x(x), tiled, ws, forced_ids=torch.from_numpy(fid).cuda(), y_dtype=torch.float32)
    assert debug_moe.get_status(ws) == -4  # MOE_ERR_BAD_FORCED_ID, not MOE_ERR_INDEX (-7)


def test_tiny_fp32_layer_debug_build(debug_moe):
    w = g.tiny_layer()
    L = debug_moe.Layer.from_host(w)
    x = g.make_x(g.SEED_TINY, 32, w.d, bf16=False)
    ws = debug_moe.workspace(L, 32)
    y, ids, wt = debug_moe.forward(to_dev_x(x), L, ws, y_dtype=torch.float32)
    assert debug_moe.get_status(ws) == 0
    check_free_layer(w, x, y, ids, wt, where="debug build tiny fp32")
