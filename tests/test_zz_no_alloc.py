"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a host runtime that owns all device memory through its own pool, or a serving
loop where an allocation, which may synchronise the device, is not allowed) cannot hand
moe_route a workspace.  The variant keeps its scratch in a fixed array inside the library.

This test calls it through the C ABI three times in a row on the Kolibri-shaped router
(d = 2048, 384 experts, bias N(0, 0.5)), with different inputs and sizes, so every call after
the first starts from the previous call's leftovers: 2048 tokens (the tiled SIMT router),
then 8 and 1 token (the warp-per-expert router).  Each result is checked against the CPU oracle
(ids within the near-tie rule, weights within 1e-5 wherever the ids agree) and against
moe_route on the same inputs.  It also checks that sizes beyond the array and an unknown bias
mode are refused.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests import parity
from tests.gpu_helpers import oracle_route, to_dev_x

pytestmark = pytest.mark.gpu


def _router_only_layer(moe, w, dummy):
    """A layer descriptor whose router tensors are real and whose expert pointers all name one
    small dummy buffer: routing reads only the router (d = 2048, ffn = 640, E4M3 row layout,
    so moe_route's checks pass too)."""
    Wr = torch.from_numpy(w.Wr).cuda()
    b = torch.from_numpy(w.bias).cuda()
    p = dummy.data_ptr()
    c = moe.binding.MoeLayerC(w.d, w.ffn, w.E, 6, moe.binding.MOE_E4M3, Wr.data_ptr(), b.data_ptr(), p, p, p, p, p, p,
                              p, p, moe.binding.LAYOUT_ROWS, moe.binding.BIAS_SCORE)
    return c, (Wr, b)


def test_route_noalloc_against_oracle_on_calls_in_a_row():
    import __graft_entry__
    __graft_entry__.build()
    import routed_expert_layer_fp32_gb300 as moe
    from gen import moegen as g

    lib = moe.binding.lib()
    w = g.sparse_layer(93, [], d=2048, ffn=640, E=384, bias_var=0.5)
    dummy = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    c, keep = _router_only_layer(moe, w, dummy)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, T in enumerate((2048, 8, 1)):
        x_h = g.make_x(94 + call, T, 2048, bf16=True)
        x = to_dev_x(x_h)
        ref = oracle_route(w, x_h)
        ids = torch.full((T, 6), -7, dtype=torch.int32, device="cuda")
        wt = torch.full((T, 6), -7.0, dtype=torch.float32, device="cuda")
        rc = lib.moe_route_noalloc(x.data_ptr(), moe.binding.MOE_BF16, T, ctypes.byref(c), 6, ids.data_ptr(),
                                   wt.data_ptr(), stream)
        assert rc == 0, moe.binding.status_string(rc)
        # the same routing through moe_route (workspace allocated here, by the test)
        nbytes = lib.moe_workspace_bytes(ctypes.byref(c), T)
        assert nbytes > 0
        ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        ids_r = torch.empty((T, 6), dtype=torch.int32, device="cuda")
        wt_r = torch.empty((T, 6), dtype=torch.float32, device="cuda")
        rc = lib.moe_route(x.data_ptr(), moe.binding.MOE_BF16, T, ctypes.byref(c), 6, ids_r.data_ptr(),
                           wt_r.data_ptr(), None, ws.data_ptr(), nbytes, stream)
        assert rc == 0, moe.binding.status_string(rc)
        torch.cuda.synchronize()
        ids_h, wt_h = ids.cpu().numpy(), wt.cpu().numpy()
        ok, bad, _ = parity.ids_ok(ids_h, ref["ids"], ref["p"], 384)
        assert ok, f"call {call} (T={T}): ids outside the near-tie rule: {bad}"
        same = np.all(ids_h == ref["ids"], axis=1)
        assert same.mean() > 0.99, f"call {call}: {int((~same).sum())} tokens differ from the oracle"
        okw, msg = parity.weights_ok(wt_h[same], ref["w"][same])
        assert okw, f"call {call}: weights against the oracle: {msg}"
        ids_rh, wt_rh = ids_r.cpu().numpy(), wt_r.cpu().numpy()
        ok, bad, _ = parity.ids_ok(ids_rh, ref["ids"], ref["p"], 384)
        assert ok, f"call {call}: moe_route ids outside the near-tie rule: {bad}"
        both = np.all(ids_h == ids_rh, axis=1)
        okw, msg = parity.weights_ok(wt_h[both], wt_rh[both])
        assert okw, f"call {call}: weights against moe_route: {msg}"
    # refused before any launch: a size beyond the built-in scratch, an unknown bias mode
    too_many = (1 << 20) // 384 + 1
    rc = lib.moe_route_noalloc(x.data_ptr(), moe.binding.MOE_BF16, too_many, ctypes.byref(c), 6, ids.data_ptr(),
                               wt.data_ptr(), stream)
    assert rc == -3
    c.bias_mode = 7
    rc = lib.moe_route_noalloc(x.data_ptr(), moe.binding.MOE_BF16, 1, ctypes.byref(c), 6, ids.data_ptr(),
                               wt.data_ptr(), stream)
    assert rc == -1
    del keep
