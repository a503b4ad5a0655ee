"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a host runtime that owns all device memory through its own pool, or a serving
loop where an allocation is not allowed) cannot hand moe_route a workspace.  The variant
keeps its scratch in a fixed array inside the library.  This test calls it through the C
ABI twice in a row (different inputs and sizes, so the second call starts from the first
call's leftovers) and checks each result against moe_route on the same inputs: ids equal,
weights within the tolerance the other routing tests use.  It also checks that a size beyond
the array is rejected.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_route_noalloc_matches_route_on_two_calls_in_a_row():
    import __graft_entry__
    __graft_entry__.build()
    import routed_expert_layer_fp32_gb300 as moe
    from gen import moegen as g

    lib = moe.binding.lib()
    w = g.make_layer(91, 256, 64, 384, fp8=True, bias_var=0.5)
    L = moe.Layer.from_host(w)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, T in enumerate((64, 37)):
        x = torch.from_numpy(g.make_x(92 + call, T, 256, bf16=True).view(np.int16).copy()).cuda().view(torch.bfloat16)
        ws = moe.workspace(L, T)
        ids_ref, w_ref, _ = moe.route(x, L, ws)
        ids = torch.full((T, 6), -7, dtype=torch.int32, device="cuda")
        wt = torch.full((T, 6), -7.0, dtype=torch.float32, device="cuda")
        rc = lib.moe_route_noalloc(x.data_ptr(), moe.binding.MOE_BF16, T, L.ref, 6, ids.data_ptr(), wt.data_ptr(),
                                   stream)
        assert rc == 0, moe.binding.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(ids, ids_ref), f"call {call}: ids differ from moe_route"
        assert float((wt - w_ref).abs().max()) <= 1e-5, f"call {call}: weights differ from moe_route"
    # a size beyond the built-in scratch is refused before any launch
    too_many = (1 << 20) // 384 + 1
    rc = lib.moe_route_noalloc(x.data_ptr(), moe.binding.MOE_BF16, too_many, L.ref, 6, ids.data_ptr(), wt.data_ptr(),
                               stream)
    assert rc == -3
