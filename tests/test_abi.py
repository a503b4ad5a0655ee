"""The C ABI without a GPU: the library loads, exports every symbol include/libmoe.h declares,
sizes workspaces on the host, and rejects invalid arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "libmoe.h")


@pytest.fixture(scope="module")
def lib():
    from routed_expert_layer_fp32_gb300 import _build, binding
    _build.build()
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_documented_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_forward", "moe_forward_stack", "moe_workspace_bytes", "moe_get_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from routed_expert_layer_fp32_gb300 import binding
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(binding.EXPORTS) == names


def _layer(binding, d=2048, F=640, E=384, k=6, wdt=2, null_scales=False):
    p = 1 << 20  # a fake, 16-byte aligned address: never dereferenced by host validation
    s = 0 if null_scales else p
    return binding.MoeLayerC(d, F, E, k, wdt, p, 0, p, s, p, s, p, s, p, s)


def test_workspace_bytes_on_host(lib):
    from routed_expert_layer_fp32_gb300 import binding
    L = _layer(binding)
    small = lib.moe_workspace_bytes(ctypes.byref(L), 1)
    big = lib.moe_workspace_bytes(ctypes.byref(L), 16384)
    assert 0 < small < big
    # the largest buffers: the per-row expert outputs [7T, d] (bf16 for an E4M3 layer) and the
    # E4M3 activation rows [T, d] (token order)
    assert big >= 7 * 16384 * 2048 * 2 + 16384 * 2048
    # an fp32 layer keeps fp32 expert outputs and fp32 activation rows
    big32 = lib.moe_workspace_bytes(ctypes.byref(_layer(binding, wdt=0)), 16384)
    assert big32 >= 7 * 16384 * 2048 * 4 + 16384 * 2048 * 4
    assert lib.moe_workspace_bytes(ctypes.byref(_layer(binding, k=5)), 8) == 0
    assert lib.moe_workspace_bytes(None, 8) == 0


def test_host_validation_rejects_before_any_launch(lib):
    from routed_expert_layer_fp32_gb300 import binding
    good = _layer(binding)
    p, ws = 1 << 20, 1 << 21
    fwd = lib.moe_forward
    # k != 6 is unsupported
    assert fwd(p, 1, 4, ctypes.byref(_layer(binding, k=8)), None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -2
    # null layer / null x / misaligned y / forced_w without forced_ids / bad dtype / bad flags
    assert fwd(p, 1, 4, None, None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -1
    assert fwd(None, 1, 4, ctypes.byref(good), None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -1
    assert fwd(p, 1, 4, ctypes.byref(good), None, None, None, None, p + 4, 0, 0, ws, 1 << 40, None) == -1
    assert fwd(p, 1, 4, ctypes.byref(good), None, p, None, None, p, 0, 0, ws, 1 << 40, None) == -1
    assert fwd(p, 7, 4, ctypes.byref(good), None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -1
    assert fwd(p, 1, 4, ctypes.byref(good), None, None, None, None, p, 0, 64, ws, 1 << 40, None) == -1
    # FP8 layer without scales, unsupported shapes
    assert fwd(p, 1, 4, ctypes.byref(_layer(binding, null_scales=True)), None, None, None, None, p, 0, 0, ws,
               1 << 40, None) == -1
    assert fwd(p, 1, 4, ctypes.byref(_layer(binding, d=2000)), None, None, None, None, p, 0, 0, ws, 1 << 40,
               None) == -2
    # workspace too small
    assert fwd(p, 1, 4, ctypes.byref(good), None, None, None, None, p, 0, 0, ws, 1024, None) == -3
    # T == 0 is a no-op
    assert fwd(p, 1, 0, ctypes.byref(good), None, None, None, None, p, 0, 0, ws, 0, None) == 0
    # negative T
    assert fwd(p, 1, -1, ctypes.byref(good), None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -1
    # route: k mismatch; stack: empty
    assert lib.moe_route(p, 1, 4, ctypes.byref(good), 5, p, p, None, ws, 1 << 40, None) == -2
    arr = (binding.MoeLayerC * 1)(good)
    assert lib.moe_forward_stack(arr, 0, p, 4, None, 0, ws, 1 << 40, None) == -1
    assert lib.moe_forward_stack(arr, 1, p, 4, None, 0, ws, 16, None) == -3
    assert lib.moe_dispatch(p, 4, 384, 7, p, p, p, p, ws, 1 << 40, None) == -2
    # weight layouts: an unknown layout, a tiled fp32 layer, a tiled layer with ffn % 128 != 0
    bad_layout = _layer(binding)
    bad_layout.w_layout = 5
    assert fwd(p, 1, 4, ctypes.byref(bad_layout), None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -1
    tiled_f32 = _layer(binding, wdt=0)
    tiled_f32.w_layout = binding.LAYOUT_TILED
    assert fwd(p, 1, 4, ctypes.byref(tiled_f32), None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -1
    tiled_odd = _layer(binding, F=576)
    tiled_odd.w_layout = binding.LAYOUT_TILED
    assert fwd(p, 1, 4, ctypes.byref(tiled_odd), None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -2
    # an unknown bias mode
    bad_bias = _layer(binding)
    bad_bias.bias_mode = 2
    assert fwd(p, 1, 4, ctypes.byref(bad_bias), None, None, None, None, p, 0, 0, ws, 1 << 40, None) == -1
    assert lib.moe_route(p, 1, 4, ctypes.byref(bad_bias), 6, p, p, None, ws, 1 << 40, None) == -1
    # the no-allocation router refuses what moe_route refuses, and sizes beyond its scratch
    assert lib.moe_route_noalloc(p, 1, 4, ctypes.byref(bad_bias), 6, p, p, None) == -1
    assert lib.moe_route_noalloc(p, 1, 4, ctypes.byref(good), 5, p, p, None) == -2
    assert lib.moe_route_noalloc(p, 1, (1 << 20) // 384 + 1, ctypes.byref(good), 6, p, p, None) == -3
    assert lib.moe_route_noalloc(None, 1, 4, ctypes.byref(good), 6, p, p, None) == -1
    assert lib.moe_route_noalloc(p, 1, 0, ctypes.byref(good), 6, p, p, None) == 0
    # packing: needs E4M3 rows with d, ffn multiples of 128, and four aligned destinations
    pack = lib.moe_pack_weights
    assert pack(ctypes.byref(_layer(binding, F=576)), p, p, p, p, None) == -2
    tiled = _layer(binding)
    tiled.w_layout = binding.LAYOUT_TILED
    assert pack(ctypes.byref(tiled), p, p, p, p, None) == -1
    assert pack(ctypes.byref(good), p, None, p, p, None) == -1
    assert pack(ctypes.byref(good), p, p + 8, p, p, None) == -1
    assert pack(None, p, p, p, p, None) == -1


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.moe_status_string(code)
