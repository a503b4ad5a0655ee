"""Python binding of libmoe (ctypes): argument marshalling only.

Every step of the layer runs in libmoe's CUDA kernels; this module turns torch tensors into
device pointers, passes torch's current CUDA stream, and raises on a non-OK status.  There is
no fallback: without the compiled library every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_F32, MOE_BF16, MOE_E4M3, MOE_E2M1 = 0, 1, 2, 3
LAYOUT_ROWS, LAYOUT_TILED = 0, 1
BIAS_SCORE, BIAS_SELECT = 0, 1
PATH_AUTO, PATH_STREAM, PATH_TC = 0, 1, 2
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_WORKSPACE",
          -4: "MOE_ERR_BAD_FORCED_ID", -5: "MOE_ERR_TIMEOUT", -6: "MOE_ERR_CUDA", -7: "MOE_ERR_INDEX"}

# every entry point include/libmoe.h declares
EXPORTS = ("moe_workspace_bytes", "moe_workspace_init", "moe_route", "moe_dispatch", "moe_forward",
           "moe_forward_stack", "moe_forward_traced", "moe_forward_stack_traced", "moe_get_status",
           "moe_status_string", "moe_e4m3_encode", "moe_route_noalloc", "moe_selftest_wait_timeout",
           "moe_pack_weights")
TRACE_POINTS = 9
TRACE_STAGES = ("router", "select", "dispatch", "act_quant", "gate_up", "h_quant", "down", "combine")


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


class MoeLayerC(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("ffn", ctypes.c_int), ("n_experts", ctypes.c_int),
                ("top_k", ctypes.c_int), ("w_dtype", ctypes.c_int),
                ("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("w_gate_up", ctypes.c_void_p), ("s_gate_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("sh_gate_up", ctypes.c_void_p), ("sh_s_gate_up", ctypes.c_void_p),
                ("sh_down", ctypes.c_void_p), ("sh_s_down", ctypes.c_void_p), ("w_layout", ctypes.c_int),
                ("bias_mode", ctypes.c_int)]


_lib = None


def lib():
    """The loaded libmoe.so.  Raises if it has not been built (no CPU fallback exists)."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def use_library(path: Optional[str]):
    """Route every call of this module through the libmoe build at `path` (e.g. the MOE_DEBUG
    build); None goes back to libmoe.so.  Returns the library in use before."""
    global _lib
    before = _lib
    _lib = load(path) if path else None
    return before


def load(path: str):
    """A libmoe build at `path` with every entry point's argument and result types set."""
    if not os.path.exists(path):
        raise ImportError(f"libmoe not built ({path}); run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64, sz, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint
    L.moe_workspace_bytes.argtypes = [vp, i32]
    L.moe_workspace_bytes.restype = sz
    L.moe_workspace_init.argtypes = [vp, sz, vp]
    L.moe_route.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp, vp, sz, vp]
    L.moe_dispatch.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    L.moe_forward.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp, i32, u32, vp, sz, vp]
    L.moe_forward_stack.argtypes = [vp, i32, vp, i32, vp, u32, vp, sz, vp]
    L.moe_forward_traced.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp, i32, u32, vp, sz, vp, vp]
    L.moe_forward_stack_traced.argtypes = [vp, i32, vp, i32, vp, u32, vp, sz, vp, vp]
    L.moe_get_status.argtypes = [vp, vp]
    L.moe_status_string.argtypes = [i32]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_e4m3_encode.argtypes = [vp, vp, i64, vp]
    L.moe_route_noalloc.argtypes = [vp, i32, i32, vp, i32, vp, vp, vp]
    L.moe_selftest_wait_timeout.argtypes = [vp, sz, u32, vp]
    L.moe_pack_weights.argtypes = [vp, vp, vp, vp, vp, vp]
    for f in ("moe_workspace_init", "moe_route", "moe_dispatch", "moe_forward", "moe_forward_stack",
              "moe_forward_traced", "moe_forward_stack_traced", "moe_get_status", "moe_e4m3_encode",
              "moe_route_noalloc", "moe_selftest_wait_timeout", "moe_pack_weights"):
        getattr(L, f).restype = i32
    return L


def status_string(status: int) -> str:
    try:
        return lib().moe_status_string(status).decode()
    except ImportError:
        return STATUS.get(status, "unknown")


def _check(rc: int, what: str):
    if rc != 0:
        raise MoeError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmoe takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MOE_F32
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    raise ValueError(f"unsupported activation dtype {t.dtype}")


class Layer:
    """One layer's weights as device tensors, plus the C descriptor that borrows them.

    FP8 layers take uint8 E4M3 codes (or torch.float8_e4m3fn tensors) and fp32 scales; the
    four weight tensors keep their shapes ([E,2,F,d], [E,d,F], [2,F,d], [d,F]) in either byte
    order (`layout`: LAYOUT_ROWS, or LAYOUT_TILED as written by moe_pack_weights).
    `bias_mode`: BIAS_SCORE (the bias is added to the logits) or BIAS_SELECT (it only ranks)."""

    def __init__(self, w_router, router_bias, w_gate_up, w_down, sh_gate_up, sh_down,
                 s_gate_up=None, s_down=None, sh_s_gate_up=None, sh_s_down=None, top_k: int = 6,
                 layout: int = LAYOUT_ROWS, bias_mode: int = BIAS_SCORE, w_dtype: Optional[int] = None):
        self.tensors = dict(w_router=w_router, router_bias=router_bias, w_gate_up=w_gate_up, w_down=w_down,
                            sh_gate_up=sh_gate_up, sh_down=sh_down, s_gate_up=s_gate_up, s_down=s_down,
                            sh_s_gate_up=sh_s_gate_up, sh_s_down=sh_s_down)
        E, two, F, d = w_gate_up.shape
        assert two == 2
        if w_dtype is None:  # uint8 / float8 codes are E4M3; E2M1 codes must be named
            w_dtype = MOE_E4M3 if w_gate_up.dtype in (torch.uint8, torch.float8_e4m3fn) else MOE_F32
        if w_dtype == MOE_E2M1:
            d *= 2  # two codes per byte
        fp8 = w_dtype in (MOE_E4M3, MOE_E2M1)
        self.d, self.F, self.E, self.k, self.fp8, self.layout = d, F, E, top_k, fp8, layout
        self.bias_mode, self.w_dtype = bias_mode, w_dtype
        self.c = MoeLayerC(d, F, E, top_k, w_dtype,
                           _ptr(w_router), _ptr(router_bias), _ptr(w_gate_up), _ptr(s_gate_up), _ptr(w_down),
                           _ptr(s_down), _ptr(sh_gate_up), _ptr(sh_s_gate_up), _ptr(sh_down), _ptr(sh_s_down),
                           layout, bias_mode)

    def tiled(self) -> "Layer":
        """The same layer with its E4M3 weights rewritten in the tiled layout (moe_pack_weights)."""
        assert self.layout == LAYOUT_ROWS
        t = self.tensors
        out = {k: torch.empty_like(t[k]) for k in ("w_gate_up", "w_down", "sh_gate_up", "sh_down")}
        _check(lib().moe_pack_weights(self.ref, _ptr(out["w_gate_up"]), _ptr(out["w_down"]), _ptr(out["sh_gate_up"]),
                                      _ptr(out["sh_down"]), _stream()), "moe_pack_weights")
        return Layer(**{**t, **out}, top_k=self.k, layout=LAYOUT_TILED, bias_mode=self.bias_mode,
                     w_dtype=self.w_dtype)

    def clone(self) -> "Layer":
        """A copy at other device addresses (same values, layout and bias mode)."""
        return Layer(**{k: (v.clone() if v is not None else None) for k, v in self.tensors.items()}, top_k=self.k,
                     layout=self.layout, bias_mode=self.bias_mode, w_dtype=self.w_dtype)

    @classmethod
    def from_host(cls, w, device="cuda", top_k: int = 6, tiled: Optional[bool] = None, bias_mode: int = BIAS_SCORE):
        """From a gen.moegen.LayerWeights-like object of numpy arrays.  tiled=None: the tiled
        layout (tensor-core expert kernels) whenever the weights are E4M3 with d_model and ffn
        multiples of 128; the row layout (weight-streaming kernels) otherwise."""
        def dev(a):
            return None if a is None else torch.from_numpy(a).to(device)
        fp4 = getattr(w, "fp4", False)
        rows = cls(dev(w.Wr), dev(w.bias), dev(w.Wgu), dev(w.Wd), dev(w.sh_Wgu), dev(w.sh_Wd),
                   dev(w.sgu), dev(w.sd), dev(w.sh_sgu), dev(w.sh_sd), top_k=top_k, bias_mode=bias_mode,
                   w_dtype=MOE_E2M1 if fp4 else None)
        if tiled is None or fp4:  # 4-bit weights run tiled only
            tiled = fp4 or (rows.fp8 and rows.d % 128 == 0 and rows.F % 128 == 0)
        if not tiled:
            return rows
        packed = rows.tiled()
        del rows  # the row-layout copies are released once the tiled ones exist
        return packed

    @property
    def ref(self):
        return ctypes.byref(self.c)


def workspace_bytes(layer: Layer, T: int) -> int:
    return int(lib().moe_workspace_bytes(layer.ref, T))


def workspace(layer: Layer, T: int, device="cuda") -> torch.Tensor:
    n = max(workspace_bytes(layer, T), 256)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _check(lib().moe_workspace_init(_ptr(ws), n, _stream()), "moe_workspace_init")
    return ws


def route(x: torch.Tensor, layer: Layer, ws: torch.Tensor, logits: bool = False):
    """Free routing.  Returns (ids [T,k] int32, w [T,k] fp32, logits [T,E] or None)."""
    T = x.shape[0]
    ids = torch.empty((T, layer.k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, layer.k), dtype=torch.float32, device=x.device)
    lg = torch.empty((T, layer.E), dtype=torch.float32, device=x.device) if logits else None
    _check(lib().moe_route(_ptr(x), _dtype_code(x), T, layer.ref, layer.k, _ptr(ids), _ptr(w), _ptr(lg), _ptr(ws),
                           ws.numel(), _stream()), "moe_route")
    return ids, w, lg


def route_noalloc(x: torch.Tensor, layer: Layer):
    """Free routing without a workspace (moe_route_noalloc): for callers that cannot allocate
    device memory.  Returns (ids [T,k] int32, w [T,k] fp32); the caller still owns the
    outputs.  Calls that overlap on the GPU share the library's scratch and must not run
    concurrently."""
    T = x.shape[0]
    ids = torch.empty((T, layer.k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, layer.k), dtype=torch.float32, device=x.device)
    _check(lib().moe_route_noalloc(_ptr(x), _dtype_code(x), T, layer.ref, layer.k, _ptr(ids), _ptr(w), _stream()),
           "moe_route_noalloc")
    return ids, w


def dispatch(ids: torch.Tensor, n_experts: int, ws: torch.Tensor):
    T, k = ids.shape
    dev = ids.device
    counts = torch.empty(n_experts + 1, dtype=torch.int32, device=dev)
    offsets = torch.empty(n_experts + 2, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k + T, dtype=torch.int32, device=dev)
    pos = torch.empty((T, k), dtype=torch.int32, device=dev)
    _check(lib().moe_dispatch(_ptr(ids), T, n_experts, k, _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(pos),
                              _ptr(ws), ws.numel(), _stream()), "moe_dispatch")
    return dict(counts=counts, offsets=offsets, perm=perm, pos=pos)


def event_array(events):
    """ctypes array of raw cudaEvent_t handles from torch.cuda.Event objects (or None)."""
    if events is None:
        return None
    handles = [e.cuda_event for e in events]
    if not all(handles):
        raise ValueError("timing events must exist on the device: torch creates them at their first record()")
    return (ctypes.c_void_p * len(events))(*handles)


def forward(x: torch.Tensor, layer: Layer, ws: torch.Tensor, forced_ids=None, forced_w=None,
            y_dtype=torch.float32, flags: int = PATH_AUTO, out=None, ids=None, w=None, events=None):
    """The layer.  Returns (y [T,d], ids [T,k], w [T,k]).  `events`: TRACE_POINTS
    torch.cuda.Event(enable_timing=True) recorded at the stage boundaries (moe_forward_traced)."""
    T = x.shape[0]
    ids = ids if ids is not None else torch.empty((T, layer.k), dtype=torch.int32, device=x.device)
    w = w if w is not None else torch.empty((T, layer.k), dtype=torch.float32, device=x.device)
    y = out if out is not None else torch.empty((T, layer.d), dtype=y_dtype, device=x.device)
    if events is None:
        rc = lib().moe_forward(_ptr(x), _dtype_code(x), T, layer.ref, _ptr(forced_ids), _ptr(forced_w), _ptr(ids),
                               _ptr(w), _ptr(y), _dtype_code(y), flags, _ptr(ws), ws.numel(), _stream())
    else:
        assert len(events) == TRACE_POINTS
        rc = lib().moe_forward_traced(_ptr(x), _dtype_code(x), T, layer.ref, _ptr(forced_ids), _ptr(forced_w),
                                      _ptr(ids), _ptr(w), _ptr(y), _dtype_code(y), flags, _ptr(ws), ws.numel(),
                                      _stream(), event_array(events))
    _check(rc, "moe_forward")
    return y, ids, w


class GraphedForward:
    """One forward step on fixed buffers, captured once as a CUDA graph and replayed with one
    launch: optionally the copy of x from pinned host memory, the layer's kernels, optionally
    the copy of y back to pinned host memory.  For serving loops, where issuing the step's
    launches from the host one by one costs more than the layer at decode sizes.  The buffers
    (and their contents' shapes) are those given here; write new inputs into `x_host` (or
    `x`) before each replay()."""

    def __init__(self, x: torch.Tensor, layer: Layer, ws: torch.Tensor, out: torch.Tensor, ids: torch.Tensor,
                 w: torch.Tensor, flags: int = PATH_AUTO, x_host: Optional[torch.Tensor] = None,
                 y_host: Optional[torch.Tensor] = None):
        self.buffers = (x, layer, ws, out, ids, w, x_host, y_host)  # kept alive with the graph
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # one plain call first: one-time attribute setup is not captured
            forward(x, layer, ws, out=out, ids=ids, w=w, flags=flags)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            if x_host is not None:
                x.copy_(x_host, non_blocking=True)
            forward(x, layer, ws, out=out, ids=ids, w=w, flags=flags)
            if y_host is not None:
                y_host.copy_(out, non_blocking=True)

    def replay(self):
        self.graph.replay()


def layer_array(layers: Sequence[Layer]):
    arr = (MoeLayerC * len(layers))(*[l.c for l in layers])
    return arr


def forward_stack(layers: Sequence[Layer], residual: torch.Tensor, ws: torch.Tensor, ids_out=None,
                  flags: int = PATH_AUTO, layer_arr=None, events=None):
    """residual [T, d] bf16, updated in place.  ids_out [L, T, k] int32 or None.  `events`:
    L * TRACE_POINTS timing events (moe_forward_stack_traced) or None."""
    arr = layer_arr if layer_arr is not None else layer_array(layers)
    n = len(arr)
    T = residual.shape[0]
    if events is None:
        rc = lib().moe_forward_stack(arr, n, _ptr(residual), T, _ptr(ids_out), flags, _ptr(ws), ws.numel(),
                                     _stream())
    else:
        assert len(events) == n * TRACE_POINTS
        rc = lib().moe_forward_stack_traced(arr, n, _ptr(residual), T, _ptr(ids_out), flags, _ptr(ws), ws.numel(),
                                            _stream(), event_array(events))
    _check(rc, "moe_forward_stack")
    return residual


class GraphedStack:
    """One step of the layer stack on fixed buffers, captured once as a CUDA graph and replayed
    with one launch: optionally the copy of the step's input `x` into the residual, then the L
    layers of moe_forward_stack.  At small batches a layer's kernels take a few microseconds
    each, and issuing the L x 5 launches one by one from the host shows between them.  The
    constructor runs the step once before capturing it (one-time attribute setup), so the
    residual holds one step's result afterwards."""

    def __init__(self, layers: Sequence[Layer], residual: torch.Tensor, ws: torch.Tensor,
                 x: Optional[torch.Tensor] = None, ids_out=None, flags: int = PATH_AUTO, layer_arr=None):
        arr = layer_arr if layer_arr is not None else layer_array(layers)
        self.buffers = (layers, residual, ws, x, ids_out, arr)  # kept alive with the graph
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            if x is not None:
                residual.copy_(x)
            forward_stack(layers, residual, ws, ids_out=ids_out, flags=flags, layer_arr=arr)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=side):
            if x is not None:
                residual.copy_(x, non_blocking=True)
            forward_stack(layers, residual, ws, ids_out=ids_out, flags=flags, layer_arr=arr)

    def replay(self):
        self.graph.replay()


def get_status(ws: torch.Tensor) -> int:
    """Synchronises the current stream; returns (and clears) the device-side status code."""
    return int(lib().moe_get_status(_ptr(ws), _stream()))


def selftest_wait_timeout(ws: torch.Tensor, timeout_us: int = 10000):
    """Launch the bounded-wait self-test; moe_get_status(ws) then reports MOE_ERR_TIMEOUT."""
    _check(lib().moe_selftest_wait_timeout(_ptr(ws), ws.numel(), timeout_us, _stream()), "moe_selftest_wait_timeout")


def e4m3_encode(v: torch.Tensor) -> torch.Tensor:
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _check(lib().moe_e4m3_encode(_ptr(v), _ptr(out), v.numel(), _stream()), "moe_e4m3_encode")
    return out
