"""ctypes wrapper of the CPU oracle (oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by tests/, by __graft_entry__.smoke() and by bench.py's
CPU-baseline leg.  The product library never imports, links or runs anything here.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

MUT_NONE, MUT_BF16_ROUTER, MUT_UNBIASED_SELECT, MUT_HIGH_INDEX_TIE, MUT_NO_RENORM, MUT_NO_SHARED, \
    MUT_SORTED_SUM, MUT_SWAP_GATE_UP, MUT_SCALE_AXIS, MUT_DISPATCH_SHIFT, MUT_BIASED_WEIGHTS = range(11)
MUTANTS = {
    "bf16_router": MUT_BF16_ROUTER, "unbiased_select": MUT_UNBIASED_SELECT,
    "high_index_tie": MUT_HIGH_INDEX_TIE, "no_renorm": MUT_NO_RENORM, "no_shared": MUT_NO_SHARED,
    "sorted_sum": MUT_SORTED_SUM, "swap_gate_up": MUT_SWAP_GATE_UP, "scale_axis": MUT_SCALE_AXIS,
    "dispatch_shift": MUT_DISPATCH_SHIFT, "biased_weights": MUT_BIASED_WEIGHTS,
}
ACT_W8A8, ACT_W8A16 = 0, 1
# the per-expert bias: added to the logits (selection and weights), or to the selection only
BIAS_SCORE, BIAS_SELECT = 0, 1


class OracleLayer(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("ffn", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("w_fp8", ctypes.c_int), ("act_mode", ctypes.c_int), ("mutant", ctypes.c_int),
                ("Wr", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("Wgu", ctypes.c_void_p), ("sgu", ctypes.c_void_p),
                ("Wd", ctypes.c_void_p), ("sd", ctypes.c_void_p),
                ("sh_Wgu", ctypes.c_void_p), ("sh_sgu", ctypes.c_void_p),
                ("sh_Wd", ctypes.c_void_p), ("sh_sd", ctypes.c_void_p), ("bias_mode", ctypes.c_int)]


_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (plain g++ -O2, no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-pthread", _SRC, "-o", _LIB + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = ctypes.c_float
        L.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1_decode.restype = ctypes.c_float
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_bf16_rne.argtypes = [ctypes.c_float]
        L.oracle_bf16_rne.restype = ctypes.c_uint16
        L.oracle_e4m3_encode_n.argtypes = [vp, i64, vp]
        L.oracle_bf16_rne_n.argtypes = [vp, i64, vp]
        L.oracle_router_logits.argtypes = [vp, vp, vp]
        L.oracle_softmax.argtypes = [vp, i32, vp]
        L.oracle_topk.argtypes = [vp, i32, i32, i32, vp]
        L.oracle_renorm.argtypes = [vp, vp, i32, i32, vp]
        L.oracle_expert.argtypes = [vp, i32, vp, vp]
        L.oracle_layer_forward.argtypes = [vp, vp, i32, i64, vp, vp, vp, vp, vp, vp, vp, i32]
        L.oracle_layer_forward.restype = i32
        L.oracle_layer_forward_range.argtypes = [vp, vp, i32, i64, i64, vp, vp, vp, vp, vp, vp, vp, i32]
        L.oracle_layer_forward_range.restype = i32
        L.oracle_stack_forward.argtypes = [vp, i32, vp, i64, vp, vp, i32]
        L.oracle_stack_forward.restype = i32
        L.oracle_dispatch.argtypes = [vp, i64, i32, i32, i32, vp, vp, vp, vp]
        for f in ("oracle_e4m3_encode_n", "oracle_bf16_rne_n", "oracle_router_logits", "oracle_softmax",
                  "oracle_topk", "oracle_renorm", "oracle_expert", "oracle_dispatch"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


class Layer:
    """Binds a gen.moegen.LayerWeights (host numpy arrays) to the oracle's C struct."""

    def __init__(self, w, k: int = 6, act_mode: int = ACT_W8A8, mutant: int = MUT_NONE,
                 bias_mode: int = BIAS_SCORE):
        self.w = w
        self.k = k
        wfmt = 2 if getattr(w, "fp4", False) else (1 if w.fp8 else 0)  # E2M1, E4M3 or fp32 weights
        self.s = OracleLayer(w.d, w.ffn, w.E, k, wfmt, act_mode, mutant,
                             _p(w.Wr), _p(w.bias), _p(w.Wgu), _p(w.sgu), _p(w.Wd), _p(w.sd),
                             _p(w.sh_Wgu), _p(w.sh_sgu), _p(w.sh_Wd), _p(w.sh_sd), bias_mode)

    @property
    def ptr(self):
        return ctypes.byref(self.s)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def layer_forward(layer: Layer, x: np.ndarray, forced_ids=None, forced_w=None, want_probs=False,
                  nthreads: int = 1, t0: int = 0, t1: Optional[int] = None):
    """x: [T, d] uint16 (bf16 bits) or float32.  Returns dict(ids, w, y[, logits, p]).
    With t0/t1 only that token range is computed (the rest of the outputs stay zero)."""
    x = np.ascontiguousarray(x)
    T, d = x.shape
    t1 = T if t1 is None else t1
    k, E = layer.k, layer.w.E
    xb = 1 if x.dtype == np.uint16 else 0
    assert x.dtype in (np.uint16, np.float32)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    y = np.zeros((T, d), np.float32)
    logits = np.zeros((T, E), np.float32) if want_probs else None
    p = np.zeros((T, E), np.float32) if want_probs else None
    fi = None if forced_ids is None else np.ascontiguousarray(forced_ids, np.int32)
    fw = None if forced_w is None else np.ascontiguousarray(forced_w, np.float32)
    rc = lib().oracle_layer_forward_range(layer.ptr, _p(x), xb, t0, t1, _p(fi), _p(fw), _p(ids), _p(w), _p(y),
                                          _p(logits), _p(p), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_layer_forward: bad forced ids (rc={rc})")
    out = dict(ids=ids, w=w, y=y)
    if want_probs:
        out.update(logits=logits, p=p)
    return out


def stack_forward(layers, residual: np.ndarray, forced_ids=None, nthreads: int = 1):
    """residual: [T, d] uint16 (bf16 bits), returned updated (a copy).  forced_ids: [L, T, k]."""
    arr = (OracleLayer * len(layers))(*[l.s for l in layers])
    r = np.ascontiguousarray(residual, np.uint16).copy()
    T = r.shape[0]
    k = layers[0].k
    ids = np.zeros((len(layers), T, k), np.int32)
    fi = None if forced_ids is None else np.ascontiguousarray(forced_ids, np.int32)
    rc = lib().oracle_stack_forward(arr, len(layers), _p(r), T, _p(fi), _p(ids), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_stack_forward failed rc={rc}")
    return r, ids


def expert(layer: Layer, e: int, xf: np.ndarray) -> np.ndarray:
    xf = np.ascontiguousarray(xf, np.float32)
    ye = np.zeros(layer.w.d, np.float32)
    lib().oracle_expert(layer.ptr, e, _p(xf), _p(ye))
    return ye


def router_logits(layer: Layer, xf: np.ndarray) -> np.ndarray:
    xf = np.ascontiguousarray(xf, np.float32)
    out = np.zeros(layer.w.E, np.float32)
    lib().oracle_router_logits(layer.ptr, _p(xf), _p(out))
    return out


def softmax(logits: np.ndarray) -> np.ndarray:
    logits = np.ascontiguousarray(logits, np.float32)
    p = np.zeros_like(logits)
    lib().oracle_softmax(_p(logits), logits.shape[0], _p(p))
    return p


def topk(p: np.ndarray, k: int, mutant: int = MUT_NONE) -> np.ndarray:
    p = np.ascontiguousarray(p, np.float32)
    ids = np.zeros(k, np.int32)
    lib().oracle_topk(_p(p), p.shape[0], k, mutant, _p(ids))
    return ids


def renorm(p: np.ndarray, ids: np.ndarray, mutant: int = MUT_NONE) -> np.ndarray:
    p = np.ascontiguousarray(p, np.float32)
    ids = np.ascontiguousarray(ids, np.int32)
    w = np.zeros(ids.shape[0], np.float32)
    lib().oracle_renorm(_p(p), _p(ids), ids.shape[0], mutant, _p(w))
    return w


def dispatch(ids: np.ndarray, E: int, mutant: int = MUT_NONE):
    ids = np.ascontiguousarray(ids, np.int32)
    T, k = ids.shape
    counts = np.zeros(E + 1, np.int32)
    offsets = np.zeros(E + 2, np.int32)
    perm = np.zeros(T * k + T, np.int32)
    pos = np.zeros((T, k), np.int32)
    lib().oracle_dispatch(_p(ids), T, E, k, mutant, _p(counts), _p(offsets), _p(perm), _p(pos))
    return dict(counts=counts, offsets=offsets, perm=perm, pos=pos)


def e4m3_decode_all() -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e4m3_decode(c) for c in range(256)], np.float32)


def e2m1_decode_all() -> np.ndarray:
    """The values of the 16 E2M1 codes."""
    L = lib()
    return np.array([L.oracle_e2m1_decode(c) for c in range(16)], np.float32)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float32)
    out = np.zeros(v.shape, np.uint8)
    lib().oracle_e4m3_encode_n(_p(v), v.size, _p(out))
    return out


def bf16_rne(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float32)
    out = np.zeros(v.shape, np.uint16)
    lib().oracle_bf16_rne_n(_p(v), v.size, _p(out))
    return out
