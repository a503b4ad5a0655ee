"""Seeded synthetic inputs for the routed expert layer (input data only).

This module is shared, as a source of DATA, by the CUDA library's tests/bench and by the
CPU oracle.  It contains none of the layer's arithmetic (router, selection, expert FFN,
combine); it draws Gaussians from a counter-based SplitMix64 stream and applies the
checkpoint-conversion recipe (per-output-row E4M3 codes with scale = rowabsmax / 448).

Recipes (Kolibri-1 layer shapes: 384 routed experts, top-6, one shared expert; the model
description in "We Ported Aleph Alpha's Kolibri to a MacBook. Our Own Gate Said No.",
section "The gate"):
  x       ~ N(0, 1)         [T, d]   bf16 (fp32 for the tiny all-fp32 layer)
  Wr      ~ N(0, 1/d)       [E, d]   fp32
  bias    ~ N(0, 0.5)       [E]      fp32 (variance 0.5), or absent
  Wg, Wu  ~ N(0, 1/d)       [E, 2, ffn, d]  E4M3 codes + [E, 2, ffn] scales (or fp32)
  Wd      ~ N(0, 1/ffn)     [E, d, ffn]     E4M3 codes + [E, d] scales (or fp32)
  shared expert: same recipe, its own streams.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moegen.cpp")
_LIB = os.path.join(_HERE, "libmoegen.so")

# stream ids (the "tensor" coordinate of a stream)
T_X, T_WR, T_BIAS, T_WGU, T_WD, T_SH_WGU, T_SH_WD, T_FORCED_IDS, T_FORCED_W, T_SAMPLE = range(10)

_lib = None


def build(force: bool = False) -> str:
    """Compile libmoegen.so next to its source (plain g++, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               _SRC, "-o", _LIB + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, u32, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_double, ctypes.c_void_p)
        L.moegen_normal_f32.argtypes = [u64, u32, u32, u64, i64, dbl, vp, i32]
        L.moegen_normal_bf16.argtypes = [u64, u32, u32, u64, i64, dbl, vp, i32]
        L.moegen_normal_e4m3_rows.argtypes = [u64, u32, u32, i64, i64, i64, dbl, vp, vp, i32]
        L.moegen_quant_rows_e4m3.argtypes = [vp, i64, i64, vp, vp]
        L.moegen_normal_e2m1_rows.argtypes = [u64, u32, u32, i64, i64, i64, dbl, vp, vp, i32]
        L.moegen_quant_e2m1_n.argtypes = [vp, i64, vp]
        L.moegen_zipf_ids.argtypes = [u64, u32, u32, i32, i32, i32, dbl, vp]
        L.moegen_dirichlet_w.argtypes = [u64, u32, u32, i32, i32, vp]
        L.moegen_uniform_int.argtypes = [u64, u32, u32, i64, i64, vp]
        for f in ("moegen_normal_f32", "moegen_normal_bf16", "moegen_normal_e4m3_rows",
                  "moegen_quant_rows_e4m3", "moegen_normal_e2m1_rows", "moegen_quant_e2m1_n", "moegen_zipf_ids", "moegen_dirichlet_w", "moegen_uniform_int"):
            getattr(L, f).restype = None
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_f32(seed, layer, tensor, shape, var, out=None, start=0, nthreads=None):
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, np.float32)
    lib().moegen_normal_f32(seed, layer, tensor, start, n, var, _ptr(out), nthreads or default_threads())
    return out


def normal_bf16_bits(seed, layer, tensor, shape, var, out=None, start=0, nthreads=None):
    """bf16 bit patterns (uint16) of N(0, var) draws."""
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, np.uint16)
    lib().moegen_normal_bf16(seed, layer, tensor, start, n, var, _ptr(out), nthreads or default_threads())
    return out


def normal_e4m3_rows(seed, layer, tensor, row0, rows, cols, var, codes=None, scales=None, nthreads=None):
    if codes is None:
        codes = np.empty((rows, cols), np.uint8)
    if scales is None:
        scales = np.empty((rows,), np.float32)
    lib().moegen_normal_e4m3_rows(seed, layer, tensor, row0, rows, cols, var, _ptr(codes), _ptr(scales),
                                  nthreads or default_threads())
    return codes, scales


def normal_e2m1_rows(seed, layer, tensor, row0, rows, cols, var, codes=None, scales=None, nthreads=None):
    """The 4-bit checkpoint of rows [row0, row0 + rows): packed E2M1 codes [rows, cols / 2]
    (element 2i in the low nibble of byte i) and scales rowabsmax / 6."""
    if codes is None:
        codes = np.empty((rows, cols // 2), np.uint8)
    if scales is None:
        scales = np.empty((rows,), np.float32)
    lib().moegen_normal_e2m1_rows(seed, layer, tensor, row0, rows, cols, var, _ptr(codes), _ptr(scales),
                                  nthreads or default_threads())
    return codes, scales


def quant_e2m1(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().moegen_quant_e2m1_n(_ptr(v), v.size, _ptr(out))
    return out


def quant_rows_e4m3(w: np.ndarray):
    w = np.ascontiguousarray(w, np.float32)
    rows, cols = int(np.prod(w.shape[:-1])), w.shape[-1]
    codes = np.empty(w.shape, np.uint8)
    scales = np.empty(w.shape[:-1], np.float32)
    lib().moegen_quant_rows_e4m3(_ptr(w), rows, cols, _ptr(codes), _ptr(scales))
    return codes, scales


def zipf_ids(seed, layer, T, E, k, s):
    ids = np.empty((T, k), np.int32)
    lib().moegen_zipf_ids(seed, layer, T_FORCED_IDS, T, E, k, s, _ptr(ids))
    return ids


def dirichlet_w(seed, layer, T, k):
    w = np.empty((T, k), np.float32)
    lib().moegen_dirichlet_w(seed, layer, T_FORCED_W, T, k, _ptr(w))
    return w


def uniform_int(seed, count, n, tensor=T_SAMPLE, layer=0):
    out = np.empty((count,), np.int64)
    lib().moegen_uniform_int(seed, layer, tensor, count, n, _ptr(out))
    return out


@dataclass
class LayerWeights:
    """Host arrays of one layer.  fp8=True: E4M3 codes + fp32 per-row scales; fp4=True: packed
    E2M1 codes (two per byte, the last dimension halved) + fp32 per-row scales; else fp32."""
    d: int
    ffn: int
    E: int
    fp8: bool
    Wr: np.ndarray
    bias: Optional[np.ndarray]
    Wgu: np.ndarray          # [E, 2, ffn, d]
    Wd: np.ndarray           # [E, d, ffn]
    sh_Wgu: np.ndarray       # [2, ffn, d]
    sh_Wd: np.ndarray        # [d, ffn]
    sgu: Optional[np.ndarray] = None     # [E, 2, ffn]
    sd: Optional[np.ndarray] = None      # [E, d]
    sh_sgu: Optional[np.ndarray] = None  # [2, ffn]
    sh_sd: Optional[np.ndarray] = None   # [d]
    meta: dict = field(default_factory=dict)
    fp4: bool = False


def make_layer(seed: int, d: int, ffn: int, E: int, fp8: bool, bias_var: Optional[float],
               layer: int = 0, nthreads: Optional[int] = None, out: Optional[dict] = None,
               down_var: Optional[float] = None, fp4: bool = False) -> LayerWeights:
    """One layer's weights from the recipe above.  `out` may supply preallocated arrays
    (e.g. pinned host buffers) keyed like the LayerWeights fields.  `down_var` replaces the
    down-projection variance 1/ffn (used by the stack, see stack_layer).  fp4=True: the 4-bit
    checkpoint of the same Gaussian weights (E2M1 codes, scale rowabsmax / 6)."""
    nt = nthreads or default_threads()
    dv = down_var if down_var is not None else 1.0 / ffn
    o = out or {}
    Wr = normal_f32(seed, layer, T_WR, (E, d), 1.0 / d, out=o.get("Wr"), nthreads=nt)
    bias = normal_f32(seed, layer, T_BIAS, (E,), bias_var, out=o.get("bias"), nthreads=nt) if bias_var else None
    if fp4:
        Wgu = np.empty((E, 2, ffn, d // 2), np.uint8)
        sgu = np.empty((E, 2, ffn), np.float32)
        normal_e2m1_rows(seed, layer, T_WGU, 0, E * 2 * ffn, d, 1.0 / d, Wgu.reshape(E * 2 * ffn, d // 2),
                         sgu.reshape(-1), nthreads=nt)
        Wd = np.empty((E, d, ffn // 2), np.uint8)
        sd = np.empty((E, d), np.float32)
        normal_e2m1_rows(seed, layer, T_WD, 0, E * d, ffn, dv, Wd.reshape(E * d, ffn // 2), sd.reshape(-1),
                         nthreads=nt)
        sh_Wgu = np.empty((2, ffn, d // 2), np.uint8)
        sh_sgu = np.empty((2, ffn), np.float32)
        normal_e2m1_rows(seed, layer, T_SH_WGU, 0, 2 * ffn, d, 1.0 / d, sh_Wgu.reshape(2 * ffn, d // 2),
                         sh_sgu.reshape(-1), nthreads=nt)
        sh_Wd = np.empty((d, ffn // 2), np.uint8)
        sh_sd = np.empty((d,), np.float32)
        normal_e2m1_rows(seed, layer, T_SH_WD, 0, d, ffn, dv, sh_Wd, sh_sd, nthreads=nt)
        return LayerWeights(d, ffn, E, False, Wr, bias, Wgu, Wd, sh_Wgu, sh_Wd, sgu, sd, sh_sgu, sh_sd, fp4=True)
    if fp8:
        Wgu = o.get("Wgu", np.empty((E, 2, ffn, d), np.uint8))
        sgu = o.get("sgu", np.empty((E, 2, ffn), np.float32))
        normal_e4m3_rows(seed, layer, T_WGU, 0, E * 2 * ffn, d, 1.0 / d,
                         Wgu.reshape(E * 2 * ffn, d), sgu.reshape(-1), nthreads=nt)
        Wd = o.get("Wd", np.empty((E, d, ffn), np.uint8))
        sd = o.get("sd", np.empty((E, d), np.float32))
        normal_e4m3_rows(seed, layer, T_WD, 0, E * d, ffn, dv, Wd.reshape(E * d, ffn), sd.reshape(-1),
                         nthreads=nt)
        sh_Wgu = o.get("sh_Wgu", np.empty((2, ffn, d), np.uint8))
        sh_sgu = o.get("sh_sgu", np.empty((2, ffn), np.float32))
        normal_e4m3_rows(seed, layer, T_SH_WGU, 0, 2 * ffn, d, 1.0 / d, sh_Wgu.reshape(2 * ffn, d),
                         sh_sgu.reshape(-1), nthreads=nt)
        sh_Wd = o.get("sh_Wd", np.empty((d, ffn), np.uint8))
        sh_sd = o.get("sh_sd", np.empty((d,), np.float32))
        normal_e4m3_rows(seed, layer, T_SH_WD, 0, d, ffn, dv, sh_Wd, sh_sd, nthreads=nt)
        return LayerWeights(d, ffn, E, True, Wr, bias, Wgu, Wd, sh_Wgu, sh_Wd, sgu, sd, sh_sgu, sh_sd)
    Wgu = normal_f32(seed, layer, T_WGU, (E, 2, ffn, d), 1.0 / d, nthreads=nt)
    Wd = normal_f32(seed, layer, T_WD, (E, d, ffn), dv, nthreads=nt)
    sh_Wgu = normal_f32(seed, layer, T_SH_WGU, (2, ffn, d), 1.0 / d, nthreads=nt)
    sh_Wd = normal_f32(seed, layer, T_SH_WD, (d, ffn), dv, nthreads=nt)
    return LayerWeights(d, ffn, E, False, Wr, bias, Wgu, Wd, sh_Wgu, sh_Wd)


def make_x(seed: int, T: int, d: int, bf16: bool, start_token: int = 0, layer: int = 0, var: float = 1.0):
    """Activations x[T, d] ~ N(0, var): bf16 bit patterns (uint16) or fp32.
    start_token selects a window of a longer sequence (element index = token * d + k)."""
    if bf16:
        return normal_bf16_bits(seed, layer, T_X, (T, d), var, start=start_token * d)
    return normal_f32(seed, layer, T_X, (T, d), var, start=start_token * d)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp32 (the bits land in the high half)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---- the five workloads -------------------------------------------------------------------
# (d, ffn, E, k) of the Kolibri-1 layer as these configurations fix it; the tiny layer keeps
# E and k and shrinks d and ffn.
KOLIBRI = dict(d=2048, ffn=640, E=384, k=6)
TINY = dict(d=256, ffn=128, E=384, k=6)

SEED_TINY, SEED_DECODE, SEED_PREFILL, SEED_ZIPF, SEED_STACK_X = 1, 2, 3, 4, 5
STACK_LAYER_SEED0 = 5000


def tiny_layer():
    return make_layer(SEED_TINY, TINY["d"], TINY["ffn"], TINY["E"], fp8=False, bias_var=None)


def kolibri_layer(seed: int, layer: int = 0, out=None, nthreads=None, down_var=None, fp4: bool = False):
    return make_layer(seed, KOLIBRI["d"], KOLIBRI["ffn"], KOLIBRI["E"], fp8=not fp4, bias_var=0.5,
                      layer=layer, out=out, nthreads=nthreads, down_var=down_var, fp4=fp4)


# The 50-layer stack applies r <- r + moe(r) with no normalisation; with the single-layer
# recipe (down projection ~ N(0, 1/ffn)) the residual grows doubly exponentially (the SwiGLU
# is quadratic in x for large x) and overflows fp32 after 8 layers.  The stack therefore
# scales every residual-branch output projection (routed and shared down weights) by
# 1/sqrt(L), the initialisation Radford et al. use for deep residual stacks (GPT-2, 2019,
# section 2.3): down ~ N(0, 1/(ffn * L)).
STACK_LAYERS = 50
STACK_DOWN_VAR = 1.0 / (KOLIBRI["ffn"] * STACK_LAYERS)


def stack_layer(l: int, out=None, nthreads=None):
    return kolibri_layer(STACK_LAYER_SEED0 + l, out=out, nthreads=nthreads, down_var=STACK_DOWN_VAR)


def sparse_layer(seed: int, experts, d: int = 2048, ffn: int = 640, E: int = 384, bias_var: float = 0.5,
                 layer: int = 0, nthreads=None, down_var: Optional[float] = None) -> LayerWeights:
    """The same layer as kolibri_layer(seed), but only the listed routed experts (plus the
    router and the shared expert) are generated; the other experts' weight arrays are left
    unwritten (allocated lazily, never read by a forced-route evaluation that avoids them).
    Every stream is counter-based, so each generated row equals the full layer's row."""
    nt = nthreads or default_threads()
    dv = down_var if down_var is not None else 1.0 / ffn
    Wr = normal_f32(seed, layer, T_WR, (E, d), 1.0 / d, nthreads=nt)
    bias = normal_f32(seed, layer, T_BIAS, (E,), bias_var, nthreads=nt) if bias_var else None
    Wgu = np.empty((E, 2, ffn, d), np.uint8)
    sgu = np.zeros((E, 2, ffn), np.float32)
    Wd = np.empty((E, d, ffn), np.uint8)
    sd = np.zeros((E, d), np.float32)
    for e in sorted(set(int(v) for v in experts)):
        normal_e4m3_rows(seed, layer, T_WGU, e * 2 * ffn, 2 * ffn, d, 1.0 / d, Wgu[e].reshape(2 * ffn, d),
                         sgu[e].reshape(-1), nthreads=nt)
        normal_e4m3_rows(seed, layer, T_WD, e * d, d, ffn, dv, Wd[e], sd[e], nthreads=nt)
    sh_Wgu = np.empty((2, ffn, d), np.uint8)
    sh_sgu = np.empty((2, ffn), np.float32)
    normal_e4m3_rows(seed, layer, T_SH_WGU, 0, 2 * ffn, d, 1.0 / d, sh_Wgu.reshape(2 * ffn, d), sh_sgu.reshape(-1),
                     nthreads=nt)
    sh_Wd = np.empty((d, ffn), np.uint8)
    sh_sd = np.empty((d,), np.float32)
    normal_e4m3_rows(seed, layer, T_SH_WD, 0, d, ffn, dv, sh_Wd, sh_sd, nthreads=nt)
    return LayerWeights(d, ffn, E, True, Wr, bias, Wgu, Wd, sh_Wgu, sh_Wd, sgu, sd, sh_sgu, sh_sd)


def stack_x(T: int, start_token: int = 0):
    """Residual stream input of the 50-layer stack: bf16 N(0,1), seed 5."""
    return make_x(SEED_STACK_X, T, KOLIBRI["d"], bf16=True, start_token=start_token)
