"""Helpers shared by the GPU tests: host<->device moves and GPU-vs-oracle comparisons."""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as o
from tests import parity


def to_dev_x(x: np.ndarray) -> torch.Tensor:
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


def to_host_bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_free_layer(w, x, y_gpu, ids_gpu, w_gpu, nthreads=None, where="", bias_mode=o.BIAS_SCORE):
    """Free routing: ids within the near-tie rule of the oracle's; then the outputs against
    the oracle run with the GPU's ids forced (weights from the oracle's own router)."""
    nt = nthreads or o.default_threads()
    L = o.Layer(w, bias_mode=bias_mode)
    ref = o.layer_forward(L, x, want_probs=True, nthreads=nt)
    ids = ids_gpu.cpu().numpy()
    ok, bad, ndiff = parity.ids_ok(ids, ref["ids"], ref["p"], w.E)
    assert ok, f"{where}: ids outside the near-tie rule: {bad}"
    forced = ref if ndiff == 0 else o.layer_forward(L, x, forced_ids=ids, nthreads=nt)
    okw, msg = parity.weights_ok(w_gpu.cpu().numpy(), forced["w"])
    assert okw, f"{where}: routing weights: {msg}"
    oky, msg = parity.outputs_ok(y_gpu.float().cpu().numpy(), forced["y"])
    assert oky, f"{where}: outputs: {msg}"
    return ref, msg, ndiff


def check_forced_layer(w, x, forced_ids, forced_w, y_gpu, ids_gpu, nthreads=None, where="", bias_mode=o.BIAS_SCORE):
    nt = nthreads or o.default_threads()
    ref = o.layer_forward(o.Layer(w, bias_mode=bias_mode), x, forced_ids=forced_ids, forced_w=forced_w, nthreads=nt)
    assert np.array_equal(ids_gpu.cpu().numpy(), forced_ids), f"{where}: forced ids not bit-exact"
    oky, msg = parity.outputs_ok(y_gpu.float().cpu().numpy(), ref["y"])
    assert oky, f"{where}: outputs: {msg}"
    return ref, msg


def oracle_route(w, x, k=6):
    """Router-only oracle pass, one token at a time: logits, p, ids, w."""
    L = o.Layer(w)
    xf = x.view(np.uint16) if x.dtype == np.uint16 else x
    T = x.shape[0]
    logits = np.zeros((T, w.E), np.float32)
    p = np.zeros((T, w.E), np.float32)
    ids = np.zeros((T, k), np.int32)
    wt = np.zeros((T, k), np.float32)
    for t in range(T):
        row = (xf[t].astype(np.uint32) << 16).view(np.float32) if x.dtype == np.uint16 else x[t]
        logits[t] = o.router_logits(L, row)
        p[t] = o.softmax(logits[t])
        ids[t] = o.topk(p[t], k)
        wt[t] = o.renorm(p[t], ids[t])
    return dict(logits=logits, p=p, ids=ids, w=wt)
