#!/usr/bin/env python
"""Benchmark of the routed MoE expert layer (libmoe) on GB300: MoE-layer tokens/s and the
fraction of the HBM roofline of the selected experts' bytes.

Workload (headline): one Kolibri-1-shaped MoE layer (d_model 2048, ffn 640, 384 E4M3 experts
with per-row fp32 scales, top-6 + 1 shared, fp32 router with a N(0, 0.5) per-expert bias),
decode batch of 64 bf16 tokens, free routing.  A step is one moe_forward over the batch.
The same layer at batch 1 and 8 is reported under "extra".  Inputs are synthetic (seeded
counter-based generator).  Eight copies of the layer's weights are rotated across steps so
that consecutive steps never find their experts in L2 (inputs larger than L2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 (under torchrun) every rank runs an independent replica (the layer has
no cross-token exchange); the time is the maximum over ranks and the value counts the
tokens of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D, FFN, E, K = 2048, 640, 384, 6
EXPERT_BYTES = 3 * D * FFN + (2 * FFN + D) * 4          # E4M3 codes + fp32 row scales
ROUTER_BYTES = E * D * 4 + E * 4                         # fp32 router weights + bias
GATEUP_EXPERT_BYTES = 2 * FFN * D + 2 * FFN * 4
EXPERT_BYTES_W4 = 3 * D * FFN // 2 + (2 * FFN + D) * 4  # E2M1 codes (two per byte) + fp32 row scales
N_COPIES = 8
HEADLINE_T = 64
KERNELS_PER_FORWARD = 5  # router (quantises x, selects, then dispatches in its last CTA), gate_up, h_quant, down, combine (free routing, T <= 128)
PATH_FLAGS = {"auto": 0, "stream": 1, "tc": 2}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tokens", type=int, default=HEADLINE_T)
    ap.add_argument("--no-extra", action="store_true", help="skip the batch-1/8 extras")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copies", type=int, default=N_COPIES, help="weight copies rotated across steps")
    ap.add_argument("--path", choices=sorted(PATH_FLAGS), default="auto", help="expert kernels")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill extras")
    ap.add_argument("--no-stack", action="store_true", help="skip the 50-layer stack extras")
    ap.add_argument("--no-w4", action="store_true", help="skip the 4-bit weight extras")
    ap.add_argument("--weights", choices=["e4m3", "e2m1"], default="e4m3",
                    help="expert weight format of the timed layer (e2m1: the 4-bit checkpoint)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profiled_traffic(kernel_key: str):
    """DRAM bytes per launch of `kernel_key` from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken (sha256 of the sources)."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", "k_expert_tc_decode_T64.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch " + re.escape(kernel_key) + r" decode_T64: (\d+)", text)
    sh = re.search(r"source_sha256: ([0-9a-f]+)", text)
    if not m or not sh:
        return None
    h = hashlib.sha256()
    for f in ("experts_tc.cu", "tcgen05.cuh", "tma.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "routed_expert_layer_fp32_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return int(m.group(1)) if h.hexdigest() == sh.group(1) else None


def fp8_peak():
    """Dense FP8 tensor peak: the measured bf16 GEMM peak times the nominal fp8/bf16 ratio
    (4.5 / 2.25 PFLOP/s = 2); burst figure for a kernel timed alone."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        kind = "measured bf16 x 2 (nominal fp8/bf16)"
        clk = p.get("clocks_under_load", {})
        if clk.get("sm_mhz_median"):  # the bf16 GEMM was measured at this clock, under the power cap
            kind += (f"; the bf16 GEMM ran at a median SM clock of {clk['sm_mhz_median']:.0f} MHz "
                     f"(max {clk.get('sm_max_mhz', 0):.0f}) at up to {clk.get('power_w_max', 0):.0f} W")
        return 2.0 * float(p["bf16_tflops"]), kind
    return 2.0 * 1900.0, "fallback bf16 x 2"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def summary(self):
        self.file.seek(0)
        rows = [l.strip().split(",") for l in self.file.read().splitlines() if l.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except (ValueError, IndexError):
                continue
            for i, n in enumerate(names):
                if len(r) > 5 + i and r[5 + i].strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float) -> float:
    """The maximum of `value` over the ranks of the default process group (replica timing)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: int, steps: int, world: int, elapsed_ms_max: float) -> float:
    """Whole-job throughput of `world` independent replicas: every rank's units over the
    slowest rank's time."""
    return world * units_per_rank * steps / (elapsed_ms_max / 1e3)


def layer_bytes(ids: np.ndarray, T: int, w4: bool = False):
    """Algorithmic HBM bytes of one forward: the used experts (and the shared one) once, the
    router once, x read and y written in bf16."""
    U = len(np.unique(ids[ids >= 0]))
    return (U + 1) * (EXPERT_BYTES_W4 if w4 else EXPERT_BYTES) + ROUTER_BYTES + 4 * T * D, U


def gateup_bytes(U: int, T: int, w4: bool = False):
    """Algorithmic bytes of one gate/up launch: the used experts' gate/up codes and scales,
    each token's E4M3 activation row once (the kernel gathers a token's routed copies by
    token), h written once in fp32 for every (token, slot) and shared row."""
    R = (K + 1) * T
    per_expert = (FFN * D + 2 * FFN * 4) if w4 else GATEUP_EXPERT_BYTES
    return (U + 1) * per_expert + T * D + R * FFN * 4


# ------------------------------------------------------------------------------ ours ------

def run_ours(args):
    import torch
    import __graft_entry__
    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    import routed_expert_layer_fp32_gb300 as moe
    from gen import moegen as g

    hbm_peak, peak_kind = peaks()
    w4 = args.weights == "e2m1"
    w = g.kolibri_layer(g.SEED_DECODE, fp4=w4)
    base = moe.Layer.from_host(w, tiled=(args.path != "stream"))
    layers = [base]
    for _ in range(args.copies - 1):  # copies at other addresses: same values, no L2 reuse between steps
        layers.append(base.clone())
    T = args.tokens
    x_host = g.make_x(g.SEED_DECODE, T, D, bf16=True)
    x = torch.from_numpy(x_host.view(np.int16).copy()).cuda().view(torch.bfloat16)
    ws = moe.workspace(base, T)
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, K), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    flags = PATH_FLAGS[args.path]

    def step(i, ev=None):
        moe.forward(x, layers[i % len(layers)], ws, out=y, ids=ids, w=wt, events=ev, flags=flags)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # timed region: K plain steps (the kernels of a step overlap their launches, PDL)
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(args.steps):
            step(i)
        stop.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop))
    clocks = clk.summary()
    # per-kernel durations: the same steps again with events at every stage boundary (an
    # event between two kernels makes the second wait for the first to finish, so this pass
    # is only used for the per-stage split, not for the step time)
    n_trace = min(args.steps, 500)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.binding.TRACE_POINTS)] for _ in range(n_trace)]
    for row in evs:  # torch creates an event's CUDA handle at its first record()
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for i in range(n_trace):
        step(i, evs[i])
    torch.cuda.synchronize()
    stage_ms = {}
    for si, name in enumerate(moe.binding.TRACE_STAGES):
        stage_ms[name] = statistics.mean(evs[i][si].elapsed_time(evs[i][si + 1]) for i in range(n_trace))
    traced_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][-1]) for i in range(n_trace))
    ids_h = ids.cpu().numpy()
    nbytes, U = layer_bytes(ids_h, T, w4)
    gu_bytes = gateup_bytes(U, T, w4)
    ms_step = elapsed_ms / args.steps
    value = replica_throughput(T, args.steps, world, elapsed_ms)
    gu_ms = stage_ms["gate_up"]
    gu_kernel = "k_gateup_fp8" if args.path == "stream" else (
        "k_expert_tc<16,gate_up,e2m1>" if w4 else "k_expert_tc<16,gate_up>")
    traffic = profiled_traffic(gu_kernel) if (args.path != "stream" and T == HEADLINE_T) else None
    roof = {"bound": "hbm", "kernel": gu_kernel, "achieved": gu_bytes / (gu_ms * 1e-3) / 1e9,
            "peak": hbm_peak, "unit": "GB/s", "peak_kind": peak_kind,
            "frac": gu_bytes / (gu_ms * 1e-3) / 1e9 / hbm_peak, "traffic": traffic,
            "algorithmic_bytes_per_launch": gu_bytes, "launch_ms": gu_ms}
    layer_frac = nbytes / (ms_step * 1e-3) / 1e9 / hbm_peak

    # end to end through the public API a serving loop uses: per step, the copy of that step's
    # x from pinned host memory, one moe.GraphedForward replay of the layer, and the copy of y
    # back to pinned host memory.  The copies run on a second stream, double-buffered: step
    # i + 1's input comes in and step i - 1's output goes out while step i computes (events
    # order every buffer's reuse).  Every step's copies are inside the timed region.
    x_pin = torch.from_numpy(x_host.view(np.int16).copy()).pin_memory().view(torch.bfloat16)
    y_pin = [torch.empty((T, D), dtype=torch.int16).pin_memory().view(torch.bfloat16) for _ in range(2)]
    xd = [torch.empty((T, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    yd = [torch.empty((T, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    n_l = len(layers)
    fwd = [[moe.GraphedForward(xd[b], layers[i], ws, yd[b], ids, wt, flags=flags) for i in range(n_l)]
           for b in range(2)]
    io = torch.cuda.Stream()

    def e2e_run(n_steps, t0=None, t1=None):
        ev_x = [torch.cuda.Event() for _ in range(2)]    # x[b] has landed
        ev_f = [torch.cuda.Event() for _ in range(2)]    # the forward on buffer b is done
        ev_y = [torch.cuda.Event() for _ in range(2)]    # y[b] has been read back
        io.wait_stream(stream)
        if t0 is not None:
            t0.record(io)
        with torch.cuda.stream(io):
            xd[0].copy_(x_pin, non_blocking=True)
            ev_x[0].record(io)
        for i in range(n_steps):
            b = i & 1
            stream.wait_event(ev_x[b])
            if i >= 2:
                stream.wait_event(ev_y[b])  # y[b] of step i - 2 is out before it is overwritten
            fwd[b][i % n_l].replay()
            ev_f[b].record(stream)
            with torch.cuda.stream(io):
                if i + 1 < n_steps:  # the next input, once step i - 1 is done reading that buffer
                    if i >= 1:
                        io.wait_event(ev_f[1 - b])
                    xd[1 - b].copy_(x_pin, non_blocking=True)
                    ev_x[1 - b].record(io)
                io.wait_event(ev_f[b])
                y_pin[b].copy_(yd[b], non_blocking=True)
                ev_y[b].record(io)
        stream.wait_stream(io)
        if t1 is not None:
            t1.record(stream)

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, e0, e1)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))
    e2e = {"value": replica_throughput(T, args.steps, world, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 2}

    l2_label = f"inputs larger than L2: {len(layers)} weight copies rotated across steps"
    extra = {"layer_hbm_frac": layer_frac, "layer_bytes_per_step": nbytes, "unique_experts": U,
             "stage_ms": stage_ms, "traced_ms_per_step": traced_ms}
    if not w4:
        extra["w8a8_drift_T64"] = w8a8_drift(w, x_host, y, ids, wt)
    if not args.no_extra:
        for Tx in (1, 8):
            extra[f"decode_T{Tx}"] = small_batch(moe, g, layers, Tx, args, hbm_peak, flags)
        extra["zipf_forced_T128"] = zipf_forced(moe, g, layers, args, hbm_peak, flags)
    if not args.no_prefill:
        for Tx in (2048, 16384):
            extra[f"prefill_T{Tx}"] = prefill(moe, g, layers[0], Tx, flags)
        extra["prefill_T2048_as_4x512_forced"] = prefill_forced_chunks(moe, g, layers[0], flags)
    if not args.no_w4 and args.path != "stream":
        extra.update(w4_bench(moe, g, args, hbm_peak, n_copies=len(layers), prefill_too=not args.no_prefill))
    if not args.no_stack:
        del layers[1:]
        torch.cuda.empty_cache()
        extra.update(stack_bench(moe, g, hbm_peak, flags))

    status = moe.get_status(ws)
    out = {
        "metric": "MoE-layer tokens/s (decode, batch 64); % of HBM roofline",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e2m1 weights, bf16 activations, fp32 accumulate (W4A8)" if w4 else
                  "e4m3 weights, bf16 activations, fp32 accumulate (W8A8)"), "data": "synthetic (seeded)",
        "config": {"workload": f"kolibri moe layer decode T={T} (d=2048, ffn=640, 384 experts top-6 + 1 shared, "
                               f"{'E2M1' if w4 else 'E4M3'} weights, bias N(0,0.5))", "tokens": T, "layers": 1,
                   "l2": l2_label,
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "clocks": clocks, "e2e": e2e,
        "gpu_launches": args.steps * KERNELS_PER_FORWARD, "device_status": status, "extra": extra,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, x_host)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


def prefill(moe, g, layer, T, flags, warmup=3, iters=10, expert_bytes=None):
    """One prefill-sized layer call (free routing): `ms_per_layer` over back-to-back calls
    (events around the loop), `traced_ms_per_layer` and `stage_ms` with an event at every stage
    boundary (which also stops the next kernel from starting early).  Two rooflines: the
    expert FLOPs 7T x 3 x 2 x d x ffn (six routed rows and one shared row per token) against
    the FP8 peak, and the bytes of the experts the call touches (at a few thousand tokens
    nearly all of them) against HBM."""
    import torch
    peak, kind = fp8_peak()
    hbm_peak, _ = peaks()
    x = torch.from_numpy(g.make_x(g.SEED_PREFILL, T, D, bf16=True).view(np.int16).copy()).cuda().view(torch.bfloat16)
    ws = moe.workspace(layer, T)
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    for _ in range(warmup):
        _, ids, _ = moe.forward(x, layer, ws, out=y, flags=flags)
    torch.cuda.synchronize()
    unique = len(np.unique(ids.cpu().numpy()))
    nbytes = (unique + 1) * (expert_bytes or EXPERT_BYTES) + ROUTER_BYTES + 2 * T * D
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        moe.forward(x, layer, ws, out=y, flags=flags)
    e1.record()
    torch.cuda.synchronize()
    plain = e0.elapsed_time(e1) / iters
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.binding.TRACE_POINTS)] for _ in range(iters)]
    for row in evs:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(iters):
        moe.forward(x, layer, ws, out=y, flags=flags, events=evs[i])
    torch.cuda.synchronize()
    total = statistics.mean(evs[i][0].elapsed_time(evs[i][-1]) for i in range(iters))
    stage = {n: statistics.mean(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(iters))
             for k, n in enumerate(moe.binding.TRACE_STAGES)}
    flops = 7 * T * 3 * 2 * D * FFN
    gemm_ms = stage["gate_up"] + stage["down"]
    return {"tokens_per_s": T / (plain * 1e-3), "ms_per_layer": plain, "traced_ms_per_layer": total,
            "expert_tflops": flops / (plain * 1e-3) / 1e12, "fp8_frac": flops / (plain * 1e-3) / 1e12 / peak,
            "gemm_fp8_frac": flops / (gemm_ms * 1e-3) / 1e12 / peak, "unique_experts": unique, "bytes": nbytes,
            "hbm_frac": nbytes / (plain * 1e-3) / 1e9 / hbm_peak, "fp8_peak_tflops": peak, "peak_kind": kind,
            "stage_ms": stage}


def stack_bench(moe, g, hbm_peak, flags):
    """The 50-layer stack (r <- bf16(r + moe(r)), free routing, ~76 GB of E4M3 weights
    resident): decode with 32 tokens and a 16,384-token prefill, each one moe_forward_stack
    call per step, timed with CUDA events (the residual is reset from the input every step).
    The decode step is replayed as one CUDA graph (GraphedStack: the input copy and the 50
    layers' launches), as a serving loop would run it; the prefill step is called directly."""
    import torch
    t0 = time.time()
    layers = [moe.Layer.from_host(g.stack_layer(l)) for l in range(g.STACK_LAYERS)]
    gen_s = time.time() - t0
    arr = moe.binding.layer_array(layers)
    peak8, kind8 = fp8_peak()
    out = {}
    for T, iters in ((32, 20), (16384, 3)):
        x = torch.from_numpy(g.stack_x(T).view(np.int16).copy()).cuda().view(torch.bfloat16)
        r = x.clone()
        ws = moe.workspace(layers[0], T)
        ids = torch.empty((len(layers), T, K), dtype=torch.int32, device="cuda")
        if T == 32:
            graphed = moe.GraphedStack(layers, r, ws, x=x, ids_out=ids, flags=flags, layer_arr=arr)
            step = graphed.replay
        else:
            def step():
                r.copy_(x)
                moe.forward_stack(layers, r, ws, ids_out=ids, flags=flags, layer_arr=arr)
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            step()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        idh = ids.cpu().numpy()
        us = [len(np.unique(idh[l])) for l in range(len(layers))]
        if T == 32:
            nbytes = sum((u + 1) * EXPERT_BYTES + ROUTER_BYTES + 4 * T * D for u in us)
            out["stack_decode_T32"] = {"tokens_per_s": T / (ms * 1e-3), "ms_per_stack": ms,
                                       "ms_per_layer": ms / len(layers), "bytes": nbytes,
                                       "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
                                       "unique_experts_mean": float(np.mean(us)), "layers": len(layers),
                                       "step": "one CUDA graph (GraphedStack)"}
        else:
            flops = len(layers) * 7 * T * 3 * 2 * D * FFN
            out["stack_prefill_T16384"] = {"tokens_per_s": T / (ms * 1e-3), "ms_per_stack": ms,
                                           "ms_per_layer": ms / len(layers), "expert_tflops": flops / (ms * 1e-3) / 1e12,
                                           "fp8_frac": flops / (ms * 1e-3) / 1e12 / peak8, "fp8_peak_tflops": peak8,
                                           "peak_kind": kind8, "layers": len(layers)}
        status = moe.get_status(ws)
        out[f"stack_T{T}_device_status"] = status
    out["stack_weight_generation_s"] = gen_s
    del layers
    torch.cuda.empty_cache()
    return out


def small_batch(moe, g, layers, T, args, hbm_peak, flags=0):
    """Batch-T decode of the same layer, captured in a CUDA graph (launch overhead excluded)."""
    import torch
    x_host = g.make_x(g.SEED_DECODE, T, D, bf16=True)
    x = torch.from_numpy(x_host.view(np.int16).copy()).cuda().view(torch.bfloat16)
    ws = moe.workspace(layers[0], T)
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, K), dtype=torch.float32, device="cuda")
    n = len(layers)
    for i in range(n):
        moe.forward(x, layers[i], ws, out=y, ids=ids, w=wt, flags=flags)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for i in range(n):
                moe.forward(x, layers[i], ws, out=y, ids=ids, w=wt, flags=flags)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // n)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * n)
    nbytes, U = layer_bytes(ids.cpu().numpy(), T)
    stage_ms, traced_ms = traced_stages(moe, layers, x, ws, y, ids, wt, flags, iters=min(200, args.steps))
    return {"tokens_per_s": T / (ms * 1e-3), "ms_per_layer": ms, "unique_experts": U, "bytes": nbytes,
            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm_peak, "timing": f"CUDA graph over {n} layer copies",
            "stage_ms": stage_ms, "traced_ms_per_layer": traced_ms,
            "stage_note": "eager launches with an event at every stage boundary (each stage waits for the "
                          "previous one to finish), so the stages sum to more than the graphed layer time"}


def traced_stages(moe, layers, x, ws, y, ids, wt, flags, iters):
    """Mean duration of each kernel stage: eager forwards over the rotated layer copies with
    events at the stage boundaries."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.binding.TRACE_POINTS)] for _ in range(iters)]
    for row in evs:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(iters):
        moe.forward(x, layers[i % len(layers)], ws, out=y, ids=ids, w=wt, events=evs[i], flags=flags)
    torch.cuda.synchronize()
    stage = {nm: statistics.mean(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(iters))
             for k, nm in enumerate(moe.binding.TRACE_STAGES)}
    return stage, statistics.mean(evs[i][0].elapsed_time(evs[i][-1]) for i in range(iters))


def w8a8_drift(w, x_host, y_dev, ids_dev, w_dev):
    """Distance of the GPU layer (W8A8: E4M3 weights and per-row E4M3 activations) from a W8A16
    evaluation of the same layer: dequantised E4M3 weights times their row scales, activations
    kept in fp32, the GPU's own ids and routing weights, evaluated with torch on the host in
    float64.  Reported, not gated (the activation quantisation is this library's reading of the
    pages' FP8 contractions)."""
    import torch
    T = x_host.shape[0]
    x = torch.from_numpy((x_host.astype(np.uint32) << 16).view(np.float32)).double()
    ids = ids_dev.cpu().numpy()
    wts = torch.from_numpy(w_dev.cpu().numpy()).double()
    y_gpu = y_dev.float().cpu().double()

    def deq(codes, scales):
        return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double() * \
            torch.from_numpy(np.ascontiguousarray(scales)).double()[:, None]

    def ffn(gu, sgu, dn, sd, xs):
        g_ = xs @ deq(gu[0], sgu[0]).T
        u_ = xs @ deq(gu[1], sgu[1]).T
        return (g_ / (1 + torch.exp(-g_)) * u_) @ deq(dn, sd).T

    y_ref = ffn(w.sh_Wgu, w.sh_sgu, w.sh_Wd, w.sh_sd, x)
    for e in np.unique(ids):
        tt, slot = np.nonzero(ids == e)
        ye = ffn(w.Wgu[e], w.sgu[e], w.Wd[e], w.sd[e], x[tt])
        y_ref[tt] += wts[tt, slot][:, None] * ye
    diff = y_gpu - y_ref
    return {"rel_l2": float(diff.norm() / y_ref.norm()),
            "max_err_frac": float(diff.abs().max() / y_ref.abs().max()), "tokens": T,
            "reference": "W8A16 on the host (torch float64, dequantised E4M3 weights, fp32 activations, "
                         "the GPU's ids and weights)"}


def w4_bench(moe, g, args, hbm_peak, n_copies, prefill_too):
    """The same Kolibri-shaped layer with 4-bit expert weights (E2M1 codes + fp32 row scales,
    W4A8): decode at batch 1, 8 and 64 (CUDA graph over rotated weight copies, as small_batch)
    with the HBM fraction over the 4-bit bytes of the selected experts, and the 16k prefill."""
    import torch
    w = g.kolibri_layer(g.SEED_DECODE, fp4=True)
    base = moe.Layer.from_host(w)
    layers = [base] + [base.clone() for _ in range(n_copies - 1)]
    out = {}
    for T in (1, 8, 64):
        x = torch.from_numpy(g.make_x(g.SEED_DECODE, T, D, bf16=True).view(np.int16).copy()).cuda().view(torch.bfloat16)
        ws = moe.workspace(base, T)
        y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
        ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
        wt = torch.empty((T, K), dtype=torch.float32, device="cuda")
        for lay in layers:
            moe.forward(x, lay, ws, out=y, ids=ids, w=wt)
        torch.cuda.synchronize()
        st = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(st):
            with torch.cuda.graph(graph, stream=st):
                for lay in layers:
                    moe.forward(x, lay, ws, out=y, ids=ids, w=wt)
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        reps = max(1, args.steps // len(layers))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * len(layers))
        U = len(np.unique(ids.cpu().numpy()))
        nbytes = (U + 1) * EXPERT_BYTES_W4 + ROUTER_BYTES + 4 * T * D
        stage_ms, traced = traced_stages(moe, layers, x, ws, y, ids, wt, 0, iters=min(200, args.steps))
        out[f"w4_decode_T{T}"] = {"tokens_per_s": T / (ms * 1e-3), "ms_per_layer": ms, "unique_experts": U,
                                  "bytes": nbytes, "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
                                  "weights": "E2M1 + fp32 row scales", "stage_ms": stage_ms,
                                  "timing": f"CUDA graph over {len(layers)} layer copies"}
        if T == 64:  # the gate/up kernel alone, over its algorithmic bytes
            gu_bytes = (U + 1) * (FFN * D + 2 * FFN * 4) + T * D + (K + 1) * T * FFN * 4
            out["w4_decode_T64"]["gate_up_hbm_frac"] = gu_bytes / (stage_ms["gate_up"] * 1e-3) / 1e9 / hbm_peak
    del layers
    if prefill_too:
        out["w4_prefill_T16384"] = prefill(moe, g, base, 16384, 0, expert_bytes=EXPERT_BYTES_W4)
    torch.cuda.empty_cache()
    return out


def zipf_forced(moe, g, layers, args, hbm_peak, flags=0, T=128):
    """Batched decode of 128 tokens with forced routing: Zipf(1.1) expert ids (six per token,
    without replacement) and Dirichlet(1) weights, the load-imbalanced grouped GEMM; CUDA graph
    over the rotated layer copies, as small_batch."""
    import torch
    x = torch.from_numpy(g.make_x(g.SEED_ZIPF, T, D, bf16=True).view(np.int16).copy()).cuda().view(torch.bfloat16)
    fid_h = g.zipf_ids(g.SEED_ZIPF, 0, T, 384, K, 1.1)
    fid = torch.from_numpy(fid_h).cuda()
    fw = torch.from_numpy(g.dirichlet_w(g.SEED_ZIPF, 0, T, K)).cuda()
    ws = moe.workspace(layers[0], T)
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, K), dtype=torch.float32, device="cuda")
    n = len(layers)

    def run():
        for i in range(n):
            moe.forward(x, layers[i], ws, forced_ids=fid, forced_w=fw, out=y, ids=ids, w=wt, flags=flags)

    run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    reps = max(1, args.steps // n)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * n)
    nbytes, U = layer_bytes(fid_h, T)
    return {"tokens_per_s": T / (ms * 1e-3), "ms_per_layer": ms, "unique_experts": U, "bytes": nbytes,
            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm_peak, "timing": f"CUDA graph over {n} layer copies"}


def prefill_forced_chunks(moe, g, layer, flags, T=2048, chunk=512, iters=10):
    """The 2048-token prefill run free once (recording ids), then replayed as four 512-token
    calls with routing forced from the recorded ids (weights from each call's own router);
    tokens/s over the four forced calls, timed with CUDA events."""
    import torch
    x = torch.from_numpy(g.make_x(g.SEED_PREFILL, T, D, bf16=True).view(np.int16).copy()).cuda().view(torch.bfloat16)
    ws = moe.workspace(layer, T)
    y = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")
    _, ids, _ = moe.forward(x, layer, ws, out=y, flags=flags)
    ids = ids.clone()
    yc = torch.empty((T, D), dtype=torch.bfloat16, device="cuda")

    def run():
        for c in range(0, T, chunk):
            moe.forward(x[c:c + chunk], layer, ws, forced_ids=ids[c:c + chunk], out=yc[c:c + chunk], flags=flags)

    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    idh = ids.cpu().numpy()
    nbytes = sum((len(np.unique(idh[c:c + chunk])) + 1) * EXPERT_BYTES + ROUTER_BYTES + 2 * chunk * D
                 for c in range(0, T, chunk))
    return {"tokens_per_s": T / (ms * 1e-3), "ms_per_2048_tokens": ms, "calls": T // chunk, "bytes": nbytes,
            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peaks()[0]}


# ---------------------------------------------------------------------------- oracle ------

def cpu_baseline(w, x_host, budget_s=10.0):
    """The CPU oracle as it stands, token-sharded over all host cores, on repeats of the same
    64-token batch until about budget_s seconds have passed."""
    from oracle import oracle as o
    cores = os.cpu_count() or 1
    L = o.Layer(w)
    T = x_host.shape[0]
    n = 0
    t0 = time.time()
    while time.time() - t0 < budget_s:
        o.layer_forward(L, x_host, nthreads=cores)
        n += 1
    dt = time.time() - t0
    return {"value": n * T / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} x the {T}-token decode batch ({n * T} token-layers), {dt:.1f} s wall"}


def run_reference(args):
    world, rank, local = dist_setup(args)
    if rank != 0:
        return
    from gen import moegen as g
    from oracle import oracle as o
    o.build()
    w = g.kolibri_layer(g.SEED_DECODE)
    T = args.tokens
    x_host = g.make_x(g.SEED_DECODE, T, D, bf16=True)
    cores = os.cpu_count() or 1
    L = o.Layer(w)
    for _ in range(args.warmup):
        o.layer_forward(L, x_host, nthreads=cores)
    t0 = time.time()
    for _ in range(args.steps):
        o.layer_forward(L, x_host, nthreads=cores)
    dt = time.time() - t0
    value = T * args.steps / dt
    out = {"metric": "MoE-layer tokens/s (decode, batch 64); % of HBM roofline", "value": value,
           "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "e4m3 weights, bf16 activations, fp32 accumulate (W8A8)", "data": "synthetic (seeded)",
           "config": {"workload": f"kolibri moe layer decode T={T} (d=2048, ffn=640, 384 experts top-6 + 1 shared, "
                                  f"E4M3 weights, bias N(0,0.5))", "tokens": T, "layers": 1,
                      "parallelism": "host cores"},
           "impl": "reference",
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": f"{args.steps} timed steps of the {T}-token batch"},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
