#!/usr/bin/env python
"""MoE layer forward+backward tokens/s on one GB300 (the layer's hot path).

One step = route (top-k) -> schedule -> dispatch -> gate/up GEMM + SwiGLU ->
down GEMM -> combine -> reverse-combine (+ d routing weights) -> down
dgrad (+ SwiGLU backward) -> down wgrad -> gate/up dgrad -> gate/up wgrad ->
reverse-dispatch, on one batch of seeded synthetic input already resident in
HBM. Default workload: N=16384 tokens, H=4096, I=1536, E=128 experts, top-8,
bf16, router logits plus a Zipf(1.2) per-expert bias (skewed expert loads).

Multi-GPU (torchrun, N ranks): replicas only -- every rank runs its own batch
with no collective on the data path ("scaling": "weak"); the barrier and the
max over ranks of the timed region stay.

--impl reference times the CPU oracle (fp64 C++, all host cores) on a
bounded sample of the same workload; it is a deliberately slow correctness
reference, not a tuned competitor.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd tokens/s on 1 GB300; GEMM TFLOP/s as % of tensor peak"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=None,
                    help="workload name (default: skewed fwd+bwd) or "
                         "N,H,I,E,k[,zipf][,T=..][,mxfp8][,fwd] (fwd: forward only)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=0,
                    help="oracle sample size in tokens (0 = sized for ~15 s)")
    ap.add_argument("--phase-report", action="store_true", help="print per-phase timings")
    ap.add_argument("--router", action="store_true",
                    help="start from x: the router GEMM (x . Wr^T) and its backward run on the "
                         "GPU inside the step (default: the step starts from router logits)")
    ap.add_argument("--stages", type=int, default=0, choices=[0, 4, 5, 6],
                    help="ring stages of the bf16 SM-pair GEMMs (0: the library's per-shape choice)")
    ap.add_argument("--tile-n", type=int, default=0, choices=[0, 256, 512],
                    help="pair-tile width of the bf16 token-row GEMMs (0: the library's choice)")
    ap.add_argument("--sweep-stages", action="store_true",
                    help="time the workload with 4, 5 and 6 GEMM ring stages (256-wide pair "
                         "tiles) and with 512-wide token-row tiles, and print every GEMM "
                         "phase's time at each and its best setting")
    ap.add_argument("--sweep-T", action="store_true",
                    help="the minibatch knob sweep: run the workload at minibatch_rows T = 128, "
                         "256, 512, 1024 and print one line with every T's result and the best")
    ap.add_argument("--overlap", action="store_true",
                    help="bf16 backward through moe_backward_overlap (the reverse-combine run "
                         "by side warps of the down data-gradient GEMM), timed as one phase")
    ap.add_argument("--inference", action="store_true",
                    help="forward-only workloads: time the context-free forward (no G, U or "
                         "context stored) instead of the training forward")
    ap.add_argument("--fused", action="store_true",
                    help="bf16 training forward: time dispatch, gate/up and down as one "
                         "persistent launch (moe_dispatch_expert_ffn) instead of three")
    ap.add_argument("--unfused", action="store_true",
                    help="bf16 context-free forward (--inference): time dispatch, gate/up and "
                         "down as three launches instead of moe_dispatch_expert_ffn")
    ap.add_argument("--tensor-peaks", action="store_true",
                    help="measure the dense bf16 and FP8 (E4M3) tensor-core peaks with library "
                         "GEMMs of 8192^3 (best of 10, and back to back for 4 s) and print them")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured once in a CUDA graph and replayed "
                         "(reported as \"graph\"; the headline stays the eager step)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws_, device):
    """The largest x over all ranks: the slowest replica sets the job's time."""
    if ws_ <= 1:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_step, steps, ws_, elapsed_ms):
    """Whole-job tokens/s of ws_ replicas that each process tokens_per_step
    tokens per step (weak scaling), over the slowest replica's time."""
    return tokens_per_step * steps * ws_ / (elapsed_ms * 1e-3)


def output_tensors(layer, backward, dw_router=None):
    """The step's outputs, in the fixed order the digest reads them."""
    out = {"y": layer.y}
    if backward:
        g = layer.grads
        out.update(dx=g.dx, dw_gate=g.dw_gate, dw_up=g.dw_up, dw_down=g.dw_down,
                   d_topk_w=g.d_topk_w)
        if dw_router is not None:
            out["dw_router"] = dw_router
    return out


def output_digest(tensors, chunk_bytes=1 << 28):
    """SHA-256 over the bytes of every tensor (in dict order), read back in
    chunks so the host never holds more than one chunk."""
    import hashlib

    import torch
    h = hashlib.sha256()
    for t in tensors.values():
        b = t.detach().reshape(-1).view(torch.uint8)
        for i in range(0, b.numel(), chunk_bytes):
            h.update(b[i:i + chunk_bytes].cpu().numpy().tobytes())
    return h.hexdigest()


def rerun_check(step, outputs, digest_keys=("y", "dx", "d_topk_w")):
    """Run one more step on the same inputs and compare every output with the
    previous step's, byte for byte (the combine and every reduction have a
    fixed order, so reruns must be identical). The SHA-256 fingerprint covers
    the token-sized outputs only (the fp32 weight gradients are compared on
    the device but not read back)."""
    import torch
    first = {k: v.clone() for k, v in outputs.items()}
    digest = output_digest({k: first[k] for k in digest_keys if k in first})
    step()
    if torch.cuda.is_available():
        torch.cuda.synchronize()
    same = {k: bool(torch.equal(first[k].reshape(-1).view(torch.uint8),
                                v.reshape(-1).view(torch.uint8))) for k, v in outputs.items()}
    del first
    return {"rerun_bitwise_equal": all(same.values()), "compared": list(outputs),
            "sha256": digest, "sha256_of": [k for k in digest_keys if k in outputs]}


def graph_timing(step, warmup, K, ws_, tokens, dev):
    """The same step captured once in a CUDA graph, replayed warmup + K times;
    the K replays timed with CUDA events like the eager steps. The library
    enqueues everything on the capturing stream and never allocates or
    synchronises, so the capture holds the whole pass."""
    import torch
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    if ws_ > 1:
        torch.distributed.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    t0.record(s)
    for _ in range(K):
        graph.replay()
    t1.record(s)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), ws_, dev)
    del graph
    return {"ms_per_step": round(ms / K, 4),
            "value": round(replica_throughput(tokens, K, ws_, ms), 1)}


def expert_loads(counts, tile_rows=128):
    """Tokens per expert (m_e) and the share of grouped-GEMM rows that are
    padding when each expert's rows are rounded up to whole tiles."""
    m = [int(c) for c in counts]
    A = sum(m)
    padded = sum(-(-c // tile_rows) * tile_rows for c in m)
    return {"m_e_max": max(m), "m_e_mean": A / len(m), "m_e_min": min(m),
            "empty_experts": sum(c == 0 for c in m), "tile_rows": tile_rows,
            "padded_row_frac": round((padded - A) / padded, 4) if padded else 0.0}


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# grouped-GEMM phases, from one single-pass ncu capture of the default
# workload (summary in profiles/). A value is reported only while the GEMM
# kernel source still hashes to the value it was captured with.
GEMM_SRC = ("mixture_experts_layer_schedule_gb300/csrc/grouped_gemm.cu",
            "mixture_experts_layer_schedule_gb300/csrc/moe_common.cuh")
MEASURED_TRAFFIC = {
    "src_sha256": "77f82cf6ac992b7cce412d0585002b8e66c2dee7852f35c0bbb2ab736af31521",
    "workload": "skewed_fwd_bwd_N16384_H4096_I1536_E128_k8_zipf1.2",
    "bytes": {"gate_up": 5.381e9 + 1.299e9,
              "down": 2.072e9 + 1.145e9,
              "down_dgrad": 3.920e9 + 0.855e9,
              "down_wgrad": 2.378e9 + 3.168e9,
              "gate_up_dgrad": 4.762e9 + 1.156e9,
              "gate_up_wgrad": 4.751e9 + 6.393e9},
}

def measured_traffic(workload_name, phase):
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SRC:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != MEASURED_TRAFFIC["src_sha256"]:
        return None
    if workload_name != MEASURED_TRAFFIC["workload"]:
        return None
    return MEASURED_TRAFFIC["bytes"].get(phase)


# The dense FP8 tensor-core peak of the GB300s, measured with
# `python bench.py --tensor-peaks` (a library E4M3 GEMM, torch._scaled_mm with
# per-tensor scales, 8192^3, CUDA events; sustained = back to back for 4 s
# under the power cap). Without it the FP8 fractions would use the bf16 peak
# times the nominal FP8 / bf16 ratio. One GB300, 2070 MHz maximum clock; the
# sustained run held the power cap at a median 1432 MHz (the bf16 GEMM beside
# it: 1919 burst, 1711 sustained, matching the copy/GEMM peak file). The
# burst figure is the best of 10 isolated launches and came out below the
# sustained one; the roofline uses the sustained figure, as the GEMMs run
# inside a long step.
MEASURED_FP8 = {"burst_tflops": 2967.7, "sustained_tflops": 3360.1, "gpu": "GB300",
                "when": "2026-12-03"}


def tensor_peaks(seconds=4.0):
    """Dense bf16 and FP8 GEMM throughput of 8192^3 problems on this GPU:
    best of 10 launches (burst) and the mean over `seconds` of back-to-back
    launches (sustained), with the SM clock sampled meanwhile."""
    import torch
    n = 8192
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn((n, n), device=dev, generator=g).to(torch.bfloat16)
    b = torch.randn((n, n), device=dev, generator=g).to(torch.bfloat16)
    a8 = (a * 0.25).to(torch.float8_e4m3fn)
    b8 = (b * 0.25).to(torch.float8_e4m3fn)
    one = torch.ones((), device=dev, dtype=torch.float32)
    runs = {"bf16": lambda: torch.matmul(a, b.t()),
            "fp8_e4m3": lambda: torch._scaled_mm(a8, b8.t(), scale_a=one, scale_b=one,
                                                 out_dtype=torch.bfloat16)}
    flops = 2.0 * n ** 3
    out = {}
    for name, fn in runs.items():
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        per = max(1, int(seconds * 1e3 / best))
        clk = ClockSampler(torch.cuda.current_device())
        clk.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(per):
            fn()
        e1.record()
        torch.cuda.synchronize()
        clocks = clk.stop()
        sus = e0.elapsed_time(e1) / per
        out[name] = {"burst_tflops": round(flops / (best * 1e-3) / 1e12, 1),
                     "sustained_tflops": round(flops / (sus * 1e-3) / 1e12, 1),
                     "launches_sustained": per, "clocks": clocks}
    out["how"] = ("8192^3 GEMMs, bf16 torch.matmul and E4M3 torch._scaled_mm (per-tensor scales, "
                  "bf16 out); burst = best of 10, sustained = back to back for "
                  f"{seconds:.0f} s; CUDA events")
    return out


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        pk = dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                  bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                  source="measured")
    else:
        pk = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                  source="fallback")
    if MEASURED_FP8 is not None:
        pk.update(fp8_tflops=MEASURED_FP8["burst_tflops"],
                  fp8_tflops_sustained=MEASURED_FP8["sustained_tflops"],
                  fp8_source="measured (bench.py --tensor-peaks)")
    else:
        pk.update(fp8_tflops=2.0 * pk["bf16_tflops"],
                  fp8_tflops_sustained=2.0 * pk["bf16_tflops_sustained"],
                  fp8_source=f"{pk['source']} bf16 x 2 (nominal FP8/bf16 ratio)")
    return pk


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def phase_flops(shape):
    """Algorithmic flops of each GEMM phase (padding rows excluded)."""
    A, H, I = shape.N * shape.k, shape.H, shape.I
    return {"gate_up": 4 * A * H * I,
            "gate_up_act": 4 * A * H * I, "experts_fwd": 6 * A * H * I,
            "experts_fwd_inf": 6 * A * H * I,
            "down": 2 * A * H * I, "down_dgrad": 2 * A * H * I,
            "down_wgrad": 2 * A * H * I, "gate_up_dgrad": 4 * A * H * I,
            "gate_up_wgrad": 4 * A * H * I, "forward": 6 * A * H * I, "backward": 12 * A * H * I}


def gemm_bytes(shape):
    """Least HBM bytes of each bf16 GEMM phase: every operand read once and
    every output written once (padding rows excluded). Set against the
    phase's time this places a GEMM on the bandwidth roofline too, which
    matters where few tokens per expert meet large weights."""
    N, A, H, I, E = shape.N, shape.N * shape.k, shape.H, shape.I, shape.E
    W = 2 * E * H * I  # one bf16 weight tensor
    return {"experts_fwd": 2 * N * H + 2 * A * H + 3 * W + 3 * 2 * A * I + 2 * A * H,
            "experts_fwd_inf": 2 * N * H + 3 * W + 2 * A * H,
            "gate_up": 2 * A * H + 2 * W + 3 * 2 * A * I,
            "gate_up_act": 2 * A * H + 2 * W + 2 * A * I,
            "down": 2 * A * I + W + 2 * A * H,
            "down_dgrad": 2 * A * H + W + 2 * 2 * A * I + 2 * 2 * A * I,
            "down_wgrad": 2 * A * H + 2 * A * I + 2 * W,
            "gate_up_dgrad": 2 * 2 * A * I + 2 * W + 2 * A * H,
            "gate_up_wgrad": 2 * 2 * A * I + 2 * A * H + 4 * W}


def phase_bytes(shape, R, router=False):
    """Algorithmic HBM bytes of the data-movement phases."""
    N, A, H, E, k = shape.N, shape.N * shape.k, shape.H, shape.E, shape.k
    # route: logits in, ids and weights out; with the router GEMM, x and Wr in instead
    route = (2 * N * H + 2 * E * H if router else 4 * N * E) + 8 * N * k
    return {"route": route, "schedule": 4 * A + 12 * A + 8 * E,
            # dz, the router share of dx (dx read and written), Xe read once, dWr written
            "router_backward": 16 * A + 4 * N * H + 2 * A * H + 4 * E * H,
            "dispatch": 2 * N * H + 2 * A * H + 4 * A,
            "combine": 2 * A * H + 8 * A + 2 * N * H,
            "reverse_combine": 2 * N * H + 2 * A * H + 8 * A + 2 * A * H + 4 * A,
            "reverse_dispatch": 2 * A * H + 4 * A + 2 * N * H}


def workload(name):
    """A named workload, or "N,H,I,E,k[,zipf_s]" for a profiling case."""
    from mixture_experts_layer_schedule_gb300 import inputs
    if not name:
        return inputs.SKEWED
    if name in inputs.ALL:
        return inputs.ALL[name]
    f = name.split(",")
    dtype, T, backward = "bf16", 128, True
    while len(f) > 5 and (f[-1] in ("mxfp8", "fwd") or f[-1].startswith("T=")):
        tok = f.pop()
        if tok == "mxfp8":
            dtype = tok
        elif tok == "fwd":
            backward = False
        else:
            T = int(tok[2:])
    N, H, I, E, k = (int(v) for v in f[:5])
    z = float(f[5]) if len(f) > 5 and float(f[5]) > 0 else None
    return inputs.LayerShape(f"custom_N{N}_H{H}_I{I}_E{E}_k{k}" + (f"_zipf{z}" if z else "")
                             + f"_T{T}" + ("_mxfp8" if dtype == "mxfp8" else "")
                             + ("" if backward else "_fwd"), N, H, I, E, k,
                             zipf_s=z, minibatch_rows=T, dtype=dtype, backward=backward)


def run_ours(args, ws_, rank, local, shape=None, stages=None, tile_n=None):
    import torch
    from mixture_experts_layer_schedule_gb300 import MoELayer, _lib, inputs

    shape = shape or workload(args.config)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # replicas: the same parameters, their own tokens and upstream gradients
    inp = inputs.make_inputs(shape, seed=rank, device=dev, weight_seed=0)
    mx = shape.dtype == "mxfp8"
    stages = args.stages if stages is None else stages
    tile_n = args.tile_n if tile_n is None else tile_n
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev,
                     minibatch_rows=shape.minibatch_rows, dtype=shape.dtype,
                     pipeline_stages=stages, tile_n=tile_n)
    p, wsb = layer.p, layer.ws
    wbwd = mxw = None
    if mx:  # weights pre-quantised once, outside the timed steps
        fwd_w, wbwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
        mxw = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
        inp["w_src"] = (inp["wg"], inp["wu"], inp["wd"])  # the bf16 weights, for the oracle
        inp["wg"], inp["wu"], inp["wd"] = fwd_w
    mxs = mxw.struct if mxw is not None else None
    w = _lib.weights(inp["wg"], inp["wu"], inp["wd"], mx=mxs)
    wfull = _lib.weights(inp["wg"], inp["wu"], inp["wd"], *(wbwd or (None, None, None)), mx=mxs)
    sv = layer.saved_tensors()
    g = layer.grads
    dyxe = torch.empty((layer.R, shape.H), dtype=torch.bfloat16, device=dev)
    dgb = torch.empty((layer.R, shape.I), dtype=torch.bfloat16, device=dev)
    dub = torch.empty((layer.R, shape.I), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    backward = shape.backward

    inference = args.inference and not backward
    fwd = ["experts_fwd"] if args.fused else ["dispatch", "gate_up", "down"]
    phases = ["route", "schedule"] + fwd + ["combine"]
    if inference:
        phases = (["route", "schedule", "dispatch", "gate_up_act", "down", "combine"] if args.unfused
                  else ["route", "schedule", "experts_fwd_inf", "combine"])
    if mx:  # MXFP8: the composite passes (they add the activation quantisations)
        phases = ["route", "schedule", "forward"] + (["backward"] if backward else [])
    elif backward and args.overlap:
        phases += ["backward"]
    elif backward:
        phases += ["reverse_combine", "down_dgrad", "down_wgrad", "gate_up_dgrad",
                   "gate_up_wgrad", "reverse_dispatch"]
    router = args.router
    if router and backward:
        phases += ["router_backward"]
    dwr = torch.empty((shape.E, shape.H), dtype=torch.float32, device=dev) if router else None
    calls = {
        "route": (lambda: _lib.moe_route(p, inp["x"], inp["w_router"], inp["bias"], None,
                                         layer.topk_ids, layer.topk_w, wsb)) if router else
                 (lambda: _lib.moe_route_topk(p, inp["logits"], inp["bias"], layer.topk_ids,
                                              layer.topk_w, wsb)),
        "router_backward": lambda: _lib.moe_router_backward(
            p, layer.saved, inp["w_router"], layer.topk_ids, layer.topk_w, g.d_topk_w, g.dx, dwr,
            wsb),
        "schedule": lambda: _lib.moe_build_schedule(p, layer.topk_ids, wsb),
        "dispatch": lambda: _lib.moe_dispatch(p, wsb, inp["x"], sv["xe"]),
        "experts_fwd": lambda: _lib.moe_dispatch_expert_ffn(p, wsb, inp["x"], w, sv["xe"], sv["g"],
                                                            sv["u"], sv["act"], sv["ye"]),
        # context-free: Xe and Ye share the Ye rows the combine reads
        "experts_fwd_inf": lambda: _lib.moe_dispatch_expert_ffn(p, wsb, inp["x"], w, sv["ye"], None,
                                                                None, sv["act"], sv["ye"]),
        "gate_up": lambda: _lib.moe_expert_gate_up(p, wsb, sv["xe"], w, sv["g"], sv["u"],
                                                   sv["act"]),
        "gate_up_act": lambda: _lib.moe_expert_gate_up(p, wsb, sv["xe"], w, None, None, sv["act"]),
        "down": lambda: _lib.moe_expert_down(p, wsb, sv["act"], w, sv["ye"]),
        "combine": lambda: _lib.moe_combine(p, wsb, sv["ye"], layer.topk_w, layer.y),
        "reverse_combine": lambda: _lib.moe_reverse_combine(p, wsb, inp["dy"], sv["ye"],
                                                            layer.topk_w, dyxe, g.d_topk_w),
        "down_dgrad": lambda: _lib.moe_expert_down_dgrad(p, wsb, dyxe, sv["g"], sv["u"], w, dgb,
                                                         dub),
        "down_wgrad": lambda: _lib.moe_expert_down_wgrad(p, wsb, dyxe, sv["act"], g.dw_down),
        "gate_up_dgrad": lambda: _lib.moe_expert_gate_up_dgrad(p, wsb, dgb, dub, w, dyxe),
        "gate_up_wgrad": lambda: _lib.moe_expert_gate_up_wgrad(p, wsb, dgb, dub, sv["xe"],
                                                               g.dw_gate, g.dw_up),
        "reverse_dispatch": lambda: _lib.moe_reverse_dispatch(p, wsb, dyxe, g.dx),
        "forward": lambda: _lib.moe_forward(p, inp["x"], w, layer.topk_w, layer.y, layer.saved,
                                            wsb),
        "backward": lambda: (_lib.moe_backward_overlap if args.overlap else _lib.moe_backward)(
            p, layer.saved, wfull, layer.topk_w, inp["dy"], g.dx, g.dw_gate, g.dw_up, g.dw_down,
            g.d_topk_w, wsb),
    }

    def step(events=None):
        for i, ph in enumerate(phases):
            if events is not None:
                events[i].record(stream)
            calls[ph]()
        if events is not None:
            events[len(phases)].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert layer.device_error() == 0, "device error during warm-up"

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)] for _ in range(K)]
    n0 = _lib.moe_launch_count()
    clk = ClockSampler(local)
    clk.start()
    if ws_ > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(K):
        step(ev[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    if ws_ > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    launches = _lib.moe_launch_count() - n0
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), ws_, dev)
    ph_ms = {ph: statistics.mean(ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(K))
             for i, ph in enumerate(phases)}
    assert layer.device_error() == 0, "device error in the timed region"

    graph = graph_timing(step, args.warmup, K, ws_, shape.N, dev) if args.graph else None

    # ---- end to end through the public API with host buffers ----
    # Every step copies its inputs (x, logits, dy) from pinned host memory and
    # reads its outputs (y, dx) back. Two buffer sets (two MoELayer objects)
    # let the copies of neighbouring steps run on a copy stream while a step
    # computes; the timed region spans the first upload to the last download.
    pin = {k: inp[k].cpu().pin_memory() for k in ("x", "logits", "dy") if inp.get(k) is not None}
    if router:
        pin.pop("logits")
    if inference or not backward:
        pin.pop("dy", None)
    layers = [layer, MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev,
                              allocate_grads=backward, minibatch_rows=shape.minibatch_rows,
                              dtype=shape.dtype, pipeline_stages=stages, tile_n=tile_n)]
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in pin.items()} for _ in range(2)]
    outs = [{"y": torch.empty((shape.N, shape.H), dtype=torch.bfloat16).pin_memory(),
             "dx": torch.empty((shape.N, shape.H), dtype=torch.bfloat16).pin_memory()}
            for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = shape.N * shape.H * 2 * (2 if backward else 1)
    # uploads and read-backs on streams of their own: the two directions overlap
    copy_s = torch.cuda.Stream(device=dev)
    read_s = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run_one(lay, din):
        if router:
            lay.route_from_x(din["x"], inp["w_router"], inp["bias"])
            lay.build_schedule()
            if inference:
                lay.forward_inference(din["x"], inp["wg"], inp["wu"], inp["wd"], mx=mxw)
                return
            lay.forward(din["x"], inp["wg"], inp["wu"], inp["wd"], mx=mxw)
            if backward:
                lay.backward(din["dy"], inp["wg"], inp["wu"], inp["wd"], bwd=wbwd, mx=mxw,
                             overlap=args.overlap)
                lay.router_backward(inp["w_router"], dwr)
        elif inference:
            lay.route(din["logits"], inp["bias"])
            lay.build_schedule()
            lay.forward_inference(din["x"], inp["wg"], inp["wu"], inp["wd"], mx=mxw)
        else:
            lay.step(din["x"], din["logits"], inp["bias"], inp["wg"], inp["wu"], inp["wd"],
                     din.get("dy"), backward=backward, bwd=wbwd, mx=mxw, overlap=args.overlap)

    def upload(b):
        with torch.cuda.stream(copy_s):
            for k, v in pin.items():
                dev_in[b][k].copy_(v, non_blocking=True)
            ev_in[b].record(copy_s)

    run_one(layers[1], {k: inp[k] for k in pin})  # warm the second buffer set
    torch.cuda.synchronize()
    n_e2e = max(args.e2e_steps, 2)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_s.wait_event(e0)
    upload(0)
    for i in range(n_e2e):
        b = i % 2
        if i + 1 < n_e2e:
            if i >= 1:
                copy_s.wait_event(ev_comp[1 - b])  # step i-1 is done with buffer set 1-b
            upload(1 - b)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # step i-2's outputs have been read back
        run_one(layers[b], dev_in[b])
        ev_comp[b].record(stream)
        with torch.cuda.stream(read_s):
            read_s.wait_event(ev_comp[b])
            outs[b]["y"].copy_(layers[b].y, non_blocking=True)
            if backward:
                outs[b]["dx"].copy_(layers[b].grads.dx, non_blocking=True)
            ev_out[b].record(read_s)
    stream.wait_stream(copy_s)
    stream.wait_stream(read_s)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, ws_, dev)
    del layers[1]
    # the last e2e steps ran from uploaded copies of the same inputs: one
    # more step on the resident ones must reproduce their outputs exactly
    determinism = rerun_check(step, output_tensors(layer, backward, dwr))
    loads = expert_loads(layer.schedule_tensors()["counts"].cpu(), shape.minibatch_rows)

    # ---- roofline of the dominant kernel ----
    peaks = load_peaks()
    fl = phase_flops(shape)
    by = phase_bytes(shape, layer.R, router)
    dominant = max((ph for ph in ph_ms if ph in fl or ph in by), key=ph_ms.get)
    # MXFP8 runs its GEMMs on the FP8 tensor cores, bf16 on the bf16 ones
    if mx:
        t_peak, t_kind = peaks["fp8_tflops_sustained"], peaks["fp8_source"] + " sustained"
    else:
        t_peak, t_kind = peaks["bf16_tflops_sustained"], f"{peaks['source']} bf16 sustained"
    if dominant in fl:
        achieved = fl[dominant] / (ph_ms[dominant] * 1e-3) / 1e12
        roof = {"kernel": dominant, "bound": "tensor", "achieved": round(achieved, 1),
                "peak": round(t_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / t_peak, 4),
                "peak_kind": t_kind, "traffic": measured_traffic(shape.name, dominant)}
    else:
        achieved = by[dominant] / (ph_ms[dominant] * 1e-3) / 1e9
        roof = {"kernel": dominant, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_kind": peaks["source"],
                "traffic": None}
    gemm_ms = sum(ph_ms[k] for k in fl if k in ph_ms)
    gemm_flops = sum(fl[k] for k in fl if k in ph_ms)
    gb_min = gemm_bytes(shape)
    phase_report = {}
    for ph in phases:
        d = {"ms": round(ph_ms[ph], 4)}
        if ph in fl:
            tf = fl[ph] / (ph_ms[ph] * 1e-3) / 1e12
            d.update(tflops=round(tf, 1), frac=round(tf / t_peak, 3))
            if ph in gb_min and not mx:  # the same phase on the bandwidth roofline
                gb = gb_min[ph] / (ph_ms[ph] * 1e-3) / 1e9
                d.update(min_gbs=round(gb, 1), hbm_frac=round(gb / peaks["hbm_gbs"], 3))
        elif ph in by:
            gb = by[ph] / (ph_ms[ph] * 1e-3) / 1e9
            d.update(gbs=round(gb, 1), frac=round(gb / peaks["hbm_gbs"], 3))
        phase_report[ph] = d

    step_ms = elapsed_ms / K
    value = replica_throughput(shape.N, K, ws_, elapsed_ms)
    rec = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws_, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp8 (E4M3 x E8M0 block-scaled MMAs, fp32 accumulation)" if mx else "bf16",
        "data": "synthetic (seeded Gaussian inputs and random-init expert weights)",
        "config": {"workload": shape.name, "N": shape.N, "H": shape.H, "I": shape.I,
                   "E": shape.E, "k": shape.k, "zipf_bias": shape.zipf_s,
                   "minibatch_rows": shape.minibatch_rows,
                   "pipeline_stages": stages or "library choice",
                   "tile_n": tile_n or "library choice",
                   "passes": "fwd+bwd" if backward else ("fwd (inference)" if inference
                                                           else "fwd"),
                   "l2": "inputs larger than L2 (expert weights alone "
                         f"{3 * shape.E * shape.H * shape.I * 2 / 1e9:.2f} GB)",
                   "parallelism": f"replicas x{ws_}",
                   "router": ("GPU router GEMM x.Wr^T and its backward inside the step" if router
                              else "router logits are an input (x.Wr^T formed on the host)")},
        "gemm_tflops": round(gemm_flops / (gemm_ms * 1e-3) / 1e12, 1),
        "gemm_frac_of_peak": round(gemm_flops / (gemm_ms * 1e-3) / 1e12 / t_peak, 4),
        "roofline": roof,
        "e2e": {"value": round(replica_throughput(shape.N, 1, ws_, e2e_ms), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clocks,
        "phases": phase_report,
        "determinism": determinism,
        "expert_loads": loads,
    }
    if graph is not None:
        rec["graph"] = graph
    if args.overlap and backward and not mx:
        rec["config"]["backward"] = ("moe_backward_overlap: reverse-combine run by side warps of "
                                     "the down data-gradient GEMM")
    return rec, shape, inp


MX_NOTE = "; MXFP8 weight copies quantised once before the sample, as on the GPU"
ROUTER_NOTE = "; router GEMM and router backward included"


# fp64 weight gradients above this many bytes do not fit the oracle's host run
# beside everything else; such shapes are timed per token and extrapolated.
ORACLE_DW_BYTES_MAX = 16 << 30


def oracle_extrapolates(shape):
    return shape.backward and 3 * 8 * shape.E * shape.H * shape.I > ORACLE_DW_BYTES_MAX


def cpu_sample(shape, inp, n_tok, threads, router=False):
    """Run the oracle on the first n_tok tokens of the workload (fwd+bwd with
    weight gradients; with router, the router GEMM and its backward too).
    Returns (seconds, tokens). Where the fp64 weight gradients would not fit
    (oracle_extrapolates), the oracle runs the tokens' forward and data
    gradients (tokens_bf16: 12 of the 18 H*I multiply-adds per assignment) and
    the returned time is scaled by 18/12 for the weight gradients' share."""
    import numpy as np

    import oracle
    if oracle_extrapolates(shape) and not router:
        ids, w = oracle.route_topk(inp["logits"][:n_tok].cpu().numpy(),
                                   None if inp["bias"] is None else inp["bias"].cpu().numpy(),
                                   shape.k)
        x = oracle.as_bf16_bits(inp["x"][:n_tok])
        dy = oracle.as_bf16_bits(inp["dy"][:n_tok])
        wg, wu, wd = (oracle.as_bf16_bits(t) for t in (inp["wg"], inp["wu"], inp["wd"]))
        t0 = time.perf_counter()
        oracle.tokens_bf16(x, wg, wu, wd, ids, w, dy, np.arange(n_tok), threads=threads)
        return (time.perf_counter() - t0) * 18.0 / 12.0, n_tok
    logits = inp["logits"][:n_tok].cpu().numpy()
    if router:
        t0 = time.perf_counter()
        logits = oracle.router_logits(inp["x"][:n_tok], inp["w_router"], threads).astype(np.float32)
        t_router = time.perf_counter() - t0
    bias = None if inp["bias"] is None else inp["bias"].cpu().numpy()
    x = oracle.as_bf16_bits(inp["x"][:n_tok])
    dy = oracle.as_bf16_bits(inp["dy"][:n_tok]) if inp.get("dy") is not None else None
    wg, wu, wd = (oracle.as_bf16_bits(t) for t in inp.get("w_src", (inp["wg"], inp["wu"], inp["wd"])))
    if shape.dtype == "mxfp8":
        if "oracle_w" not in inp:
            inp["oracle_w"] = oracle.mxfp8_weights(wg, wu, wd, threads=threads)
        prepared = inp["oracle_w"]
    t0 = time.perf_counter()
    ids, w = oracle.route_topk(logits, bias, shape.k)
    oracle.build_schedule(ids, shape.E)
    if shape.dtype == "mxfp8":
        # the weights' quantisation is not part of a step (the GPU run also
        # prepares them once, before its timed steps)
        r = oracle.layer_mxfp8_prepared(x, prepared, ids, w, dy, threads=threads)
    elif shape.backward:
        oracle.forward_bf16(x, wg, wu, wd, ids, w, threads=threads)
        r = oracle.backward_bf16(x, wg, wu, wd, ids, w, dy, threads=threads)
    else:
        oracle.forward_bf16(x, wg, wu, wd, ids, w, threads=threads)
    if router and shape.backward:
        oracle.router_backward(x, inp["w_router"], ids, w, r["dw"], threads)
    return time.perf_counter() - t0 + (t_router if router else 0.0), n_tok


def one_core(shape, inp, router=False, n_tok=8):
    """The oracle on one host thread, on the first n_tok tokens: the baseline's
    single-core rate beside its all-cores one."""
    secs, n = cpu_sample(shape, inp, n_tok, 1, router)
    return {"value": round(n / secs, 3), "unit": UNIT, "cores": 1,
            "sample": f"first {n} tokens, {secs:.1f} s"}


def run_reference(args, ws_, rank):
    """The oracle, timed on the host cores, on bounded samples of the workload."""
    if rank != 0:
        return None
    import torch

    from mixture_experts_layer_schedule_gb300 import inputs
    shape = workload(args.config)
    threads = os.cpu_count() or 1
    n_tok = args.cpu_tokens or 16
    inp = inputs.make_inputs(shape.with_(N=n_tok), seed=0, device="cpu")
    for _ in range(args.warmup):
        cpu_sample(shape, inp, n_tok, threads, args.router)
    times = [cpu_sample(shape, inp, n_tok, threads, args.router)[0] for _ in range(args.steps)]
    tot = sum(times)
    value = n_tok * args.steps / tot
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Gaussian inputs and random-init expert weights)",
        "config": {"workload": shape.name, "N": shape.N, "H": shape.H, "I": shape.I,
                   "E": shape.E, "k": shape.k, "zipf_bias": shape.zipf_s,
                   "passes": "fwd+bwd" if shape.backward else "fwd"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads,
                         "kind": "oracle",
                         "sample": f"first {n_tok} tokens of the workload per step "
                                   f"(full expert weights, fwd+bwd with weight gradients"
                                   f"{MX_NOTE if shape.dtype == 'mxfp8' else ''}"
                                   f"{ROUTER_NOTE if args.router else ''})",
                         "one_core": one_core(shape, inp, args.router)},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    ws_, rank, local = dist_env()
    if ws_ > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
    if args.tensor_peaks:
        import torch
        torch.cuda.set_device(local)
        print(json.dumps(tensor_peaks()), flush=True)
        return
    if args.impl == "reference":
        rec = run_reference(args, ws_, rank)
        if rec is not None:
            print(json.dumps(rec), flush=True)
        return
    if args.sweep_stages:
        import torch
        base = workload(args.config)
        res = {}
        for S in (4, 5, 6, "wide"):
            args.phase_report = True
            r, _, _ = run_ours(args, ws_, rank, local, base, stages=0 if S == "wide" else S,
                               tile_n=512 if S == "wide" else 256)
            res[S] = {"value": r["value"], "ms_per_step": r["ms_per_step"],
                      "phases": {k: v["ms"] for k, v in r["phases"].items()},
                      "clocks": r["clocks"]}
            del r
            torch.cuda.empty_cache()
        gemm = [k for k in res[6]["phases"] if k in phase_flops(base)]
        best = {k: min(res, key=lambda S: res[S]["phases"][k]) for k in gemm}
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, "sweep": "pipeline_stages",
                              "workload": base.name, "steps": args.steps, "warmup": args.warmup,
                              "results": res, "best_stages_per_phase": best,
                              "best_stages_step": max(res, key=lambda S: res[S]["value"])}),
                  flush=True)
        return
    if args.sweep_T:
        import torch
        base = workload(args.config)
        res = {}
        for T in (128, 256, 512, 1024):
            r, _, _ = run_ours(args, ws_, rank, local,
                               base.with_(name=f"{base.name}_T{T}", minibatch_rows=T))
            res[T] = {"value": r["value"], "ms_per_step": r["ms_per_step"],
                      "gemm_tflops": r["gemm_tflops"], "clocks": r["clocks"]}
            del r
            torch.cuda.empty_cache()
        best = max(res, key=lambda t: res[t]["value"])
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, "higher_is_better": True,
                              "sweep": "minibatch_rows", "workload": base.name, "n_gpus": ws_,
                              "steps": args.steps, "warmup": args.warmup, "results": res,
                              "best_minibatch_rows": best, "value": res[best]["value"]}),
                  flush=True)
        return
    rec, shape, inp = run_ours(args, ws_, rank, local)
    if rank == 0 and ws_ == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        n_tok = args.cpu_tokens or 256
        ext = oracle_extrapolates(shape) and not args.router
        if ext:
            n_tok = min(n_tok, 16)
        secs, n = cpu_sample(shape, inp, n_tok, threads, args.router)
        rec["cpu_baseline"] = {"value": round(n / secs, 3), "unit": UNIT, "cores": threads,
                               "kind": "oracle",
                               "sample": (f"first {n} tokens of the workload: forward and data "
                                          f"gradients timed, x 18/12 for the weight gradients "
                                          f"(extrapolated: fp64 weight gradients of this shape "
                                          f"exceed host memory), {secs:.1f} s" if ext else
                                          f"first {n} tokens of the workload (full expert "
                                          f"weights, fwd+bwd with weight gradients"
                                          f"{MX_NOTE if shape.dtype == 'mxfp8' else ''}"
                                          f"{ROUTER_NOTE if args.router else ''}), "
                                          f"{secs:.1f} s"),
                               "full_layer_seconds": round(shape.N * secs / n, 1)}
        if not ext:
            rec["cpu_baseline"]["one_core"] = one_core(shape, inp, args.router)
    if rank == 0:
        if not args.phase_report:
            rec.pop("phases", None)
        print(json.dumps(rec), flush=True)
    if ws_ > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
