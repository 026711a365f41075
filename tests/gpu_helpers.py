"""Shared helpers for the GPU parity tests (CUDA path vs the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, inputs

BF16_TOL = 2e-2      # max|err| <= 2e-2 * max|ref| per tensor (bf16 path)
W_RTOL = 2e-6        # routing weights: fp32 expf + k-term sum + divide vs fp64


def dev():
    return torch.device("cuda:0")


def max_rel(got, ref) -> float:
    g = got.float().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    ref = np.asarray(ref, dtype=np.float64)
    denom = max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(g.astype(np.float64) - ref)) / denom)


def assert_close(name, got, ref, tol=BF16_TOL):
    e = max_rel(got, ref)
    assert e <= tol, f"{name}: max|err|/max|ref| = {e:.3e} > {tol}"
    return e


def to_dev(d):
    return {k: (v.to(dev()) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def custom_shape(N, H, I, E, k, zipf_s=None, name="custom", T=128):
    return inputs.LayerShape(name, N, H, I, E, k, zipf_s=zipf_s, minibatch_rows=T)


def run_layer(shape, inp_dev, backward=True):
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows)
    layer.step(inp_dev["x"], inp_dev["logits"], inp_dev["bias"], inp_dev["wg"], inp_dev["wu"],
               inp_dev["wd"], inp_dev.get("dy"), backward=backward)
    torch.cuda.synchronize()
    return layer
