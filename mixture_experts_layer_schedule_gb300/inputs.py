"""Seeded synthetic inputs for the MoE layer (shared by tests and the bench).

This module holds none of the layer's arithmetic: it only draws the inputs.
The pages' workload (production training of a coding model) has no public
dataset, so seeded Gaussian tensors of the stated shapes stand in for it:

  x  ~ N(0, 1)          [N, H]      bf16 (round-to-nearest-even)
  Wr ~ N(0, 1/H)        [H, E]      fp32, only used to form the logits
  Wg, Wu ~ N(0, 1/H)    [E, I, H]   bf16
  Wd ~ N(0, 1/H)        [E, H, I]   bf16 (scale taken literally as 1/H)
  dY ~ N(0, 1)          [N, H]      bf16
  logits = fl32(x . Wr) evaluated in fp64 from the bf16 x values
  bias (skewed configs) = -s * ln(r_e), r a seeded permutation of 1..E, so the
       per-expert prior is proportional to rank^-s (Zipf, s = 1.2)

Each tensor has its own generator stream keyed by (seed, tensor id) in a
fixed id order (x=0, Wr=1, Wg=2, Wu=3, Wd=4, bias permutation=5, dY=6).
Large weight tensors are drawn one expert at a time from their stream, so
the host never holds an fp32 copy of a whole weight tensor.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

TENSOR_IDS = dict(x=0, wr=1, wg=2, wu=3, wd=4, bias=5, dy=6)


@dataclass(frozen=True)
class LayerShape:
    name: str
    N: int
    H: int
    I: int
    E: int
    k: int
    zipf_s: float | None = None      # per-expert Zipf bias exponent, None = uniform
    dtype: str = "bf16"              # "bf16" or "mxfp8" (expert weights)
    backward: bool = True
    minibatch_rows: int = 128        # T: rows per ring slot / tile height
    extra: dict = field(default_factory=dict)

    @property
    def A(self) -> int:
        return self.N * self.k

    def with_(self, **kw) -> "LayerShape":
        return replace(self, **kw)


# The workloads the pages' method is exercised on (sizes as stated for them).
TINY = LayerShape("tiny_N256_H256_I512_E8_k2", 256, 256, 512, 8, 2)
FINE_GRAINED_FWD = LayerShape("fine_grained_fwd_N4096_H2048_I1024_E64_k8", 4096, 2048, 1024, 64,
                              8, backward=False)
SKEWED = LayerShape("skewed_fwd_bwd_N16384_H4096_I1536_E128_k8_zipf1.2", 16384, 4096, 1536, 128,
                    8, zipf_s=1.2)
SKEWED_MXFP8 = SKEWED.with_(name="skewed_mxfp8_N16384_H4096_I1536_E128_k8_zipf1.2",
                            dtype="mxfp8")


def large_batch(N: int, T: int = 128) -> LayerShape:
    return LayerShape(f"large_batch_N{N}_H7168_I2048_E256_k8_T{T}", N, 7168, 2048, 256, 8,
                      minibatch_rows=T)


LARGE_BATCH_N = (8192, 32768, 65536)
LARGE_BATCH_T = (128, 256, 512, 1024)

ALL = {s.name: s for s in (TINY, FINE_GRAINED_FWD, SKEWED, SKEWED_MXFP8)}
for _n in LARGE_BATCH_N:
    for _t in LARGE_BATCH_T:
        ALL[large_batch(_n, _t).name] = large_batch(_n, _t)


def _gen(seed: int, tensor: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + TENSOR_IDS[tensor] * 7919 + 12345) & 0x7FFF_FFFF_FFFF)
    return g


def _normal(shape, std, gen, device, dtype=torch.bfloat16):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _expert_stack(E, rows, cols, std, gen, device):
    out = torch.empty((E, rows, cols), dtype=torch.bfloat16, device=device)
    for e in range(E):
        out[e] = _normal((rows, cols), std, gen, device)
    return out


def make_inputs(shape: LayerShape, seed: int = 0, device="cpu", with_dy: bool = True,
                weight_seed: int = None) -> dict:
    """Draw every input of one layer call. Returns torch tensors on `device`.
    weight_seed (default: seed) draws the parameters -- router and expert
    weights, expert bias -- so data-parallel replicas can share them while
    their tokens and upstream gradients (seed) differ."""
    N, H, I, E = shape.N, shape.H, shape.I, shape.E
    dev = torch.device(device)
    std = 1.0 / math.sqrt(H)
    pseed = seed if weight_seed is None else weight_seed
    x = _normal((N, H), 1.0, _gen(seed, "x", dev), dev)
    wr = _normal((H, E), std, _gen(pseed, "wr", dev), dev, dtype=torch.float32)
    wg = _expert_stack(E, I, H, std, _gen(pseed, "wg", dev), dev)
    wu = _expert_stack(E, I, H, std, _gen(pseed, "wu", dev), dev)
    wd = _expert_stack(E, H, I, std, _gen(pseed, "wd", dev), dev)
    logits = (x.double() @ wr.double()).float().contiguous()
    bias = None
    if shape.zipf_s is not None:
        g = _gen(pseed, "bias", torch.device("cpu"))
        r = torch.randperm(E, generator=g).double() + 1.0
        bias = (-shape.zipf_s * torch.log(r)).float().to(dev)
    # the same router weights as the device router GEMM reads them: bf16 [E, H]
    w_router = wr.t().contiguous().to(torch.bfloat16)
    out = dict(x=x, wg=wg, wu=wu, wd=wd, logits=logits, bias=bias, w_router=w_router)
    if with_dy:
        out["dy"] = _normal((N, H), 1.0, _gen(seed, "dy", dev), dev)
    return out
