"""GPU MXFP8 quantiser vs the oracle, bit-exact codes and scales.

The quantise op of the project summary "Mixture-of-Kittens (MoK)" (core
concepts, MXFP8 row), with the OCP MX v1.0 scale rule and E4M3 elements."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import _lib

from gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _run(src_bf16: torch.Tensor):
    rows, cols = src_bf16.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device=dev())
    s = torch.empty((rows, cols // 32), dtype=torch.uint8, device=dev())
    _lib.mxfp8_quantize(src_bf16.to(dev()).contiguous(), rows, cols, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def test_random_magnitudes_bit_exact():
    g = torch.Generator().manual_seed(0)
    rows, cols = 1024, 2048
    x = torch.randn((rows, cols), generator=g) * torch.exp(
        torch.empty((rows, 1)).uniform_(-40, 40, generator=g))
    src = x.bfloat16()
    q, s = _run(src)
    qr, sr = oracle.mxfp8_quantize(src)
    np.testing.assert_array_equal(s, sr)
    np.testing.assert_array_equal(q, qr)


def test_every_bf16_pattern_and_special_blocks():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    src = bits.view(torch.bfloat16).reshape(-1, 256).clone()
    finite = torch.isfinite(src.float())
    src[~finite] = 0  # the quantiser is specified for finite inputs
    extra = torch.zeros((8, 256), dtype=torch.float32)
    extra[1] = 448.0
    extra[2, :32] = torch.tensor([2.0 ** i for i in range(-10, 22)])
    extra[3] = 1.9375 * 2.0 ** 10  # scaled into (448, 512): saturates
    extra[4] = -(2.0 ** -130)       # bf16 subnormals: scale code clamps to 0
    extra[5, ::2] = 1e-30
    extra[6] = torch.linspace(-500, 500, 256)
    src = torch.cat([src, extra.bfloat16()])
    q, s = _run(src)
    qr, sr = oracle.mxfp8_quantize(src)
    np.testing.assert_array_equal(s, sr)
    np.testing.assert_array_equal(q, qr)


def test_expert_weight_shapes():
    E, I, H = 8, 512, 256
    w = (torch.randn((E * I, H), generator=torch.Generator().manual_seed(3)) / 16).bfloat16()
    q, s = _run(w)
    qr, sr = oracle.mxfp8_quantize(w)
    np.testing.assert_array_equal(q, qr)
    np.testing.assert_array_equal(s, sr)
