"""MXFP8 layer on the GPU: quantise-dequantise kernels bit-exact against the
oracle quantiser, and the whole MXFP8 forward + backward against the oracle's
MXFP8 layer within max|err| <= 6e-2 * max|ref| per tensor (the MXFP8 bound of
the workload statement)."""
import math

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, _lib, inputs

from gpu_helpers import assert_close, custom_shape, dev, to_dev

pytestmark = pytest.mark.gpu

MX_TOL = 6e-2


def _oracle_qdq(bits2d, axis):
    a = bits2d if axis == 0 else np.ascontiguousarray(bits2d.T)
    q, s = oracle.mxfp8_quantize(a)
    dec = np.vectorize(oracle.e4m3_decode)(q) if q.size < 300000 else None
    if dec is None:
        table = np.array([oracle.e4m3_decode(c) for c in range(256)])
        dec = table[q]
    v = dec * np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
    return v if axis == 0 else v.T


@pytest.mark.parametrize("axis", [0, 1])
def test_qdq_matches_oracle_quantiser(axis):
    g = torch.Generator().manual_seed(axis)
    x = (torch.randn((256, 512), generator=g) * torch.exp(torch.empty((256, 1)).uniform_(-8, 8, generator=g))).bfloat16()
    out = torch.empty_like(x, device=dev())
    _lib.mxfp8_qdq(x.to(dev()), out, 256, 512, axis)
    torch.cuda.synchronize()
    ref = _oracle_qdq(oracle.as_bf16_bits(x), axis)
    np.testing.assert_array_equal(out.float().cpu().numpy().astype(np.float64), ref)


SHAPES = [inputs.TINY.with_(name="tiny_mxfp8", dtype="mxfp8"),
          custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_skewed_mxfp8").with_(dtype="mxfp8"),
          custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_T256_mxfp8", T=256).with_(dtype="mxfp8")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_mxfp8_layer_matches_oracle(shape):
    inp_cpu = inputs.make_inputs(shape, seed=3, device="cpu")
    inp = to_dev(inp_cpu)
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows, dtype="mxfp8")
    fwd, bwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    layer.step(inp["x"], inp["logits"], inp["bias"], *fwd, inp["dy"], bwd=bwd)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    logits = inp_cpu["logits"].numpy()
    bias = None if inp_cpu["bias"] is None else inp_cpu["bias"].numpy()
    ids, w = oracle.route_topk(logits, bias, shape.k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids)
    r = oracle.layer_mxfp8(inp_cpu["x"], inp_cpu["wg"], inp_cpu["wu"], inp_cpu["wd"], ids, w,
                           inp_cpu["dy"], quantize=True)
    g = layer.grads
    assert_close("y", layer.y, r["y"], MX_TOL)
    for name, got, key in (("dx", g.dx, "dx"), ("dw_gate", g.dw_gate, "dwg"),
                           ("dw_up", g.dw_up, "dwu"), ("dw_down", g.dw_down, "dwd"),
                           ("d_topk_w", g.d_topk_w, "dw")):
        assert_close(name, got, r[key], MX_TOL)
