"""Router on the GPU (the GEMM in front of the routing, and its backward).

* logits = x . Wr^T on the tensor cores against the oracle's fp64 logits:
  max|err| <= 1e-4 * max|ref| (fp32 accumulation of exact bf16 products over H);
* top-k ids bit-exact and weights within 2e-6 relative against the oracle's
  routing fed the GPU's logits (top-k is only comparable on identical
  logits); against the oracle's own fp64 logits every differing token must be
  a near tie (the k-th and (k+1)-th logits within twice the logit tolerance);
* router backward against the oracle fed the GPU's ids, weights and
  d(routing weights): dWr within 1e-4 * max|ref|, dx (expert part + router
  part) within the bf16 bound 2e-2 * max|ref| of the whole-layer oracle;
* bitwise reruns.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, inputs

from gpu_helpers import BF16_TOL, W_RTOL, assert_close, custom_shape, dev, max_rel, to_dev

pytestmark = pytest.mark.gpu

LOGIT_TOL = 1e-4
SHAPES = [inputs.TINY, custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_skewed"),
          custom_shape(1000, 1024, 512, 64, 8, name="e64_k8"),
          custom_shape(513, 256, 256, 256, 8, name="e256")]


def _layer(shape):
    return MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                    minibatch_rows=shape.minibatch_rows)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_router_logits_and_routing(shape):
    inp_cpu = inputs.make_inputs(shape, seed=2, device="cpu")
    inp = to_dev(inp_cpu)
    layer = _layer(shape)
    logits = torch.empty((shape.N, shape.E), dtype=torch.float32, device=dev())
    layer.route_from_x(inp["x"], inp["w_router"], inp["bias"], logits)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ref = oracle.router_logits(inp_cpu["x"], inp_cpu["w_router"])
    assert max_rel(logits, ref) <= LOGIT_TOL
    bias = None if inp_cpu["bias"] is None else inp_cpu["bias"].numpy()
    got = logits.cpu().numpy()
    ids, w = oracle.route_topk(got, bias, shape.k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids)
    assert np.max(np.abs(layer.topk_w.cpu().numpy().astype(np.float64) - w) / w) <= W_RTOL
    # routing from the oracle's own logits differs only at near ties
    ids64, _ = oracle.route_topk(ref.astype(np.float32), bias, shape.k)
    tol = 2 * LOGIT_TOL * np.max(np.abs(ref))
    z = ref + (0.0 if bias is None else bias.astype(np.float64))
    for t in np.flatnonzero(np.any(np.sort(ids64, 1) != np.sort(ids, 1), axis=1)):
        srt = np.sort(z[t])[::-1]
        assert srt[shape.k - 1] - srt[shape.k] <= tol, (t, srt[shape.k - 1] - srt[shape.k])


@pytest.mark.parametrize("shape", SHAPES[:3], ids=lambda s: s.name)
def test_router_backward(shape):
    inp_cpu = inputs.make_inputs(shape, seed=4, device="cpu")
    inp = to_dev(inp_cpu)
    layer = _layer(shape)
    layer.route_from_x(inp["x"], inp["w_router"], inp["bias"])
    layer.build_schedule()
    layer.forward(inp["x"], inp["wg"], inp["wu"], inp["wd"])
    layer.backward(inp["dy"], inp["wg"], inp["wu"], inp["wd"])
    dx_experts = layer.grads.dx.clone()
    dwr = torch.empty((shape.E, shape.H), dtype=torch.float32, device=dev())
    layer.router_backward(inp["w_router"], dwr)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ids = layer.topk_ids.cpu().numpy()
    w = layer.topk_w.cpu().numpy().astype(np.float64)
    dw = layer.grads.d_topk_w.cpu().numpy().astype(np.float64)
    r = oracle.router_backward(inp_cpu["x"], inp_cpu["w_router"], ids, w, dw)
    assert_close("dw_router", dwr, r["dwr"], 1e-4)
    # the whole dx: experts (oracle layer backward on the GPU's routing) + router
    rb = oracle.backward_bf16(inp_cpu["x"], inp_cpu["wg"], inp_cpu["wu"], inp_cpu["wd"], ids, w,
                              inp_cpu["dy"])
    assert_close("dx", layer.grads.dx, rb["dx"] + r["dx"], BF16_TOL)
    # bitwise rerun from the same expert part
    dx1, dwr1 = layer.grads.dx.clone(), dwr.clone()
    layer.grads.dx.copy_(dx_experts)
    layer.router_backward(inp["w_router"], dwr)
    torch.cuda.synchronize()
    assert torch.equal(layer.grads.dx, dx1) and torch.equal(dwr, dwr1)


def test_router_empty_batch_and_unsupported_sizes():
    shape = custom_shape(16, 256, 256, 8, 2, name="small")
    inp = to_dev(inputs.make_inputs(shape, seed=1, device="cpu"))
    empty = custom_shape(0, 256, 256, 8, 2, name="empty")
    layer = _layer(empty)
    layer.route_from_x(inp["x"][:0], inp["w_router"], None)
    layer.build_schedule()
    layer.forward(inp["x"][:0], inp["wg"], inp["wu"], inp["wd"])
    layer.backward(inp["dy"][:0], inp["wg"], inp["wu"], inp["wd"])
    dwr = torch.full((8, 256), 1.0, dtype=torch.float32, device=dev())
    layer.router_backward(inp["w_router"], dwr)
    torch.cuda.synchronize()
    assert layer.device_error() == 0 and torch.all(dwr == 0)
    # E = 6 (not a multiple of 4) and E > 256 are rejected before any launch
    from mixture_experts_layer_schedule_gb300 import _lib
    for E in (6, 512):
        bad = MoELayer(16, 256, 256, E, 2, device=dev())
        wr = torch.zeros((E, 256), dtype=torch.bfloat16, device=dev())
        with pytest.raises(_lib.MoEError):
            bad.route_from_x(inp["x"], wr, None)
