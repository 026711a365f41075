"""Gate/up with the dispatch fused into its producer (TMA gather of token rows)
and the context-free forward built on it.

The fused path must reproduce, on every real row, the G/U/Act of the unfused
dispatch + gate/up (same tensor-core products in the same order, so
bit-exact), and moe_forward_inference must reproduce moe_forward's y; both are
also checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, _lib, inputs

from gpu_helpers import assert_close, custom_shape, dev, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [inputs.TINY, custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_skewed"),
          custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_skewed_T256", T=256),
          custom_shape(1000, 1024, 512, 32, 8, name="wider")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_gathered_gate_up_matches_dispatch_then_gate_up(shape):
    inp_cpu = inputs.make_inputs(shape, seed=5, device="cpu")
    inp = to_dev(inp_cpu)
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows)
    layer.route(inp["logits"], inp["bias"])
    layer.build_schedule()
    p, ws = layer.p, layer.ws
    w = _lib.weights(inp["wg"], inp["wu"], inp["wd"])
    sv = layer.saved_tensors()
    _lib.moe_dispatch(p, ws, inp["x"], sv["xe"])
    _lib.moe_expert_gate_up(p, ws, sv["xe"], w, sv["g"], sv["u"], sv["act"])
    g2, u2, a2 = (torch.full_like(sv["g"], 9.0) for _ in range(3))
    _lib.moe_expert_gate_up_gather(p, ws, inp["x"], w, g2, u2, a2)
    a3 = torch.full_like(sv["act"], 9.0)
    _lib.moe_expert_gate_up_gather(p, ws, inp["x"], w, None, None, a3)
    torch.cuda.synchronize()
    src = layer.schedule_tensors()["src_of_row"]
    rows = int(layer.schedule_tensors()["pad_offsets"][shape.E])
    real = torch.nonzero(src[:rows] >= 0).squeeze(1)
    for name, ref, got in (("G", sv["g"], g2), ("U", sv["u"], u2), ("Act", sv["act"], a2),
                           ("Act only", sv["act"], a3)):
        assert torch.equal(got[real], ref[real]), name
    assert torch.all(torch.isfinite(a2[:rows].float()))
    assert torch.all(g2[rows:] == 9.0)  # rows past the used segments untouched
    assert layer.device_error() == 0


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_forward_inference_matches_forward_and_oracle(shape):
    inp_cpu = inputs.make_inputs(shape, seed=6, device="cpu")
    inp = to_dev(inp_cpu)
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows)
    layer.route(inp["logits"], inp["bias"])
    layer.build_schedule()
    y1 = layer.forward(inp["x"], inp["wg"], inp["wu"], inp["wd"]).clone()
    y2 = layer.forward_inference(inp["x"], inp["wg"], inp["wu"], inp["wd"]).clone()
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    logits = inp_cpu["logits"].numpy()
    bias = None if inp_cpu["bias"] is None else inp_cpu["bias"].numpy()
    ids, wts = oracle.route_topk(logits, bias, shape.k)
    yref = oracle.forward_bf16(inp_cpu["x"], inp_cpu["wg"], inp_cpu["wu"], inp_cpu["wd"], ids, wts)
    assert_close("y", y2, yref)
    assert layer.device_error() == 0
