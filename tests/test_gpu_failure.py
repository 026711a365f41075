"""Failure detection on the GPU without a fault: a barrier wait that can never
complete runs out of time (about a second), records MOE_DEVERR_TIMEOUT in the
workspace error word and returns; the host reads the code, clears it, and the
same context then runs the layer correctly."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, _lib, inputs

from gpu_helpers import assert_close, dev, to_dev

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_stays_usable():
    shape = inputs.TINY
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev())
    assert layer.device_error() == 0
    _lib.moe_test_wait_timeout(layer.p, layer.ws)
    torch.cuda.synchronize()
    assert layer.device_error() == _lib.MOE_DEVERR_TIMEOUT
    layer.clear_device_error()
    assert layer.device_error() == 0
    inp_cpu = inputs.make_inputs(shape, seed=0, device="cpu")
    inp = to_dev(inp_cpu)
    layer.step(inp["x"], inp["logits"], inp["bias"], inp["wg"], inp["wu"], inp["wd"], inp["dy"])
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ids, w = oracle.route_topk(inp_cpu["logits"].numpy(), None, shape.k)
    y = oracle.forward_bf16(inp_cpu["x"], inp_cpu["wg"], inp_cpu["wu"], inp_cpu["wd"], ids, w)
    assert_close("y", layer.y, y)
