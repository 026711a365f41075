"""A whole layer pass captured in a CUDA graph and replayed.

The library allocates nothing, never synchronises and enqueues every step on
the caller's stream, so a route -> schedule -> forward -> backward pass can be
captured once and replayed: the graph must give the eager results bit for
bit, and, with new values written into the same input buffers, the results of
an eager pass on those values (the graph reads its buffers at replay time;
the schedule is rebuilt on the device inside the graph, so new routing is
handled too)."""
import pytest
import torch

from mixture_experts_layer_schedule_gb300 import MoELayer, inputs

from gpu_helpers import custom_shape, dev, to_dev

pytestmark = pytest.mark.gpu

CASES = [("bf16", False), ("bf16", True), ("mxfp8", False)]


def _outputs(layer):
    g = layer.grads
    return {"y": layer.y, "dx": g.dx, "dw_gate": g.dw_gate, "dw_up": g.dw_up,
            "dw_down": g.dw_down, "d_topk_w": g.d_topk_w, "topk_ids": layer.topk_ids}


def _bytes(t):
    return t.reshape(-1).view(torch.uint8)


@pytest.mark.parametrize("dtype,overlap", CASES, ids=lambda v: str(v))
def test_graph_replay_matches_eager(dtype, overlap):
    shape = custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="graph")
    d = dev()
    inp = to_dev(inputs.make_inputs(shape, seed=21, device="cpu"))
    new = to_dev(inputs.make_inputs(shape, seed=22, device="cpu"))
    fwd = (inp["wg"], inp["wu"], inp["wd"])
    bwd = mx = None
    if dtype == "mxfp8":
        fwd, bwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
        mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=d, dtype=dtype)
    x, logits, dy = inp["x"].clone(), inp["logits"].clone(), inp["dy"].clone()

    def step():
        layer.step(x, logits, inp["bias"], *fwd, dy, bwd=bwd, mx=mx, overlap=overlap)

    side = torch.cuda.Stream(device=d)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # eager pass: one-time setup happens here
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    eager = {k: v.clone() for k, v in _outputs(layer).items()}

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in _outputs(layer).values():  # stale values must not survive a replay
        _bytes(t).fill_(0xA5)
    graph.replay()
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    for k, t in _outputs(layer).items():
        assert torch.equal(_bytes(t), _bytes(eager[k])), k

    # new token values in the same buffers: replay against a fresh eager pass
    x.copy_(new["x"])
    logits.copy_(new["logits"])
    dy.copy_(new["dy"])
    graph.replay()
    torch.cuda.synchronize()
    replayed = {k: v.clone() for k, v in _outputs(layer).items()}
    assert not torch.equal(replayed["y"], eager["y"])
    step()
    torch.cuda.synchronize()
    for k, t in _outputs(layer).items():
        assert torch.equal(_bytes(t), _bytes(replayed[k])), k
