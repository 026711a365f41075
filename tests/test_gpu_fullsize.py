"""Full-size parity on the workloads the layer is measured on, in the launch
configuration bench.py times (same kernels, same grids, inputs drawn on the
device by the shared generator).

At these sizes the oracle cannot run the whole layer, so:
  * routing ids and every schedule table are compared bit-exactly over the
    whole batch (the oracle's routing and schedule are cheap);
  * y, dx and d(routing weights) are compared on a seeded sample of tokens,
    each computed by the oracle from that token's own assignments;
  * weight-gradient rows are compared for sampled experts (the smallest
    non-empty one, the median one and the largest one, whose long token
    panels run the chunked weight-gradient plan on the skewed workload) and
    sampled rows, each computed by the oracle over every token routed to that
    expert;
  * the tolerance is the bf16 bound, max|err| <= 2e-2 * max|ref| over the
    sampled elements of each tensor; ids and tables are exact;
  * the fused dispatch + expert FFN launch (moe_forward_inference) reproduces
    the checked y bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, inputs

from gpu_helpers import BF16_TOL, W_RTOL, assert_close, dev

pytestmark = pytest.mark.gpu

FULL = [inputs.FINE_GRAINED_FWD, inputs.SKEWED, inputs.SKEWED.with_(name=inputs.SKEWED.name + "_T256", minibatch_rows=256),
        inputs.large_batch(8192, 256), inputs.large_batch(65536, 1024)]


def _host(t):
    return None if t is None else t.cpu()


@pytest.mark.parametrize("shape", FULL, ids=lambda s: s.name)
def test_full_size_sampled_parity(shape):
    torch.cuda.empty_cache()
    d = dev()
    inp = inputs.make_inputs(shape, seed=0, device=d)
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=d,
                     allocate_grads=shape.backward, minibatch_rows=shape.minibatch_rows)
    layer.step(inp["x"], inp["logits"], inp["bias"], inp["wg"], inp["wu"], inp["wd"],
               inp.get("dy"), backward=shape.backward)
    torch.cuda.synchronize()
    assert layer.device_error() == 0

    # routing and schedule: exact over the whole batch
    logits = inp["logits"].cpu().numpy()
    bias = None if inp["bias"] is None else inp["bias"].cpu().numpy()
    ids, w = oracle.route_topk(logits, bias, shape.k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids)
    wg_gpu = layer.topk_w.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(wg_gpu - w) / w) <= W_RTOL
    ref = oracle.build_schedule(ids, shape.E, 128, shape.minibatch_rows)
    got = {k: v.cpu().numpy() for k, v in layer.schedule_tensors().items()}
    for key in ("counts", "offsets", "pad_offsets"):
        np.testing.assert_array_equal(got[key], ref[key])
    np.testing.assert_array_equal(got["slot_of"], ref["slot_of"].ravel())
    rows = int(ref["pad_offsets"][shape.E])
    np.testing.assert_array_equal(got["src_of_row"][:rows], ref["src_of_row"])
    np.testing.assert_array_equal(got["tiles"].reshape(-1, 3)[:ref["n_tiles"]], ref["tiles"])

    # the fused dispatch + expert FFN launch (the context-free forward's path)
    # gives the training forward's y bit for bit at this size as well
    y_train = layer.y.clone()
    layer.forward_inference(inp["x"], inp["wg"], inp["wu"], inp["wd"])
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(layer.y.view(torch.int16), y_train.view(torch.int16))

    # sampled tokens: y (and dx, d routing weights when the pass has a backward)
    x, wgt, wut, wdt = (_host(inp[k]) for k in ("x", "wg", "wu", "wd"))
    dy = _host(inp["dy"]) if shape.backward else torch.zeros_like(x)
    rng = np.random.default_rng(shape.N)
    tok = np.sort(rng.choice(shape.N, 16, replace=False))
    s = oracle.tokens_bf16(x, wgt, wut, wdt, ids, w, dy, tok)
    assert_close("y", layer.y[torch.as_tensor(tok)], s["y"])
    if not shape.backward:
        return
    g = layer.grads
    assert_close("dx", g.dx[torch.as_tensor(tok)], s["dx"])
    assert_close("d_topk_w", g.d_topk_w[torch.as_tensor(tok)], s["dw"])

    # sampled weight-gradient rows of three experts: smallest, median, largest
    counts = ref["counts"]
    nonzero = np.flatnonzero(counts)
    by_size = nonzero[np.argsort(counts[nonzero], kind="stable")]
    experts = sorted({int(by_size[0]), int(by_size[len(by_size) // 2]), int(by_size[-1])})
    il = np.sort(rng.choice(shape.I, 4, replace=False)).astype(np.int32)
    hl = np.sort(rng.choice(shape.H, 4, replace=False)).astype(np.int32)
    for e in experts:
        r = oracle.expert_wgrad_bf16(x, wgt, wut, wdt, ids, w, dy, e, il, hl)
        assert_close(f"dw_gate[{e}]", g.dw_gate[e][torch.as_tensor(il).long()], r["dwg"])
        assert_close(f"dw_up[{e}]", g.dw_up[e][torch.as_tensor(il).long()], r["dwu"])
        assert_close(f"dw_down[{e}]", g.dw_down[e][torch.as_tensor(hl).long()], r["dwd"])
    # an expert without tokens (if any) has an all-zero gradient
    empty = np.flatnonzero(counts == 0)
    if len(empty):
        e = int(empty[0])
        assert torch.all(g.dw_gate[e] == 0) and torch.all(g.dw_down[e] == 0)
    del layer, inp
    torch.cuda.empty_cache()
