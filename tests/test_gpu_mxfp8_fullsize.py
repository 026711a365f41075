"""Full-size MXFP8 parity against the oracle on the skewed MXFP8 workload
(N=16384, H=4096, I=1536, E=128, top-8, Zipf 1.2), in the launch
configuration bench.py times: FP8 tensor-core GEMMs, weights quantised once.

The oracle cannot run this whole layer, but most of it is local:
  * every forward operand and the dX-path operands are quantised along K,
    one row at a time, so a token's y, dx and d(routing weights) depend only
    on its own row and its k experts' weights -- the oracle runs that token
    alone against just those k experts;
  * an expert's weight gradients quantise their operands along the token
    axis in 32-row blocks that restart at the expert's segment (its tokens in
    ascending order), so the oracle runs exactly that expert's tokens against
    that expert alone (k = 1, each token's own routing weight) and the whole
    dW_gate[e], dW_up[e], dW_down[e] are compared.
Tolerance: the MXFP8 bound, max|err| <= 6e-2 * max|ref| over the sampled
elements of each tensor; the routing ids are exact."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, inputs

from gpu_helpers import assert_close, dev

pytestmark = pytest.mark.gpu

MX_TOL = 6e-2


def test_mxfp8_full_size_sampled_parity():
    torch.cuda.empty_cache()
    shape = inputs.SKEWED_MXFP8
    d = dev()
    inp = inputs.make_inputs(shape, seed=0, device=d)
    fwd, bwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=d,
                     minibatch_rows=shape.minibatch_rows, dtype="mxfp8")
    layer.step(inp["x"], inp["logits"], inp["bias"], *fwd, inp["dy"], bwd=bwd, mx=mx)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    del fwd, bwd, mx

    ids, w = oracle.route_topk(inp["logits"].cpu().numpy(), inp["bias"].cpu().numpy(), shape.k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids)
    x, dy = (oracle.as_bf16_bits(inp[n]) for n in ("x", "dy"))
    wg, wu, wd = (oracle.as_bf16_bits(inp[n]) for n in ("wg", "wu", "wd"))
    g = layer.grads

    # sampled tokens: each alone, against its own k experts in its j order
    rng = np.random.default_rng(shape.N)
    tok = np.sort(rng.choice(shape.N, 4, replace=False))
    ref = {n: [] for n in ("y", "dx", "dw")}
    own = np.arange(shape.k, dtype=np.int32)[None]
    for t in tok:
        ex = ids[t]
        r = oracle.layer_mxfp8(x[t:t + 1], wg[ex], wu[ex], wd[ex], own, w[t:t + 1], dy[t:t + 1])
        for n in ref:
            ref[n].append(r[n][0])
    sel = torch.as_tensor(tok)
    assert_close("y", layer.y[sel], np.stack(ref["y"]), MX_TOL)
    assert_close("dx", g.dx[sel], np.stack(ref["dx"]), MX_TOL)
    assert_close("d_topk_w", g.d_topk_w[sel], np.stack(ref["dw"]), MX_TOL)

    # whole weight gradients of three experts: one token; 33 tokens (a ragged
    # 32-row block); the first with more than 128 (a second 128-row tile)
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    picks = []
    for lo in (1, 33, 129):
        cand = np.flatnonzero(counts >= lo)
        picks.append(int(cand[np.argmin(counts[cand])]))
    for e in sorted(set(picks)):
        hit = ids == e
        toks = np.flatnonzero(hit.any(axis=1))
        we = w[hit][:, None]  # row-major order of hit = ascending tokens
        r = oracle.layer_mxfp8(x[toks], wg[e:e + 1], wu[e:e + 1], wd[e:e + 1],
                               np.zeros((len(toks), 1), np.int32), we, dy[toks])
        assert_close(f"dw_gate[{e}] (m_e={len(toks)})", g.dw_gate[e], r["dwg"][0], MX_TOL)
        assert_close(f"dw_up[{e}] (m_e={len(toks)})", g.dw_up[e], r["dwu"][0], MX_TOL)
        assert_close(f"dw_down[{e}] (m_e={len(toks)})", g.dw_down[e], r["dwd"][0], MX_TOL)
    del layer, inp
    torch.cuda.empty_cache()
