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
    ascending order), each column on its own, so sampled entries of dW need
    only the sampled rows and columns of that expert's operands
    (oracle.expert_wgrad_mxfp8) -- cheap even for the expert that takes
    almost every token.
Tolerance: the MXFP8 bound, max|err| <= 6e-2 * max|ref| over the sampled
elements of each tensor (all sampled experts together, as the bound is per
tensor); the routing ids are exact. A single expert's slice is not the
tensor: with few tokens, one E4M3 code that flips between the two sides
(an intermediate next to a rounding boundary, fp32 against fp64) moves a
small expert's dW by several percent of that expert's own maximum."""
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

    # weight gradients: sampled entries of five experts, from one token to the
    # dominant expert (its long tiles go through the chunked weight-gradient
    # plan): 1, 33 (a ragged 32-token block), the first above 128 (a second
    # 128-row tile), the median and the largest expert
    counts = np.bincount(ids.reshape(-1), minlength=shape.E)
    nz = np.flatnonzero(counts)
    picks = {int(nz[np.argmin(counts[nz])]), int(np.argmax(counts)),
             int(nz[np.argsort(counts[nz], kind="stable")[len(nz) // 2]])}
    for lo in (33, 129):
        cand = np.flatnonzero(counts >= lo)
        picks.add(int(cand[np.argmin(counts[cand])]))
    il = np.sort(rng.choice(shape.I, 16, replace=False)).astype(np.int32)
    hl = np.sort(rng.choice(shape.H, 32, replace=False)).astype(np.int32)
    il_t, hl_t = torch.as_tensor(il, device=d).long(), torch.as_tensor(hl, device=d).long()
    got = {n: [] for n in ("dwg", "dwu", "dwd")}
    want = {n: [] for n in got}
    for e in sorted(picks):
        r = oracle.expert_wgrad_mxfp8(x, wg, wu, wd, ids, w, dy, e, il, hl)
        got["dwg"].append(g.dw_gate[e][il_t][:, hl_t])
        got["dwu"].append(g.dw_up[e][il_t][:, hl_t])
        got["dwd"].append(g.dw_down[e][hl_t][:, il_t])
        for n in want:
            want[n].append(r[n])
            # gross-error screen per expert: a flipped E4M3 code moves a
            # product by at most 2^-3 of itself, so two flips on the dominant
            # product stay under a quarter of the expert's own maximum
            assert_close(f"{n}[{e}] (m_e={counts[e]})", got[n][-1], r[n], 0.25)
    # the bound is per tensor: max|err| over the sampled entries of all five
    # experts against max|ref| over the same entries
    for n, name in (("dwg", "dw_gate"), ("dwu", "dw_up"), ("dwd", "dw_down")):
        assert_close(f"{name} (experts {sorted(picks)}, m_e {sorted(counts[list(picks)])})",
                     torch.cat(got[n]), np.concatenate(want[n]), MX_TOL)
    del layer, inp
    torch.cuda.empty_cache()
