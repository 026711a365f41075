"""GPU layer parity.

1. Each phase kernel against a plain PyTorch fp32 reference of the same op,
   computed from the kernel's own inputs (isolates each GEMM mode).
2. The whole forward + backward against the fp64 oracle, element by element,
   max|err| <= 2e-2 * max|ref| per tensor, on sizes spanning several tiles
   with ragged tails and empty experts.
3. Identity experts (expert output := expert input), and bitwise-identical
   reruns (clip "Mixture-of-Kittens: Cursor open-sources an MoE training
   megakernel", key point 5 and "how to" item 6: fixed accumulation order).
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, _lib, inputs

from gpu_helpers import BF16_TOL, assert_close, custom_shape, dev, max_rel, run_layer, to_dev

pytestmark = pytest.mark.gpu

RAGGED = custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_skewed")


def _phase_setup(shape, seed=0):
    inp = to_dev(inputs.make_inputs(shape, seed=seed, device="cpu"))
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows)
    layer.route(inp["logits"], inp["bias"])
    layer.build_schedule()
    return inp, layer


def _segments(layer):
    s = {k: v.cpu().numpy() for k, v in layer.schedule_tensors().items()}
    return [(e, int(s["pad_offsets"][e]), int(s["counts"][e])) for e in range(layer.E)], s


PHASE_SHAPES = [inputs.TINY, RAGGED, inputs.TINY.with_(name="tiny_T256", minibatch_rows=256),
                RAGGED.with_(name="ragged_skewed_T256", minibatch_rows=256),
                # experts of 3568, 2130 and 1098 rows (weight-gradient tiles issued in
                # chunks, with short-K tiles of other experts between the chunks), one
                # of 527 rows, and twelve of at most 312 (seed 0)
                custom_shape(4096, 1024, 512, 16, 2, zipf_s=1.5, name="wgrad_chunked_and_short")]


@pytest.mark.parametrize("shape", PHASE_SHAPES, ids=lambda s: s.name)
def test_phases_match_torch_fp32(shape):
    inp, layer = _phase_setup(shape)
    p, ws = layer.p, layer.ws
    w = _lib.weights(inp["wg"], inp["wu"], inp["wd"])
    sv = layer.saved_tensors()
    xe, g, u, act, ye = sv["xe"], sv["g"], sv["u"], sv["act"], sv["ye"]
    sv["xe"].fill_(7.0)  # poison: padding rows must come back zero
    _lib.moe_dispatch(p, ws, inp["x"], xe)
    torch.cuda.synchronize()
    segs, s = _segments(layer)
    slot_of = s["slot_of"].reshape(shape.N, shape.k)
    x = inp["x"]
    # dispatch: exact copies, zero padding
    np.testing.assert_array_equal(
        xe[torch.as_tensor(slot_of.ravel(), device=dev()).long()].view(torch.int16).cpu().numpy(),
        x.repeat_interleave(shape.k, 0).view(torch.int16).cpu().numpy())
    for e, r0, c in segs:
        pad_rows = xe[r0 + c: int(s["pad_offsets"][e + 1])]
        assert torch.all(pad_rows == 0)

    _lib.moe_expert_gate_up(p, ws, xe, w, g, u, act)
    _lib.moe_expert_down(p, ws, act, w, ye)
    torch.cuda.synchronize()
    wg, wu, wd = (inp[k].float() for k in ("wg", "wu", "wd"))
    for e, r0, c in segs:
        if c == 0:
            continue
        rows = slice(r0, r0 + c)
        G = xe[rows].float() @ wg[e].T
        U = xe[rows].float() @ wu[e].T
        assert_close(f"G[{e}]", g[rows], G.double().cpu().numpy(), 1e-2)
        assert_close(f"U[{e}]", u[rows], U.double().cpu().numpy(), 1e-2)
        A = torch.nn.functional.silu(G) * U
        assert_close(f"Act[{e}]", act[rows], A.double().cpu().numpy(), 1e-2)
        Y = act[rows].float() @ wd[e].T
        assert_close(f"Ye[{e}]", ye[rows], Y.double().cpu().numpy(), 1e-2)

    # combine
    _lib.moe_combine(p, ws, ye, layer.topk_w, layer.y)
    torch.cuda.synchronize()
    sl = torch.as_tensor(slot_of, device=dev()).long()
    yref = (layer.topk_w.unsqueeze(-1) * ye[sl].float()).sum(1)
    assert_close("y", layer.y, yref.double().cpu().numpy(), 1e-2)

    # backward phases
    dy = inp["dy"]
    dye = torch.empty_like(ye)
    dye.fill_(3.0)
    dtw = torch.empty_like(layer.topk_w)
    _lib.moe_reverse_combine(p, ws, dy, ye, layer.topk_w, dye, dtw)
    torch.cuda.synchronize()
    dye_ref = (layer.topk_w.unsqueeze(-1) * dy.float().unsqueeze(1)).bfloat16()
    assert torch.equal(dye[sl], dye_ref)
    for e, r0, c in segs:
        assert torch.all(dye[r0 + c: int(s["pad_offsets"][e + 1])] == 0)
    dw_ref = (dy.float().unsqueeze(1) * ye[sl].float()).sum(-1)
    assert_close("d_topk_w", dtw, dw_ref.double().cpu().numpy(), 1e-4)

    dg, du = torch.empty_like(g), torch.empty_like(u)
    dwd = torch.full((shape.E, shape.H, shape.I), 5.0, device=dev())
    _lib.moe_expert_down_dgrad(p, ws, dye, g, u, w, dg, du)
    _lib.moe_expert_down_wgrad(p, ws, dye, act, dwd)
    torch.cuda.synchronize()
    for e, r0, c in segs:
        rows = slice(r0, r0 + c)
        if c == 0:
            assert torch.all(dwd[e] == 0)
            continue
        dA = dye[rows].float() @ wd[e]
        G, U = g[rows].float(), u[rows].float()
        sg = torch.sigmoid(G)
        assert_close(f"dG[{e}]", dg[rows], (dA * U * sg * (1 + G * (1 - sg))).double().cpu().numpy(), 1e-2)
        assert_close(f"dU[{e}]", du[rows], (dA * G * sg).double().cpu().numpy(), 1e-2)
        assert_close(f"dWd[{e}]", dwd[e], (dye[rows].float().T @ act[rows].float()).double().cpu().numpy(), 1e-3)

    dxe = torch.empty_like(xe)
    dwg = torch.full((shape.E, shape.I, shape.H), 5.0, device=dev())
    dwu = torch.full_like(dwg, 5.0)
    _lib.moe_expert_gate_up_dgrad(p, ws, dg, du, w, dxe)
    _lib.moe_expert_gate_up_wgrad(p, ws, dg, du, xe, dwg, dwu)
    torch.cuda.synchronize()
    for e, r0, c in segs:
        rows = slice(r0, r0 + c)
        if c == 0:
            assert torch.all(dwg[e] == 0) and torch.all(dwu[e] == 0)
            continue
        ref = dg[rows].float() @ wg[e] + du[rows].float() @ wu[e]
        assert_close(f"dXe[{e}]", dxe[rows], ref.double().cpu().numpy(), 1e-2)
        assert_close(f"dWg[{e}]", dwg[e], (dg[rows].float().T @ xe[rows].float()).double().cpu().numpy(), 1e-3)
        assert_close(f"dWu[{e}]", dwu[e], (du[rows].float().T @ xe[rows].float()).double().cpu().numpy(), 1e-3)

    dx = torch.empty_like(x)
    _lib.moe_reverse_dispatch(p, ws, dxe, dx)
    torch.cuda.synchronize()
    assert_close("dx", dx, dxe[sl].float().sum(1).double().cpu().numpy(), 1e-2)
    assert layer.device_error() == 0


def _oracle_compare(shape, inp_cpu, layer, backward=True):
    logits = inp_cpu["logits"].numpy()
    bias = None if inp_cpu["bias"] is None else inp_cpu["bias"].numpy()
    ids, w = oracle.route_topk(logits, bias, shape.k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids)
    y = oracle.forward_bf16(inp_cpu["x"], inp_cpu["wg"], inp_cpu["wu"], inp_cpu["wd"], ids, w)
    errs = {"y": assert_close("y", layer.y, y)}
    if backward:
        r = oracle.backward_bf16(inp_cpu["x"], inp_cpu["wg"], inp_cpu["wu"], inp_cpu["wd"], ids,
                                 w, inp_cpu["dy"])
        g = layer.grads
        for name, got, key in (("dx", g.dx, "dx"), ("dw_gate", g.dw_gate, "dwg"),
                               ("dw_up", g.dw_up, "dwu"), ("dw_down", g.dw_down, "dwd"),
                               ("d_topk_w", g.d_topk_w, "dw")):
            errs[name] = assert_close(name, got, r[key])
    return errs


LAYER_SHAPES = [
    inputs.TINY,
    RAGGED,
    custom_shape(129, 256, 256, 4, 2, name="one_over_tile"),
    custom_shape(64, 1024, 512, 32, 8, name="many_empty_experts"),
    custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_skewed_T256", T=256),
    custom_shape(129, 256, 512, 4, 2, name="one_over_tile_T1024", T=1024),
    custom_shape(64, 1024, 512, 32, 8, name="many_empty_experts_T512", T=512),
    custom_shape(1, 256, 256, 4, 1, name="one_token_k1"),
    custom_shape(100, 256, 512, 4, 4, name="k_equals_E"),
    custom_shape(77, 512, 256, 1, 1, name="single_expert"),
]


@pytest.mark.parametrize("shape", LAYER_SHAPES, ids=lambda s: s.name)
def test_layer_matches_oracle(shape):
    inp = inputs.make_inputs(shape, seed=1, device="cpu")
    layer = run_layer(shape, to_dev(inp))
    assert layer.device_error() == 0
    _oracle_compare(shape, inp, layer)


def test_expert_without_tokens_gets_zero_weight_gradient():
    shape = custom_shape(200, 256, 512, 8, 2, name="forced_empty")
    inp = inputs.make_inputs(shape, seed=2, device="cpu")
    inp["bias"] = torch.zeros(8)
    inp["bias"][[3, 6]] = -1e4  # never selected
    layer = run_layer(shape, to_dev(inp))
    g = layer.grads
    for e in (3, 6):
        assert torch.all(g.dw_gate[e] == 0) and torch.all(g.dw_up[e] == 0)
        assert torch.all(g.dw_down[e] == 0)
    _oracle_compare(shape, inp, layer)


def test_identity_experts():
    """Expert output := expert input. With weights summing to 1 the combine
    returns x up to one bf16 rounding; the reverse rounds return dy and
    d_topk_w = <dy, x>."""
    shape = RAGGED
    inp, layer = _phase_setup(shape, seed=3)
    p, ws = layer.p, layer.ws
    sv = layer.saved_tensors()
    _lib.moe_dispatch(p, ws, inp["x"], sv["xe"])
    _lib.moe_combine(p, ws, sv["xe"], layer.topk_w, layer.y)
    torch.cuda.synchronize()
    x = inp["x"].float()
    assert torch.max(torch.abs(layer.y.float() - x)) <= 2.0 ** -7 * torch.max(torch.abs(x))
    dy = inp["dy"]
    dye = torch.empty_like(sv["xe"])
    dtw = torch.empty_like(layer.topk_w)
    _lib.moe_reverse_combine(p, ws, dy, sv["xe"], layer.topk_w, dye, dtw)
    dx = torch.empty_like(inp["x"])
    _lib.moe_reverse_dispatch(p, ws, dye, dx)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(dx.float() - dy.float())) <= 2.0 ** -6 * torch.max(torch.abs(dy.float()))
    ref = (dy.double() * inp["x"].double()).sum(1, keepdim=True).expand(-1, shape.k)
    assert max_rel(dtw, ref.cpu().numpy()) <= 1e-5


def test_reruns_are_bitwise_identical():
    shape = RAGGED
    inp = to_dev(inputs.make_inputs(shape, seed=4, device="cpu"))
    a = run_layer(shape, inp)
    b = run_layer(shape, inp)
    assert torch.equal(a.y, b.y)
    rows = int(a.schedule_tensors()["pad_offsets"][shape.E])
    for key, t in a.saved_tensors().items():
        assert torch.equal(t[:rows], b.saved_tensors()[key][:rows]), key
    for f in ("dx", "dw_gate", "dw_up", "dw_down", "d_topk_w"):
        assert torch.equal(getattr(a.grads, f), getattr(b.grads, f)), f


CHAIN_SHAPES = [RAGGED, RAGGED.with_(name="ragged_skewed_T256", minibatch_rows=256),
                custom_shape(2048, 1024, 512, 16, 4, zipf_s=1.2, name="many_tiles_skewed")]


@pytest.mark.parametrize("overlap", [False, True], ids=["moe_backward", "moe_backward_overlap"])
@pytest.mark.parametrize("shape", CHAIN_SHAPES, ids=lambda s: s.name)
def test_backward_equals_phase_chain(shape, overlap):
    """moe_backward, and moe_backward_overlap (the reverse-combine inside the
    down data-gradient GEMM: side warps publish finished tiles, the GEMM waits
    for each tile it loads), must equal, bit for bit, the chain of the
    separate phase entry points on the same inputs."""
    inp = to_dev(inputs.make_inputs(shape, seed=5, device="cpu"))
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows)
    layer.step(inp["x"], inp["logits"], inp["bias"], inp["wg"], inp["wu"], inp["wd"], inp["dy"],
               overlap=overlap)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    p, ws = layer.p, layer.ws
    w = _lib.weights(inp["wg"], inp["wu"], inp["wd"])
    sv = layer.saved_tensors()
    dye = torch.empty_like(sv["xe"])
    dtw = torch.empty_like(layer.topk_w)
    dg = torch.empty_like(sv["g"])
    du = torch.empty_like(sv["u"])
    dxe = torch.empty_like(sv["xe"])
    dwg = torch.empty_like(layer.grads.dw_gate)
    dwu = torch.empty_like(layer.grads.dw_up)
    dwd = torch.empty_like(layer.grads.dw_down)
    dx = torch.empty_like(inp["x"])
    _lib.moe_reverse_combine(p, ws, inp["dy"], sv["ye"], layer.topk_w, dye, dtw)
    _lib.moe_expert_down_dgrad(p, ws, dye, sv["g"], sv["u"], w, dg, du)
    _lib.moe_expert_down_wgrad(p, ws, dye, sv["act"], dwd)
    _lib.moe_expert_gate_up_dgrad(p, ws, dg, du, w, dxe)
    _lib.moe_expert_gate_up_wgrad(p, ws, dg, du, sv["xe"], dwg, dwu)
    _lib.moe_reverse_dispatch(p, ws, dxe, dx)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    g = layer.grads
    for name, got, want in (("d_topk_w", g.d_topk_w, dtw), ("dx", g.dx, dx),
                            ("dw_gate", g.dw_gate, dwg), ("dw_up", g.dw_up, dwu),
                            ("dw_down", g.dw_down, dwd)):
        assert torch.equal(got, want), name


# Shapes whose context-free forward runs Xe and Act through the ring of
# minibatch slots, wrapping around it several times: the ring has lag + 4
# slots, lag = max(2, ceil(3 * CTA pairs / (I / 128 + H / 256))), and needs
# ring * 256 * (H + I) <= R * I rows of scratch (R >= N * k); with at most 76
# CTA pairs that holds here, for about 130 and 260 pair items.
RING_SHAPES = [custom_shape(4096, 1024, 1024, 16, 8, zipf_s=1.2, name="ring_wraps_skewed"),
               custom_shape(8192, 2048, 1024, 32, 8, name="ring_wraps_uniform")]

FUSED_SHAPES = CHAIN_SHAPES + [LAYER_SHAPES[i] for i in (2, 3, 5, 7, 8, 9)] + [
    custom_shape(3000, 1024, 768, 16, 8, zipf_s=1.2, name="fused_skewed_odd_items")] + RING_SHAPES


@pytest.mark.parametrize("inference", [False, True], ids=["training", "inference"])
@pytest.mark.parametrize("shape", FUSED_SHAPES, ids=lambda s: s.name)
def test_fused_forward_equals_phase_chain(shape, inference):
    """moe_dispatch_expert_ffn (dispatch, gate/up + SwiGLU and down in one
    persistent launch) followed by the combine must equal, bit for bit,
    moe_dispatch + moe_expert_gate_up + moe_expert_down + moe_combine on the
    same inputs: Xe (padding rows zero), G, U, Act, Ye and y. The context-free
    forward (moe_forward_inference: the fused launch with Xe and Act in a ring
    of 256-row minibatch slots where the scratch holds one, else with Xe and
    Ye sharing one scratch buffer) gives the same y."""
    inp = to_dev(inputs.make_inputs(shape, seed=4, device="cpu"))
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows, allocate_grads=False)
    layer.route(inp["logits"], inp["bias"])
    layer.build_schedule()
    sv = layer.saved_tensors()
    for t in sv.values():
        t.fill_(float("nan"))  # rows the fused launch must write
    p, ws = layer.p, layer.ws
    w = _lib.weights(inp["wg"], inp["wu"], inp["wd"])
    if inference:
        y = layer.forward_inference(inp["x"], inp["wg"], inp["wu"], inp["wd"]).clone()
    else:
        _lib.moe_dispatch_expert_ffn(p, ws, inp["x"], w, sv["xe"], sv["g"], sv["u"], sv["act"],
                                     sv["ye"])
        _lib.moe_combine(p, ws, sv["ye"], layer.topk_w, layer.y)
        y = layer.y.clone()
        got = {k: v.clone() for k, v in sv.items()}
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ref = {k: torch.empty_like(v) for k, v in sv.items()}
    y_ref = torch.empty_like(y)
    _lib.moe_dispatch(p, ws, inp["x"], ref["xe"])
    _lib.moe_expert_gate_up(p, ws, ref["xe"], w, ref["g"], ref["u"], ref["act"])
    _lib.moe_expert_down(p, ws, ref["act"], w, ref["ye"])
    _lib.moe_combine(p, ws, ref["ye"], layer.topk_w, y_ref)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(y, y_ref)
    if inference:
        return
    rows = int(layer.schedule_tensors()["pad_offsets"][shape.E])
    for name in ("xe", "g", "u", "act", "ye"):
        assert torch.equal(got[name][:rows].view(torch.int16), ref[name][:rows].view(torch.int16)), name


@pytest.mark.parametrize("shape", RING_SHAPES, ids=lambda s: s.name)
def test_ring_forward_reruns_are_bitwise_identical(shape):
    """The ring forward's slot recycling depends on timing (which CTA frees a
    slot first); its results must not."""
    inp = to_dev(inputs.make_inputs(shape, seed=9, device="cpu"))
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(), allocate_grads=False)
    layer.route(inp["logits"], inp["bias"])
    layer.build_schedule()
    ys = [layer.forward_inference(inp["x"], inp["wg"], inp["wu"], inp["wd"]).clone()
          for _ in range(3)]
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.isfinite(ys[0].float()).all()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_fused_forward_reruns_are_bitwise_identical():
    shape = custom_shape(3000, 1024, 768, 16, 8, zipf_s=1.2, name="fused_rerun")
    inp = to_dev(inputs.make_inputs(shape, seed=8, device="cpu"))
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(), allocate_grads=False)
    layer.route(inp["logits"], inp["bias"])
    layer.build_schedule()
    w = _lib.weights(inp["wg"], inp["wu"], inp["wd"])
    sv = layer.saved_tensors()
    outs = []
    for _ in range(3):
        _lib.moe_dispatch_expert_ffn(layer.p, layer.ws, inp["x"], w, sv["xe"], sv["g"], sv["u"],
                                     sv["act"], sv["ye"])
        _lib.moe_combine(layer.p, layer.ws, sv["ye"], layer.topk_w, layer.y)
        outs.append((layer.y.clone(), layer.saved.clone()))
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    for y, s in outs[1:]:
        assert torch.equal(y.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(s, outs[0][1])


def test_weight_gradient_of_a_dominant_expert():
    """One expert takes every token (K = 4096 rows = 64 k-blocks): its weight-
    gradient tiles are long enough to be issued in chunks with the other
    experts' tiles between them. Gradients match the oracle and reruns are
    bitwise identical."""
    shape = custom_shape(4096, 256, 512, 8, 2, name="dominant_expert")
    inp = inputs.make_inputs(shape, seed=6, device="cpu")
    inp["bias"] = torch.zeros(8)
    inp["bias"][0] = 1e4  # always selected
    a = run_layer(shape, to_dev(inp))
    assert a.device_error() == 0
    counts = a.schedule_tensors()["counts"].cpu().numpy()
    assert counts[0] == shape.N
    _oracle_compare(shape, inp, a)
    b = run_layer(shape, to_dev(inp))
    for f in ("dw_gate", "dw_up", "dw_down"):
        assert torch.equal(getattr(a.grads, f), getattr(b.grads, f)), f


def test_empty_batch():
    """N = 0: every phase is a no-op; the weight gradients are written as zeros."""
    shape = custom_shape(0, 256, 512, 8, 2, name="empty")
    inp = to_dev(inputs.make_inputs(custom_shape(4, 256, 512, 8, 2), seed=7, device="cpu"))
    layer = MoELayer(0, 256, 512, 8, 2, device=dev())
    for t in (layer.grads.dw_gate, layer.grads.dw_up, layer.grads.dw_down):
        t.fill_(3.0)
    empty = {k: v[:0] for k, v in inp.items() if k in ("x", "logits", "dy")}
    layer.step(empty["x"], empty["logits"], None, inp["wg"], inp["wu"], inp["wd"], empty["dy"])
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert layer.y.shape == (0, 256) and layer.grads.dx.shape == (0, 256)
    for t in (layer.grads.dw_gate, layer.grads.dw_up, layer.grads.dw_down):
        assert torch.all(t == 0)
    # the fused dispatch + expert FFN launch on an empty batch: nothing to do,
    # and no counter wait is left waiting
    layer.forward_inference(empty["x"], inp["wg"], inp["wu"], inp["wd"])
    torch.cuda.synchronize()
    assert layer.device_error() == 0


@pytest.mark.parametrize("stages,tile_n", [(4, 256), (5, 256), (6, 256), (0, 512), (0, 256)])
def test_results_do_not_depend_on_the_ring_depth(stages, tile_n):
    """moe_problem.pipeline_stages only changes how many k-blocks the SM-pair
    GEMMs keep in flight, and tile_n = 512 only makes two N tiles share each
    staged A k-block (two pair MMAs per k-step into the two halves of TMEM):
    the MMAs of every 256-column block, their order and the epilogues are the
    same, so every output equals the library's default choice bit for bit
    (ragged experts, odd last 128-row items, several N tiles)."""
    shape = custom_shape(2048, 1024, 512, 16, 4, zipf_s=1.2, name="ring_depth")
    inp = to_dev(inputs.make_inputs(shape, seed=5, device="cpu"))
    ref = run_layer(shape, inp)
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     pipeline_stages=stages, tile_n=tile_n)
    layer.step(inp["x"], inp["logits"], inp["bias"], inp["wg"], inp["wu"], inp["wd"], inp["dy"])
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(layer.y.view(torch.int16), ref.y.view(torch.int16))
    rows = int(ref.schedule_tensors()["pad_offsets"][shape.E])  # rows past it are never written
    got, want = layer.saved_tensors(), ref.saved_tensors()
    for name in want:
        assert torch.equal(got[name][:rows].view(torch.int16), want[name][:rows].view(torch.int16)), name
    for name in ("dx", "dw_gate", "dw_up", "dw_down", "d_topk_w"):
        a, b = getattr(layer.grads, name), getattr(ref.grads, name)
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), name


@pytest.mark.parametrize("shape", [LAYER_SHAPES[i] for i in (0, 1, 3, 4, 5, 9)], ids=lambda s: s.name)
def test_wide_tiles_match_oracle(shape):
    """The whole layer with 512-wide pair tiles in the token-row GEMMs, against
    the fp64 oracle (bf16 bound), on ragged, empty-expert, T = 256 / 1024 and
    single-expert shapes."""
    inp = inputs.make_inputs(shape, seed=1, device="cpu")
    d = to_dev(inp)
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows, tile_n=512)
    layer.step(d["x"], d["logits"], d["bias"], d["wg"], d["wu"], d["wd"], d["dy"])
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    _oracle_compare(shape, inp, layer)
