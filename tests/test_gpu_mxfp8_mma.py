"""MXFP8 on the block-scaled tensor cores (tcgen05 kind::mxf8f6f4).

* The MMA-layout quantiser, row and transposed forms, gives the oracle
  quantiser's E4M3 codes bit-exactly and its E8M0 scales at the chunk
  positions include/moe.h documents.
* The MXFP8 forward and backward on FP8 MMAs match the same passes on bf16
  MMAs of the exact MXFP8 values (the same products, fp32 sums in another
  order; an intermediate that lands next to a rounding boundary may quantise
  to the neighbouring code) to 1e-2 * max|ref| per tensor, also at the full
  skewed size, are bitwise identical across reruns, and the whole FP8 layer
  matches the oracle's MXFP8 layer within 6e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, _lib, inputs

from gpu_helpers import assert_close, custom_shape, dev, max_rel, to_dev

pytestmark = pytest.mark.gpu

MX_TOL = 6e-2
SAME_PRODUCTS_TOL = 1e-2


def untile_scales(s, rows, k):
    """Scales [rows, k/32] from the 512-byte chunk layout of a K-major operand."""
    r = np.arange(rows)[:, None]
    j = np.arange(k // 32)[None, :]
    idx = ((j // 4) * (rows // 128) + r // 128) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (j % 4)
    return s[idx]


@pytest.mark.parametrize("transpose", [0, 1])
@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 384), (384, 1024)])
def test_quantize_mma_matches_oracle(transpose, rows, cols):
    g = torch.Generator().manual_seed(rows + cols + transpose)
    spread = torch.exp(torch.empty((rows, 1)).uniform_(-8, 8, generator=g))
    x = (torch.randn((rows, cols), generator=g) * spread).bfloat16()
    x[0, :64] = 0.0  # all-zero blocks take scale code 0
    q = torch.empty(rows * cols, dtype=torch.uint8, device=dev())
    s = torch.empty(rows * cols // 32, dtype=torch.uint8, device=dev())
    _lib.mxfp8_quantize_mma(x.to(dev()), rows, cols, transpose, q, s)
    torch.cuda.synchronize()
    src = oracle.as_bf16_bits(x)
    if transpose:
        src = np.ascontiguousarray(src.T)
    ref_q, ref_s = oracle.mxfp8_quantize(src)
    R, K = ref_q.shape
    np.testing.assert_array_equal(q.cpu().numpy().reshape(R, K), ref_q)
    np.testing.assert_array_equal(untile_scales(s.cpu().numpy(), R, K), ref_s)


@pytest.mark.parametrize("shape", [custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged"),
                                   custom_shape(300, 512, 768, 16, 4, name="ragged_T256", T=256),
                                   custom_shape(64, 1024, 512, 32, 8, name="many_empty")],
                         ids=lambda s: s.name)
def test_dispatch_mxfp8_equals_dispatch_then_quantise(shape):
    """The fused dispatch + row quantiser writes Xe, its codes and its scales
    exactly as moe_dispatch followed by mxfp8_quantize_mma on every row of the
    used expert segments; padding rows get zero codes and scales."""
    inp_cpu = inputs.make_inputs(shape, seed=8, device="cpu")
    g = torch.Generator().manual_seed(8)
    spread = torch.exp(torch.empty((shape.N, 1)).uniform_(-8, 8, generator=g))
    inp_cpu["x"] = (inp_cpu["x"].float() * spread).bfloat16()
    inp_cpu["x"][0, :64] = 0.0
    inp = to_dev(inp_cpu)
    layer = MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                     minibatch_rows=shape.minibatch_rows)
    layer.route(inp["logits"], inp["bias"])
    layer.build_schedule()
    p, ws, R, H = layer.p, layer.ws, layer.R, shape.H
    xe1 = torch.full((R, H), 5.0, dtype=torch.bfloat16, device=dev())
    xe2 = torch.full((R, H), 7.0, dtype=torch.bfloat16, device=dev())
    q1 = torch.empty(R * H, dtype=torch.uint8, device=dev())
    s1 = torch.empty(R * H // 32, dtype=torch.uint8, device=dev())
    q2 = torch.full((R * H,), 0x55, dtype=torch.uint8, device=dev())
    s2 = torch.full((R * H // 32,), 0x55, dtype=torch.uint8, device=dev())
    _lib.moe_dispatch(p, ws, inp["x"], xe1)
    _lib.mxfp8_quantize_mma(xe1, R, H, 0, q1, s1)
    _lib.moe_dispatch_mxfp8(p, ws, inp["x"], xe2, q2, s2)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    used = int(layer.schedule_tensors()["pad_offsets"][shape.E])
    assert torch.equal(xe2[:used], xe1[:used])
    qa, qb = q1.view(R, H)[:used], q2.view(R, H)[:used]
    assert torch.equal(qa, qb)
    sa = untile_scales(s1.cpu().numpy(), R, H)[:used]
    sb = untile_scales(s2.cpu().numpy(), R, H)[:used]
    np.testing.assert_array_equal(sb, sa)
    src = layer.schedule_tensors()["src_of_row"][:used].cpu().numpy()
    pad = np.nonzero(src < 0)[0]
    assert np.all(sb[pad] == 0) and torch.all(qb[torch.as_tensor(pad, device=dev())] == 0)


def test_quantize_mma_rejects_unaligned_sizes():
    x = torch.zeros((128, 96), dtype=torch.bfloat16, device=dev())
    q = torch.empty(128 * 96, dtype=torch.uint8, device=dev())
    s = torch.empty(128 * 3, dtype=torch.uint8, device=dev())
    with pytest.raises(_lib.MoEError):
        _lib.mxfp8_quantize_mma(x, 128, 96, 0, q, s)


SHAPES = [inputs.TINY.with_(name="tiny_mxfp8", dtype="mxfp8"),
          custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_skewed_mxfp8").with_(dtype="mxfp8"),
          custom_shape(300, 768, 512, 16, 4, name="odd_h_tiles_mxfp8").with_(dtype="mxfp8"),
          custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name="ragged_T256_mxfp8", T=256).with_(dtype="mxfp8")]


def _layer(shape):
    return MoELayer(shape.N, shape.H, shape.I, shape.E, shape.k, device=dev(),
                    minibatch_rows=shape.minibatch_rows, dtype="mxfp8")


class _DevBytes:
    """A raw device buffer of n bytes as a CUDA-array-interface object."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "|u1", "data": (ptr, False),
                                         "version": 3}


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_fp8_forward_operands_equal_the_quantiser(shape):
    """The MXFP8 forward quantises Xe's rows in the dispatch and Act's rows in
    the gate/up epilogue. Both must equal, bit for bit, mxfp8_quantize_mma of
    the saved bf16 Xe and Act on every row of the used expert segments."""
    inp = to_dev(inputs.make_inputs(shape, seed=9, device="cpu"))
    fwd, _ = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"], backward=False)
    layer = _layer(shape)
    layer.route(inp["logits"], inp["bias"])
    layer.build_schedule()
    layer.forward(inp["x"], *fwd, mx=mx)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    R, used = layer.R, int(layer.schedule_tensors()["pad_offsets"][shape.E])
    sv = layer.saved_tensors()
    ops = _lib.moe_mxfp8_forward_operands(layer.p, layer.ws)
    for (q_ptr, s_ptr), src, K in zip(ops, (sv["xe"], sv["act"]), (shape.H, shape.I)):
        q_ref = torch.empty(R * K, dtype=torch.uint8, device=dev())
        s_ref = torch.empty(R * K // 32, dtype=torch.uint8, device=dev())
        _lib.mxfp8_quantize_mma(src, R, K, 0, q_ref, s_ref)
        q_got = torch.as_tensor(_DevBytes(q_ptr, R * K), device=dev()).clone()
        s_got = torch.as_tensor(_DevBytes(s_ptr, R * K // 32), device=dev()).clone()
        torch.cuda.synchronize()
        assert torch.equal(q_got.view(R, K)[:used], q_ref.view(R, K)[:used]), K
        np.testing.assert_array_equal(untile_scales(s_got.cpu().numpy(), R, K)[:used],
                                      untile_scales(s_ref.cpu().numpy(), R, K)[:used])


@pytest.mark.parametrize("shape", SHAPES + [custom_shape(2048, 512, 768, 16, 8, zipf_s=1.2,
                                                       name="many_tiles_mxfp8").with_(dtype="mxfp8")],
                         ids=lambda s: s.name)
def test_fp8_backward_operands_equal_the_quantiser(shape):
    """The MXFP8 backward quantises dG and dU into both forms the later GEMMs
    read: rows along I (gate/up data gradient) and the transposed form along
    the token axis (gate/up weight gradient). Each must equal, bit for bit,
    mxfp8_quantize_mma of the bf16 dG and dU the down data gradient wrote, on
    every row (token) of the used expert segments."""
    inp = to_dev(inputs.make_inputs(shape, seed=10, device="cpu"))
    fwd, bwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    layer = _layer(shape)
    layer.step(inp["x"], inp["logits"], inp["bias"], *fwd, inp["dy"], bwd=bwd, mx=mx)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    R, I = layer.R, shape.I
    used = int(layer.schedule_tensors()["pad_offsets"][shape.E])
    ops = _lib.moe_mxfp8_backward_operands(layer.p, layer.ws)
    for t in ("dg", "du"):
        src = torch.as_tensor(_DevBytes(ops[t], R * I * 2), device=dev()).view(torch.bfloat16)
        src = src.view(R, I).clone()
        for form, tr in (("_rows", 0), ("_cols", 1)):
            q_ref = torch.empty(R * I, dtype=torch.uint8, device=dev())
            s_ref = torch.empty(R * I // 32, dtype=torch.uint8, device=dev())
            _lib.mxfp8_quantize_mma(src, R, I, tr, q_ref, s_ref)
            q_ptr, s_ptr = ops[t + form]
            q_got = torch.as_tensor(_DevBytes(q_ptr, R * I), device=dev()).clone()
            s_got = torch.as_tensor(_DevBytes(s_ptr, R * I // 32), device=dev()).clone()
            torch.cuda.synchronize()
            if tr == 0:
                assert torch.equal(q_got.view(R, I)[:used], q_ref.view(R, I)[:used]), t + form
                np.testing.assert_array_equal(untile_scales(s_got.cpu().numpy(), R, I)[:used],
                                              untile_scales(s_ref.cpu().numpy(), R, I)[:used])
            else:
                assert torch.equal(q_got.view(I, R)[:, :used], q_ref.view(I, R)[:, :used]), t + form
                np.testing.assert_array_equal(
                    untile_scales(s_got.cpu().numpy(), I, R)[:, :used // 32],
                    untile_scales(s_ref.cpu().numpy(), I, R)[:, :used // 32])


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_fp8_forward_matches_bf16_mma_forward(shape):
    inp = to_dev(inputs.make_inputs(shape, seed=5, device="cpu"))
    fwd, _ = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    a, b = _layer(shape), _layer(shape)
    for lay in (a, b):
        lay.route(inp["logits"], inp["bias"])
        lay.build_schedule()
    a.forward(inp["x"], *fwd, mx=mx)
    b.forward(inp["x"], *fwd)
    torch.cuda.synchronize()
    assert a.device_error() == 0 and b.device_error() == 0
    rows = int(a.schedule_tensors()["pad_offsets"][shape.E].item())
    sa, sb = a.saved_tensors(), b.saved_tensors()
    for name in ("g", "u", "act", "ye"):
        e = max_rel(sa[name][:rows], sb[name][:rows].float().cpu().numpy())
        assert e <= SAME_PRODUCTS_TOL, (name, e)
    e = max_rel(a.y, b.y.float().cpu().numpy())
    assert e <= SAME_PRODUCTS_TOL, ("y", e)
    y1 = a.y.clone()
    a.forward(inp["x"], *fwd, mx=mx)
    torch.cuda.synchronize()
    assert torch.equal(a.y, y1), "FP8 forward is not bitwise reproducible"


@pytest.mark.parametrize("shape", SHAPES[:2], ids=lambda s: s.name)
def test_fp8_layer_matches_oracle(shape):
    inp_cpu = inputs.make_inputs(shape, seed=3, device="cpu")
    inp = to_dev(inp_cpu)
    fwd, bwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    layer = _layer(shape)
    layer.step(inp["x"], inp["logits"], inp["bias"], *fwd, inp["dy"], bwd=bwd, mx=mx)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    logits = inp_cpu["logits"].numpy()
    bias = None if inp_cpu["bias"] is None else inp_cpu["bias"].numpy()
    ids, w = oracle.route_topk(logits, bias, shape.k)
    r = oracle.layer_mxfp8(inp_cpu["x"], inp_cpu["wg"], inp_cpu["wu"], inp_cpu["wd"], ids, w,
                           inp_cpu["dy"], quantize=True)
    g = layer.grads
    assert_close("y", layer.y, r["y"], MX_TOL)
    for name, got, key in (("dx", g.dx, "dx"), ("dw_gate", g.dw_gate, "dwg"),
                           ("dw_up", g.dw_up, "dwu"), ("dw_down", g.dw_down, "dwd"),
                           ("d_topk_w", g.d_topk_w, "dw")):
        assert_close(name, got, r[key], MX_TOL)


def test_fp8_inference_forward_matches_training_forward():
    shape = SHAPES[1]
    inp = to_dev(inputs.make_inputs(shape, seed=9, device="cpu"))
    fwd, _ = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    a, b = _layer(shape), _layer(shape)
    for lay in (a, b):
        lay.route(inp["logits"], inp["bias"])
        lay.build_schedule()
    a.forward(inp["x"], *fwd, mx=mx)
    b.forward_inference(inp["x"], *fwd, mx=mx)
    torch.cuda.synchronize()
    assert torch.equal(a.y, b.y)


def _step_pair(shape, seed):
    """The same MXFP8 layer pass on FP8 MMAs (a) and on bf16 MMAs of the same
    MXFP8 values (b)."""
    inp = to_dev(inputs.make_inputs(shape, seed=seed, device="cpu"))
    fwd, bwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    a, b = _layer(shape), _layer(shape)
    a.step(inp["x"], inp["logits"], inp["bias"], *fwd, inp["dy"], bwd=bwd, mx=mx)
    b.step(inp["x"], inp["logits"], inp["bias"], *fwd, inp["dy"], bwd=bwd)
    torch.cuda.synchronize()
    assert a.device_error() == 0 and b.device_error() == 0
    return a, b, inp, fwd, bwd, mx


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_fp8_backward_matches_bf16_mma_backward(shape):
    a, b, inp, fwd, bwd, mx = _step_pair(shape, 11)
    for name in ("dx", "dw_gate", "dw_up", "dw_down", "d_topk_w"):
        ref = getattr(b.grads, name).float().cpu().numpy()
        e = max_rel(getattr(a.grads, name), ref)
        assert e <= SAME_PRODUCTS_TOL, (name, e)
    # bitwise reproducible
    saved = {n: getattr(a.grads, n).clone() for n in ("dx", "dw_gate", "dw_up", "dw_down")}
    a.step(inp["x"], inp["logits"], inp["bias"], *fwd, inp["dy"], bwd=bwd, mx=mx)
    torch.cuda.synchronize()
    for n, t in saved.items():
        assert torch.equal(getattr(a.grads, n), t), n


def test_fp8_path_matches_bf16_mma_path_at_full_size():
    """The skewed MXFP8 workload at full size (N=16384, H=4096, I=1536, E=128,
    top-8): every output of the FP8 tensor-core pass against the same pass on
    bf16 MMAs of the same MXFP8 values."""
    torch.cuda.empty_cache()
    a, b, *_ = _step_pair(inputs.SKEWED_MXFP8, 0)
    e = max_rel(a.y, b.y.float().cpu().numpy())
    assert e <= SAME_PRODUCTS_TOL, ("y", e)
    for name in ("dx", "dw_gate", "dw_up", "dw_down", "d_topk_w"):
        ref = getattr(b.grads, name).float().cpu().numpy()
        e = max_rel(getattr(a.grads, name), ref)
        assert e <= SAME_PRODUCTS_TOL, (name, e)
    del a, b
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T", [512, 1024])
def test_fp8_layer_large_minibatch_rows(T):
    """Expert segments padded to 512 / 1024 rows (many all-padding tiles)."""
    shape = custom_shape(300, 512, 768, 16, 4, zipf_s=1.2, name=f"T{T}_mxfp8", T=T).with_(
        dtype="mxfp8")
    a, b, *_ = _step_pair(shape, 13)
    for name in ("dx", "dw_gate", "dw_up", "dw_down"):
        ref = getattr(b.grads, name).float().cpu().numpy()
        assert max_rel(getattr(a.grads, name), ref) <= SAME_PRODUCTS_TOL, name


def test_fp8_layer_empty_batch():
    """N = 0: nothing routed; every weight gradient is zero, nothing faults."""
    shape = custom_shape(0, 512, 512, 8, 2, name="empty_mxfp8").with_(dtype="mxfp8")
    inp = to_dev(inputs.make_inputs(custom_shape(8, 512, 512, 8, 2), seed=1, device="cpu"))
    empty = {k: (v[:0] if k in ("x", "logits", "dy") else v) for k, v in inp.items()}
    fwd, bwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    layer = _layer(shape)
    layer.grads.dw_gate.fill_(1.0)
    layer.step(empty["x"], empty["logits"], empty["bias"], *fwd, empty["dy"], bwd=bwd, mx=mx)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.all(layer.grads.dw_gate == 0) and torch.all(layer.grads.dw_down == 0)


def _decode_rows(q_ptr, s_ptr, rows, k):
    """Values [rows, k] of a row-form MXFP8 operand in device memory."""
    q = torch.as_tensor(_DevBytes(q_ptr, rows * k), device=dev()).cpu().numpy().reshape(rows, k)
    s = torch.as_tensor(_DevBytes(s_ptr, rows * k // 32), device=dev()).cpu().numpy()
    table = np.array([oracle.e4m3_decode(c) for c in range(256)])
    scale = 2.0 ** (untile_scales(s, rows, k).astype(np.float64) - 127)
    return table[q] * np.repeat(scale, 32, axis=1)


def test_fp8_error_budget_at_the_tiny_shape():
    """Where the MXFP8 error against the oracle comes from, on the tiny
    workload (seed 0, as in smoke): the GPU forms dG and dU from the G and U it
    saved in bf16, the oracle from fp64 G and U; the two sides can then round
    a dG or dU value to a neighbouring bf16 value and quantise it to a
    neighbouring E4M3 code (or, through the block maximum, another scale).
    The oracle's diagnostic switch that reads G and U as bf16 values (never
    a parity reference) shows how much of the dx / dWg / dWu error that
    explains: the GPU's quantised dG/dU rows (read back from the workspace)
    disagree with it in far fewer codes, and the errors shrink."""
    shape = SHAPES[0]
    inp_cpu = inputs.make_inputs(shape, seed=0, device="cpu")
    inp = to_dev(inp_cpu)
    fwd, bwd = MoELayer.prepare_mxfp8_weights(inp["wg"], inp["wu"], inp["wd"])
    mx = MoELayer.prepare_mxfp8_mma_weights(inp["wg"], inp["wu"], inp["wd"])
    layer = _layer(shape)
    layer.step(inp["x"], inp["logits"], inp["bias"], *fwd, inp["dy"], bwd=bwd, mx=mx)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    ids, w = oracle.route_topk(inp_cpu["logits"].numpy(), None, shape.k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids)
    prep = oracle.mxfp8_weights(inp_cpu["wg"], inp_cpu["wu"], inp_cpu["wd"])
    ref = {gb: oracle.layer_mxfp8_trace(inp_cpu["x"], prep, ids, w, inp_cpu["dy"], gu_bf16=gb)
           for gb in (False, True)}
    slot = layer.schedule_tensors()["slot_of"].cpu().numpy().reshape(-1)
    ops = _lib.moe_mxfp8_backward_operands(layer.p, layer.ws)
    (gq, gs), (uq, us) = ops["dg_rows"], ops["du_rows"]
    got_rows = {"dg": _decode_rows(gq, gs, layer.R, shape.I)[slot],
                "du": _decode_rows(uq, us, layer.R, shape.I)[slot]}
    g = layer.grads
    report = {}
    for gb, r in ref.items():
        key = "oracle_bf16_gu" if gb else "oracle"
        report[key] = {
            "dg_code_mismatch": float(np.mean(got_rows["dg"] != r["dg_rows"])),
            "du_code_mismatch": float(np.mean(got_rows["du"] != r["du_rows"])),
            **{n: max_rel(t, r[k]) for n, t, k in (("dx", g.dx, "dx"), ("dw_gate", g.dw_gate, "dwg"),
                                                    ("dw_up", g.dw_up, "dwu"),
                                                    ("dw_down", g.dw_down, "dwd"))}}
    print("error budget", report)
    # measured on a GB300 (seed 0): against the fp64 reference 4.3% / 1.5% of
    # the dG / dU codes differ and dWg is off by 4.7e-2, dx by 3.7e-2; against
    # the diagnostic one code in 262144 differs, dWg is off by 8e-6, dWu by
    # 6e-4, dx by 4e-3. The checks keep a margin above those figures.
    a, b = report["oracle"], report["oracle_bf16_gu"]
    for n in ("dx", "dw_gate", "dw_up", "dw_down"):
        assert a[n] <= MX_TOL, n
    assert b["dg_code_mismatch"] <= 1e-4 and b["du_code_mismatch"] <= 1e-4
    assert b["dw_gate"] <= 5e-3 and b["dw_up"] <= 5e-3 and b["dx"] <= 1.5e-2
    assert b["dw_gate"] < a["dw_gate"] / 5 and b["dx"] < a["dx"] / 5
