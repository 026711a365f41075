"""Functional front end over the C ABI: workspace once per problem size,
schedule from the router's top-k experts, forward -> (y, context), backward
-> gradients. This mirrors the functional API described in the project
summary "Mixture-of-Kittens (MoK)" (section "use the functional API"). torch
only allocates device memory and supplies the stream; every step of the
layer runs in the CUDA library.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib


class MXFP8MMAWeights:
    """E4M3 codes + E8M0 scale chunks of the expert weights (tensors kept
    alive here) and the C struct that points at them."""

    def __init__(self, operands: dict):
        self.operands = operands
        self.struct = _lib.mxfp8_weights(operands)


@dataclass
class Grads:
    dx: torch.Tensor
    dw_gate: torch.Tensor
    dw_up: torch.Tensor
    dw_down: torch.Tensor
    d_topk_w: torch.Tensor


class MoELayer:
    """Buffers of one problem size on one device, reused across calls."""

    def __init__(self, N, H, I, E, k, device="cuda", allocate_grads=True, minibatch_rows=128,
                 dtype="bf16", pipeline_stages=0, tile_n=0):
        self.N, self.H, self.I, self.E, self.k = int(N), int(H), int(I), int(E), int(k)
        self.T = int(minibatch_rows)
        self.dtype = dtype
        self.device = torch.device(device)
        self.p = _lib.problem(N, H, I, E, k,
                              dtype=_lib.MOE_MXFP8 if dtype == "mxfp8" else _lib.MOE_BF16,
                              minibatch_rows=self.T, pipeline_stages=pipeline_stages,
                              tile_n=tile_n)
        self.R = _lib.moe_grouped_rows(self.p)
        dev = self.device
        self.ws = torch.empty(_lib.moe_workspace_bytes(self.p), dtype=torch.uint8, device=dev)
        self.saved = torch.empty(_lib.moe_saved_bytes(self.p), dtype=torch.uint8, device=dev)
        self.ws.zero_()  # clears the device error word
        self.topk_ids = torch.empty((N, k), dtype=torch.int32, device=dev)
        self.topk_w = torch.empty((N, k), dtype=torch.float32, device=dev)
        self.y = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        self.grads = None
        if allocate_grads:
            self.grads = Grads(
                dx=torch.empty((N, H), dtype=torch.bfloat16, device=dev),
                dw_gate=torch.empty((E, I, H), dtype=torch.float32, device=dev),
                dw_up=torch.empty((E, I, H), dtype=torch.float32, device=dev),
                dw_down=torch.empty((E, H, I), dtype=torch.float32, device=dev),
                d_topk_w=torch.empty((N, k), dtype=torch.float32, device=dev))

    # -- views -------------------------------------------------------------
    def saved_tensors(self) -> dict:
        v = _lib.moe_saved_layout(self.p, self.saved)
        base = self.saved.data_ptr()
        out = {}
        for name, cols in (("xe", self.H), ("g", self.I), ("u", self.I), ("act", self.I),
                           ("ye", self.H)):
            off = getattr(v, name) - base
            nbytes = self.R * cols * 2
            out[name] = self.saved[off:off + nbytes].view(torch.bfloat16).view(self.R, cols)
        return out

    def schedule_tensors(self) -> dict:
        s = _lib.moe_schedule_view(self.p, self.ws)
        base = self.ws.data_ptr()
        sizes = dict(counts=self.E, offsets=self.E + 1, pad_offsets=self.E + 1,
                     slot_of=self.N * self.k, src_of_row=self.R, tiles=3 * (self.R // 128),
                     n_tiles=1)
        out = {}
        for name, n in sizes.items():
            off = getattr(s, name) - base
            out[name] = self.ws[off:off + 4 * n].view(torch.int32)
        return out

    # -- steps -------------------------------------------------------------
    def route(self, logits, bias=None, stream=None):
        _lib.moe_route_topk(self.p, logits, bias, self.topk_ids, self.topk_w, self.ws, stream)
        return self.topk_ids, self.topk_w

    def route_from_x(self, x, w_router, bias=None, logits=None, stream=None):
        """Router GEMM (logits = x . w_router^T on the tensor cores) + top-k."""
        _lib.moe_route(self.p, x, w_router, bias, logits, self.topk_ids, self.topk_w, self.ws,
                       stream)
        return self.topk_ids, self.topk_w

    def router_backward(self, w_router, dw_router, stream=None):
        """Router share of dx (added to grads.dx) and dw_router [E, H] fp32; call
        after backward() of the same batch."""
        g = self.grads
        _lib.moe_router_backward(self.p, self.saved, w_router, self.topk_ids, self.topk_w,
                                 g.d_topk_w, g.dx, dw_router, self.ws, stream)
        return dw_router

    def build_schedule(self, topk_ids=None, stream=None):
        _lib.moe_build_schedule(self.p, self.topk_ids if topk_ids is None else topk_ids, self.ws,
                                stream)

    @staticmethod
    def prepare_mxfp8_weights(wg, wu, wd, stream=None):
        """MXFP8 weights as the GEMMs read them (exact bf16 values of the MXFP8
        numbers): forward -- gate/up along H, down along I; backward -- gate/up
        along I, down along H. Returns ((wg, wu, wd), (wg_bwd, wu_bwd, wd_bwd))."""
        E, I, H = wg.shape
        fwd, bwd = [], []
        for t, rows, cols in ((wg, E * I, H), (wu, E * I, H), (wd, E * H, I)):
            f = torch.empty_like(t)
            b = torch.empty_like(t)
            _lib.mxfp8_qdq(t, f, rows, cols, 0, stream)
            _lib.mxfp8_qdq(t, b, rows, cols, 1, stream)
            fwd.append(f)
            bwd.append(b)
        return tuple(fwd), tuple(bwd)

    @staticmethod
    def prepare_mxfp8_mma_weights(wg, wu, wd, stream=None, backward=True) -> "MXFP8MMAWeights":
        """MXFP8 weights for the block-scaled tensor-core GEMMs: E4M3 codes and
        E8M0 scale chunks of gate/up [E*I, H] and down [E*H, I] (forward) and,
        with backward, of their transposes [H, E*I] and [I, E*H] quantised
        along I and H (the K of the data-gradient GEMMs)."""
        E, I, H = wg.shape
        dev = wg.device
        ops = {}
        todo = [("gate", wg, E * I, H, 0), ("up", wu, E * I, H, 0), ("down", wd, E * H, I, 0)]
        if backward:
            todo += [("gate_t", wg, E * I, H, 1), ("up_t", wu, E * I, H, 1),
                     ("down_t", wd, E * H, I, 1)]
        for name, t, rows, cols, tr in todo:
            shape = (cols, rows) if tr else (rows, cols)
            q = torch.empty(shape, dtype=torch.uint8, device=dev)
            sc = torch.empty((rows * cols // 32,), dtype=torch.uint8, device=dev)
            _lib.mxfp8_quantize_mma(t, rows, cols, tr, q, sc, stream)
            ops[name] = (q, sc)
        return MXFP8MMAWeights(ops)

    def forward(self, x, wg, wu, wd, topk_w=None, stream=None, mx=None):
        """mx: MXFP8MMAWeights (MXFP8 layers): run the GEMMs on the FP8 tensor cores."""
        w = _lib.weights(wg, wu, wd, mx=mx.struct if mx is not None else None)
        _lib.moe_forward(self.p, x, w, self.topk_w if topk_w is None else topk_w, self.y,
                         self.saved, self.ws, stream)
        return self.y

    def forward_inference(self, x, wg, wu, wd, topk_w=None, stream=None, mx=None):
        """Forward without a saved context (inference): dispatch, gate/up
        storing Act only and down in one persistent launch (bf16: Xe and Act in
        a ring of 256-row minibatch slots in workspace scratch), then the
        combine; same y as forward()."""
        w = _lib.weights(wg, wu, wd, mx=mx.struct if mx is not None else None)
        _lib.moe_forward_inference(self.p, x, w, self.topk_w if topk_w is None else topk_w,
                                   self.y, self.ws, stream)
        return self.y

    def backward(self, dy, wg, wu, wd, topk_w=None, stream=None, bwd=None, mx=None,
                 overlap=False) -> Grads:
        """MXFP8: mx (MXFP8MMAWeights with the transposed copies) runs the GEMMs on
        the FP8 tensor cores; otherwise bwd (the backward-direction bf16 MXFP8
        values) feeds bf16 MMAs. overlap: the reverse-combine runs inside the
        down data-gradient GEMM (moe_backward_overlap; same results)."""
        g = self.grads
        w = _lib.weights(wg, wu, wd, *(bwd if bwd is not None else (None, None, None)),
                         mx=mx.struct if mx is not None else None)
        fn = _lib.moe_backward_overlap if overlap else _lib.moe_backward
        fn(self.p, self.saved, w, self.topk_w if topk_w is None else topk_w, dy, g.dx, g.dw_gate,
           g.dw_up, g.dw_down, g.d_topk_w, self.ws, stream)
        return g

    def step(self, x, logits, bias, wg, wu, wd, dy, stream=None, backward=True, bwd=None,
             mx=None, overlap=False):
        """Route, schedule, forward and (optionally) backward: one layer pass."""
        self.route(logits, bias, stream)
        self.build_schedule(None, stream)
        y = self.forward(x, wg, wu, wd, None, stream, mx=mx)
        if backward:
            self.backward(dy, wg, wu, wd, None, stream, bwd=bwd, mx=mx, overlap=overlap)
        return y

    def device_error(self, stream=None) -> int:
        return _lib.moe_get_device_error(self.p, self.ws, stream)

    def clear_device_error(self, stream=None):
        _lib.moe_clear_device_error(self.p, self.ws, stream)
