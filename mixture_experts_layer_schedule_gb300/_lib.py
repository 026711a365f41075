"""ctypes binding of the C ABI in include/moe.h (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
tensors (device memory) and passes their data pointers plus the current CUDA
stream. All arithmetic happens in the CUDA library; if the library has not
been built this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(5)
MOE_DEVERR_NONE, MOE_DEVERR_BAD_EXPERT, MOE_DEVERR_NAN_LOGIT, MOE_DEVERR_TIMEOUT = range(4)
MOE_BF16, MOE_MXFP8 = 0, 1

c_i64, c_i32, c_vp, c_sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t


class Problem(ctypes.Structure):
    _fields_ = [("N", c_i64), ("H", c_i32), ("I", c_i32), ("E", c_i32), ("k", c_i32),
                ("dtype", c_i32), ("minibatch_rows", c_i32), ("pipeline_stages", c_i32),
                ("tile_n", c_i32)]


class MXFP8Operand(ctypes.Structure):
    _fields_ = [("q", c_vp), ("s", c_vp)]


MXFP8_WEIGHT_OPERANDS = ("gate", "up", "down", "gate_t", "up_t", "down_t")


class MXFP8Weights(ctypes.Structure):
    _fields_ = [(n, MXFP8Operand) for n in MXFP8_WEIGHT_OPERANDS]


class Weights(ctypes.Structure):
    _fields_ = [("w_gate", c_vp), ("w_up", c_vp), ("w_down", c_vp),
                ("w_gate_bwd", c_vp), ("w_up_bwd", c_vp), ("w_down_bwd", c_vp),
                ("mx", ctypes.POINTER(MXFP8Weights))]


class Schedule(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("counts", "offsets", "pad_offsets", "slot_of", "src_of_row",
                                    "tiles", "n_tiles")]


class SavedView(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("xe", "g", "u", "act", "ye")]


class MoEError(RuntimeError):
    def __init__(self, fn, status, lib):
        msg = lib.moe_status_string(status).decode() if lib is not None else str(status)
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None

_SIGS = {
    "moe_grouped_rows": ([c_vp], c_i64),
    "moe_workspace_bytes": ([c_vp, c_vp], c_i32),
    "moe_saved_bytes": ([c_vp, c_vp], c_i32),
    "moe_saved_layout": ([c_vp, c_vp, c_vp], c_i32),
    "moe_schedule_view": ([c_vp, c_vp, c_vp], c_i32),
    "moe_route_topk": ([c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp], c_i32),
    "moe_build_schedule": ([c_vp, c_vp, c_vp, c_vp], c_i32),
    "moe_route": ([c_vp] * 9, c_i32),
    "moe_router_backward": ([c_vp] * 10, c_i32),
    "moe_build_schedule_noalloc": ([c_vp, c_vp, c_vp, c_vp, c_vp], c_i32),
    "moe_dispatch": ([c_vp, c_vp, c_vp, c_vp, c_vp], c_i32),
    "moe_expert_gate_up": ([c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp], c_i32),
    "moe_expert_down": ([c_vp, c_vp, c_vp, c_vp, c_vp, c_vp], c_i32),
    "moe_combine": ([c_vp, c_vp, c_vp, c_vp, c_vp, c_vp], c_i32),
    "moe_forward": ([c_vp] * 8, c_i32),
    "moe_forward_inference": ([c_vp] * 7, c_i32),
    "moe_reverse_combine": ([c_vp] * 8, c_i32),
    "moe_expert_down_dgrad": ([c_vp] * 9, c_i32),
    "moe_expert_down_wgrad": ([c_vp] * 6, c_i32),
    "moe_expert_gate_up_dgrad": ([c_vp] * 7, c_i32),
    "moe_expert_gate_up_wgrad": ([c_vp] * 8, c_i32),
    "moe_reverse_dispatch": ([c_vp] * 5, c_i32),
    "moe_backward": ([c_vp] * 12, c_i32),
    "moe_mxfp8_forward_operands": ([c_vp] * 4, c_i32),
    "moe_mxfp8_backward_operands": ([c_vp] * 8, c_i32),
    "moe_dispatch_expert_ffn": ([c_vp] * 10, c_i32),
    "moe_dispatch_mxfp8": ([c_vp] * 7, c_i32),
    "moe_backward_overlap": ([c_vp] * 12, c_i32),
    "mxfp8_quantize": ([c_vp, c_i64, c_i64, c_vp, c_vp, c_vp], c_i32),
    "mxfp8_qdq": ([c_vp, c_vp, c_i64, c_i64, c_i32, c_vp], c_i32),
    "mxfp8_quantize_mma": ([c_vp, c_i64, c_i64, c_i32, c_vp, c_vp, c_vp], c_i32),
    "moe_get_device_error": ([c_vp, c_vp, c_vp, c_vp], c_i32),
    "moe_clear_device_error": ([c_vp, c_vp, c_vp], c_i32),
    "moe_status_string": ([c_i32], ctypes.c_char_p),
    "moe_test_wait_timeout": ([c_vp, c_vp, c_vp], c_i32),
    "moe_launch_count": ([], ctypes.c_uint64),
}

EXPORTED = tuple(_SIGS)


def load(path: str = LIB_PATH):
    """Load the CUDA library. Raises if it is missing (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def _check(name, status):
    if status != MOE_OK:
        raise MoEError(name, status, _lib)


def _ptr(t):
    """Device address of a tensor argument (None -> NULL; an int is taken as a
    raw address). The kernels read and write dense row-major device buffers,
    so a strided view or a host tensor raises here, before the library sees
    it: a host address would fault on the GPU instead of failing cleanly."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got strides {tuple(t.stride())} "
                         f"for shape {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"expected a CUDA tensor, got one on {t.device}")
    return t.data_ptr()


def _host_ptr(t):
    """Address of a pinned host tensor (the library's host-side outputs)."""
    if not t.is_pinned():
        raise ValueError("expected a pinned host tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return stream


def problem(N, H, I, E, k, dtype=MOE_BF16, minibatch_rows=128, pipeline_stages=0,
            tile_n=0) -> Problem:
    return Problem(int(N), int(H), int(I), int(E), int(k), int(dtype), int(minibatch_rows),
                   int(pipeline_stages), int(tile_n))


def mxfp8_weights(operands: dict) -> MXFP8Weights:
    """operands: name -> (q, s) tensors (names of MXFP8_WEIGHT_OPERANDS; missing ones NULL)."""
    st = MXFP8Weights()
    for n in MXFP8_WEIGHT_OPERANDS:
        q, sc = operands.get(n, (None, None))
        setattr(st, n, MXFP8Operand(_ptr(q), _ptr(sc)))
    return st


def weights(wg, wu, wd, wg_bwd=None, wu_bwd=None, wd_bwd=None, mx: MXFP8Weights = None) -> Weights:
    w = Weights(_ptr(wg), _ptr(wu), _ptr(wd), _ptr(wg_bwd), _ptr(wu_bwd), _ptr(wd_bwd),
                ctypes.pointer(mx) if mx is not None else None)
    w._keep = mx  # the pointed-to struct lives as long as this one
    return w


def _call(name, *args):
    _check(name, getattr(load(), name)(*args))


# ---- sizes and views -----------------------------------------------------

def moe_grouped_rows(p: Problem) -> int:
    r = load().moe_grouped_rows(ctypes.byref(p))
    if r < 0:
        raise MoEError("moe_grouped_rows", MOE_ERR_INVALID_ARG, _lib)
    return int(r)


def moe_workspace_bytes(p: Problem) -> int:
    out = c_sz(0)
    _call("moe_workspace_bytes", ctypes.byref(p), ctypes.byref(out))
    return out.value


def moe_saved_bytes(p: Problem) -> int:
    out = c_sz(0)
    _call("moe_saved_bytes", ctypes.byref(p), ctypes.byref(out))
    return out.value


def moe_saved_layout(p: Problem, saved) -> SavedView:
    v = SavedView()
    _call("moe_saved_layout", ctypes.byref(p), _ptr(saved), ctypes.byref(v))
    return v


def moe_schedule_view(p: Problem, ws) -> Schedule:
    v = Schedule()
    _call("moe_schedule_view", ctypes.byref(p), _ptr(ws), ctypes.byref(v))
    return v


# ---- layer entry points ----------------------------------------------------

def moe_route_topk(p, logits, bias, topk_ids, topk_w, ws, stream=None):
    _call("moe_route_topk", ctypes.byref(p), _ptr(logits), _ptr(bias), _ptr(topk_ids),
          _ptr(topk_w), _ptr(ws), _stream(stream))


def moe_build_schedule(p, topk_ids, ws, stream=None):
    _call("moe_build_schedule", ctypes.byref(p), _ptr(topk_ids), _ptr(ws), _stream(stream))


def moe_build_schedule_noalloc(p, topk_ids, out: Schedule, err_word, stream=None):
    """Schedule tables into the caller's arrays; scan scratch is a static device
    array inside the library (no allocation)."""
    _call("moe_build_schedule_noalloc", ctypes.byref(p), _ptr(topk_ids), ctypes.byref(out),
          _ptr(err_word), _stream(stream))


def moe_dispatch(p, ws, x, xe, stream=None):
    _call("moe_dispatch", ctypes.byref(p), _ptr(ws), _ptr(x), _ptr(xe), _stream(stream))


def moe_mxfp8_forward_operands(p, ws):
    """Device addresses (q, s) of Xe's and Act's row-form MXFP8 operands in ws."""
    xe, act = MXFP8Operand(), MXFP8Operand()
    _call("moe_mxfp8_forward_operands", ctypes.byref(p), _ptr(ws), ctypes.byref(xe),
          ctypes.byref(act))
    return (xe.q, xe.s), (act.q, act.s)


def moe_mxfp8_backward_operands(p, ws):
    """Device addresses in ws of what the MXFP8 tensor-core backward leaves for
    dG and dU: {"dg_rows", "du_rows", "dg_cols", "du_cols"} -> (q, s) of the
    row and transposed MXFP8 forms, {"dg", "du"} -> the bf16 [R, I] values."""
    ops = [MXFP8Operand() for _ in range(4)]
    dg, du = ctypes.c_void_p(), ctypes.c_void_p()
    _call("moe_mxfp8_backward_operands", ctypes.byref(p), _ptr(ws), *(ctypes.byref(o) for o in ops),
          ctypes.byref(dg), ctypes.byref(du))
    out = {k: (o.q, o.s) for k, o in zip(("dg_rows", "du_rows", "dg_cols", "du_cols"), ops)}
    out.update(dg=dg.value, du=du.value)
    return out


def moe_dispatch_expert_ffn(p, ws, x, w: Weights, xe, g, u, act, ye, stream=None):
    """Dispatch + gate/up + SwiGLU + down in one persistent launch."""
    _call("moe_dispatch_expert_ffn", ctypes.byref(p), _ptr(ws), _ptr(x), ctypes.byref(w), _ptr(xe),
          _ptr(g), _ptr(u), _ptr(act), _ptr(ye), _stream(stream))


def moe_dispatch_mxfp8(p, ws, x, xe, q, s, stream=None):
    _call("moe_dispatch_mxfp8", ctypes.byref(p), _ptr(ws), _ptr(x), _ptr(xe), _ptr(q), _ptr(s),
          _stream(stream))


def moe_expert_gate_up(p, ws, xe, w: Weights, g, u, act, stream=None):
    _call("moe_expert_gate_up", ctypes.byref(p), _ptr(ws), _ptr(xe), ctypes.byref(w), _ptr(g),
          _ptr(u), _ptr(act), _stream(stream))


def moe_expert_down(p, ws, act, w: Weights, ye, stream=None):
    _call("moe_expert_down", ctypes.byref(p), _ptr(ws), _ptr(act), ctypes.byref(w), _ptr(ye),
          _stream(stream))


def moe_combine(p, ws, ye, topk_w, y, stream=None):
    _call("moe_combine", ctypes.byref(p), _ptr(ws), _ptr(ye), _ptr(topk_w), _ptr(y),
          _stream(stream))


def moe_forward(p, x, w: Weights, topk_w, y, saved, ws, stream=None):
    _call("moe_forward", ctypes.byref(p), _ptr(x), ctypes.byref(w), _ptr(topk_w), _ptr(y),
          _ptr(saved), _ptr(ws), _stream(stream))


def moe_forward_inference(p, x, w: Weights, topk_w, y, ws, stream=None):
    _call("moe_forward_inference", ctypes.byref(p), _ptr(x), ctypes.byref(w), _ptr(topk_w),
          _ptr(y), _ptr(ws), _stream(stream))


def moe_reverse_combine(p, ws, dy, ye, topk_w, dye, d_topk_w, stream=None):
    _call("moe_reverse_combine", ctypes.byref(p), _ptr(ws), _ptr(dy), _ptr(ye), _ptr(topk_w),
          _ptr(dye), _ptr(d_topk_w), _stream(stream))


def moe_expert_down_dgrad(p, ws, dye, g, u, w: Weights, dg, du, stream=None):
    _call("moe_expert_down_dgrad", ctypes.byref(p), _ptr(ws), _ptr(dye), _ptr(g), _ptr(u),
          ctypes.byref(w), _ptr(dg), _ptr(du), _stream(stream))


def moe_expert_down_wgrad(p, ws, dye, act, dw_down, stream=None):
    _call("moe_expert_down_wgrad", ctypes.byref(p), _ptr(ws), _ptr(dye), _ptr(act),
          _ptr(dw_down), _stream(stream))


def moe_expert_gate_up_dgrad(p, ws, dg, du, w: Weights, dxe, stream=None):
    _call("moe_expert_gate_up_dgrad", ctypes.byref(p), _ptr(ws), _ptr(dg), _ptr(du),
          ctypes.byref(w), _ptr(dxe), _stream(stream))


def moe_expert_gate_up_wgrad(p, ws, dg, du, xe, dw_gate, dw_up, stream=None):
    _call("moe_expert_gate_up_wgrad", ctypes.byref(p), _ptr(ws), _ptr(dg), _ptr(du), _ptr(xe),
          _ptr(dw_gate), _ptr(dw_up), _stream(stream))


def moe_reverse_dispatch(p, ws, dxe, dx, stream=None):
    _call("moe_reverse_dispatch", ctypes.byref(p), _ptr(ws), _ptr(dxe), _ptr(dx),
          _stream(stream))


def moe_backward(p, saved, w: Weights, topk_w, dy, dx, dw_gate, dw_up, dw_down, d_topk_w, ws,
                 stream=None):
    _call("moe_backward", ctypes.byref(p), _ptr(saved), ctypes.byref(w), _ptr(topk_w), _ptr(dy),
          _ptr(dx), _ptr(dw_gate), _ptr(dw_up), _ptr(dw_down), _ptr(d_topk_w), _ptr(ws),
          _stream(stream))


def moe_backward_overlap(p, saved, w: Weights, topk_w, dy, dx, dw_gate, dw_up, dw_down, d_topk_w,
                         ws, stream=None):
    _call("moe_backward_overlap", ctypes.byref(p), _ptr(saved), ctypes.byref(w), _ptr(topk_w),
          _ptr(dy), _ptr(dx), _ptr(dw_gate), _ptr(dw_up), _ptr(dw_down), _ptr(d_topk_w), _ptr(ws),
          _stream(stream))


def moe_route(p, x, w_router, bias, logits, topk_ids, topk_w, ws, stream=None):
    _call("moe_route", ctypes.byref(p), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(logits),
          _ptr(topk_ids), _ptr(topk_w), _ptr(ws), _stream(stream))


def moe_router_backward(p, saved, w_router, topk_ids, topk_w, d_topk_w, dx, dw_router, ws,
                        stream=None):
    _call("moe_router_backward", ctypes.byref(p), _ptr(saved), _ptr(w_router), _ptr(topk_ids),
          _ptr(topk_w), _ptr(d_topk_w), _ptr(dx), _ptr(dw_router), _ptr(ws), _stream(stream))


def mxfp8_quantize(src, rows, cols, q, scale, stream=None):
    _call("mxfp8_quantize", _ptr(src), int(rows), int(cols), _ptr(q), _ptr(scale),
          _stream(stream))


def mxfp8_quantize_mma(src, rows, cols, transpose, q, s, stream=None):
    _call("mxfp8_quantize_mma", _ptr(src), int(rows), int(cols), int(transpose), _ptr(q), _ptr(s),
          _stream(stream))


def mxfp8_qdq(src, dst, rows, cols, axis, stream=None):
    _call("mxfp8_qdq", _ptr(src), _ptr(dst), int(rows), int(cols), int(axis), _stream(stream))


def moe_get_device_error(p, ws, stream=None) -> int:
    """Reads the device error word (synchronises the stream)."""
    out = torch.zeros(1, dtype=torch.int32, pin_memory=True)
    _call("moe_get_device_error", ctypes.byref(p), _ptr(ws), _host_ptr(out), _stream(stream))
    (torch.cuda.current_stream() if stream is None else stream).synchronize() \
        if not isinstance(stream, int) else torch.cuda.synchronize()
    return int(out.item())


def moe_test_wait_timeout(p, ws, stream=None):
    _call("moe_test_wait_timeout", ctypes.byref(p), _ptr(ws), _stream(stream))


def moe_launch_count() -> int:
    return int(load().moe_launch_count())


def moe_clear_device_error(p, ws, stream=None):
    _call("moe_clear_device_error", ctypes.byref(p), _ptr(ws), _stream(stream))
