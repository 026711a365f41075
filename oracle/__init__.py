"""fp64 CPU oracle of the top-k SwiGLU mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
(the CUDA library and its Python binding) never does. It shares no code with
the CUDA path: it is a plain C++ library (``moe_oracle.cpp``) loaded with
ctypes, plus the numpy marshalling below.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` and
``tests/test_golden.py`` (brute force, closed forms, finite differences,
library routines, code points fixed by the OCP MXFP8 specifications, a flush
pin for every MXFP8 quantisation point, and bit-exact agreement of the
sampled functions with the whole-layer ones); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_ERR_ARG, ORC_ERR_NAN = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (no CUDA involved)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                               os.path.getmtime(os.path.join(_HERE, "moe_oracle.h")))):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([
            "g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
            "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            L.orc_route_topk.argtypes = [i64, i32, i32, vp, vp, vp, vp]
            L.orc_build_schedule.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, vp,
                                             vp, i64, vp, i64, vp]
            L.orc_build_schedule_padded.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp,
                                                    vp, vp, i64, vp, i64, vp]
            fw = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
            L.orc_forward_f64.argtypes = fw
            L.orc_forward_bf16.argtypes = fw
            bw = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                  ctypes.c_int]
            L.orc_backward_f64.argtypes = bw
            L.orc_backward_bf16.argtypes = bw
            L.orc_tokens_bf16.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                          vp, i64, vp, vp, vp, vp, ctypes.c_int]
            L.orc_expert_wgrad_bf16.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp,
                                                vp, vp, vp, i32, i64, vp, i64, vp, vp, vp,
                                                vp, ctypes.c_int]
            L.orc_expert_wgrad_mxfp8.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                                 vp, vp, i32, i64, vp, i64, vp, ctypes.c_int,
                                                 vp, vp, vp, ctypes.c_int]
            L.orc_mxfp8_quantize.argtypes = [i64, i64, vp, vp, vp]
            L.orc_layer_mxfp8.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp,
                                          ctypes.c_int, vp, vp, vp, vp, vp, vp, ctypes.c_int]
            L.orc_mxfp8_weights.argtypes = [i32, i32, i32, vp, vp, vp, ctypes.c_int, vp, vp, vp,
                                            vp, vp, vp, ctypes.c_int]
            L.orc_layer_mxfp8_prepared.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                                   vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp,
                                                   vp, vp, vp, ctypes.c_int]
            L.orc_layer_mxfp8_trace.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                                vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                                vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int]
            L.orc_router_logits.argtypes = [i64, i32, i32, vp, vp, vp, ctypes.c_int]
            L.orc_router_backward.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                              ctypes.c_int]
            L.orc_e4m3_encode.argtypes = [ctypes.c_double]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_decode.restype = ctypes.c_double
            _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc):
    if rc != ORC_OK:
        raise OracleError({ORC_ERR_ARG: "invalid argument", ORC_ERR_NAN: "NaN logit"}.get(rc, rc))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def as_bf16_bits(a) -> np.ndarray:
    """Accept a uint16 bit-pattern array or a torch bf16 tensor."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # torch is only a container here
    assert a.dtype == torch.bfloat16
    return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def route_topk(logits, bias, k):
    logits = _c(logits, np.float32)
    N, E = logits.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((N, k), np.int32)
    w = np.empty((N, k), np.float64)
    _check(lib().orc_route_topk(N, E, k, _p(logits), _p(b), _p(ids), _p(w)))
    return ids, w


def router_logits(x, wr, threads=0):
    """logits = x . Wr^T in fp64 (x bf16 [N, H], Wr bf16 [E, H])."""
    x, wr = as_bf16_bits(x), as_bf16_bits(wr)
    N, H = x.shape
    E = wr.shape[0]
    out = np.empty((N, E))
    _check(lib().orc_router_logits(N, H, E, _p(x), _p(wr), _p(out), threads))
    return out


def router_backward(x, wr, ids, w, dw, threads=0):
    """dz [N, k], dWr [E, H], router share of dx [N, H] (fp64; routing held fixed)."""
    x, wr = as_bf16_bits(x), as_bf16_bits(wr)
    ids, w, dw = _c(ids, np.int32), _c(w, np.float64), _c(dw, np.float64)
    N, H = x.shape
    E = wr.shape[0]
    k = ids.shape[1]
    dz = np.empty((N, k))
    dwr = np.empty((E, H))
    dx = np.empty((N, H))
    _check(lib().orc_router_backward(N, H, E, k, _p(x), _p(wr), _p(ids), _p(w), _p(dw), _p(dz),
                                     _p(dwr), _p(dx), threads))
    return dict(dz=dz, dwr=dwr, dx=dx)


def build_schedule(ids, E, tile_m=128, pad_m=None):
    """Schedule tables; expert segments padded to pad_m (default tile_m) rows."""
    pad_m = tile_m if pad_m is None else pad_m
    ids = _c(ids, np.int32)
    N, k = ids.shape
    A = N * k
    rows_cap = A + E * (pad_m - 1)
    tiles_cap = rows_cap // tile_m + 1
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    pad_offsets = np.empty(E + 1, np.int32)
    slot_of = np.empty(A, np.int32)
    src_of_row = np.empty(rows_cap, np.int32)
    tiles = np.empty((tiles_cap, 3), np.int32)
    n_tiles = np.zeros(1, np.int32)
    _check(lib().orc_build_schedule_padded(N, k, E, tile_m, pad_m, _p(ids), _p(counts),
                                           _p(offsets), _p(pad_offsets), _p(slot_of),
                                           _p(src_of_row), rows_cap, _p(tiles), tiles_cap,
                                           _p(n_tiles)))
    rows = int(pad_offsets[E])
    nt = int(n_tiles[0])
    return dict(counts=counts, offsets=offsets, pad_offsets=pad_offsets,
                slot_of=slot_of.reshape(N, k), src_of_row=src_of_row[:rows].copy(),
                tiles=tiles[:nt].copy(), n_tiles=nt)


def forward_f64(x, wg, wu, wd, ids, w, threads=0, want_ye=False):
    x, wg, wu, wd = (_c(a, np.float64) for a in (x, wg, wu, wd))
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    N, H = x.shape
    E, I, _ = wg.shape
    k = ids.shape[1]
    y = np.empty((N, H), np.float64)
    ye = np.empty((N * k, H), np.float64) if want_ye else None
    _check(lib().orc_forward_f64(N, H, I, E, k, _p(x), _p(wg), _p(wu), _p(wd), _p(ids),
                                 _p(w), _p(y), _p(ye), threads))
    return (y, ye) if want_ye else y


def forward_bf16(x, wg, wu, wd, ids, w, threads=0, want_ye=False):
    x, wg, wu, wd = (as_bf16_bits(a) for a in (x, wg, wu, wd))
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    N, H = x.shape
    E, I, _ = wg.shape
    k = ids.shape[1]
    y = np.empty((N, H), np.float64)
    ye = np.empty((N * k, H), np.float64) if want_ye else None
    _check(lib().orc_forward_bf16(N, H, I, E, k, _p(x), _p(wg), _p(wu), _p(wd), _p(ids),
                                  _p(w), _p(y), _p(ye), threads))
    return (y, ye) if want_ye else y


def _bw_out(N, H, I, E, k):
    return (np.empty((N, H)), np.empty((E, I, H)), np.empty((E, I, H)), np.empty((E, H, I)),
            np.empty((N, k)))


def backward_f64(x, wg, wu, wd, ids, w, dy, threads=0):
    x, wg, wu, wd, dy = (_c(a, np.float64) for a in (x, wg, wu, wd, dy))
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    N, H = x.shape
    E, I, _ = wg.shape
    k = ids.shape[1]
    dx, dwg, dwu, dwd, dw = _bw_out(N, H, I, E, k)
    _check(lib().orc_backward_f64(N, H, I, E, k, _p(x), _p(wg), _p(wu), _p(wd), _p(ids),
                                  _p(w), _p(dy), _p(dx), _p(dwg), _p(dwu), _p(dwd), _p(dw),
                                  threads))
    return dict(dx=dx, dwg=dwg, dwu=dwu, dwd=dwd, dw=dw)


def backward_bf16(x, wg, wu, wd, ids, w, dy, threads=0):
    x, wg, wu, wd, dy = (as_bf16_bits(a) for a in (x, wg, wu, wd, dy))
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    N, H = x.shape
    E, I, _ = wg.shape
    k = ids.shape[1]
    dx, dwg, dwu, dwd, dw = _bw_out(N, H, I, E, k)
    _check(lib().orc_backward_bf16(N, H, I, E, k, _p(x), _p(wg), _p(wu), _p(wd), _p(ids),
                                   _p(w), _p(dy), _p(dx), _p(dwg), _p(dwu), _p(dwd), _p(dw),
                                   threads))
    return dict(dx=dx, dwg=dwg, dwu=dwu, dwd=dwd, dw=dw)


def tokens_bf16(x, wg, wu, wd, ids, w, dy, tokens, threads=0):
    """y, dx, dw of the listed tokens only (sampled parity at full size)."""
    x, wg, wu, wd, dy = (as_bf16_bits(a) for a in (x, wg, wu, wd, dy))
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    tok = _c(tokens, np.int64)
    N, H = x.shape
    E, I, _ = wg.shape
    k = ids.shape[1]
    n = tok.shape[0]
    y, dx, dw = np.empty((n, H)), np.empty((n, H)), np.empty((n, k))
    _check(lib().orc_tokens_bf16(N, H, I, E, k, _p(x), _p(wg), _p(wu), _p(wd), _p(ids),
                                 _p(w), _p(dy), n, _p(tok), _p(y), _p(dx), _p(dw), threads))
    return dict(y=y, dx=dx, dw=dw)


def expert_wgrad_bf16(x, wg, wu, wd, ids, w, dy, e, i_list, h_list, threads=0):
    """Rows i_list of dWg[e], dWu[e] and rows h_list of dWd[e]."""
    x, wg, wu, wd, dy = (as_bf16_bits(a) for a in (x, wg, wu, wd, dy))
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    il, hl = _c(i_list, np.int32), _c(h_list, np.int32)
    N, H = x.shape
    E, I, _ = wg.shape
    k = ids.shape[1]
    dwg, dwu, dwd = np.empty((len(il), H)), np.empty((len(il), H)), np.empty((len(hl), I))
    _check(lib().orc_expert_wgrad_bf16(N, H, I, E, k, _p(x), _p(wg), _p(wu), _p(wd), _p(ids),
                                       _p(w), _p(dy), int(e), len(il), _p(il), len(hl), _p(hl),
                                       _p(dwg), _p(dwu), _p(dwd), threads))
    return dict(dwg=dwg, dwu=dwu, dwd=dwd)


def layer_mxfp8(x, wg, wu, wd, ids, w, dy, quantize=True, threads=0):
    """MXFP8 layer forward + backward (quantised GEMM operands, fp64 sums)."""
    x, wg, wu, wd, dy = (as_bf16_bits(a) for a in (x, wg, wu, wd, dy))
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    N, H = x.shape
    E, I, _ = wg.shape
    k = ids.shape[1]
    y = np.empty((N, H))
    dx, dwg, dwu, dwd, dw = _bw_out(N, H, I, E, k)
    _check(lib().orc_layer_mxfp8(N, H, I, E, k, _p(x), _p(wg), _p(wu), _p(wd), _p(ids), _p(w),
                                 _p(dy), 1 if quantize else 0, _p(y), _p(dx), _p(dwg), _p(dwu),
                                 _p(dwd), _p(dw), threads))
    return dict(y=y, dx=dx, dwg=dwg, dwu=dwu, dwd=dwd, dw=dw)


def expert_wgrad_mxfp8(x, wg, wu, wd, ids, w, dy, e, i_list, h_list, quantize=True, threads=0):
    """Entries of expert e's MXFP8 weight gradients (those of layer_mxfp8):
    dwg, dwu [len(i_list), len(h_list)] and dwd [len(h_list), len(i_list)]."""
    x, wg, wu, wd, dy = (as_bf16_bits(a) for a in (x, wg, wu, wd, dy))
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    il, hl = _c(i_list, np.int32), _c(h_list, np.int32)
    N, H = x.shape
    E, I, _ = wg.shape
    k = ids.shape[1]
    dwg, dwu = np.empty((len(il), len(hl))), np.empty((len(il), len(hl)))
    dwd = np.empty((len(hl), len(il)))
    _check(lib().orc_expert_wgrad_mxfp8(N, H, I, E, k, _p(x), _p(wg), _p(wu), _p(wd), _p(ids),
                                        _p(w), _p(dy), int(e), len(il), _p(il), len(hl), _p(hl),
                                        1 if quantize else 0, _p(dwg), _p(dwu), _p(dwd), threads))
    return dict(dwg=dwg, dwu=dwu, dwd=dwd)


MXFP8_WEIGHT_COPIES = ("wg_h", "wu_h", "wd_i", "wd_h", "wg_i", "wu_i")


def mxfp8_weights(wg, wu, wd, quantize=True, threads=0):
    """The six quantised weight copies the MXFP8 layer reads (see
    orc_mxfp8_weights), as a dict of fp64 arrays."""
    wg, wu, wd = (as_bf16_bits(a) for a in (wg, wu, wd))
    E, I, H = wg.shape
    out = {n: np.empty(wg.shape if n[1] != "d" else wd.shape) for n in MXFP8_WEIGHT_COPIES}
    _check(lib().orc_mxfp8_weights(H, I, E, _p(wg), _p(wu), _p(wd), 1 if quantize else 0,
                                   *(_p(out[n]) for n in MXFP8_WEIGHT_COPIES), threads))
    return out


def layer_mxfp8_prepared(x, prepared, ids, w, dy, quantize=True, threads=0):
    """layer_mxfp8 on weights from mxfp8_weights (same quantize flag)."""
    x, dy = as_bf16_bits(x), as_bf16_bits(dy)
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    N, H = x.shape
    E, I, _ = prepared["wg_h"].shape
    k = ids.shape[1]
    y = np.empty((N, H))
    dx, dwg, dwu, dwd, dw = _bw_out(N, H, I, E, k)
    _check(lib().orc_layer_mxfp8_prepared(
        N, H, I, E, k, _p(x), *(_p(prepared[n]) for n in MXFP8_WEIGHT_COPIES), _p(ids), _p(w),
        _p(dy), 1 if quantize else 0, _p(y), _p(dx), _p(dwg), _p(dwu), _p(dwd), _p(dw), threads))
    return dict(y=y, dx=dx, dwg=dwg, dwu=dwu, dwd=dwd, dw=dw)


def layer_mxfp8_trace(x, prepared, ids, w, dy, gu_bf16=False, threads=0):
    """layer_mxfp8_prepared (quantisation on) plus the quantised dG and dU rows
    [N*k, I] the gate/up data gradient reads; gu_bf16 rounds G and U to bf16
    before the SwiGLU backward (an error-accounting diagnostic, not a parity
    reference)."""
    x, dy = as_bf16_bits(x), as_bf16_bits(dy)
    ids, w = _c(ids, np.int32), _c(w, np.float64)
    N, H = x.shape
    E, I, _ = prepared["wg_h"].shape
    k = ids.shape[1]
    y = np.empty((N, H))
    dx, dwg, dwu, dwd, dw = _bw_out(N, H, I, E, k)
    dg_rows, du_rows = np.empty((N * k, I)), np.empty((N * k, I))
    _check(lib().orc_layer_mxfp8_trace(
        N, H, I, E, k, _p(x), *(_p(prepared[n]) for n in MXFP8_WEIGHT_COPIES), _p(ids), _p(w),
        _p(dy), 1, 1 if gu_bf16 else 0, _p(y), _p(dx), _p(dwg), _p(dwu), _p(dwd), _p(dw),
        _p(dg_rows), _p(du_rows), threads))
    return dict(y=y, dx=dx, dwg=dwg, dwu=dwu, dwd=dwd, dw=dw, dg_rows=dg_rows, du_rows=du_rows)


def mxfp8_quantize(src_bits):
    src = as_bf16_bits(src_bits)
    rows, cols = src.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // 32), np.uint8)
    _check(lib().orc_mxfp8_quantize(rows, cols, _p(src), _p(q), _p(s)))
    return q, s


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(int(code)))
