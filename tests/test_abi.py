"""The C-ABI library loads and exports every entry point include/moe.h
declares; host-only entry points (sizes, validation) behave as documented.
No compute call is made, so this runs without a GPU."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_schedule_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_binding_names():
    declared = _header_functions()
    assert "moe_forward" in declared and "mxfp8_quantize" in declared
    assert sorted(declared) == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name


def test_sizes_and_validation(lib):
    p = _lib.problem(256, 256, 512, 8, 2)
    assert _lib.moe_grouped_rows(p) == ((512 + 8 * 127 + 127) // 128) * 128
    ws = _lib.moe_workspace_bytes(p)
    sv = _lib.moe_saved_bytes(p)
    R = _lib.moe_grouped_rows(p)
    assert sv >= R * (2 * 256 + 3 * 512) * 2 and sv % 256 == 0
    assert ws >= R * (256 + 2 * 512) * 2
    for bad, status in (((256, 200, 512, 8, 2), _lib.MOE_ERR_UNSUPPORTED),
                        ((256, 256, 512, 8, 9), _lib.MOE_ERR_INVALID_ARG),
                        ((256, 256, 512, 2048, 2), _lib.MOE_ERR_UNSUPPORTED),
                        ((-1, 256, 512, 8, 2), _lib.MOE_ERR_INVALID_ARG),
                        # int32 rows on the device: N * k (+ padding) must fit
                        ((2 ** 62, 256, 512, 8, 8), _lib.MOE_ERR_UNSUPPORTED),
                        ((2 ** 28, 256, 512, 8, 8), _lib.MOE_ERR_UNSUPPORTED),
                        # N * k = 2^31 - 512 fits, but not with E * (T - 1) padding rows
                        ((2 ** 28 - 64, 256, 512, 8, 8), _lib.MOE_ERR_UNSUPPORTED)):
        with pytest.raises(_lib.MoEError) as ei:
            _lib.moe_workspace_bytes(_lib.problem(*bad))
        assert ei.value.status == status
    # the largest sizes below the bound are accepted (host-side sizing only)
    assert _lib.moe_workspace_bytes(_lib.problem(2 ** 28 - 2 ** 16, 256, 512, 8, 8)) > 0
    for bad_kw in (dict(dtype=7), dict(minibatch_rows=192), dict(minibatch_rows=2048),
                   dict(pipeline_stages=3), dict(pipeline_stages=7), dict(pipeline_stages=-1),
                   dict(tile_n=128), dict(tile_n=1024)):
        with pytest.raises(_lib.MoEError) as ei:
            _lib.moe_workspace_bytes(_lib.problem(256, 256, 512, 8, 2, **bad_kw))
        assert ei.value.status == _lib.MOE_ERR_UNSUPPORTED
    for good in (4, 5, 6):  # the ring depths the GEMMs are built for; sizes do not change
        assert _lib.moe_workspace_bytes(_lib.problem(256, 256, 512, 8, 2, pipeline_stages=good)) == ws
    for good in (256, 512):
        assert _lib.moe_workspace_bytes(_lib.problem(256, 256, 512, 8, 2, tile_n=good)) == ws
    # MXFP8 adds the quantised-operand buffers; T = 256 grows the padded rows
    mx = _lib.moe_workspace_bytes(_lib.problem(256, 256, 512, 8, 2, dtype=_lib.MOE_MXFP8))
    assert mx > ws + R * (2 * 256 + 4 * 512) * 2 - 4096
    assert _lib.moe_grouped_rows(_lib.problem(256, 256, 512, 8, 2, minibatch_rows=256)) == \
        ((512 + 8 * 255 + 255) // 256) * 256


def test_null_and_misaligned_pointers_are_rejected_before_any_launch(lib):
    p = _lib.problem(64, 256, 256, 4, 2)
    st = lib.moe_build_schedule(ctypes.byref(p), None, None, None)
    assert st == _lib.MOE_ERR_INVALID_ARG
    st = lib.moe_dispatch(ctypes.byref(p), 256, 16, 0, None)  # xe NULL
    assert st == _lib.MOE_ERR_INVALID_ARG
    st = lib.moe_dispatch(ctypes.byref(p), 256 + 8, 16, 16, None)  # ws misaligned
    assert st == _lib.MOE_ERR_INVALID_ARG
    st = lib.mxfp8_quantize(16, 4, 48, 16, 16, None)  # cols not a multiple of 32
    assert st == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_status_string(_lib.MOE_ERR_CUDA) == b"CUDA runtime or driver error"


def test_binding_rejects_host_and_strided_tensors_before_the_library():
    """A host tensor would hand the kernels a host address (a GPU fault, not an
    error status), and a strided view the wrong layout: the binding raises on
    both before any library call."""
    torch = pytest.importorskip("torch")
    p = _lib.problem(64, 256, 256, 4, 2)
    host = torch.zeros(64, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        _lib.moe_dispatch(p, 256, host, 512)
    with pytest.raises(ValueError, match="contiguous"):
        _lib.moe_dispatch(p, 256, host.t(), 512)
    with pytest.raises(ValueError, match="contiguous"):
        _lib.mxfp8_quantize(host[:, ::2], 64, 128, 256, 512)
    assert _lib._ptr(None) is None and _lib._ptr(4096) == 4096


@pytest.mark.parametrize("N,H,I,E,k,dtype,T", [(256, 256, 512, 8, 2, 0, 128),
                                               (300, 512, 768, 16, 4, 1, 256),
                                               (16384, 4096, 1536, 128, 8, 1, 128),
                                               (0, 256, 256, 4, 2, 0, 1024)])
def test_workspace_and_context_regions_are_disjoint_and_aligned(lib, N, H, I, E, k, dtype, T):
    """The host-side carving of the workspace (schedule tables) and of the
    saved context (Xe, G, U, Act, Ye): every region 256-byte aligned, inside
    its buffer and disjoint from the others, at the documented sizes. Pure
    address arithmetic on a fake base address; nothing is launched."""
    p = _lib.problem(N, H, I, E, k, dtype=dtype, minibatch_rows=T)
    R = _lib.moe_grouped_rows(p)
    base = 1 << 40
    ws_bytes, sv_bytes = _lib.moe_workspace_bytes(p), _lib.moe_saved_bytes(p)

    def check(regions, total):
        spans = sorted((addr - base, n, name) for name, addr, n in regions)
        for off, n, name in spans:
            assert off % 256 == 0 and 0 <= off and off + n <= total, name
        for (o1, n1, a), (o2, _, b) in zip(spans, spans[1:]):
            assert o1 + n1 <= o2, (a, b)

    sched = _lib.Schedule()
    assert lib.moe_schedule_view(ctypes.byref(p), base, ctypes.byref(sched)) == _lib.MOE_OK
    A = N * k
    regions = [("counts", sched.counts, 4 * E), ("offsets", sched.offsets, 4 * (E + 1)),
               ("pad_offsets", sched.pad_offsets, 4 * (E + 1)), ("slot_of", sched.slot_of, 4 * A),
               ("src_of_row", sched.src_of_row, 4 * R), ("tiles", sched.tiles, 12 * (R // 128)),
               ("n_tiles", sched.n_tiles, 4)]
    if dtype == _lib.MOE_MXFP8:  # the forward's row-form MXFP8 operands of Xe and Act
        (xq, xs), (aq, as_) = _lib.moe_mxfp8_forward_operands(p, base)
        fwd = [("xe_q", xq, R * H), ("xe_s", xs, R * H // 32), ("act_q", aq, R * I),
               ("act_s", as_, R * I // 32)]
        # the backward's dG / dU row operands (dG reuses Act's buffer after the
        # forward's last reader): checked beside the tables, apart from the forward's
        ops = _lib.moe_mxfp8_backward_operands(p, base)
        bwd = [("dg", ops["dg"], 2 * R * I), ("du", ops["du"], 2 * R * I)]
        for name in ("dg_rows", "du_rows", "dg_cols", "du_cols"):
            q, sc = ops[name]
            bwd += [(name + "_q", q, R * I), (name + "_s", sc, R * I // 32)]
        check(regions + bwd, ws_bytes)
        regions += fwd
    check(regions, ws_bytes)
    sv = _lib.SavedView()
    assert lib.moe_saved_layout(ctypes.byref(p), base, ctypes.byref(sv)) == _lib.MOE_OK
    check([("xe", sv.xe, 2 * R * H), ("g", sv.g, 2 * R * I), ("u", sv.u, 2 * R * I),
           ("act", sv.act, 2 * R * I), ("ye", sv.ye, 2 * R * H)], sv_bytes)
