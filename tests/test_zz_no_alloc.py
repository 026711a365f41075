"""The allocation-free schedule entry point, moe_build_schedule_noalloc.

It exists for callers that cannot allocate device memory (for example a
plugin whose host application owns the device memory pool, or a loop that
must never call the allocator): its scan scratch is a static device array in
the library instead of a caller-provided workspace. The test calls it through
the C ABI twice in a row, on different routings, into the same output arrays,
and checks every table against moe_build_schedule's (bit-exact, as all
schedule tests are). This file is collected last so that a run stopping at
the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_schedule_gb300 import MoELayer, _lib

pytestmark = pytest.mark.gpu


def _ids(N, E, k, seed):
    """k distinct experts per token, drawn with Zipf(1.2) weights (Gumbel top-k)."""
    rng = np.random.default_rng(seed)
    logp = -1.2 * np.log(np.arange(1, E + 1, dtype=np.float64))
    keys = logp[None, :] + rng.gumbel(size=(N, E))
    return np.argsort(-keys, axis=1)[:, :k].astype(np.int32)


def _outputs(E, N, k, R, dev):
    return {name: torch.full((max(n, 1),), -7, dtype=torch.int32, device=dev)
            for name, n in (("counts", E), ("offsets", E + 1), ("pad_offsets", E + 1),
                            ("slot_of", N * k), ("src_of_row", R), ("tiles", 3 * (R // 128)),
                            ("n_tiles", 1))}


def _view(out):
    return _lib.Schedule(*(out[n].data_ptr() for n, _ in _lib.Schedule._fields_))


def _check_equal(out, ref, E, tag):
    rows = int(ref["pad_offsets"][E])
    nt = int(ref["n_tiles"][0])
    for name in ("counts", "offsets", "pad_offsets", "slot_of", "n_tiles"):
        assert torch.equal(out[name][:ref[name].numel()], ref[name]), (tag, name)
    assert torch.equal(out["src_of_row"][:rows], ref["src_of_row"][:rows]), tag
    assert torch.equal(out["tiles"][:3 * nt], ref["tiles"][:3 * nt]), tag


def test_noalloc_schedule_matches_workspace_schedule_on_two_calls():
    N, E, k = 3000, 64, 8
    dev = torch.device("cuda:0")
    ref_layer = MoELayer(N, 256, 256, E, k, device=dev, allocate_grads=False)
    p = ref_layer.p
    out = _outputs(E, N, k, _lib.moe_grouped_rows(p), dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    view = _view(out)
    for call, seed in enumerate((11, 12)):
        ids = torch.as_tensor(_ids(N, E, k, seed)).to(dev)
        _lib.moe_build_schedule(p, ids, ref_layer.ws)
        _lib.moe_build_schedule_noalloc(p, ids, view, err)
        torch.cuda.synchronize()
        _check_equal(out, ref_layer.schedule_tensors(), E, call)
        assert int(err.item()) == 0


def test_noalloc_largest_accepted_problem():
    """E * ceil(N*k / 256) = 256 * 2048 = 524288: the whole static array in use."""
    N, E, k = 65536, 256, 8
    dev = torch.device("cuda:0")
    ref_layer = MoELayer(N, 256, 256, E, k, device=dev, allocate_grads=False)
    p = ref_layer.p
    out = _outputs(E, N, k, _lib.moe_grouped_rows(p), dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ids = torch.as_tensor(_ids(N, E, k, 5)).to(dev)
    _lib.moe_build_schedule(p, ids, ref_layer.ws)
    _lib.moe_build_schedule_noalloc(p, ids, _view(out), err)
    torch.cuda.synchronize()
    _check_equal(out, ref_layer.schedule_tensors(), E, "largest")
    assert int(err.item()) == 0


def test_noalloc_empty_batch_gives_zero_counts():
    N, E, k = 0, 16, 2
    dev = torch.device("cuda:0")
    p = _lib.problem(N, 256, 256, E, k)
    out = _outputs(E, 1, k, _lib.moe_grouped_rows(p), dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ids = torch.zeros((1, k), dtype=torch.int32, device=dev)  # not read when N = 0
    _lib.moe_build_schedule_noalloc(p, ids, _view(out), err)
    torch.cuda.synchronize()
    assert torch.equal(out["counts"], torch.zeros(E, dtype=torch.int32, device=dev))
    assert torch.equal(out["offsets"], torch.zeros(E + 1, dtype=torch.int32, device=dev))
    assert torch.equal(out["pad_offsets"], torch.zeros(E + 1, dtype=torch.int32, device=dev))
    assert int(out["n_tiles"][0]) == 0 and int(err.item()) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    view = _lib.Schedule(*([16] * 7))
    # one schedule warp over the limit: ceil(65537 * 8 / 256) = 2049 warps x 256 experts
    for N in (65537, 65536 * 4):
        p = _lib.problem(N, 256, 256, 256, 8)
        st = lib.moe_build_schedule_noalloc(ctypes.byref(p), 16, ctypes.byref(view), 16, None)
        assert st == _lib.MOE_ERR_UNSUPPORTED, N
