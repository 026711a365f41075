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
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.2
    p /= p.sum()
    return np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(N)]).astype(np.int32)


def test_noalloc_schedule_matches_workspace_schedule_on_two_calls():
    N, E, k = 3000, 64, 8
    dev = torch.device("cuda:0")
    ref_layer = MoELayer(N, 256, 256, E, k, device=dev, allocate_grads=False)
    p = ref_layer.p
    R = _lib.moe_grouped_rows(p)
    out = {name: torch.full((n,), -7, dtype=torch.int32, device=dev)
           for name, n in (("counts", E), ("offsets", E + 1), ("pad_offsets", E + 1),
                           ("slot_of", N * k), ("src_of_row", R), ("tiles", 3 * (R // 128)),
                           ("n_tiles", 1))}
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    view = _lib.Schedule(*(out[n].data_ptr() for n, _ in _lib.Schedule._fields_))
    for call, seed in enumerate((11, 12)):
        ids = torch.as_tensor(_ids(N, E, k, seed)).to(dev)
        _lib.moe_build_schedule(p, ids, ref_layer.ws)
        _lib.moe_build_schedule_noalloc(p, ids, view, err)
        torch.cuda.synchronize()
        ref = ref_layer.schedule_tensors()
        rows = int(ref["pad_offsets"][E])
        nt = int(ref["n_tiles"][0])
        for name in ("counts", "offsets", "pad_offsets", "slot_of", "n_tiles"):
            assert torch.equal(out[name], ref[name]), (call, name)
        assert torch.equal(out["src_of_row"][:rows], ref["src_of_row"][:rows]), call
        assert torch.equal(out["tiles"][:3 * nt], ref["tiles"][:3 * nt]), call
        assert int(err.item()) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    p = _lib.problem(65536 * 4, 256, 256, 256, 8)  # E * ceil(N*k/256) > 524288
    view = _lib.Schedule(*([16] * 7))
    st = lib.moe_build_schedule_noalloc(ctypes.byref(p), 16, ctypes.byref(view), 16, None)
    assert st == _lib.MOE_ERR_UNSUPPORTED
