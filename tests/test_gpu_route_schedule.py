"""GPU routing and schedule vs the oracle: bit-exact ids, counts, offsets,
permutation and tile list; routing weights within the fp32 bound.

Routing: "Router picks top-k experts" (clip "Mixture-of-Kittens: Cursor
open-sources an MoE training megakernel", key flowchart). Schedule: counts,
prefix sums and permutation built on the GPU with no host sync and no token
dropping (same page, key point 4).
"""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_schedule_gb300 import MoELayer, _lib, inputs

from gpu_helpers import W_RTOL, dev

pytestmark = pytest.mark.gpu


def _route_and_schedule(N, E, k, logits, bias, H=256, I=256, T=128):
    layer = MoELayer(N, H, I, E, k, device=dev(), allocate_grads=False, minibatch_rows=T)
    lg = torch.as_tensor(logits).to(dev())
    bs = None if bias is None else torch.as_tensor(bias).to(dev())
    layer.route(lg, bs)
    layer.build_schedule()
    torch.cuda.synchronize()
    return layer


def _check_schedule(layer, ids_np, E):
    ref = oracle.build_schedule(ids_np, E, 128, layer.T)
    got = {k: v.cpu().numpy() for k, v in layer.schedule_tensors().items()}
    np.testing.assert_array_equal(got["counts"], ref["counts"])
    np.testing.assert_array_equal(got["offsets"], ref["offsets"])
    np.testing.assert_array_equal(got["pad_offsets"], ref["pad_offsets"])
    np.testing.assert_array_equal(got["slot_of"], ref["slot_of"].ravel())
    rows = int(ref["pad_offsets"][E])
    np.testing.assert_array_equal(got["src_of_row"][:rows], ref["src_of_row"])
    assert int(got["n_tiles"][0]) == ref["n_tiles"]
    np.testing.assert_array_equal(got["tiles"].reshape(-1, 3)[:ref["n_tiles"]], ref["tiles"])


CASES = [
    ("tiny", 256, 8, 2, None),
    ("fine_grained", 4096, 64, 8, None),
    ("skewed_zipf", 16384, 128, 8, 1.2),
    ("e256_ragged_n", 1001, 256, 8, None),
    ("k_equals_e", 77, 8, 8, None),
    ("single_token", 1, 32, 4, None),
    ("e1024", 300, 1024, 32, None),
]


@pytest.mark.parametrize("T", [128, 256, 1024])
@pytest.mark.parametrize("name,N,E,k,zipf", CASES, ids=[c[0] for c in CASES])
def test_route_and_schedule_match_oracle(name, N, E, k, zipf, T):
    g = torch.Generator().manual_seed(N * 31 + E)
    logits = torch.randn((N, E), generator=g).float().numpy()
    bias = None
    if zipf is not None:
        r = torch.randperm(E, generator=g).double() + 1.0
        bias = (-zipf * torch.log(r)).float().numpy()
    layer = _route_and_schedule(N, E, k, logits, bias, T=T)
    ids_ref, w_ref = oracle.route_topk(logits, bias, k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids_ref)
    w = layer.topk_w.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(w - w_ref) / w_ref) <= W_RTOL
    _check_schedule(layer, ids_ref, E)
    assert layer.device_error() == 0


def test_ties_and_signed_zeros():
    N, E, k = 512, 16, 4
    g = torch.Generator().manual_seed(5)
    logits = torch.randint(-2, 3, (N, E), generator=g).float().numpy()  # many exact ties
    logits[::7] = 0.0
    logits[1::7, ::2] = -0.0
    layer = _route_and_schedule(N, E, k, logits, None)
    ids_ref, _ = oracle.route_topk(logits, None, k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids_ref)
    _check_schedule(layer, ids_ref, E)


def test_all_tokens_to_one_expert_and_empty_experts():
    N, E, k = 1000, 16, 1
    logits = np.zeros((N, E), np.float32)
    logits[:, 5] = 10.0  # every token -> expert 5; 15 experts get no token
    layer = _route_and_schedule(N, E, k, logits, None)
    ids_ref, _ = oracle.route_topk(logits, None, k)
    np.testing.assert_array_equal(layer.topk_ids.cpu().numpy(), ids_ref)
    _check_schedule(layer, ids_ref, E)
    s = layer.schedule_tensors()
    assert int(s["counts"][5]) == N and int(s["n_tiles"][0]) == (N + 127) // 128


def test_schedule_from_given_ids_edge_sizes():
    for N, E, k in ((128, 4, 1), (129, 4, 2), (2048, 3, 3), (1, 1, 1)):
        rng = np.random.default_rng(N)
        ids = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
        layer = MoELayer(N, 256, 256, E, k, device=dev(), allocate_grads=False)
        layer.build_schedule(torch.as_tensor(ids).to(dev()))
        torch.cuda.synchronize()
        _check_schedule(layer, ids, E)


def test_bad_expert_id_sets_device_error_without_fault():
    N, E, k = 300, 8, 2
    ids = np.tile(np.array([[0, 1]], np.int32), (N, 1))
    ids[17, 1] = 9
    ids[200, 0] = -3
    layer = MoELayer(N, 256, 256, E, k, device=dev(), allocate_grads=False)
    layer.build_schedule(torch.as_tensor(ids).to(dev()))
    x = torch.zeros((N, 256), dtype=torch.bfloat16, device=dev())
    sv = layer.saved_tensors()
    _lib.moe_dispatch(layer.p, layer.ws, x, sv["xe"])  # unplaced assignments are skipped
    torch.cuda.synchronize()
    assert layer.device_error() == _lib.MOE_DEVERR_BAD_EXPERT
    layer.clear_device_error()
    assert layer.device_error() == 0


def test_nan_logit_sets_device_error():
    N, E, k = 64, 8, 2
    logits = np.random.default_rng(0).standard_normal((N, E)).astype(np.float32)
    logits[10, 3] = np.nan
    layer = _route_and_schedule(N, E, k, logits, None)
    assert layer.device_error() == _lib.MOE_DEVERR_NAN_LOGIT


def test_schedule_is_deterministic_across_runs():
    N, E, k = 16384, 128, 8
    logits = torch.randn((N, E), generator=torch.Generator().manual_seed(1)).numpy()
    a = _route_and_schedule(N, E, k, logits, None)
    b = _route_and_schedule(N, E, k, logits, None)
    for key, t in a.schedule_tensors().items():
        assert torch.equal(t, b.schedule_tensors()[key]), key
    assert torch.equal(a.topk_w, b.topk_w)
