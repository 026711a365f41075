"""Pins for the oracle's router (the GEMM in front of the top-k routing and its
backward with the selection held fixed).

* logits equal numpy's fp64 matmul of the same bf16 values;
* the backward equals PyTorch fp64 autograd through "logits = x Wr^T, w =
  softmax over the selected logits, L = sum w * g" (autograd differentiates
  the forward definition; nothing of the oracle's hand-derived formulas is
  reused), for dz, dWr and dx;
* softmax-backward invariants: the dz of a token sum to zero, and k = 1
  gives dz = 0 (a single selected weight is always 1).
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")


def _bf16(a):
    return torch.as_tensor(np.asarray(a, np.float32)).bfloat16()


def _case(N, H, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((N, H), generator=g).bfloat16()
    wr = (torch.randn((E, H), generator=g) / H ** 0.5).bfloat16()
    logits = oracle.router_logits(x, wr)
    ids, w = oracle.route_topk(logits.astype(np.float32), None, k)
    dw = torch.randn((N, k), generator=g, dtype=torch.float64).numpy()
    return x, wr, logits, ids, w, dw


def test_logits_equal_numpy_fp64_matmul():
    x, wr, logits, *_ = _case(37, 96, 12, 3, 0)
    ref = x.double().numpy() @ wr.double().numpy().T
    np.testing.assert_allclose(logits, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("N,H,E,k", [(9, 64, 8, 2), (33, 96, 16, 4), (5, 32, 4, 4)])
def test_backward_equals_autograd(N, H, E, k):
    x, wr, logits, ids, _, dw = _case(N, H, E, k, N + H)
    xt = x.double().clone().requires_grad_(True)
    wt = wr.double().clone().requires_grad_(True)
    lg = xt @ wt.T
    z = torch.gather(lg, 1, torch.as_tensor(ids, dtype=torch.int64))
    w = torch.softmax(z, dim=1)
    (w * torch.as_tensor(dw)).sum().backward()
    r = oracle.router_backward(x, wr, ids, w.detach().numpy(), dw)
    # dL/dz via autograd on z directly
    zt = z.detach().clone().requires_grad_(True)
    (torch.softmax(zt, dim=1) * torch.as_tensor(dw)).sum().backward()
    np.testing.assert_allclose(r["dz"], zt.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["dwr"], wt.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(r["dx"], xt.grad.numpy(), rtol=1e-11, atol=1e-13)


def test_softmax_backward_invariants():
    x, wr, _, ids, w, dw = _case(20, 64, 8, 3, 5)
    r = oracle.router_backward(x, wr, ids, w, dw)
    np.testing.assert_allclose(r["dz"].sum(axis=1), 0.0, atol=1e-15)
    x1, wr1, _, ids1, w1, dw1 = _case(20, 64, 8, 1, 6)
    r1 = oracle.router_backward(x1, wr1, ids1, w1, dw1)
    assert np.all(r1["dz"] == 0.0) and np.all(r1["dwr"] == 0.0) and np.all(r1["dx"] == 0.0)


def test_rejects_bad_expert_ids():
    x, wr, _, ids, w, dw = _case(4, 32, 4, 2, 7)
    ids = ids.copy()
    ids[1, 0] = 4
    with pytest.raises(RuntimeError):
        oracle.router_backward(x, wr, ids, w, dw)
