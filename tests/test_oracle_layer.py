"""Pins for the oracle's layer forward and backward.

The layer: router top-k -> dispatch -> expert FFN with SwiGLU (gate/up,
silu*mul, down) -> combine as the routing-weighted sum (clip "Mixture-of-
Kittens: Cursor open-sources an MoE training megakernel", key flowchart and
key point 5); the backward mirrors it (key point 2: reverse-combine,
reverse-dispatch). Pins used here:
  * hand-derived closed forms on 2x2 experts whose gate/up/down matrices are
    not symmetric, so a transposed operand or swapped gate/up fails;
  * central finite differences of L = <dY, y> for every gradient;
  * invariants: shared-weight experts collapse to one dense FFN (weights sum
    to 1), token independence, expert relabelling, exact linearity in Wu and
    Wd, thread-count independence;
  * the sampled entry points agree bitwise with the whole-layer ones.
"""
import math

import numpy as np
import pytest

import oracle

LN3 = math.log(3.0)


def test_closed_form_single_expert():
    # x = [1, 2]; Wg rows: [ln3, 0], [ln3, -ln3] -> g = [ln3, -ln3]
    # sigmoid(ln3) = 3/4, sigmoid(-ln3) = 1/4
    # Wu rows [1, 1], [0, 1] -> u = [3, 2]
    # a = silu(g) * u = [ln3*3/4*3, -ln3/4*2] = [9 ln3/4, -ln3/2]
    # Wd rows [1, 0], [2, 3] -> ye = [a0, 2 a0 + 3 a1] = [9 ln3/4, 3 ln3]
    x = np.array([[1.0, 2.0]])
    wg = np.array([[[LN3, 0.0], [LN3, -LN3]]])
    wu = np.array([[[1.0, 1.0], [0.0, 1.0]]])
    wd = np.array([[[1.0, 0.0], [2.0, 3.0]]])
    y = oracle.forward_f64(x, wg, wu, wd, np.array([[0]]), np.array([[1.0]]))
    np.testing.assert_allclose(y, [[9 * LN3 / 4, 3 * LN3]], rtol=1e-14)


def test_closed_form_two_experts_weighted_sum():
    # expert 0 as above (ye0 = [9 ln3/4, 3 ln3]);
    # expert 1: Wg rows [0, ln3/2], [0, 0] -> g = [ln3, 0]; Wu rows [1,0],[0,0]
    # -> u = [1, 0]; a = [3 ln3/4, 0]; Wd rows [0,0],[4,0] -> ye1 = [0, 3 ln3]
    # y = 0.25 ye0 + 0.75 ye1 = [9 ln3/16, 3 ln3]
    x = np.array([[1.0, 2.0]])
    wg = np.array([[[LN3, 0.0], [LN3, -LN3]], [[0.0, LN3 / 2], [0.0, 0.0]]])
    wu = np.array([[[1.0, 1.0], [0.0, 1.0]], [[1.0, 0.0], [0.0, 0.0]]])
    wd = np.array([[[1.0, 0.0], [2.0, 3.0]], [[0.0, 0.0], [4.0, 0.0]]])
    y = oracle.forward_f64(x, wg, wu, wd, np.array([[0, 1]]), np.array([[0.25, 0.75]]))
    np.testing.assert_allclose(y, [[9 * LN3 / 16, 3 * LN3]], rtol=1e-14)
    # swapping the ranks' experts swaps the weights they receive
    y2 = oracle.forward_f64(x, wg, wu, wd, np.array([[1, 0]]), np.array([[0.75, 0.25]]))
    np.testing.assert_allclose(y2, y, rtol=1e-15)


def test_closed_form_scalar_backward():
    # H = I = 1: y = wd * silu(wg x) * (wu x); with x = 1, wg = ln3, wu = 2,
    # wd = 5, dY = 1: g = ln3, s = 3/4, u = 2, a = 3 ln3/2, y = 15 ln3/2.
    # da = wd = 5; dg = da u s (1 + g (1-s)) = 5*2*3/4*(1 + ln3/4); du = da g s
    # dx = wg dg + wu du; dWd = a; dWg = dg x; dWu = du x; dw = <dY, ye> = y
    x, wg, wu, wd, dy = (np.array(v, float).reshape(s) for v, s in
                         ((1.0, (1, 1)), (LN3, (1, 1, 1)), (2.0, (1, 1, 1)),
                          (5.0, (1, 1, 1)), (1.0, (1, 1))))
    r = oracle.backward_f64(x, wg, wu, wd, np.array([[0]]), np.array([[1.0]]), dy)
    dg = 5 * 2 * 0.75 * (1 + LN3 / 4)
    du = 5 * LN3 * 0.75
    np.testing.assert_allclose(r["dx"], [[LN3 * dg + 2 * du]], rtol=1e-14)
    np.testing.assert_allclose(r["dwd"], [[[1.5 * LN3]]], rtol=1e-14)
    np.testing.assert_allclose(r["dwg"], [[[dg]]], rtol=1e-14)
    np.testing.assert_allclose(r["dwu"], [[[du]]], rtol=1e-14)
    np.testing.assert_allclose(r["dw"], [[7.5 * LN3]], rtol=1e-14)


def _rand_layer(N, H, I, E, k, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((N, H))
    wg = rng.standard_normal((E, I, H)) / math.sqrt(H)
    wu = rng.standard_normal((E, I, H)) / math.sqrt(H)
    wd = rng.standard_normal((E, H, I)) / math.sqrt(I)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    w = rng.random((N, k)) + 0.1
    w /= w.sum(axis=1, keepdims=True)
    dy = rng.standard_normal((N, H))
    return x, wg, wu, wd, ids, w, dy


def _fd(fun, arr, h=1e-5):
    g = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + h
        lp = fun()
        arr[i] = old - h
        lm = fun()
        arr[i] = old
        g[i] = (lp - lm) / (2 * h)
    return g


@pytest.mark.parametrize("N,H,I,E,k", [(4, 5, 7, 3, 2), (3, 8, 4, 4, 3)])
def test_backward_matches_finite_differences(N, H, I, E, k):
    x, wg, wu, wd, ids, w, dy = _rand_layer(N, H, I, E, k, seed=N * 100 + H)

    def loss():
        return float(np.sum(dy * oracle.forward_f64(x, wg, wu, wd, ids, w, threads=1)))

    r = oracle.backward_f64(x, wg, wu, wd, ids, w, dy, threads=1)
    for name, arr in (("dx", x), ("dwg", wg), ("dwu", wu), ("dwd", wd), ("dw", w)):
        fd = _fd(loss, arr)
        err = np.max(np.abs(fd - r[name])) / np.max(np.abs(fd))
        assert err < 1e-7, (name, err)


def test_shared_weights_collapse_to_dense_ffn():
    N, H, I, E, k = 6, 8, 12, 5, 3
    x, wg, wu, wd, ids, w, dy = _rand_layer(N, H, I, E, k, seed=3)
    wg[:] = wg[0]
    wu[:] = wu[0]
    wd[:] = wd[0]
    y = oracle.forward_f64(x, wg, wu, wd, ids, w)
    dense = oracle.forward_f64(x, wg[:1], wu[:1], wd[:1], np.zeros((N, 1), np.int32),
                               np.ones((N, 1)))
    np.testing.assert_allclose(y, dense, rtol=1e-12, atol=1e-14)


def test_token_independence_and_relabelling():
    N, H, I, E, k = 7, 6, 10, 4, 2
    x, wg, wu, wd, ids, w, dy = _rand_layer(N, H, I, E, k, seed=5)
    y = oracle.forward_f64(x, wg, wu, wd, ids, w)
    for t in range(N):
        yt = oracle.forward_f64(x[t:t + 1], wg, wu, wd, ids[t:t + 1], w[t:t + 1])
        np.testing.assert_array_equal(yt[0], y[t])
    perm = np.array([2, 0, 3, 1])  # new expert p holds old expert perm[p]
    inv = np.argsort(perm)
    y2 = oracle.forward_f64(x, wg[perm], wu[perm], wd[perm], inv[ids].astype(np.int32), w)
    np.testing.assert_array_equal(y2, y)


def test_linearity_in_up_and_down_weights():
    x, wg, wu, wd, ids, w, dy = _rand_layer(5, 6, 9, 3, 2, seed=8)
    y = oracle.forward_f64(x, wg, wu, wd, ids, w)
    np.testing.assert_array_equal(oracle.forward_f64(x, wg, 2 * wu, wd, ids, w), 2 * y)
    np.testing.assert_array_equal(oracle.forward_f64(x, wg, wu, 0.5 * wd, ids, w), 0.5 * y)


def test_thread_count_does_not_change_results():
    x, wg, wu, wd, ids, w, dy = _rand_layer(9, 16, 24, 4, 2, seed=11)
    a = oracle.backward_f64(x, wg, wu, wd, ids, w, dy, threads=1)
    b = oracle.backward_f64(x, wg, wu, wd, ids, w, dy, threads=5)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def _bf16_round(a):
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def test_bf16_entry_points_and_sampled_forms_agree():
    N, H, I, E, k = 11, 16, 24, 5, 2
    x, wg, wu, wd, ids, w, dy = _rand_layer(N, H, I, E, k, seed=13)
    xb, wgb, wub, wdb, dyb = (_bf16_round(a) for a in (x, wg, wu, wd, dy))
    xf, wgf, wuf, wdf, dyf = (oracle.bf16_bits_to_f64(a) for a in (xb, wgb, wub, wdb, dyb))
    yb, yeb = oracle.forward_bf16(xb, wgb, wub, wdb, ids, w, want_ye=True)
    yf = oracle.forward_f64(xf, wgf, wuf, wdf, ids, w)
    np.testing.assert_array_equal(yb, yf)
    rb = oracle.backward_bf16(xb, wgb, wub, wdb, ids, w, dyb)
    rf = oracle.backward_f64(xf, wgf, wuf, wdf, ids, w, dyf)
    for key in rb:
        np.testing.assert_array_equal(rb[key], rf[key])
    # ye rows combine to y
    np.testing.assert_allclose((w[:, :, None] * yeb.reshape(N, k, H)).sum(1), yb, rtol=1e-12,
                               atol=1e-14)
    tok = np.array([10, 0, 4])
    s = oracle.tokens_bf16(xb, wgb, wub, wdb, ids, w, dyb, tok)
    np.testing.assert_array_equal(s["y"], yb[tok])
    np.testing.assert_array_equal(s["dx"], rb["dx"][tok])
    np.testing.assert_array_equal(s["dw"], rb["dw"][tok])
    for e in range(E):
        il, hl = np.array([0, 5, 23]), np.array([15, 1])
        g = oracle.expert_wgrad_bf16(xb, wgb, wub, wdb, ids, w, dyb, e, il, hl)
        np.testing.assert_array_equal(g["dwg"], rb["dwg"][e, il])
        np.testing.assert_array_equal(g["dwu"], rb["dwu"][e, il])
        np.testing.assert_array_equal(g["dwd"], rb["dwd"][e, hl])


def test_expert_with_no_tokens_has_zero_gradient():
    x, wg, wu, wd, ids, w, dy = _rand_layer(4, 4, 6, 3, 1, seed=2)
    ids[:] = 1
    r = oracle.backward_f64(x, wg, wu, wd, ids, w, dy)
    assert np.all(r["dwg"][[0, 2]] == 0) and np.all(r["dwd"][[0, 2]] == 0)
    assert np.any(r["dwg"][1] != 0)


def test_forward_and_backward_equal_torch_autograd():
    """An independent library routine: the layer written with torch CPU fp64
    ops (F.silu for the activation, index_add for the weighted combine) and
    differentiated by autograd gives the oracle's y and every gradient, at
    the tiny workload's shape (N=256, H=256, I=512, E=8, top-2)."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    N, H, I, E, k = 256, 256, 512, 8, 2
    rng = np.random.default_rng(31)
    x = rng.standard_normal((N, H))
    wg, wu, wd = (rng.standard_normal(s) / np.sqrt(H) for s in ((E, I, H), (E, I, H), (E, H, I)))
    dy = rng.standard_normal((N, H))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    w = rng.random((N, k)) + 0.05
    w /= w.sum(1, keepdims=True)
    y_ref = oracle.forward_f64(x, wg, wu, wd, ids, w)
    g_ref = oracle.backward_f64(x, wg, wu, wd, ids, w, dy)

    X, WG, WU, WD, W = (torch.tensor(a, requires_grad=True) for a in (x, wg, wu, wd, w))
    y = torch.zeros(N, H, dtype=torch.float64)
    ids_t = torch.as_tensor(ids, dtype=torch.long)
    for j in range(k):
        for e in range(E):
            sel = torch.nonzero(ids_t[:, j] == e).flatten()
            if len(sel) == 0:
                continue
            xs = X[sel]
            act = F.silu(xs @ WG[e].T) * (xs @ WU[e].T)
            y = y.index_add(0, sel, W[sel, j:j + 1] * (act @ WD[e].T))
    (y * torch.as_tensor(dy)).sum().backward()

    def close(got, ref):
        scale = np.max(np.abs(ref))
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12 * scale)

    close(y.detach().numpy(), y_ref)
    close(X.grad.numpy(), g_ref["dx"])
    close(WG.grad.numpy(), g_ref["dwg"])
    close(WU.grad.numpy(), g_ref["dwu"])
    close(WD.grad.numpy(), g_ref["dwd"])
    close(W.grad.numpy(), g_ref["dw"])
