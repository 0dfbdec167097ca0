"""Pins for the oracle's forward (Schedule -> Dispatch -> Expert FFN ->
Combine -> weighted merge, leiphone "MoK..." 03) and backward (reverse
combine / reverse dispatch, leiphone 02; routing-weight gradient through the
SwiGLU backward, Marktechpost "Cursor开源MoK..." three design decisions)."""
import math

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O


def _problem(T, d, f, E, k, seed, x_std=None):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, E)).astype(np.float32)
    x = rng.standard_normal((T, d)) * (x_std if x_std else 1 / math.sqrt(d))
    W1 = rng.standard_normal((E, d, 2 * f)) / math.sqrt(d)
    W2 = rng.standard_normal((E, f, d)) / math.sqrt(f)
    dO = rng.standard_normal((T, d))
    ids, g = O.route(z, k)
    return z, x, W1, W2, dO, ids, g


@pytest.mark.parametrize("shape", [(64, 128, 64, 8, 2), (40, 32, 16, 6, 3)])
def test_forward_equals_per_token_brute_force(shape):
    z, x, W1, W2, dO, ids, g = _problem(*shape, seed=1, x_std=1.0)
    out, Yts = O.forward(x, W1, W2, ids, g)
    bf = O.forward_tokens(x, W1, W2, ids, g)
    np.testing.assert_allclose(out, bf, rtol=1e-12, atol=1e-12)
    # a pure-python loop per token and slot, for a few tokens
    f = W2.shape[1]
    for t in (0, 7, 31):
        acc = np.zeros(x.shape[1])
        for j in range(ids.shape[1]):
            e = ids[t, j]
            h = [sum(x[t, i] * W1[e, i, c] for i in range(x.shape[1])) for c in range(2 * f)]
            a = [h[c] / (1 + math.exp(-h[c])) * h[f + c] for c in range(f)]
            y = [sum(a[c] * W2[e, c, o] for c in range(f)) for o in range(x.shape[1])]
            acc += g[t, j] * np.array(y)
        np.testing.assert_allclose(out[t], acc, rtol=1e-11, atol=1e-12)


def test_forward_k1_is_identity_merge():
    z, x, W1, W2, dO, ids, g = _problem(50, 32, 16, 5, 1, seed=2, x_std=1.0)
    assert np.all(g == 1.0)
    out, Yts = O.forward(x, W1, W2, ids, g)
    assert np.array_equal(out, Yts[:, 0])


def test_forward_single_expert_is_dense_swiglu_ffn():
    z, x, W1, W2, dO, ids, g = _problem(33, 48, 24, 1, 1, seed=3, x_std=1.0)
    out, _ = O.forward(x, W1, W2, ids, g)
    X = torch.tensor(x, dtype=torch.float64)
    H = X @ torch.tensor(W1[0])
    A = torch.nn.functional.silu(H[:, :24]) * H[:, 24:]
    want = (A @ torch.tensor(W2[0])).numpy()
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-13)


def test_forward_hand_example_gate_then_up():
    # d = 2, f = 1, one expert: x = [1, 0] picks row 0 of W1 -> H = [a, b]
    a, b, p, q = 0.7, -1.3, 2.0, 0.5
    x = np.array([[1.0, 0.0]])
    W1 = np.array([[[a, b], [5.0, 6.0]]])
    W2 = np.array([[[p, q]]])
    out, _ = O.forward(x, W1, W2, np.array([[0]]), np.array([[1.0]]))
    s = a / (1 + math.exp(-a)) * b
    np.testing.assert_allclose(out[0], [s * p, s * q], rtol=1e-15)


def test_forward_linear_in_W2():
    z, x, W1, W2, dO, ids, g = _problem(30, 32, 16, 4, 2, seed=4, x_std=1.0)
    W2b = np.random.default_rng(9).standard_normal(W2.shape)
    al, be = 0.37, -1.9
    o1, _ = O.forward(x, W1, W2, ids, g)
    o2, _ = O.forward(x, W1, W2b, ids, g)
    o3, _ = O.forward(x, W1, al * W2 + be * W2b, ids, g)
    np.testing.assert_allclose(o3, al * o1 + be * o2, rtol=1e-12, atol=1e-12)


def _loss(x, W1, W2, ids, g, dO):
    out, _ = O.forward(x, W1, W2, ids, g)
    return float(np.sum(out * dO))


def _fd(fun, arr, idx, h):
    old = arr[idx]
    arr[idx] = old + h
    lp = fun()
    arr[idx] = old - h
    lm = fun()
    arr[idx] = old
    return (lp - lm) / (2 * h)


@pytest.mark.parametrize("x_std", [None, 1.0])
def test_backward_finite_differences(x_std):
    T, d, f, E, k = 64, 128, 64, 8, 2
    z, x, W1, W2, dO, ids, g = _problem(T, d, f, E, k, seed=5, x_std=x_std)
    B = O.backward(x, W1, W2, ids, g, dO)
    np.testing.assert_allclose(B["dg"], B["dg_fused"], rtol=1e-10, atol=1e-12)
    rng = np.random.default_rng(11)
    fun = lambda: _loss(x, W1, W2, ids, g, dO)  # noqa: E731
    for name, arr, grad in (("x", x, B["dx"]), ("W1", W1, B["dW1"]), ("W2", W2, B["dW2"])):
        flat_idx = rng.choice(arr.size, 24, replace=False)
        # make sure touched experts' weights are sampled too
        if name != "x":
            e0 = int(ids[0, 0])
            flat_idx[:6] = np.ravel_multi_index((np.full(6, e0), rng.integers(0, arr.shape[1], 6),
                                                  rng.integers(0, arr.shape[2], 6)), arr.shape)
        for fi in flat_idx:
            idx = np.unravel_index(fi, arr.shape)
            h = 1e-6 * max(1.0, abs(arr[idx]))
            num = _fd(fun, arr, idx, h)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, grad[idx])
    for t in range(0, T, 9):
        for j in range(k):
            h = 1e-6
            num = _fd(fun, g, (t, j), h)
            assert abs(num - B["dg"][t, j]) <= 1e-6 * max(1.0, abs(num))


def test_backward_dlogits_finite_differences():
    T, d, f, E, k = 64, 128, 64, 8, 2
    z, x, W1, W2, dO, ids, g = _problem(T, d, f, E, k, seed=6, x_std=1.0)
    B = O.backward(x, W1, W2, ids, g, dO)
    zs = np.sort(z, axis=1)[:, ::-1]
    margin = zs[:, k - 1] - zs[:, k]
    z64 = z.astype(np.float64)

    def loss_of_logits(zz):
        # route in fp64 with the selection held fixed (valid while the margin holds)
        sel = np.take_along_axis(zz, ids.astype(np.int64), 1)
        ex = np.exp(sel - sel[:, :1])
        gg = ex / ex.sum(1, keepdims=True)
        return _loss(x, W1, W2, ids, gg, dO)

    checked = 0
    for t in np.nonzero(margin > 1e-3)[0][:12]:
        for e in range(E):
            h = 1e-6
            zp = z64.copy(); zp[t, e] += h
            zm = z64.copy(); zm[t, e] -= h
            num = (loss_of_logits(zp) - loss_of_logits(zm)) / (2 * h)
            assert abs(num - B["dlogits"][t, e]) <= 1e-6 * max(1.0, abs(num))
            checked += 1
    assert checked >= 8 * E
    # rows of dlogits sum to zero (softmax is shift invariant)
    np.testing.assert_allclose(B["dlogits"].sum(1), 0, atol=1e-12)


def test_backward_subsets_match_full():
    T, d, f, E, k = 48, 64, 32, 6, 2
    z, x, W1, W2, dO, ids, g = _problem(T, d, f, E, k, seed=8, x_std=1.0)
    B = O.backward(x, W1, W2, ids, g, dO)
    ex = O.backward_experts(x, W1, W2, ids, g, dO, range(E))
    for e in range(E):
        np.testing.assert_allclose(ex[e][0], B["dW1"][e], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(ex[e][1], B["dW2"][e], rtol=1e-12, atol=1e-13)
    toks = [0, 5, 17, 47]
    bt = O.backward_tokens(x, W1, W2, ids, g, dO, toks)
    np.testing.assert_allclose(bt["dx"], B["dx"][toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(bt["dg"], B["dg"][toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(bt["dlogits"], B["dlogits"][toks], rtol=1e-12, atol=1e-13)


def test_backward_empty_expert_has_zero_weight_grads():
    ids = np.array([[0, 1], [1, 0]], np.int32)
    g = np.array([[0.6, 0.4], [0.5, 0.5]])
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 8)); W1 = rng.standard_normal((3, 8, 8)); W2 = rng.standard_normal((3, 4, 8))
    B = O.backward(x, W1, W2, ids, g, rng.standard_normal((2, 8)))
    assert np.all(B["dW1"][2] == 0) and np.all(B["dW2"][2] == 0)
