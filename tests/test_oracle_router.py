"""Pins of the oracle's router projection (CPU): a brute-force triple loop,
central finite differences of a scalar loss, and shapes chosen non-square so
that a transposed operand cannot pass."""
import numpy as np

from oracle import moe_oracle as O


def _case(T=5, d=7, E=3, seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, d)), rng.standard_normal((E, d)), rng.standard_normal((T, E))


def test_router_logits_brute_force():
    x, Wr, _ = _case()
    T, d = x.shape
    E = Wr.shape[0]
    want = np.zeros((T, E))
    for t in range(T):
        for e in range(E):
            acc = 0.0
            for i in range(d):
                acc += x[t, i] * Wr[e, i]
            want[t, e] = acc
    got = O.router_logits(x, Wr)
    assert got.shape == (T, E)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def test_router_backward_brute_force():
    x, Wr, dl = _case(seed=1)
    T, d = x.shape
    E = Wr.shape[0]
    dx, dW = O.router_backward(x, Wr, dl)
    assert dx.shape == (T, d) and dW.shape == (E, d)
    for t in range(T):
        for i in range(d):
            assert abs(dx[t, i] - sum(dl[t, e] * Wr[e, i] for e in range(E))) < 1e-12
    for e in range(E):
        for i in range(d):
            assert abs(dW[e, i] - sum(dl[t, e] * x[t, i] for t in range(T))) < 1e-12


def test_router_backward_finite_differences():
    x, Wr, C = _case(T=4, d=6, E=5, seed=2)

    def loss(x_, W_):
        return float(np.sum(O.router_logits(x_, W_) * C))

    dx, dW = O.router_backward(x, Wr, C)
    h = 1e-6
    for (t, i) in [(0, 0), (3, 5), (2, 1)]:
        xp, xm = x.copy(), x.copy()
        xp[t, i] += h
        xm[t, i] -= h
        assert abs((loss(xp, Wr) - loss(xm, Wr)) / (2 * h) - dx[t, i]) < 1e-7
    for (e, i) in [(0, 0), (4, 5), (2, 3)]:
        Wp, Wm = Wr.copy(), Wr.copy()
        Wp[e, i] += h
        Wm[e, i] -= h
        assert abs((loss(x, Wp) - loss(x, Wm)) / (2 * h) - dW[e, i]) < 1e-7


def test_router_feeds_route():
    # the router's logits, rounded to fp32, are valid routing input
    x, Wr, _ = _case(T=9, d=4, E=6, seed=3)
    z = O.router_logits(x, Wr).astype(np.float32)
    ids, g = O.route(z, 2)
    assert ids.shape == (9, 2)
    np.testing.assert_allclose(g.sum(axis=1), 1.0)
    assert np.all(z[np.arange(9), ids[:, 0]] >= z[np.arange(9), ids[:, 1]])
