"""Pins for the oracle's routing and schedule table (CPU).

Routing follows the per-step top-k choice of experts (leiphone "MoK..." 01);
the schedule is the per-expert count / placement / contiguity table of the
same section and of Marktechpost "Cursor开源MoK..." (three design decisions).
"""
import math

import numpy as np
import pytest
import scipy.special

from oracle import moe_oracle as O


def _brute_route(z, k):
    T, E = z.shape
    ids = np.zeros((T, k), np.int64)
    g = np.zeros((T, k))
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(z[t, e]), e))
        sel = order[:k]
        ids[t] = sel
        w = [math.exp(float(z[t, e]) - float(z[t, sel[0]])) for e in sel]
        s = math.fsum(w)
        g[t] = [v / s for v in w]
    return ids, g


@pytest.mark.parametrize("T,E,k,seed", [(64, 8, 2, 0), (50, 16, 4, 1), (7, 5, 5, 2), (9, 3, 1, 3)])
def test_route_matches_python_sorted(T, E, k, seed):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, E)).astype(np.float32)
    ids, g = O.route(z, k)
    bi, bg = _brute_route(z, k)
    assert np.array_equal(ids, bi)
    np.testing.assert_allclose(g, bg, rtol=1e-13, atol=0)


def test_route_ties_lower_id_wins_and_signed_zero():
    rng = np.random.default_rng(5)
    z = rng.integers(-2, 3, size=(200, 12)).astype(np.float32)
    z[z == 0] = np.where(rng.random(np.count_nonzero(z == 0)) < 0.5, -0.0, 0.0)
    for k in (1, 3, 6, 12):
        ids, _ = O.route(z, k)
        bi, _ = _brute_route(z, k)
        assert np.array_equal(ids, bi)
    z1 = np.array([[1.0, 3.0, 3.0, 2.0], [-0.0, 0.0, -1.0, -0.0]], np.float32)
    ids, g = O.route(z1, 2)
    assert ids.tolist() == [[1, 2], [0, 1]]
    np.testing.assert_allclose(g, [[0.5, 0.5], [0.5, 0.5]], rtol=0, atol=1e-15)


def test_route_hand_example_weights():
    z = np.array([[0.0, math.log(3.0), -5.0]], np.float32)
    ids, g = O.route(z, 2)
    assert ids.tolist() == [[1, 0]]
    # exp(ln3) : exp(0) = 3 : 1 -> renormalised 0.75 / 0.25 (up to fp32 ln 3)
    z3 = float(np.float32(math.log(3.0)))
    want = [math.exp(z3) / (math.exp(z3) + 1), 1 / (math.exp(z3) + 1)]
    np.testing.assert_allclose(g[0], want, rtol=1e-15)
    np.testing.assert_allclose(g[0], [0.75, 0.25], rtol=1e-7)


def test_route_equals_full_softmax_renormalised():
    rng = np.random.default_rng(7)
    z = (rng.standard_normal((300, 64)) * 3).astype(np.float32)
    ids, g = O.route(z, 8)
    p = scipy.special.softmax(z.astype(np.float64), axis=1)
    ps = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(g, ps / ps.sum(1, keepdims=True), rtol=1e-12)
    assert np.all(np.diff(np.take_along_axis(z, ids.astype(np.int64), 1), axis=1) <= 0)


def test_route_rejects_bad_input():
    with pytest.raises(ValueError):
        O.route(np.array([[np.nan, 1.0]], np.float32), 1)
    with pytest.raises(ValueError):
        O.route(np.zeros((2, 3), np.float32), 4)
    with pytest.raises(TypeError):
        O.route(np.zeros((2, 3), np.float64), 1)


def _brute_schedule(ids, E):
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    counts = [0] * E
    for e in flat:
        counts[e] += 1
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    nxt = offsets[:-1].copy()
    perm = [0] * len(flat)
    for r, e in enumerate(flat):
        perm[nxt[e]] = r
        nxt[e] += 1
    return counts, offsets, perm


@pytest.mark.parametrize("T,E,k,seed", [(64, 8, 2, 0), (333, 17, 3, 1), (1, 4, 4, 2), (100, 64, 8, 3)])
def test_schedule_matches_counting_sort(T, E, k, seed):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = O.route(z, k)
    counts, offsets, perm, inv = O.schedule(ids, E)
    bc, bo, bp = _brute_schedule(ids, E)
    assert counts.tolist() == bc and offsets.tolist() == bo and perm.tolist() == bp
    R = T * k
    assert counts.sum() == R and offsets[-1] == R and np.all(np.diff(offsets) >= 0)
    assert np.array_equal(np.sort(perm), np.arange(R))
    assert np.array_equal(inv[perm], np.arange(R)) and np.array_equal(perm[inv], np.arange(R))
    flat = ids.reshape(-1)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    for t in range(T):
        assert len(set(ids[t].tolist())) == k


def test_schedule_skewed_and_empty_experts():
    ids = np.array([[3, 0], [3, 1], [3, 0], [0, 3]], np.int32)
    counts, offsets, perm, inv = O.schedule(ids, 5)
    assert counts.tolist() == [3, 1, 0, 4, 0]
    assert offsets.tolist() == [0, 3, 4, 4, 8, 8]
    assert perm.tolist() == [1, 5, 6, 3, 0, 2, 4, 7]
