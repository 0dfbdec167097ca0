"""Pins of the oracle's MXFP8 forward (activation quantisation on the dispatch
and SwiGLU data path, leiphone "MoK..." 02; the BF16 and MXFP8 modes of
Marktechpost "Cursor开源MoK..." three design decisions).  Reading: each GEMM
quantises both operands along its own contraction dimension -- x and W1 along
d, the SwiGLU output A and W2 along f -- in OCP MX blocks of 32.

1. With the identity in place of the quantiser it is the exact layer (the
   per-token brute force, itself pinned by the permuted forward and by a
   dense-FFN reduction), so any wiring mistake shows.
2. With MXFP8 the error against the exact layer is that of 3-bit mantissas.
3. Axes, one operand at a time (the others left unquantised): inputs whose
   blocks along that operand's contraction axis each hold one power-of-two
   scale times small integers quantise losslessly, so the result equals the
   unquantised layer; the same operand quantised along its other axis mixes
   magnitudes 16 binades apart in a block and loses bits.  A transposed
   operand or a block along the wrong dimension fails one of these.
4. A power-of-two scale of x passes exactly through every block scale.
"""
import numpy as np
import pytest

from oracle import moe_oracle as O


def _case(T=40, d=64, f=32, E=4, k=2, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    W1 = [rng.standard_normal((d, 2 * f)) / 8 for _ in range(E)]
    W2 = [rng.standard_normal((f, d)) / 6 for _ in range(E)]
    z = rng.standard_normal((T, E)).astype(np.float32)
    ids, g = O.route(z, k)
    return x, W1, W2, ids, g


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _maxrel(a, b):
    return float(np.max(np.abs(a - b) / np.abs(b)))


def _ident(v, axis):
    return v


def _qdq_any(v, axis):
    """MXFP8 quantise-dequantise along `axis` of any length (zero-padded)."""
    n = v.shape[axis]
    pad = (-n) % 32
    if pad:
        widths = [(0, 0), (0, 0)]
        widths[axis] = (0, pad)
        v = np.pad(v, widths)
    out = O.mxfp8_dequantize(*O.mxfp8_quantize(v, axis), axis)
    return np.take(out, np.arange(n), axis=axis)


def _swapped(v, axis):
    return _qdq_any(v, 1 - axis)


def _grid(rng, shape, lo=-7, hi=8):
    """Small integers: exact in E4M3 under any block scale that keeps the
    block maximum in range."""
    return rng.integers(lo, hi, size=shape).astype(np.float64)


def _binades(rng, n):
    """Powers of two 16 binades apart (2^8 or 2^-8), more than E4M3 spans
    below a block's maximum, so a block holding both loses the small ones."""
    return np.ldexp(1.0, 8 * rng.choice([-1, 1], size=n))


@pytest.mark.parametrize("shape", [dict(), dict(T=77, d=96, f=64, E=5, k=3, seed=1),
                                   dict(T=9, E=8, k=8, seed=2)])
def test_identity_quantiser_is_the_exact_forward(shape):
    x, W1, W2, ids, g = _case(**shape)
    ref = O.forward_tokens(x, W1, W2, ids, g)
    got = O.forward_mxfp8(x, W1, W2, ids, g, qdq=_ident)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    toks = np.array([0, 3, len(x) - 1])
    np.testing.assert_allclose(O.forward_mxfp8(x, W1, W2, ids, g, toks, qdq=_ident), ref[toks],
                               rtol=0, atol=1e-12 * np.abs(ref).max())


def test_mxfp8_error_is_that_of_e4m3():
    x, W1, W2, ids, g = _case(T=96, d=128, f=64, E=4, k=2, seed=3)
    ref = O.forward_tokens(x, W1, W2, ids, g)
    e = _rel(O.forward_mxfp8(x, W1, W2, ids, g), ref)
    # up to 2^-4 relative per quantised element, two quantised operands per
    # product, two chained GEMMs
    assert 1e-3 < e < 0.1, e
    for op in O.FORWARD_OPERANDS:  # each operand alone does quantise something
        e1 = _rel(O.forward_mxfp8(x, W1, W2, ids, g, quantise=[op]), ref)
        assert 1e-4 < e1 < 0.08, (op, e1)


def _axis_case(op, seed):
    """Inputs on which operand `op` is exactly representable blockwise along
    its contraction axis only."""
    rng = np.random.default_rng(seed)
    T, d, f, E, k = 96, 64, 64, 3, 2
    x = rng.standard_normal((T, d))
    W1 = [rng.standard_normal((d, 2 * f)) / 8 for _ in range(E)]
    W2 = [rng.standard_normal((f, d)) / 8 for _ in range(E)]
    if op == "fwd.x":      # blocks along d: one scale per token row
        x = _grid(rng, (T, d)) * _binades(rng, (T, 1))
    elif op == "fwd.W1":   # W1e [d, 2f], blocks along d: one scale per column
        W1 = [_grid(rng, (d, 2 * f)) * _binades(rng, (1, 2 * f)) for _ in range(E)]
    elif op == "fwd.W2":   # W2e [f, d], blocks along f: one scale per column
        W2 = [_grid(rng, (f, d)) * _binades(rng, (1, d)) for _ in range(E)]
    elif op == "fwd.A":
        # A [m, f] blocks along f: one scale per token row.  x[t] = c_t e_i(t)
        # (one nonzero), the gate weights 2^14 so that the gate pre-activation
        # is >= 2^10 and SiLU is exactly the identity there, the up weights
        # small integers times 2^-14: A[t, j] = c_t^2 * n[i(t), j] with
        # c_t^2 = 2^8 or 2^-8.
        c = np.ldexp(1.0, 4 * rng.choice([-1, 1], size=T))
        x = np.zeros((T, d))
        x[np.arange(T), rng.integers(0, d, size=T)] = c
        W1 = [np.concatenate([np.full((d, f), 2.0 ** 14), _grid(rng, (d, f)) * 2.0 ** -14], axis=1)
              for _ in range(E)]
    z = rng.standard_normal((T, E)).astype(np.float32)
    ids, g = O.route(z, k)
    return x, W1, W2, ids, g


@pytest.mark.filterwarnings("ignore:overflow encountered in exp")  # SiLU of large negative inputs: exactly 0
@pytest.mark.parametrize("op", O.FORWARD_OPERANDS)
def test_quantisation_axis_of_each_operand(op):
    x, W1, W2, ids, g = _axis_case(op, seed=10 + O.FORWARD_OPERANDS.index(op))
    ref = O.forward_mxfp8(x, W1, W2, ids, g, qdq=_ident)
    assert np.all(np.isfinite(ref)) and np.all(ref != 0)
    got = O.forward_mxfp8(x, W1, W2, ids, g, quantise=[op])
    assert _maxrel(got, ref) < 1e-12, op
    # control: the same operand blocked along its other axis loses bits
    bad = O.forward_mxfp8(x, W1, W2, ids, g, qdq=_swapped, quantise=[op])
    assert _maxrel(bad, ref) > 1e-2, op


def test_all_operands_on_one_grid_case_are_exact():
    # one case on which all four operands are blockwise exact along their
    # contraction axes at once (the A construction above, with W2 scaled per
    # column): the fully quantised forward equals the exact layer
    rng = np.random.default_rng(20)
    x, W1, _, ids, g = _axis_case("fwd.A", seed=20)
    W2 = [_grid(rng, (64, 64)) * _binades(rng, (1, 64)) for _ in range(3)]
    ref = O.forward_mxfp8(x, W1, W2, ids, g, qdq=_ident)
    got = O.forward_mxfp8(x, W1, W2, ids, g)
    assert _maxrel(got, ref) < 1e-12
    # A's rows of one expert mix c^2 = 2^8 and 2^-8 and W2's rows mix column
    # scales, so each blocked along its other axis loses bits (x's values are
    # powers of two and W1's 32-column blocks never straddle gate and up, so
    # those two survive either way here; their own cases above cover them)
    for op in ("fwd.A", "fwd.W2"):
        bad = O.forward_mxfp8(x, W1, W2, ids, g, qdq=_swapped, quantise=[op])
        assert _maxrel(bad, ref) > 1e-2, op


def test_power_of_two_scaling_of_x_is_exact():
    # the UE8M0 block scale absorbs a power of two: quantising 2^5 x gives
    # exactly 2^5 times the quantised x, so the layer on 2^5 x with x
    # quantised equals the unquantised layer on 2^5 q(x); a scale rule that
    # is not a power of two, or one that rounds the scale, breaks this
    x, W1, W2, ids, g = _case(T=64, d=64, f=32, E=3, k=2, seed=6)
    xq = O.mxfp8_dequantize(*O.mxfp8_quantize(x, 1), 1)
    b = O.forward_mxfp8(32.0 * x, W1, W2, ids, g, quantise=["fwd.x"])
    c = O.forward_mxfp8(32.0 * xq, W1, W2, ids, g, qdq=_ident)
    np.testing.assert_array_equal(b, c)


def test_unknown_operand_name_is_rejected():
    x, W1, W2, ids, g = _case()
    with pytest.raises(ValueError):
        O.forward_mxfp8(x, W1, W2, ids, g, quantise=["fwd.y"])
