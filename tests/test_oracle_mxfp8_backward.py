"""Pins of the oracle's MXFP8 backward (each backward GEMM quantises both
operands along its own contraction dimension).

1. With the identity in place of the quantiser it is the BF16 backward, which
   finite differences pin (test_oracle_forward_backward.py): any wiring
   mistake (an operand, a transpose, the weight on the wrong side) shows.
2. With MXFP8 the error against the exact backward is that of 3-bit
   mantissas: clearly nonzero (the quantiser is applied) and bounded.
3. Quantisation axes: inputs whose 32-blocks along the contraction dimension
   of the forward GEMM1 (d) and of dgrad2 (d) each hold one power-of-two
   scale times small integers quantise losslessly along that axis and lossily
   along the other (rows of different scale share a block).  The fused
   routing-weight gradient <dOut W2^T, A> then comes out exact; the same
   inputs with the axes swapped do not.
4. A power-of-two scaling of dOut scales every output exactly.
5. Separation: one token's dOut row scaled by 2^12 changes only that token's
   dx and dg (exactly by 2^12): dgrad2 and dgrad1 quantise within rows.  One
   column of dOut scaled by 2^12 changes only that column of dW2: wgrad2
   quantises dOut along the rows.  One row of W2 scaled by 2^12 changes only
   the matching gate and up columns of dW1: wgrad1 quantises dH along the
   rows.

6. Every operand on its own (the tests at the end): quantising one operand
   alone reproduces the unquantised backward exactly on inputs that are
   blockwise exact along that operand's contraction axis, and loses bits when
   the same operand is blocked along its other axis -- all ten operands,
   including dgrad1's W1, wgrad1's X and wgrad2's g*A.  The weight-gradient
   row blocks start at each expert's segment (a reading): an input exact
   under that anchoring is lossy under blocks keyed to the global position.
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
    dO = rng.standard_normal((T, d))
    return x, W1, W2, ids, g, dO


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("shape", [dict(), dict(T=77, d=96, f=64, E=5, k=3, seed=1), dict(T=9, E=8, k=8, seed=2)])
def test_identity_quantiser_is_the_bf16_backward(shape):
    x, W1, W2, ids, g, dO = _case(**shape)
    ref = O.backward(x, W1, W2, ids, g, dO)
    got = O.backward_mxfp8(x, W1, W2, ids, g, dO, qdq=lambda v, axis: v)
    for name in ("dx", "dW1", "dW2", "dlogits"):
        np.testing.assert_allclose(got[name], ref[name], rtol=0, atol=1e-12 * np.abs(ref[name]).max())
    np.testing.assert_allclose(got["dg"], ref["dg_fused"], rtol=0, atol=1e-12 * np.abs(ref["dg_fused"]).max())


def test_mxfp8_error_is_that_of_e4m3():
    x, W1, W2, ids, g, dO = _case(T=96, d=128, f=64, E=4, k=2, seed=3)
    ref = O.backward(x, W1, W2, ids, g, dO)
    got = O.backward_mxfp8(x, W1, W2, ids, g, dO)
    for name, r in (("dx", ref["dx"]), ("dW1", ref["dW1"]), ("dW2", ref["dW2"]), ("dg", ref["dg_fused"])):
        e = _rel(got[name], r)
        # a rounding error of up to 2^-4 relative per element, two quantised
        # operands per product, two chained GEMMs for dx and dW1
        assert 1e-3 < e < 0.15, (name, e)


def _grid(rng, shape):
    """Small integers times 2^-3: exact in E4M3 at any block scale that keeps
    the block maximum in range."""
    return rng.integers(-7, 8, size=shape).astype(np.float64) * 0.125


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


def test_quantisation_axes_of_forward_and_dgrad2():
    # E4M3 keeps 4 significant bits over 15 binades below a block's maximum,
    # so a block loses bits only when it mixes magnitudes further apart: the
    # rows (or columns) here sit at 2^8 or 2^-8, 16 binades apart
    rng = np.random.default_rng(4)
    T, d, f, E, k = 64, 64, 32, 3, 2
    sc_row = lambda n: np.ldexp(1.0, 8 * rng.choice([-1, 1], size=(n, 1)))
    sc_col = lambda n: np.ldexp(1.0, 8 * rng.choice([-1, 1], size=(1, n)))
    x = _grid(rng, (T, d)) * sc_row(T)                                 # blocks along d: one scale each
    W1 = [_grid(rng, (d, 2 * f)) * sc_col(2 * f) for _ in range(E)]    # K = d = axis 0: per column
    W2 = [_grid(rng, (f, d)) * sc_row(f) for _ in range(E)]            # dgrad2 K = d = axis 1: per row
    dO = _grid(rng, (T, d)) * sc_row(T)                                # dgrad2 K = d: per token row
    z = rng.standard_normal((T, E)).astype(np.float32)
    ids, g = O.route(z, k)
    with np.errstate(over="ignore"):  # silu of pre-activations near -2^16: exp overflows to the exact limit 0
        ref = O.backward(x, W1, W2, ids, g, dO)["dg_fused"]
        got = O.backward_mxfp8(x, W1, W2, ids, g, dO)["dg"]
        # control: the same inputs quantised along the other axis lose bits
        swapped = O.backward_mxfp8(x, W1, W2, ids, g, dO, qdq=lambda v, axis: _qdq_any(v, 1 - axis))["dg"]
    # entries span many binades: compare each entry to itself
    maxrel = lambda a: float(np.max(np.abs(a - ref) / np.abs(ref)))
    assert np.all(np.isfinite(ref)) and np.all(ref != 0)
    assert maxrel(got) < 1e-12
    assert maxrel(swapped) > 1e-2


def test_power_of_two_upstream_scaling_is_exact():
    # the UE8M0 block scales absorb a power of two: every quantised operand
    # that carries dOut (dOut, dH, and through dH the weight gradients) scales
    # exactly, so every output does; a scale rule that is not a power of two,
    # or a rounding of the scale, breaks this.  Row counts that are not a
    # multiple of 32 exercise the zero-padded last row block.
    x, W1, W2, ids, g, dO = _case(T=45, d=64, f=32, E=2, k=1, seed=5)
    a = O.backward_mxfp8(x, W1, W2, ids, g, dO)
    b = O.backward_mxfp8(x, W1, W2, ids, g, 8.0 * dO)
    for name in ("dW1", "dW2", "dx", "dg"):
        np.testing.assert_array_equal(b[name], 8.0 * a[name])


def test_tokens_stay_separate_in_dgrad2_and_dgrad1():
    # dgrad2 (K = d) and dgrad1 (K = 2f) quantise within a row, so a token's
    # upstream row scaled by 2^12 scales its own dx and dg exactly and leaves
    # every other token's bit-identical; a block across rows would not
    x, W1, W2, ids, g, dO = _case(T=64, d=64, f=32, E=3, k=2, seed=6)
    t0 = 17
    dO2 = dO.copy()
    dO2[t0] *= 2.0 ** 12
    a = O.backward_mxfp8(x, W1, W2, ids, g, dO)
    b = O.backward_mxfp8(x, W1, W2, ids, g, dO2)
    others = np.arange(64) != t0
    np.testing.assert_array_equal(b["dx"][others], a["dx"][others])
    np.testing.assert_array_equal(b["dg"][others], a["dg"][others])
    np.testing.assert_array_equal(b["dx"][t0], 2.0 ** 12 * a["dx"][t0])
    np.testing.assert_array_equal(b["dg"][t0], 2.0 ** 12 * a["dg"][t0])


def test_weight_gradient_blocks_run_along_the_rows():
    # wgrad2 quantises dOut along the expert's rows, within one column: a
    # column of dOut scaled by 2^12 scales that column of every dW2 exactly and
    # leaves the other columns bit-identical; blocks along d would mix columns
    x, W1, W2, ids, g, dO = _case(T=70, d=64, f=32, E=3, k=2, seed=7)
    j = 5
    dO2 = dO.copy()
    dO2[:, j] *= 2.0 ** 12
    a = O.backward_mxfp8(x, W1, W2, ids, g, dO)
    b = O.backward_mxfp8(x, W1, W2, ids, g, dO2)
    cols = np.arange(64) != j
    np.testing.assert_array_equal(b["dW2"][:, :, cols], a["dW2"][:, :, cols])
    np.testing.assert_array_equal(b["dW2"][:, :, j], 2.0 ** 12 * a["dW2"][:, :, j])


def test_wgrad1_blocks_dh_along_the_rows():
    # row r of every W2 scaled by 2^12: dgrad2 (blocks within W2's rows) scales
    # column r of dA' exactly, so the gate and up columns r and f + r of dH
    # scale exactly; wgrad1 quantises dH along the rows, within a column, so
    # exactly those two columns of every dW1 scale and the rest stay
    # bit-identical; dW2 does not involve W2 at all
    x, W1, W2, ids, g, dO = _case(T=70, d=64, f=32, E=3, k=2, seed=8)
    r, f = 3, 32
    W2s = [w.copy() for w in W2]
    for w in W2s:
        w[r] *= 2.0 ** 12
    a = O.backward_mxfp8(x, W1, W2, ids, g, dO)
    b = O.backward_mxfp8(x, W1, W2s, ids, g, dO)
    cols = np.ones(2 * f, dtype=bool)
    cols[[r, f + r]] = False
    np.testing.assert_array_equal(b["dW1"][:, :, cols], a["dW1"][:, :, cols])
    np.testing.assert_array_equal(b["dW1"][:, :, ~cols], 2.0 ** 12 * a["dW1"][:, :, ~cols])
    np.testing.assert_array_equal(b["dW2"], a["dW2"])


# ---------------------------------------------------------------------------
# Every operand on its own.  For each quantised operand of the backward, an
# input on which that operand holds one power-of-two scale per 32-block along
# its contraction axis (and small integers) quantises losslessly there, so
# quantising only it reproduces the unquantised backward exactly; blocked
# along its other axis it mixes magnitudes 16 binades apart and loses bits.
# dH and g*A are computed, so their cases are built from one-hot token rows
# (x[t] = c_t e_i(t), dOut[t] = e_l(t)), top-1 routing (g = 1) and gate
# weights of at least 2^6, where sigmoid(H_gate) is exactly 1 in fp64: then
# SiLU(H_gate) = H_gate, dH_gate = dA * H_up and dH_up = dA * H_gate exactly.
# ---------------------------------------------------------------------------
def _ident(v, axis):
    return v


def _swapped(v, axis):
    return _qdq_any(v, 1 - axis)


def _binades(rng, shape):
    return np.ldexp(1.0, 8 * rng.choice([-1, 1], size=shape))


def _pow2(rng, shape, top=2):
    """+-2^j, j in [0, top]: products of a few stay exact in E4M3."""
    return rng.choice([-1, 1], size=shape) * np.ldexp(1.0, rng.integers(0, top + 1, size=shape))


def _onehot_rows(rng, T, n, scale):
    v = np.zeros((T, n))
    v[np.arange(T), rng.integers(0, n, size=T)] = scale
    return v


def _operand_case(op, seed):
    rng = np.random.default_rng(seed)
    T, d, f, E = 96, 64, 64, 3
    k = 2
    x = rng.standard_normal((T, d))
    W1 = [rng.standard_normal((d, 2 * f)) / 8 for _ in range(E)]
    W2 = [rng.standard_normal((f, d)) / 8 for _ in range(E)]
    dO = rng.standard_normal((T, d))
    if op == "fwd.x":          # [m, d] along d: a scale per row
        x = _grid(rng, (T, d)) * _binades(rng, (T, 1))
    elif op == "fwd.W1":       # [d, 2f] along d: a scale per column
        W1 = [_grid(rng, (d, 2 * f)) * _binades(rng, (1, 2 * f)) for _ in range(E)]
    elif op == "dgrad2.dO":    # [m, d] along d: a scale per row
        dO = _grid(rng, (T, d)) * _binades(rng, (T, 1))
    elif op == "dgrad2.W2":    # W2e [f, d] along d: a scale per row
        W2 = [_grid(rng, (f, d)) * _binades(rng, (f, 1)) for _ in range(E)]
    elif op == "dgrad1.W1":    # W1e [d, 2f] along 2f: a scale per row
        W1 = [_grid(rng, (d, 2 * f)) * _binades(rng, (d, 1)) for _ in range(E)]
    elif op == "wgrad1.X":     # [m, d] along the rows: a scale per column
        x = _grid(rng, (T, d)) * _binades(rng, (1, d))
    elif op == "wgrad2.dO":    # [m, d] along the rows: a scale per column
        dO = _grid(rng, (T, d)) * _binades(rng, (1, d))
    else:
        k = 1
        dO = _onehot_rows(rng, T, d, 1.0)
        W2 = [_pow2(rng, (f, d), 1) for _ in range(E)]
        if op == "wgrad2.gA":
            # A[t, j] = n[i, j] 2^s_j: a scale per column of g*A
            x = _onehot_rows(rng, T, d, 1.0)
            W1 = [np.concatenate([np.full((d, f), 64.0),
                                  _grid(rng, (d, f)) * _binades(rng, (1, f)) / 64.0], axis=1)
                  for _ in range(E)]
        elif op == "dgrad1.dH":
            # x[t] = c_t e_i with c_t = 2^8 or 2^-8, gate weights 2^14, up
            # weights +-2^j 2^-14, W2 +-2^j: dH_gate = c_t W2 up and dH_up =
            # c_t W2 2^14 (gate and up in separate 32-blocks): one scale per
            # row in each half
            c = _binades(rng, T)
            x = _onehot_rows(rng, T, d, 1.0) * c[:, None]
            W1 = [np.concatenate([np.full((d, f), 2.0 ** 14), _pow2(rng, (d, f)) * 2.0 ** -14], axis=1)
                  for _ in range(E)]
        elif op == "wgrad1.dH":
            # one scale per column: gate columns 2^(14 + 16 b_j), up columns
            # +-2^j 2^(-14 + 8 s_j); token rows all of scale 1
            x = _onehot_rows(rng, T, d, 1.0)
            gate = np.ldexp(1.0, 14 + 16 * rng.integers(0, 2, size=(1, f)))
            W1 = [np.concatenate([np.ones((d, 1)) * gate,
                                  _pow2(rng, (d, f)) * 2.0 ** -14 * _binades(rng, (1, f))], axis=1)
                  for _ in range(E)]
        else:
            raise ValueError(op)
    z = rng.standard_normal((T, E)).astype(np.float32)
    ids, g = O.route(z, k)
    return x, W1, W2, ids, g, dO


def _worst(got, ref):
    """Largest relative deviation over every output (exact zeros must stay)."""
    w = 0.0
    for name in ("dx", "dW1", "dW2", "dg"):
        a, b = got[name], ref[name]
        nz = b != 0
        if np.any(nz):
            w = max(w, float(np.max(np.abs(a[nz] - b[nz]) / np.abs(b[nz]))))
        if np.any(~nz):
            w = max(w, float(np.max(np.abs(a[~nz]))) / max(float(np.max(np.abs(b))), 1e-300))
    return w


@pytest.mark.filterwarnings("ignore:overflow encountered in exp")  # sigmoid / SiLU limits, exact
@pytest.mark.parametrize("op", O.BACKWARD_OPERANDS)
def test_quantisation_axis_of_each_backward_operand(op):
    x, W1, W2, ids, g, dO = _operand_case(op, seed=30 + O.BACKWARD_OPERANDS.index(op))
    ref = O.backward_mxfp8(x, W1, W2, ids, g, dO, qdq=_ident)
    assert all(np.all(np.isfinite(ref[n])) for n in ("dx", "dW1", "dW2", "dg"))
    got = O.backward_mxfp8(x, W1, W2, ids, g, dO, quantise=[op])
    assert _worst(got, ref) < 1e-12, op
    bad = O.backward_mxfp8(x, W1, W2, ids, g, dO, qdq=_swapped, quantise=[op])
    assert _worst(bad, ref) > 1e-2, op


def test_weight_gradient_row_blocks_start_at_each_expert_segment():
    # Reading: the weight gradients' 32-row blocks run from the start of each
    # expert's rows (in the stable expert order).  Top-1 routing with segment
    # lengths that are not multiples of 32; x scaled 2^8 / 2^-8 by the block
    # parity of its row's position in its expert's segment quantises
    # losslessly under that reading -- and the same construction keyed to the
    # global expert-ordered position (blocks straddling segments) does not.
    rng = np.random.default_rng(40)
    T, d, f, E = 150, 64, 32, 3
    z = rng.standard_normal((T, E)).astype(np.float32)
    ids, g = O.route(z, 1)
    counts, offsets, perm, inv = O.schedule(ids, E)
    assert np.any(offsets[1:E] % 32 != 0) and np.any(counts % 32 != 0)
    pos = np.empty(T, np.int64)
    seg = np.empty(T, np.int64)
    pos[perm] = np.arange(T)
    e_of = ids[:, 0]
    seg = pos - offsets[e_of]
    base = _grid(rng, (T, d))
    W1 = [rng.standard_normal((d, 2 * f)) / 8 for _ in range(E)]
    W2 = [rng.standard_normal((f, d)) / 8 for _ in range(E)]
    dO = rng.standard_normal((T, d))

    def dev(blockpos):
        x = base * np.ldexp(1.0, 8 * np.where((blockpos // 32) % 2 == 0, 1, -1))[:, None]
        ref = O.backward_mxfp8(x, W1, W2, ids, g, dO, qdq=_ident)["dW1"]
        got = O.backward_mxfp8(x, W1, W2, ids, g, dO, quantise=["wgrad1.X"])["dW1"]
        return float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))

    # lossless: the quantised X is X itself, so dW1 is the same bits; lossy:
    # the 2^-8 rows lose bits, visible far above fp64 rounding although they
    # weigh 2^-16 of the 2^8 rows in each sum
    assert dev(seg) == 0.0
    assert dev(pos) > 1e-13


def test_per_expert_variant_matches_the_full_backward():
    x, W1, W2, ids, g, dO = _case(T=50, d=64, f=32, E=4, k=2, seed=9)
    full = O.backward_mxfp8(x, W1, W2, ids, g, dO)
    part = O.backward_mxfp8_experts(x, W1, W2, ids, g, dO, [0, 2, 3])
    for e, (dW1, dW2, rows, dg_rows) in part.items():
        np.testing.assert_array_equal(dW1, full["dW1"][e])
        np.testing.assert_array_equal(dW2, full["dW2"][e])
        np.testing.assert_array_equal(dg_rows, full["dg"].reshape(-1)[rows])
