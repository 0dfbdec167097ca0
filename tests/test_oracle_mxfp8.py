"""Pins for the oracle's MXFP8 quantiser (activation quantisation on the
dispatch / SwiGLU data path, leiphone "MoK..." 02; the BF16 and MXFP8 modes of
Marktechpost "Cursor开源MoK..." three design decisions).  Block format read
as OCP MX: 32 elements share a UE8M0 scale, elements are FP8 E4M3."""
import numpy as np
import torch

from oracle import moe_oracle as O


def _all_bf16_finite():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    v = bits.float()
    return v[torch.isfinite(v)]


def test_e4m3_encode_matches_torch_cast_on_every_bf16_in_range():
    v = _all_bf16_finite()
    v = v[v.abs() <= 464.0]
    got = O.e4m3_encode(v.double().numpy())
    want = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_e4m3_saturates_and_decodes():
    assert O.e4m3_encode(np.array([500.0, -1e6, 448.0]))[:].tolist() == [0x7E, 0xFE, 0x7E]
    codes = np.arange(256)
    dec = O.e4m3_decode(codes)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(dec), nan)
    assert np.array_equal(dec[~nan], ref[~nan])
    # round trip on every finite code (sign of zero kept)
    fin = codes[~nan]
    assert np.array_equal(O.e4m3_encode(dec[~nan]), fin)


def test_e4m3_ties_to_even_and_subnormals():
    cases = {1.0 + 1 / 16: 0x38, 1.0 + 3 / 16: 0x3A, 1.5 * 2 ** -9: 0x02, 0.5 * 2 ** -9: 0x00,
             2.5 * 2 ** -9: 0x02, 2 ** -6: 0x08, 7 * 2 ** -9: 0x07, 7.5 * 2 ** -9: 0x08,
             -0.0: 0x80, -(0.25 * 2 ** -9): 0x80}
    for v, c in cases.items():
        assert int(O.e4m3_encode(np.array([v]))[0]) == c, (v, c)


def test_scale_rule_closed_forms():
    for s in (-20, -3, 0, 5, 40):
        blk = np.zeros(32)
        blk[3] = 448.0 * 2.0 ** s            # exactly representable at scale s
        blk[4] = -1.0 * 2.0 ** s
        c, sc = O.mxfp8_quantize(blk)
        assert int(sc[0]) == s + 127 and int(c[3]) == 0x7E and int(c[4]) == 0xB8
        blk[3] = 449.0 * 2.0 ** s            # just above -> next scale, no saturation
        c, sc = O.mxfp8_quantize(blk)
        assert int(sc[0]) == s + 128
        blk[3] = 2.0 ** (s + 9)              # 512 * 2^s: mantissa 0.5 -> s+1 as well
        c, sc = O.mxfp8_quantize(blk)
        assert int(sc[0]) == s + 128 and int(c[3]) == 0x78
    c, sc = O.mxfp8_quantize(np.zeros((2, 64)))
    assert np.all(sc == 0) and np.all(c == 0)
    tiny = np.full(32, 2.0 ** -140)         # scale clamps at 2^-127
    c, sc = O.mxfp8_quantize(tiny)
    assert int(sc[0]) == 0 and int(c[0]) == O.e4m3_encode(np.array([2.0 ** -13]))[0]


def test_quantise_error_bound_and_axis():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((16, 96)) * np.exp(rng.standard_normal((16, 1)) * 4)
    c, sc = O.mxfp8_quantize(v, axis=1)
    dq = O.mxfp8_dequantize(c, sc, axis=1)
    blk = v.reshape(16, 3, 32)
    s = sc.astype(np.int64) - 127
    amax = np.abs(blk).max(-1)
    assert np.all(amax <= 448 * 2.0 ** s) and np.all(amax > 224 * 2.0 ** s)
    y = np.abs(blk) * 2.0 ** (-s[..., None])
    e = np.maximum(np.floor(np.log2(np.maximum(y, 1e-300))), -6)
    bound = 2.0 ** (e - 4) * 2.0 ** s[..., None]
    assert np.all(np.abs(dq.reshape(16, 3, 32) - blk) <= bound * (1 + 1e-12))
    c0, s0 = O.mxfp8_quantize(v.T, axis=0)
    assert np.array_equal(c0, c.T) and np.array_equal(s0, sc.T)
