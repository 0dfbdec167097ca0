"""MXFP8 mode on the GPU against the oracle.

The quantisers (E4M3 codes + UE8M0 scale per 32 along K) must be bit-exact:
the weight quantiser, and the quantising gather's codes and scale tiles read
back from the workspace.  The codes GEMM1's epilogue writes for A come from
fp32 H (the oracle's from fp64 H of the same quantised operands): every scale
byte must match except where the block maximum sits within fp32 rounding of a
scale boundary, and every code within one E4M3 step, both counted.  The MXFP8
forward is compared with the oracle's forward on operands it quantises itself
(x along d, W1 along d, the SwiGLU output A along f, W2 along f): normwise
relative error <= 6e-2 on random inputs; on grid inputs whose blocks are
exact along the right axes (and 16 binades apart across them) every token
must be within 1e-2 (bf16 rounding of Y alone: 2e-3), so x or A blocked
along the wrong axis (0.37 and 1.0 on this case, checked on the CPU) or a
scale read for the wrong block (a 2^16 factor) fails.  The weights' axes are
pinned by the byte-exact weight quantiser: lost bits of a weight block sit
15 binades below its largest element, too small to show in any output.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_stable_gb300 import binding as B
from mixture_experts_layer_stable_gb300.configs import CONFIGS
from mixture_experts_layer_stable_gb300.inputs import make_inputs
from oracle import moe_oracle as O

from gpu_util import Layer, cfg_struct, padded_positions, with_config
from helpers import ExpertView, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL_MX = 6e-2


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield


def tile_scales(sc_rows_k):
    """Arrange scales [rows, K/32] (rows and K multiples of 128) into the
    library's 512-byte scale tiles (documented with moe_quantize_mxfp8)."""
    rows, nkb = sc_rows_k.shape
    r = np.arange(rows)[:, None]
    kb = np.arange(nkb)[None, :]
    off = ((r // 128) * (nkb // 4) + kb // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + kb % 4
    out = np.zeros(rows * nkb, np.uint8)
    out[off.reshape(-1)] = sc_rows_k.reshape(-1)
    return out


def quantize_weights(W):
    """[E, K, N] bf16 on the GPU -> (codes [E, N, K], scale tiles) via the C ABI."""
    E, K, N = W.shape
    q = torch.empty(E, N, K, dtype=torch.uint8, device="cuda")
    s = torch.empty(E * N * K // 32, dtype=torch.uint8, device="cuda")
    B.moe_quantize_mxfp8(W, E, K, N, q, s)
    return q, s


@pytest.mark.parametrize("E,K,N", [(2, 128, 128), (3, 256, 384)])
def test_weight_quantizer_bit_exact(E, K, N):
    g = torch.Generator().manual_seed(E * 1000 + K + N)
    mag = torch.exp(torch.randn(E, K // 32, 1, N, generator=g) * 3)  # per-block magnitudes
    W = torch.randn(E, K, N, generator=g) * mag.repeat_interleave(32, 1).reshape(E, K, N)
    W = W.to(torch.bfloat16)
    W[0, :32, 0] = 0.0                          # an all-zero block
    W[0, 32:64, 1] = 448.0                      # amax exactly 448 * 2^0
    W[0, 64:96, 2] = torch.tensor(2.0 ** -130)  # tiny block: scale clamps at 2^-127
    W[-1, :32, -1] = -3.0e38                    # huge block
    q, s = quantize_weights(W.cuda())
    Wn = W.float().numpy().astype(np.float64)
    for e in range(E):
        codes, _ = O.mxfp8_quantize(Wn[e], axis=0)          # codes [K, N]
        assert np.array_equal(q[e].cpu().numpy(), codes.T), e
    sc_all = np.concatenate([O.mxfp8_quantize(Wn[e], axis=0)[1].T for e in range(E)], 0)
    assert np.array_equal(s.cpu().numpy(), tile_scales(sc_all))


def _mx_forward_case(cfg, x_std=None, tokens=None, device_inputs=False):
    if device_inputs:
        dev = make_inputs(cfg, device="cuda", with_grad=False, x_std=x_std)
        logits = dev["logits"].cpu().numpy()
    else:
        host = make_inputs(cfg, with_grad=False, x_std=x_std)
        dev = {k: v.cuda() for k, v in host.items()}
        logits = host["logits"].numpy()
    L = Layer(cfg, cfg_struct(cfg, prec="mxfp8"))
    w1q, w1s = quantize_weights(dev["W1"])
    w2q, w2s = quantize_weights(dev["W2"])
    L.schedule(dev["logits"])
    out = L.forward(dev["x"], w1q, w2q, save=False, w1s=w1s, w2s=w2s)
    torch.cuda.synchronize()
    assert L.status() == 0
    ids, g = O.route(logits, cfg.k)
    assert np.array_equal(L.sched_np()["topk_ids"], ids)
    want = O.forward_mxfp8(to_np(dev["x"]), ExpertView(dev["W1"]), ExpertView(dev["W2"]), ids, g,
                           tokens)
    got = out.float().cpu().numpy()
    if tokens is not None:
        got = got[tokens]
    err = rel_err(got, want)
    print(f"mxfp8 forward rel err {err:.3e}")
    return err, got, dev, ids, g


@pytest.mark.parametrize("kw,x_std", [(dict(f=128), None), (dict(f=128), 1.0),
                                      (dict(f=256, d=256, T=300, E=6, k=3), 1.0)])
def test_mxfp8_forward_tiny(kw, x_std):
    cfg = with_config("tiny", prec="mxfp8", **kw)
    err, *_ = _mx_forward_case(cfg, x_std)
    assert err <= TOL_MX


def test_mxfp8_forward_balanced_shape():
    cfg = with_config("balanced", prec="mxfp8")
    toks = np.arange(0, 2048, 16)
    err, got, dev, ids, g = _mx_forward_case(cfg, tokens=toks)
    assert err <= TOL_MX
    # against the unquantised fp64 layer: the size of the quantisation error itself
    want = O.forward_tokens(to_np(dev["x"]), ExpertView(dev["W1"]), ExpertView(dev["W2"]), ids, g,
                            toks)
    assert rel_err(got, want) <= 0.15


@pytest.mark.slow
def test_kimi_mxfp8_forward_sampled():
    cfg = CONFIGS["kimi_mxfp8"]
    toks = np.sort(np.random.default_rng(3).choice(cfg.T, 24, replace=False))
    err, *_ = _mx_forward_case(cfg, tokens=toks, device_inputs=True)
    assert err <= TOL_MX


# ---------------------------------------------------------------- bytes
def _region(L, region):
    off, n = B.moe_workspace_region(L.c, region)
    return L.ws[off:off + n].cpu().numpy()


def _row_of_pad(L):
    """Flat routed row of every written padded position (-1: padding)."""
    s = L.sched_np()
    c = s["counts"].astype(np.int64)
    rp = int(((c + 127) // 128 * 128).sum())
    rop = np.full(rp, -1, np.int64)
    rop[padded_positions(c, s["offsets"])] = s["perm"]
    return rop


def _tile_index(rows, K):
    """Index into the scale-tile bytes of every (row, 32-block) of a [rows, K]
    operand (byte 16*(r%32) + 4*((r%128)//32) + kb%4 of tile (r//128, kb//4))."""
    r = np.arange(rows)[:, None]
    kb = np.arange(K // 32)[None, :]
    return ((r // 128) * (K // 128) + kb // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + kb % 4


def _untile(tiles, rows, K):
    return tiles[_tile_index(rows, K)]


def _mx_run(cfg, dev):
    L = Layer(cfg, cfg_struct(cfg, prec="mxfp8"))
    w1q, w1s = quantize_weights(dev["W1"])
    w2q, w2s = quantize_weights(dev["W2"])
    L.schedule(dev["logits"])
    L.forward(dev["x"], w1q, w2q, save=False, w1s=w1s, w2s=w2s)
    torch.cuda.synchronize()
    assert L.status() == 0
    return L


@pytest.mark.parametrize("name,kw", [("tiny", dict(f=128, d=256, T=300, E=6, k=3)),
                                     ("tiny", dict(f=128, d=256, T=99, E=40, k=32)),
                                     ("tiny", dict(f=128, d=256, T=77, E=3, k=1)),
                                     ("balanced", {})])
def test_gather_codes_and_scales_bit_exact(name, kw):
    cfg = with_config(name, prec="mxfp8", **kw)
    host = make_inputs(cfg, with_grad=False, x_std=1.0)
    # blocks of very different magnitude, an all-zero block and a tiny one
    host["x"][::7, :32] *= 2.0 ** 20
    host["x"][1::5, 32:64] = 0.0
    host["x"][2::9, 64:96] = 2.0 ** -120
    dev = {k: v.cuda() for k, v in host.items()}
    L = _mx_run(cfg, dev)
    rop = _row_of_pad(L)
    rp, d = len(rop), cfg.d
    codes = _region(L, B.MOE_WS_XQ_CODES)[:rp * d].reshape(rp, d)
    scales = _region(L, B.MOE_WS_XQ_SCALES)[:rp * d // 32]
    x = host["x"].float().numpy().astype(np.float64)
    src = np.where(rop[:, None] >= 0, x[np.maximum(rop, 0) // cfg.k], 0.0)
    want_c, want_s = O.mxfp8_quantize(src, axis=1)
    # every routed row's codes and scale bytes (padding rows are not written:
    # GEMM1 zeroes what it computes from them)
    real = rop >= 0
    assert np.array_equal(codes[real], want_c[real])
    got_s = _untile(scales, rp, d)
    assert np.array_equal(got_s[real], want_s[real])


def _ordinal(c):
    c = c.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


@pytest.mark.parametrize("name,kw,x_std", [("tiny", dict(f=128, d=256, T=300, E=6, k=3), 1.0),
                                           ("balanced", {}, None)])
def test_gemm1_quantised_a_within_one_step(name, kw, x_std):
    cfg = with_config(name, prec="mxfp8", **kw)
    host = make_inputs(cfg, with_grad=False, x_std=x_std)
    dev = {k: v.cuda() for k, v in host.items()}
    L = _mx_run(cfg, dev)
    rop = _row_of_pad(L)
    rp, f = len(rop), cfg.f
    codes = _region(L, B.MOE_WS_AQ_CODES)[:rp * f].reshape(rp, f)
    sc_t = _region(L, B.MOE_WS_AQ_SCALES)[:rp * f // 32]
    # the scale tiles back to [rows, f/32]
    r = np.arange(rp)[:, None]
    kb = np.arange(f // 32)[None, :]
    sc = sc_t[((r // 128) * (f // 128) + kb // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + kb % 4]
    real = np.nonzero(rop >= 0)[0]
    pad = np.nonzero(rop < 0)[0]
    assert np.all(codes[pad] == 0) and np.all(sc[pad] == 0)
    sample = real[np.linspace(0, len(real) - 1, min(len(real), 384)).astype(np.int64)]
    ids = L.sched_np()["topk_ids"].reshape(-1)
    x = host["x"].float().numpy().astype(np.float64)
    xq = O.mxfp8_dequantize(*O.mxfp8_quantize(x, 1), 1)
    W1 = ExpertView(dev["W1"])
    n_blocks = n_scale_diff = n_code_diff = n_codes = 0
    for e in np.unique(ids[rop[sample]]):
        rows = sample[ids[rop[sample]] == e]
        W1q = O.mxfp8_dequantize(*O.mxfp8_quantize(W1[e], 0), 0)
        H = xq[rop[rows] // cfg.k] @ W1q
        A = O.silu(H[:, :f]) * H[:, f:]
        wc, ws = O.mxfp8_quantize(A, axis=1)
        amax = np.abs(A).reshape(len(rows), f // 32, 32).max(-1)
        s_o = ws.astype(np.int64) - 127
        same = sc[rows] == ws
        # a scale may differ only where amax is within fp32 rounding of the
        # boundary 448 * 2^s between two scales
        near = np.abs(amax / (448.0 * np.ldexp(1.0, s_o - 1)) - 1) < 1e-5
        near |= np.abs(amax / (448.0 * np.ldexp(1.0, s_o)) - 1) < 1e-5
        assert np.all(same | near), (e, np.argwhere(~(same | near))[:4])
        n_blocks += same.size
        n_scale_diff += int((~same).sum())
        ok = np.repeat(same, 32, axis=1)
        dif = np.abs(_ordinal(codes[rows]) - _ordinal(wc))
        assert np.all(dif[ok] <= 1), e
        n_code_diff += int((dif[ok] > 0).sum())
        n_codes += int(ok.sum())
    print(f"A: {n_scale_diff}/{n_blocks} scale bytes differ, {n_code_diff}/{n_codes} codes one step apart")
    assert n_scale_diff <= max(2, n_blocks // 1000)
    assert n_code_diff <= max(8, n_codes // 1000)


def _grid_inputs(cfg, seed=0):
    """bf16 inputs whose MXFP8 blocks along each GEMM's contraction axis hold
    one power-of-two scale and small integers: x a scale per token row, W1 a
    scale per column (its K = d), W2 a scale per column (its K = f).  The
    scales are 2^8 or 2^-8 at random: across the other axis a block mixes
    magnitudes 16 binades apart, more than E4M3 keeps."""
    g = torch.Generator().manual_seed(seed)
    T, d, f, E = cfg.T, cfg.d, cfg.f, cfg.E

    def grid(*shape):
        return torch.randint(-7, 8, shape, generator=g).double()

    def binades(*shape):
        return torch.pow(2.0, 8.0 * (2 * torch.randint(0, 2, shape, generator=g) - 1).double())

    x = (grid(T, d) * binades(T, 1) * 2.0 ** -4).to(torch.bfloat16)
    W1 = (grid(E, d, 2 * f) * binades(E, 1, 2 * f) * 2.0 ** -8).to(torch.bfloat16)
    W2 = (grid(E, f, d) * binades(E, 1, d) * 2.0 ** -8).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g)
    return {"x": x, "W1": W1, "W2": W2, "logits": logits}


def test_mxfp8_forward_grid_inputs_per_token():
    cfg = with_config("tiny", prec="mxfp8", f=256, d=256, T=300, E=6, k=3)
    host = _grid_inputs(cfg)
    dev = {k: v.cuda() for k, v in host.items()}
    L = _mx_run(cfg, dev)
    ids, g = O.route(host["logits"].numpy(), cfg.k)
    assert np.array_equal(L.sched_np()["topk_ids"], ids)
    want = O.forward_mxfp8(to_np(host["x"]), ExpertView(host["W1"]), ExpertView(host["W2"]), ids, g)
    got = L.out.double().cpu().numpy()
    per_tok = np.linalg.norm(got - want, axis=1) / np.linalg.norm(want, axis=1)
    print(f"grid mxfp8 forward: worst token {per_tok.max():.2e}, normwise {rel_err(got, want):.2e}")
    assert np.all(np.isfinite(got))
    assert per_tok.max() <= 1e-2


def test_mxfp8_forward_bitwise_deterministic_over_10_runs():
    cfg = with_config("balanced", prec="mxfp8")
    dev = make_inputs(cfg, device="cuda", with_grad=False)
    L = Layer(cfg, cfg_struct(cfg, prec="mxfp8"))
    w1q, w1s = quantize_weights(dev["W1"])
    w2q, w2s = quantize_weights(dev["W2"])
    ref = None
    for _ in range(10):
        L.schedule(dev["logits"])
        L.forward(dev["x"], w1q, w2q, save=True, w1s=w1s, w2s=w2s)
        got = [L.out.clone(), L.saved["H"].clone(), L.saved["A"].clone()]
        if ref is None:
            ref = got
        for a, b in zip(ref, got):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert L.status() == 0
