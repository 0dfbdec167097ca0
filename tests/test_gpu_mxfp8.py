"""MXFP8 mode on the GPU against the oracle.

The quantiser (E4M3 codes + UE8M0 scale per 32 along K) must be bit-exact.
The MXFP8 forward is compared with the oracle's forward on operands it
quantises itself (x along d, W1 along d, the SwiGLU output A along f, W2 along
f): normwise relative error <= 6e-2.  The GPU quantises A from fp32 H while
the oracle quantises from fp64 H, so codes next to a rounding boundary may
differ by one step; that and the bf16 rounding of Y bound the error.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_stable_gb300 import binding as B
from mixture_experts_layer_stable_gb300.configs import CONFIGS
from mixture_experts_layer_stable_gb300.inputs import make_inputs
from oracle import moe_oracle as O

from gpu_util import Layer, cfg_struct, with_config
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
