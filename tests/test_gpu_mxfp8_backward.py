"""The MXFP8 backward on the GPU against the oracle (moe_backward_mxfp8).

Reading (the oracle's backward_mxfp8): every backward GEMM quantises both
operands along its own contraction dimension -- dgrad2 dOut and W2 along d,
dgrad1 dH and W1 along 2f, the weight gradients x, dH, g*A and dOut along the
expert's rows in blocks of 32 from the segment start.

* Quantised operands that come from the inputs are compared byte for byte
  with the oracle's quantiser: the weights quantised along their rows, dOut
  along d, x and dOut transposed along the rows (read back from the
  workspace with moe_workspace_region).
* dH (along 2f, and transposed along the rows) and g*A (transposed) are
  quantised in dgrad2's epilogue from fp32 values; the expected codes are the
  oracle's quantisation of the same quantities formed in fp64 from the GPU's
  own inputs to that step (its saved H and A, its quantised dOut and W2):
  every scale byte equal except where the block maximum sits within fp32
  rounding of a scale boundary, every code within one E4M3 step, both
  counted.
* Outputs and gradients against backward_mxfp8: normwise relative error
  <= 6e-2; bitwise identical over repeat runs.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_stable_gb300 import binding as B
from mixture_experts_layer_stable_gb300.inputs import make_inputs
from oracle import moe_oracle as O

from gpu_util import Layer, cfg_struct, padded_positions, with_config
from helpers import ExpertView, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL_MX = 6e-2


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield


def _tile_index(rows, nkb):
    """Byte of (row r, 32-block kb) in the 512-byte scale tiles of a [rows, 32 nkb] operand."""
    r = np.arange(rows)[:, None]
    kb = np.arange(nkb)[None, :]
    return ((r // 128) * (nkb // 4) + kb // 4) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + kb % 4


def _scales(buf, rows, K):
    return buf[_tile_index(rows, K // 32)]


def _region(L, region, shape=None):
    off, n = B.moe_workspace_region(L.c, region)
    a = L.ws[off:off + n].cpu().numpy()
    return a.reshape(shape) if shape is not None else a


class MxBackward:
    def __init__(self, cfg, dev):
        self.cfg = cfg
        E, d, f = cfg.E, cfg.d, cfg.f
        self.L = Layer(cfg, cfg_struct(cfg, prec="mxfp8"))
        # forward weights quantised along K (their first dimension), backward
        # weights along their rows (the other dimension)
        self.w1q = torch.empty(E, 2 * f, d, dtype=torch.uint8, device="cuda")
        self.w1s = torch.empty(E * 2 * f * d // 32, dtype=torch.uint8, device="cuda")
        self.w2q = torch.empty(E, d, f, dtype=torch.uint8, device="cuda")
        self.w2s = torch.empty(E * d * f // 32, dtype=torch.uint8, device="cuda")
        B.moe_quantize_mxfp8(dev["W1"], E, d, 2 * f, self.w1q, self.w1s)
        B.moe_quantize_mxfp8(dev["W2"], E, f, d, self.w2q, self.w2s)
        self.w1r = torch.empty(E, d, 2 * f, dtype=torch.uint8, device="cuda")
        self.w1rs = torch.empty(E * d * 2 * f // 32, dtype=torch.uint8, device="cuda")
        self.w2r = torch.empty(E, f, d, dtype=torch.uint8, device="cuda")
        self.w2rs = torch.empty(E * f * d // 32, dtype=torch.uint8, device="cuda")
        B.moe_quantize_mxfp8_rows(dev["W1"], E * d, 2 * f, self.w1r, self.w1rs)
        B.moe_quantize_mxfp8_rows(dev["W2"], E * f, d, self.w2r, self.w2rs)
        self.dev = dev
        L = self.L
        L.dW1 = torch.empty_like(dev["W1"])
        L.dW2 = torch.empty_like(dev["W2"])

    def run(self):
        L, dev = self.L, self.dev
        L.schedule(dev["logits"])
        L.forward(dev["x"], self.w1q, self.w2q, save=True, w1s=self.w1s, w2s=self.w2s)
        B.moe_backward_mxfp8(L.c, dev["dOut"], dev["x"], self.w1r, self.w1rs, self.w2r, self.w2rs,
                             L.sched, L.saved, L.dx, L.dW1, L.dW2, L.dtopk_w, L.dlogits, L.ws)
        torch.cuda.synchronize()
        assert L.status() == 0
        return L


def _padded_rows(L):
    s = L.sched_np()
    c = s["counts"].astype(np.int64)
    pc = (c + 127) // 128 * 128
    rp = int(pc.sum())
    rop = np.full(rp, -1, np.int64)
    rop[padded_positions(c, s["offsets"])] = s["perm"]
    poff = np.concatenate([[0], np.cumsum(pc)])
    return rop, poff


def test_weight_row_quantiser_bit_exact():
    g = torch.Generator().manual_seed(11)
    W = (torch.randn(3, 256, 384, generator=g) * torch.exp(torch.randn(3, 256, 12, 1, generator=g) * 3)
         .repeat_interleave(32, 3).reshape(3, 256, 384)).to(torch.bfloat16)
    W[0, 0, :32] = 0.0
    q = torch.empty(3, 256, 384, dtype=torch.uint8, device="cuda")
    s = torch.empty(3 * 256 * 384 // 32, dtype=torch.uint8, device="cuda")
    B.moe_quantize_mxfp8_rows(W.cuda(), 3 * 256, 384, q, s)
    codes, sc = O.mxfp8_quantize(W.double().numpy().reshape(768, 384), axis=1)
    assert np.array_equal(q.cpu().numpy().reshape(768, 384), codes)
    assert np.array_equal(_scales(s.cpu().numpy(), 768, 384), sc)


def _ordinal(c):
    c = c.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def _compare_codes(got_c, got_s, want_c, want_s, amax, what):
    """Scales equal except near a boundary; codes of equal-scale blocks within one step."""
    s_o = want_s.astype(np.int64) - 127
    same = got_s == want_s
    near = np.abs(amax / (448.0 * np.ldexp(1.0, s_o - 1)) - 1) < 1e-5
    near |= np.abs(amax / (448.0 * np.ldexp(1.0, s_o)) - 1) < 1e-5
    assert np.all(same | near), (what, int((~(same | near)).sum()))
    return same


@pytest.mark.parametrize("name,kw,x_std", [("tiny", dict(f=128, d=256, T=300, E=6, k=3), 1.0),
                                           ("balanced", {}, None)])
def test_backward_quantised_operands(name, kw, x_std):
    cfg = with_config(name, prec="mxfp8", passes="fwd+bwd", **kw)
    host = make_inputs(cfg, x_std=x_std)
    dev = {k: v.cuda() for k, v in host.items()}
    mb = MxBackward(cfg, dev)
    L = mb.run()
    rop, poff = _padded_rows(L)
    rp_total, Rp, d, f, k = len(rop), B.moe_saved_rows(L.c), cfg.d, cfg.f, cfg.k
    x = to_np(host["x"])
    dO = to_np(host["dOut"])
    real = rop >= 0
    xp = np.where(real[:, None], x[np.maximum(rop, 0) // k], 0.0)
    dyp = np.where(real[:, None], dO[np.maximum(rop, 0) // k], 0.0)
    # dOut along d: bit-exact
    c = _region(L, B.MOE_WS_DYQ_CODES, (Rp, d))[:rp_total]
    s = _scales(_region(L, B.MOE_WS_DYQ_SCALES), Rp, d)[:rp_total]
    wc, ws_ = O.mxfp8_quantize(dyp, axis=1)
    assert np.array_equal(c, wc) and np.array_equal(s, ws_)
    # x and dOut transposed along the rows (32-row blocks of the padded order,
    # which start every expert's segment): bit-exact
    for region, src in ((B.MOE_WS_XQT_CODES, xp), (B.MOE_WS_DYQT_CODES, dyp)):
        ct = _region(L, region, (d, Rp))[:, :rp_total]
        st = _scales(_region(L, region + 1), d, Rp)[:, :rp_total // 32]
        wc, ws_ = O.mxfp8_quantize(src, axis=0)
        assert np.array_equal(ct, wc.T), region
        assert np.array_equal(st, ws_.T), region
    # dH and g*A from the epilogue, on a sample of rows
    H = L.saved["H"].double().cpu().numpy()[:rp_total]
    A = L.saved["A"].double().cpu().numpy()[:rp_total]
    ids = L.sched_np()["topk_ids"].reshape(-1)
    gw = L.sched_np()["topk_w"].reshape(-1).astype(np.float64)
    g_pad = np.where(real, gw[np.maximum(rop, 0)], 0.0)
    dyq = O.mxfp8_dequantize(*O.mxfp8_quantize(dyp, 1), 1)
    dHq = _region(L, B.MOE_WS_DHQ_CODES, (Rp, 2 * f))[:rp_total]
    dHs = _scales(_region(L, B.MOE_WS_DHQ_SCALES), Rp, 2 * f)[:rp_total]
    dHqT = _region(L, B.MOE_WS_DHQT_CODES, (2 * f, Rp))[:, :rp_total]
    dHsT = _scales(_region(L, B.MOE_WS_DHQT_SCALES), 2 * f, Rp)[:, :rp_total // 32]
    gAqT = _region(L, B.MOE_WS_GAQT_CODES, (f, Rp))[:, :rp_total]
    gAsT = _scales(_region(L, B.MOE_WS_GAQT_SCALES), f, Rp)[:, :rp_total // 32]
    W2 = ExpertView(host["W2"])
    counts = L.sched_np()["counts"]
    n = {"blocks": 0, "scale_diff": 0, "codes": 0, "code_diff": 0}
    for e in np.nonzero(counts)[0][:: max(1, len(np.nonzero(counts)[0]) // 6)]:
        a, b = int(poff[e]), int(poff[e + 1])        # the expert's padded rows
        W2r = O.mxfp8_dequantize(*O.mxfp8_quantize(W2[e], 1), 1)
        dAp = dyq[a:b] @ W2r.T
        dHg, dHu = O.swiglu_backward(H[a:b, :f], H[a:b, f:], g_pad[a:b, None] * dAp)
        dH = np.concatenate([dHg, dHu], axis=1)
        gA = g_pad[a:b, None] * A[a:b]
        checks = [(dHq[a:b], dHs[a:b], dH, 1), (dHqT[:, a:b].T, dHsT[:, a // 32:b // 32].T, dH, 0),
                  (gAqT[:, a:b].T, gAsT[:, a // 32:b // 32].T, gA, 0)]
        for gc, gs, v, axis in checks:
            wc, ws_ = O.mxfp8_quantize(v, axis=axis)
            blk = np.abs(v).reshape(v.shape[0], -1, 32).max(-1) if axis == 1 else \
                np.abs(v).reshape(-1, 32, v.shape[1]).max(1)
            same = _compare_codes(gc, gs, wc, ws_, blk, (e, axis))
            ok = np.repeat(same, 32, axis=axis)
            dif = np.abs(_ordinal(gc) - _ordinal(wc))
            assert np.all(dif[ok] <= 1), (e, axis)
            n["blocks"] += same.size
            n["scale_diff"] += int((~same).sum())
            n["codes"] += int(ok.sum())
            n["code_diff"] += int((dif[ok] > 0).sum())
    print("mxfp8 backward epilogue quantisation:", n)
    assert n["scale_diff"] <= max(2, n["blocks"] // 1000)
    assert n["code_diff"] <= max(8, n["codes"] // 1000)


def _against_oracle(cfg, host, L, tokens=None, experts=None):
    x, dO = to_np(host["x"]), to_np(host["dOut"])
    ids, g = O.route(host["logits"].numpy(), cfg.k)
    assert np.array_equal(L.sched_np()["topk_ids"], ids)
    want = O.backward_mxfp8(x, ExpertView(host["W1"]), ExpertView(host["W2"]), ids, g, dO)
    errs = {"dx": rel_err(L.dx.double().cpu().numpy(), want["dx"]),
            "dW1": rel_err(L.dW1.double().cpu().numpy(), want["dW1"]),
            "dW2": rel_err(L.dW2.double().cpu().numpy(), want["dW2"]),
            "dg": rel_err(L.dtopk_w.cpu().numpy().reshape(cfg.T, cfg.k), want["dg"]),
            "dlogits": rel_err(L.dlogits.cpu().numpy(), want["dlogits"])}
    print("mxfp8 backward vs oracle:", {k: f"{v:.2e}" for k, v in errs.items()})
    return errs


@pytest.mark.parametrize("kw,x_std", [(dict(f=128, d=256, T=300, E=6, k=3), 1.0),
                                      (dict(f=128, d=128, T=64, E=8, k=2), None),
                                      (dict(f=256, d=384, T=1, E=8, k=8), 1.0)])
def test_mxfp8_backward_tiny(kw, x_std):
    cfg = with_config("tiny", prec="mxfp8", passes="fwd+bwd", **kw)
    host = make_inputs(cfg, x_std=x_std)
    dev = {k: v.cuda() for k, v in host.items()}
    L = MxBackward(cfg, dev).run()
    errs = _against_oracle(cfg, host, L)
    assert all(v <= TOL_MX for v in errs.values()), errs
    counts = L.sched_np()["counts"]
    for e in np.nonzero(counts == 0)[0]:
        assert torch.count_nonzero(L.dW1[e]) == 0 and torch.count_nonzero(L.dW2[e]) == 0


def test_mxfp8_backward_balanced_shape():
    cfg = with_config("balanced", prec="mxfp8", passes="fwd+bwd")
    host = make_inputs(cfg)
    dev = {k: v.cuda() for k, v in host.items()}
    L = MxBackward(cfg, dev).run()
    errs = _against_oracle(cfg, host, L)
    assert all(v <= TOL_MX for v in errs.values()), errs


def test_mxfp8_backward_bitwise_deterministic():
    cfg = with_config("balanced", prec="mxfp8", passes="fwd+bwd")
    dev = make_inputs(cfg, device="cuda")
    mb = MxBackward(cfg, dev)
    ref = None
    for _ in range(5):
        L = mb.run()
        got = [t.clone() for t in (L.dx, L.dW1, L.dW2, L.dtopk_w, L.dlogits)]
        if ref is None:
            ref = got
        for a, b in zip(ref, got):
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b)


@pytest.mark.slow
def test_kimi_mxfp8_backward_sampled():
    cfg = with_config("kimi_bwd", prec="mxfp8")
    dev = make_inputs(cfg, device="cuda")
    L = MxBackward(cfg, dev).run()
    ids, g = O.route(dev["logits"].cpu().numpy(), cfg.k)
    assert np.array_equal(L.sched_np()["topk_ids"], ids)
    counts = L.sched_np()["counts"]
    nz = np.nonzero(counts)[0]
    small = nz[np.argmin(counts[nz])]
    experts = [int(np.argsort(counts)[-3]), int(small), int(nz[len(nz) // 2])]
    ex = O.backward_mxfp8_experts(to_np(dev["x"]), ExpertView(dev["W1"]), ExpertView(dev["W2"]), ids, g,
                                  to_np(dev["dOut"]), experts)
    dg = L.dtopk_w.cpu().numpy()
    for e in experts:
        dW1, dW2, rows, dg_rows = ex[e]
        assert rel_err(L.dW1[e].double().cpu().numpy(), dW1) <= TOL_MX, e
        assert rel_err(L.dW2[e].double().cpu().numpy(), dW2) <= TOL_MX, e
        assert rel_err(dg[rows], dg_rows) <= TOL_MX, e
    empty = np.nonzero(counts == 0)[0]
    if len(empty):
        assert torch.count_nonzero(L.dW1[int(empty[0])]) == 0
