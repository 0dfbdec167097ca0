"""The persistent ring forward (SM split into gather and GEMM CTAs, minibatch
windows handed over through device counters, leiphone "MoK..." section 02).

It computes the same tiles in the same K order as the kernel-chain forward, so
its outputs and saved activations must be bitwise identical to that path, for
every minibatch size and ring depth (the results do not depend on the
minibatch), and within 1e-2 of the oracle.  A withheld window must end in
MOE_ERR_TIMEOUT through the bounded waits, leaving the context usable.
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

HDR_INJECT = 8  # workspace header word of the wait test hook (int32 index)


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield


def _run(cfg, dev, mb=0, slots=0, gather=0, save=True, backward=False):
    L = Layer(cfg, cfg_struct(cfg, minibatch_rows=mb, ring_slots=slots, gather_ctas=gather))
    L.schedule(dev["logits"])
    L.forward(dev["x"], dev["W1"], dev["W2"], save=save)
    if backward:
        L.backward(dev["dOut"], dev["x"], dev["W1"], dev["W2"])
    torch.cuda.synchronize()
    assert L.status() == 0
    return L


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _rows_written(L):
    """Rows of the saved activations the forward writes: the padded total."""
    c = L.sched["counts"].cpu().numpy().astype(np.int64)
    return int(((c + 127) // 128 * 128).sum())


@pytest.mark.parametrize("name,kw,mbs", [
    ("tiny", {}, [(128, 2), (256, 3)]),
    ("tiny", dict(f=192, d=256, T=300), [(128, 2), (384, 2)]),
    ("tiny", dict(T=1, k=8), [(128, 2)]),
    ("balanced", {}, [(1024, 2), (512, 4), (2368, 2), (8192, 2)]),
])
def test_ring_equals_chain_bitwise(name, kw, mbs):
    cfg = with_config(name, **kw)
    inp = make_inputs(cfg, x_std=1.0 if name == "tiny" else None)
    dev = {k: v.cuda() for k, v in inp.items()}
    ref = _run(cfg, dev)
    for mb, slots in mbs:
        for gather in (0, 3):  # a gather warp in every CTA; three gather-only CTAs
            L = _run(cfg, dev, mb, slots, gather)
            assert _same(L.out, ref.out), (mb, slots, gather)
            rp = _rows_written(ref)
            assert _same(L.saved["H"][:rp], ref.saved["H"][:rp])
            assert _same(L.saved["A"][:rp], ref.saved["A"][:rp])
    ids, g = O.route(inp["logits"].numpy(), cfg.k)
    want, _ = O.forward(to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), ids, g)
    assert rel_err(ref.out.float().cpu().numpy(), want) <= 1e-2


def test_ring_two_tile_units_and_thin_tiles_bitwise():
    # hidden 5120 and enough rows (8 units of 256 rows per SM): the ring takes
    # two 128-row tiles of one expert per unit, and tiles of at most 32 rows
    # run thin in GEMM1 and GEMM2; a hot expert spans several windows, a few
    # experts get 1-40 rows, one none
    cfg = with_config("tiny", T=10240, d=5120, f=2048, E=12, k=2)
    inp = make_inputs(cfg, x_std=1.0)
    z = inp["logits"]
    z[:, 0] += 6.0                   # hot: most tokens' first choice
    z[:, 11] -= 40.0                 # never chosen
    for e, lo, hi in ((8, 0, 1), (9, 1, 18), (10, 18, 58)):  # exactly tokens [lo, hi) pick e
        z[:, e] -= 40.0
        z[lo:hi, e] += 80.0
    dev = {k: v.cuda() for k, v in inp.items()}
    ref = _run(cfg, dev)
    counts = ref.sched["counts"].cpu().numpy()
    assert counts[11] == 0 and counts[8] == 1 and counts[9] == 17 and counts[10] == 40
    for mb, slots in ((1024, 3), (384, 4)):
        L = _run(cfg, dev, mb, slots)
        assert _same(L.out, ref.out), (mb, slots)
        rp = _rows_written(ref)
        assert _same(L.saved["H"][:rp], ref.saved["H"][:rp])
        assert _same(L.saved["A"][:rp], ref.saved["A"][:rp])
    # the chain against the oracle on the light experts' tokens and a sample
    ids, g = O.route(inp["logits"].numpy(), cfg.k)
    toks = np.concatenate([np.arange(58), np.linspace(58, cfg.T - 1, 40).astype(np.int64)])
    want = O.forward_tokens(to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), ids, g, toks)
    assert rel_err(ref.out.float().cpu().numpy()[toks], want) <= 1e-2


def test_ring_forward_then_backward():
    cfg = with_config("tiny", T=256)
    inp = make_inputs(cfg, x_std=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    ref = _run(cfg, dev, backward=True)
    L = _run(cfg, dev, 128, 2, backward=True)
    for a, b in ((L.dx, ref.dx), (L.dW1, ref.dW1), (L.dW2, ref.dW2)):
        assert _same(a, b)
    assert torch.equal(L.dtopk_w, ref.dtopk_w)


def test_ring_inference_without_saved():
    cfg = with_config("balanced")
    dev = {k: v.cuda() for k, v in make_inputs(cfg, with_grad=False).items()}
    ref = _run(cfg, dev, save=False)
    L = _run(cfg, dev, 1024, 2, save=False)
    assert _same(L.out, ref.out)


@pytest.mark.parametrize("gather", [0, 8])
def test_ring_withheld_window_times_out_cleanly(gather):
    cfg = with_config("balanced")
    dev = {k: v.cuda() for k, v in make_inputs(cfg, with_grad=False).items()}
    c = cfg_struct(cfg, minibatch_rows=1024, ring_slots=2, gather_ctas=gather)
    L = Layer(cfg, c)
    L.schedule(dev["logits"])
    hdr = L.ws[:64 * 4].view(torch.int32)
    hdr[HDR_INJECT] = 3       # window 2's arrival is never released
    hdr[HDR_INJECT + 1] = 50  # bounded waits give up after 50 ms
    L.forward(dev["x"], dev["W1"], dev["W2"])
    assert L.status() == B.MOE_ERR_TIMEOUT
    # the context is still usable and a normal call succeeds afterwards
    L.schedule(dev["logits"])
    L.forward(dev["x"], dev["W1"], dev["W2"])
    torch.cuda.synchronize()
    assert L.status() == 0
    ref = _run(cfg, dev)
    assert _same(L.out, ref.out)


def test_ring_argument_errors_return_before_gpu_work():
    # rejected on the host: an MXFP8 ring forward without weight scales, a
    # BF16 one with scales, an SM split that leaves no compute CTA
    cfg = with_config("tiny", f=128, prec="mxfp8")
    dev = {k: v.cuda() for k, v in make_inputs(cfg, with_grad=False).items()}
    c = cfg_struct(cfg, minibatch_rows=128, ring_slots=2)
    L = Layer(cfg, c)
    L.schedule(dev["logits"])
    w = torch.zeros(64, dtype=torch.uint8, device="cuda")  # never read: the checks come first
    with pytest.raises(B.MoeError) as ei:
        B.moe_forward(c, dev["x"], w, None, w, None, L.sched, L.out, None, L.ws)
    assert ei.value.code == B.MOE_ERR_INVALID_ARG
    cb = with_config("tiny", f=128)
    c2 = cfg_struct(cb, minibatch_rows=128, ring_slots=2)
    L2 = Layer(cb, c2)
    with pytest.raises(B.MoeError) as ei:
        B.moe_forward(c2, dev["x"], w, w, w, w, L2.sched, L2.out, None, L2.ws)
    assert ei.value.code == B.MOE_ERR_INVALID_ARG
    c3 = cfg_struct(cb, minibatch_rows=128, ring_slots=2, gather_ctas=100000)
    L3 = Layer(cb, c3)
    with pytest.raises(B.MoeError) as ei:
        B.moe_forward(c3, dev["x"], w, None, w, None, L3.sched, L3.out, None, L3.ws)
    assert ei.value.code == B.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.slow
def test_kimi_zipf_ring_equals_chain():
    cfg = CONFIGS["kimi_zipf"]
    dev = make_inputs(cfg, device="cuda", with_grad=False)
    ref = _run(cfg, dev, save=False)
    for mb, gather in ((512, 0), (2368, 0), (4096, 0), (1024, 9)):
        L = _run(cfg, dev, mb, 4, gather, save=False)
        assert _same(L.out, ref.out), (mb, gather)


# ---------------------------------------------------------------- MXFP8
def _quantized(dev):
    out = {}
    for name in ("W1", "W2"):
        W = dev[name]
        E, K, N = W.shape
        q = torch.empty(E, N, K, dtype=torch.uint8, device="cuda")
        s = torch.empty(E * N * K // 32, dtype=torch.uint8, device="cuda")
        B.moe_quantize_mxfp8(W, E, K, N, q, s)
        out[name] = (q, s)
    return out


def _run_mx(cfg, dev, wq, mb=0, slots=0, gather=0, save=True):
    L = Layer(cfg, cfg_struct(cfg, prec="mxfp8", minibatch_rows=mb, ring_slots=slots, gather_ctas=gather))
    L.schedule(dev["logits"])
    L.forward(dev["x"], wq["W1"][0], wq["W2"][0], save=save, w1s=wq["W1"][1], w2s=wq["W2"][1])
    torch.cuda.synchronize()
    assert L.status() == 0
    return L


@pytest.mark.parametrize("name,kw,mbs", [
    ("tiny", dict(f=128, d=256, T=300, E=6, k=3), [(128, 2), (256, 3)]),
    ("tiny", dict(f=256, d=384, T=1, k=8), [(128, 2)]),
    ("balanced", {}, [(1024, 2), (512, 4), (2368, 2), (8192, 2)]),
])
def test_mxfp8_ring_equals_chain_bitwise(name, kw, mbs):
    cfg = with_config(name, prec="mxfp8", **kw)
    inp = make_inputs(cfg, with_grad=False, x_std=1.0 if name == "tiny" else None)
    dev = {k: v.cuda() for k, v in inp.items()}
    wq = _quantized(dev)
    ref = _run_mx(cfg, dev, wq)
    rp = _rows_written(ref)
    for mb, slots in mbs:
        for gather in (0, 3):
            L = _run_mx(cfg, dev, wq, mb, slots, gather)
            assert _same(L.out, ref.out), (mb, slots, gather)
            assert _same(L.saved["H"][:rp], ref.saved["H"][:rp])
            assert _same(L.saved["A"][:rp], ref.saved["A"][:rp])
    L = _run_mx(cfg, dev, wq, mbs[0][0], mbs[0][1], save=False)  # inference: no bf16 A / H
    assert _same(L.out, ref.out)
    ids, g = O.route(inp["logits"].numpy(), cfg.k)
    toks = np.arange(0, cfg.T, max(1, cfg.T // 128))
    want = O.forward_mxfp8(to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), ids, g, toks)
    assert rel_err(ref.out.float().cpu().numpy()[toks], want) <= 6e-2


def test_mxfp8_ring_bitwise_deterministic_over_10_runs():
    cfg = with_config("balanced", prec="mxfp8")
    dev = make_inputs(cfg, device="cuda", with_grad=False)
    wq = _quantized(dev)
    L = Layer(cfg, cfg_struct(cfg, prec="mxfp8", minibatch_rows=1024, ring_slots=4))
    ref = None
    for _ in range(10):
        L.schedule(dev["logits"])
        L.forward(dev["x"], wq["W1"][0], wq["W2"][0], save=False, w1s=wq["W1"][1], w2s=wq["W2"][1])
        out = L.out.clone()
        if ref is None:
            ref = out
        assert _same(out, ref)
    assert L.status() == 0


@pytest.mark.slow
def test_kimi_mxfp8_ring_equals_chain():
    cfg = CONFIGS["kimi_mxfp8"]
    dev = make_inputs(cfg, device="cuda", with_grad=False)
    wq = _quantized(dev)
    ref = _run_mx(cfg, dev, wq, save=False)
    for mb, gather in ((1024, 0), (2368, 0), (1024, 9)):
        L = _run_mx(cfg, dev, wq, mb, 4, gather, save=False)
        assert _same(L.out, ref.out), (mb, gather)
