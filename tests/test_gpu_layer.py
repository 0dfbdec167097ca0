"""GPU parity of the MoE layer against the fp64 oracle, through the C ABI.

Bars: routing ids, counts, offsets, perm and inv bit-exact; routing weights
within 4e-6 relative (fp32 softmax of <= 32 terms: a few ulp); outputs and
gradients within a normwise relative error of 1e-2 (BF16 path: H, A and Y are
rounded to bf16 once each, fp32 accumulation); bitwise identical outputs
across repeat runs.
"""
import math

import numpy as np
import pytest
import torch

from mixture_experts_layer_stable_gb300.configs import CONFIGS
from mixture_experts_layer_stable_gb300.inputs import make_inputs
from oracle import moe_oracle as O

from gpu_util import Layer, padded_positions, with_config
from helpers import ExpertView, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2
TOL_W = 4e-6


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    torch.manual_seed(0)
    yield


def _check_schedule(L, logits_cpu, k):
    E = logits_cpu.shape[1]
    ids, g = O.route(logits_cpu.numpy(), k)
    counts, offsets, perm, inv = O.schedule(ids, E)
    s = L.sched_np()
    assert np.array_equal(s["topk_ids"], ids)
    assert np.array_equal(s["counts"], counts)
    assert np.array_equal(s["offsets"], offsets)
    assert np.array_equal(s["perm"], perm)
    assert np.array_equal(s["inv"], inv)
    np.testing.assert_allclose(s["topk_w"], g, rtol=TOL_W, atol=0)
    return ids, g


@pytest.mark.parametrize("name", ["tiny", "balanced", "kimi_zipf", "kimi_mxfp8", "kimi_bwd",
                                  "local_slice"])
def test_schedule_bit_exact(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg, parts=("logits",))
    L = Layer(cfg)
    L.schedule(inp["logits"].cuda())
    _check_schedule(L, inp["logits"], cfg.k)
    assert L.status() == 0


@pytest.mark.parametrize("T,E,k,kind", [
    (1, 8, 8, "normal"), (100, 5, 1, "normal"), (333, 1, 1, "normal"), (130, 16, 4, "ties"),
    (257, 64, 8, "hot"), (70, 1000, 32, "normal"), (64, 256, 8, "allsame")])
def test_schedule_edge_cases(T, E, k, kind):
    g = torch.Generator().manual_seed(T * 7 + E)
    z = torch.randn(T, E, generator=g)
    if kind == "ties":
        z = torch.randint(-2, 3, (T, E), generator=g).float()
        z[z == 0] = -0.0
        z[::3][z[::3] == -0.0] = 0.0
    elif kind == "hot":
        z[:, 3] += 50.0
    elif kind == "allsame":
        z = torch.zeros(T, E)
    cfg = with_config("tiny", T=T, E=E, k=k)
    L = Layer(cfg)
    L.schedule(z.contiguous().cuda())
    _check_schedule(L, z, k)


def _run_forward(cfg, inp):
    L = Layer(cfg)
    dev = {k: v.cuda() for k, v in inp.items()}
    L.schedule(dev["logits"])
    out = L.forward(dev["x"], dev["W1"], dev["W2"], save=True)
    torch.cuda.synchronize()
    assert L.status() == 0
    return L, dev, out.float().cpu().numpy()


@pytest.mark.parametrize("name,kw,x_std", [
    ("tiny", {}, None), ("tiny", {}, 1.0), ("tiny", dict(f=192, d=256), 1.0),
    ("tiny", dict(d=64, f=128, E=3, k=3, T=200), 1.0), ("tiny", dict(T=1, k=8), 1.0),
    # the token-order gather at its widest and narrowest fan-out
    ("tiny", dict(T=97, E=40, k=32), 1.0), ("tiny", dict(T=133, E=5, k=1), 1.0),
    ("balanced", {}, None)])
def test_forward_full(name, kw, x_std):
    cfg = with_config(name, **kw)
    inp = make_inputs(cfg, x_std=x_std)
    L, dev, out = _run_forward(cfg, inp)
    ids, g = _check_schedule(L, inp["logits"], cfg.k)
    want, _ = O.forward(to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), ids, g)
    assert rel_err(out, want) <= TOL_BF16
    # saved H rows are X W1 of the row's expert (documented saved layout)
    s = L.sched_np()
    pp = padded_positions(s["counts"], s["offsets"])
    H = L.saved["H"].float().cpu().numpy()
    x = to_np(inp["x"])
    for p in list(range(0, len(pp), max(1, len(pp) // 16)))[:16]:
        r = int(s["perm"][p])
        e = int(ids.reshape(-1)[r])
        h = x[r // cfg.k] @ to_np(inp["W1"][e])
        assert rel_err(H[pp[p]], h) <= TOL_BF16


def test_forward_skewed_one_hot_expert():
    cfg = with_config("tiny", T=512, E=8, k=2)
    inp = make_inputs(cfg, x_std=1.0)
    inp["logits"][:, 5] += 30.0   # every token routes to expert 5 first
    inp["logits"][:, 2] -= 30.0   # expert 2 never chosen
    L, dev, out = _run_forward(cfg, inp)
    ids, g = _check_schedule(L, inp["logits"], cfg.k)
    assert L.sched_np()["counts"][5] == 512 and L.sched_np()["counts"][2] == 0
    want, _ = O.forward(to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), ids, g)
    assert rel_err(out, want) <= TOL_BF16


def _backward_case(cfg, x_std=None, logits_fn=None):
    inp = make_inputs(cfg, x_std=x_std)
    if logits_fn:
        logits_fn(inp["logits"])
    L, dev, out = _run_forward(cfg, inp)
    L.backward(dev["dOut"], dev["x"], dev["W1"], dev["W2"])
    torch.cuda.synchronize()
    assert L.status() == 0
    ids, g = _check_schedule(L, inp["logits"], cfg.k)
    want = O.backward(to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), ids, g,
                      to_np(inp["dOut"]))
    return L, want


@pytest.mark.parametrize("kw,x_std", [({}, None), ({}, 1.0), (dict(f=192, d=256, T=300), 1.0),
                                      (dict(T=97, E=40, k=32), 1.0), (dict(T=133, E=5, k=1), 1.0),
                                      (dict(T=1, k=8), 1.0), (dict(d=64, E=3, k=3), 1.0)])
def test_backward_tiny(kw, x_std):
    cfg = with_config("tiny", **kw)
    L, want = _backward_case(cfg, x_std)
    assert rel_err(L.dx.float().cpu().numpy(), want["dx"]) <= TOL_BF16
    assert rel_err(L.dW1.float().cpu().numpy(), want["dW1"]) <= TOL_BF16
    assert rel_err(L.dW2.float().cpu().numpy(), want["dW2"]) <= TOL_BF16
    assert rel_err(L.dtopk_w.cpu().numpy().reshape(cfg.T, cfg.k), want["dg"]) <= TOL_BF16
    assert rel_err(L.dlogits.cpu().numpy(), want["dlogits"]) <= TOL_BF16
    counts = L.sched_np()["counts"]
    for e in np.nonzero(counts == 0)[0]:
        assert torch.count_nonzero(L.dW1[e]) == 0 and torch.count_nonzero(L.dW2[e]) == 0


def test_backward_balanced_shape():
    cfg = with_config("balanced", passes="fwd+bwd")
    L, want = _backward_case(cfg)
    assert rel_err(L.dx.float().cpu().numpy(), want["dx"]) <= TOL_BF16
    assert rel_err(L.dW1.float().cpu().numpy(), want["dW1"]) <= TOL_BF16
    assert rel_err(L.dW2.float().cpu().numpy(), want["dW2"]) <= TOL_BF16
    assert rel_err(L.dtopk_w.cpu().numpy().reshape(cfg.T, cfg.k), want["dg"]) <= TOL_BF16
    assert rel_err(L.dlogits.cpu().numpy(), want["dlogits"]) <= TOL_BF16


def test_backward_empty_and_hot_experts():
    cfg = with_config("tiny", T=256, E=8, k=2)

    def skew(z):
        z[:, 1] += 30.0
        z[:, 6] -= 30.0

    L, want = _backward_case(cfg, 1.0, skew)
    assert L.sched_np()["counts"][6] == 0
    assert rel_err(L.dW1.float().cpu().numpy(), want["dW1"]) <= TOL_BF16
    assert rel_err(L.dW2.float().cpu().numpy(), want["dW2"]) <= TOL_BF16
    assert rel_err(L.dx.float().cpu().numpy(), want["dx"]) <= TOL_BF16
    assert torch.count_nonzero(L.dW1[6]) == 0


def test_bitwise_deterministic_over_10_runs():
    cfg = with_config("balanced", passes="fwd+bwd")
    inp = {k: v.cuda() for k, v in make_inputs(cfg).items()}
    L = Layer(cfg)
    ref = None
    for _ in range(10):
        L.schedule(inp["logits"])
        L.forward(inp["x"], inp["W1"], inp["W2"])
        L.backward(inp["dOut"], inp["x"], inp["W1"], inp["W2"])
        got = [L.out.clone(), L.dx.clone(), L.dW1.clone(), L.dW2.clone(), L.dtopk_w.clone(),
               L.dlogits.clone(), L.sched["perm"].clone(), L.sched["topk_w"].clone()]
        if ref is None:
            ref = got
        else:
            for a, b in zip(ref, got):
                assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                                   b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)
    assert L.status() == 0


# ---------------------------------------------------------------- full sizes
def _sample_tokens(T, n, seed=0):
    return np.sort(np.random.default_rng(seed).choice(T, n, replace=False))


@pytest.mark.slow
def test_kimi_zipf_forward_sampled():
    cfg = CONFIGS["kimi_zipf"]
    dev = make_inputs(cfg, device="cuda", with_grad=False)
    L = Layer(cfg)
    L.schedule(dev["logits"])
    out = L.forward(dev["x"], dev["W1"], dev["W2"], save=False)
    torch.cuda.synchronize()
    assert L.status() == 0
    logits = dev["logits"].cpu()
    ids, g = _check_schedule(L, logits, cfg.k)
    toks = _sample_tokens(cfg.T, 48)
    want = O.forward_tokens(to_np(dev["x"]), ExpertView(dev["W1"]), ExpertView(dev["W2"]), ids, g,
                            toks)
    got = out.float().cpu().numpy()[toks]
    assert rel_err(got, want) <= TOL_BF16
    for i in range(len(toks)):
        assert rel_err(got[i], want[i]) <= 3 * TOL_BF16


@pytest.mark.slow
def test_local_slice_forward_sampled():
    # k = 1 over 4 experts of about 4,096 rows each: every unit a full pair
    cfg = CONFIGS["local_slice"]
    dev = make_inputs(cfg, device="cuda", with_grad=False)
    L = Layer(cfg)
    L.schedule(dev["logits"])
    out = L.forward(dev["x"], dev["W1"], dev["W2"], save=False)
    torch.cuda.synchronize()
    assert L.status() == 0
    ids, g = _check_schedule(L, dev["logits"].cpu(), cfg.k)
    assert np.all(g == 1.0)  # one expert per token: the renormalised weight is 1
    toks = _sample_tokens(cfg.T, 48, seed=2)
    want = O.forward_tokens(to_np(dev["x"]), ExpertView(dev["W1"]), ExpertView(dev["W2"]), ids, g,
                            toks)
    got = out.float().cpu().numpy()[toks]
    assert rel_err(got, want) <= TOL_BF16
    for i in range(len(toks)):
        assert rel_err(got[i], want[i]) <= 3 * TOL_BF16


@pytest.mark.slow
def test_kimi_backward_sampled():
    cfg = CONFIGS["kimi_bwd"]
    dev = make_inputs(cfg, device="cuda")
    L = Layer(cfg)
    L.schedule(dev["logits"])
    L.forward(dev["x"], dev["W1"], dev["W2"], save=True)
    L.backward(dev["dOut"], dev["x"], dev["W1"], dev["W2"])
    torch.cuda.synchronize()
    assert L.status() == 0
    ids, g = _check_schedule(L, dev["logits"].cpu(), cfg.k)
    counts = L.sched_np()["counts"]
    x = to_np(dev["x"])
    dO = to_np(dev["dOut"])
    toks = _sample_tokens(cfg.T, 24, seed=1)
    bt = O.backward_tokens(x, ExpertView(dev["W1"]), ExpertView(dev["W2"]), ids, g, dO, toks)
    assert rel_err(L.dx.float().cpu().numpy()[toks], bt["dx"]) <= TOL_BF16
    assert rel_err(L.dtopk_w.cpu().numpy().reshape(cfg.T, cfg.k)[toks], bt["dg"]) <= TOL_BF16
    assert rel_err(L.dlogits.cpu().numpy()[toks], bt["dlogits"]) <= TOL_BF16
    nz = np.nonzero(counts)[0]
    small = nz[np.argmin(counts[nz])]
    experts = [int(np.argsort(counts)[-3]), int(small), int(nz[len(nz) // 2])]
    empty = np.nonzero(counts == 0)[0]
    ex = O.backward_experts(x, ExpertView(dev["W1"]), ExpertView(dev["W2"]), ids, g, dO, experts)
    for e in experts:
        assert rel_err(L.dW1[e].float().cpu().numpy(), ex[e][0]) <= TOL_BF16, e
        assert rel_err(L.dW2[e].float().cpu().numpy(), ex[e][1]) <= TOL_BF16, e
    if len(empty):
        assert torch.count_nonzero(L.dW1[int(empty[0])]) == 0
        assert torch.count_nonzero(L.dW2[int(empty[0])]) == 0


@pytest.mark.slow
def test_kimi_zipf_forward_bitwise_deterministic():
    cfg = CONFIGS["kimi_zipf"]
    dev = make_inputs(cfg, device="cuda", with_grad=False)
    L = Layer(cfg)
    ref = None
    for _ in range(5):
        L.schedule(dev["logits"])
        out = L.forward(dev["x"], dev["W1"], dev["W2"], save=False).clone()
        if ref is None:
            ref = out
        assert torch.equal(ref.view(torch.int16), out.view(torch.int16))
    assert L.status() == 0
