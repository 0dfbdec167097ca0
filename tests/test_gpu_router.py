"""GPU parity of the router projection (moe_route, moe_router_backward) against
the fp64 oracle, through the C ABI.

Bars: logits within a normwise relative error of 1e-5 of the fp64 product
(bf16 inputs, products exact in fp32, fp32 accumulation); routing decisions
bit-exact against the oracle's top-k of the GPU's own fp32 logits (the
decision is taken in the same precision on both sides) and bitwise equal to
moe_schedule on those logits; weights within 4e-6; the schedule bit-exact;
router gradients within 1e-2 of the oracle fed the same bf16 operands.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_stable_gb300 import binding as B
from oracle import moe_oracle as O

from gpu_util import Layer, with_config
from helpers import rel_err, to_np

pytestmark = pytest.mark.gpu

TOL_LOGITS = 1e-5
TOL_W = 4e-6
TOL_BF16 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield


def _router_inputs(T, d, E, seed=0, skew=0.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    Wr = (torch.randn(E, d, generator=g) / d ** 0.5).to(torch.bfloat16)
    if skew:
        Wr[3] += skew  # a popular expert
    return x, Wr


def _route(cfg, x, Wr, with_logits=True):
    L = Layer(cfg)
    logits = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda") if with_logits else None
    B.moe_route(L.c, x.cuda(), Wr.cuda(), logits, L.sched, L.ws)
    torch.cuda.synchronize()
    assert L.status() == 0
    return L, logits


@pytest.mark.parametrize("T,d,E,k", [(64, 128, 8, 2), (300, 256, 64, 8), (1000, 512, 256, 8),
                                     (97, 128, 300, 4), (2048, 2048, 64, 8), (129, 192, 3, 3)])
def test_route_matches_oracle_and_schedule(T, d, E, k):
    cfg = with_config("tiny", T=T, d=d, f=64, E=E, k=k)
    x, Wr = _router_inputs(T, d, E, seed=T + E)
    L, logits = _route(cfg, x, Wr)
    z = logits.cpu().numpy()
    assert rel_err(z, O.router_logits(to_np(x), to_np(Wr))) <= TOL_LOGITS
    ids, g = O.route(z, k)
    counts, offsets, perm, inv = O.schedule(ids, E)
    s = L.sched_np()
    assert np.array_equal(s["topk_ids"], ids)
    np.testing.assert_allclose(s["topk_w"], g, rtol=TOL_W, atol=0)
    for name, want in (("counts", counts), ("offsets", offsets), ("perm", perm), ("inv", inv)):
        assert np.array_equal(s[name], want), name
    # the same decisions, bit for bit, as the separate schedule on these logits
    L2 = Layer(cfg)
    L2.schedule(logits)
    torch.cuda.synchronize()
    for name in ("topk_ids", "topk_w", "counts", "offsets", "perm", "inv"):
        assert torch.equal(L.sched[name], L2.sched[name]), name


@pytest.mark.parametrize("E", [8, 256])
def test_route_without_logits_output(E):
    cfg = with_config("tiny", T=333, d=256, f=64, E=E, k=min(8, E))
    x, Wr = _router_inputs(333, 256, E, seed=7, skew=0.05)
    La, _ = _route(cfg, x, Wr, with_logits=True)
    Lb, _ = _route(cfg, x, Wr, with_logits=False)
    for name in ("topk_ids", "topk_w", "counts", "perm"):
        assert torch.equal(La.sched[name], Lb.sched[name]), name


def test_route_needs_logits_buffer_past_256_experts():
    cfg = with_config("tiny", T=64, d=128, f=64, E=300, k=4)
    L = Layer(cfg)
    x, Wr = _router_inputs(64, 128, 300)
    with pytest.raises(B.MoeError):
        B.moe_route(L.c, x.cuda(), Wr.cuda(), None, L.sched, L.ws)


@pytest.mark.parametrize("T,d,E", [(64, 128, 8), (300, 256, 64), (1000, 512, 256), (129, 192, 3),
                                   (97, 128, 300)])
def test_router_backward(T, d, E):
    cfg = with_config("tiny", T=T, d=d, f=64, E=E, k=min(2, E))
    x, Wr = _router_inputs(T, d, E, seed=3)
    dl = torch.randn(T, E, generator=torch.Generator().manual_seed(5))
    L = Layer(cfg)
    dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(E, d, dtype=torch.bfloat16, device="cuda")
    B.moe_router_backward(L.c, x.cuda(), Wr.cuda(), dl.cuda(), dx, dW, L.ws)
    torch.cuda.synchronize()
    assert L.status() == 0
    # the oracle is fed the same operands: dlogits rounded to bf16
    wx, wW = O.router_backward(to_np(x), to_np(Wr), to_np(dl.to(torch.bfloat16)))
    assert rel_err(dx.float().cpu().numpy(), wx) <= TOL_BF16
    assert rel_err(dW.float().cpu().numpy(), wW) <= TOL_BF16


def test_route_kimi_shape():
    cfg = with_config("kimi_zipf")
    x, Wr = _router_inputs(cfg.T, cfg.d, cfg.E, seed=11, skew=0.02)
    L, logits = _route(cfg, x, Wr)
    z = logits.cpu().numpy()
    assert rel_err(z, O.router_logits(to_np(x), to_np(Wr))) <= TOL_LOGITS
    ids, g = O.route(z, cfg.k)
    s = L.sched_np()
    assert np.array_equal(s["topk_ids"], ids)
    np.testing.assert_allclose(s["topk_w"], g, rtol=TOL_W, atol=0)
    counts, offsets, perm, inv = O.schedule(ids, cfg.E)
    assert np.array_equal(s["perm"], perm) and np.array_equal(s["counts"], counts)


@pytest.mark.parametrize("T,d,E", [(2048, 2048, 64), (300, 256, 300)])
def test_route_and_router_backward_bitwise_deterministic_over_10_runs(T, d, E):
    cfg = with_config("tiny", T=T, d=d, f=64, E=E, k=8)
    x, Wr = _router_inputs(T, d, E, seed=9, skew=0.03)
    x, Wr = x.cuda(), Wr.cuda()
    dl = torch.randn(T, E, generator=torch.Generator().manual_seed(6)).cuda()
    L = Layer(cfg)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(E, d, dtype=torch.bfloat16, device="cuda")
    ref = None
    for _ in range(10):
        B.moe_route(L.c, x, Wr, logits, L.sched, L.ws)
        B.moe_router_backward(L.c, x, Wr, dl, dx, dW, L.ws)
        got = [logits.clone(), dx.clone().view(torch.int16), dW.clone().view(torch.int16)]
        got += [L.sched[n].clone() for n in ("topk_ids", "topk_w", "perm")]
        if ref is None:
            ref = got
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    assert L.status() == 0
