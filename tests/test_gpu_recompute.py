"""The backward without saved activations, and its reverse traversal of the
ring (Marktechpost "Cursor开源MoK..." three design decisions: the ring buffer
is traversed in reverse to replay as few forward activations as possible).

moe_backward with saved = NULL recomputes H and A with the forward's own
GEMM1 on the re-gathered rows -- the same tiles in the same K order -- so
every gradient must be bitwise identical to the backward from saved H and A.
After a ring forward the backward's re-gather walks the rows from the last to
the first and takes the rows of the ring's last windows from the ring: the
gradients must again be bitwise identical to the kernel-chain path, for
window counts below, at and above the ring depth.  Both stay within 1e-2 of
the oracle.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_stable_gb300.configs import CONFIGS
from mixture_experts_layer_stable_gb300.inputs import make_inputs
from oracle import moe_oracle as O

from gpu_util import Layer, cfg_struct, with_config
from helpers import ExpertView, rel_err, to_np

pytestmark = pytest.mark.gpu

GRADS = ("dx", "dW1", "dW2", "dtopk_w", "dlogits")


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield


def _same(a, b):
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    return torch.equal(a, b)


def _fwd_bwd(cfg, dev, mb=0, slots=0, save=True, recompute=False):
    L = Layer(cfg, cfg_struct(cfg, minibatch_rows=mb, ring_slots=slots))
    L.schedule(dev["logits"])
    L.forward(dev["x"], dev["W1"], dev["W2"], save=save)
    L.backward(dev["dOut"], dev["x"], dev["W1"], dev["W2"], recompute=recompute)
    torch.cuda.synchronize()
    assert L.status() == 0
    return L


@pytest.mark.parametrize("name,kw,x_std", [("tiny", {}, 1.0), ("tiny", dict(f=192, d=256, T=300), 1.0),
                                           ("tiny", dict(T=1, k=8), 1.0), ("balanced", {}, None)])
def test_recompute_equals_saved_bitwise(name, kw, x_std):
    cfg = with_config(name, passes="fwd+bwd", **kw)
    inp = make_inputs(cfg, x_std=x_std)
    dev = {k: v.cuda() for k, v in inp.items()}
    ref = _fwd_bwd(cfg, dev)
    L = _fwd_bwd(cfg, dev, save=False, recompute=True)
    for n in GRADS:
        assert _same(getattr(L, n), getattr(ref, n)), n
    ids, g = O.route(inp["logits"].numpy(), cfg.k)
    if name == "tiny":
        want = O.backward(to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), ids, g,
                          to_np(inp["dOut"]))
        assert rel_err(L.dx.float().cpu().numpy(), want["dx"]) <= 1e-2
        assert rel_err(L.dW1.float().cpu().numpy(), want["dW1"]) <= 1e-2
        assert rel_err(L.dW2.float().cpu().numpy(), want["dW2"]) <= 1e-2


@pytest.mark.parametrize("mb,slots", [(1024, 2), (512, 4), (4096, 4), (8192, 2)])
def test_backward_after_ring_forward_reuses_the_ring(mb, slots):
    # balanced: about 20,000 padded rows, so 1,024-row windows over 2 slots
    # leave 2 of about 20 windows in the ring, 8,192-row windows all of them
    cfg = with_config("balanced", passes="fwd+bwd")
    dev = {k: v.cuda() for k, v in make_inputs(cfg).items()}
    ref = _fwd_bwd(cfg, dev)
    for save, recompute in ((True, False), (False, True)):
        L = _fwd_bwd(cfg, dev, mb, slots, save=save, recompute=recompute)
        for n in GRADS:
            assert _same(getattr(L, n), getattr(ref, n)), (mb, slots, save, n)


def test_backward_recompute_bitwise_deterministic():
    cfg = with_config("balanced", passes="fwd+bwd")
    dev = {k: v.cuda() for k, v in make_inputs(cfg).items()}
    L = Layer(cfg, cfg_struct(cfg, minibatch_rows=1024, ring_slots=4))
    ref = None
    for _ in range(5):
        L.schedule(dev["logits"])
        L.forward(dev["x"], dev["W1"], dev["W2"], save=False)
        L.backward(dev["dOut"], dev["x"], dev["W1"], dev["W2"], recompute=True)
        got = [getattr(L, n).clone() for n in GRADS]
        if ref is None:
            ref = got
        for a, b in zip(ref, got):
            assert _same(a, b)
    assert L.status() == 0


@pytest.mark.slow
def test_kimi_backward_recompute_equals_saved():
    cfg = CONFIGS["kimi_bwd"]
    dev = make_inputs(cfg, device="cuda")
    ref = _fwd_bwd(cfg, dev)
    L = _fwd_bwd(cfg, dev, 1024, 4, save=False, recompute=True)
    for n in GRADS:
        assert _same(getattr(L, n), getattr(ref, n)), n
