"""Cluster launch control as the weight-gradient GEMMs' tile scheduler
(Marktechpost "Cursor开源MoK..." three design decisions, last paragraph: the
megakernel schedules with Blackwell's Cluster Launch Control).

With moe_set_tile_scheduler(1) the one-CTA weight-gradient GEMMs run as a
grid of one CTA per work unit whose running CTAs cancel the launches of the
pending ones and take over their units.  Every unit is still one whole tile
computed by one CTA in the same K order, so every output must be bitwise
identical to the static walk's, whichever CTA ran which unit -- here on the
BF16 and MXFP8 backward, on a tiny, the balanced and the Kimi-like shape.
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


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    before = B.moe_get_tile_scheduler()
    yield
    B.moe_set_tile_scheduler(before)


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _grads(cfg, dev, mode):
    B.moe_set_tile_scheduler(mode)
    L = Layer(cfg)
    L.schedule(dev["logits"])
    L.forward(dev["x"], dev["W1"], dev["W2"], save=True)
    L.backward(dev["dOut"], dev["x"], dev["W1"], dev["W2"])
    torch.cuda.synchronize()
    assert L.status() == 0
    return L


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("tiny", dict(T=300, d=256, f=192, E=6, k=3)),
                                     ("balanced", {})])
def test_clc_weight_gradients_equal_the_static_walk(name, kw):
    cfg = with_config(name, passes="fwd+bwd", **kw)
    inp = make_inputs(cfg, x_std=1.0 if name == "tiny" else None)
    dev = {k: v.cuda() for k, v in inp.items()}
    ref = _grads(cfg, dev, 0)
    L = _grads(cfg, dev, 1)
    for n in ("dW1", "dW2", "dx", "dtopk_w"):
        assert torch.equal(_bits(getattr(L, n)), _bits(getattr(ref, n))), n
    if name == "tiny":
        ids, g = O.route(inp["logits"].numpy(), cfg.k)
        want = O.backward(to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), ids, g,
                          to_np(inp["dOut"]))
        assert rel_err(L.dW1.float().cpu().numpy(), want["dW1"]) <= 1e-2


def test_clc_mxfp8_weight_gradients_equal_the_static_walk():
    from test_gpu_mxfp8_backward import MxBackward
    cfg = with_config("tiny", prec="mxfp8", passes="fwd+bwd", f=128, d=256, T=300, E=6, k=3)
    dev = {k: v.cuda() for k, v in make_inputs(cfg, x_std=1.0).items()}
    out = []
    for mode in (0, 1):
        B.moe_set_tile_scheduler(mode)
        L = MxBackward(cfg, dev).run()
        out.append([L.dW1.clone(), L.dW2.clone()])
    for a, b in zip(*out):
        assert torch.equal(_bits(a), _bits(b))


@pytest.mark.slow
def test_clc_kimi_backward_equal_the_static_walk():
    cfg = CONFIGS["kimi_bwd"]
    dev = make_inputs(cfg, device="cuda")
    ref = _grads(cfg, dev, 0)
    dW1, dW2 = ref.dW1.clone(), ref.dW2.clone()
    del ref
    L = _grads(cfg, dev, 1)
    assert torch.equal(_bits(L.dW1), _bits(dW1))
    assert torch.equal(_bits(L.dW2), _bits(dW2))


def test_scheduler_setting_is_validated():
    with pytest.raises(B.MoeError):
        B.moe_set_tile_scheduler(2)
