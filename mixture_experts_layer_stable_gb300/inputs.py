"""Seeded synthetic inputs for the MoE layer.

This module holds no arithmetic of the layer itself: it only draws random
tensors.  Both the CUDA path (tests, bench) and the fp64 oracle are fed from
here.  Recipe (one torch.Generator per tensor, seed = base + index):

  index 0  logits  fp32 [T,E]   ~ N(0, logit_std); with zipf = s > 0 the
                                  per-expert bias ln p_e, p_e ~ (e+1)^-s
                                  normalised, is added (a few experts hot)
  index 1  x       bf16 [T,d]   ~ N(0, 1/sqrt(d))      (std = 1/sqrt(fan_in))
  index 2  W1      bf16 [E,d,2f] ~ N(0, 1/sqrt(d)), drawn expert by expert;
                                  columns [0,f) gate, [f,2f) up
  index 3  W2      bf16 [E,f,d] ~ N(0, 1/sqrt(f)), drawn expert by expert
  index 4  dOut    bf16 [T,d]   ~ N(0, 1)

fp32 draws are rounded to bf16 by torch's round-to-nearest-even cast.  Values
depend on the device the generator runs on (CPU and CUDA streams differ), so a
test draws once and copies to the other side.
"""

import math

import torch

from .configs import CONFIGS, LayerConfig


def zipf_bias(E: int, s: float) -> torch.Tensor:
    p = torch.arange(1, E + 1, dtype=torch.float64) ** (-s)
    p = p / p.sum()
    return torch.log(p).to(torch.float32)


def make_inputs(cfg, device="cpu", seed: int = 0, with_grad: bool = True,
                x_std=None, parts=("logits", "x", "W1", "W2", "dOut"), experts=None):
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    assert isinstance(cfg, LayerConfig)
    T, d, f, E = cfg.T, cfg.d, cfg.f, cfg.E
    dev = torch.device(device)

    def gen(i):
        return torch.Generator(device=dev).manual_seed(seed + i)

    nE = E if experts is None else min(E, int(experts))  # first nE experts' weights only
    out = {}
    if "logits" in parts:
        logits = torch.randn(T, E, generator=gen(0), device=dev) * cfg.logit_std
        if cfg.zipf > 0:
            logits = logits + zipf_bias(E, cfg.zipf).to(dev)
        out["logits"] = logits.contiguous()
    if "x" in parts:
        xs = (1.0 / math.sqrt(d)) if x_std is None else x_std
        out["x"] = (torch.randn(T, d, generator=gen(1), device=dev) * xs).to(torch.bfloat16)
    if "W1" in parts:
        g2 = gen(2)
        W1 = torch.empty(nE, d, 2 * f, dtype=torch.bfloat16, device=dev)
        for e in range(nE):
            W1[e] = (torch.randn(d, 2 * f, generator=g2, device=dev) / math.sqrt(d)).to(torch.bfloat16)
        out["W1"] = W1
    if "W2" in parts:
        g3 = gen(3)
        W2 = torch.empty(nE, f, d, dtype=torch.bfloat16, device=dev)
        for e in range(nE):
            W2[e] = (torch.randn(f, d, generator=g3, device=dev) / math.sqrt(f)).to(torch.bfloat16)
        out["W2"] = W2
    if with_grad and "dOut" in parts:
        out["dOut"] = torch.randn(T, d, generator=gen(4), device=dev).to(torch.bfloat16)
    return out
