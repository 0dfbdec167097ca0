"""Helpers for the GPU tests: run the layer through the C-ABI binding and pull
results back to the host.  No layer arithmetic lives here."""
import numpy as np
import torch

from mixture_experts_layer_stable_gb300 import binding as B
from mixture_experts_layer_stable_gb300.configs import CONFIGS, LayerConfig


def cfg_struct(cfg: LayerConfig, prec=None, minibatch_rows=0, ring_slots=0, gather_ctas=0):
    p = B.MOE_MXFP8 if (prec or cfg.prec) == "mxfp8" else B.MOE_BF16
    return B.make_config(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, p, minibatch_rows, ring_slots, gather_ctas)


class Layer:
    """Buffers for one layer configuration on the current CUDA device."""

    def __init__(self, cfg: LayerConfig, c=None):
        self.cfg = cfg
        self.c = c if c is not None else cfg_struct(cfg)
        self.sched = B.alloc_sched(self.c)
        self.ws = B.alloc_workspace(self.c)
        self.saved = B.alloc_saved(self.c)
        T, d, f, E = cfg.T, cfg.d, cfg.f, cfg.E
        self.out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
        self.dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
        self.dtopk_w = torch.empty(T * cfg.k, dtype=torch.float32, device="cuda")
        self.dlogits = torch.empty(T, E, dtype=torch.float32, device="cuda")
        self.dW1 = None
        self.dW2 = None

    def schedule(self, logits):
        B.moe_schedule(self.c, logits, self.sched, self.ws)

    def forward(self, x, W1, W2, save=True, w1s=None, w2s=None):
        B.moe_forward(self.c, x, W1, w1s, W2, w2s, self.sched, self.out,
                      self.saved if save else None, self.ws)
        return self.out

    def backward(self, dOut, x, W1, W2, dlogits=True, recompute=False):
        if self.dW1 is None:
            self.dW1 = torch.empty_like(W1)
            self.dW2 = torch.empty_like(W2)
        B.moe_backward(self.c, dOut, x, W1, W2, self.sched, None if recompute else self.saved,
                       self.dx, self.dW1, self.dW2, self.dtopk_w, self.dlogits if dlogits else None,
                       self.ws)

    def status(self):
        return B.moe_read_status(self.ws)

    def sched_np(self):
        s = {k: v.cpu().numpy() for k, v in self.sched.items()}
        s["topk_ids"] = s["topk_ids"].reshape(self.cfg.T, self.cfg.k)
        s["topk_w"] = s["topk_w"].reshape(self.cfg.T, self.cfg.k)
        return s


def padded_positions(counts, offsets, bm=128):
    """Padded expert-ordered row of every expert-ordered position p (host
    restatement of the documented saved-activation layout)."""
    counts = np.asarray(counts, np.int64)
    pc = (counts + bm - 1) // bm * bm
    poff = np.concatenate([[0], np.cumsum(pc)])
    R = int(np.sum(counts))
    pp = np.empty(R, np.int64)
    for e in range(len(counts)):
        a, b = int(offsets[e]), int(offsets[e + 1])
        pp[a:b] = poff[e] + np.arange(b - a)
    return pp


def with_config(name, **kw):
    c = CONFIGS[name]
    d = c.as_dict()
    d.update(kw)
    return LayerConfig(**d)
