"""Small test helpers shared by the CPU and GPU tests (no layer arithmetic)."""
import numpy as np
import torch


class ExpertView:
    """Index a torch bf16 weight tensor [E, ...] by expert, yielding float64 numpy."""

    def __init__(self, t):
        self.t = t

    def __len__(self):
        return self.t.shape[0]

    def __getitem__(self, e):
        return self.t[e].detach().to("cpu", torch.float64).numpy()


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))
