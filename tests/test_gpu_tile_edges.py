"""GPU parity where the grouped GEMM's tile plan has its edge cases.

Experts hold row counts on and next to the 32-row (thin units round their
rows up to 32), 128-row (one tile) and 256-row (one pair of tiles)
boundaries, plus an empty expert, so that the run has full pair units,
pair units whose odd tile is partial, thin units of every rounding and
experts with no work.  Every token picks two distinct experts, so routing
weights and their gradients vary.  Forward and backward are compared with
the fp64 oracle at the BF16 bar (normwise relative error 1e-2); the saved
activations' padding rows and the empty expert's weight gradients must be
exact zeros.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_stable_gb300.inputs import make_inputs
from oracle import moe_oracle as O

from gpu_util import Layer, padded_positions, with_config
from helpers import ExpertView, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL_BF16 = 1e-2
COUNTS = [1, 31, 32, 33, 127, 128, 129, 255, 256, 257, 383, 0]


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    yield


def _logits_for_counts(counts, seed=0):
    """fp32 logits [T, E] whose top-2 gives expert e exactly counts[e] rows."""
    rng = np.random.default_rng(seed)
    slots = np.repeat(np.arange(len(counts)), counts)
    rng.shuffle(slots)
    pairs = slots.reshape(-1, 2)
    # make the two choices of every token distinct by swapping second choices
    for i in range(len(pairs)):
        if pairs[i, 0] == pairs[i, 1]:
            for j in range(len(pairs)):
                if pairs[j, 1] != pairs[i, 0] and pairs[j, 0] != pairs[i, 1]:
                    pairs[i, 1], pairs[j, 1] = pairs[j, 1], pairs[i, 1]
                    break
    assert np.all(pairs[:, 0] != pairs[:, 1])
    T, E = len(pairs), len(counts)
    z = 0.1 * rng.standard_normal((T, E))
    z[np.arange(T), pairs[:, 0]] += 20.0
    z[np.arange(T), pairs[:, 1]] += 19.0 + rng.uniform(-0.5, 0.5, T)
    return torch.tensor(z, dtype=torch.float32)


@pytest.mark.parametrize("d,f", [(256, 256), (128, 384)])
def test_tile_boundary_counts_forward_backward(d, f):
    logits = _logits_for_counts(COUNTS)
    T, E = logits.shape
    cfg = with_config("tiny", T=T, d=d, f=f, E=E, k=2)
    inp = make_inputs(cfg, x_std=1.0)
    inp["logits"] = logits
    dev = {k: v.cuda() for k, v in inp.items()}
    L = Layer(cfg)
    L.schedule(dev["logits"])
    out = L.forward(dev["x"], dev["W1"], dev["W2"], save=True)
    L.backward(dev["dOut"], dev["x"], dev["W1"], dev["W2"])
    torch.cuda.synchronize()
    assert L.status() == 0

    ids, g = O.route(logits.numpy(), 2)
    counts, offsets, perm, inv = O.schedule(ids, E)
    assert list(counts) == COUNTS
    s = L.sched_np()
    assert np.array_equal(s["counts"], counts) and np.array_equal(s["perm"], perm)

    x, W1, W2, dO = to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), to_np(inp["dOut"])
    want, _ = O.forward(x, W1, W2, ids, g)
    assert rel_err(out.float().cpu().numpy(), want) <= TOL_BF16
    wb = O.backward(x, W1, W2, ids, g, dO)
    assert rel_err(L.dx.float().cpu().numpy(), wb["dx"]) <= TOL_BF16
    assert rel_err(L.dW1.float().cpu().numpy(), wb["dW1"]) <= TOL_BF16
    assert rel_err(L.dW2.float().cpu().numpy(), wb["dW2"]) <= TOL_BF16
    assert rel_err(L.dtopk_w.cpu().numpy().reshape(T, 2), wb["dg"]) <= TOL_BF16
    assert rel_err(L.dlogits.cpu().numpy(), wb["dlogits"]) <= TOL_BF16

    # every expert's dW against its own oracle value (small experts get lost in a normwise
    # error over all experts)
    for e in range(E):
        if counts[e] == 0:
            assert torch.count_nonzero(L.dW1[e]) == 0 and torch.count_nonzero(L.dW2[e]) == 0
            continue
        assert rel_err(L.dW1[e].float().cpu().numpy(), wb["dW1"][e]) <= TOL_BF16, e
        assert rel_err(L.dW2[e].float().cpu().numpy(), wb["dW2"][e]) <= TOL_BF16, e

    # saved activations: rows of the padded layout that hold no routed row are zero
    pp = padded_positions(counts, offsets)
    rp_total = int(sum((c + 127) // 128 * 128 for c in counts))
    pad = np.ones(rp_total, dtype=bool)
    pad[pp] = False
    H = L.saved["H"][:rp_total]
    A = L.saved["A"][:rp_total]
    pad_t = torch.from_numpy(pad).cuda()
    assert torch.count_nonzero(H[pad_t]) == 0
    assert torch.count_nonzero(A[pad_t]) == 0


def test_rows_wider_than_the_bulk_gather_buffers():
    # d = 40960: a bf16 row (80 KB) leaves no room for two shared-memory row
    # buffers per warp, so both gathers take their plain-load kernel; the
    # grouped GEMMs run K = 40960 (GEMM1, dgrad2) and N = 40960 (GEMM2)
    cfg = with_config("tiny", T=96, d=40960, f=64, E=4, k=2)
    inp = make_inputs(cfg, x_std=1.0)
    dev = {k: v.cuda() for k, v in inp.items()}
    L = Layer(cfg)
    L.schedule(dev["logits"])
    out = L.forward(dev["x"], dev["W1"], dev["W2"], save=True)
    L.backward(dev["dOut"], dev["x"], dev["W1"], dev["W2"])
    torch.cuda.synchronize()
    assert L.status() == 0
    ids, g = O.route(inp["logits"].numpy(), 2)
    x, W1, W2, dO = to_np(inp["x"]), ExpertView(inp["W1"]), ExpertView(inp["W2"]), to_np(inp["dOut"])
    want, _ = O.forward(x, W1, W2, ids, g)
    assert rel_err(out.float().cpu().numpy(), want) <= TOL_BF16
    wb = O.backward(x, W1, W2, ids, g, dO)
    for name, got in (("dx", L.dx), ("dW1", L.dW1), ("dW2", L.dW2)):
        assert rel_err(got.float().cpu().numpy(), wb[name]) <= TOL_BF16, name
