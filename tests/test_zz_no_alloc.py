"""moe_schedule_noalloc: the schedule call for callers that cannot allocate
device memory (no workspace argument; the library's built-in device scratch
is used instead).  Its results must equal moe_schedule's, bit for bit, on two
calls in a row -- the built-in scratch keeps the previous call's contents, so
the second call shows that nothing stale leaks into a new result.

This file is collected last on purpose; it passes alone in a fresh process and
after the other tests.
"""
import ctypes

import pytest
import torch

from mixture_experts_layer_stable_gb300 import binding as B
from mixture_experts_layer_stable_gb300.inputs import make_inputs

from gpu_util import cfg_struct, with_config

pytestmark = pytest.mark.gpu

NAMES = ("topk_ids", "topk_w", "counts", "offsets", "perm", "inv")


def _reference(c, logits):
    s = B.alloc_sched(c)
    ws = B.alloc_workspace(c)
    B.moe_schedule(c, logits, s, ws)
    return s


def test_noalloc_schedule_equals_workspace_schedule_twice(cuda_lib):
    cases = [with_config("balanced"), with_config("balanced", logit_std=1.0, zipf=1.2),
             with_config("tiny", T=333, E=16, k=4)]
    for cfg in cases:
        c = cfg_struct(cfg)
        logits = make_inputs(cfg, parts=("logits",))["logits"].cuda()
        want = _reference(c, logits)
        outs = [B.alloc_sched(c) for _ in range(2)]
        for got in outs:
            for t in got.values():
                t.fill_(-7)
        B.moe_schedule_noalloc(c, logits, outs[0])  # first call on this device: address lookup
        torch.cuda.synchronize()
        # the second call allocates nothing: neither device memory nor through torch
        free0 = torch.cuda.mem_get_info()[0]
        stats0 = torch.cuda.memory_stats()
        B.moe_schedule_noalloc(c, logits, outs[1])
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0
        stats1 = torch.cuda.memory_stats()
        for key in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
            assert stats1.get(key) == stats0.get(key), key
        for got in outs:  # two calls in a row on the shared scratch
            for n in NAMES:
                assert torch.equal(got[n], want[n]), (cfg.name, n)


def test_noalloc_rejects_configs_beyond_its_scratch(cuda_lib):
    L = B.lib()
    big = B.make_config(65536, 128, 64, 1024, 8)
    fake = 1 << 20  # never dereferenced: the size check comes first
    s = B.moe_sched(fake, fake, fake, fake, fake, fake)
    assert L.moe_schedule_noalloc(ctypes.byref(big), fake, s, None) == B.MOE_ERR_INVALID_ARG
