"""The C-ABI library loads, exports every symbol include/moe.h declares, and
its host-side logic (validation, sizing, the minibatch heuristic) behaves --
all without a GPU (no call here reaches a CUDA kernel)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from mixture_experts_layer_stable_gb300 import build, binding
    build.build()
    binding.lib()
    return binding


def _declared():
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", txt)))


def test_exports_every_declared_symbol(B):
    names = _declared()
    assert len(names) >= 9
    L = B.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(B.EXPORTED) <= set(names)


def test_min_minibatch_matches_pages_figure(B):
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "min_minibatch.txt"))
            if l.strip() and not l.startswith("#")]
    for sms, bm, bn, n, want in rows:
        assert B.moe_min_minibatch(int(sms), int(bm), int(bn), int(n)) == int(want)
    assert B.moe_min_minibatch(0, 128, 256, 4096) == 0
    assert B.moe_min_minibatch(152, 128, 256, 4096) == 2432
    assert B.moe_min_minibatch(1, 1, 1, 3) == 1  # ceiling


def test_workspace_and_saved_sizes(B):
    c = B.make_config(64, 128, 64, 8, 2)
    ws = B.moe_workspace_bytes(c)
    assert ws > 0 and ws % 1024 == 0
    rows = B.moe_saved_rows(c)
    # R = 128 routed rows, at most 8 experts each padded by < 128 rows
    assert rows % 128 == 0 and 128 <= rows <= 128 + 8 * 127 + 127
    big = B.make_config(4096, 7168, 2048, 256, 8)
    assert B.moe_saved_rows(big) == 32768 + 256 * 127 + (128 - (32768 + 256 * 127) % 128) % 128
    for bad in (B.make_config(64, 100, 64, 8, 2), B.make_config(64, 128, 64, 8, 9),
                B.make_config(0, 128, 64, 8, 2), B.make_config(64, 128, 64, 2000, 2),
                B.make_config(64, 128, 64, 64, 33), B.make_config(64, 128, 64, 8, 2, prec=7),
                B.make_config(64, 128, 64, 8, 2, minibatch_rows=-1, ring_slots=2),
                B.make_config(64, 128, 64, 8, 2, minibatch_rows=128, ring_slots=65),
                B.make_config(64, 128, 64, 8, 2, gather_ctas=-1),
                B.make_config(64, 128, 64, 8, 2, minibatch_rows=128, ring_slots=1)):
        assert B.moe_workspace_bytes(bad) == 0
        assert B.moe_saved_rows(bad) == 0
    # a ring window of 100 rows rounds up to one 128-row tile: valid, with ring space
    ring = B.make_config(64, 128, 64, 8, 2, minibatch_rows=100, ring_slots=2)
    assert B.moe_workspace_bytes(ring) >= ws + 2 * 128 * 128 * 2


def test_host_validation_returns_before_any_gpu_work(B):
    L = B.lib()
    c = B.make_config(64, 128, 64, 8, 2)
    fake = 1 << 20  # aligned, never dereferenced: validation fails first
    s = B.moe_sched(fake, fake, fake, fake, fake, fake)
    null_s = B.moe_sched(None, fake, fake, fake, fake, fake)
    need = B.moe_workspace_bytes(c)
    assert L.moe_schedule(ctypes.byref(c), fake, null_s, fake, need, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_schedule(ctypes.byref(c), fake + 4, s, fake, need, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_schedule(ctypes.byref(c), fake, s, fake, need - 1, None) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    bad = B.make_config(64, 128, 64, 8, 9)
    assert L.moe_schedule(ctypes.byref(bad), fake, s, fake, need, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_forward(ctypes.byref(c), fake, fake, None, fake, None, s, None, None, fake, need,
                         None) == B.MOE_ERR_INVALID_ARG
    # saved activations, when given, must be aligned (NULL asks for a recompute)
    bad_saved = ctypes.byref(B.moe_saved(fake + 2, fake))
    assert L.moe_backward(ctypes.byref(c), fake, fake, fake, fake, s, bad_saved, fake, fake, fake, fake,
                          None, fake, need, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_backward(ctypes.byref(c), fake, fake, fake, fake, null_s, None, fake, fake, fake, fake,
                          None, fake, need, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_mxfp8(fake, 1, 100, 64, fake, fake, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_read_status(fake + 1, None) == B.MOE_ERR_INVALID_ARG


def test_status_strings(B):
    for code in range(7):
        assert B.moe_status_string(code) not in ("", "unknown status")
    assert B.moe_status_string(99) == "unknown status"


def test_workspace_regions_lie_inside_the_workspace(B):
    c = B.make_config(300, 256, 128, 6, 3, B.MOE_MXFP8)
    total = B.moe_workspace_bytes(c)
    rows = B.moe_saved_rows(c)
    d, f = 256, 128
    want = {B.MOE_WS_XQ_CODES: rows * d, B.MOE_WS_XQ_SCALES: rows * d // 32,
            B.MOE_WS_AQ_CODES: rows * f, B.MOE_WS_AQ_SCALES: rows * f // 32,
            B.MOE_WS_DYQ_CODES: rows * d, B.MOE_WS_DYQ_SCALES: rows * d // 32,
            B.MOE_WS_XQT_CODES: d * rows, B.MOE_WS_XQT_SCALES: d * rows // 32,
            B.MOE_WS_DYQT_CODES: d * rows, B.MOE_WS_DYQT_SCALES: d * rows // 32,
            B.MOE_WS_DHQ_CODES: rows * 2 * f, B.MOE_WS_DHQ_SCALES: rows * 2 * f // 32,
            B.MOE_WS_DHQT_CODES: 2 * f * rows, B.MOE_WS_DHQT_SCALES: 2 * f * rows // 32,
            B.MOE_WS_GAQT_CODES: f * rows, B.MOE_WS_GAQT_SCALES: f * rows // 32}
    spans = []
    for region, n_want in want.items():
        off, n = B.moe_workspace_region(c, region)
        assert n == n_want and off % 16 == 0 and off + n <= total, region
        spans.append((off, off + n))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))  # no overlap
    with pytest.raises(B.MoeError):
        B.moe_workspace_region(c, 16)
    with pytest.raises(B.MoeError):  # a BF16 layer has no quantised buffers
        B.moe_workspace_region(B.make_config(300, 256, 128, 6, 3), B.MOE_WS_XQ_CODES)
