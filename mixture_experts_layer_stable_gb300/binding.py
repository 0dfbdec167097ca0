"""ctypes binding of libmoe.so (include/moe.h).  Argument marshalling only:
every step of the layer runs in the library's CUDA kernels.  Tensors are torch
CUDA tensors (PyTorch provides device memory and streams); their data
pointers are passed through unchanged.

The functions keep the C names.  Each raises MoeError when the library
returns a status other than MOE_OK.  There is no fallback: if the library has
not been built, the first call raises.
"""

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

MOE_BF16 = 0
MOE_MXFP8 = 1

EXPORTED = [
    "moe_workspace_bytes", "moe_saved_rows", "moe_min_minibatch", "moe_schedule",
    "moe_quantize_mxfp8", "moe_forward", "moe_backward", "moe_read_status", "moe_status_string",
    "moe_trace_enable", "moe_trace_count", "moe_trace_read", "moe_schedule_noalloc",
    "moe_route", "moe_router_backward", "moe_workspace_region", "moe_quantize_mxfp8_rows",
    "moe_backward_mxfp8", "moe_set_tile_scheduler", "moe_get_tile_scheduler",
]

MOE_WS_XQ_CODES = 0
MOE_WS_XQ_SCALES = 1
MOE_WS_AQ_CODES = 2
MOE_WS_AQ_SCALES = 3
MOE_WS_DYQ_CODES, MOE_WS_DYQ_SCALES = 4, 5
MOE_WS_XQT_CODES, MOE_WS_XQT_SCALES = 6, 7
MOE_WS_DYQT_CODES, MOE_WS_DYQT_SCALES = 8, 9
MOE_WS_DHQ_CODES, MOE_WS_DHQ_SCALES = 10, 11
MOE_WS_DHQT_CODES, MOE_WS_DHQT_SCALES = 12, 13
MOE_WS_GAQT_CODES, MOE_WS_GAQT_SCALES = 14, 15


class MoeError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {moe_status_string(code)} ({code})")


class moe_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("T", "d", "f", "E", "k", "prec", "minibatch_rows", "ring_slots", "gather_ctas")]


class moe_sched(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("topk_ids", "topk_w", "counts", "offsets", "perm", "inv")]


class moe_saved(ctypes.Structure):
    _fields_ = [("H", ctypes.c_void_p), ("A", ctypes.c_void_p)]


_lib = None


def lib():
    """Load libmoe.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() "
                               "(or python -m mixture_experts_layer_stable_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(moe_config)
        savp = ctypes.POINTER(moe_saved)
        L.moe_workspace_bytes.argtypes = [cfgp]
        L.moe_workspace_bytes.restype = sz
        L.moe_saved_rows.argtypes = [cfgp]
        L.moe_saved_rows.restype = i64
        L.moe_min_minibatch.argtypes = [i32, i32, i32, i32]
        L.moe_min_minibatch.restype = i32
        L.moe_schedule.argtypes = [cfgp, vp, moe_sched, vp, sz, vp]
        L.moe_schedule.restype = ctypes.c_int
        L.moe_quantize_mxfp8.argtypes = [vp, i64, i32, i32, vp, vp, vp]
        L.moe_quantize_mxfp8.restype = ctypes.c_int
        L.moe_forward.argtypes = [cfgp, vp, vp, vp, vp, vp, moe_sched, vp, savp, vp, sz, vp]
        L.moe_forward.restype = ctypes.c_int
        L.moe_backward.argtypes = [cfgp, vp, vp, vp, vp, moe_sched, savp, vp, vp, vp, vp, vp, vp,
                                   sz, vp]
        L.moe_backward.restype = ctypes.c_int
        L.moe_read_status.argtypes = [vp, vp]
        L.moe_read_status.restype = ctypes.c_int
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_trace_enable.argtypes = [i32]
        L.moe_trace_enable.restype = ctypes.c_int
        L.moe_trace_count.argtypes = []
        L.moe_trace_count.restype = i32
        L.moe_trace_read.argtypes = [i32, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]
        L.moe_trace_read.restype = ctypes.c_int
        L.moe_schedule_noalloc.argtypes = [cfgp, vp, moe_sched, vp]
        L.moe_schedule_noalloc.restype = ctypes.c_int
        L.moe_route.argtypes = [cfgp, vp, vp, vp, moe_sched, vp, sz, vp]
        L.moe_route.restype = ctypes.c_int
        L.moe_router_backward.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.moe_router_backward.restype = ctypes.c_int
        L.moe_workspace_region.argtypes = [cfgp, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
        L.moe_workspace_region.restype = ctypes.c_int
        L.moe_quantize_mxfp8_rows.argtypes = [vp, i64, i32, vp, vp, vp]
        L.moe_quantize_mxfp8_rows.restype = ctypes.c_int
        L.moe_backward_mxfp8.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, moe_sched, savp, vp, vp, vp, vp,
                                         vp, vp, sz, vp]
        L.moe_backward_mxfp8.restype = ctypes.c_int
        L.moe_set_tile_scheduler.argtypes = [i32]
        L.moe_set_tile_scheduler.restype = ctypes.c_int
        L.moe_get_tile_scheduler.argtypes = []
        L.moe_get_tile_scheduler.restype = i32
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code, where):
    if code != MOE_OK:
        raise MoeError(code, where)


def make_config(T, d, f, E, k, prec=MOE_BF16, minibatch_rows=0, ring_slots=0, gather_ctas=0):
    return moe_config(T, d, f, E, k, prec, minibatch_rows, ring_slots, gather_ctas)


def moe_status_string(code):
    return lib().moe_status_string(int(code)).decode()


def moe_workspace_bytes(cfg):
    return int(lib().moe_workspace_bytes(ctypes.byref(cfg)))


def moe_saved_rows(cfg):
    return int(lib().moe_saved_rows(ctypes.byref(cfg)))


def moe_min_minibatch(compute_sms, bm, bn, n_cols):
    return int(lib().moe_min_minibatch(compute_sms, bm, bn, n_cols))


def sched_struct(s):
    return moe_sched(*(_ptr(s[n]) for n in ("topk_ids", "topk_w", "counts", "offsets", "perm", "inv")))


def moe_schedule(cfg, logits, sched, ws, stream=None):
    _check(lib().moe_schedule(ctypes.byref(cfg), _ptr(logits), sched_struct(sched), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "moe_schedule")


def moe_route(cfg, x, w_router, logits, sched, ws, stream=None):
    """Router projection + routing + schedule (logits may be None when E <= 256)."""
    _check(lib().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(w_router),
                           None if logits is None else _ptr(logits), sched_struct(sched), _ptr(ws),
                           ws.numel() * ws.element_size(), _stream(stream)), "moe_route")


def moe_router_backward(cfg, x, w_router, dlogits, dx_router, dw_router, ws, stream=None):
    _check(lib().moe_router_backward(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(dlogits),
                                     _ptr(dx_router), _ptr(dw_router), _ptr(ws),
                                     ws.numel() * ws.element_size(), _stream(stream)),
           "moe_router_backward")


def moe_schedule_noalloc(cfg, logits, sched, stream=None):
    """moe_schedule for callers that cannot allocate: no workspace argument;
    the library's built-in 1.5 MiB device scratch is used (calls share it)."""
    _check(lib().moe_schedule_noalloc(ctypes.byref(cfg), _ptr(logits), sched_struct(sched),
                                      _stream(stream)), "moe_schedule_noalloc")


def moe_quantize_mxfp8(w, batch, K, N, q, scales, stream=None):
    _check(lib().moe_quantize_mxfp8(_ptr(w), batch, K, N, _ptr(q), _ptr(scales), _stream(stream)),
           "moe_quantize_mxfp8")


def moe_forward(cfg, x, w1, w1_scales, w2, w2_scales, sched, out, saved, ws, stream=None):
    sv = None if saved is None else ctypes.byref(moe_saved(_ptr(saved["H"]), _ptr(saved["A"])))
    _check(lib().moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(w1), _ptr(w1_scales), _ptr(w2),
                             _ptr(w2_scales), sched_struct(sched), _ptr(out), sv, _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "moe_forward")


def moe_backward(cfg, dout, x, w1, w2, sched, saved, dx, dw1, dw2, dtopk_w, dlogits, ws, stream=None):
    """saved: the dict moe_forward filled, or None (H and A are recomputed)."""
    sv = None if saved is None else ctypes.byref(moe_saved(_ptr(saved["H"]), _ptr(saved["A"])))
    _check(lib().moe_backward(ctypes.byref(cfg), _ptr(dout), _ptr(x), _ptr(w1), _ptr(w2),
                              sched_struct(sched), sv, _ptr(dx), _ptr(dw1), _ptr(dw2),
                              _ptr(dtopk_w), _ptr(dlogits), _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "moe_backward")


def moe_workspace_region(cfg, region):
    """(byte offset, bytes) of an intermediate buffer inside the workspace."""
    off, n = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().moe_workspace_region(ctypes.byref(cfg), int(region), ctypes.byref(off),
                                      ctypes.byref(n)), "moe_workspace_region")
    return int(off.value), int(n.value)


def moe_quantize_mxfp8_rows(w, rows, K, q, scales, stream=None):
    _check(lib().moe_quantize_mxfp8_rows(_ptr(w), rows, K, _ptr(q), _ptr(scales), _stream(stream)),
           "moe_quantize_mxfp8_rows")


def moe_backward_mxfp8(cfg, dout, x, w1q, w1s, w2q, w2s, sched, saved, dx, dw1, dw2, dtopk_w, dlogits,
                       ws, stream=None):
    sv = None if saved is None else ctypes.byref(moe_saved(_ptr(saved["H"]), _ptr(saved["A"])))
    _check(lib().moe_backward_mxfp8(ctypes.byref(cfg), _ptr(dout), _ptr(x), _ptr(w1q), _ptr(w1s),
                                    _ptr(w2q), _ptr(w2s), sched_struct(sched), sv, _ptr(dx), _ptr(dw1),
                                    _ptr(dw2), _ptr(dtopk_w), _ptr(dlogits), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)), "moe_backward_mxfp8")


def moe_set_tile_scheduler(mode):
    """0: static walk; 1: cluster launch control (one-CTA weight gradients)."""
    _check(lib().moe_set_tile_scheduler(int(mode)), "moe_set_tile_scheduler")


def moe_get_tile_scheduler():
    return int(lib().moe_get_tile_scheduler())


def moe_read_status(ws, stream=None):
    return int(lib().moe_read_status(_ptr(ws), _stream(stream)))


def moe_trace_enable(capacity):
    _check(lib().moe_trace_enable(int(capacity)), "moe_trace_enable")


def moe_trace_count():
    return int(lib().moe_trace_count())


def moe_trace_read(i):
    name = ctypes.c_char_p()
    ms = ctypes.c_float()
    _check(lib().moe_trace_read(int(i), ctypes.byref(name), ctypes.byref(ms)), "moe_trace_read")
    return name.value.decode(), float(ms.value)


# ---------------------------------------------------------------- buffers
def alloc_sched(cfg, device="cuda"):
    """Schedule arrays for cfg (torch allocates; the library only writes)."""
    R = cfg.T * cfg.k
    i32 = dict(dtype=torch.int32, device=device)
    return {
        "topk_ids": torch.empty(R, **i32),
        "topk_w": torch.empty(R, dtype=torch.float32, device=device),
        "counts": torch.empty(cfg.E, **i32),
        "offsets": torch.empty(cfg.E + 1, **i32),
        "perm": torch.empty(R, **i32),
        "inv": torch.empty(R, **i32),
    }


def alloc_workspace(cfg, device="cuda"):
    n = moe_workspace_bytes(cfg)
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def alloc_saved(cfg, device="cuda"):
    rows = moe_saved_rows(cfg)
    return {"H": torch.empty(rows, 2 * cfg.f, dtype=torch.bfloat16, device=device),
            "A": torch.empty(rows, cfg.f, dtype=torch.bfloat16, device=device)}
