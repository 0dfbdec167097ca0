"""Plain, slow, fp64 CPU oracle for the single-GPU mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The product path (the CUDA library and its Python binding) never does,
and this module never imports the product package: the two share no code.

Sources (web pages on Cursor's "Mixture-of-Kittens" (MoK) MoE megakernel):
  [LP]  leiphone, "MoK：把 token 调度、跨 GPU 通信和专家计算塞进同一个 GPU 内核"
        sections 01 "MoE 的「通信税」" / 02 "怎么让 token 一边传，一边算" /
        03 "一整套高度特化的执行方式"
  [MT]  Marktechpost (Chinese translation), "Cursor开源MoK：GB300 NVL72机架上的
        确定性MoE训练大内核", sections "三个重要的设计决策" (three design
        decisions), "基准测试" (benchmarks), "关键要点" (key points)

The pages print no formula, listing or worked example.  The layer they
benchmark is, in order, Schedule -> Dispatch -> Expert FFN -> Combine ->
weighted merge ([LP] 03, first paragraph); the expert FFN is a SwiGLU FFN
([MT] three design decisions, last paragraph; [LP] 02, MXFP8 paragraph).
Each function below writes out the plain definition of one of those steps.
Where the pages leave a detail open the reading taken is stated in the
docstring (the full list of readings is in the repository's design notes).

Everything is fp64.  bf16 / fp32 inputs widen exactly to fp64; no
intermediate is rounded back to bf16 (the GPU path does round H, A and Y to
bf16; the parity tolerance covers those roundings).

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against brute force, closed forms, library routines or finite differences.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "router_logits",
    "router_backward",
    "route",
    "schedule",
    "silu",
    "swiglu_backward",
    "expert_ffn",
    "forward",
    "forward_tokens",
    "backward",
    "backward_experts",
    "backward_tokens",
    "dlogits_from_dg",
    "e4m3_encode",
    "e4m3_decode",
    "mxfp8_quantize",
    "mxfp8_dequantize",
    "forward_mxfp8",
    "backward_mxfp8",
    "backward_mxfp8_experts",
]


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Router projection: the logits that routing reads come from the router of
# [LP] 01 (it decides afresh every step which experts each token goes to).
# Reading: a bias-free linear map of the token row, the router weight stored
# expert by expert, logits[t, e] = sum_i x[t, i] * Wr[e, i]; and its backward.
# --------------------------------------------------------------------------
def router_logits(x, Wr):
    """logits [T, E] = x [T, d] . Wr [E, d]^T, in fp64."""
    return _f64(x) @ _f64(Wr).T


def router_backward(x, Wr, dlogits):
    """Backward of router_logits for an upstream gradient dlogits [T, E]:
    dx [T, d] = dlogits . Wr and dWr [E, d] = dlogits^T . x, in fp64."""
    dl = _f64(dlogits)
    return dl @ _f64(Wr), dl.T @ _f64(x)


# --------------------------------------------------------------------------
# Routing: [LP] 01 (the router picks experts afresh every step for every
# token).  Reading: plain top-k of the fp32 logits, ties to the lower expert
# id, weights = softmax over the k selected logits (identical to a softmax
# over all E logits renormalised over the k selected).  Slot j is the rank.
# --------------------------------------------------------------------------
def route(logits, k: int):
    """Top-k routing.

    logits: float32 [T, E] (finite).  Returns (ids int32 [T,k], g fp64 [T,k]).
    Experts are ordered by (logit descending, expert id ascending); comparison
    is on the fp32 values exactly as given (-0.0 ties with +0.0).
    g[t, j] = exp(z_j - z_0) / sum_l exp(z_l - z_0) over the k selected.
    """
    z = np.asarray(logits)
    if z.dtype != np.float32:
        raise TypeError("logits must be float32")
    if not np.all(np.isfinite(z)):
        raise ValueError("logits must be finite")
    T, E = z.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    z64 = z.astype(np.float64)
    eidx = np.broadcast_to(np.arange(E), (T, E))
    # lexsort: last key is primary -> primary -z ascending, then e ascending.
    order = np.lexsort((eidx, -z64), axis=-1)
    ids = order[:, :k].astype(np.int32)
    zs = np.take_along_axis(z64, ids.astype(np.int64), axis=1)
    ex = np.exp(zs - zs[:, :1])
    g = ex / ex.sum(axis=1, keepdims=True)
    return ids, g


# --------------------------------------------------------------------------
# Schedule table: [LP] 01 (count tokens per expert, decide where each goes,
# keep each expert's tokens contiguous for the grouped GEMM); [MT] three
# design decisions (one table serves all four transfer modes).
# Reading: stable counting sort of flat rows r = t*k + j by expert.
# --------------------------------------------------------------------------
def schedule(ids, E: int):
    """counts[E], offsets[E+1] (exclusive scan, offsets[E] = T*k),
    perm[R] (expert-contiguous, ascending r inside an expert), inv = perm^-1."""
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = flat.size
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    if counts.size != E:
        raise ValueError("expert id out of range")
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable")
    inv = np.empty(R, dtype=np.int64)
    inv[perm] = np.arange(R)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            perm.astype(np.int32), inv.astype(np.int32))


# --------------------------------------------------------------------------
# Expert FFN: SwiGLU ([MT] three design decisions; [LP] 02).  W1 [d, 2f]
# holds the gate in columns [0, f) and the up projection in [f, 2f).
# --------------------------------------------------------------------------
def silu(u):
    return u / (1.0 + np.exp(-u))


def _sigmoid(u):
    return 1.0 / (1.0 + np.exp(-u))


def expert_ffn(xrows, W1e, W2e):
    """Y = (silu(X W1_gate) * (X W1_up)) W2 for the rows X of one expert.

    Returns (Y, H, A) with H = X W1e [m, 2f] and A = silu(H_gate) * H_up."""
    X = _f64(xrows)
    W1e = _f64(W1e)
    W2e = _f64(W2e)
    f = W2e.shape[0]
    H = X @ W1e
    A = silu(H[:, :f]) * H[:, f:]
    return A @ W2e, H, A


# --------------------------------------------------------------------------
# Forward: Schedule -> Dispatch -> Expert FFN -> Combine -> weighted merge
# ([LP] 03, first paragraph; dispatch/combine directions [LP] 02).
# --------------------------------------------------------------------------
def forward(x, W1, W2, ids, g):
    """Permuted forward.  x [T,d]; W1[e] -> [d,2f]; W2[e] -> [f,d] (anything
    indexable by expert id); ids [T,k]; g [T,k].  Returns (out [T,d], Yts [T,k,d]).

    Dispatch gathers Xp[p] = x[perm[p] // k] into expert order, each expert's
    FFN runs on its contiguous rows, combine writes Y back to its (t, j) slot
    (Yts), and the merge sums g[t,j] * Yts[t,j] over j."""
    x = _f64(x)
    T, d = x.shape
    ids = np.asarray(ids)
    k = ids.shape[1]
    E = len(W1)
    counts, offsets, perm, inv = schedule(ids, E)
    Xp = x[perm // k]
    Yts = np.zeros((T * k, d))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        Y, _, _ = expert_ffn(Xp[a:b], W1[e], W2[e])
        Yts[perm[a:b]] = Y
    Yts = Yts.reshape(T, k, d)
    gg = _f64(g)
    out = np.zeros((T, d))
    for j in range(k):
        out += gg[:, j:j + 1] * Yts[:, j]
    return out, Yts


def forward_tokens(x, W1, W2, ids, g, tokens=None):
    """Per-token brute force, no permutation: out[t] = sum_j g[t,j] FFN_ids[t,j](x[t]).

    Only the listed tokens are computed (all when tokens is None); rows are
    grouped by expert only so that each expert's weights are widened once."""
    x = _f64(x)
    ids = np.asarray(ids)
    T, k = ids.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    gg = _f64(g)
    out = np.zeros((len(tokens), x.shape[1]))
    pairs = {}
    for i, t in enumerate(tokens):
        for j in range(k):
            pairs.setdefault(int(ids[t, j]), []).append((i, int(t), j))
    for e, lst in pairs.items():
        rows = np.array([t for (_, t, _) in lst])
        Y, _, _ = expert_ffn(x[rows], W1[e], W2[e])
        for q, (i, t, j) in enumerate(lst):
            out[i] += gg[t, j] * Y[q]
    return out


# --------------------------------------------------------------------------
# Backward: the mirror of the forward ([LP] 02: pull reverse-combine, push
# reverse-dispatch) with the routing-weight gradient taken from the SwiGLU
# backward ([MT] three design decisions, last paragraph).
# --------------------------------------------------------------------------
def swiglu_backward(Hg, Hu, dA):
    """Gradient of A = silu(Hg) * Hu for an upstream dA: returns (dHg, dHu),
    dHg = dA * Hu * s (1 + Hg (1 - s)) with s = sigmoid(Hg), dHu = dA * silu(Hg)."""
    sg = _sigmoid(Hg)
    return dA * Hu * sg * (1.0 + Hg * (1.0 - sg)), dA * (Hg * sg)


def _expert_backward(Xe, W1e, W2e, ge, dOe):
    """Backward of one expert over its rows.

    Xe [m,d] rows of x, ge [m] routing weights, dOe [m,d] upstream grads of
    the tokens those rows belong to.  Returns dict with dg (both ways), dXe,
    dW1e, dW2e."""
    W1e = _f64(W1e)
    W2e = _f64(W2e)
    f = W2e.shape[0]
    Y, H, A = expert_ffn(Xe, W1e, W2e)
    Hg, Hu = H[:, :f], H[:, f:]
    dg_def = np.einsum("md,md->m", dOe, Y)            # <dOut_t, Y>
    dAp = dOe @ W2e.T                                  # dOut_t W2^T
    dg_fused = np.einsum("mf,mf->m", dAp, A)           # <dOut_t W2^T, A>
    dA = ge[:, None] * dAp
    dHg, dHu = swiglu_backward(Hg, Hu, dA)
    dH = np.concatenate([dHg, dHu], axis=1)
    dW2e = A.T @ (ge[:, None] * dOe)
    dW1e = _f64(Xe).T @ dH
    dXe = dH @ W1e.T
    return {"dg": dg_def, "dg_fused": dg_fused, "dX": dXe, "dW1": dW1e, "dW2": dW2e}


def dlogits_from_dg(g, ids, dg, E: int):
    """Gradient through top-k + renormalised softmax: for selected expert
    ids[t,l]: g_l (dg_l - sum_j g_j dg_j); zero for unselected experts (the
    selection is piecewise constant in the logits)."""
    g = _f64(g)
    dg = _f64(dg)
    T, k = g.shape
    s = (g * dg).sum(axis=1, keepdims=True)
    dz_sel = g * (dg - s)
    out = np.zeros((T, E))
    np.put_along_axis(out, np.asarray(ids, dtype=np.int64), dz_sel, axis=1)
    return out


def backward(x, W1, W2, ids, g, dOut):
    """Full backward.  Returns dict: dx [T,d], dW1 [E,d,2f], dW2 [E,f,d],
    dg [T,k] (= d loss / d g), dg_fused [T,k] (same value through the SwiGLU
    identity), dlogits [T,E]."""
    x = _f64(x)
    dOut = _f64(dOut)
    ids = np.asarray(ids)
    T, d = x.shape
    k = ids.shape[1]
    E = len(W1)
    gg = _f64(g)
    W1e0 = np.asarray(W1[0])
    twof = W1e0.shape[1]
    f = twof // 2
    counts, offsets, perm, inv = schedule(ids, E)
    dx = np.zeros((T, d))
    dW1 = np.zeros((E, d, twof))
    dW2 = np.zeros((E, f, d))
    dg = np.zeros(T * k)
    dgf = np.zeros(T * k)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        rows = perm[a:b]
        tok = rows // k
        r = _expert_backward(x[tok], W1[e], W2[e], gg.reshape(-1)[rows], dOut[tok])
        dg[rows] = r["dg"]
        dgf[rows] = r["dg_fused"]
        dW1[e] = r["dW1"]
        dW2[e] = r["dW2"]
        np.add.at(dx, tok, r["dX"])
    dg = dg.reshape(T, k)
    return {"dx": dx, "dW1": dW1, "dW2": dW2, "dg": dg,
            "dg_fused": dgf.reshape(T, k),
            "dlogits": dlogits_from_dg(gg, ids, dg, E)}


def backward_experts(x, W1, W2, ids, g, dOut, experts):
    """dW1[e], dW2[e] for the listed experts only (needs only their rows)."""
    x = _f64(x)
    ids = np.asarray(ids)
    k = ids.shape[1]
    flat = ids.reshape(-1)
    gflat = _f64(g).reshape(-1)
    res = {}
    for e in experts:
        rows = np.nonzero(flat == e)[0]          # ascending r, as perm orders them
        W2e = _f64(W2[e])
        f, d = W2e.shape
        if rows.size == 0:
            res[int(e)] = (np.zeros((d, 2 * f)), np.zeros((f, d)))
            continue
        tok = rows // k
        r = _expert_backward(x[tok], W1[e], W2e, gflat[rows], _f64(dOut[tok]))
        res[int(e)] = (r["dW1"], r["dW2"])
    return res


def backward_tokens(x, W1, W2, ids, g, dOut, tokens):
    """dx[t], dg[t,:] and dlogits[t,:] for the listed tokens only."""
    x = _f64(x)
    ids = np.asarray(ids)
    T, k = ids.shape
    E = len(W1)
    gg = _f64(g)
    tokens = np.asarray(tokens)
    dx = np.zeros((len(tokens), x.shape[1]))
    dg = np.zeros((len(tokens), k))
    pairs = {}
    for i, t in enumerate(tokens):
        for j in range(k):
            pairs.setdefault(int(ids[t, j]), []).append((i, int(t), j))
    for e, lst in pairs.items():
        tok = np.array([t for (_, t, _) in lst])
        ge = np.array([gg[t, j] for (_, t, j) in lst])
        r = _expert_backward(x[tok], W1[e], W2[e], ge, _f64(dOut[tok]))
        for q, (i, t, j) in enumerate(lst):
            dx[i] += r["dX"][q]
            dg[i, j] = r["dg"][q]
    dl = dlogits_from_dg(gg[tokens], ids[tokens], dg, E)
    return {"dx": dx, "dg": dg, "dlogits": dl}


# --------------------------------------------------------------------------
# MXFP8 ([LP] 02, MXFP8 paragraph; [MT] three design decisions, on its BF16 and MXFP8 modes).
# The pages do not give the block format; the reading is the OCP MX format:
# blocks of 32 consecutive elements along the contraction dimension share a
# UE8M0 power-of-two scale 2^s; elements are FP8 E4M3 (bias 7, max 448,
# subnormals down to 2^-9, no infinities, S.1111.111 = NaN).
# Scale reading: the smallest s with amax <= 448 * 2^s (never saturates),
# clamped to [-127, 127]; an all-zero block takes s = -127.
# --------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_encode(y):
    """Round-to-nearest-even of fp64 values into E4M3 codes (uint8), with
    saturation to +-448 (satfinite).  The sign bit is kept (so -0.0 -> 0x80)."""
    y = _f64(y)
    if np.any(~np.isfinite(y)):
        raise ValueError("non-finite input")
    sign = np.signbit(y)
    a = np.abs(y)
    _, q = np.frexp(a)                   # a = m * 2^q, m in [0.5, 1); a == 0 -> q = 0
    e = np.maximum(q - 1, -6)            # binade exponent; subnormals share 2^-6's quantum
    quantum = np.ldexp(1.0, e - 3)       # 3 mantissa bits
    r = np.round(a / quantum) * quantum  # np.round: half to even; a/quantum is exact
    r = np.minimum(r, E4M3_MAX)
    code = np.zeros(a.shape, dtype=np.int64)
    normal = r >= 2.0 ** -6
    _, qr = np.frexp(np.where(normal, r, 1.0))
    er = qr - 1                          # floor(log2 r) for normal r
    mant = np.where(normal, np.round((r / np.ldexp(1.0, er) - 1.0) * 8.0), 0)
    code = np.where(normal, ((er + 7) << 3) | mant.astype(np.int64),
                    np.round(r / 2.0 ** -9).astype(np.int64))
    code = code | (sign.astype(np.int64) << 7)
    return code.astype(np.uint8)


def e4m3_decode(codes):
    """Value of E4M3 codes (fp64); 0x7F / 0xFF decode to NaN."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where((c >> 7) & 1, -1.0, 1.0)
    E = (c >> 3) & 0xF
    M = c & 0x7
    v = np.where(E == 0, M * 2.0 ** -9, (1.0 + M / 8.0) * np.ldexp(1.0, E - 7))
    v = np.where((c & 0x7F) == 0x7F, np.nan, v)
    return s * v


def mxfp8_quantize(v, axis: int = -1):
    """Quantise along `axis` in blocks of 32.  Returns (codes uint8, same shape
    as v; scales uint8 with the axis length divided by 32; byte = s + 127)."""
    v = np.moveaxis(_f64(v), axis, -1)
    K = v.shape[-1]
    if K % 32:
        raise ValueError("axis length must be a multiple of 32")
    b = v.reshape(*v.shape[:-1], K // 32, 32)
    amax = np.abs(b).max(axis=-1)
    m, q = np.frexp(amax)
    s = np.where(m <= 0.875, q - 9, q - 8)
    s = np.where(amax == 0, -127, s)
    s = np.clip(s, -127, 127)
    y = b * np.ldexp(1.0, -s)[..., None]
    codes = e4m3_encode(y).reshape(v.shape)
    scales = (s + 127).astype(np.uint8)
    return np.moveaxis(codes, -1, axis), np.moveaxis(scales, -1, axis)


def mxfp8_dequantize(codes, scales, axis: int = -1):
    c = np.moveaxis(np.asarray(codes), axis, -1)
    sc = np.moveaxis(np.asarray(scales), axis, -1).astype(np.int64)
    K = c.shape[-1]
    vals = e4m3_decode(c).reshape(*c.shape[:-1], K // 32, 32)
    vals = vals * np.ldexp(1.0, sc - 127)[..., None]
    return np.moveaxis(vals.reshape(c.shape), -1, axis)


def _qdq(v, axis):
    c, s = mxfp8_quantize(v, axis)
    return mxfp8_dequantize(c, s, axis)


# Names of the quantised GEMM operands, "<GEMM>.<operand>".  The MXFP8 forward
# and backward below quantise every one of them by default; `quantise` may
# name a subset (the others pass through unchanged) so that each operand's
# quantisation axis can be checked on its own.
FORWARD_OPERANDS = ("fwd.x", "fwd.W1", "fwd.A", "fwd.W2")
BACKWARD_OPERANDS = ("fwd.x", "fwd.W1", "dgrad2.dO", "dgrad2.W2", "dgrad1.dH", "dgrad1.W1",
                     "wgrad1.X", "wgrad1.dH", "wgrad2.gA", "wgrad2.dO")


def _quantiser(qdq, quantise, names):
    """apply(v, axis, name): qdq(v, axis) (MXFP8 by default) when `name` is
    among `quantise` (all of `names` when None), else v unchanged."""
    q = _qdq if qdq is None else qdq
    chosen = set(names if quantise is None else quantise)
    unknown = chosen - set(names)
    if unknown:
        raise ValueError(f"unknown operands {sorted(unknown)}")

    def apply(v, axis, name):
        return q(v, axis) if name in chosen else v
    return apply


def forward_mxfp8(x, W1, W2, ids, g, tokens=None, qdq=None, quantise=None):
    """Per-token forward with MXFP8 operands ([LP] 02: activation quantisation
    fused into dispatch and into the SwiGLU data path).  Each GEMM quantises
    both operands along its contraction dimension: x along d and W1[e] [d, 2f]
    along d (GEMM1), the SwiGLU output A along f and W2[e] [f, d] along f
    (GEMM2); every product is then exact in fp64.  qdq(v, axis) is the
    quantise-dequantise step (MXFP8 by default; the identity gives the
    unquantised layer); `quantise` names the operands it applies to
    (FORWARD_OPERANDS; all by default).  Returns out for `tokens`."""
    q = _quantiser(qdq, quantise, FORWARD_OPERANDS)
    x = _f64(x)
    ids = np.asarray(ids)
    T, k = ids.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens)
    gg = _f64(g)
    xq = q(x[tokens], 1, "fwd.x")
    out = np.zeros((len(tokens), x.shape[1]))
    pairs = {}
    for i, t in enumerate(tokens):
        for j in range(k):
            pairs.setdefault(int(ids[t, j]), []).append((i, int(t), j))
    for e, lst in pairs.items():
        W1q = q(_f64(W1[e]), 0, "fwd.W1")
        W2q = q(_f64(W2[e]), 0, "fwd.W2")
        f = W2q.shape[0]
        Xe = xq[[i for (i, _, _) in lst]]
        H = Xe @ W1q
        A = silu(H[:, :f]) * H[:, f:]
        Aq = q(A, 1, "fwd.A")
        Y = Aq @ W2q
        for r, (i, t, j) in enumerate(lst):
            out[i] += gg[t, j] * Y[r]
    return out


def _pad_rows(v, mult: int = 32):
    """v [m, n] with zero rows appended up to a multiple of `mult` rows."""
    m = v.shape[0]
    pad = (-m) % mult
    return np.concatenate([v, np.zeros((pad, v.shape[1]))], axis=0) if pad else v


def _expert_backward_mxfp8(Xe, W1e, W2e, ge, dOe, q):
    """One expert's MXFP8 backward over its rows (in the stable expert order):
    q(v, axis, name) quantises operand `name`.  Returns dict dg, dX, dW1, dW2."""
    W1e = _f64(W1e)
    W2e = _f64(W2e)
    f = W2e.shape[0]
    H = q(Xe, 1, "fwd.x") @ q(W1e, 0, "fwd.W1")
    Hg, Hu = H[:, :f], H[:, f:]
    A = silu(Hg) * Hu
    dAp = q(dOe, 1, "dgrad2.dO") @ q(W2e, 1, "dgrad2.W2").T
    dg = np.einsum("mf,mf->m", dAp, A)
    dA = ge[:, None] * dAp
    dH = np.concatenate(swiglu_backward(Hg, Hu, dA), axis=1)
    return {"dg": dg,
            "dX": q(dH, 1, "dgrad1.dH") @ q(W1e, 1, "dgrad1.W1").T,
            "dW1": q(_pad_rows(Xe), 0, "wgrad1.X").T @ q(_pad_rows(dH), 0, "wgrad1.dH"),
            "dW2": q(_pad_rows(ge[:, None] * A), 0, "wgrad2.gA").T @ q(_pad_rows(dOe), 0, "wgrad2.dO")}


def backward_mxfp8(x, W1, W2, ids, g, dOut, qdq=None, quantise=None):
    """Full backward with MXFP8 operands.

    Reading (the pages name an MXFP8 mode for the layer, [MT] three design
    decisions, on its BF16 and MXFP8 modes, and put the quantisation on the
    GEMMs' data path, [LP] 02, but do not say how the backward quantises):
    every GEMM quantises both
    of its operands along its own contraction dimension, in blocks of 32 with
    the scale rule above; for the weight-gradient GEMMs that dimension is the
    expert's rows in the stable expert order, blocked from the start of the
    expert's segment, the last block padded with zero rows.  Per expert e with
    rows X (of x), weights g, upstream rows dO:
      forward, as forward_mxfp8:  H = q_d(X) q_d(W1e),  A = silu(Hg) * Hu
      dgrad2   (K = d):   dA' = q_d(dO) q_d(W2e)^T        (W2e [f, d])
      routing-weight gradient fused into the SwiGLU backward: dg = <dA', A>
      SwiGLU backward (fp64) on dA = g dA'  ->  dH = [dHg | dHu]
      dgrad1   (K = 2f):  dX = q_2f(dH) q_2f(W1e)^T       (W1e [d, 2f])
      wgrad1   (K = rows): dW1e = q_m(X)^T q_m(dH)
      wgrad2   (K = rows): dW2e = q_m(g A)^T q_m(dO)
    dx[t] sums its rows' dX in slot order; dlogits follows from dg as in
    backward().  qdq(v, axis) is the quantise-dequantise step (MXFP8 by
    default); the identity turns this into backward() (its dg_fused).
    `quantise` names the operands qdq applies to (BACKWARD_OPERANDS; all by
    default).  Returns dict: dx, dW1, dW2, dg (fused), dlogits."""
    q = _quantiser(qdq, quantise, BACKWARD_OPERANDS)
    x = _f64(x)
    dOut = _f64(dOut)
    ids = np.asarray(ids)
    T, d = x.shape
    k = ids.shape[1]
    E = len(W1)
    gg = _f64(g)
    twof = np.asarray(W1[0]).shape[1]
    f = twof // 2
    counts, offsets, perm, inv = schedule(ids, E)
    dx = np.zeros((T, d))
    dW1 = np.zeros((E, d, twof))
    dW2 = np.zeros((E, f, d))
    dg = np.zeros(T * k)
    dX_rows = np.zeros((T * k, d))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        rows = perm[a:b]
        tok = rows // k
        r = _expert_backward_mxfp8(x[tok], W1[e], W2[e], gg.reshape(-1)[rows], dOut[tok], q)
        dg[rows] = r["dg"]
        dX_rows[rows] = r["dX"]
        dW1[e] = r["dW1"]
        dW2[e] = r["dW2"]
    for j in range(k):  # slot order
        dx += dX_rows[np.arange(T) * k + j]
    dg = dg.reshape(T, k)
    return {"dx": dx, "dW1": dW1, "dW2": dW2, "dg": dg,
            "dlogits": dlogits_from_dg(gg, ids, dg, E)}


def backward_mxfp8_experts(x, W1, W2, ids, g, dOut, experts):
    """dW1[e], dW2[e] and the routing-weight gradient of expert e's rows, with
    MXFP8 operands as in backward_mxfp8, for the listed experts only (each
    needs only its own rows).  Returns {e: (dW1e, dW2e, rows, dg_rows)}."""
    q = _quantiser(None, None, BACKWARD_OPERANDS)
    x = _f64(x)
    ids = np.asarray(ids)
    k = ids.shape[1]
    flat = ids.reshape(-1)
    gflat = _f64(g).reshape(-1)
    res = {}
    for e in experts:
        rows = np.nonzero(flat == e)[0]          # ascending r, as perm orders them
        W2e = _f64(W2[e])
        f, d = W2e.shape
        if rows.size == 0:
            res[int(e)] = (np.zeros((d, 2 * f)), np.zeros((f, d)), rows, np.zeros(0))
            continue
        tok = rows // k
        r = _expert_backward_mxfp8(x[tok], W1[e], W2e, gflat[rows], _f64(dOut[tok]), q)
        res[int(e)] = (r["dW1"], r["dW2"], rows, r["dg"])
    return res
