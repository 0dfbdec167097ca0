// api.cu -- the C ABI declared in include/moe.h: argument validation,
// workspace layout and the launch sequence of each call.  No call allocates
// device memory or synchronises the stream (moe_read_status excepted).
#include <cuda_bf16.h>
#include <stdio.h>
#include <string.h>

#include "moe_internal.h"

namespace moe {

int g_tile_scheduler = MOE_GEMM_CLC ? 1 : 0;

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool config_valid(const moe_config* c) {
  if (c == nullptr) return false;
  if (c->T < 1 || c->d < 64 || c->f < 64 || c->E < 1 || c->k < 1) return false;
  if (c->E > kMaxE || c->k > kMaxK || c->k > c->E) return false;
  if (c->d % 64 || c->f % 64) return false;
  if (c->prec != MOE_BF16 && c->prec != MOE_MXFP8) return false;
  if (c->prec == MOE_MXFP8 && (c->d % 128 || c->f % 128)) return false;
  if ((int64_t)c->T * c->k > (int64_t)1 << 28) return false;
  if (c->minibatch_rows < 0 || c->minibatch_rows > (1 << 24)) return false;
  if (c->minibatch_rows > 0 && (c->ring_slots < 2 || c->ring_slots > 64)) return false;
  if (c->gather_ctas < 0) return false;
  return true;
}

WsLayout ws_layout(const moe_config* c) {
  WsLayout L;
  L.R = (int64_t)c->T * c->k;
  const int64_t nonempty = c->E < L.R ? c->E : L.R;
  L.Rp_max = (int64_t)align_up((size_t)(L.R + nonempty * (kBM - 1)), kBM);
  L.MT_max = L.Rp_max / kBM;
  const int tb = sched_chunk_tokens(c->T, c->k);
  L.nblk = (c->T + tb - 1) / tb;
  L.nt_dg = (c->f + 255) / 256;
  const size_t A = 1024;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, A);
    return o;
  };
  const size_t rp = (size_t)L.Rp_max;
  L.hdr = take(kHdrWords * sizeof(int));
  L.hist = take((size_t)L.nblk * c->E * sizeof(int));
  L.poff = take((size_t)(c->E + 1) * sizeof(int));
  L.mt_off = take((size_t)(c->E + 1) * sizeof(int));
  L.E = c->E;
  L.pt_off = take((size_t)3 * (c->E + 1) * sizeof(int));  // pairs, then heavy and light units
  L.pos_pad = take((size_t)L.R * sizeof(int));
  L.row_of_pad = take(rp * sizeof(int));
  L.g_pad = take(rp * sizeof(float));
  L.Xp = take(rp * c->d * 2);     // bf16 rows; MXFP8: e4m3 rows + scales
  L.Abuf = take(rp * c->f * 2);   // SwiGLU output when nothing is saved
  L.Yp = take(rp * c->d * 2);     // expert outputs; backward: dX in expert order
  L.dYp = take(rp * c->d * 2);
  L.dH = take(rp * 2 * c->f * 2);
  L.gA = take(rp * c->f * 2);
  L.dgp = take(rp * L.nt_dg * sizeof(float));
  L.Aq = take(c->prec == MOE_MXFP8 ? rp * c->f + rp * (c->f / 32) : 0);
  L.dl16 = take((size_t)c->T * ((c->E + 63) / 64 * 64) * 2);
  L.Hrc = take(c->prec == MOE_BF16 ? rp * 2 * c->f * 2 : 0);
  // MXFP8 backward: dY along d [rp, d], X and dY transposed [d, rp] each, dH
  // along 2f [rp, 2f] and transposed [2f, rp], g*A transposed [f, rp]; codes
  // followed by their scale tiles (1/32 of the codes)
  L.bq = take(c->prec == MOE_MXFP8 ? (rp * c->d * 3 + rp * 2 * c->f * 2 + rp * c->f) / 32 * 33 : 0);
  if (c->minibatch_rows > 0) {
    L.ring = take((size_t)c->ring_slots * ring_window_rows(*c) * c->d * 2);
    L.ctr_bytes = (size_t)(2 * c->ring_slots + 3 + L.MT_max) * sizeof(int);
    L.ctr = take(L.ctr_bytes);
  }
  L.total = off;
  return L;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

static bool aligned(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 127) == 0; }

static bool sched_ok(const moe_sched& s) {
  return aligned(s.topk_ids) && aligned(s.topk_w) && aligned(s.counts) && aligned(s.offsets) &&
         aligned(s.perm) && aligned(s.inv);
}

static moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

namespace {
struct Trace {
  int cap = 0, n = 0;
  cudaEvent_t* ev = nullptr;
  const char** names = nullptr;
};
Trace g_trace;

void trace_free() {
  for (int i = 0; i < 2 * g_trace.cap; ++i) cudaEventDestroy(g_trace.ev[i]);
  delete[] g_trace.ev;
  delete[] g_trace.names;
  g_trace = Trace();
}
}  // namespace

void trace_before(const char* name, cudaStream_t st) {
  if (g_trace.n >= g_trace.cap) return;
  g_trace.names[g_trace.n] = name;
  cudaEventRecord(g_trace.ev[2 * g_trace.n], st);
}

void trace_after(cudaStream_t st) {
  if (g_trace.n >= g_trace.cap) return;
  cudaEventRecord(g_trace.ev[2 * g_trace.n + 1], st);
  ++g_trace.n;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_config* cfg) {
  if (!config_valid(cfg)) return 0;
  return ws_layout(cfg).total;
}

int64_t moe_saved_rows(const moe_config* cfg) {
  if (!config_valid(cfg)) return 0;
  return ws_layout(cfg).Rp_max;
}

int32_t moe_min_minibatch(int32_t compute_sms, int32_t bm, int32_t bn, int32_t n_cols) {
  if (compute_sms <= 0 || bm <= 0 || bn <= 0 || n_cols <= 0) return 0;
  const int64_t num = 2ll * compute_sms * bm * bn;
  const int64_t v = (num + n_cols - 1) / n_cols;
  return v > INT32_MAX ? INT32_MAX : (int32_t)v;
}

moe_status moe_schedule(const moe_config* cfg, const float* logits, moe_sched sched, void* ws,
                        size_t ws_bytes, moe_stream_t stream) {
  if (!config_valid(cfg) || !aligned(logits) || !sched_ok(sched) || !aligned(ws))
    return MOE_ERR_INVALID_ARG;
  Ws w;
  w.L = ws_layout(cfg);
  w.base = static_cast<uint8_t*>(ws);
  if (ws_bytes < w.L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_schedule(*cfg, logits, sched, w, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_route(const moe_config* cfg, const moe_bf16* x, const moe_bf16* w_router,
                     float* logits, moe_sched sched, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!config_valid(cfg) || !aligned(x) || !aligned(w_router) || !sched_ok(sched) || !aligned(ws))
    return MOE_ERR_INVALID_ARG;
  if (logits == nullptr ? cfg->E > 256 : !aligned(logits)) return MOE_ERR_INVALID_ARG;
  Ws w;
  w.L = ws_layout(cfg);
  w.base = static_cast<uint8_t*>(ws);
  if (ws_bytes < w.L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const moe_config& c = *cfg;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool fused = c.E <= 256;
  cudaError_t e = cudaMemsetAsync(w.hdr(), 0, kHdrWords * sizeof(int), st);
  if (e == cudaSuccess)
    e = router_gemm(c, w, reinterpret_cast<const __nv_bfloat16*>(x),
                    reinterpret_cast<const __nv_bfloat16*>(w_router), logits,
                    fused ? sched.topk_ids : nullptr, sched.topk_w, st);
  if (e == cudaSuccess)
    e = fused ? launch_schedule_tail(c, sched, w, st) : launch_schedule_from_logits(c, logits, sched, w, st);
  return cuda_status(e);
}

moe_status moe_router_backward(const moe_config* cfg, const moe_bf16* x, const moe_bf16* w_router,
                               const float* dlogits, moe_bf16* dx_router, moe_bf16* dw_router,
                               void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!config_valid(cfg) || !aligned(x) || !aligned(w_router) || !aligned(dlogits) ||
      !aligned(dx_router) || !aligned(dw_router) || !aligned(ws))
    return MOE_ERR_INVALID_ARG;
  Ws w;
  w.L = ws_layout(cfg);
  w.base = static_cast<uint8_t*>(ws);
  if (ws_bytes < w.L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const moe_config& c = *cfg;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int Epad = (c.E + 63) / 64 * 64;
  auto* dl16 = static_cast<__nv_bfloat16*>(w.at(w.L.dl16));
  cudaError_t e = launch_to_bf16_padded(dlogits, c.T, c.E, Epad, dl16, st);
  if (e == cudaSuccess)
    e = router_bwd(c, w, dl16, Epad, reinterpret_cast<const __nv_bfloat16*>(x),
                   reinterpret_cast<const __nv_bfloat16*>(w_router),
                   reinterpret_cast<__nv_bfloat16*>(dx_router),
                   reinterpret_cast<__nv_bfloat16*>(dw_router), st);
  return cuda_status(e);
}

moe_status moe_quantize_mxfp8(const moe_bf16* w, int64_t batch, int32_t K, int32_t N, uint8_t* q,
                              uint8_t* scales, moe_stream_t stream) {
  if (!aligned(w) || !aligned(q) || !aligned(scales) || batch < 1 || K < 128 || N < 128 ||
      K % 128 || N % 128)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_mxfp8(reinterpret_cast<const __nv_bfloat16*>(w), batch, K, N,
                                           q, scales, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_quantize_mxfp8_rows(const moe_bf16* w, int64_t rows, int32_t K, uint8_t* q,
                                   uint8_t* scales, moe_stream_t stream) {
  if (!aligned(w) || !aligned(q) || !aligned(scales) || rows < 128 || rows % 128 || K < 128 || K % 128)
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quant_rows(reinterpret_cast<const __nv_bfloat16*>(w), rows, K, nullptr, q,
                                       scales, reinterpret_cast<cudaStream_t>(stream),
                                       "quantize_weight_rows"));
}

moe_status moe_forward(const moe_config* cfg, const moe_bf16* x, const void* w1,
                       const uint8_t* w1_scales, const void* w2, const uint8_t* w2_scales,
                       moe_sched sched, moe_bf16* out, const moe_saved* saved, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  if (!config_valid(cfg) || !aligned(x) || !aligned(w1) || !aligned(w2) || !aligned(out) ||
      !sched_ok(sched) || !aligned(ws))
    return MOE_ERR_INVALID_ARG;
  if (saved != nullptr && (!aligned(saved->H) || !aligned(saved->A))) return MOE_ERR_INVALID_ARG;
  Ws W;
  W.L = ws_layout(cfg);
  W.base = static_cast<uint8_t*>(ws);
  if (ws_bytes < W.L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const moe_config& c = *cfg;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (c.minibatch_rows > 0 && c.prec == MOE_MXFP8) {
    // persistent kernel with MXFP8 operands
    if (!aligned(w1_scales) || !aligned(w2_scales)) return MOE_ERR_INVALID_ARG;
    if (c.gather_ctas >= num_sms()) return MOE_ERR_INVALID_ARG;
    const cudaError_t e = ring_forward_mx(
        c, W, sched.counts, reinterpret_cast<const __nv_bfloat16*>(x), static_cast<const uint8_t*>(w1),
        w1_scales, static_cast<const uint8_t*>(w2), w2_scales, sched.topk_w,
        saved ? reinterpret_cast<__nv_bfloat16*>(saved->A) : nullptr,
        saved ? reinterpret_cast<__nv_bfloat16*>(saved->H) : nullptr, reinterpret_cast<__nv_bfloat16*>(out), st);
    if (e == cudaErrorCooperativeLaunchTooLarge) return MOE_ERR_UNSUPPORTED;
    return cuda_status(e);
  }
  if (c.minibatch_rows > 0) {
    // persistent kernel: SM split, ring of windows, device counters
    if (w1_scales != nullptr || w2_scales != nullptr) return MOE_ERR_INVALID_ARG;
    if (c.gather_ctas >= num_sms()) return MOE_ERR_INVALID_ARG;
    auto* A = saved ? reinterpret_cast<__nv_bfloat16*>(saved->A)
                    : static_cast<__nv_bfloat16*>(W.at(W.L.Abuf));
    auto* H = saved ? reinterpret_cast<__nv_bfloat16*>(saved->H) : nullptr;
    const cudaError_t e = ring_forward(c, W, sched.counts, reinterpret_cast<const __nv_bfloat16*>(x),
                                       static_cast<const __nv_bfloat16*>(w1),
                                       static_cast<const __nv_bfloat16*>(w2), sched.topk_w, A, H,
                                       reinterpret_cast<__nv_bfloat16*>(out), st);
    if (e == cudaErrorCooperativeLaunchTooLarge) return MOE_ERR_UNSUPPORTED;
    return cuda_status(e);
  }
  if (c.prec == MOE_MXFP8) {
    if (!aligned(w1_scales) || !aligned(w2_scales)) return MOE_ERR_INVALID_ARG;
    const size_t rp = (size_t)W.L.Rp_max;
    auto* Xq = static_cast<uint8_t*>(W.at(W.L.Xp));
    uint8_t* Xs = Xq + rp * c.d;
    auto* Aq = static_cast<uint8_t*>(W.at(W.L.Aq));
    uint8_t* As = Aq + rp * c.f;
    auto* Yp = static_cast<__nv_bfloat16*>(W.at(W.L.Yp));
    cudaError_t e = launch_gather_mxfp8(c, W, reinterpret_cast<const __nv_bfloat16*>(x), Xq, Xs, st);
    if (e == cudaSuccess)
      e = gemm_fwd1_mx(c, W, sched.counts, Xq, Xs, static_cast<const uint8_t*>(w1), w1_scales, Aq, As,
                       saved ? reinterpret_cast<__nv_bfloat16*>(saved->A) : nullptr,
                       saved ? reinterpret_cast<__nv_bfloat16*>(saved->H) : nullptr, st);
    if (e == cudaSuccess)
      e = gemm_fwd2_mx(c, W, Aq, As, static_cast<const uint8_t*>(w2), w2_scales, Yp, st);
    if (e == cudaSuccess)
      e = launch_merge(c, W, Yp, sched.topk_w, reinterpret_cast<__nv_bfloat16*>(out), st);
    return cuda_status(e);
  }
  if (w1_scales != nullptr || w2_scales != nullptr) return MOE_ERR_INVALID_ARG;

  auto* Xp = static_cast<__nv_bfloat16*>(W.at(W.L.Xp));
  auto* A = saved ? reinterpret_cast<__nv_bfloat16*>(saved->A)
                  : static_cast<__nv_bfloat16*>(W.at(W.L.Abuf));
  auto* H = saved ? reinterpret_cast<__nv_bfloat16*>(saved->H) : nullptr;
  auto* Yp = static_cast<__nv_bfloat16*>(W.at(W.L.Yp));
  cudaError_t e = launch_gather(c, W, reinterpret_cast<const __nv_bfloat16*>(x), Xp, nullptr,
                                nullptr, st);
  if (e == cudaSuccess)
    e = gemm_fwd1(c, W, sched.counts, Xp, static_cast<const __nv_bfloat16*>(w1), A, H, st);
  if (e == cudaSuccess) e = gemm_fwd2(c, W, sched.counts, A, static_cast<const __nv_bfloat16*>(w2), Yp, st);
  if (e == cudaSuccess)
    e = launch_merge(c, W, Yp, sched.topk_w, reinterpret_cast<__nv_bfloat16*>(out), st);
  return cuda_status(e);
}

moe_status moe_backward(const moe_config* cfg, const moe_bf16* dout, const moe_bf16* x,
                        const moe_bf16* w1, const moe_bf16* w2, moe_sched sched,
                        const moe_saved* saved, moe_bf16* dx, moe_bf16* dw1, moe_bf16* dw2,
                        float* dtopk_w, float* dlogits, void* ws, size_t ws_bytes,
                        moe_stream_t stream) {
  if (!config_valid(cfg) || !aligned(dout) || !aligned(x) || !aligned(w1) || !aligned(w2) ||
      !sched_ok(sched) || !aligned(dx) || !aligned(dw1) || !aligned(dw2) || !aligned(dtopk_w) ||
      !aligned(ws))
    return MOE_ERR_INVALID_ARG;
  if (dlogits != nullptr && !aligned(dlogits)) return MOE_ERR_INVALID_ARG;
  if (saved != nullptr && (!aligned(saved->H) || !aligned(saved->A))) return MOE_ERR_INVALID_ARG;
  if (cfg->prec != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  Ws W;
  W.L = ws_layout(cfg);
  W.base = static_cast<uint8_t*>(ws);
  if (ws_bytes < W.L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const moe_config& c = *cfg;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto bf = [](const moe_bf16* p) { return reinterpret_cast<const __nv_bfloat16*>(p); };
  auto* Xp = static_cast<__nv_bfloat16*>(W.at(W.L.Xp));
  auto* dYp = static_cast<__nv_bfloat16*>(W.at(W.L.dYp));
  auto* dH = static_cast<__nv_bfloat16*>(W.at(W.L.dH));
  auto* gA = static_cast<__nv_bfloat16*>(W.at(W.L.gA));
  auto* dXp = static_cast<__nv_bfloat16*>(W.at(W.L.Yp));
  auto* dgp = static_cast<float*>(W.at(W.L.dgp));
  // without saved activations H and A are recomputed from the re-gathered
  // rows by the forward's own GEMM1 (same tiles, same K order: the same bits)
  auto* Hrc = static_cast<__nv_bfloat16*>(W.at(W.L.Hrc));
  auto* Arc = static_cast<__nv_bfloat16*>(W.at(W.L.Abuf));
  const auto* Hs = saved ? reinterpret_cast<const __nv_bfloat16*>(saved->H) : Hrc;
  const auto* As = saved ? reinterpret_cast<const __nv_bfloat16*>(saved->A) : Arc;

  // after a ring forward its last windows are still in the ring: the
  // re-gather walks the rows in reverse and takes those from the ring
  RingSrc rs;
  rs.ring = static_cast<const __nv_bfloat16*>(W.at(W.L.ring));
  rs.mb = ring_window_rows(c);
  rs.slots = c.ring_slots;
  cudaError_t e = launch_gather(c, W, bf(x), Xp, bf(dout), dYp, st, c.minibatch_rows > 0 ? &rs : nullptr);
  if (e == cudaSuccess && saved == nullptr)
    e = gemm_fwd1(c, W, sched.counts, Xp, bf(w1), Arc, Hrc, st, "recompute_gemm1");
  if (e == cudaSuccess) e = gemm_dgrad2(c, W, dYp, bf(w2), Hs, As, dH, gA, dgp, st);
  if (e == cudaSuccess) e = launch_dg_reduce(c, W, sched, dtopk_w, dlogits, st);
  if (e == cudaSuccess)
    e = gemm_wgrad(c, W, sched, gA, c.f, dYp, c.d, reinterpret_cast<__nv_bfloat16*>(dw2), st);
  if (e == cudaSuccess)
    e = gemm_wgrad(c, W, sched, Xp, c.d, dH, 2 * c.f, reinterpret_cast<__nv_bfloat16*>(dw1), st);
  if (e == cudaSuccess) e = gemm_dgrad1(c, W, sched.counts, dH, bf(w1), dXp, st);
  if (e == cudaSuccess) e = launch_merge(c, W, dXp, nullptr, reinterpret_cast<__nv_bfloat16*>(dx), st);
  return cuda_status(e);
}

moe_status moe_workspace_region(const moe_config* cfg, int32_t region, size_t* offset,
                                size_t* bytes) {
  if (!config_valid(cfg) || offset == nullptr || bytes == nullptr) return MOE_ERR_INVALID_ARG;
  if (cfg->prec != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(cfg);
  const size_t rp = (size_t)L.Rp_max;
  switch (region) {
    case MOE_WS_XQ_CODES: *offset = L.Xp; *bytes = rp * cfg->d; return MOE_OK;
    case MOE_WS_XQ_SCALES: *offset = L.Xp + rp * cfg->d; *bytes = rp * (cfg->d / 32); return MOE_OK;
    case MOE_WS_AQ_CODES: *offset = L.Aq; *bytes = rp * cfg->f; return MOE_OK;
    case MOE_WS_AQ_SCALES: *offset = L.Aq + rp * cfg->f; *bytes = rp * (cfg->f / 32); return MOE_OK;
    default: break;
  }
  // the MXFP8 backward's operands, in the order moe_backward_mxfp8 carves them
  const size_t d = cfg->d, f = cfg->f;
  const size_t sizes[6] = {rp * d, d * rp, d * rp, rp * 2 * f, 2 * f * rp, f * rp};
  const int first = MOE_WS_DYQ_CODES;
  if (region < first || region >= first + 12) return MOE_ERR_INVALID_ARG;
  size_t off = L.bq;
  const int i = (region - first) / 2;
  for (int j = 0; j < i; ++j) off += sizes[j] + sizes[j] / 32;
  if ((region - first) % 2 == 0) {
    *offset = off;
    *bytes = sizes[i];
  } else {
    *offset = off + sizes[i];
    *bytes = sizes[i] / 32;
  }
  return MOE_OK;
}

moe_status moe_backward_mxfp8(const moe_config* cfg, const moe_bf16* dout, const moe_bf16* x,
                              const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q,
                              const uint8_t* w2s, moe_sched sched, const moe_saved* saved, moe_bf16* dx,
                              moe_bf16* dw1, moe_bf16* dw2, float* dtopk_w, float* dlogits, void* ws,
                              size_t ws_bytes, moe_stream_t stream) {
  if (!config_valid(cfg) || cfg->prec != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
  if (!aligned(dout) || !aligned(x) || !aligned(w1q) || !aligned(w1s) || !aligned(w2q) || !aligned(w2s) ||
      !sched_ok(sched) || !aligned(dx) || !aligned(dw1) || !aligned(dw2) || !aligned(dtopk_w) ||
      !aligned(ws))
    return MOE_ERR_INVALID_ARG;
  if (dlogits != nullptr && !aligned(dlogits)) return MOE_ERR_INVALID_ARG;
  if (saved == nullptr || !aligned(saved->H) || !aligned(saved->A)) return MOE_ERR_INVALID_ARG;
  Ws W;
  W.L = ws_layout(cfg);
  W.base = static_cast<uint8_t*>(ws);
  if (ws_bytes < W.L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const moe_config& c = *cfg;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto bf = [](const moe_bf16* p) { return reinterpret_cast<const __nv_bfloat16*>(p); };
  const size_t rp = (size_t)W.L.Rp_max, d = c.d, f = c.f;
  auto* Xp = static_cast<__nv_bfloat16*>(W.at(W.L.Xp));
  auto* dYp = static_cast<__nv_bfloat16*>(W.at(W.L.dYp));
  auto* dXp = static_cast<__nv_bfloat16*>(W.at(W.L.Yp));
  auto* dgp = static_cast<float*>(W.at(W.L.dgp));
  // quantised operands, codes then scale tiles
  uint8_t* b = static_cast<uint8_t*>(W.at(W.L.bq));
  auto carve = [&](size_t n) {
    uint8_t* q = b;
    b += n + n / 32;
    return q;
  };
  uint8_t* dYq = carve(rp * d);
  uint8_t* XqT = carve(d * rp);
  uint8_t* dYqT = carve(d * rp);
  uint8_t* dHq = carve(rp * 2 * f);
  uint8_t* dHqT = carve(2 * f * rp);
  uint8_t* gAqT = carve(f * rp);
  auto sc = [](uint8_t* q, size_t n) { return q + n; };
  const int* rows = W.hdr() + kHdrRpTotal;
  const auto* Hs = reinterpret_cast<const __nv_bfloat16*>(saved->H);
  const auto* As = reinterpret_cast<const __nv_bfloat16*>(saved->A);

  cudaError_t e = launch_gather(c, W, bf(x), Xp, bf(dout), dYp, st);
  if (e == cudaSuccess) e = launch_quant_rows(dYp, (int64_t)rp, c.d, rows, dYq, sc(dYq, rp * d), st, "quant_dy_rows");
  if (e == cudaSuccess)
    e = launch_quant_cols(Xp, (int64_t)rp, c.d, rows, XqT, sc(XqT, d * rp), (int)rp, st, "quant_x_cols");
  if (e == cudaSuccess)
    e = launch_quant_cols(dYp, (int64_t)rp, c.d, rows, dYqT, sc(dYqT, d * rp), (int)rp, st, "quant_dy_cols");
  if (e == cudaSuccess)
    e = gemm_dgrad2_mx(c, W, dYq, sc(dYq, rp * d), w2q, w2s, Hs, As, dHq, sc(dHq, rp * 2 * f), dHqT,
                       sc(dHqT, 2 * f * rp), gAqT, sc(gAqT, f * rp), dgp, st);
  if (e == cudaSuccess) e = launch_dg_reduce(c, W, sched, dtopk_w, dlogits, st);
  if (e == cudaSuccess)
    e = gemm_wgrad_mx(c, W, sched, gAqT, sc(gAqT, f * rp), c.f, dYqT, sc(dYqT, d * rp), c.d,
                      reinterpret_cast<__nv_bfloat16*>(dw2), "wgrad2_mxfp8", st);
  if (e == cudaSuccess)
    e = gemm_wgrad_mx(c, W, sched, XqT, sc(XqT, d * rp), c.d, dHqT, sc(dHqT, 2 * f * rp), 2 * c.f,
                      reinterpret_cast<__nv_bfloat16*>(dw1), "wgrad1_mxfp8", st);
  if (e == cudaSuccess) e = gemm_dgrad1_mx(c, W, dHq, sc(dHq, rp * 2 * f), w1q, w1s, dXp, st);
  if (e == cudaSuccess) e = launch_merge(c, W, dXp, nullptr, reinterpret_cast<__nv_bfloat16*>(dx), st);
  return cuda_status(e);
}

moe_status moe_read_status(const void* ws, moe_stream_t stream) {
  if (!aligned(ws)) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(h[0]);
}

moe_status moe_trace_enable(int32_t capacity) {
  if (capacity < 0 || capacity > (1 << 22)) return MOE_ERR_INVALID_ARG;
  trace_free();
  if (capacity == 0) return MOE_OK;
  g_trace.ev = new cudaEvent_t[2 * (size_t)capacity];
  g_trace.names = new const char*[capacity];
  for (int i = 0; i < 2 * capacity; ++i) {
    if (cudaEventCreate(&g_trace.ev[i]) != cudaSuccess) {
      g_trace.cap = i / 2;
      trace_free();
      return MOE_ERR_CUDA;
    }
    g_trace.cap = (i + 1) / 2;
  }
  g_trace.cap = capacity;
  g_trace.n = 0;
  return MOE_OK;
}

int32_t moe_trace_count(void) { return g_trace.n; }

moe_status moe_trace_read(int32_t i, const char** name, float* ms) {
  if (i < 0 || i >= g_trace.n || name == nullptr || ms == nullptr) return MOE_ERR_INVALID_ARG;
  if (cudaEventSynchronize(g_trace.ev[2 * i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaEventElapsedTime(ms, g_trace.ev[2 * i], g_trace.ev[2 * i + 1]) != cudaSuccess)
    return MOE_ERR_CUDA;
  *name = g_trace.names[i];
  return MOE_OK;
}

moe_status moe_set_tile_scheduler(int32_t mode) {
  if (mode != 0 && mode != 1) return MOE_ERR_INVALID_ARG;
  g_tile_scheduler = mode;
  return MOE_OK;
}

int32_t moe_get_tile_scheduler(void) { return g_tile_scheduler; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "device bounds check failed";
  }
  return "unknown status";
}

}  // extern "C"
