// moe_internal.h -- workspace layout and kernel launchers shared by the
// translation units of libmoe.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kBM = 128;           // rows of an expert tile; expert segments are padded to it

// "Thin" GEMM1 tiles: an expert's last, partial 128-row tile is computed
// swapped -- its gate / up weight slices on the MMA's M side and its rows on N
// (rounded up to 16) -- so no padding rows are multiplied.  Measured on GB300
// it pays off when the contraction is short (d = 2048: GEMM1 -20 %) and costs
// a few percent at d = 7168, so it is enabled for d <= 4096 only (and needs
// 128-column gate / up slices).  The chain and ring paths use the same rule,
// so their results stay bitwise identical.
__host__ __device__ inline bool thin_tile(int rows, int /*cnt*/) { return rows >= 1 && rows < kBM; }
inline bool gemm1_thin_enabled(const moe_config& c) { return c.f % 128 == 0 && c.d <= 4096; }

// The bf16 grouped GEMMs of the chain path can run on CTA pairs: a cluster of
// two CTAs shares one tcgen05 MMA of 256 rows (128 per CTA) whose B operand
// is split between them, so each SM loads a third less per FLOP than with a
// one-CTA 128-row tile.  That pays where the contraction is long (the row
// GEMMs, K = d, f or 2f); the weight-gradient GEMMs contract over one
// expert's rows, often a handful of 64-row steps, and run one CTA per tile.
// MOE_GEMM_PAIR=0 / 2 at build time forces one mode for every GEMM.
enum GemmKind { kGemmFwd1, kGemmFwd2, kGemmDgrad2, kGemmDgrad1, kGemmWgrad };
#ifndef MOE_GEMM_PAIR
#define MOE_GEMM_PAIR 1
#endif
inline bool gemm_pair_enabled(const moe_config&, GemmKind k) {
  if (MOE_GEMM_PAIR == 0) return false;
  if (MOE_GEMM_PAIR == 2) return true;
  return k != kGemmWgrad;
}

// Split units: a pair GEMM runs as two kernels side by side on every SM --
// the heavy units (pairs of full tiles) with fewer pipeline stages and one
// accumulator, and the light units (an expert's lone last tile of at most
// kLightRows rows, which mostly streams its weight slice from HBM) in the
// shared memory and TMEM left over -- so that the light units' weight
// streaming overlaps the heavy units' tensor work.  MOE_SPLIT_UNITS=1 at
// build time turns it on.
#ifndef MOE_SPLIT_UNITS
#define MOE_SPLIT_UNITS 0
#endif
inline bool gemm_split_units(const moe_config&) { return MOE_SPLIT_UNITS != 0; }

// The one-CTA weight-gradient GEMMs can take their work units from the
// hardware's cluster launch control instead of a static walk: a grid of one
// CTA per unit, the running CTAs cancelling the launches of the pending ones
// and taking over their units.  Chosen process-wide with
// moe_set_tile_scheduler (default MOE_GEMM_CLC at build time).
#ifndef MOE_GEMM_CLC
#define MOE_GEMM_CLC 0
#endif
extern int g_tile_scheduler;  // 0 static walk, 1 cluster launch control
inline bool gemm_clc_enabled(const moe_config&) { return g_tile_scheduler == 1; }

// A light unit: an expert's lone last 128-row tile with at most this many
// rows (the thin pair unit of an expert with a few rows), which streams its
// weight slice with little to compute.
constexpr int kLightRows = 32;
constexpr int kSchedChunk = 256;   // at most this many routed rows per histogram / scatter block
constexpr int kSchedBlocks = 152;  // chunks shrink until the schedule has this many blocks
// Tokens per schedule chunk: whole tokens (their k rows each), at most
// kSchedChunk rows, fewer for small T so that the schedule kernels still
// spread over about kSchedBlocks blocks.
__host__ __device__ inline int sched_chunk_tokens(int T, int k) {
  const int cap = kSchedChunk / k > 0 ? kSchedChunk / k : 1;
  const int want = (T + kSchedBlocks - 1) / kSchedBlocks;
  return want < 1 ? 1 : (want < cap ? want : cap);
}
constexpr int kSchedThreads = 256;
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;

// Header words at the start of the workspace.
enum HdrWord {
  kHdrStatus = 0,     // device status (moe_status code), first error wins
  kHdrWhere = 1,      // which wait / check reported it
  kHdrDone = 2,       // schedule: blocks finished (last-block ticket)
  kHdrSchedGo = 3,    // one-launch schedule: the table is ready (set by the last block)
  kHdrRpTotal = 4,    // padded rows of all experts (multiple of kBM)
  kHdrMtTotal = 5,    // kRpTotal / kBM
  kHdrInject = 8,     // fault-injection words for tests of the bounded waits (8 and 9)
  kHdrRingValid = 12, // set by the ring forward once every window has passed through the ring
  kHdrWords = 64
};

struct WsLayout {
  int64_t R = 0, Rp_max = 0, MT_max = 0, nblk = 0, nt_dg = 0, E = 0;
  size_t hdr = 0, hist = 0, poff = 0, mt_off = 0, pt_off = 0, pos_pad = 0, row_of_pad = 0, g_pad = 0;
  size_t Xp = 0, Abuf = 0, Yp = 0, dYp = 0, dH = 0, gA = 0, dgp = 0, Aq = 0, ring = 0;
  size_t Hrc = 0;   // backward without saved activations: H recomputed [Rp, 2f]
  size_t bq = 0;    // MXFP8 backward: quantised operands (see ws_layout)
  size_t dl16 = 0;  // router backward: dlogits in bf16 [T, E rounded up to 64]
  size_t ctr = 0, ctr_bytes = 0;  // ring path: window counters
  size_t total = 0;
};

bool config_valid(const moe_config* c);
WsLayout ws_layout(const moe_config* c);

// Pointers into a workspace, typed.
struct Ws {
  WsLayout L;
  uint8_t* base = nullptr;
  int* hdr() const { return reinterpret_cast<int*>(base + L.hdr); }
  int* hist() const { return reinterpret_cast<int*>(base + L.hist); }
  int* poff() const { return reinterpret_cast<int*>(base + L.poff); }
  int* mt_off() const { return reinterpret_cast<int*>(base + L.mt_off); }
  int* pt_off() const { return reinterpret_cast<int*>(base + L.pt_off); }
  int* hv_off() const { return pt_off() + (L.E + 1); }   // heavy units per expert (prefix)
  int* lt_off() const { return pt_off() + 2 * (L.E + 1); }  // light units per expert (prefix)
  int* pos_pad() const { return reinterpret_cast<int*>(base + L.pos_pad); }
  int* row_of_pad() const { return reinterpret_cast<int*>(base + L.row_of_pad); }
  float* g_pad() const { return reinterpret_cast<float*>(base + L.g_pad); }
  void* at(size_t off) const { return base + off; }
};

int num_sms();

// Ring path: rows per window (minibatch_rows rounded up to 128-row tiles).
inline int ring_window_rows(const moe_config& c) { return (c.minibatch_rows + kBM - 1) / kBM * kBM; }

// Tracing hooks around every kernel launch (no-ops unless moe_trace_enable).
void trace_before(const char* name, cudaStream_t st);
void trace_after(cudaStream_t st);
struct TraceScope {
  cudaStream_t st;
  TraceScope(const char* name, cudaStream_t s) : st(s) { trace_before(name, s); }
  ~TraceScope() { trace_after(st); }
};

// ---- launchers (return a cudaError_t from the launch) ----
cudaError_t launch_schedule(const moe_config& c, const float* logits, const moe_sched& s,
                            const Ws& ws, cudaStream_t st);
// The parts of it (both expect the header words zeroed): the table from
// fp32 logits (top-k with the histograms, then the stable scatter), and the
// table from ids chosen elsewhere (histograms, scans, stable scatter).
cudaError_t launch_schedule_from_logits(const moe_config& c, const float* logits, const moe_sched& s,
                                        const Ws& ws, cudaStream_t st);
cudaError_t launch_schedule_tail(const moe_config& c, const moe_sched& s, const Ws& ws,
                                 cudaStream_t st);
// dst [T, Epad] bf16 = src [T, E] fp32 rounded, zero in columns [E, Epad).
cudaError_t launch_to_bf16_padded(const float* src, int T, int E, int Epad, __nv_bfloat16* dst,
                                  cudaStream_t st);
// The ring of windows a ring forward leaves behind: once it completed (header
// word kHdrRingValid), slot w % slots still holds the rows of each of the
// last `slots` windows w of `mb` padded rows (padding rows zero).
struct RingSrc {
  const __nv_bfloat16* ring;
  int mb, slots;
};
// dst[pp] = src[row_of_pad[pp] / k] (zero rows for padding), pp < Rp_total.
// With `ring`, the rows of src that the last windows of a completed ring
// forward still hold are read from the ring instead, and the padded rows are
// walked from the last to the first (the backward's reverse traversal).
cudaError_t launch_gather(const moe_config& c, const Ws& ws, const __nv_bfloat16* src,
                          __nv_bfloat16* dst, const __nv_bfloat16* src2, __nv_bfloat16* dst2,
                          cudaStream_t st, const RingSrc* ring = nullptr);
// MXFP8 gather: E4M3 codes [Rp, d] and UE8M0 scale tiles (mx.cuh layout).
cudaError_t launch_gather_mxfp8(const moe_config& c, const Ws& ws, const __nv_bfloat16* src,
                                uint8_t* q, uint8_t* sc, cudaStream_t st);
// out[t] = sum_j w[t,j] * rows[pos_pad[t*k+j]] (w == nullptr: plain sum).
cudaError_t launch_merge(const moe_config& c, const Ws& ws, const __nv_bfloat16* rows,
                         const float* w, __nv_bfloat16* out, cudaStream_t st);
cudaError_t launch_dg_reduce(const moe_config& c, const Ws& ws, const moe_sched& s,
                             float* dtopk_w, float* dlogits, cudaStream_t st);
cudaError_t launch_quantize_mxfp8(const __nv_bfloat16* w, int64_t batch, int K, int N, uint8_t* q,
                                  uint8_t* sc, cudaStream_t st);

// MXFP8 along the contiguous dimension: w [rows, K] -> codes [rows, K] and
// scale tiles (mx.cuh layout, k_groups = K / 128); rows_dev (nullable) caps
// the rows at a device-side count.
cudaError_t launch_quant_rows(const __nv_bfloat16* w, int64_t rows, int K, const int* rows_dev,
                              uint8_t* q, uint8_t* sc, cudaStream_t st, const char* name);
// Transposed: src [*rows_dev, K] -> codes [K, ld] (rows contiguous) and scale
// tiles over [K, ld] (blocks of 32 rows; ld a multiple of 128 >= max_rows).
cudaError_t launch_quant_cols(const __nv_bfloat16* src, int64_t max_rows, int K, const int* rows_dev,
                              uint8_t* qt, uint8_t* sct, int ld, cudaStream_t st, const char* name);
// Grouped GEMMs on tcgen05 (gemm.cu).
cudaError_t gemm_fwd1(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* Xp,
                      const __nv_bfloat16* W1, __nv_bfloat16* A, __nv_bfloat16* H, cudaStream_t st,
                      const char* name = "gemm1_swiglu");
cudaError_t gemm_fwd2(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* A,
                      const __nv_bfloat16* W2, __nv_bfloat16* Yp, cudaStream_t st);
cudaError_t gemm_dgrad2(const moe_config& c, const Ws& ws, const __nv_bfloat16* dYp,
                        const __nv_bfloat16* W2, const __nv_bfloat16* Hs, const __nv_bfloat16* As,
                        __nv_bfloat16* dH, __nv_bfloat16* gA, float* dgp, cudaStream_t st);
cudaError_t gemm_dgrad1(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* dH,
                        const __nv_bfloat16* W1, __nv_bfloat16* dXp, cudaStream_t st);
cudaError_t gemm_wgrad(const moe_config& c, const Ws& ws, const moe_sched& s,
                       const __nv_bfloat16* Amn, int M, const __nv_bfloat16* Bmn, int N,
                       __nv_bfloat16* dW, cudaStream_t st);
// MXFP8 backward GEMMs (gemm.cu): dgrad2 with the SwiGLU backward and the
// quantisation of dH (along 2f, and transposed along the rows) and of g*A
// (transposed), dgrad1, and the weight gradients over transposed operands.
cudaError_t gemm_dgrad2_mx(const moe_config& c, const Ws& ws, const uint8_t* dYq, const uint8_t* dYs,
                           const uint8_t* W2q, const uint8_t* W2s, const __nv_bfloat16* Hs,
                           const __nv_bfloat16* As, uint8_t* dHq, uint8_t* dHs, uint8_t* dHqT,
                           uint8_t* dHsT, uint8_t* gAqT, uint8_t* gAsT, float* dgp, cudaStream_t st);
cudaError_t gemm_dgrad1_mx(const moe_config& c, const Ws& ws, const uint8_t* dHq, const uint8_t* dHs,
                           const uint8_t* W1q, const uint8_t* W1s, __nv_bfloat16* dXp, cudaStream_t st);
cudaError_t gemm_wgrad_mx(const moe_config& c, const Ws& ws, const moe_sched& s, const uint8_t* AqT,
                          const uint8_t* AsT, int M, const uint8_t* BqT, const uint8_t* BsT, int N,
                          __nv_bfloat16* dW, const char* name, cudaStream_t st);
// Persistent forward with an SM split and a ring of windows (ring.cu).
cudaError_t ring_forward(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* x,
                         const __nv_bfloat16* W1, const __nv_bfloat16* W2, const float* topk_w,
                         __nv_bfloat16* A, __nv_bfloat16* H, __nv_bfloat16* out, cudaStream_t st);
// The same with MXFP8 operands: the gather quantises rows in the ring, the
// weights come as E4M3 codes and scale tiles (moe_quantize_mxfp8); A is saved
// in bf16 only when A / H are given.
cudaError_t ring_forward_mx(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* x,
                            const uint8_t* W1q, const uint8_t* W1s, const uint8_t* W2q, const uint8_t* W2s,
                            const float* topk_w, __nv_bfloat16* A, __nv_bfloat16* H, __nv_bfloat16* out,
                            cudaStream_t st);
// Router projection (gemm.cu): logits = x Wr^T with the top-k fused when E <= 256,
// and its backward (dx_r = dlogits Wr, dWr = dlogits^T x).
cudaError_t router_gemm(const moe_config& c, const Ws& ws, const __nv_bfloat16* x,
                        const __nv_bfloat16* Wr, float* logits, int* topk_ids, float* topk_w,
                        cudaStream_t st);
cudaError_t router_bwd(const moe_config& c, const Ws& ws, const __nv_bfloat16* dl16, int Epad,
                       const __nv_bfloat16* x, const __nv_bfloat16* Wr, __nv_bfloat16* dx_r,
                       __nv_bfloat16* dWr, cudaStream_t st);
cudaError_t gemm_fwd1_mx(const moe_config& c, const Ws& ws, const int* counts, const uint8_t* Xq,
                         const uint8_t* Xs, const uint8_t* W1q, const uint8_t* W1s, uint8_t* Aq,
                         uint8_t* As, __nv_bfloat16* A, __nv_bfloat16* H, cudaStream_t st);
cudaError_t gemm_fwd2_mx(const moe_config& c, const Ws& ws, const uint8_t* Aq, const uint8_t* As,
                         const uint8_t* W2q, const uint8_t* W2s, __nv_bfloat16* Yp,
                         cudaStream_t st);

}  // namespace moe
