/*
 * moe.h -- C ABI of the single-GPU mixture-of-experts layer for GB300 (sm_103a).
 *
 * One MoE layer: top-k routing, a schedule table (per-expert counts, prefix-sum
 * offsets, stable expert-contiguous permutation), a gather of token rows into
 * expert order, a grouped SwiGLU expert FFN on tcgen05 tensor cores, and a
 * fixed-order weighted merge back to token order; forward and backward.
 *
 * Sources (web pages on Cursor's "Mixture-of-Kittens" MoE megakernel):
 *   [LP] leiphone, "MoK：把 token 调度、跨 GPU 通信和专家计算塞进同一个 GPU 内核",
 *        sections 01 (communication tax), 02 (transfer while computing),
 *        03 (specialised execution)
 *   [MT] Marktechpost, "Cursor开源MoK：GB300 NVL72机架上的确定性MoE训练大内核",
 *        sections "three design decisions", "benchmarks", "key points"
 *
 * Conventions for every call:
 *  - Ownership: the caller owns every buffer.  The library never allocates
 *    device memory and never synchronises the stream (moe_read_status is the
 *    one exception).  Device pointers must be 128-byte aligned.
 *  - Layouts are row-major.  bf16 tensors are passed as moe_bf16 (raw bits).
 *    W1 is [E, d, 2f] with the gate in columns [0, f) and the up projection
 *    in [f, 2f); W2 is [E, f, d].
 *  - Errors: argument errors return at once without touching the GPU
 *    (MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE_TOO_SMALL).
 *    Launch failures return MOE_ERR_CUDA.  Conditions found on the device
 *    (a bounded wait that ran out) are written to a status word inside the
 *    workspace and read back with moe_read_status; nothing traps.
 *  - Determinism: for the same inputs, configuration and device every output
 *    is bitwise identical from run to run (the pages' megakernel is fully
 *    deterministic: [MT] three design decisions, last paragraph).  No
 *    floating-point atomics are used; every reduction has a fixed order.
 *  - Workspace: moe_schedule, moe_forward and moe_backward of one layer call
 *    must share the same workspace (it carries the padded expert layout from
 *    the schedule to the FFN) and the same moe_sched arrays.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */
typedef uint16_t moe_bf16;                /* bfloat16 bit pattern */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, bad size, misalignment, k > E ... */
  MOE_ERR_UNSUPPORTED = 2,         /* valid request this build does not implement */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < moe_workspace_bytes(cfg) */
  MOE_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5,             /* a bounded device wait ran out (status word) */
  MOE_ERR_DEVICE_CHECK = 6         /* a device-side bounds check failed (status word) */
} moe_status;

typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1 } moe_precision;

/* Layer configuration.
 *   T tokens, d hidden size, f expert intermediate size, E experts, k top-k.
 *   Limits: 1 <= k <= min(E, 32); 1 <= E <= 1024; T >= 1; d and f multiples
 *   of 64 (d also of 128 in MXFP8 mode).
 *   minibatch_rows: 0 runs the layer as a chain of kernels over the whole
 *     expert-ordered buffer.  > 0 runs the forward (BF16 or MXFP8) as one
 *     persistent cooperative kernel that hands windows of this many expert-ordered rows
 *     (rounded up to a multiple of 128) from gather warps or CTAs to GEMM
 *     warps through a ring of ring_slots slots, with GPU-side counters and
 *     the weighted merge at the end ([LP] 02: SM partition, local counters,
 *     minibatch, ring token buffer).  Results are bitwise identical to the chain path
 *     of the same precision for every window size (in MXFP8 mode the gather
 *     side quantises each window's rows into the ring slot).  The backward
 *     runs as a chain of kernels; after a BF16 ring forward it reuses the
 *     rows the ring still holds (see moe_backward).
 *   ring_slots: ring depth, 2..64, when minibatch_rows > 0.
 *   gather_ctas: how the work is split when minibatch_rows > 0.  0 (the
 *     default): every CTA runs the GEMM warps and one gather warp, so all
 *     SMs compute.  G > 0 (below the SM count): CTAs [0, G) only gather, with
 *     bulk copies staged through shared memory, and the other CTAs only
 *     compute. */
typedef struct {
  int32_t T, d, f, E, k;
  int32_t prec; /* moe_precision */
  int32_t minibatch_rows;
  int32_t ring_slots;
  int32_t gather_ctas;
} moe_config;

/* Schedule table, all device arrays written by moe_schedule ([LP] 01: count
 * tokens per expert, decide where each goes, keep an expert's tokens
 * contiguous; [MT] three design decisions: one table serves all four
 * transfer modes).  Flat routed row r = t*k + j, j = slot = rank.
 *   topk_ids [T*k] int32   expert of row r (ranked by logit, ties -> lower id)
 *   topk_w   [T*k] fp32    renormalised softmax weight of row r
 *   counts   [E]   int32   rows routed to each expert
 *   offsets  [E+1] int32   exclusive prefix sum of counts, offsets[E] = T*k
 *   perm     [T*k] int32   perm[p] = r: expert-major, ascending r within an expert
 *   inv      [T*k] int32   inverse of perm */
typedef struct {
  int32_t* topk_ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
} moe_sched;

/* Activations the forward saves for the backward, in the library's padded
 * expert order (each expert's rows start on a multiple of 128; padding rows
 * are zero).  H: [moe_saved_rows(cfg), 2f] bf16 (X W1 before SwiGLU);
 * A: [moe_saved_rows(cfg), f] bf16 (SwiGLU output).  Opaque to the caller. */
typedef struct {
  moe_bf16* H;
  moe_bf16* A;
} moe_saved;

/* Bytes of device workspace moe_schedule / moe_forward / moe_backward need
 * for cfg (pure host arithmetic; 0 if cfg is invalid). */
size_t moe_workspace_bytes(const moe_config* cfg);

/* Rows of the saved H / A buffers (pure host arithmetic; 0 if invalid). */
int64_t moe_saved_rows(const moe_config* cfg);

/* Smallest minibatch (rows) that gives the grouped GEMM at least two full
 * waves of tiles on compute_sms SMs: ceil(2 * compute_sms * bm * bn / n_cols)
 * with n_cols the GEMM's output width ([LP] 02 and [MT] three design
 * decisions: two full waves of tiles at least; for hidden 7168 / intermediate
 * 2048 the pages quote ~2,368 tokens).  Returns 0 on non-positive input. */
int32_t moe_min_minibatch(int32_t compute_sms, int32_t bm, int32_t bn, int32_t n_cols);

/* Routing + schedule table ([LP] 01; [MT] three design decisions).
 *   logits: device fp32 [T, E] (finite; non-finite logits give unspecified
 *   routing).  Writes every array of `sched` and the padded expert layout in
 *   `ws`; clears the workspace status word. */
moe_status moe_schedule(const moe_config* cfg, const float* logits, moe_sched sched,
                        void* ws, size_t ws_bytes, moe_stream_t stream);

/* Router projection + routing + schedule table: the logits are computed from
 * the token rows by the router ([LP] 01: the router decides every step which
 * experts each token goes to), then routed and scheduled exactly as
 * moe_schedule does.  Reading: a bias-free linear router,
 *   logits[t, e] = sum_i x[t, i] * w_router[e, i]
 * with bf16 products accumulated in fp32 on the tensor cores.
 *   x: device bf16 [T, d]; w_router: device bf16 [E, d] (row e = expert e).
 *   logits: device fp32 [T, E] output; may be NULL when E <= 256, where the
 *   top-k and its weights are taken in the GEMM's epilogue and the logits are
 *   never written (E > 256: required; the top-k runs on the stored logits).
 *   The routing decisions are those of moe_schedule on the same fp32 logits,
 *   bit for bit.  Writes every array of `sched` and the workspace as
 *   moe_schedule does. */
moe_status moe_route(const moe_config* cfg, const moe_bf16* x, const moe_bf16* w_router,
                     float* logits, moe_sched sched, void* ws, size_t ws_bytes,
                     moe_stream_t stream);

/* Backward of the router projection for an upstream gradient dlogits (as
 * moe_backward writes it):
 *   dx_router[t, i] = sum_e dlogits[t, e] * w_router[e, i]   (add it to dx)
 *   dw_router[e, i] = sum_t dlogits[t, e] * x[t, i]
 * dlogits: device fp32 [T, E], rounded to bf16 for the tensor cores;
 * dx_router: device bf16 [T, d] output; dw_router: device bf16 [E, d] output.
 * Uses the workspace (not the schedule in it). */
moe_status moe_router_backward(const moe_config* cfg, const moe_bf16* x, const moe_bf16* w_router,
                               const float* dlogits, moe_bf16* dx_router, moe_bf16* dw_router,
                               void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_schedule without a workspace.  The pages have no counterpart: this is a
 * convenience for callers that cannot allocate device memory -- for example a
 * plugin running inside a host framework that hands it only its input and
 * output tensors and forbids cudaMalloc after start-up (cudaMalloc may
 * synchronise the device and bypasses the framework's own allocator).
 * Computes the same `sched` arrays as moe_schedule, bit for bit, from the same
 * kernels, whose scratch (status and ticket words, per-block histograms,
 * padded offsets, row positions) is a 1.5 MiB array in the library's own
 * device data; every GPU that loads the library holds it until the process
 * exits.  No device memory is allocated and no allocating routine is called.
 * Limit: configurations whose schedule scratch exceeds 1.5 MiB return
 * MOE_ERR_INVALID_ARG; T <= 16384, E <= 256 and T*k <= 65536 always fit.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.  The
 * address is kept for as long as the device's CUDA context stays the same; a
 * call after a device reset (or in a new context) looks it up again, and that
 * call too should come before any stream capture.
 * All calls share the one array and leave their contents in it: calls that
 * overlap on the GPU (different streams, or different host threads, without
 * ordering between them) race and give undefined results.  The result does
 * not carry over to moe_forward / moe_backward, which need the workspace
 * written by moe_schedule. */
moe_status moe_schedule_noalloc(const moe_config* cfg, const float* logits, moe_sched sched,
                                moe_stream_t stream);

/* MXFP8 quantisation of weights for the MXFP8 forward ([LP] 02 MXFP8
 * paragraph; [MT] on the BF16 and MXFP8 modes).  w: device bf16 [batch, K, N]
 * (a W1 or W2 stack).  Writes q: e4m3 [batch, N, K] (K contiguous) and
 * scales: one UE8M0 byte per 32 consecutive K elements (batch*N*K/32 bytes;
 * scale 2^s with s the smallest exponent such that the block's max |v| <=
 * 448 * 2^s, clamped to [-127, 127]; elements rounded to nearest even with
 * saturation).  Scales are stored in 512-byte tiles, one per 128 rows
 * (rows = batch*N) x 128 K elements, tiles ordered row-block-major; within a
 * tile the scale of row r, 32-element block kb is at byte
 * 16*(r%32) + 4*((r%128)/32) + kb%4 (the order the tensor cores read them).
 * K and N must be multiples of 128. */
moe_status moe_quantize_mxfp8(const moe_bf16* w, int64_t batch, int32_t K, int32_t N,
                              uint8_t* q, uint8_t* scales, moe_stream_t stream);

/* MXFP8 quantisation along the contiguous dimension (the weights of the MXFP8
 * backward, whose GEMMs contract over the weights' other dimension): w [rows,
 * K] bf16 -> q [rows, K] E4M3 and one UE8M0 scale per 32 consecutive K
 * elements, with the scale rule, rounding and 512-byte tile layout of
 * moe_quantize_mxfp8 (row r, block kb at byte 16*(r%32) + 4*((r%128)/32) +
 * kb%4 of tile (r/128, kb/4)).  rows and K multiples of 128.  W1 [E, d, 2f]
 * for the MXFP8 backward: rows = E*d, K = 2f; W2 [E, f, d]: rows = E*f,
 * K = d. */
moe_status moe_quantize_mxfp8_rows(const moe_bf16* w, int64_t rows, int32_t K, uint8_t* q,
                                   uint8_t* scales, moe_stream_t stream);

/* Forward: Dispatch -> Expert FFN -> Combine -> weighted merge ([LP] 03;
 * dispatch by pull, combine by push, [LP] 02).
 *   x [T, d] bf16.  BF16 mode: w1 = W1 bf16 [E, d, 2f], w2 = W2 bf16 [E, f, d],
 *   w1_scales = w2_scales = NULL.  MXFP8 mode: w1/w2 and their scales as
 *   written by moe_quantize_mxfp8 from W1 / W2.
 *   out [T, d] bf16: out[t] = sum_j topk_w[t,j] * FFN_{topk_ids[t,j]}(x[t]),
 *   summed in slot order in fp32, rounded once to bf16.
 *   saved: NULL for inference; else H and A are written for moe_backward. */
moe_status moe_forward(const moe_config* cfg, const moe_bf16* x, const void* w1,
                       const uint8_t* w1_scales, const void* w2, const uint8_t* w2_scales,
                       moe_sched sched, moe_bf16* out, const moe_saved* saved, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/* Backward (BF16): reverse combine, expert FFN dgrad / wgrad, SwiGLU backward
 * fused with the routing-weight gradient, reverse dispatch ([LP] 02: pull
 * reverse-combine, push reverse-dispatch; [MT] three design decisions: the
 * routing-weight gradient is fused into the SwiGLU backward, and the ring
 * buffer is traversed in reverse to replay as few forward activations as
 * possible).
 *   dout [T, d] bf16 upstream gradient; x, w1, w2 as in the forward; saved
 *   as written by moe_forward with the same sched and ws, or NULL: then H and
 *   A are recomputed from the re-gathered rows by the forward's GEMM1 (the
 *   same bits as the saved ones) in workspace buffers.
 *   The token rows are re-gathered into expert order walking the rows from
 *   the last to the first; after a ring forward (minibatch_rows > 0, same
 *   ws) the rows of its last ring_slots windows, still held in the ring, are
 *   taken from there instead of from x.
 *   dx [T, d] bf16; dw1 [E, d, 2f] bf16; dw2 [E, f, d] bf16 (experts with no
 *   rows get exact zeros); dtopk_w [T*k] fp32 = d loss / d topk_w;
 *   dlogits [T, E] fp32 or NULL: gradient through the renormalised softmax
 *   (zero for unselected experts).
 *   An MXFP8 configuration returns MOE_ERR_UNSUPPORTED: its backward is
 *   moe_backward_mxfp8. */
moe_status moe_backward(const moe_config* cfg, const moe_bf16* dout, const moe_bf16* x,
                        const moe_bf16* w1, const moe_bf16* w2, moe_sched sched,
                        const moe_saved* saved, moe_bf16* dx, moe_bf16* dw1, moe_bf16* dw2,
                        float* dtopk_w, float* dlogits, void* ws, size_t ws_bytes,
                        moe_stream_t stream);

/* Where an intermediate buffer of the layer lies inside the workspace, for
 * tests and debugging (the pages describe no such call).  Pure host
 * arithmetic: writes the byte offset from the workspace start and the size
 * in bytes, or returns MOE_ERR_INVALID_ARG for an invalid cfg, an unknown
 * region, a null pointer, or a region the configuration does not have.
 *   MOE_WS_XQ_CODES   MXFP8: E4M3 codes of the gathered token rows,
 *                     [moe_saved_rows(cfg), d] in the padded expert order
 *                     (moe_forward writes the routed rows; padding rows
 *                     are not written, and GEMM1 zeroes what it computes
 *                     from them)
 *   MOE_WS_XQ_SCALES  their UE8M0 scales in 512-byte tiles (the layout
 *                     moe_quantize_mxfp8 documents, K = d)
 *   MOE_WS_AQ_CODES   MXFP8: E4M3 codes of the SwiGLU output A that GEMM1's
 *                     epilogue quantises for GEMM2, [moe_saved_rows(cfg), f]
 *   MOE_WS_AQ_SCALES  their scales in 512-byte tiles (K = f)
 * The operands moe_backward_mxfp8 quantises, each a codes region followed by
 * its scales region (tiles as above; Rp = moe_saved_rows(cfg)):
 *   MOE_WS_DYQ_*      dOut rows in expert order, blocks along d: [Rp, d]
 *   MOE_WS_XQT_*      x rows in expert order, transposed, blocks of 32 rows
 *                     from each expert's segment start: [d, Rp]
 *   MOE_WS_DYQT_*     dOut rows the same way: [d, Rp]
 *   MOE_WS_DHQ_*      dH, blocks along 2f: [Rp, 2f]
 *   MOE_WS_DHQT_*     dH transposed, blocks of 32 rows: [2f, Rp]
 *   MOE_WS_GAQT_*     g*A transposed, blocks of 32 rows: [f, Rp] */
typedef enum {
  MOE_WS_XQ_CODES = 0,
  MOE_WS_XQ_SCALES = 1,
  MOE_WS_AQ_CODES = 2,
  MOE_WS_AQ_SCALES = 3,
  MOE_WS_DYQ_CODES = 4,
  MOE_WS_DYQ_SCALES = 5,
  MOE_WS_XQT_CODES = 6,
  MOE_WS_XQT_SCALES = 7,
  MOE_WS_DYQT_CODES = 8,
  MOE_WS_DYQT_SCALES = 9,
  MOE_WS_DHQ_CODES = 10,
  MOE_WS_DHQ_SCALES = 11,
  MOE_WS_DHQT_CODES = 12,
  MOE_WS_DHQT_SCALES = 13,
  MOE_WS_GAQT_CODES = 14,
  MOE_WS_GAQT_SCALES = 15
} moe_ws_region;
moe_status moe_workspace_region(const moe_config* cfg, int32_t region, size_t* offset,
                                size_t* bytes);

/* Backward in MXFP8 ([MT] three design decisions: BF16 and MXFP8 precision
 * modes; [LP] 03: the MXFP8 backward is among the layer's measured passes).
 * The pages do not say how the backward quantises; reading: every backward
 * GEMM quantises both operands along its own contraction dimension, with the
 * forward's block format --
 *   dgrad2 (K = d):   dOut rows and W2 along d
 *   dgrad1 (K = 2f):  dH and W1 along 2f
 *   wgrad2 (K = the expert's rows): g*A and dOut along the rows
 *   wgrad1 (K = the expert's rows): x rows and dH along the rows
 * the row blocks of 32 counted from the start of each expert's rows (the
 * padded expert order; the last block holds zero rows).  The SwiGLU backward
 * and the routing-weight gradient run in fp32 in dgrad2's epilogue, which
 * also quantises dH (both ways) and g*A.
 *   cfg->prec must be MOE_MXFP8.  dout, x: as moe_backward.  w1q / w1s: W1
 *   quantised by moe_quantize_mxfp8_rows(W1, E*d, 2f); w2q / w2s: W2 by
 *   moe_quantize_mxfp8_rows(W2, E*f, d).  saved: required, written by the
 *   MXFP8 moe_forward (H and A in bf16) with the same sched and ws.
 *   Outputs as moe_backward (dx, dw1, dw2 bf16; dtopk_w, dlogits fp32). */
moe_status moe_backward_mxfp8(const moe_config* cfg, const moe_bf16* dout, const moe_bf16* x,
                              const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q,
                              const uint8_t* w2s, moe_sched sched, const moe_saved* saved, moe_bf16* dx,
                              moe_bf16* dw1, moe_bf16* dw2, float* dtopk_w, float* dlogits, void* ws,
                              size_t ws_bytes, moe_stream_t stream);

/* Synchronises `stream` and returns the device status word of `ws` (MOE_OK,
 * MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK).  Test / debug use. */
moe_status moe_read_status(const void* ws, moe_stream_t stream);

/* Static English name of a status code. */
const char* moe_status_string(moe_status s);

/* How the one-CTA weight-gradient GEMMs (moe_backward, moe_backward_mxfp8)
 * hand out their work units ([MT] three design decisions, last paragraph:
 * the megakernel schedules its tiles with Blackwell's Cluster Launch
 * Control).  0: a static walk -- a persistent grid of one CTA per SM, CTA i
 * taking units i, i + grid, ...  1: cluster launch control -- a grid of one
 * CTA per unit; each running CTA, while it works on a unit, has the hardware
 * cancel the launch of a CTA that has not started yet and takes over that
 * CTA's unit, so the units go to whichever SM frees up first.  Both give
 * bitwise identical results (the same tiles, each computed whole by one
 * CTA).  Process-wide, not thread-safe; takes effect for later calls.
 * Returns MOE_ERR_INVALID_ARG for another mode. */
moe_status moe_set_tile_scheduler(int32_t mode);
int32_t moe_get_tile_scheduler(void);

/* Tracing (profiling aid; the pages describe none).  moe_trace_enable(n)
 * creates 2n CUDA events on the current device; from then on every kernel the
 * library launches records one event before and one after its launch, on the
 * call's stream, until n launches have been recorded.  moe_trace_enable(0)
 * turns tracing off and frees the events.  moe_trace_count returns the number
 * of launches recorded; moe_trace_read(i, ...) waits for launch i's second
 * event and returns the kernel's static name and its duration in ms.  Tracing
 * state is process-wide and not thread-safe. */
moe_status moe_trace_enable(int32_t capacity);
int32_t moe_trace_count(void);
moe_status moe_trace_read(int32_t i, const char** name, float* ms);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
