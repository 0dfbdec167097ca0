// ring.cu -- the forward pass as one persistent kernel.
//
// The pages' megakernel splits the GPU's SMs into a side that moves tokens
// (dispatch, combine, state) and a side that runs the expert FFN; the moving
// side tells the compute side through GPU-local counters when a full
// minibatch has arrived, the compute side signals back when it is done, and
// a fixed-size ring token buffer is recycled minibatch by minibatch, with no
// CPU in the loop (leiphone "MoK..." section 02; Marktechpost "Cursor开源MoK..."
// three design decisions).  On one GPU the moving side is an HBM gather.
//
// Layout of one launch (cooperative, so every CTA is co-resident), for
// windows w of `mb` consecutive rows of the padded expert order held in ring
// slot w % S:
//   gather         either (G = 0, the default) the last kGatherWarps warps of
//                  every CTA, each copying its share of a window with plain
//                  loads and stores, or (G > 0) CTAs [0, G), whose warps stage
//                  rows through shared memory with bulk copies; each waits
//                  until the slot is free (freed), copies the window's token
//                  rows in and releases ready[slot].
//   compute        the warp-specialised tcgen05 pipeline of gemm.cu (TMA
//                  producer, MMA issuer, four epilogue warps) in every CTA that
//                  is not a gather CTA, over the unit stream G1(0) ... G1(lag-1),
//                  [G1(lag), G2(0)], ..., G2(last); each CTA claims the next
//                  unit from a global counter when its producer is ready for
//                  one, so units of mixed cost balance themselves.  A unit is
//                  one N tile of two M-adjacent 128-row tiles of a window (BF16;
//                  one tile in MXFP8): when both belong to one expert and
//                  neither is thin, each stage holds both A tiles and the
//                  shared B tile and the MMAs feed two accumulators, so B
//                  crosses the SM's L2 ingress once for 256 rows; otherwise
//                  the tiles run one after the other.  GEMM1 + SwiGLU tiles of
//                  window w read the ring slot after acquiring ready[slot] and
//                  release freed[slot] once their loads have landed; GEMM2
//                  tiles of a 128-row tile wait for that tile's GEMM1
//                  epilogues (a_ready) and store Y in expert order.
//   all CTAs       after the last GEMM2 store (done2), the fixed-order
//                  weighted merge of every token.
// MXFP8 mode: the gather quantises each row into E4M3 codes and UE8M0 scale
// tiles in the ring slot (one scale per 32 elements along d), GEMM1 and GEMM2
// are block-scaled (tcgen05.mma kind::mxf8f6f4, scales staged into TMEM),
// GEMM1's epilogue quantises A along f for GEMM2 -- the same tiles in the
// same order as the kernel chain's MXFP8 GEMMs, so the results are the
// chain's bit for bit.
// Every tile waits only on tiles and windows earlier in the stream, so the
// stream always makes progress.  Every wait is bounded: on expiry the kernel
// sets a global abort word, reports MOE_ERR_TIMEOUT in the workspace status
// word and every CTA winds down (no trap).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "mx.cuh"
#include "ptx.cuh"
#include "bulk_rows.cuh"
#include "rowops.cuh"

namespace moe {

namespace {

constexpr int BK = 64;
constexpr int BK8 = 128;                       // MXFP8: K elements (bytes) per stage
constexpr int kABytes = kBM * BK * 2;          // 16 KB (MXFP8: 128 rows x 128 bytes, the same)
constexpr int kBBox = 64 * BK * 2;             // 8 KB: 64 columns x 64 K rows, MN-major
constexpr int kSfBytes = 1536;                 // MXFP8: A scale tile + two B scale tiles a stage
constexpr int kEpiWarps = 4;
constexpr int kGatherWarps = 2;  // gather warps of a CTA in the warp split
constexpr int kThreads = (2 + kEpiWarps + kGatherWarps) * 32;  // producer, MMA, epilogue, gather
constexpr int kOutTile = 32 * 128;
constexpr int kTmemCols = 512;
constexpr int kTmemSf = 256;                   // MXFP8: scale columns of stage s at 256 + 16 s
constexpr int kQ = 4;  // depth of the per-CTA queue of claimed tile indices
// The stage region holds four stages of one A tile and B (48 KB each) or,
// for units of two tiles (bf16, see the unit stream), three stages of two A
// tiles and B (64 KB each).  bf16: staging tiles for the Y stores (and the
// thin tiles' transposes) after it; MXFP8 (units of one tile): per-stage
// scale tiles instead (Y leaves with direct stores).
constexpr int kMaxStages = 4;
constexpr int kStageRegion = 4 * (kABytes + 4 * kBBox);
static_assert(kStageRegion == 3 * (2 * kABytes + 4 * kBBox), "both stage layouts fill the region");
template <bool FP8>
struct RingCfg {
  static constexpr size_t kExtra = FP8 ? (size_t)kMaxStages * kSfBytes : (size_t)kEpiWarps * 2 * kOutTile;
  static constexpr size_t kSmem = 1024 + (size_t)kStageRegion + (kExtra + 1023) / 1024 * 1024 + 256;
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct RingParams {
  int T, d, f, E, k;
  int G, S, mb, mtw;          // gather CTAs (0: a gather warp in every CTA), ring slots, rows per
                              // window, 128-row tiles per window
  int nrel;                   // arrivals that complete one window (gather CTAs or gather warps)
  int gw, nbw;                // gather warps per CTA issuing bulk copies, row buffers per such warp
  int lag;                    // windows between a window's GEMM1 and GEMM2 tiles in the stream
  int tpu;                    // 128-row tiles per unit (bf16: 1 or 2; selects the kernel)
  int hn, nt1, nt2, kb1, kb2;  // GEMM1 half width, N tiles of GEMM1 / GEMM2, K blocks
  const int* mt_off;
  const int* counts;   // rows per expert: a partial last tile runs thin (swapped)
  int thin;
  int thin_rows;        // largest partial tile that runs thin
  int thin2;            // GEMM2 tiles of at most 32 rows run thin (bf16)
  const int* hdr;
  const int* row_of_pad;
  const int* pos_pad;
  const float* topk_w;
  const __nv_bfloat16* x;
  __nv_bfloat16* ring;  // [S * mb, d]  (MXFP8: E4M3 codes [S * mb, d], then their scale tiles)
  uint8_t* ring_sf;     // MXFP8: scale tiles of the ring rows
  uint8_t* Aq;          // MXFP8: E4M3 codes of A [Rp, f] and their scale tiles
  uint8_t* As;
  const uint8_t* W1s;   // MXFP8: scale tiles of the quantised weights
  const uint8_t* W2s;
  __nv_bfloat16* A;     // [Rp, f]
  __nv_bfloat16* H;     // [Rp, 2f] or null
  __nv_bfloat16* Y;     // [Rp, d]
  __nv_bfloat16* out;   // [T, d]
  int* ready;           // [S]  gather arrivals per slot
  int* freed;           // [S]  GEMM1 tiles done reading per slot
  int* a_ready;         // [MT] GEMM1 epilogue warps done per 128-row tile
  int* done2;           // GEMM2 epilogue warps done
  int* tile_next;       // next unclaimed tile of the stream
  int* gabort;          // set once by the first wait that gives up
  int* status;
  int* ring_valid;      // header word: set once every window has passed through the ring
};

// Window geometry of this call (from the padded row total the schedule wrote).
// The stream is counted in units of up to tpu 128-row tiles (the tiles of a
// window are grouped along M: tiles 2u and 2u + 1 form unit u when tpu = 2).
struct Geo {
  int rp, nW, mt_last;
  int F1;          // GEMM1 tiles of a full window (the ring slot's readers)
  int um, uml;     // units along M of a full window / of the last window
  int U1, U2;      // GEMM1 / GEMM2 units of a full window
  int total;       // units in the stream
  int total2;      // GEMM2 tiles in the stream
};

__device__ __forceinline__ Geo make_geo(const RingParams& p, int tpu) {
  Geo g;
  g.rp = p.hdr[kHdrRpTotal];
  g.nW = (g.rp + p.mb - 1) / p.mb;
  g.mt_last = (g.rp - (g.nW - 1) * p.mb) / kBM;
  g.F1 = p.mtw * p.nt1;
  g.um = (p.mtw + tpu - 1) / tpu;
  g.uml = (g.mt_last + tpu - 1) / tpu;
  g.U1 = g.um * p.nt1;
  g.U2 = g.um * p.nt2;
  g.total = (g.nW - 1) * (g.U1 + g.U2) + g.uml * (p.nt1 + p.nt2);
  g.total2 = (g.nW - 1) * p.mtw * p.nt2 + g.mt_last * p.nt2;
  return g;
}

struct RTile {
  int phase, w, mloc, mt, n, e;
  int rows;   // valid rows of the 128-row tile
  bool thin;  // computed as (weights)^T x (rows)^T with the tokens on N
};

// A unit of the stream: one or two tiles of one window, phase and N tile.
// pair: two tiles of the same expert, neither thin -- their MMAs share each
// stage's B operand, one accumulator each; otherwise the tiles run one after
// the other.
struct RUnit {
  RTile t[2];
  int nt;     // tiles in the unit (1 or 2)
  bool pair;
};

// A 32-token x 32-column block held one column per lane is written to rows
// [0, nrows) at dst through a shared transpose tile (see gemm.cu).
__device__ __forceinline__ void ring_store_cols_t(uint8_t* tr, const float* v, __nv_bfloat16* dst,
                                                  size_t ld, int nrows, int lane) {
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 32; ++i)
    *reinterpret_cast<__nv_bfloat16*>(tr + i * 80 + lane * 2) = __float2bfloat16_rn(v[i]);
  __syncwarp();
  if (lane < nrows) {
    const uint4* s = reinterpret_cast<const uint4*>(tr + lane * 80);
    uint4* d = reinterpret_cast<uint4*>(dst + (size_t)lane * ld);
    d[0] = s[0];
    d[1] = s[1];
    d[2] = s[2];
    d[3] = s[3];
  }
}

// Unit L of the stream G1(0), ..., G1(lag - 1), [G1(lag) G2(0)], [G1(lag + 1)
// G2(1)], ..., [G1(nW - 1) G2(nW - 1 - lag)], G2(nW - lag), ..., G2(nW - 1):
// GEMM2 of a window is claimed `lag` windows after its GEMM1, by when its
// GEMM1 tiles are mostly done.  Inside a phase block, units run
// N-tile-major so that the units sharing an expert's weight slice are
// adjacent.  Only the last window can be short (mt_last tiles).
__device__ __forceinline__ RUnit ring_decode(const RingParams& p, const Geo& g, int L, int tpu) {
  int phase, w, loc;
  const int u1l = g.uml * p.nt1;
  const int lag = min(p.lag, g.nW);
  if (lag == g.nW) {
    // every GEMM1 unit, then every GEMM2 unit
    const int n1 = (g.nW - 1) * g.U1 + u1l;
    phase = L < n1 ? 1 : 2;
    const int l = L < n1 ? L : L - n1;
    const int F = phase == 1 ? g.U1 : g.U2;
    w = min(l / F, g.nW - 1);
    loc = l - w * F;
  } else if (L < lag * g.U1) {
    phase = 1; w = L / g.U1; loc = L % g.U1;
  } else {
    int l = L - lag * g.U1;
    const int blk = g.U1 + g.U2;
    const int nfull = g.nW - 1 - lag;  // blocks [G1(b) G2(b - lag)] of full windows
    if (l < nfull * blk) {
      const int b = lag + l / blk, r = l % blk;
      if (r < g.U1) { phase = 1; w = b; loc = r; }
      else { phase = 2; w = b - lag; loc = r - g.U1; }
    } else {
      l -= nfull * blk;
      if (l < u1l) { phase = 1; w = g.nW - 1; loc = l; }
      else if ((l -= u1l) < g.U2) { phase = 2; w = g.nW - 1 - lag; loc = l; }
      else {
        l -= g.U2;
        phase = 2;
        w = min(g.nW - lag + l / g.U2, g.nW - 1);
        loc = l - (w - (g.nW - lag)) * g.U2;
      }
    }
  }
  const bool last = (w == g.nW - 1);
  const int umw = last ? g.uml : g.um;
  const int mtw = last ? g.mt_last : p.mtw;
  const int mu = loc % umw, n = loc / umw;
  auto tile = [&](int mloc) {
    RTile t;
    t.phase = phase;
    t.w = w;
    t.mloc = mloc;
    t.n = n;
    t.mt = w * p.mtw + mloc;
    t.e = find_expert(p.mt_off, p.E, t.mt);
    t.rows = kBM;
    t.thin = false;
    if ((p.thin && phase == 1) || (p.thin2 && phase == 2)) {
      const int cnt = __ldg(p.counts + t.e);
      const int rows = cnt - (t.mt - __ldg(p.mt_off + t.e)) * kBM;
      if (thin_tile(rows, cnt) && rows <= (phase == 1 ? p.thin_rows : 32)) {
        t.rows = rows;
        t.thin = true;
      }
    }
    return t;
  };
  RUnit u;
  u.t[0] = tile(mu * tpu);
  u.nt = (tpu == 2 && mu * 2 + 1 < mtw) ? 2 : 1;
  if (u.nt == 2) u.t[1] = tile(mu * 2 + 1);
  else u.t[1] = u.t[0];
  u.pair = u.nt == 2 && u.t[0].e == u.t[1].e && !u.t[0].thin && !u.t[1].thin;
  return u;
}

// MXFP8: one warp quantises the source row of routed row r (zeros for a
// padding row, r < 0) into ring row rr -- E4M3 codes and one UE8M0 scale per
// 32 elements along d, lane b taking blocks b, b + 32, ... -- with the
// quantiser of the chain's gather (the same codes, bit for bit).
__device__ __forceinline__ void ring_quant_row(const RingParams& p, int r, size_t rr, int lane) {
  const int nblk = p.d >> 5;
  const uint4* sv = reinterpret_cast<const uint4*>(p.x + (size_t)(r < 0 ? 0 : r / p.k) * p.d);
  uint8_t* q = reinterpret_cast<uint8_t*>(p.ring) + rr * p.d;
  for (int b = lane; b < nblk; b += 32) {
    float v[32];
#pragma unroll
    for (int u = 0; u < 4; ++u) unpack8(r >= 0 ? ldg_nc_v4(sv + b * 4 + u) : make_uint4(0, 0, 0, 0), v + 8 * u);
    uint4 lo, hi;
    const uint8_t sc = mx_quant32(v, lo, hi);
    stg_v4(q + b * 32, lo);
    stg_v4(q + b * 32 + 16, hi);
    p.ring_sf[mx_sf_offset(rr, b, p.d >> 7)] = sc;
  }
}

template <bool FP8, int TPU>
__global__ void __launch_bounds__(kThreads, 1)
    ring_forward_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW1,
                        const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW2,
                        const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmX16,
                        const __grid_constant__ CUtensorMap tmA16, const __grid_constant__ CUtensorMap tmAo,
                        const __grid_constant__ CUtensorMap tmHo, const RingParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_ok;
  __shared__ int s_gab;
  __shared__ int s_pos[kMaxK];
  __shared__ float s_w[kMaxK];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kAcc = FP8 ? 1 : 2;  // MXFP8: one accumulator, the scales in TMEM columns 256..
  // tiles per unit (the host's choice, 1 in MXFP8) and the stage layout it implies
  static_assert(TPU == 1 || (TPU == 2 && !FP8), "two-tile units are bf16 only");
  constexpr int kTpu = TPU;
  constexpr int kStages = kTpu == 2 ? 3 : 4;
  constexpr int kStageBytes = kTpu * kABytes + 4 * kBBox;
  const Geo geo = make_geo(p, kTpu);
  const int inject = p.hdr[kHdrInject];        // test hook: window + 1 whose arrival is withheld
  const int lim_ms = p.hdr[kHdrInject + 1];    // test hook: wait limit in ms (0: default)
  const uint64_t limit = lim_ms > 0 ? (uint64_t)lim_ms * 1000000ull : kWaitLimitNs;

  if (blockIdx.x < (unsigned)p.G) {
    // ====================================================== gather side
    // Warps [0, gw) each move their share of a window's rows with bulk copies
    // staged through nbw row buffers of their own (bulk_rows.cuh); padding
    // rows of the expert order leave from a zero row.
    // (MXFP8: warps quantise rows from registers; no row buffers)
    const uint32_t rb = (uint32_t)p.d * 2u;
    const bool issuer = warp < p.gw;
    RowPipe rp;
    rp.zrow = smem_u32(smem);
    rp.rb = rb;
    rp.wbuf = rp.zrow + rb + (uint32_t)(warp * p.nbw) * rb;
    rp.bars = reinterpret_cast<uint64_t*>(smem + (size_t)(1 + p.gw * p.nbw) * rb) + warp * p.nbw;
    rp.nbw = p.nbw;
    rp.depth = p.nbw / 2;
    rp.ph = rp.pend = 0;
    rp.hints = 0;  // the ring's rows are read by the GEMM warps right away: normal priority
    rp.ld_pol = rp.st_pol = 0;
    if constexpr (!FP8) {
      for (uint32_t i = threadIdx.x; i < rb / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();  // the zero row is read by bulk stores
      if (issuer && lane == 0) {
        for (int b = 0; b < p.nbw; ++b) mbar_init(&rp.bars[b], 1);
        fence_mbar_init();
      }
    }
    if (threadIdx.x == 0) s_gab = 0;
    __syncthreads();
    const int gid = blockIdx.x * p.gw + warp, ni = p.G * p.gw;
    for (int w = 0; w < geo.nW; ++w) {
      const int s = w % p.S, gen = w / p.S;
      if (threadIdx.x == 0)
        s_ok = (gen == 0) || wait_counter(&p.freed[s], gen * geo.F1, p.gabort, p.status, 500 + s, limit);
      __syncthreads();
      const bool ok = s_ok;
      __syncthreads();  // everyone has read s_ok before thread 0 writes it again
      if (!ok) break;
      const int r0 = w * p.mb, r1 = min(r0 + p.mb, geo.rp);
      if constexpr (FP8) {
        // every warp of the CTA quantises its share of the window's rows
        const int gq = blockIdx.x * (kThreads / 32) + warp, nq = p.G * (kThreads / 32);
        for (int pp = r0 + gq; pp < r1; pp += nq)
          ring_quant_row(p, __ldg(p.row_of_pad + pp), (size_t)s * p.mb + (pp - r0), lane);
        __syncthreads();
        if (threadIdx.x == 0) {
          __threadfence();
          if (inject != w + 1) red_release_add(&p.ready[s], 1);
        }
        continue;
      }
      const int n = (issuer && r0 + gid < r1) ? (r1 - r0 - gid + ni - 1) / ni : 0;
      if (n > 0) {
        __nv_bfloat16* slot = p.ring + (size_t)s * p.mb * p.d;
        const int* rop = p.row_of_pad + r0 + gid;
        if (lane == 0) fence_proxy_async_global();  // the slot's earlier readers are done (freed acquired above)
        const bool done = bulk_rows(
            rp, n,
            [&](int i) {
              const int r = __ldg(rop + (size_t)i * ni);
              return r >= 0 ? r : kRowZero;
            },
            [&](int r) { return p.x + (size_t)(r / p.k) * p.d; },
            [&](int i) { return slot + (size_t)(gid + i * ni) * p.d; }, &s_gab, p.status, 550);
        if (lane == 0) {
          bulk_wait<0>();  // this warp's rows are in global memory
          fence_proxy_async_global();
          if (!done || s_gab) {
            atomicExch(p.gabort, 1);
            for (int b = 0; b < p.nbw; ++b)  // no copy may still target shared memory at exit
              if ((rp.pend >> b) & 1u) mbar_wait_drain(&rp.bars[b], (rp.ph >> b) & 1u);
          }
        }
        __syncwarp();
      }
      __syncthreads();
      if (s_gab) break;
      if (threadIdx.x == 0) {
        __threadfence();
        if (inject != w + 1) red_release_add(&p.ready[s], 1);
      }
    }
  } else {
    // ====================================================== compute side
    uint8_t* stages = smem;
    uint8_t* staging = smem + (size_t)kStageRegion;  // MXFP8: the stages' scale tiles
    uint8_t* sfbuf = staging;
    uint8_t* ctrl = staging + (RingCfg<FP8>::kExtra + 1023) / 1024 * 1024;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* qfull = drain + 1;     // tile queue: claimed tile index published
    uint64_t* qempty = qfull + kQ;   // tile queue: slot read by the MMA and epilogue warps
    int* qtile = reinterpret_cast<int*>(qempty + kQ);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qtile + kQ);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    if (threadIdx.x == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(&tfull[a], 1);
        mbar_init(&tempty[a], kEpiWarps * 32);
      }
      mbar_init(drain, 1);
      for (int i = 0; i < kQ; ++i) {
        mbar_init(&qfull[i], 1);
        mbar_init(&qempty[i], 1 + kEpiWarps);
      }
      *abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmW1);
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmW2);
      tma_prefetch_desc(&tmY);
      tma_prefetch_desc(&tmX16);
      tma_prefetch_desc(&tmA16);
    }
    if (warp == 1) {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------ TMA producer
        int s = 0;
        uint32_t ph = 0, used = 0, last_par = 0;
        for (int j = 0;; ++j) {
          // claim the next tile of the stream and hand its index to the other roles
          if (!mbar_wait(&qempty[j % kQ], ((j / kQ) & 1) ^ 1, abort_flag, p.status, 150)) goto producer_done;
          const int L = atomicAdd(p.tile_next, 1);
          qtile[j % kQ] = L;
          mbar_arrive(&qfull[j % kQ]);
          if (L >= geo.total) break;
          const RUnit u = ring_decode(p, geo, L, kTpu);
          const bool g1 = (u.t[0].phase == 1);
          const int slot = u.t[0].w % p.S;
          bool ok;
          if (g1)
            ok = wait_counter(&p.ready[slot], p.nrel * (u.t[0].w / p.S + 1), p.gabort, p.status, 600 + slot, limit);
          else
            ok = wait_counter(&p.a_ready[u.t[0].mt], kEpiWarps * p.nt1, p.gabort, p.status, 700, limit) &&
                 (u.nt < 2 || wait_counter(&p.a_ready[u.t[1].mt], kEpiWarps * p.nt1, p.gabort, p.status, 700, limit));
          if (!ok) {
            *abort_flag = 1;
            goto producer_done;
          }
          fence_proxy_async_global();  // rows written by other CTAs, read by TMA below
          const int nbox = g1 ? (2 * p.hn) / 64 : 4;
          const int nkb = g1 ? p.kb1 : p.kb2;
          // a pair unit: both A tiles and the shared B in one stage; otherwise
          // the unit's tiles one after the other, A then B in each stage
          const int passes = u.pair ? 1 : u.nt;
          for (int ti = 0; ti < passes; ++ti) {
          const RTile t = ti == 0 ? u.t[0] : u.t[1];
          const int na = u.pair ? 2 : 1;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, 100 + s)) goto producer_done;
            const uint32_t sa = smem_u32(stages + (size_t)s * kStageBytes);
            const uint32_t sb = sa + (uint32_t)na * kABytes;
            const uint32_t fb = smem_u32(&full[s]);
            if constexpr (FP8) {
              // K-major E4M3 tiles (128 bytes of K per row) and their scale
              // tiles, as the chain's MXFP8 GEMMs load them
              mbar_arrive_expect_tx(&full[s], (uint32_t)(kABytes + 32768 + kSfBytes));
              const uint32_t sf = smem_u32(sfbuf + (size_t)s * kSfBytes);
              if (g1) {
                const int ring_row = slot * p.mb + t.mloc * kBM;
                const int kg = p.d >> 7, nbt = (2 * p.f) >> 7;
                tma_load_2d(sa, &tmX, fb, kb * BK8, ring_row);
                tma_load_3d(sb, &tmW1, fb, kb * BK8, t.n * 128, t.e);
                tma_load_3d(sb + 16384, &tmW1, fb, kb * BK8, p.f + t.n * 128, t.e);
                bulk_load(sf, p.ring_sf + ((size_t)(ring_row >> 7) * kg + kb) * 512u, 512u, fb);
                bulk_load(sf + 512, p.W1s + (((size_t)t.e * nbt + t.n) * kg + kb) * 512u, 512u, fb);
                bulk_load(sf + 1024, p.W1s + (((size_t)t.e * nbt + (p.f >> 7) + t.n) * kg + kb) * 512u, 512u, fb);
              } else {
                const int kg = p.f >> 7, nbt = p.d >> 7;
                const int nb1 = min(2 * t.n + 1, nbt - 1);  // rows past d are zero-filled; any finite scale
                tma_load_2d(sa, &tmA, fb, kb * BK8, t.mt * kBM);
                tma_load_3d(sb, &tmW2, fb, kb * BK8, t.n * 256, t.e);
                bulk_load(sf, p.As + ((size_t)t.mt * kg + kb) * 512u, 512u, fb);
                bulk_load(sf + 512, p.W2s + (((size_t)t.e * nbt + 2 * t.n) * kg + kb) * 512u, 512u, fb);
                bulk_load(sf + 1024, p.W2s + (((size_t)t.e * nbt + nb1) * kg + kb) * 512u, 512u, fb);
              }
            } else {
            if (t.thin && (!g1 || p.thin_rows <= 32)) {
              // a thin tile of at most 32 rows (GEMM2; GEMM1 at large hidden
              // sizes) reads only the 16-row boxes that hold its rows
              const int nr16 = (t.rows + 15) >> 4;
              mbar_arrive_expect_tx(&full[s], (uint32_t)nr16 * 2048u + (uint32_t)nbox * kBBox);
              for (int i = 0; i < nr16; ++i) {
                if (g1) tma_load_2d(sa + i * 2048, &tmX16, fb, kb * BK, slot * p.mb + t.mloc * kBM + 16 * i);
                else tma_load_2d(sa + i * 2048, &tmA16, fb, kb * BK, t.mt * kBM + 16 * i);
              }
            } else {
              mbar_arrive_expect_tx(&full[s], (uint32_t)(na * kABytes) + (uint32_t)nbox * kBBox);
              for (int i = 0; i < na; ++i) {
                const RTile ta = (ti + i) == 0 ? u.t[0] : u.t[1];
                if (g1) tma_load_2d(sa + i * kABytes, &tmX, fb, kb * BK, slot * p.mb + ta.mloc * kBM);
                else tma_load_2d(sa + i * kABytes, &tmA, fb, kb * BK, ta.mt * kBM);
              }
            }
            if (g1) {
              const int half = nbox / 2;
              for (int i = 0; i < nbox; ++i) {
                const int col = (i < half) ? t.n * p.hn + 64 * i : p.f + t.n * p.hn + 64 * (i - half);
                tma_load_3d(sb + i * kBBox, &tmW1, fb, col, kb * BK, t.e);
              }
            } else {
              for (int i = 0; i < 4; ++i) tma_load_3d(sb + i * kBBox, &tmW2, fb, t.n * 256 + 64 * i, kb * BK, t.e);
            }
            }
            used |= 1u << s;
            last_par = (last_par & ~(1u << s)) | (ph << s);
            if (++s == kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
          }
        }
      producer_done:
        for (int i = 0; i < kStages; ++i)
          if ((used >> i) & 1u) mbar_wait_drain(&full[i], (last_par >> i) & 1u);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ------------------------------------------ MMA issuer
        const uint32_t idesc1 = idesc_bf16(kBM, 2 * p.hn, false, true);
        const uint32_t idesc2 = idesc_bf16(kBM, 256, false, true);
        int s = 0, acc = 0;
        uint32_t ph = 0, aph = 0;
        for (int j = 0;; ++j) {
          if (!mbar_wait(&qfull[j % kQ], (j / kQ) & 1, abort_flag, p.status, 160)) goto mma_done;
          const int L = qtile[j % kQ];
          mbar_arrive(&qempty[j % kQ]);
          if (L >= geo.total) break;
          const RUnit u = ring_decode(p, geo, L, kTpu);
          const bool g1 = (u.t[0].phase == 1);
          const int nkb = g1 ? p.kb1 : p.kb2;
          // a pair unit takes two accumulators at once (the next two in the
          // order the epilogue drains them); other units one per tile, in turn
          const int passes = u.pair ? 1 : u.nt;
          for (int ti = 0; ti < passes; ++ti) {
          const RTile t = ti == 0 ? u.t[0] : u.t[1];
          const int acc0 = acc;
          if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, p.status, 200 + acc)) goto mma_done;
          if (++acc == kAcc) {
            acc = 0;
            aph ^= 1u;
          }
          int acc1 = acc0;
          if (u.pair) {
            acc1 = acc;
            if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, p.status, 200 + acc)) goto mma_done;
            if (++acc == kAcc) {
              acc = 0;
              aph ^= 1u;
            }
          }
          tc_fence_after();
          const uint32_t dt = tmem_base + (uint32_t)acc0 * 256u;
          const uint32_t dt1 = tmem_base + (uint32_t)acc1 * 256u;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&full[s], ph, abort_flag, p.status, 300 + s)) goto mma_done;
            tc_fence_after();
            if (g1 && kb == nkb - 1) red_release_add(&p.freed[t.w % p.S], u.pair ? 2 : 1);  // ring rows landed
            const uint32_t sa = smem_u32(stages + (size_t)s * kStageBytes);
            const uint32_t sb = sa + (u.pair ? 2u : 1u) * kABytes;
            if constexpr (FP8) {
              // stage the scale tiles into this stage's TMEM columns, then 4
              // block-scaled MMAs of K = 32, each reading its block's scale byte
              const uint32_t sf = smem_u32(sfbuf + (size_t)s * kSfBytes);
              const uint32_t tsa = tmem_base + kTmemSf + (uint32_t)s * 16u;
              const uint32_t tsb = tsa + 8u;
              tc_cp_32x128b_warpx4(tsa, sdesc_plain(sf, 16, 128));
              tc_cp_32x128b_warpx4(tsb, sdesc_plain(sf + 512, 16, 128));
              tc_cp_32x128b_warpx4(tsb + 4u, sdesc_plain(sf + 1024, 16, 128));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc_mma_mxf8(dt, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024),
                            idesc_mxf8(kBM, 256, kk), tsa, tsb, (kb > 0 || kk > 0) ? 1u : 0u);
            } else if (t.thin) {
              // weight slices (MN-major) x tile rows (K-major, N = rows rounded to 16)
              const uint32_t idt = idesc_bf16(kBM, (t.rows + 15) & ~15, true, false);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t bd = sdesc_sw128(sa + kk * 32, 16, 1024);
                const uint32_t accf = (kb > 0 || kk > 0) ? 1u : 0u;
                tc_mma_f16(dt, sdesc_sw128(sb + kk * 2048, 8192, 1024), bd, idt, accf);
                tc_mma_f16(dt + 128u, sdesc_sw128(sb + 16384 + kk * 2048, 8192, 1024), bd, idt, accf);
              }
            } else {
              // each tile's accumulator sees the same MMAs in the same order
              // as a tile of its own
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                tc_mma_f16(dt, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 2048, 8192, 1024),
                           g1 ? idesc1 : idesc2, (kb > 0 || kk > 0) ? 1u : 0u);
              if (u.pair) {
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                  tc_mma_f16(dt1, sdesc_sw128(sa + kABytes + kk * 32, 16, 1024),
                             sdesc_sw128(sb + kk * 2048, 8192, 1024), g1 ? idesc1 : idesc2,
                             (kb > 0 || kk > 0) ? 1u : 0u);
              }
            }
            tc_commit(smem_u32(&empty[s]));
            if (++s == kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
          tc_commit(smem_u32(&tfull[acc0]));
          if (u.pair) tc_commit(smem_u32(&tfull[acc1]));
          }
        }
      mma_done:
        tc_commit(smem_u32(drain));
        mbar_wait_drain(drain, 0);
      }
    } else if (warp < 2 + kEpiWarps) {
      // -------------------------------------------- epilogue warps
      const int q = warp & 3;
      int acc = 0, buf = 0;
      uint32_t aph = 0;
      const uint32_t stg = smem_u32(staging) + (uint32_t)(warp - 2) * 2u * kOutTile;
      // this warp's 32 rows x 64 columns (v = this lane's row) as bf16 through
      // the next swizzled staging tile to a TMA store at (col, row) of m
      auto put64 = [&](const CUtensorMap* m, const float* v, int col, int row) {
        if (lane == 0) bulk_wait_read<1>();
        __syncwarp();
        const uint32_t sbuf = stg + (uint32_t)buf * kOutTile;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          st_shared_v4(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4),
                       pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                       pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(m, sbuf, col, row);
          bulk_commit();
        }
        buf ^= 1;
      };
      for (int j = 0;; ++j) {
        if (!mbar_wait(&qfull[j % kQ], (j / kQ) & 1, abort_flag, p.status, 170)) break;
        const int L = qtile[j % kQ];
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[j % kQ]);
        if (L >= geo.total) break;
        const RUnit un = ring_decode(p, geo, L, kTpu);
        bool eok = true;
        for (int ti = 0; ti < un.nt; ++ti) {  // the unit's tiles, in accumulator order
        const RTile t = ti == 0 ? un.t[0] : un.t[1];
        if (!mbar_wait(&tfull[acc], aph, abort_flag, p.status, 400 + acc)) {
          eok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + (uint32_t)acc * 256u + ((uint32_t)(q * 32) << 16);
        if (FP8 && t.phase == 1) {
          // SwiGLU; A quantised along f for GEMM2 (each lane's 32 columns are
          // one block), A and H in bf16 when saving
          const size_t row = (size_t)t.mt * kBM + q * 32 + lane;
          for (int c = 0; c < p.hn; c += 32) {
            float g[32], u[32], a[32];
            tmem_ld32(tb + c, g);
            tmem_ld32(tb + p.hn + c, u);
            const int col = t.n * p.hn + c;
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = silu_f(g[i]) * u[i];
            uint4 lo, hi;
            const uint8_t sc = mx_quant32(a, lo, hi);
            uint4* qd = reinterpret_cast<uint4*>(p.Aq + row * p.f + col);
            qd[0] = lo;
            qd[1] = hi;
            p.As[mx_sf_offset(row, col >> 5, p.f >> 7)] = sc;
            if (p.A != nullptr) store32_bf16(p.A + row * p.f + col, a);
            if (p.H != nullptr) {
              store32_bf16(p.H + row * (2 * p.f) + col, g);
              store32_bf16(p.H + row * (2 * p.f) + p.f + col, u);
            }
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          __threadfence();
          __syncwarp();
          if (lane == 0) red_release_add(&p.a_ready[t.mt], 1);
        } else if (FP8) {
          // Y rows in expert order with direct stores
          const size_t row = (size_t)t.mt * kBM + q * 32 + lane;
          for (int c = 0; c < 256; c += 32) {
            const int col = t.n * 256 + c;
            if (col >= p.d) break;
            float v[32];
            tmem_ld32(tb + c, v);
            store32_bf16(p.Y + row * p.d + col, v);
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          __threadfence();
          __syncwarp();
          if (lane == 0) red_release_add(p.done2, 1);
        } else if (t.thin && t.phase == 2) {
          // thin GEMM2 tile: lanes hold output columns (two halves of 128),
          // TMEM columns the tile's rows; the rows of Y go out through the
          // warp's drained staging area used as a transpose tile
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          uint8_t* tr = staging + (size_t)(warp - 2) * 2 * kOutTile;
          const int nthin = (t.rows + 15) & ~15;
          for (int h = 0; h < 2; ++h) {
            const int c0 = t.n * 256 + h * 128 + q * 32;
            if (c0 >= p.d) continue;
            for (int t0 = 0; t0 < nthin; t0 += 32) {
              float v[32];
              tmem_ld32(tb + h * 128 + t0, v);
              const size_t r0 = (size_t)t.mt * kBM + t0;
              ring_store_cols_t(tr, v, p.Y + r0 * p.d + c0, p.d, min(32, t.rows - t0), lane);
            }
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          __threadfence();
          __syncwarp();
          if (lane == 0) red_release_add(p.done2, 1);
        } else if (t.thin) {
          // thin GEMM1 tile: lanes hold gate / up columns, TMEM columns hold
          // tokens; rows go out through the warp's drained staging area used as
          // a transpose tile (all 128 rows: zeros past the expert's rows)
          if (lane == 0) bulk_wait_read<0>();
          uint8_t* tr = staging + (size_t)(warp - 2) * 2 * kOutTile;
          const int nthin = (t.rows + 15) & ~15;
          const int c0 = t.n * 128 + q * 32;
          for (int t0 = 0; t0 < kBM; t0 += 32) {
            float g[32], u[32], a[32];
            if (t0 < nthin) {
              tmem_ld32(tb + t0, g);
              tmem_ld32(tb + 128 + t0, u);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) g[i] = u[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const bool ok = t0 + i < t.rows;
              g[i] = ok ? g[i] : 0.f;
              u[i] = ok ? u[i] : 0.f;
              a[i] = ok ? silu_f(g[i]) * u[i] : 0.f;
            }
            const size_t r0 = (size_t)t.mt * kBM + t0;
            ring_store_cols_t(tr, a, p.A + r0 * p.f + c0, p.f, 32, lane);
            if (p.H != nullptr) {
              ring_store_cols_t(tr, g, p.H + r0 * (2 * p.f) + c0, 2 * p.f, 32, lane);
              ring_store_cols_t(tr, u, p.H + r0 * (2 * p.f) + p.f + c0, 2 * p.f, 32, lane);
            }
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          __threadfence();
          __syncwarp();
          if (lane == 0) red_release_add(&p.a_ready[t.mt], 1);
        } else if (t.phase == 1) {
          // SwiGLU: A (and H when saving) through swizzled staging and TMA
          // stores of 32 x 64 tiles
          const int row = t.mt * kBM + q * 32;
          for (int c = 0; c < p.hn; c += 64) {
            float g[64], u[64];
            tmem_ld32(tb + c, g);
            tmem_ld32(tb + c + 32, g + 32);
            tmem_ld32(tb + p.hn + c, u);
            tmem_ld32(tb + p.hn + c + 32, u + 32);
            const int col = t.n * p.hn + c;
            if (p.H != nullptr) {
              put64(&tmHo, g, col, row);
              put64(&tmHo, u, p.f + col, row);
            }
#pragma unroll
            for (int i = 0; i < 64; ++i) g[i] = silu_f(g[i]) * u[i];
            put64(&tmAo, g, col, row);
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          if (lane == 0) {
            bulk_wait<0>();  // this warp's A rows are in global memory before GEMM2 reads them
            fence_proxy_async_global();
            __threadfence();
            red_release_add(&p.a_ready[t.mt], 1);
          }
          __syncwarp();
        } else {
          // Y tile to expert order through swizzled staging + TMA stores
          const int row = t.mt * kBM + q * 32;
          for (int c = 0; c < 4; ++c) {
            float v[64];
            tmem_ld32(tb + c * 64, v);
            tmem_ld32(tb + c * 64 + 32, v + 32);
            const int col = t.n * 256 + c * 64;
            if (col >= p.d) continue;
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
            const uint32_t sbuf = stg + (uint32_t)buf * kOutTile;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              st_shared_v4(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4),
                           pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                           pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmY, sbuf, col, row);
              bulk_commit();
            }
            buf ^= 1;
          }
          tc_fence_before();
          mbar_arrive(&tempty[acc]);
          if (lane == 0) {
            bulk_wait<0>();              // this warp's Y rows are in global memory
            fence_proxy_async_global();
            __threadfence();
            red_release_add(p.done2, 1);
          }
          __syncwarp();
        }
        if (++acc == kAcc) {
          acc = 0;
          aph ^= 1u;
        }
        }
        if (!eok) break;
      }
      if (lane == 0) bulk_wait<0>();
    } else if (p.G == 0) {
      // -------------------------------------------- gather warps (warp split)
      // The last kGatherWarps warps of every CTA copy their share of each
      // window (rows r0 + gwi + i * ncta, gwi this warp's global index, ncta
      // the number of gather warps) into the ring slot with plain 16-byte
      // loads and stores, two rows at a time, 8 loads per lane and row in
      // flight; source-row indices are read 32 at a time and shuffled.
      const int nvec = p.d >> 3, ncta = gridDim.x * kGatherWarps;
      const int gwi = blockIdx.x * kGatherWarps + (warp - 2 - kEpiWarps);
      for (int w = 0; w < geo.nW; ++w) {
        const int s = w % p.S, gen = w / p.S;
        int ok = 1;
        if (lane == 0)
          ok = (gen == 0) || wait_counter(&p.freed[s], gen * geo.F1, p.gabort, p.status, 500 + s, limit);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const int r0 = w * p.mb, r1 = min(r0 + p.mb, geo.rp);
        const int n = (r0 + gwi < r1) ? (r1 - r0 - gwi + ncta - 1) / ncta : 0;
        __nv_bfloat16* slot = p.ring + (size_t)s * p.mb * p.d;
        if constexpr (FP8) {
          for (int i = 0; i < n; ++i) {
            const int pa = gwi + i * ncta;  // row within the window
            ring_quant_row(p, __ldg(p.row_of_pad + r0 + pa), (size_t)s * p.mb + pa, lane);
          }
        } else
        for (int c0 = 0; c0 < n; c0 += 32) {
          const int my = (c0 + lane < n) ? __ldg(p.row_of_pad + r0 + gwi + (size_t)(c0 + lane) * ncta) : -1;
          const int cn = min(32, n - c0);
          for (int i = 0; i < cn; i += 2) {
            const int ra = __shfl_sync(0xffffffffu, my, i);
            const int rb = __shfl_sync(0xffffffffu, my, (i + 1) & 31);
            const bool two = i + 1 < cn;
            const int pa = gwi + (c0 + i) * ncta;  // row within the window
            const uint4* sa = reinterpret_cast<const uint4*>(p.x + (size_t)(ra < 0 ? 0 : ra / p.k) * p.d);
            const uint4* sb = reinterpret_cast<const uint4*>(p.x + (size_t)(rb < 0 ? 0 : rb / p.k) * p.d);
            uint4* da = reinterpret_cast<uint4*>(slot + (size_t)pa * p.d);
            uint4* db = reinterpret_cast<uint4*>(slot + (size_t)(pa + ncta) * p.d);
            for (int v0 = lane; v0 < nvec; v0 += 32 * 8) {
              uint4 a[8], b[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int v = v0 + 32 * u;
                a[u] = (ra >= 0 && v < nvec) ? ldg_nc_v4(sa + v) : make_uint4(0, 0, 0, 0);
                b[u] = (two && rb >= 0 && v < nvec) ? ldg_nc_v4(sb + v) : make_uint4(0, 0, 0, 0);
              }
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int v = v0 + 32 * u;
                if (v < nvec) {
                  stg_v4(da + v, a[u]);
                  if (two) stg_v4(db + v, b[u]);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          if (inject != w + 1) red_release_add(&p.ready[s], 1);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, kTmemCols);
    }
  }

  // ======================================================== weighted merge
  if (threadIdx.x == 0)
    s_ok = wait_counter(p.done2, kEpiWarps * geo.total2, p.gabort, p.status, 800, limit);
  __syncthreads();
  if (!s_ok) return;
  // every window's GEMM1 tiles acquired its rows before GEMM2 could finish:
  // the ring now holds the last ring_slots windows for the (BF16) backward
  if (!FP8 && blockIdx.x == 0 && threadIdx.x == 0) *p.ring_valid = 1;
  for (int t = blockIdx.x; t < p.T; t += gridDim.x) {
    if (threadIdx.x < p.k) {
      s_pos[threadIdx.x] = p.pos_pad[(size_t)t * p.k + threadIdx.x];
      s_w[threadIdx.x] = p.topk_w[(size_t)t * p.k + threadIdx.x];
    }
    __syncthreads();
    merge_token<true>(p.Y, s_pos, s_w, true, t, p.k, p.d, p.out, threadIdx.x, blockDim.x);
    __syncthreads();
  }
}

}  // namespace

namespace {

// Launch of the ring kernel; W1 / W2 are bf16, or (FP8) E4M3 codes with
// their scale tiles W1s / W2s as moe_quantize_mxfp8 writes them.
template <bool FP8>
cudaError_t ring_launch(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* x,
                        const void* W1, const uint8_t* W1s, const void* W2, const uint8_t* W2s,
                        const float* topk_w, __nv_bfloat16* A, __nv_bfloat16* H, __nv_bfloat16* out,
                        cudaStream_t st) {
  constexpr size_t kSmem = RingCfg<FP8>::kSmem;
  const int sms = num_sms();
  RingParams p{};
  p.T = c.T;
  p.d = c.d;
  p.f = c.f;
  p.E = c.E;
  p.k = c.k;
  p.S = c.ring_slots;
  p.mb = ring_window_rows(c);
  p.mtw = p.mb / kBM;
  p.G = c.gather_ctas;
  if (p.G < 0 || p.G >= sms) return cudaErrorInvalidValue;
  p.nrel = p.G > 0 ? p.G : sms * kGatherWarps;
  {
    // gather row buffers (after one zero row): up to 16 per warp in all six
    // warps, at least two per issuing warp (fewer issuing warps for very wide
    // rows); MXFP8 gathers use none
    const size_t rb = (size_t)c.d * 2;
    if (kSmem <= 2048 + 3 * rb || rb >= (1u << 20)) return cudaErrorInvalidValue;
    const size_t avail = kSmem - 2048 - rb;
    p.gw = kThreads / 32;
    p.nbw = (int)std::min<size_t>(16, avail / (p.gw * rb));
    if (p.nbw < 2) {
      p.nbw = 2;
      p.gw = (int)(avail / (2 * rb));
    }
    if (p.gw < 1) return cudaErrorInvalidValue;
  }
  p.hn = (c.f % 128 == 0) ? 128 : 64;
  p.nt1 = c.f / p.hn;
  p.nt2 = (c.d + 255) / 256;
  p.kb1 = FP8 ? c.d / BK8 : c.d / BK;
  p.kb2 = FP8 ? c.f / BK8 : c.f / BK;
  // units of two tiles halve B's L2 ingress per row but halve the number of
  // units; they pay where a tile's K loop is long and the layer offers at
  // least 8 GEMM1 units of 256 rows per SM (hidden 7168, 32768 rows: ring
  // forward 3.75 -> 3.63 ms) and cost where the K loop is short (hidden 2048:
  // 0.235 -> 0.330 ms) or the units are few (512 tokens: 0.59 -> 0.68 ms)
  const long long units2 = (long long)c.T * c.k / 256 * p.nt1;
  p.tpu = (!FP8 && p.kb1 >= 64 && units2 >= 8LL * sms) ? 2 : 1;
  {
    // lag: one window more than it takes for the tiles claimed between a
    // window's GEMM1 and its GEMM2 to keep every compute CTA busy for one
    // GEMM1 tile (relative tile costs from their FLOPs: GEMM1 128 x 2hn x d,
    // GEMM2 128 x 256 x f); the extra window covers the spread of claim times
    const double t1 = 2.0 * p.hn * c.d, t2 = 256.0 * c.f;
    const double blk = p.mtw * (p.nt1 * t1 + p.nt2 * t2);
    p.lag = std::min(4, 1 + (int)std::ceil((sms - p.G) * t1 / blk));
  }
  p.mt_off = ws.mt_off();
  p.counts = counts;
  // thin GEMM1 tiles (weights on the MMA's M, the tile's rows on N): every
  // partial tile at hidden <= 4096; at larger hidden only tiles of at most 32
  // rows, which then also load just their rows
  p.thin = (!FP8 && c.f % 128 == 0) ? 1 : 0;
  p.thin_rows = gemm1_thin_enabled(c) ? kBM - 1 : 32;
  p.thin2 = (!FP8 && p.thin_rows <= 32) ? 1 : 0;  // measured: Kimi-like 3.58 -> 3.51 ms; no gain at hidden 2048
  p.hdr = ws.hdr();
  p.row_of_pad = ws.row_of_pad();
  p.pos_pad = ws.pos_pad();
  p.topk_w = topk_w;
  p.x = x;
  p.ring = static_cast<__nv_bfloat16*>(ws.at(ws.L.ring));
  p.ring_sf = static_cast<uint8_t*>(ws.at(ws.L.ring)) + (size_t)p.S * p.mb * c.d;
  p.A = A;
  p.H = H;
  p.Y = static_cast<__nv_bfloat16*>(ws.at(ws.L.Yp));
  p.out = out;
  p.W1s = W1s;
  p.W2s = W2s;
  if (FP8) {
    p.Aq = static_cast<uint8_t*>(ws.at(ws.L.Aq));
    p.As = p.Aq + (size_t)ws.L.Rp_max * c.f;
  }
  int* ctr = static_cast<int*>(ws.at(ws.L.ctr));
  p.ready = ctr;
  p.freed = ctr + p.S;
  p.done2 = ctr + 2 * p.S;
  p.gabort = ctr + 2 * p.S + 1;
  p.tile_next = ctr + 2 * p.S + 2;
  p.a_ready = ctr + 2 * p.S + 3;
  p.status = ws.hdr() + kHdrStatus;
  p.ring_valid = ws.hdr() + kHdrRingValid;

  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  CUtensorMap tmX, tmW1, tmA, tmW2, tmY, tmX16, tmA16, tmAo, tmHo;
  if (FP8) {
    // K-major E4M3: 128-byte K boxes of 128 rows (W2: 256 rows)
    if (!map2d(&tmX, p.ring, c.d, (uint64_t)p.S * p.mb, 128, kBM, true) ||
        !map3d(&tmW1, W1, c.d, 2ull * c.f, c.E, 128, 128, true) ||
        !map2d(&tmA, p.Aq, c.f, rows, 128, kBM, true) || !map3d(&tmW2, W2, c.f, c.d, c.E, 128, 256, true))
      return cudaErrorInvalidValue;
    tmY = tmX;  // Y leaves with direct stores
    tmX16 = tmX;
    tmA16 = tmA;
    tmAo = tmHo = tmX;
  } else if (!map2d(&tmX, p.ring, c.d, (uint64_t)p.S * p.mb, 64, kBM) ||
             !map2d(&tmX16, p.ring, c.d, (uint64_t)p.S * p.mb, 64, 16) ||
             !map2d(&tmA16, A, c.f, rows, 64, 16) || !map2d(&tmAo, A, c.f, rows, 64, 32) ||
             (H != nullptr ? !map2d(&tmHo, H, 2ull * c.f, rows, 64, 32) : !map2d(&tmHo, A, c.f, rows, 64, 32)) ||
             !map3d(&tmW1, W1, 2ull * c.f, c.d, c.E, 64, 64) || !map2d(&tmA, A, c.f, rows, 64, kBM) ||
             !map3d(&tmW2, W2, c.d, c.f, c.E, 64, 64) || !map2d(&tmY, p.Y, c.d, rows, 64, 32)) {
    return cudaErrorInvalidValue;
  }

  cudaError_t err = cudaMemsetAsync(ctr, 0, ws.L.ctr_bytes, st);
  if (err != cudaSuccess) return err;
  auto kern = p.tpu == 2 ? ring_forward_kernel<FP8, FP8 ? 1 : 2> : ring_forward_kernel<FP8, 1>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  void* args[] = {&tmX, &tmW1, &tmA, &tmW2, &tmY, &tmX16, &tmA16, &tmAo, &tmHo, &p};
  TraceScope ts(FP8 ? "ring_forward_mxfp8" : "ring_forward", st);
  return cudaLaunchCooperativeKernel((const void*)kern, dim3(sms), dim3(kThreads), args, kSmem, st);
}

}  // namespace

cudaError_t ring_forward(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* x,
                         const __nv_bfloat16* W1, const __nv_bfloat16* W2, const float* topk_w,
                         __nv_bfloat16* A, __nv_bfloat16* H, __nv_bfloat16* out, cudaStream_t st) {
  return ring_launch<false>(c, ws, counts, x, W1, nullptr, W2, nullptr, topk_w, A, H, out, st);
}

cudaError_t ring_forward_mx(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* x,
                            const uint8_t* W1q, const uint8_t* W1s, const uint8_t* W2q, const uint8_t* W2s,
                            const float* topk_w, __nv_bfloat16* A, __nv_bfloat16* H, __nv_bfloat16* out,
                            cudaStream_t st) {
  return ring_launch<true>(c, ws, counts, x, W1q, W1s, W2q, W2s, topk_w, A, H, out, st);
}

}  // namespace moe
