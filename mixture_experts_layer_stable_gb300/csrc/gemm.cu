// gemm.cu -- grouped expert GEMMs on the 5th-generation tensor cores (tcgen05).
//
// The expert FFN is a grouped GEMM over each expert's contiguous rows, fed to
// the tensor cores (leiphone "MoK..." sections 01 and 02); its SwiGLU and the
// SwiGLU backward with the routing-weight gradient are fused into the GEMM
// epilogues (Marktechpost "Cursor开源MoK..." three design decisions).
//
// One persistent kernel template, one CTA per SM (192 threads):
//   warp 0      TMA producer: 64-wide K slices of A and B into a 4-stage ring
//               of 128-byte-swizzled shared-memory tiles (mbarrier full/empty)
//   warp 1      TMEM allocator and MMA issuer: one thread issues
//               tcgen05.mma.cta_group::1.kind::f16 (128 x N x 16, bf16 -> fp32)
//               into one of two TMEM accumulators (2 x 256 columns), commits
//               to the stage's "empty" barrier and, per tile, to "tmem full"
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, fused math,
//               stores (TMA tensor stores through swizzled staging tiles, or
//               direct vector stores), then "tmem empty"
// Tiles (all modes 128 rows x up to 256 columns):
//   ROWS   forward / dgrad: M tiles are 128-row blocks of the padded
//          expert-ordered buffer (one expert each), N tiles across the output,
//          K = d, f or 2f.  Tile order: expert, then N tile, then M tile, so
//          tiles sharing an expert's weight slice run side by side.
//   WGRAD  weight gradients: per expert e, an (M x N) grid of tiles of
//          dW[e] = A_e^T B_e with K = the expert's rows (zero-padded to 64);
//          experts without rows produce zero tiles.
// Every wait is bounded (%globaltimer); on expiry the CTA records
// MOE_ERR_TIMEOUT in the workspace status word, stops, drains its in-flight
// copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <math.h>

#include "moe_internal.h"
#include "gemm_common.cuh"
#include "mx.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int BK = 64;                    // bf16 K elements per stage (128 bytes)
constexpr int BK8 = 128;                  // fp8 K elements per stage (128 bytes)
constexpr int kABytes = kBM * BK * 2;     // 16 KB
constexpr int kBBytes = 256 * BK * 2;     // 32 KB
constexpr int kBHalfBytes = 128 * BK * 2; // 16 KB: a CTA's half of B in pair mode
constexpr int kSfBytes = 1536;            // fp8 stage: one A scale tile + two B scale tiles
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kOutTile = 32 * 128;        // 32 rows x 64 bf16, swizzled staging tile
constexpr int kTmemCols = 512;
constexpr int kTmemSf = 256;              // fp8: per-stage scale columns start here
constexpr int kTmemSfStride = 16;         // fp8: TMEM columns per stage (A: 4, B: 8; 8-aligned)
constexpr int kTrTile = 32 * 80;          // 32 rows x (64 + 16 pad) bytes: per-warp transpose tile

enum Epi { EPI_STORE = 0, EPI_SWIGLU = 1, EPI_DSWIGLU = 2, EPI_LOGITS = 3 };

// Pipeline shape per variant.  The fp8 kernels keep one TMEM accumulator
// (256 columns) and put the per-stage scale factors (16 columns a stage) in
// the other half; the fp8 store variant has 3 stages to leave room for the
// store staging tiles.  In pair mode a stage holds the CTA's 128 rows of A
// and its half (128 columns) of B: 32 KB, so six stages fit.
// Unit sets of the pair GEMMs: all units, or (split) the heavy units and
// the light units as two kernels running side by side on every SM -- the
// heavy kernel leaves room (shared memory, TMEM) for one light CTA per SM.
// Their pipeline depths (stages) share one SM's shared memory.
enum UnitSet { UNITS_ALL = 0, UNITS_HEAVY = 1, UNITS_LIGHT = 2 };
#ifndef MOE_SPLIT_HEAVY_STAGES
#define MOE_SPLIT_HEAVY_STAGES 3
#endif
#ifndef MOE_SPLIT_LIGHT_STAGES
#define MOE_SPLIT_LIGHT_STAGES 4
#endif

template <int EPI, bool FP8, bool WGRAD, bool PAIR, int UM = UNITS_ALL>
struct KCfg {
  static_assert(!(PAIR && FP8), "pair mode is bf16 only");
  static_assert(UM == UNITS_ALL || (PAIR && !WGRAD), "unit sets split the row pair GEMMs");
  // a light unit's stage: its weight slice (MMA A) and at most 16 of its rows
  // per CTA (MMA B, nt <= kLightRows)
  static constexpr int kStageBytes = UM == UNITS_LIGHT ? kABytes + 16 * 128
                                                       : kABytes + (PAIR ? kBHalfBytes : kBBytes);
  static constexpr int kStages = UM == UNITS_HEAVY ? MOE_SPLIT_HEAVY_STAGES
                                 : UM == UNITS_LIGHT ? MOE_SPLIT_LIGHT_STAGES
                                 : PAIR ? 6 : (FP8 && EPI == EPI_STORE) ? 3 : 4;
  // swizzled staging tiles per epilogue warp for the TMA-store epilogues
  // (light units only need their transpose tiles)
  static constexpr int kOutBufs = (UM == UNITS_LIGHT && EPI == EPI_STORE) ? 1
                                  : (EPI == EPI_STORE || (EPI != EPI_LOGITS && !FP8)) ? 2 : 0;
  static constexpr int kAcc = (FP8 || UM == UNITS_HEAVY) ? 1 : 2;
  // TMEM columns and the distance between accumulators
  static constexpr uint32_t kTmemAlloc = UM == UNITS_HEAVY ? 256u : UM == UNITS_LIGHT ? 64u : 512u;
  static constexpr uint32_t kAccStride = UM == UNITS_LIGHT ? (uint32_t)kLightRows : 256u;
  // scale-tile region rounded to 1024 bytes: the swizzled staging tiles after
  // it must start on a 1024-byte boundary for the 128-byte swizzle pattern
  static constexpr size_t kSfRegion = FP8 ? ((size_t)kStages * kSfBytes + 1023) / 1024 * 1024 : 0;
  // epilogue staging: kOutBufs swizzled tiles per warp; light SwiGLU units
  // need only the gate warps' exchange buffers (32 x 32 fp32) and a
  // transpose tile per warp
  static constexpr bool kLightSwiglu = UM == UNITS_LIGHT && EPI == EPI_SWIGLU;
  static constexpr size_t kStaging = kLightSwiglu ? 2 * 4096 + (size_t)kEpiWarps * kTrTile
                                                  : (size_t)kEpiWarps * kOutBufs * kOutTile;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kSfRegion + kStaging + 512;
  // the thin tiles' transpose tile lives in the warp's staging tiles
  static_assert(EPI != EPI_SWIGLU || FP8 || kOutBufs * kOutTile >= kTrTile, "transpose tile");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct Params {
  int E;
  int num_kb;      // ROWS: K / 64
  int n_tiles;     // tiles along N
  int m_tiles_w;   // WGRAD: tiles along M
  int umma_n;      // MMA N (64..256)
  int hn;          // SWIGLU: gate (and up) columns per tile
  int f;
  int out_cols;    // output width (stores starting at or past it are skipped)
  int out_rows;    // WGRAD: output height
  const int* mt_off;  // ROWS: [E+1] prefix of 128-row tiles per expert
  const int* pt_off;  // ROWS, pair mode: [E+1] prefix of tile pairs per expert
  const int* hv_off;  // ROWS, pair mode: [E+1] prefix of heavy units per expert
  const int* lt_off;  // ROWS, pair mode: [E+1] prefix of light units per expert
  const int* counts;  // WGRAD: [E] rows per expert
  const int* poff;    // WGRAD: [E+1] padded row prefix
  __nv_bfloat16* out0;  // SWIGLU: A [rows, f]      DSWIGLU: dH [rows, 2f]
  __nv_bfloat16* out1;  // SWIGLU: H [rows, 2f] / 0 DSWIGLU: gA [rows, f]
  const __nv_bfloat16* Hs;  // DSWIGLU: saved H
  const __nv_bfloat16* As;  // DSWIGLU: saved A
  const float* g_pad;       // DSWIGLU: routing weight per padded row
  float* dgp;               // DSWIGLU: [rows, n_tiles] partial <dA', A>
  const uint8_t* sfa;       // FP8: scale tiles of A [rows, K]
  const uint8_t* sfb;       // FP8: scale tiles of the weight stack [E * b_rows, K]
  int k_groups;             // FP8: K / 128
  int b_rows;               // FP8: rows (N) of one expert's weight
  uint8_t* q_out;           // FP8 SWIGLU: E4M3 codes of A [rows, f]; DSWIGLU: of dH [rows, 2f]
  uint8_t* q_sf;            // FP8 SWIGLU: scale tiles of A; DSWIGLU: of dH (blocks along 2f)
  uint8_t* qt0;             // FP8 DSWIGLU: dH transposed [2f, ldt], blocks of 32 rows
  uint8_t* qt0_sf;
  uint8_t* qt1;             // FP8 DSWIGLU: g*A transposed [f, ldt], blocks of 32 rows
  uint8_t* qt1_sf;
  int ldt;                  // FP8: row length (K) of the transposed operands (the padded row capacity)
  int kstep;                // WGRAD: expert rows per K step (64 bf16, 128 fp8)
  int thin;                 // bf16 GEMM1: compute an expert's partial last tile swapped
  // dense mode (router GEMMs): ROWS without mt_off walks dense_mt 128-row
  // tiles of one matrix; WGRAD without counts contracts over dense_k rows
  int dense_mt, dense_k, T;
  float* logits;            // LOGITS: fp32 [T, E] output (may be null when the top-k is fused)
  int* topk_ids;            // LOGITS: fused top-k (one N tile): ids [T, k] and weights [T, k]
  float* topk_w;
  int k;
  int* status;
};

struct Tile {
  int e, m, n, kb_count, row0, krow0;
  int rows;    // valid rows of a ROWS tile
  int nt;      // thin pair unit: MMA N (rows rounded up to 32), half in each CTA
  bool thin;   // tile computed as (weights)^T x (rows)^T, tokens on N
  bool valid;  // pair mode: the odd CTA's tile past the expert's last tile is not
};

// Work units: tiles, or in pair mode pairs of M-adjacent tiles of one expert
// (the even CTA of the pair takes M tile 2j, the odd one 2j + 1).
template <int UM>
__device__ __forceinline__ const int* pair_units(const Params& p) {
  return UM == UNITS_HEAVY ? p.hv_off : UM == UNITS_LIGHT ? p.lt_off : p.pt_off;
}

template <bool WGRAD, bool PAIR, int UM = UNITS_ALL>
__device__ __forceinline__ int total_units(const Params& p) {
  if (WGRAD) return p.E * (PAIR ? (p.m_tiles_w + 1) >> 1 : p.m_tiles_w) * p.n_tiles;
  if (p.mt_off == nullptr) return p.dense_mt * p.n_tiles;
  return __ldg((PAIR ? pair_units<UM>(p) : p.mt_off) + p.E) * p.n_tiles;
}

// Position L of a CTA's (cluster's) walk -> work unit.  Units are numbered
// expert by expert; positions 2h and 2h + 1 take unit h from the front and
// unit total-1-h from the back (which one goes first flips every `stride`
// positions), so every wave mixes the first experts' units with the last
// experts' and each CTA alternates between the two.  When the expert loads
// are skewed, tiles of busy experts (limited by the tensor cores and L2) then
// run beside tiles of experts with a few rows (limited by streaming their
// weights from HBM).  A bijection on [0, total).
__device__ __forceinline__ int unit_at(int L, int total, int stride) {
  const int h = L >> 1;
  const bool swap = (((L - (L & 1)) / stride) & 1) != 0;
  const bool back = ((L & 1) != 0) != swap;
  return back ? total - 1 - h : h;
}

template <bool WGRAD, bool PAIR, int UM = UNITS_ALL>
__device__ __forceinline__ Tile decode(const Params& p, int L, int rank) {
  Tile t;
  t.valid = true;
  if (!WGRAD && p.mt_off == nullptr) {
    // dense: tile m of one [T, K] matrix
    t.e = 0;
    t.m = L / p.n_tiles;
    t.n = L - t.m * p.n_tiles;
    t.row0 = t.m * kBM;
    t.kb_count = p.num_kb;
    t.krow0 = 0;
    t.rows = min(kBM, p.T - t.row0);
    t.nt = 0;
    t.thin = false;
  } else if (!WGRAD) {
    const int* uoff = PAIR ? pair_units<UM>(p) : p.mt_off;
    const int e = find_expert(uoff, p.E, L / p.n_tiles);
    const int u0 = __ldg(uoff + e);
    const int ue = __ldg(uoff + e + 1) - u0;
    const int m0 = PAIR ? __ldg(p.mt_off + e) : u0;
    const int loc = L - u0 * p.n_tiles;
    int mrel = loc % ue;
    t.rows = kBM;
    t.nt = 0;
    t.thin = false;
    if (PAIR) {
      const int me = __ldg(p.mt_off + e + 1) - m0;
      // a light unit is its expert's last tile; other units are pairs 2j, 2j+1
      mrel = UM == UNITS_LIGHT ? me - 1 : 2 * mrel;
      if (p.thin && mrel + 1 == me) {
        // thin pair unit: the expert's last tile has no partner; both CTAs
        // compute it, each with half of the weight columns on M
        t.thin = true;
        t.rows = min(kBM, __ldg(p.counts + e) - mrel * kBM);
        t.nt = (t.rows + 31) & ~31;
      } else {
        mrel += rank;
        t.valid = mrel < me;
      }
    }
    t.e = e;
    t.n = loc / ue;
    t.m = m0 + mrel;
    t.row0 = t.m * kBM;
    t.kb_count = p.num_kb;
    t.krow0 = 0;
    if (!t.thin && p.counts != nullptr) {
      // rows of this tile that hold routed rows (<= 0 past the expert's tiles)
      const int cnt = __ldg(p.counts + e);
      t.rows = min(kBM, cnt - mrel * kBM);
      if (!PAIR && p.thin && thin_tile(t.rows, cnt)) t.thin = true;
    }
  } else {
    t.nt = 0;
    const int mu = PAIR ? (p.m_tiles_w + 1) >> 1 : p.m_tiles_w;
    const int per = mu * p.n_tiles;
    t.e = L / per;
    const int loc = L - t.e * per;
    t.m = PAIR ? 2 * (loc % mu) + rank : loc % mu;
    t.n = loc / mu;
    t.valid = t.m < p.m_tiles_w;
    if (p.counts != nullptr) {
      t.kb_count = (__ldg(p.counts + t.e) + p.kstep - 1) / p.kstep;
      t.krow0 = __ldg(p.poff + t.e);
    } else {
      t.kb_count = (p.dense_k + p.kstep - 1) / p.kstep;
      t.krow0 = 0;
    }
    t.row0 = 0;
    t.rows = kBM;
    t.thin = false;
  }
  return t;
}

// A 32-token x 32-column block held one column per lane (v[i] = token i) is
// written to rows [0, nrows) at dst (row-major, leading dimension ld) through
// a per-warp shared transpose tile, so that each lane stores a contiguous
// 64-byte row fragment.
__device__ __forceinline__ void store_cols_t(uint8_t* tr, const float* v, __nv_bfloat16* dst,
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

// The bf16 boxes this CTA copies for k-block kb of tile t: op2 / op3 get the
// box's byte offset in the stage (A at 0, B at kABytes), its tensor map and
// coordinates.
template <bool WGRAD, bool A_MN, bool B_MN, int EPI, bool PAIR, typename Op2, typename Op3>
__device__ __forceinline__ void for_each_box(const Params& p, const Tile& t, int kb, int rank,
                                             const CUtensorMap* tmA, const CUtensorMap* tmB,
                                             Op2&& op2, Op3&& op3) {
  // MN-major B arrives in 64-column boxes; in pair mode each CTA loads half
  const int nbox = PAIR ? p.umma_n / 128 : p.umma_n / 64;
  const int kr = t.krow0 + kb * BK;
  if (t.valid) {
    if (!A_MN) {
      op2(0u, tmA, kb * BK, t.row0);
    } else {
      op2(0u, tmA, t.m * kBM, kr);
      op2(8192u, tmA, t.m * kBM + 64, kr);
    }
  }
  // first column (MN-major) or row (K-major) of this CTA's part of B
  const int bpart = t.n * 256 + (PAIR ? rank * 128 : 0);
  if (WGRAD) {
    for (int i = 0; i < nbox; ++i) op2((uint32_t)(kABytes + i * 8192), tmB, bpart + 64 * i, kr);
  } else if (B_MN) {
    for (int i = 0; i < nbox; ++i) {
      int col;
      if (EPI == EPI_SWIGLU) {
        // gate columns first, then up (pair: the even CTA holds gate)
        if (PAIR) {
          col = (rank == 0 ? t.n * p.hn : p.f + t.n * p.hn) + 64 * i;
        } else {
          const int half = nbox / 2;
          col = (i < half) ? t.n * p.hn + 64 * i : p.f + t.n * p.hn + 64 * (i - half);
        }
      } else {
        col = bpart + 64 * i;
      }
      op3((uint32_t)(kABytes + i * 8192), tmB, col, kb * BK, t.e);
    }
  } else {
    op3((uint32_t)kABytes, tmB, kb * BK, bpart, t.e);
  }
}

// CLC: a grid of one CTA per work unit (an upper bound; units past the
// schedule's total are skipped).  Each CTA takes its own unit first, and
// while working on one asks the hardware (cluster launch control) to cancel
// the launch of a CTA that has not started yet and takes that CTA's unit
// next; the producer hands the units to the MMA and epilogue warps through
// a small queue in shared memory.  One-CTA (not pair) kernels only.
constexpr int kQ = 4;  // depth of the queue of units

template <bool WGRAD, bool A_MN, bool B_MN, int EPI, bool FP8, bool PAIR, int UM = UNITS_ALL,
          bool CLC = false>
__global__ void __launch_bounds__(kThreads, UM == UNITS_ALL ? 1 : 2)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmA2,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO,
                        const __grid_constant__ CUtensorMap tmO2, const Params p) {
  using Cfg = KCfg<EPI, FP8, WGRAD, PAIR, UM>;
  static_assert(!(CLC && PAIR), "the cluster-launch-control schedule is for one-CTA kernels");
  constexpr uint32_t kTmemAlloc = Cfg::kTmemAlloc;
  constexpr uint32_t kAccStride = Cfg::kAccStride;
  // split units: once every heavy CTA is resident, the light kernel queued
  // behind this one in the stream may start on the room left on each SM
  if constexpr (UM == UNITS_HEAVY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kStages = Cfg::kStages;
  constexpr int kAcc = Cfg::kAcc;
  constexpr int kStageB = Cfg::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* stages = smem;
  uint8_t* sfbuf = smem + (size_t)kStages * kStageB;  // fp8 scale tiles, kSfBytes a stage
  uint8_t* staging = sfbuf + Cfg::kSfRegion;
  uint8_t* ctrl = staging + Cfg::kStaging;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // CLC: the queue of units and the cancel request's barrier and response
  uint64_t* qfull = reinterpret_cast<uint64_t*>(ctrl + 256);
  uint64_t* qempty = qfull + kQ;
  uint64_t* cbar = qempty + kQ;
  int* qunit = reinterpret_cast<int*>(cbar + 1);
  const uint32_t cresp = smem_u32(ctrl + 256 + 96);  // 16-byte aligned

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Pair mode: the two CTAs of a cluster walk the same work units; the even
  // CTA issues the MMAs, and its "full" and "tmem empty" barriers count both
  // CTAs' copies and epilogues.
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const int unit0 = PAIR ? (int)cluster_idx() : (int)blockIdx.x;
  const int ustride = PAIR ? (int)cluster_count() : (int)gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], PAIR ? 2 * kEpiWarps : kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    if constexpr (CLC) {
      for (int i = 0; i < kQ; ++i) {
        mbar_init(&qfull[i], 1);
        mbar_init(&qempty[i], 1 + kEpiWarps);
      }
      mbar_init(cbar, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    if (PAIR && !WGRAD) tma_prefetch_desc(&tmA2);
    tma_prefetch_desc(&tmB);
    if (Cfg::kOutBufs > 0) tma_prefetch_desc(&tmO);
    if (EPI == EPI_DSWIGLU || (EPI == EPI_SWIGLU && !FP8)) tma_prefetch_desc(&tmO2);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemAlloc);  // both CTAs, collectively
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemAlloc);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the peer's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = total_units<WGRAD, PAIR, UM>(p);
  // unit j of this CTA for the MMA and epilogue roles: the static walk, or
  // the queue the producer fills (CLC); -1 ends the walk, units past the
  // total are skipped
  auto unit_of = [&](int j, bool& ok) -> int {
    ok = true;
    if constexpr (CLC) {
      ok = mbar_wait(&qfull[j % kQ], (j / kQ) & 1, abort_flag, p.status, 170);
      if (!ok) return -1;
      const int U = qunit[j % kQ];
      __syncwarp(__activemask());  // every lane of the role has read the slot
      if ((threadIdx.x & 31) == 0) mbar_arrive(&qempty[j % kQ]);
      return U;
    } else {
      const int L = unit0 + j * ustride;
      return L < total ? unit_at(L, total, ustride) : -1;
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const int nbox = PAIR ? p.umma_n / 128 : p.umma_n / 64;
      const uint32_t b_bytes = FP8 ? (uint32_t)kBBytes
                               : (B_MN ? (uint32_t)nbox * 8192u
                                       : (uint32_t)(PAIR ? kBHalfBytes : kBBytes));
      int s = 0;
      uint32_t ph = 0, used = 0, last_par = 0;
      const uint64_t pol_stream = l2_policy_evict_first();  // weights streamed once (thin units)
      int cur = (int)blockIdx.x;  // CLC: this CTA's own unit first
      uint32_t cph = 0;
      bool pending = false;       // CLC: a cancel request in flight
      for (int j = 0;; ++j) {
        int U;
        if constexpr (CLC) {
          if (!mbar_wait(&qempty[j % kQ], ((j / kQ) & 1) ^ 1, abort_flag, p.status, 150)) goto producer_done;
          qunit[j % kQ] = cur;
          mbar_arrive(&qfull[j % kQ]);
          if (cur < 0) break;
          // ask for the next unit while this one's operands go out
          mbar_arrive_expect_tx(cbar, 16);
          clc_try_cancel(cresp, smem_u32(cbar));
          pending = true;
          U = cur;
        } else {
          const int L = unit0 + j * ustride;
          if (L >= total) break;
          U = unit_at(L, total, ustride);
        }
        if (CLC && U >= total) goto next_unit;
        {
        const Tile t = decode<WGRAD, PAIR, UM>(p, U, rank);
        // bytes landing on this stage's "full" barrier (pair: both CTAs' copies)
        uint32_t tx = (t.valid ? (uint32_t)kABytes : 0u) + b_bytes + (FP8 ? (uint32_t)kSfBytes : 0u);
        if (PAIR && t.thin) tx = 16384u + (uint32_t)(t.nt / 2) * 128u;  // weights + half the rows
        if (PAIR && rank == 0)
          tx += t.thin ? tx : (decode<WGRAD, PAIR, UM>(p, U, 1).valid ? (uint32_t)kABytes : 0u) + b_bytes;
        for (int kb = 0; kb < t.kb_count; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, 100 + s)) goto producer_done;
          const uint32_t sa = smem_u32(stages + (size_t)s * kStageB);
          const uint32_t sb = sa + kABytes;
          const uint32_t fb = PAIR ? mapa_shared(smem_u32(&full[s]), 0) : smem_u32(&full[s]);
          if (!PAIR || rank == 0) mbar_arrive_expect_tx(&full[s], tx);
          if constexpr (FP8) {
            // K-major E4M3 tiles (128 bytes of K per row) plus their scale tiles
            // ROWS: A rows at row0, K from 0; WGRAD: A = the transposed
            // operand's rows m*128 (output rows), K = the expert's rows from
            // krow0 (a multiple of 128), the same for B (one matrix, e = 0)
            const int nbt = p.b_rows >> 7;  // 128-row scale tiles per expert
            const int kc = (WGRAD ? t.krow0 : 0) + kb * BK8;
            const int kg = kc >> 7;          // K group of the scale tiles
            const int arow = WGRAD ? t.m * kBM : t.row0;
            const int be = WGRAD ? 0 : t.e;
            int nb0, nb1;
            tma_load_2d(sa, &tmA, fb, kc, arow);
            if (EPI == EPI_SWIGLU) {
              tma_load_3d(sb, &tmB, fb, kc, t.n * 128, be);
              tma_load_3d(sb + 16384, &tmB, fb, kc, p.f + t.n * 128, be);
              nb0 = t.n;
              nb1 = (p.f >> 7) + t.n;
            } else {
              tma_load_3d(sb, &tmB, fb, kc, t.n * 256, be);
              nb0 = 2 * t.n;
              nb1 = min(2 * t.n + 1, nbt - 1);  // rows past N are zero-filled; any finite scale
            }
            const uint32_t sf = smem_u32(sfbuf + (size_t)s * kSfBytes);
            bulk_load(sf, p.sfa + ((size_t)(arow >> 7) * p.k_groups + kg) * 512u, 512u, fb);
            bulk_load(sf + 512, p.sfb + (((size_t)be * nbt + nb0) * p.k_groups + kg) * 512u, 512u, fb);
            bulk_load(sf + 1024, p.sfb + (((size_t)be * nbt + nb1) * p.k_groups + kg) * 512u, 512u, fb);
          } else {
            auto load2 = [&](uint32_t off, const CUtensorMap* m, int c0, int c1) {
              if constexpr (PAIR) tma_load_2d_pair(sa + off, m, fb, c0, c1);
              else tma_load_2d(sa + off, m, fb, c0, c1);
            };
            auto load3 = [&](uint32_t off, const CUtensorMap* m, int c0, int c1, int c2) {
              if constexpr (PAIR) tma_load_3d_pair(sa + off, m, fb, c0, c1, c2);
              else tma_load_3d(sa + off, m, fb, c0, c1, c2);
            };
            if (PAIR && !WGRAD && t.thin) {
              // thin pair unit: this CTA's weight columns as the MMA's A --
              // SwiGLU: 64 gate and the matching 64 up columns; otherwise 128
              // output columns (MN-major, or K-major rows for dgrad) -- then its
              // half of the rows in 16-row boxes (the MMA's B, K-major).  The
              // weight slice is read by this unit alone: it goes into L2 with
              // evict-first priority, so the stream does not push out the
              // row tiles and weight slices other units read again
              auto loadw = [&](uint32_t off, int c0, int c1) {
                if constexpr (PAIR) tma_load_3d_pair_hint(sa + off, &tmB, fb, c0, c1, t.e, pol_stream);
                else tma_load_3d_hint(sa + off, &tmB, fb, c0, c1, t.e, pol_stream);
              };
              if (EPI == EPI_SWIGLU) {
                const int c0 = t.n * p.hn + rank * 64;
                loadw(0u, c0, kb * BK);
                loadw(8192u, p.f + c0, kb * BK);
              } else if (B_MN) {
                const int c0 = t.n * 256 + rank * 128;
                loadw(0u, c0, kb * BK);
                loadw(8192u, c0 + 64, kb * BK);
              } else {
                loadw(0u, kb * BK, t.n * 256 + rank * 128);
              }
              const int nt2 = t.nt / 2;
              for (int i = 0; i < nt2; i += 16)
                load2((uint32_t)(kABytes + i * 128), &tmA2, kb * BK, t.row0 + rank * nt2 + i);
            } else {
              for_each_box<WGRAD, A_MN, B_MN, EPI, PAIR>(p, t, kb, rank, &tmA, &tmB, load2, load3);
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
      next_unit:
        if constexpr (CLC) {
          if (!mbar_wait(cbar, cph, abort_flag, p.status, 180)) goto producer_done;
          pending = false;
          cph ^= 1u;
          cur = clc_canceled_x(cresp);
          fence_proxy_async_smem();  // the response is read before the next request overwrites it
        }
      }
    producer_done:
      // no cancel request may still be writing into shared memory at exit
      if (CLC && pending) mbar_wait_drain(cbar, cph);
      // every issued copy has landed before the CTA can exit (in pair mode the
      // even CTA's "full" barriers also count the odd CTA's copies)
      if (!PAIR || rank == 0)
        for (int i = 0; i < kStages; ++i)
          if ((used >> i) & 1u) mbar_wait_drain(&full[i], (last_par >> i) & 1u);
      if constexpr (PAIR) {
        // and every stage this CTA filled has been released by the pair's MMAs,
        // so no multicast arrival is still on its way to this CTA's barriers
        for (int i = 0; i < kStages; ++i)
          if ((used >> i) & 1u)
            if (!mbar_wait_drain(&empty[i], (last_par >> i) & 1u)) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && (!PAIR || rank == 0)) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_bf16(PAIR ? 2 * kBM : kBM, p.umma_n, A_MN, B_MN);
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      for (int j = 0;; ++j) {
        bool ok;
        const int U = unit_of(j, ok);
        if (!ok) goto mma_done;
        if (U < 0) break;
        if (CLC && U >= total) continue;
        const Tile t = decode<WGRAD, PAIR, UM>(p, U, 0);
        if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, p.status, 200 + acc)) goto mma_done;
        tc_fence_after();
        const uint32_t dt = tmem_base + (uint32_t)acc * kAccStride;
        for (int kb = 0; kb < t.kb_count; ++kb) {
          if (!mbar_wait(&full[s], ph, abort_flag, p.status, 300 + s)) goto mma_done;
          tc_fence_after();
          const uint32_t sa = smem_u32(stages + (size_t)s * kStageB);
          const uint32_t sb = sa + kABytes;
          if constexpr (FP8) {
            // stage the scale tiles into this stage's TMEM columns, then 4 MMAs
            // of K = 32, each reading its 32-element block's scale byte
            const uint32_t sf = smem_u32(sfbuf + (size_t)s * kSfBytes);
            const uint32_t tsa = tmem_base + kTmemSf + (uint32_t)s * kTmemSfStride;
            const uint32_t tsb = tsa + 8u;
            tc_cp_32x128b_warpx4(tsa, sdesc_plain(sf, 16, 128));
            tc_cp_32x128b_warpx4(tsb, sdesc_plain(sf + 512, 16, 128));
            tc_cp_32x128b_warpx4(tsb + 4u, sdesc_plain(sf + 1024, 16, 128));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              tc_mma_mxf8(dt, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024),
                          idesc_mxf8(kBM, 256, kk), tsa, tsb, (kb > 0 || kk > 0) ? 1u : 0u);
            }
          } else {
            bool issued = false;
            if constexpr (!PAIR && !WGRAD && !A_MN && B_MN) {
              if (t.thin) {
                // thin tile: the gate and up weight slices (MN-major, the MMA's
                // A, M = 128 columns each) times the tile's rows (K-major, the
                // MMA's B, N = rows rounded up to 16); D columns are tokens:
                // gate at [0, N), up at [128, 128 + N)
                const uint32_t idt = idesc_bf16(kBM, (t.rows + 15) & ~15, true, false);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                  const uint64_t bd = sdesc_sw128(sa + kk * 32, 16, 1024);
                  const uint32_t accf = (kb > 0 || kk > 0) ? 1u : 0u;
                  tc_mma_f16(dt, sdesc_sw128(sb + kk * 2048, 8192, 1024), bd, idt, accf);
                  tc_mma_f16(dt + 128u, sdesc_sw128(sb + 16384 + kk * 2048, 8192, 1024), bd, idt, accf);
                }
                issued = true;
              }
            }
            if constexpr (PAIR && !WGRAD) {
              if (t.thin) {
                // thin pair unit: D^T (weight columns on TMEM lanes -- SwiGLU:
                // gate 0..63, up 64..127 in each CTA; tokens on TMEM columns)
                // = W^T x rows^T
                constexpr bool kWmn = (EPI == EPI_SWIGLU) || B_MN;  // weights MN-major in smem
                const uint32_t idt = idesc_bf16(2 * kBM, t.nt, kWmn, false);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                  tc_mma_f16_pair(dt, kWmn ? sdesc_sw128(sa + kk * 2048, 8192, 1024)
                                           : sdesc_sw128(sa + kk * 32, 16, 1024),
                                  sdesc_sw128(sb + kk * 32, 16, 1024), idt,
                                  (kb > 0 || kk > 0) ? 1u : 0u);
                issued = true;
              }
            }
            if (!issued) {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad = A_MN ? sdesc_sw128(sa + kk * 2048, 8192, 1024)
                                         : sdesc_sw128(sa + kk * 32, 16, 1024);
                const uint64_t bd = B_MN ? sdesc_sw128(sb + kk * 2048, 8192, 1024)
                                         : sdesc_sw128(sb + kk * 32, 16, 1024);
                const uint32_t accf = (kb > 0 || kk > 0) ? 1u : 0u;
                if constexpr (PAIR) tc_mma_f16_pair(dt, ad, bd, idesc, accf);
                else tc_mma_f16(dt, ad, bd, idesc, accf);
              }
            }
          }
          if constexpr (PAIR) tc_commit_pair(smem_u32(&empty[s]), 3);
          else tc_commit(smem_u32(&empty[s]));
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if constexpr (PAIR) tc_commit_pair(smem_u32(&tfull[acc]), 3);
        else tc_commit(smem_u32(&tfull[acc]));
        if (++acc == kAcc) {
          acc = 0;
          aph ^= 1u;
        }
      }
    mma_done:
      // all issued MMAs complete before TMEM is released
      if constexpr (PAIR) tc_commit_pair(smem_u32(drain), 1);
      else tc_commit(smem_u32(drain));
      mbar_wait_drain(drain, 0);
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0, buf = 0;
    uint32_t aph = 0;
    const uint32_t stg = smem_u32(staging) + (uint32_t)(warp - 2) * (uint32_t)Cfg::kOutBufs * kOutTile;
    // This warp's 32 rows x 64 columns (v = this lane's row) as bf16 through
    // the next swizzled staging tile to a TMA store at (col, row) of m.  A
    // tile is rewritten only after the store issued from it two tiles ago has
    // finished reading it.
    auto put_tile = [&](const CUtensorMap* m, const float* v, int col, int row) {
      if (lane == 0) bulk_wait_read<(Cfg::kOutBufs > 0 ? Cfg::kOutBufs - 1 : 0)>();
      __syncwarp();
      const uint32_t sbuf = stg + (uint32_t)buf * kOutTile;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        st_shared_v4(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4), pack_bf16x2(v[8 * j + 0], v[8 * j + 1]),
                     pack_bf16x2(v[8 * j + 2], v[8 * j + 3]), pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                     pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(m, sbuf, col, row);
        bulk_commit();
      }
      if (++buf == Cfg::kOutBufs) buf = 0;
    };
    // The same for 32 rows x 32 columns through 2 KB tiles with the 64-byte
    // swizzle (16-byte chunk j of row r at r * 64 + ((j ^ ((r >> 1) & 3)) << 4)),
    // four of them rotating in this warp's staging space.
    int buf32 = 0;
    auto put_tile32 = [&](const CUtensorMap* m, const float* v, int col, int row) {
      if (lane == 0) bulk_wait_read<(Cfg::kOutBufs > 0 ? 2 * Cfg::kOutBufs - 1 : 0)>();
      __syncwarp();
      const uint32_t sbuf = stg + (uint32_t)buf32 * (kOutTile / 2);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        st_shared_v4(sbuf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), pack_bf16x2(v[8 * j + 0], v[8 * j + 1]),
                     pack_bf16x2(v[8 * j + 2], v[8 * j + 3]), pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                     pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(m, sbuf, col, row);
        bulk_commit();
      }
      if (++buf32 == 2 * Cfg::kOutBufs) buf32 = 0;
    };
    for (int j = 0;; ++j) {
      bool ok;
      const int U = unit_of(j, ok);
      if (!ok || U < 0) break;
      if (CLC && U >= total) continue;
      const Tile t = decode<WGRAD, PAIR, UM>(p, U, rank);
      if (!mbar_wait(&tfull[acc], aph, abort_flag, p.status, 400 + acc)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (uint32_t)acc * kAccStride + ((uint32_t)(q * 32) << 16);
      const bool zero = (t.kb_count == 0);

      if (!t.valid) {
        // pair mode: the odd CTA's rows past the expert's last tile
      } else if (EPI == EPI_STORE && PAIR && !WGRAD && t.thin) {
        // thin pair unit: lane = output column, TMEM columns = tokens; rows
        // [row0, row0 + nt) are written (zeros past the expert's rows)
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint8_t* tr = staging + (size_t)(warp - 2) * Cfg::kOutBufs * kOutTile;
        const int c0 = t.n * 256 + rank * 128 + q * 32;
        if (c0 < p.out_cols) {
          for (int t0 = 0; t0 < t.nt; t0 += 32) {
            float v[32];
            tmem_ld32(tb + t0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = (t0 + i < t.rows) ? v[i] : 0.f;
            store_cols_t(tr, v, p.out0 + ((size_t)t.row0 + t0) * p.out_cols + c0, p.out_cols, 32, lane);
          }
        }
      } else if constexpr (EPI == EPI_STORE) {
        const int row = (WGRAD ? t.m * kBM : t.row0) + q * 32;
        for (int c = 0; c < p.umma_n / 64; ++c) {
          float v[64];
          if (!zero) {
            tmem_ld32(tb + c * 64, v);
            tmem_ld32(tb + c * 64 + 32, v + 32);
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = 0.f;
          }
          const int col = t.n * 256 + c * 64;
          if (col >= p.out_cols || (WGRAD && row >= p.out_rows)) continue;
          if (!WGRAD) {
            put_tile(&tmO, v, col, row);
            continue;
          }
          if (lane == 0) bulk_wait_read<Cfg::kOutBufs - 1>();
          __syncwarp();
          const uint32_t sbuf = stg + (uint32_t)buf * kOutTile;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            st_shared_v4(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4),
                         pack_bf16x2(v[8 * j + 0], v[8 * j + 1]),
                         pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                         pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                         pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmO, sbuf, col, row, t.e);
            bulk_commit();
          }
          if (++buf == Cfg::kOutBufs) buf = 0;
        }
      } else if (EPI == EPI_SWIGLU && !FP8 && !PAIR && t.thin) {
        // thin tile: lane = gate / up column, TMEM columns = tokens.  All 128
        // rows are written (zeros past the expert's rows) so that the saved
        // activations of the padding rows stay zero.
        // the transpose tile reuses this warp's staging tiles once the TMA
        // stores reading them are done
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint8_t* tr = staging + (size_t)(warp - 2) * Cfg::kOutBufs * kOutTile;
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
          const size_t r0 = (size_t)t.row0 + t0;
          store_cols_t(tr, a, p.out0 + r0 * p.f + c0, p.f, 32, lane);
          if (p.out1 != nullptr) {
            store_cols_t(tr, g, p.out1 + r0 * (2 * p.f) + c0, 2 * p.f, 32, lane);
            store_cols_t(tr, u, p.out1 + r0 * (2 * p.f) + p.f + c0, 2 * p.f, 32, lane);
          }
        }
      } else if (EPI == EPI_SWIGLU && !FP8 && PAIR && t.thin) {
        // thin pair unit: TMEM lane = weight column (gate in lane quarters 0-1,
        // up in 2-3, the same 64 columns), TMEM column = token.  Each up warp
        // hands its values to the gate warp of the same columns through
        // shared memory.  All 128 rows are written (zeros past the expert's
        // rows) so that the saved activations of the padding rows stay zero.
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        const bool is_gate = q < 2;
        uint8_t* tr = Cfg::kLightSwiglu ? staging + 2 * 4096 + (size_t)(warp - 2) * kTrTile
                                        : staging + (size_t)(warp - 2) * Cfg::kOutBufs * kOutTile + 4096;
        float* xb = reinterpret_cast<float*>(
            staging + (size_t)(is_gate ? q : q - 2) * (Cfg::kLightSwiglu ? 4096 : Cfg::kOutBufs * kOutTile));
        const int c0 = t.n * p.hn + rank * 64 + (q & 1) * 32;
        for (int t0 = 0; t0 < kBM; t0 += 32) {
          float v[32];
          if (t0 < t.nt) {
            tmem_ld32(tb + t0, v);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = (t0 + i < t.rows) ? v[i] : 0.f;
          const size_t r0 = (size_t)t.row0 + t0;
          if (!is_gate) {
#pragma unroll
            for (int i = 0; i < 32; ++i) xb[i * 32 + lane] = v[i];
            if (p.out1 != nullptr) store_cols_t(tr, v, p.out1 + r0 * (2 * p.f) + p.f + c0, 2 * p.f, 32, lane);
          }
          named_bar_sync(1, kEpiWarps * 32);
          if (is_gate) {
            float a[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = silu_f(v[i]) * xb[i * 32 + lane];
            store_cols_t(tr, a, p.out0 + r0 * p.f + c0, p.f, 32, lane);
            if (p.out1 != nullptr) store_cols_t(tr, v, p.out1 + r0 * (2 * p.f) + c0, 2 * p.f, 32, lane);
          }
          named_bar_sync(1, kEpiWarps * 32);
        }
      } else if constexpr (EPI == EPI_SWIGLU && !FP8) {
        // 64 gate and 64 up columns at a time: H (gate, up) and A = SiLU(gate) * up
        // leave through TMA stores of 32-row x 64-column tiles
        const int row = t.row0 + q * 32;
        for (int c = 0; c < p.hn; c += 64) {
          float g[64], u[64];
          tmem_ld32(tb + c, g);
          tmem_ld32(tb + c + 32, g + 32);
          tmem_ld32(tb + p.hn + c, u);
          tmem_ld32(tb + p.hn + c + 32, u + 32);
          const int col = t.n * p.hn + c;
          if (q * 32 + lane >= t.rows) {
            // a padding row of the expert's last tile (its input row is not
            // written by the gather): saved and passed on as zeros
#pragma unroll
            for (int i = 0; i < 64; ++i) g[i] = u[i] = 0.f;
          }
          if (p.out1 != nullptr) {
            put_tile(&tmO2, g, col, row);
            put_tile(&tmO2, u, p.f + col, row);
          }
#pragma unroll
          for (int i = 0; i < 64; ++i) g[i] = silu_f(g[i]) * u[i];
          put_tile(&tmO, g, col, row);
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        const size_t row = (size_t)t.row0 + q * 32 + lane;
        // a padding row of the expert's last tile (its input row is not
        // written by the gather): saved and passed on as zeros
        const bool pad_row = q * 32 + lane >= t.rows;
        for (int c = 0; c < p.hn; c += 32) {
          float g[32], u[32], a[32];
          tmem_ld32(tb + c, g);
          tmem_ld32(tb + p.hn + c, u);
          if (pad_row) {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = u[i] = 0.f;
          }
          const int col = t.n * p.hn + c;
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = silu_f(g[i]) * u[i];
          if constexpr (FP8) {
            // quantise A for the fp8 GEMM2: this thread's 32 columns are one block
            uint4 lo, hi;
            const uint8_t sc = mx_quant32(a, lo, hi);
            uint4* qd = reinterpret_cast<uint4*>(p.q_out + row * p.f + col);
            qd[0] = lo;
            qd[1] = hi;
            p.q_sf[mx_sf_offset(row, col >> 5, p.f >> 7)] = sc;
          }
          if (p.out0 != nullptr) store32_bf16(p.out0 + row * p.f + col, a);
          if (p.out1 != nullptr) {
            store32_bf16(p.out1 + row * (2 * p.f) + col, g);
            store32_bf16(p.out1 + row * (2 * p.f) + p.f + col, u);
          }
        }
      } else if constexpr (EPI == EPI_LOGITS) {
        // router: this thread's row of fp32 logits for experts [n*256, n*256+256)
        const int r = t.row0 + q * 32 + lane;
        if (p.logits != nullptr) {
          for (int c = 0; c < p.umma_n; c += 32) {
            float v[32];
            tmem_ld32(tb + c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int e = t.n * 256 + c + i;
              if (r < p.T && e < p.E) p.logits[(size_t)r * p.E + e] = v[i];
            }
          }
        }
        if (p.topk_ids != nullptr) {
          // one N tile holds the whole row: its top-k in k rounds, round j
          // taking the best (value descending, id ascending) strictly after
          // round j-1's pick; weights exp(z_j - z_0) summed in slot order and
          // divided by the sum -- the same fp32 steps as sched_topk
          float pv = INFINITY, z0 = 0.f, ssum = 0.f;
          int pi = -1;
          for (int j = 0; j < p.k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int c = 0; c < p.umma_n; c += 32) {
              float v[32];
              tmem_ld32(tb + c, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int e = c + i;
                const bool after = v[i] < pv || (v[i] == pv && e > pi);
                if (e < p.E && after && (v[i] > bv || (v[i] == bv && e < bi))) {
                  bv = v[i];
                  bi = e;
                }
              }
            }
            if (j == 0) z0 = bv;
            const float ex = expf(bv - z0);
            ssum += ex;
            if (r < p.T) {
              p.topk_ids[(size_t)r * p.k + j] = bi;
              p.topk_w[(size_t)r * p.k + j] = ex;
            }
            pv = bv;
            pi = bi;
          }
          if (r < p.T)
            for (int j = 0; j < p.k; ++j) p.topk_w[(size_t)r * p.k + j] /= ssum;
        }
      } else if constexpr (EPI == EPI_DSWIGLU && FP8) {
        // MXFP8 SwiGLU backward: acc = dA' for f columns [n*256, n*256+256).
        // dH is quantised along 2f for dgrad1 (this lane's 32 gate and 32 up
        // values are one block each), and dH and g*A along the rows for the
        // weight gradients (the warp's 32 lanes are one 32-row block of every
        // column), written transposed.
        const size_t row = (size_t)t.row0 + q * 32 + lane;
        const int rblk = (t.row0 + q * 32) >> 5;
        const int kq = (2 * p.f) >> 7, kt = p.ldt >> 7;
        const float gw = p.g_pad[row];
        float dg = 0.f;
        // fragments of A, H_gate, H_up for the next 32 columns are loaded while
        // the current ones are processed
        uint4 nxt[12];
        auto fetch = [&](int col) {
          const uint4* a = reinterpret_cast<const uint4*>(p.As + row * p.f + col);
          const uint4* g = reinterpret_cast<const uint4*>(p.Hs + row * (2 * p.f) + col);
          const uint4* u = reinterpret_cast<const uint4*>(p.Hs + row * (2 * p.f) + p.f + col);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            nxt[i] = __ldg(a + i);
            nxt[4 + i] = __ldg(g + i);
            nxt[8 + i] = __ldg(u + i);
          }
        };
        if (t.n * 256 < p.f) fetch(t.n * 256);
        for (int c = 0; c < 256; c += 32) {
          const int col = t.n * 256 + c;
          if (col >= p.f) break;
          float da[32], av[32], hg[32], hu[32], o1[32], o2[32], o3[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            unpack8(nxt[i], av + 8 * i);
            unpack8(nxt[4 + i], hg + 8 * i);
            unpack8(nxt[8 + i], hu + 8 * i);
          }
          if (c + 32 < 256 && col + 32 < p.f) fetch(col + 32);
          tmem_ld32(tb + c, da);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            dg = fmaf(da[i], av[i], dg);
            const float dA = gw * da[i];
            const float sg = sigmoid_f(hg[i]);
            o1[i] = dA * hu[i] * sg * (1.0f + hg[i] * (1.0f - sg));  // d gate
            o2[i] = dA * hg[i] * sg;                                // d up
            o3[i] = gw * av[i];                                     // g * A (for dW2)
          }
          uint4 lo, hi;
          uint8_t sc = mx_quant32(o1, lo, hi);
          uint4* qd = reinterpret_cast<uint4*>(p.q_out + row * (2 * p.f) + col);
          qd[0] = lo;
          qd[1] = hi;
          p.q_sf[mx_sf_offset(row, col >> 5, kq)] = sc;
          sc = mx_quant32(o2, lo, hi);
          qd = reinterpret_cast<uint4*>(p.q_out + row * (2 * p.f) + p.f + col);
          qd[0] = lo;
          qd[1] = hi;
          p.q_sf[mx_sf_offset(row, (p.f + col) >> 5, kq)] = sc;
          // column i's scale bytes (the same in every lane) are kept by lane
          // i, which stores them after the loop
          uint8_t m1 = 0, m2 = 0, m3 = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            uint8_t s1, s2, s3;
            const uint8_t c1 = mx_quant_lane(o1[i], &s1);
            const uint8_t c2 = mx_quant_lane(o2[i], &s2);
            const uint8_t c3 = mx_quant_lane(o3[i], &s3);
            p.qt0[(size_t)(col + i) * p.ldt + row] = c1;
            p.qt0[(size_t)(p.f + col + i) * p.ldt + row] = c2;
            p.qt1[(size_t)(col + i) * p.ldt + row] = c3;
            if (lane == i) {
              m1 = s1;
              m2 = s2;
              m3 = s3;
            }
          }
          p.qt0_sf[mx_sf_offset((size_t)(col + lane), rblk, kt)] = m1;
          p.qt0_sf[mx_sf_offset((size_t)(p.f + col + lane), rblk, kt)] = m2;
          p.qt1_sf[mx_sf_offset((size_t)(col + lane), rblk, kt)] = m3;
        }
        p.dgp[row * p.n_tiles + t.n] = dg;
      } else {
        // EPI_DSWIGLU: acc = dA' = dOut_p W2^T for f columns [n*256, n*256+256);
        // dH (gate, up) and g*A leave through TMA stores of 32 x 32 tiles
        const size_t row = (size_t)t.row0 + q * 32 + lane;
        const int wrow = t.row0 + q * 32;
        const float gw = p.g_pad[row];
        float dg = 0.f;
        // fragments of A, H_gate, H_up for the next 32 columns are loaded while
        // the current ones are processed
        uint4 nxt[12];
        auto fetch = [&](int col) {
          const uint4* a = reinterpret_cast<const uint4*>(p.As + row * p.f + col);
          const uint4* g = reinterpret_cast<const uint4*>(p.Hs + row * (2 * p.f) + col);
          const uint4* u = reinterpret_cast<const uint4*>(p.Hs + row * (2 * p.f) + p.f + col);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            nxt[i] = __ldg(a + i);
            nxt[4 + i] = __ldg(g + i);
            nxt[8 + i] = __ldg(u + i);
          }
        };
        if (t.n * 256 < p.f) fetch(t.n * 256);
        for (int c = 0; c < 256; c += 32) {
          const int col = t.n * 256 + c;
          if (col >= p.f) break;
          float da[32], av[32], hg[32], hu[32], o1[32], o2[32], o3[32];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            unpack8(nxt[i], av + 8 * i);
            unpack8(nxt[4 + i], hg + 8 * i);
            unpack8(nxt[8 + i], hu + 8 * i);
          }
          if (c + 32 < 256 && col + 32 < p.f) fetch(col + 32);
          tmem_ld32(tb + c, da);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            dg = fmaf(da[i], av[i], dg);
            const float dA = gw * da[i];
            const float sg = sigmoid_f(hg[i]);
            o1[i] = dA * hu[i] * sg * (1.0f + hg[i] * (1.0f - sg));  // d gate
            o2[i] = dA * hg[i] * sg;                                // d up
            o3[i] = gw * av[i];                                     // g * A (for dW2)
          }
          put_tile32(&tmO, o1, col, wrow);
          put_tile32(&tmO, o2, p.f + col, wrow);
          put_tile32(&tmO2, o3, col, wrow);
        }
        p.dgp[row * p.n_tiles + t.n] = dg;
      }
      tc_fence_before();
      if constexpr (PAIR) {
        // one arrival per warp on the even CTA's barrier
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[acc]), 0));
      } else {
        mbar_arrive(&tempty[acc]);
      }
      if (++acc == kAcc) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if (Cfg::kOutBufs > 0 && lane == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the pair's MMAs and remote arrivals are done
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, kTmemAlloc);
    else tmem_dealloc(tmem_base, kTmemAlloc);
  }
  // split units: the light kernel ends after the heavy one it runs beside,
  // so the next kernel in the stream sees both finished
  if constexpr (UM == UNITS_LIGHT) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ host side
template <bool WGRAD, bool A_MN, bool B_MN, int EPI, bool FP8 = false, bool PAIR = false, int UM = UNITS_ALL,
          bool CLC = false>
cudaError_t launch(const char* name, const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                   const CUtensorMap& o, const CUtensorMap& o2, const Params& p, long long max_units,
                   cudaStream_t st) {
  auto kern = grouped_gemm_kernel<WGRAD, A_MN, B_MN, EPI, FP8, PAIR, UM, CLC>;
  const size_t smem = KCfg<EPI, FP8, WGRAD, PAIR, UM>::kSmem;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if constexpr (CLC) {
    // one CTA per unit; the running CTAs cancel the launches of the others
    if (max_units < 1 || max_units > 0x7fffffffLL) return cudaErrorInvalidValue;
    TraceScope ts(name, st);
    kern<<<(unsigned)max_units, kThreads, smem, st>>>(a, a2, b, o, o2, p);
    return cudaGetLastError();
  } else if constexpr (!PAIR) {
    long long grid = num_sms();
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    TraceScope ts(name, st);
    kern<<<(int)grid, kThreads, smem, st>>>(a, a2, b, o, o2, p);
    return cudaGetLastError();
  } else {
    // persistent clusters of two CTAs: as many as can be resident at once
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms() & ~1));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (UM == UNITS_LIGHT) {
      // beside the heavy kernel queued just before it: one CTA per SM, started
      // as soon as every heavy CTA is resident (programmatic dependent launch)
      cudaLaunchAttribute attr2[2] = {attr[0], {}};
      attr2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr2[1].val.programmaticStreamSerializationAllowed = 1;
      long long clusters = num_sms() / 2;
      if (max_units < clusters) clusters = max_units;
      if (clusters < 1) clusters = 1;
      cfg.gridDim = dim3((unsigned)(2 * clusters));
      cfg.attrs = attr2;
      cfg.numAttrs = 2;
      TraceScope ts(name, st);
      return cudaLaunchKernelEx(&cfg, kern, a, a2, b, o, o2, p);
    }
    static int resident[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    if (resident[dev] == 0) {
      int n = 0;
      err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (err != cudaSuccess) return err;
      if (n < 1) return cudaErrorInvalidConfiguration;
      resident[dev] = n;
    }
    long long clusters = resident[dev];
    if (max_units < clusters) clusters = max_units;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    TraceScope ts(name, st);
    return cudaLaunchKernelEx(&cfg, kern, a, a2, b, o, o2, p);
  }
}

Params base_params(const moe_config& c, const Ws& ws) {
  Params p{};
  p.E = c.E;
  p.f = c.f;
  p.kstep = BK;
  p.mt_off = ws.mt_off();
  p.pt_off = ws.pt_off();
  p.hv_off = ws.hv_off();
  p.lt_off = ws.lt_off();
  p.poff = ws.poff();
  p.status = ws.hdr() + kHdrStatus;
  return p;
}

}  // namespace

cudaError_t gemm_fwd1(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* Xp,
                      const __nv_bfloat16* W1, __nv_bfloat16* A, __nv_bfloat16* H, cudaStream_t st,
                      const char* name) {
  CUtensorMap ta, tb, to;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.hn = (c.f % 128 == 0) ? 128 : 64;
  p.umma_n = 2 * p.hn;
  p.n_tiles = c.f / p.hn;
  p.num_kb = c.d / BK;
  p.out_cols = c.f;
  p.out0 = A;
  p.out1 = H;
  p.counts = counts;
  const bool pair = gemm_pair_enabled(c, kGemmFwd1);
  // one CTA: partial last tiles swapped when gemm1_thin_enabled; pairs: an
  // expert's unpartnered last tile as a thin pair unit (128-column slices)
  p.thin = (pair ? p.hn == 128 : gemm1_thin_enabled(c)) ? 1 : 0;
  // outputs: A [rows, f] and (when saved) H [rows, 2f], stored as 32 x 64 tiles
  CUtensorMap th, ta16;
  if (!map2d(&ta, Xp, c.d, rows, 64, kBM) || !map2d(&ta16, Xp, c.d, rows, 64, 16) ||
      !map3d(&tb, W1, 2ull * c.f, c.d, c.E, 64, 64) ||
      !map2d(&to, A, c.f, rows, 64, 32) || (H != nullptr && !map2d(&th, H, 2ull * c.f, rows, 64, 32)))
    return cudaErrorInvalidValue;
  if (H == nullptr) th = to;
  static_assert(KCfg<EPI_SWIGLU, false, false, true, UNITS_HEAVY>::kSmem +
                    KCfg<EPI_SWIGLU, false, false, true, UNITS_LIGHT>::kSmem + 2048 <= 233472,
                "heavy and light GEMM1 CTAs share an SM");
  if (pair && p.thin && gemm_split_units(c)) {
    const cudaError_t e = launch<false, false, true, EPI_SWIGLU, false, true, UNITS_HEAVY>(
        name, ta, ta16, tb, to, th, p, ws.L.MT_max * p.n_tiles, st);
    if (e != cudaSuccess) return e;
    return launch<false, false, true, EPI_SWIGLU, false, true, UNITS_LIGHT>(
        "gemm1_light", ta, ta16, tb, to, th, p, (long long)c.E * p.n_tiles, st);
  }
  if (pair)
    return launch<false, false, true, EPI_SWIGLU, false, true>(name, ta, ta16, tb, to, th, p,
                                                               ws.L.MT_max * p.n_tiles, st);
  return launch<false, false, true, EPI_SWIGLU>(name, ta, ta, tb, to, th, p, ws.L.MT_max * p.n_tiles, st);
}

cudaError_t gemm_fwd2(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* A,
                      const __nv_bfloat16* W2, __nv_bfloat16* Yp, cudaStream_t st) {
  CUtensorMap ta, ta16, tb, to;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.umma_n = 256;
  p.n_tiles = (c.d + 255) / 256;
  p.num_kb = c.f / BK;
  p.out_cols = c.d;
  p.out0 = Yp;
  p.counts = counts;
  const bool pair = gemm_pair_enabled(c, kGemmFwd2);
  p.thin = pair ? 1 : 0;  // an expert's unpartnered last tile as a thin pair unit
  if (!map2d(&ta, A, c.f, rows, 64, kBM) || !map2d(&ta16, A, c.f, rows, 64, 16) ||
      !map3d(&tb, W2, c.d, c.f, c.E, 64, 64) || !map2d(&to, Yp, c.d, rows, 64, 32))
    return cudaErrorInvalidValue;
  static_assert(KCfg<EPI_STORE, false, false, true, UNITS_HEAVY>::kSmem +
                    KCfg<EPI_STORE, false, false, true, UNITS_LIGHT>::kSmem + 2048 <= 233472,
                "heavy and light GEMM2 CTAs share an SM");
  if (pair && p.thin && gemm_split_units(c)) {
    const cudaError_t e = launch<false, false, true, EPI_STORE, false, true, UNITS_HEAVY>(
        "gemm2", ta, ta16, tb, to, to, p, ws.L.MT_max * p.n_tiles, st);
    if (e != cudaSuccess) return e;
    return launch<false, false, true, EPI_STORE, false, true, UNITS_LIGHT>(
        "gemm2_light", ta, ta16, tb, to, to, p, (long long)c.E * p.n_tiles, st);
  }
  if (pair)
    return launch<false, false, true, EPI_STORE, false, true>("gemm2", ta, ta16, tb, to, to, p,
                                                              ws.L.MT_max * p.n_tiles, st);
  return launch<false, false, true, EPI_STORE>("gemm2", ta, ta, tb, to, to, p, ws.L.MT_max * p.n_tiles, st);
}

cudaError_t gemm_dgrad2(const moe_config& c, const Ws& ws, const __nv_bfloat16* dYp,
                        const __nv_bfloat16* W2, const __nv_bfloat16* Hs, const __nv_bfloat16* As,
                        __nv_bfloat16* dH, __nv_bfloat16* gA, float* dgp, cudaStream_t st) {
  CUtensorMap ta, tb, to;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.umma_n = 256;
  p.n_tiles = (int)ws.L.nt_dg;
  p.num_kb = c.d / BK;
  p.out_cols = c.f;
  p.out0 = dH;
  p.out1 = gA;
  p.Hs = Hs;
  p.As = As;
  p.g_pad = ws.g_pad();
  p.dgp = dgp;
  // B = W2[e]^T: K = d contiguous, N = f rows -> K-major box of 256 rows (pair: 128 a CTA)
  const bool pair = gemm_pair_enabled(c, kGemmDgrad2);
  // outputs dH [rows, 2f] and g*A [rows, f] as 32 x 32 tiles (64-byte swizzle)
  CUtensorMap tg;
  if (!map2d(&ta, dYp, c.d, rows, 64, kBM) || !map3d(&tb, W2, c.d, c.f, c.E, 64, pair ? 128 : 256) ||
      !map2d(&to, dH, 2ull * c.f, rows, 32, 32, false, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !map2d(&tg, gA, c.f, rows, 32, 32, false, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (pair)
    return launch<false, false, false, EPI_DSWIGLU, false, true>("dgrad2_dswiglu", ta, ta, tb, to, tg, p,
                                                                 ws.L.MT_max * p.n_tiles, st);
  return launch<false, false, false, EPI_DSWIGLU>("dgrad2_dswiglu", ta, ta, tb, to, tg, p,
                                                 ws.L.MT_max * p.n_tiles, st);
}

cudaError_t gemm_dgrad1(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* dH,
                        const __nv_bfloat16* W1, __nv_bfloat16* dXp, cudaStream_t st) {
  CUtensorMap ta, ta16, tb, to;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.umma_n = 256;
  p.n_tiles = (c.d + 255) / 256;
  p.num_kb = 2 * c.f / BK;
  p.out_cols = c.d;
  p.out0 = dXp;
  p.counts = counts;
  // B = W1[e]^T: K = 2f contiguous, N = d rows (box of 256 rows; pair: 128 a CTA)
  const bool pair = gemm_pair_enabled(c, kGemmDgrad1);
  p.thin = pair ? 1 : 0;  // an expert's unpartnered last tile as a thin pair unit
  if (!map2d(&ta, dH, 2ull * c.f, rows, 64, kBM) || !map2d(&ta16, dH, 2ull * c.f, rows, 64, 16) ||
      !map3d(&tb, W1, 2ull * c.f, c.d, c.E, 64, pair ? 128 : 256) || !map2d(&to, dXp, c.d, rows, 64, 32))
    return cudaErrorInvalidValue;
  if (pair)
    return launch<false, false, false, EPI_STORE, false, true>("dgrad1", ta, ta16, tb, to, to, p,
                                                               ws.L.MT_max * p.n_tiles, st);
  return launch<false, false, false, EPI_STORE>("dgrad1", ta, ta, tb, to, to, p, ws.L.MT_max * p.n_tiles, st);
}

cudaError_t gemm_wgrad(const moe_config& c, const Ws& ws, const moe_sched& s,
                       const __nv_bfloat16* Amn, int M, const __nv_bfloat16* Bmn, int N,
                       __nv_bfloat16* dW, cudaStream_t st) {
  CUtensorMap ta, tb, to;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.umma_n = 256;
  p.m_tiles_w = (M + kBM - 1) / kBM;
  p.n_tiles = (N + 255) / 256;
  p.out_cols = N;
  p.out_rows = M;
  p.counts = s.counts;
  if (!map2d(&ta, Amn, M, rows, 64, 64) || !map2d(&tb, Bmn, N, rows, 64, 64) ||
      !map3d(&to, dW, N, M, c.E, 64, 32))
    return cudaErrorInvalidValue;
  const char* name = M == c.f ? "wgrad2" : "wgrad1";
  if (gemm_pair_enabled(c, kGemmWgrad))
    return launch<true, true, true, EPI_STORE, false, true>(
        name, ta, ta, tb, to, to, p, (long long)c.E * ((p.m_tiles_w + 1) / 2) * p.n_tiles, st);
  if (gemm_clc_enabled(c))
    return launch<true, true, true, EPI_STORE, false, false, UNITS_ALL, true>(
        name, ta, ta, tb, to, to, p, (long long)c.E * p.m_tiles_w * p.n_tiles, st);
  return launch<true, true, true, EPI_STORE>(name, ta, ta, tb, to, to, p,
                                             (long long)c.E * p.m_tiles_w * p.n_tiles, st);
}

// Router logits [T, E] = x [T, d] . Wr [E, d]^T (fp32 accumulation), one CTA
// per 128 x 256 tile; with E <= 256 and topk_ids given the epilogue also takes
// each row's top-k and weights.
cudaError_t router_gemm(const moe_config& c, const Ws& ws, const __nv_bfloat16* x,
                        const __nv_bfloat16* Wr, float* logits, int* topk_ids, float* topk_w,
                        cudaStream_t st) {
  CUtensorMap ta, tb;
  Params p = base_params(c, ws);
  p.mt_off = nullptr;
  p.T = c.T;
  p.dense_mt = (c.T + kBM - 1) / kBM;
  p.n_tiles = (c.E + 255) / 256;
  p.umma_n = p.n_tiles > 1 ? 256 : (c.E + 15) / 16 * 16;
  p.num_kb = c.d / BK;
  p.logits = logits;
  p.topk_ids = p.n_tiles == 1 ? topk_ids : nullptr;
  p.topk_w = topk_w;
  p.k = c.k;
  if (!map2d(&ta, x, c.d, (uint64_t)c.T, 64, kBM) || !map3d(&tb, Wr, c.d, c.E, 1, 64, 256))
    return cudaErrorInvalidValue;
  return launch<false, false, false, EPI_LOGITS>("router_logits", ta, ta, tb, ta, ta, p,
                                                 (long long)p.dense_mt * p.n_tiles, st);
}

// Router backward: dx_r [T, d] = dlogits [T, Epad] . Wr [E, d] and
// dWr [E, d] = dlogits^T . x; dlogits in bf16 with Epad (E rounded up to 64)
// columns, zero past E.
cudaError_t router_bwd(const moe_config& c, const Ws& ws, const __nv_bfloat16* dl16, int Epad,
                       const __nv_bfloat16* x, const __nv_bfloat16* Wr, __nv_bfloat16* dx_r,
                       __nv_bfloat16* dWr, cudaStream_t st) {
  CUtensorMap ta, tb, to;
  {
    Params p = base_params(c, ws);
    p.mt_off = nullptr;
    p.T = c.T;
    p.dense_mt = (c.T + kBM - 1) / kBM;
    p.umma_n = 256;
    p.n_tiles = (c.d + 255) / 256;
    p.num_kb = Epad / BK;
    p.out_cols = c.d;
    if (!map2d(&ta, dl16, (uint64_t)Epad, (uint64_t)c.T, 64, kBM) ||
        !map3d(&tb, Wr, c.d, c.E, 1, 64, 64) || !map2d(&to, dx_r, c.d, (uint64_t)c.T, 64, 32))
      return cudaErrorInvalidValue;
    const cudaError_t e = launch<false, false, true, EPI_STORE>("router_dx", ta, ta, tb, to, to, p,
                                                                (long long)p.dense_mt * p.n_tiles, st);
    if (e != cudaSuccess) return e;
  }
  Params p = base_params(c, ws);
  p.E = 1;
  p.counts = nullptr;
  p.dense_k = c.T;
  p.umma_n = 256;
  p.m_tiles_w = (c.E + kBM - 1) / kBM;
  p.n_tiles = (c.d + 255) / 256;
  p.out_cols = c.d;
  p.out_rows = c.E;
  if (!map2d(&ta, dl16, (uint64_t)Epad, (uint64_t)c.T, 64, 64) || !map2d(&tb, x, c.d, (uint64_t)c.T, 64, 64) ||
      !map3d(&to, dWr, c.d, c.E, 1, 64, 32))
    return cudaErrorInvalidValue;
  return launch<true, true, true, EPI_STORE>("router_dw", ta, ta, tb, to, to, p,
                                             (long long)p.m_tiles_w * p.n_tiles, st);
}

// MXFP8 GEMM1: Xq [rows, d] E4M3 (+ scale tiles) x W1q [E, 2f, d] E4M3 (+ scale
// tiles) -> SwiGLU -> Aq [rows, f] E4M3 + scale tiles; optionally A and H in bf16.
cudaError_t gemm_fwd1_mx(const moe_config& c, const Ws& ws, const int* counts, const uint8_t* Xq,
                         const uint8_t* Xs, const uint8_t* W1q, const uint8_t* W1s, uint8_t* Aq,
                         uint8_t* As, __nv_bfloat16* A, __nv_bfloat16* H, cudaStream_t st) {
  CUtensorMap ta, tb, to;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.counts = counts;  // the rows of each tile: padding rows leave as zeros
  p.hn = 128;
  p.umma_n = 256;
  p.n_tiles = c.f / 128;
  p.num_kb = c.d / BK8;
  p.out_cols = c.f;
  p.out0 = A;
  p.out1 = H;
  p.sfa = Xs;
  p.sfb = W1s;
  p.k_groups = c.d / 128;
  p.b_rows = 2 * c.f;
  p.q_out = Aq;
  p.q_sf = As;
  if (!map2d(&ta, Xq, c.d, rows, 128, kBM, true) ||
      !map3d(&tb, W1q, c.d, 2ull * c.f, c.E, 128, 128, true))
    return cudaErrorInvalidValue;
  to = tb;
  return launch<false, false, false, EPI_SWIGLU, true>("gemm1_swiglu_mxfp8", ta, ta, tb, to, to, p,
                                                       ws.L.MT_max * p.n_tiles, st);
}

// MXFP8 GEMM2: Aq [rows, f] x W2q [E, d, f] -> Y [rows, d] bf16.
cudaError_t gemm_fwd2_mx(const moe_config& c, const Ws& ws, const uint8_t* Aq, const uint8_t* As,
                         const uint8_t* W2q, const uint8_t* W2s, __nv_bfloat16* Yp,
                         cudaStream_t st) {
  CUtensorMap ta, tb, to;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.umma_n = 256;
  p.n_tiles = (c.d + 255) / 256;
  p.num_kb = c.f / BK8;
  p.out_cols = c.d;
  p.sfa = As;
  p.sfb = W2s;
  p.k_groups = c.f / 128;
  p.b_rows = c.d;
  if (!map2d(&ta, Aq, c.f, rows, 128, kBM, true) ||
      !map3d(&tb, W2q, c.f, c.d, c.E, 128, 256, true) || !map2d(&to, Yp, c.d, rows, 64, 32))
    return cudaErrorInvalidValue;
  return launch<false, false, false, EPI_STORE, true>("gemm2_mxfp8", ta, ta, tb, to, to, p,
                                                      ws.L.MT_max * p.n_tiles, st);
}

// ---------------------------------------------------------------- MXFP8 backward
// dgrad2: dYq [rows, d] E4M3 (blocks along d) x W2 quantised along d
// (W2q [E, f, d], its scale tiles over [E*f, d]) -> SwiGLU backward with the
// routing-weight gradient; dH quantised along 2f (dHq, dHs), dH and g*A
// quantised along the rows and written transposed (dHqT [2f, ldt], gAqT
// [f, ldt], ldt = the padded row capacity), dg partials.
cudaError_t gemm_dgrad2_mx(const moe_config& c, const Ws& ws, const uint8_t* dYq, const uint8_t* dYs,
                           const uint8_t* W2q, const uint8_t* W2s, const __nv_bfloat16* Hs,
                           const __nv_bfloat16* As, uint8_t* dHq, uint8_t* dHs, uint8_t* dHqT,
                           uint8_t* dHsT, uint8_t* gAqT, uint8_t* gAsT, float* dgp, cudaStream_t st) {
  CUtensorMap ta, tb;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.umma_n = 256;
  p.n_tiles = (int)ws.L.nt_dg;
  p.num_kb = c.d / BK8;
  p.out_cols = c.f;
  p.Hs = Hs;
  p.As = As;
  p.g_pad = ws.g_pad();
  p.dgp = dgp;
  p.sfa = dYs;
  p.sfb = W2s;
  p.k_groups = c.d / 128;
  p.b_rows = c.f;
  p.q_out = dHq;
  p.q_sf = dHs;
  p.qt0 = dHqT;
  p.qt0_sf = dHsT;
  p.qt1 = gAqT;
  p.qt1_sf = gAsT;
  p.ldt = (int)ws.L.Rp_max;
  if (!map2d(&ta, dYq, c.d, rows, 128, kBM, true) || !map3d(&tb, W2q, c.d, c.f, c.E, 128, 256, true))
    return cudaErrorInvalidValue;
  return launch<false, false, false, EPI_DSWIGLU, true>("dgrad2_dswiglu_mxfp8", ta, ta, tb, ta, ta, p,
                                                        ws.L.MT_max * p.n_tiles, st);
}

// dgrad1: dHq [rows, 2f] (blocks along 2f) x W1 quantised along 2f (W1q
// [E, d, 2f], scale tiles over [E*d, 2f]) -> dX [rows, d] bf16 in expert order.
cudaError_t gemm_dgrad1_mx(const moe_config& c, const Ws& ws, const uint8_t* dHq, const uint8_t* dHs,
                           const uint8_t* W1q, const uint8_t* W1s, __nv_bfloat16* dXp, cudaStream_t st) {
  CUtensorMap ta, tb, to;
  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.umma_n = 256;
  p.n_tiles = (c.d + 255) / 256;
  p.num_kb = 2 * c.f / BK8;
  p.out_cols = c.d;
  p.sfa = dHs;
  p.sfb = W1s;
  p.k_groups = 2 * c.f / 128;
  p.b_rows = c.d;
  if (!map2d(&ta, dHq, 2ull * c.f, rows, 128, kBM, true) ||
      !map3d(&tb, W1q, 2ull * c.f, c.d, c.E, 128, 256, true) || !map2d(&to, dXp, c.d, rows, 64, 32))
    return cudaErrorInvalidValue;
  return launch<false, false, false, EPI_STORE, true>("dgrad1_mxfp8", ta, ta, tb, to, to, p,
                                                      ws.L.MT_max * p.n_tiles, st);
}

// Weight gradient dW[e] [M, N] = A_e^T B_e over expert e's rows with both
// operands quantised along the rows and stored transposed: AqT [M, ldt],
// BqT [N, ldt] (scale tiles over them, blocks of 32 rows from each expert's
// padded segment start), K steps of 128 rows.
cudaError_t gemm_wgrad_mx(const moe_config& c, const Ws& ws, const moe_sched& s, const uint8_t* AqT,
                          const uint8_t* AsT, int M, const uint8_t* BqT, const uint8_t* BsT, int N,
                          __nv_bfloat16* dW, const char* name, cudaStream_t st) {
  CUtensorMap ta, tb, to;
  const uint64_t ldt = (uint64_t)ws.L.Rp_max;
  Params p = base_params(c, ws);
  p.umma_n = 256;
  p.m_tiles_w = (M + kBM - 1) / kBM;
  p.n_tiles = (N + 255) / 256;
  p.out_cols = N;
  p.out_rows = M;
  p.counts = s.counts;
  p.kstep = BK8;
  p.sfa = AsT;
  p.sfb = BsT;
  p.k_groups = (int)(ldt / 128);
  p.b_rows = N;
  if (!map2d(&ta, AqT, ldt, (uint64_t)M, 128, kBM, true) || !map3d(&tb, BqT, ldt, (uint64_t)N, 1, 128, 256, true) ||
      !map3d(&to, dW, N, M, c.E, 64, 32))
    return cudaErrorInvalidValue;
  if (gemm_clc_enabled(c))
    return launch<true, false, false, EPI_STORE, true, false, UNITS_ALL, true>(
        name, ta, ta, tb, to, to, p, (long long)c.E * p.m_tiles_w * p.n_tiles, st);
  return launch<true, false, false, EPI_STORE, true>(name, ta, ta, tb, to, to, p,
                                                     (long long)c.E * p.m_tiles_w * p.n_tiles, st);
}

}  // namespace moe
