// ring.cu -- the forward pass as one persistent kernel with an SM partition.
//
// The pages' megakernel splits the GPU's SMs into a side that moves tokens
// (dispatch, combine, state) and a side that runs the expert FFN; the moving
// side tells the compute side through GPU-local counters when a full
// minibatch has arrived, the compute side signals back when it is done, and
// a fixed-size ring token buffer is recycled minibatch by minibatch, with no
// CPU in the loop (leiphone "MoK..." section 02; Marktechpost "Cursor开源MoK..."
// three design decisions).  On one GPU the moving side is an HBM gather.
//
// Layout of one launch (cooperative, so every CTA is co-resident):
//   CTAs [0, G)       gather side: for every window w of `mb` consecutive rows
//                     of the padded expert order, wait until ring slot
//                     w % S is free, copy the window's token rows into it,
//                     then release ready[slot].
//   CTAs [G, grid)    compute side: the warp-specialised tcgen05 pipeline of
//                     gemm.cu over a tile stream ordered
//                     G1(0), [G1(1), G2(0)], [G1(2), G2(1)], ..., G2(last):
//                     GEMM1 + SwiGLU tiles of window w read the ring slot after
//                     acquiring ready[slot] and release freed[slot] once their
//                     loads have landed; GEMM2 tiles of a 128-row tile wait for
//                     that tile's GEMM1 epilogues (a_ready) and store Y in
//                     expert order.
//   all CTAs          after the last GEMM2 store (done2), the fixed-order
//                     weighted merge of every token.
// Every tile waits only on tiles and windows earlier in the stream, so the
// stream always makes progress.  Every wait is bounded: on expiry the kernel
// sets a global abort word, reports MOE_ERR_TIMEOUT in the workspace status
// word and every CTA winds down (no trap).
#include <cuda_bf16.h>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "rowops.cuh"

namespace moe {

namespace {

constexpr int BK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * BK * 2;          // 16 KB
constexpr int kBBox = 64 * BK * 2;             // 8 KB: 64 columns x 64 K rows, MN-major
constexpr int kStageBytes = kABytes + 4 * kBBox;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kOutTile = 32 * 128;
constexpr int kTmemCols = 512;
constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kEpiWarps * 2 * kOutTile + 256;
static_assert(kSmem <= 232448, "shared memory budget");

struct RingParams {
  int T, d, f, E, k;
  int G, S, mb, mtw;          // gather CTAs, ring slots, rows per window, 128-row tiles per window
  int hn, nt1, nt2, kb1, kb2;  // GEMM1 half width, N tiles of GEMM1 / GEMM2, K blocks
  const int* mt_off;
  const int* counts;   // rows per expert: a partial last tile runs thin (swapped)
  int thin;
  const int* hdr;
  const int* row_of_pad;
  const int* pos_pad;
  const float* topk_w;
  const __nv_bfloat16* x;
  __nv_bfloat16* ring;  // [S * mb, d]
  __nv_bfloat16* A;     // [Rp, f]
  __nv_bfloat16* H;     // [Rp, 2f] or null
  __nv_bfloat16* Y;     // [Rp, d]
  __nv_bfloat16* out;   // [T, d]
  int* ready;           // [S]  gather arrivals per slot
  int* freed;           // [S]  GEMM1 tiles done reading per slot
  int* a_ready;         // [MT] GEMM1 epilogue warps done per 128-row tile
  int* done2;           // GEMM2 epilogue warps done
  int* gabort;          // set once by the first wait that gives up
  int* status;
};

// Window geometry of this call (from the padded row total the schedule wrote).
struct Geo {
  int rp, nW, mt_last, F1, F2, total, total2;
};

__device__ __forceinline__ Geo make_geo(const RingParams& p) {
  Geo g;
  g.rp = p.hdr[kHdrRpTotal];
  g.nW = (g.rp + p.mb - 1) / p.mb;
  g.mt_last = (g.rp - (g.nW - 1) * p.mb) / kBM;
  g.F1 = p.mtw * p.nt1;
  g.F2 = p.mtw * p.nt2;
  g.total = (g.nW - 1) * (g.F1 + g.F2) + g.mt_last * (p.nt1 + p.nt2);
  g.total2 = (g.nW - 1) * g.F2 + g.mt_last * p.nt2;
  return g;
}

struct RTile {
  int phase, w, mloc, mt, n, e;
  int rows;   // valid rows of the 128-row tile
  bool thin;  // computed as (weights)^T x (rows)^T with the tokens on N
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

// Tile L of the stream G1(0), [G1(1) G2(0)], ..., [G1(nW-1) G2(nW-2)], G2(nW-1).
// Inside a phase block, tiles run N-tile-major so that the tiles sharing an
// expert's weight slice are adjacent.
__device__ __forceinline__ RTile ring_decode(const RingParams& p, const Geo& g, int L) {
  int phase, w, loc;
  const int t1l = g.mt_last * p.nt1;
  if (g.nW == 1) {
    if (L < t1l) { phase = 1; w = 0; loc = L; }
    else { phase = 2; w = 0; loc = L - t1l; }
  } else if (L < g.F1) {
    phase = 1; w = 0; loc = L;
  } else {
    int l = L - g.F1;
    const int blk = g.F1 + g.F2;
    const int nfull = g.nW - 2;
    if (l < nfull * blk) {
      const int b = 1 + l / blk, r = l % blk;
      if (r < g.F1) { phase = 1; w = b; loc = r; }
      else { phase = 2; w = b - 1; loc = r - g.F1; }
    } else {
      l -= nfull * blk;
      if (l < t1l) { phase = 1; w = g.nW - 1; loc = l; }
      else if (l < t1l + g.F2) { phase = 2; w = g.nW - 2; loc = l - t1l; }
      else { phase = 2; w = g.nW - 1; loc = l - t1l - g.F2; }
    }
  }
  const int mtw = (w == g.nW - 1) ? g.mt_last : p.mtw;
  RTile t;
  t.phase = phase;
  t.w = w;
  t.mloc = loc % mtw;
  t.n = loc / mtw;
  t.mt = w * p.mtw + t.mloc;
  t.e = find_expert(p.mt_off, p.E, t.mt);
  t.rows = kBM;
  t.thin = false;
  if (p.thin && t.phase == 1) {
    const int cnt = __ldg(p.counts + t.e);
    const int rows = cnt - (t.mt - __ldg(p.mt_off + t.e)) * kBM;
    if (thin_tile(rows, cnt)) {
      t.rows = rows;
      t.thin = true;
    }
  }
  return t;
}

__global__ void __launch_bounds__(kThreads, 1)
    ring_forward_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW1,
                        const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmW2,
                        const __grid_constant__ CUtensorMap tmY, const RingParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_ok;
  __shared__ int s_pos[kMaxK];
  __shared__ float s_w[kMaxK];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Geo geo = make_geo(p);
  const int inject = p.hdr[kHdrInject];        // test hook: window + 1 whose arrival is withheld
  const int lim_ms = p.hdr[kHdrInject + 1];    // test hook: wait limit in ms (0: default)
  const uint64_t limit = lim_ms > 0 ? (uint64_t)lim_ms * 1000000ull : kWaitLimitNs;

  if (blockIdx.x < (unsigned)p.G) {
    // ====================================================== gather side
    const int nwarp = kThreads / 32;
    for (int w = 0; w < geo.nW; ++w) {
      const int s = w % p.S, gen = w / p.S;
      if (threadIdx.x == 0)
        s_ok = (gen == 0) || wait_counter(&p.freed[s], gen * geo.F1, p.gabort, p.status, 500 + s, limit);
      __syncthreads();
      const bool ok = s_ok;
      __syncthreads();  // everyone has read s_ok before thread 0 writes it again
      if (!ok) break;
      const int r0 = w * p.mb, r1 = min(r0 + p.mb, geo.rp);
      const int nvec = p.d >> 3;
      for (int pp = r0 + blockIdx.x * nwarp + warp; pp < r1; pp += p.G * nwarp) {
        const int r = p.row_of_pad[pp];
        const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)(r < 0 ? 0 : r / p.k) * p.d);
        uint4* dst = reinterpret_cast<uint4*>(p.ring + ((size_t)s * p.mb + (pp - r0)) * p.d);
        for (int v0 = lane; v0 < nvec; v0 += 32 * 4) {
          uint4 buf[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int v = v0 + u * 32;
            buf[u] = (r >= 0 && v < nvec) ? ldg_nc_v4(src + v) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (v0 + u * 32 < nvec) stg_v4(dst + v0 + u * 32, buf[u]);
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        if (inject != w + 1) red_release_add(&p.ready[s], 1);
      }
    }
  } else {
    // ====================================================== compute side
    uint8_t* stages = smem;
    uint8_t* staging = smem + (size_t)kStages * kStageBytes;
    uint8_t* ctrl = staging + kEpiWarps * 2 * kOutTile;
    uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
    uint64_t* empty = full + kStages;
    uint64_t* tfull = empty + kStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int cta = blockIdx.x - p.G, ncta = gridDim.x - p.G;

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
      *abort_flag = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmW1);
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmW2);
      tma_prefetch_desc(&tmY);
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
        for (int L = cta; L < geo.total; L += ncta) {
          const RTile t = ring_decode(p, geo, L);
          const bool g1 = (t.phase == 1);
          const int slot = t.w % p.S;
          bool ok;
          if (g1)
            ok = wait_counter(&p.ready[slot], p.G * (t.w / p.S + 1), p.gabort, p.status, 600 + slot, limit);
          else
            ok = wait_counter(&p.a_ready[t.mt], kEpiWarps * p.nt1, p.gabort, p.status, 700, limit);
          if (!ok) {
            *abort_flag = 1;
            goto producer_done;
          }
          fence_proxy_async_global();  // rows written by other CTAs, read by TMA below
          const int nbox = g1 ? (2 * p.hn) / 64 : 4;
          const int nkb = g1 ? p.kb1 : p.kb2;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, 100 + s)) goto producer_done;
            const uint32_t sa = smem_u32(stages + (size_t)s * kStageBytes);
            const uint32_t sb = sa + kABytes;
            const uint32_t fb = smem_u32(&full[s]);
            mbar_arrive_expect_tx(&full[s], (uint32_t)kABytes + (uint32_t)nbox * kBBox);
            if (g1) {
              tma_load_2d(sa, &tmX, fb, kb * BK, slot * p.mb + t.mloc * kBM);
              const int half = nbox / 2;
              for (int i = 0; i < nbox; ++i) {
                const int col = (i < half) ? t.n * p.hn + 64 * i : p.f + t.n * p.hn + 64 * (i - half);
                tma_load_3d(sb + i * kBBox, &tmW1, fb, col, kb * BK, t.e);
              }
            } else {
              tma_load_2d(sa, &tmA, fb, kb * BK, t.mt * kBM);
              for (int i = 0; i < 4; ++i) tma_load_3d(sb + i * kBBox, &tmW2, fb, t.n * 256 + 64 * i, kb * BK, t.e);
            }
            used |= 1u << s;
            last_par = (last_par & ~(1u << s)) | (ph << s);
            if (++s == kStages) {
              s = 0;
              ph ^= 1u;
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
        for (int L = cta; L < geo.total; L += ncta) {
          const RTile t = ring_decode(p, geo, L);
          const bool g1 = (t.phase == 1);
          const int nkb = g1 ? p.kb1 : p.kb2;
          if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, p.status, 200 + acc)) goto mma_done;
          tc_fence_after();
          const uint32_t dt = tmem_base + (uint32_t)acc * 256u;
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&full[s], ph, abort_flag, p.status, 300 + s)) goto mma_done;
            tc_fence_after();
            if (g1 && kb == nkb - 1) red_release_add(&p.freed[t.w % p.S], 1);  // ring rows landed
            const uint32_t sa = smem_u32(stages + (size_t)s * kStageBytes);
            const uint32_t sb = sa + kABytes;
            if (t.thin) {
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
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                tc_mma_f16(dt, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 2048, 8192, 1024),
                           g1 ? idesc1 : idesc2, (kb > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(smem_u32(&empty[s]));
            if (++s == kStages) {
              s = 0;
              ph ^= 1u;
            }
          }
          tc_commit(smem_u32(&tfull[acc]));
          if (++acc == 2) {
            acc = 0;
            aph ^= 1u;
          }
        }
      mma_done:
        tc_commit(smem_u32(drain));
        mbar_wait_drain(drain, 0);
      }
    } else {
      // -------------------------------------------- epilogue warps
      const int q = warp & 3;
      int acc = 0, buf = 0;
      uint32_t aph = 0;
      const uint32_t stg = smem_u32(staging) + (uint32_t)(warp - 2) * 2u * kOutTile;
      for (int L = cta; L < geo.total; L += ncta) {
        const RTile t = ring_decode(p, geo, L);
        if (!mbar_wait(&tfull[acc], aph, abort_flag, p.status, 400 + acc)) break;
        tc_fence_after();
        const uint32_t tb = tmem_base + (uint32_t)acc * 256u + ((uint32_t)(q * 32) << 16);
        if (t.thin) {
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
          // SwiGLU: A (and H when saving) with direct row stores
          const size_t row = (size_t)t.mt * kBM + q * 32 + lane;
          for (int c = 0; c < p.hn; c += 32) {
            float g[32], u[32], a[32];
            tmem_ld32(tb + c, g);
            tmem_ld32(tb + p.hn + c, u);
            const int col = t.n * p.hn + c;
#pragma unroll
            for (int i = 0; i < 32; ++i) a[i] = silu_f(g[i]) * u[i];
            store32_bf16(p.A + row * p.f + col, a);
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
        if (++acc == 2) {
          acc = 0;
          aph ^= 1u;
        }
      }
      if (lane == 0) bulk_wait<0>();
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

cudaError_t ring_forward(const moe_config& c, const Ws& ws, const int* counts, const __nv_bfloat16* x,
                         const __nv_bfloat16* W1, const __nv_bfloat16* W2, const float* topk_w,
                         __nv_bfloat16* A, __nv_bfloat16* H, __nv_bfloat16* out, cudaStream_t st) {
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
  p.G = c.gather_ctas > 0 ? c.gather_ctas : ring_default_gather_ctas(sms);
  if (p.G >= sms) return cudaErrorInvalidValue;
  p.hn = (c.f % 128 == 0) ? 128 : 64;
  p.nt1 = c.f / p.hn;
  p.nt2 = (c.d + 255) / 256;
  p.kb1 = c.d / BK;
  p.kb2 = c.f / BK;
  p.mt_off = ws.mt_off();
  p.counts = counts;
  p.thin = gemm1_thin_enabled(c) ? 1 : 0;
  p.hdr = ws.hdr();
  p.row_of_pad = ws.row_of_pad();
  p.pos_pad = ws.pos_pad();
  p.topk_w = topk_w;
  p.x = x;
  p.ring = static_cast<__nv_bfloat16*>(ws.at(ws.L.ring));
  p.A = A;
  p.H = H;
  p.Y = static_cast<__nv_bfloat16*>(ws.at(ws.L.Yp));
  p.out = out;
  int* ctr = static_cast<int*>(ws.at(ws.L.ctr));
  p.ready = ctr;
  p.freed = ctr + p.S;
  p.done2 = ctr + 2 * p.S;
  p.gabort = ctr + 2 * p.S + 1;
  p.a_ready = ctr + 2 * p.S + 2;
  p.status = ws.hdr() + kHdrStatus;

  const uint64_t rows = (uint64_t)ws.L.Rp_max;
  CUtensorMap tmX, tmW1, tmA, tmW2, tmY;
  if (!map2d(&tmX, p.ring, c.d, (uint64_t)p.S * p.mb, 64, kBM) ||
      !map3d(&tmW1, W1, 2ull * c.f, c.d, c.E, 64, 64) || !map2d(&tmA, A, c.f, rows, 64, kBM) ||
      !map3d(&tmW2, W2, c.d, c.f, c.E, 64, 64) || !map2d(&tmY, p.Y, c.d, rows, 64, 32))
    return cudaErrorInvalidValue;

  cudaError_t err = cudaMemsetAsync(ctr, 0, ws.L.ctr_bytes, st);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(ring_forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ring_forward_kernel, kThreads, kSmem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  void* args[] = {&tmX, &tmW1, &tmA, &tmW2, &tmY, &p};
  TraceScope ts("ring_forward", st);
  return cudaLaunchCooperativeKernel((const void*)ring_forward_kernel, dim3(sms), dim3(kThreads), args,
                                     kSmem, st);
}

}  // namespace moe
