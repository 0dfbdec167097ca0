// gather_merge.cu -- the memory-bound steps of the layer.
//
//  * gather (dispatch, leiphone "MoK..." section 02): every routed token row
//    lands in its expert's segment of the padded expert-ordered buffer.  On
//    one GPU this is an HBM row copy.  Without a ring it walks the tokens:
//    each token row is read from HBM once and written from shared memory to
//    its k positions (the buffer a pull by the expert side would build, with
//    each source row read once instead of k times).  After a ring forward the
//    backward's gather walks the padded rows instead (the pull order), so
//    that it can take the rows the ring still holds.  The forward's gather
//    leaves padding rows alone (GEMM1 zeroes what it computes from them); the
//    backward's writes them as zeros, which the weight gradients' K loop over
//    padded rows relies on.
//  * merge (combine + final weighted merge, leiphone section 03): each token
//    sums its k expert outputs in slot order in fp32 and rounds once to bf16.
//    The same kernel without weights is the backward's reverse dispatch.
//  * dg reduce: the routing-weight gradient, summed from the per-tile partials
//    of the fused SwiGLU backward (Marktechpost "Cursor开源MoK..." three design
//    decisions, last paragraph), and its softmax backward to the logits.
//  * MXFP8 quantisation (leiphone section 02, MXFP8 paragraph): fused into the
//    gather for activations (each token row quantised once, its codes and
//    scales written to its k positions); a separate pass for weights.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#ifndef MOE_BULK_GATHER
#define MOE_BULK_GATHER 1  // 0: the plain-load gather everywhere
#endif

// L2 priorities of the gathers' copies.  A token's k rows lie in k different
// experts' segments, so its source row is read again only after a large part
// of the (larger than L2) gathered buffer has been written; the gathered rows
// themselves are read again only by the next kernel, which starts from the
// first rows.  1: the gathered rows are written evict-first, so that the
// source rows stay in L2 between their k reads; 2: the source rows are in
// addition read evict-last; 0: no policy.
#ifndef MOE_GATHER_L2
#define MOE_GATHER_L2 1
#endif

#include "bulk_rows.cuh"
#include "moe_internal.h"
#include "mx.cuh"
#include "rowops.cuh"

namespace moe {

namespace {

// First padded row that a completed ring forward left in its ring (its last
// `slots` windows of mb rows), or `rows` when there is no such ring.
__device__ __forceinline__ int ring_first_row(const __nv_bfloat16* ring, const int* hdr, int rows,
                                              int mb, int slots) {
  if (ring == nullptr || hdr[kHdrRingValid] == 0) return rows;
  const int nw = (rows + mb - 1) / mb;
  return max(0, nw - slots) * mb;
}

// Ring slot row that holds padded row pp (pp at or past ring_first_row).
__device__ __forceinline__ const __nv_bfloat16* ring_row(const __nv_bfloat16* ring, int pp, int mb,
                                                         int slots, int d) {
  const int w = pp / mb;
  return ring + ((size_t)(w % slots) * mb + (pp - w * mb)) * d;
}

// One warp per padded row; 16-byte vectors; up to 8 loads in flight per lane.
// Padding rows are zero-filled when zero_pad, else skipped.  With a ring
// (backward), rows are walked from the last to the first and the first
// source's rows that the ring still holds are read from it.
__global__ void __launch_bounds__(256) gather_kernel(const __nv_bfloat16* __restrict__ src,
                                                     __nv_bfloat16* __restrict__ dst,
                                                     const __nv_bfloat16* __restrict__ src2,
                                                     __nv_bfloat16* __restrict__ dst2,
                                                     const int* __restrict__ row_of_pad,
                                                     const int* __restrict__ hdr, int k, int d,
                                                     int zero_pad, const __nv_bfloat16* __restrict__ ring,
                                                     int ring_mb, int ring_slots) {
  const int rows = hdr[kHdrRpTotal];
  const int rb = ring_first_row(ring, hdr, rows, ring_mb, ring_slots);
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int nvec = d >> 3;
  for (int q = gw; q < rows; q += nw) {
    const int pp = ring != nullptr ? rows - 1 - q : q;
    const int r = row_of_pad[pp];
    if (r < 0 && !zero_pad) continue;
    for (int pass = 0; pass < 2; ++pass) {
      const __nv_bfloat16* s = pass ? src2 : src;
      __nv_bfloat16* o = pass ? dst2 : dst;
      if (o == nullptr) break;
      const __nv_bfloat16* srow = (pass == 0 && r >= 0 && pp >= rb) ? ring_row(ring, pp, ring_mb, ring_slots, d)
                                                                    : s + (size_t)(r < 0 ? 0 : r / k) * d;
      const uint4* sv = reinterpret_cast<const uint4*>(srow);
      uint4* ov = reinterpret_cast<uint4*>(o + (size_t)pp * d);
      for (int v0 = lane; v0 < nvec; v0 += 32 * 8) {
        uint4 buf[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32;
          buf[u] = (r >= 0 && v < nvec) ? ldg_nc_v4(sv + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32;
          if (v < nvec) stg_v4(ov + v, buf[u]);
        }
      }
    }
  }
}

// The same gather staged through shared memory with bulk copies: one CTA per
// SM, warps [0, gw) each with nbw row buffers (bulk_rows.cuh).  Item i of a
// warp is the q-th padded row, q = gid + (i / npass) * ni (walked from the
// last row down when a ring is given), from src (pass 0) or src2 (pass 1).
// Item codes: r * npass + pass for row r of a source, R * npass + pp for
// padded row pp read from the ring.
__global__ void __launch_bounds__(256, 1) gather_bulk_kernel(
    const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst,
    const __nv_bfloat16* __restrict__ src2, __nv_bfloat16* __restrict__ dst2,
    const int* __restrict__ row_of_pad, const int* __restrict__ hdr, int k, int d, int zero_pad,
    int gw, int nbw, int* status, int R, const __nv_bfloat16* __restrict__ ring, int ring_mb,
    int ring_slots) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rb = (uint32_t)d * 2u;
  RowPipe rp;
  rp.zrow = smem_u32(smem);
  rp.rb = rb;
  rp.wbuf = rp.zrow + rb + (uint32_t)(warp * nbw) * rb;
  rp.bars = reinterpret_cast<uint64_t*>(smem + (size_t)(1 + gw * nbw) * rb) + warp * nbw;
  rp.nbw = nbw;
  rp.depth = nbw / 2;
  rp.ph = rp.pend = 0;
  rp.hints = MOE_GATHER_L2 >= 2 ? 3u : MOE_GATHER_L2 == 1 ? 2u : 0u;
  rp.ld_pol = MOE_GATHER_L2 >= 2 ? l2_policy_evict_last() : 0;
  rp.st_pol = MOE_GATHER_L2 >= 1 ? l2_policy_evict_first() : 0;
  if (zero_pad) {
    for (uint32_t i = threadIdx.x; i < rb / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();  // the zero row is read by bulk stores
  }
  if (warp < gw && lane == 0) {
    for (int b = 0; b < nbw; ++b) mbar_init(&rp.bars[b], 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) s_abort = 0;
  __syncthreads();
  if (warp >= gw) return;
  const int rows = hdr[kHdrRpTotal];
  const int ring0 = ring_first_row(ring, hdr, rows, ring_mb, ring_slots);
  const bool rev = ring != nullptr;
  const int npass = dst2 != nullptr ? 2 : 1;
  const int gid = blockIdx.x * gw + warp, ni = gridDim.x * gw;
  const int n = gid < rows ? (rows - gid + ni - 1) / ni * npass : 0;
  if (n == 0) return;
  auto pad_of = [&](int i) {
    const int q = gid + (i / npass) * ni;
    return rev ? rows - 1 - q : q;
  };
  const bool done = bulk_rows(
      rp, n,
      [&](int i) {
        const int pp = pad_of(i);
        const int r = __ldg(row_of_pad + pp);
        if (r < 0) return zero_pad ? kRowZero : kRowSkip;
        if (i % npass == 0 && pp >= ring0) return R * npass + pp;
        return r * npass + i % npass;
      },
      [&](int code) {
        if (code >= R * npass) return ring_row(ring, code - R * npass, ring_mb, ring_slots, d);
        const __nv_bfloat16* s = (code % npass) ? src2 : src;
        return s + (size_t)(code / npass / k) * d;
      },
      [&](int i) { return ((i % npass) ? dst2 : dst) + (size_t)pad_of(i) * d; },
      &s_abort, status, 900);
  if (lane == 0) {
    bulk_wait<0>();
    if (!done)
      for (int b = 0; b < nbw; ++b)  // no copy may still target shared memory at exit
        if ((rp.pend >> b) & 1u) mbar_wait_drain(&rp.bars[b], (rp.ph >> b) & 1u);
  }
}

// Quantise 32 bf16 values (4 x uint4) to E4M3 codes with one UE8M0 scale.
__device__ __forceinline__ void quant32(const uint4 (&in)[4], uint4 (&out)[2], uint8_t& scale) {
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&in[i]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      v[i * 8 + j * 2] = f.x;
      v[i * 8 + j * 2 + 1] = f.y;
    }
  }
  scale = mx_quant32(v, out[0], out[1]);
}

// Shared-memory layout of the bulk-copy gathers: a zero row, gw warps x nbw
// row buffers of rb bytes, then one mbarrier per buffer (and, for the MXFP8
// gather, gw scale rows of sb bytes after the barriers).
struct GatherSmem {
  uint8_t* base;
  RowPipe rp;
};

__device__ __forceinline__ GatherSmem gather_smem_init(uint8_t* smem_raw, uint32_t rb, int gw, int nbw,
                                                       int warp, int lane) {
  GatherSmem g;
  g.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                      ~static_cast<uintptr_t>(127));
  RowPipe& rp = g.rp;
  rp.zrow = smem_u32(g.base);
  rp.rb = rb;
  rp.wbuf = rp.zrow + rb + (uint32_t)(warp * nbw) * rb;
  rp.bars = reinterpret_cast<uint64_t*>(g.base + (size_t)(1 + gw * nbw) * rb) + warp * nbw;
  rp.nbw = nbw;
  rp.depth = nbw / 2;
  rp.ph = rp.pend = 0;
  rp.hints = MOE_GATHER_L2 >= 2 ? 3u : MOE_GATHER_L2 == 1 ? 2u : 0u;
  rp.ld_pol = MOE_GATHER_L2 >= 2 ? l2_policy_evict_last() : 0;
  rp.st_pol = MOE_GATHER_L2 >= 1 ? l2_policy_evict_first() : 0;
  for (uint32_t i = threadIdx.x; i < rb / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(g.base)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();  // the zero row is read by bulk stores
  if (warp < gw && lane == 0) {
    for (int b = 0; b < nbw; ++b) mbar_init(&rp.bars[b], 1);
    fence_mbar_init();
  }
  return g;
}

// Gather in token order (no ring): each source row is read from HBM once and
// written from shared memory to each of its k padded positions (pos_pad).
// Items of the warps' walk: tokens (with two sources, item 2t + pass), then,
// with zero_pad, every padded position, written as a zero row in both
// destinations where it holds no routed row.
__global__ void __launch_bounds__(256, 1) gather_tokens_kernel(
    const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst,
    const __nv_bfloat16* __restrict__ src2, __nv_bfloat16* __restrict__ dst2,
    const int* __restrict__ pos_pad, const int* __restrict__ row_of_pad, const int* __restrict__ hdr,
    int T, int k, int d, int zero_pad, int gw, int nbw, int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  GatherSmem gs = gather_smem_init(smem_raw, (uint32_t)d * 2u, gw, nbw, warp, lane);
  RowPipe& rp = gs.rp;
  if (threadIdx.x == 0) s_abort = 0;
  __syncthreads();
  if (warp >= gw) return;
  const int rows = hdr[kHdrRpTotal];
  const int npass = dst2 != nullptr ? 2 : 1;
  const int ntok = T * npass;
  const int N = ntok + (zero_pad ? rows : 0);
  const int gid = blockIdx.x * gw + warp, ni = gridDim.x * gw;
  const int n = gid < N ? (N - gid + ni - 1) / ni : 0;
  if (n == 0) return;
  const bool done = bulk_rows_fan(
      rp, n, max(k, npass), rp.rb,
      [&](int i) {
        const int g = gid + i * ni;
        if (g < ntok) return g;
        return __ldg(row_of_pad + (g - ntok)) < 0 ? kRowZero : kRowSkip;
      },
      [&](int code) { return ((code % npass) ? src2 : src) + (size_t)(code / npass) * d; },
      [&](int i, int j) -> __nv_bfloat16* {
        const int g = gid + i * ni;
        if (g < ntok) {
          if (j >= k) return nullptr;
          const int pp = __ldg(pos_pad + (size_t)(g / npass) * k + j);
          return ((g % npass) ? dst2 : dst) + (size_t)pp * d;
        }
        if (j >= npass) return nullptr;
        return (j ? dst2 : dst) + (size_t)(g - ntok) * d;
      },
      RowAsIs(), &s_abort, status, 920);
  if (lane == 0) {
    bulk_wait<0>();
    if (!done)
      for (int b = 0; b < nbw; ++b)  // no copy may still target shared memory at exit
        if ((rp.pend >> b) & 1u) mbar_wait_drain(&rp.bars[b], (rp.ph >> b) & 1u);
  }
}

// The MXFP8 gather in token order: each token row is read once, quantised
// once in its shared-memory buffer (codes over the first d bytes, block
// scales into the warp's scale row), and its codes and scales are written to
// each of its k padded positions.  Padding rows are left alone: the MXFP8
// GEMM1 writes zeros for them whatever they hold.
__global__ void __launch_bounds__(256, 1) gather_tokens_mxfp8_kernel(
    const __nv_bfloat16* __restrict__ src, uint8_t* __restrict__ q, uint8_t* __restrict__ sc,
    const int* __restrict__ pos_pad, int T, int k, int d, int gw, int nbw, int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rb = (uint32_t)d * 2u;
  GatherSmem gs = gather_smem_init(smem_raw, rb, gw, nbw, warp, lane);
  RowPipe& rp = gs.rp;
  const int nblk = d >> 5, kgroups = d >> 7;
  uint8_t* srow = gs.base + (size_t)(1 + gw * nbw) * rb + (size_t)gw * nbw * 8 + (size_t)warp * nblk;
  if (threadIdx.x == 0) s_abort = 0;
  __syncthreads();
  if (warp >= gw) return;
  const int gid = blockIdx.x * gw + warp, ni = gridDim.x * gw;
  const int n = gid < T ? (T - gid + ni - 1) / ni : 0;
  if (n == 0) return;
  auto xform = [&](int i, int, uint32_t buf) {
    const int g = gid + i * ni;
    {
      // quantise in place: iteration m reads blocks 32m..32m+31 (bf16 bytes
      // [2048m, 2048m + 2048)) before any lane writes their codes at
      // [1024m, 1024m + 1024), which only overlap bytes read before
      uint8_t* row = gs.base + (buf - rp.zrow);
      for (int b0 = 0; b0 < nblk; b0 += 32) {
        const int blk = b0 + lane;
        uint4 in[4], out[2];
        uint8_t s8 = 0;
        if (blk < nblk)
#pragma unroll
          for (int u = 0; u < 4; ++u) in[u] = reinterpret_cast<const uint4*>(row)[blk * 4 + u];
        __syncwarp();
        if (blk < nblk) {
          quant32(in, out, s8);
          reinterpret_cast<uint4*>(row)[blk * 2] = out[0];
          reinterpret_cast<uint4*>(row)[blk * 2 + 1] = out[1];
          srow[blk] = s8;
        }
      }
      __syncwarp();
      // the scales of blocks 4w..4w+3 of a row are one 32-bit word of its
      // 128-row scale tile: lane l writes words l, l + 32, ... of every copy
      const int my_pp = lane < k ? __ldg(pos_pad + (size_t)g * k + lane) : 0;
      for (int j = 0; j < k; ++j) {
        const int pp = __shfl_sync(0xffffffffu, my_pp, j);
        uint8_t* tile = sc + (size_t)(pp >> 7) * kgroups * 512u + mx_sf_byte(pp & 127, 0);
        for (int w = lane; w < kgroups; w += 32)
          *reinterpret_cast<uint32_t*>(tile + (size_t)w * 512u) = reinterpret_cast<const uint32_t*>(srow)[w];
      }
      fence_proxy_async_smem();  // the codes are read by bulk stores, the buffer refilled by bulk loads
      __syncwarp();
    }
  };
  const bool done = bulk_rows_fan(
      rp, n, k, (uint32_t)d, [&](int i) { return gid + i * ni; },
      [&](int code) { return src + (size_t)code * d; },
      [&](int i, int j) { return q + (size_t)__ldg(pos_pad + (size_t)(gid + i * ni) * k + j) * d; },
      xform, &s_abort, status, 930);
  if (lane == 0) {
    bulk_wait<0>();
    if (!done)
      for (int b = 0; b < nbw; ++b)  // no copy may still target shared memory at exit
        if ((rp.pend >> b) & 1u) mbar_wait_drain(&rp.bars[b], (rp.ph >> b) & 1u);
  }
}


// Gather + quantise: one warp per padded row, each lane one block of 32.
__global__ void __launch_bounds__(256) gather_mxfp8_kernel(const __nv_bfloat16* __restrict__ src,
                                                           uint8_t* __restrict__ q,
                                                           uint8_t* __restrict__ sc,
                                                           const int* __restrict__ row_of_pad,
                                                           const int* __restrict__ hdr, int k,
                                                           int d) {
  const int rows = hdr[kHdrRpTotal];
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int nblk = d >> 5;
  for (int pp = gw; pp < rows; pp += nw) {
    const int r = row_of_pad[pp];
    const uint4* sv = reinterpret_cast<const uint4*>(src + (size_t)(r < 0 ? 0 : r / k) * d);
    for (int b = lane; b < nblk; b += 32) {
      uint4 in[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) in[i] = (r >= 0) ? ldg_nc_v4(sv + b * 4 + i) : make_uint4(0, 0, 0, 0);
      uint4 out[2];
      uint8_t s;
      quant32(in, out, s);
      uint4* qv = reinterpret_cast<uint4*>(q + (size_t)pp * d + b * 32);
      stg_v4(qv, out[0]);
      stg_v4(qv + 1, out[1]);
      sc[mx_sf_offset((size_t)pp, b, d >> 7)] = s;
    }
  }
}

// Weights [batch, K, N] bf16 -> codes [batch, N, K] and scale tiles over [batch*N, K].
// One thread per (batch, n, 32-block of K): reads a strided column block.
__global__ void __launch_bounds__(256) quant_weights_kernel(const __nv_bfloat16* __restrict__ w,
                                                            int64_t batch, int K, int N,
                                                            uint8_t* __restrict__ q,
                                                            uint8_t* __restrict__ sc) {
  const int nkb = K >> 5;
  const int64_t total = batch * (int64_t)N * nkb;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    // consecutive threads take consecutive n so the strided reads coalesce
    const int n = (int)(i % N);
    const int64_t rest = i / N;
    const int kb = (int)(rest % nkb);
    const int64_t b = rest / nkb;
    const __nv_bfloat16* col = w + (b * K + (int64_t)kb * 32) * N + n;
    uint4 in[4];
    uint16_t* hv = reinterpret_cast<uint16_t*>(in);
#pragma unroll
    for (int j = 0; j < 32; ++j) hv[j] = __bfloat16_as_ushort(col[(int64_t)j * N]);
    uint4 out[2];
    uint8_t s;
    quant32(in, out, s);
    uint4* qv = reinterpret_cast<uint4*>(q + (b * N + n) * (int64_t)K + kb * 32);
    stg_v4(qv, out[0]);
    stg_v4(qv + 1, out[1]);
    sc[mx_sf_offset((size_t)(b * N + n), kb, K >> 7)] = s;
  }
}

// Rows [rows, K] bf16 (K contiguous) -> E4M3 codes [rows, K] and scale tiles,
// blocks of 32 along K.  A warp takes 4 x 512 contiguous bytes at a time, all
// four 16-byte loads of a lane in flight together; a lane holds 8 consecutive
// elements of each, the 4 lanes of a 32-element block share its maximum
// through two shuffles, and each lane stores its 8 codes.  The same scale rule
// and rounding steps as mx_quant32.  rows_dev (optional) caps the rows at a
// device-side count (the padded row total of the schedule).
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ w,
                                                         int64_t rows, int K, const int* rows_dev,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ sc) {
  constexpr int kU = 4;  // 512-byte segments per warp iteration
  const int lane = threadIdx.x & 31;
  const int64_t nr = rows_dev ? (int64_t)*rows_dev : rows;
  const int64_t nv = nr * (K >> 3);  // 8-element vectors; K % 32 == 0, so a block never straddles segments
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t base = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * (32 * kU); base < nv;
       base += nw * 32 * kU) {
    uint4 raw[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = base + u * 32 + lane;
      raw[u] = i < nv ? ldg_nc_v4(reinterpret_cast<const uint4*>(w) + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = base + u * 32 + lane;
      float f[8];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 p2 = __bfloat1622float2(h[j]);
        f[2 * j] = p2.x;
        f[2 * j + 1] = p2.y;
      }
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const int sx = mx_scale_exp(amax);
      const int s1 = -sx / 2, s2 = -sx - s1;
      const float f1 = mx_exp2i(s1), f2 = mx_exp2i(s2);
      if (i < nv) {
        uint2 cw;
        cw.x = mx_pack4(f[0] * f1 * f2, f[1] * f1 * f2, f[2] * f1 * f2, f[3] * f1 * f2);
        cw.y = mx_pack4(f[4] * f1 * f2, f[5] * f1 * f2, f[6] * f1 * f2, f[7] * f1 * f2);
        *reinterpret_cast<uint2*>(q + i * 8) = cw;
        if ((lane & 3) == 0) {
          const int64_t r = (i * 8) / K;
          const int kb = (int)((i * 8 - r * K) >> 5);
          sc[mx_sf_offset((size_t)r, kb, K >> 7)] = (uint8_t)(sx + 127);
        }
      }
    }
  }
}

// Transposing quantiser: src [rows, K] bf16 (rows of the padded expert order,
// K contiguous) -> codes qt [K, ld] (row k holds column k of src, rows
// contiguous) and scale tiles over [K, ld], blocks of 32 rows: the K-major
// operand of a weight-gradient GEMM that contracts over the rows.  A CTA
// stages 64 rows x 256 columns through shared memory; thread c then holds
// column c's values, two blocks of 32.  Rows past the device-side count
// (*rows_dev) are left alone.
__global__ void __launch_bounds__(256) quant_cols_kernel(const __nv_bfloat16* __restrict__ src, int K,
                                                         const int* __restrict__ rows_dev, int ld,
                                                         uint8_t* __restrict__ qt, uint8_t* __restrict__ sct) {
  constexpr int kR = 64;  // rows per block: two 32-row blocks per column
  __shared__ __align__(16) __nv_bfloat16 tile[kR][256 + 8];
  const int rows = *rows_dev;
  const int r0 = blockIdx.x * kR, c0 = blockIdx.y * 256;
  if (r0 >= rows) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // each warp loads 8 rows of 256 columns: 32 lanes x 8 columns (16 bytes),
  // all eight loads in flight before the first store to shared memory
  uint4 v8[kR / 8];
#pragma unroll
  for (int j = 0; j < kR / 8; ++j) {
    const int rr = warp + 8 * j, c = c0 + lane * 8;
    v8[j] = (c < K && r0 + rr < rows) ? ldg_nc_v4(src + (size_t)(r0 + rr) * K + c) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int j = 0; j < kR / 8; ++j) *reinterpret_cast<uint4*>(&tile[warp + 8 * j][lane * 8]) = v8[j];
  __syncthreads();
  const int c = c0 + tid;
  if (c >= K) return;
#pragma unroll
  for (int h = 0; h < kR / 32; ++h) {
    if (r0 + 32 * h >= rows) break;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __bfloat162float(tile[32 * h + i][tid]);
    uint4 lo, hi;
    const uint8_t s8 = mx_quant32(v, lo, hi);
    uint4* qv = reinterpret_cast<uint4*>(qt + (size_t)c * ld + r0 + 32 * h);
    stg_v4(qv, lo);
    stg_v4(qv + 1, hi);
    sct[mx_sf_offset((size_t)c, (r0 >> 5) + h, ld >> 7)] = s8;
  }
}

// One CTA per token (grid-stride); each thread owns 8-column vectors.
__global__ void __launch_bounds__(128) merge_kernel(const __nv_bfloat16* __restrict__ rows,
                                                    const int* __restrict__ pos_pad,
                                                    const float* __restrict__ w, int T, int k,
                                                    int d, __nv_bfloat16* __restrict__ out) {
  __shared__ int sp[kMaxK];
  __shared__ float sw[kMaxK];
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) {
      sp[threadIdx.x] = pos_pad[(size_t)t * k + threadIdx.x];
      sw[threadIdx.x] = w ? w[(size_t)t * k + threadIdx.x] : 1.f;
    }
    __syncthreads();
    merge_token<false>(rows, sp, sw, w != nullptr, t, k, d, out, threadIdx.x, blockDim.x);
  }
}

// One warp per token: dg[t,j] = sum of the fused-epilogue partials (tile
// order), dlogits = g_l (dg_l - sum_j g_j dg_j) at the selected experts.
__global__ void __launch_bounds__(256) dg_reduce_kernel(
    const float* __restrict__ dgp, int nt, const int* __restrict__ pos_pad,
    const float* __restrict__ w, const int* __restrict__ ids, int T, int k, int E,
    float* __restrict__ dtopk_w, float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  float dg = 0.f, g = 0.f;
  int id = 0;
  if (lane < k) {
    const int pp = pos_pad[(size_t)t * k + lane];
    for (int n = 0; n < nt; ++n) dg += dgp[(size_t)pp * nt + n];
    g = w[(size_t)t * k + lane];
    id = ids[(size_t)t * k + lane];
    dtopk_w[(size_t)t * k + lane] = dg;
  }
  if (dlogits == nullptr) return;
  float s = 0.f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, g * dg, j);
  float* row = dlogits + (size_t)t * E;
  for (int e = lane; e < E; e += 32) row[e] = 0.f;
  __syncwarp();
  if (lane < k) row[id] = g * (dg - s);
}

}  // namespace

cudaError_t launch_gather(const moe_config& c, const Ws& ws, const __nv_bfloat16* src,
                          __nv_bfloat16* dst, const __nv_bfloat16* src2, __nv_bfloat16* dst2,
                          cudaStream_t st, const RingSrc* ring) {
  TraceScope ts(dst2 ? "gather_x_dy" : "gather", st);
  // the backward's gather (two sources) zero-fills padding rows for the weight gradients
  const int zero_pad = dst2 != nullptr ? 1 : 0;
  const __nv_bfloat16* rg = ring ? ring->ring : nullptr;
  const int rmb = ring ? ring->mb : 1, rsl = ring ? ring->slots : 1;
  // bulk-copy gather: a zero row and up to 16 row buffers in each of 8 warps
  // (fewer warps for wide rows, at least two buffers each), one CTA per SM
  constexpr size_t kBudget = 227 * 1024 - 128 - 8 * 16 * 8;
  const size_t rb = (size_t)c.d * 2;
  if (kBudget >= 3 * rb && MOE_BULK_GATHER) {
    int gw = 8;
    int nbw = (int)std::min<size_t>(16, (kBudget - rb) / (gw * rb));
    if (nbw < 2) {
      nbw = 2;
      gw = (int)((kBudget - rb) / (2 * rb));
    }
    const size_t smem = 128 + (1 + (size_t)gw * nbw) * rb + (size_t)gw * nbw * 8;
    if (ring == nullptr) {
      // token order: every source row read once, written to its k positions
      cudaError_t err = cudaFuncSetAttribute(gather_tokens_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      gather_tokens_kernel<<<num_sms(), 256, smem, st>>>(src, dst, src2, dst2, ws.pos_pad(), ws.row_of_pad(),
                                                         ws.hdr(), c.T, c.k, c.d, zero_pad, gw, nbw,
                                                         ws.hdr() + kHdrStatus);
      return cudaGetLastError();
    }
    // after a ring forward: padded order, the rows the ring still holds read from it
    cudaError_t err = cudaFuncSetAttribute(gather_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    gather_bulk_kernel<<<num_sms(), 256, smem, st>>>(src, dst, src2, dst2, ws.row_of_pad(), ws.hdr(), c.k,
                                                     c.d, zero_pad, gw, nbw, ws.hdr() + kHdrStatus,
                                                     c.T * c.k, rg, rmb, rsl);
    return cudaGetLastError();
  }
  // rows too wide for two shared-memory buffers per warp: plain loads and stores
  gather_kernel<<<num_sms() * 8, 256, 0, st>>>(src, dst, src2, dst2, ws.row_of_pad(), ws.hdr(), c.k, c.d,
                                               zero_pad, rg, rmb, rsl);
  return cudaGetLastError();
}

cudaError_t launch_gather_mxfp8(const moe_config& c, const Ws& ws, const __nv_bfloat16* src,
                                uint8_t* q, uint8_t* sc, cudaStream_t st) {
  TraceScope ts("gather_mxfp8", st);
  // token order, bf16 rows staged through shared memory: a zero row, up to
  // 16 buffers in each of 8 warps (fewer warps for wide rows, at least two
  // buffers each) and a scale row per warp
  const size_t rb = (size_t)c.d * 2, sb = (size_t)c.d / 32;
  constexpr size_t kBudget = 227 * 1024 - 128 - 8 * 16 * 8;
  if (kBudget >= 3 * rb + 8 * sb && MOE_BULK_GATHER) {
    int gw = 8;
    int nbw = (int)std::min<size_t>(16, (kBudget - rb - gw * sb) / (gw * rb));
    if (nbw < 2) {
      nbw = 2;
      gw = (int)((kBudget - rb) / (2 * rb + sb));
    }
    const size_t smem = 128 + (1 + (size_t)gw * nbw) * rb + (size_t)gw * nbw * 8 + (size_t)gw * sb;
    cudaError_t err = cudaFuncSetAttribute(gather_tokens_mxfp8_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    gather_tokens_mxfp8_kernel<<<num_sms(), 256, smem, st>>>(src, q, sc, ws.pos_pad(), c.T, c.k, c.d, gw,
                                                             nbw, ws.hdr() + kHdrStatus);
    return cudaGetLastError();
  }
  gather_mxfp8_kernel<<<num_sms() * 8, 256, 0, st>>>(src, q, sc, ws.row_of_pad(), ws.hdr(), c.k, c.d);
  return cudaGetLastError();
}

cudaError_t launch_merge(const moe_config& c, const Ws& ws, const __nv_bfloat16* rows,
                         const float* w, __nv_bfloat16* out, cudaStream_t st) {
  const int grid = c.T < num_sms() * 16 ? c.T : num_sms() * 16;
  TraceScope ts(w ? "merge" : "reverse_dispatch", st);
  merge_kernel<<<grid, 128, 0, st>>>(rows, ws.pos_pad(), w, c.T, c.k, c.d, out);
  return cudaGetLastError();
}

cudaError_t launch_dg_reduce(const moe_config& c, const Ws& ws, const moe_sched& s,
                             float* dtopk_w, float* dlogits, cudaStream_t st) {
  const int grid = (c.T * 32 + 255) / 256;
  TraceScope ts("dg_reduce", st);
  dg_reduce_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float*>(ws.at(ws.L.dgp)),
                                          (int)ws.L.nt_dg, ws.pos_pad(), s.topk_w, s.topk_ids,
                                          c.T, c.k, c.E, dtopk_w, dlogits);
  return cudaGetLastError();
}

cudaError_t launch_quantize_mxfp8(const __nv_bfloat16* w, int64_t batch, int K, int N, uint8_t* q,
                                  uint8_t* sc, cudaStream_t st) {
  const int64_t total = batch * (int64_t)N * (K / 32);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  TraceScope ts("quantize_weights", st);
  quant_weights_kernel<<<(int)blocks, 256, 0, st>>>(w, batch, K, N, q, sc);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const __nv_bfloat16* w, int64_t rows, int K, const int* rows_dev,
                              uint8_t* q, uint8_t* sc, cudaStream_t st, const char* name) {
  const int64_t total = rows * (K / 8) / 4;  // four 8-element vectors per thread and iteration
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  TraceScope ts(name, st);
  quant_rows_kernel<<<(int)blocks, 256, 0, st>>>(w, rows, K, rows_dev, q, sc);
  return cudaGetLastError();
}

cudaError_t launch_quant_cols(const __nv_bfloat16* src, int64_t max_rows, int K, const int* rows_dev,
                              uint8_t* qt, uint8_t* sct, int ld, cudaStream_t st, const char* name) {
  dim3 grid((unsigned)((max_rows + 63) / 64), (unsigned)((K + 255) / 256));
  TraceScope ts(name, st);
  quant_cols_kernel<<<grid, 256, 0, st>>>(src, K, rows_dev, ld, qt, sct);
  return cudaGetLastError();
}

namespace {
__global__ void to_bf16_padded_kernel(const float* __restrict__ src, int T, int E, int Epad,
                                      __nv_bfloat16* __restrict__ dst) {
  const size_t n = (size_t)T * Epad;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / Epad), e = (int)(i % Epad);
    dst[i] = __float2bfloat16_rn(e < E ? src[(size_t)t * E + e] : 0.f);
  }
}
}  // namespace

cudaError_t launch_to_bf16_padded(const float* src, int T, int E, int Epad, __nv_bfloat16* dst,
                                  cudaStream_t st) {
  const size_t n = (size_t)T * Epad;
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  TraceScope ts("router_dlogits_bf16", st);
  to_bf16_padded_kernel<<<blocks, 256, 0, st>>>(src, T, E, Epad, dst);
  return cudaGetLastError();
}

}  // namespace moe
