// sched.cu -- routing and schedule table on the GPU.
//
// Routing: each token picks its top-k experts afresh every step (leiphone
// "MoK..." section 01).  The schedule table counts rows per expert, places
// every row and keeps an expert's rows contiguous for the grouped GEMM
// (same section; Marktechpost "Cursor开源MoK..." three design decisions:
// one table serves all four transfer modes, at < 3 % of the MoE runtime).
//
// Two kernels after a clear of the header words, no host synchronisation.
// Rows are handled in chunks of sched_chunk_tokens(T, k) tokens (their k rows
// each, at most kSchedChunk rows, about kSchedBlocks chunks for small T):
//  1. sched_topk_hist: per chunk, one warp per token runs k rounds of a warp
//     arg-max over the E fp32 logits (value descending, id ascending);
//     weights = softmax over the k selected logits in fp32, summed in slot
//     order; the chunk's integer histogram over experts is counted in shared
//     memory.  The last block to finish (atomic ticket) turns the chunk
//     histograms into per-chunk exclusive prefixes and computes counts,
//     offsets and the padded layout (each expert's segment rounded up to 128
//     rows; prefixes over experts of their 128-row tiles and of their pairs
//     of tiles).  Integer sums do not depend on order, so the table is
//     deterministic.  (sched_hist does the histogram part alone, for ids
//     chosen elsewhere: the router GEMM's fused top-k.)
//  2. sched_scatter: every chunk re-walks its rows in index order and ranks
//     each row among the earlier rows of the same expert (warp match + prefix
//     over warps), which makes the permutation stable without atomics.
#include <cuda_bf16.h>
#include <math.h>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kWarps = kSchedThreads / 32;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return (v > bv) || (v == bv && i < bi);
}

// Logits of token t for one warp: NCH chunks of 32 per lane (E <= 32 NCH);
// zeros past E (excluded from the top-k by topk_token).
template <int NCH>
__device__ __forceinline__ void load_logits(const float* __restrict__ logits, int t, int E, int lane,
                                            float (&v)[NCH]) {
  const float* zrow = logits + (size_t)t * E;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int e = c * 32 + lane;
    v[c] = e < E ? __ldg(zrow + e) : 0.f;
  }
}

// Top-k of one token's logits v (load_logits) by one warp: lane j < k
// returns the j-th pick in *id and its weight in *w.
template <int NCH>
__device__ __forceinline__ void topk_token(const float (&v)[NCH], int E, int k, int lane, int* id,
                                           float* w) {
  uint32_t taken = 0;
#pragma unroll
  for (int c = 0; c < NCH; ++c)
    if (c * 32 + lane >= E) taken |= 1u << c;
  int my_id = 0;
  float my_v = 0.f;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      if (!((taken >> c) & 1u) && better(v[c], c * 32 + lane, bv, bi)) {
        bv = v[c];
        bi = c * 32 + lane;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == r) {
      my_id = bi;
      my_v = bv;
    }
  }
  // weights: exp(z_j - z_0) / sum_l exp(z_l - z_0), summed in slot order
  const float z0 = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - z0) : 0.f;
  float s = 0.f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ex, j);
  *id = my_id;
  *w = ex / s;
}

// Per-expert exclusive prefix, in place, over chunks [c0, c1) of the chunk
// histograms, starting from `run`; returns the running sum.  Loads go out 32
// at a time so that their latencies overlap.
__device__ __forceinline__ int prefix_chunks(int* __restrict__ hist, int E, int e, int c0, int c1,
                                             int run) {
  for (int b0 = c0; b0 < c1; b0 += 32) {
    int c[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) c[u] = (b0 + u < c1) ? __ldcg(hist + (size_t)(b0 + u) * E + e) : 0;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      if (b0 + u < c1) hist[(size_t)(b0 + u) * E + e] = run;
      run += c[u];
    }
  }
  return run;
}

__device__ __forceinline__ int sum_chunks(const int* __restrict__ hist, int E, int e, int c0, int c1) {
  int run = 0;
  for (int b0 = c0; b0 < c1; b0 += 32) {
    int c[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) c[u] = (b0 + u < c1) ? __ldcg(hist + (size_t)(b0 + u) * E + e) : 0;
#pragma unroll
    for (int u = 0; u < 32; ++u) run += c[u];
  }
  return run;
}

// The last block of a chunked histogram pass: per-expert exclusive prefixes
// over the chunks (in place), counts, offsets and the padded layout.
// sh: kMaxE ints, aux: blockDim.x ints of shared memory (G * E <= blockDim.x).
__device__ void finish_histograms(int* __restrict__ hist, int nb, int E, int* __restrict__ hdr,
                                  int* __restrict__ counts, int* __restrict__ offsets,
                                  int* __restrict__ poff, int* __restrict__ mt_off,
                                  int* __restrict__ pt_off, int* sh, int* aux) {
  const int tid = threadIdx.x;
  // G thread groups split the chunks of every expert: group q sums chunks
  // [q*len, (q+1)*len), then writes their prefixes from its start
  const int G = E >= (int)blockDim.x ? 1 : min(8, (int)blockDim.x / E);
  const int len = (nb + G - 1) / G;
  const int q = tid / E;
  if (G > 1) {
    if (q < G) {
      const int e = tid - q * E;
      aux[q * E + e] = sum_chunks(hist, E, e, min(nb, q * len), min(nb, (q + 1) * len));
    }
    __syncthreads();
    if (q < G) {
      const int e = tid - q * E;
      int start = 0;
      for (int j = 0; j < q; ++j) start += aux[j * E + e];
      prefix_chunks(hist, E, e, min(nb, q * len), min(nb, (q + 1) * len), start);
      if (q == 0) {
        int tot = 0;
        for (int j = 0; j < G; ++j) tot += aux[j * E + e];
        sh[e] = tot;
        counts[e] = tot;
      }
    }
  } else {
    for (int e = tid; e < E; e += blockDim.x) {
      const int tot = prefix_chunks(hist, E, e, 0, nb, 0);
      sh[e] = tot;
      counts[e] = tot;
    }
  }
  __syncthreads();
  if (tid < 32) {
    // prefixes over experts, one warp: lane l takes experts [l*per, (l+1)*per).
    // Per expert: its rows; its padded rows (128-row tiles); pt_off: work
    // units of the CTA-pair GEMMs (pairs of 128-row tiles, an odd last tile
    // alone); hv_off / lt_off split them into heavy units and light ones (an
    // odd last tile of at most kLightRows rows)
    int* hv_off = pt_off + (E + 1);
    int* lt_off = hv_off + (E + 1);
    const int lane = tid;
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    auto sizes = [&](int e, int& o, int& po, int& pt, int& hv, int& lt) {
      const int c = sh[e];
      const int mt = (c + kBM - 1) / kBM;
      const int light = ((mt & 1) && c - (mt - 1) * kBM <= kLightRows) ? 1 : 0;
      o = c;
      po = mt * kBM;
      pt = (mt + 1) >> 1;
      hv = pt - light;
      lt = light;
    };
    int v[5] = {0, 0, 0, 0, 0};
    for (int e = e0; e < e1; ++e) {
      int d[5];
      sizes(e, d[0], d[1], d[2], d[3], d[4]);
#pragma unroll
      for (int i = 0; i < 5; ++i) v[i] += d[i];
    }
    // exclusive scan of the lanes' sums
    int x[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      int inc = v[i];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
      }
      x[i] = inc - v[i];
    }
    for (int e = e0; e < e1; ++e) {
      offsets[e] = x[0];
      poff[e] = x[1];
      mt_off[e] = x[1] / kBM;
      pt_off[e] = x[2];
      hv_off[e] = x[3];
      lt_off[e] = x[4];
      int d[5];
      sizes(e, d[0], d[1], d[2], d[3], d[4]);
#pragma unroll
      for (int i = 0; i < 5; ++i) x[i] += d[i];
    }
    if (lane == 31) {
      offsets[E] = x[0];
      poff[E] = x[1];
      mt_off[E] = x[1] / kBM;
      pt_off[E] = x[2];
      hv_off[E] = x[3];
      lt_off[E] = x[4];
      hdr[kHdrRpTotal] = x[1];
      hdr[kHdrMtTotal] = x[1] / kBM;
      hdr[kHdrDone] = 0;
    }
  }
}

// Top-k of the chunk's tokens (one warp per token) with the chunk's
// histogram, then the table in the last block (see the file comment).
template <int NCH>
__global__ void __launch_bounds__(kSchedThreads) sched_topk_hist_kernel(
    const float* __restrict__ logits, int T, int E, int k, int tb, int* __restrict__ ids,
    float* __restrict__ wts, int* __restrict__ hist, int* __restrict__ hdr, int* __restrict__ counts,
    int* __restrict__ offsets, int* __restrict__ poff, int* __restrict__ mt_off,
    int* __restrict__ pt_off) {
  __shared__ int sh[kMaxE];
  __shared__ int aux[kSchedThreads];
  __shared__ int sh_last;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * tb, t1 = min(T, t0 + tb);
  // the next token's logits are loaded while this one's top-k runs
  float v[NCH] = {}, vn[NCH] = {};
  int t = t0 + (tid >> 5);
  if (t < t1) load_logits<NCH>(logits, t, E, lane, v);
  for (; t < t1; t += kWarps) {
    if (t + kWarps < t1) load_logits<NCH>(logits, t + kWarps, E, lane, vn);
    int id;
    float w;
    topk_token<NCH>(v, E, k, lane, &id, &w);
#pragma unroll
    for (int c = 0; c < NCH; ++c) v[c] = vn[c];
    if (lane < k) {
      ids[(size_t)t * k + lane] = id;
      wts[(size_t)t * k + lane] = w;
      atomicAdd(&sh[id], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh[e];
  __threadfence();
  __syncthreads();
  if (tid == 0) sh_last = (atomicAdd(hdr + kHdrDone, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  finish_histograms(hist, gridDim.x, E, hdr, counts, offsets, poff, mt_off, pt_off, sh, aux);
}

__global__ void __launch_bounds__(kSchedThreads) sched_hist_kernel(
    const int* __restrict__ ids, int R, int E, int cr, int* __restrict__ hist, int* __restrict__ hdr,
    int* __restrict__ counts, int* __restrict__ offsets, int* __restrict__ poff,
    int* __restrict__ mt_off, int* __restrict__ pt_off) {
  __shared__ int sh[kMaxE];
  __shared__ int aux[kSchedThreads];
  __shared__ int sh_last;
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int r0 = blockIdx.x * cr, r1 = min(R, r0 + cr);
  for (int r = r0 + tid; r < r1; r += blockDim.x) atomicAdd(&sh[ids[r]], 1);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = sh[e];
  __threadfence();
  __syncthreads();
  if (tid == 0) sh_last = (atomicAdd(hdr + kHdrDone, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  finish_histograms(hist, gridDim.x, E, hdr, counts, offsets, poff, mt_off, pt_off, sh, aux);
}

__global__ void __launch_bounds__(kSchedThreads) sched_scatter_kernel(
    const int* __restrict__ ids, const float* __restrict__ wts, int R, int E,
    const int* __restrict__ hist_prefix, const int* __restrict__ counts,
    const int* __restrict__ offsets, const int* __restrict__ poff, int* __restrict__ perm,
    int* __restrict__ inv, int* __restrict__ pos_pad, int* __restrict__ row_of_pad,
    float* __restrict__ g_pad, int cr) {
  __shared__ int wcnt[kWarps][kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r_begin = blockIdx.x * cr;
  const int r_end = min(R, r_begin + cr);
  const int per_warp = (r_end - r_begin + kWarps - 1) / kWarps;
  const int w_begin = r_begin + warp * per_warp;
  const int w_end = min(r_end, w_begin + per_warp);
  for (int i = tid; i < kWarps * E; i += blockDim.x) wcnt[i / E][i % E] = 0;
  __syncthreads();
  // pass 1: per-warp counts
  for (int base = w_begin; base < w_end; base += 32) {
    const int r = base + lane;
    const int e = (r < w_end) ? ids[r] : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp][e] += __popc(peers);
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcnt[w][e];
      wcnt[w][e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass 2: stable ranks
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int base = w_begin; base < w_end; base += 32) {
    const int r = base + lane;
    const int e = (r < w_end) ? ids[r] : -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int local = 0;
    if (e >= 0) local = wcnt[warp][e] + __popc(peers & lt_mask);
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp][e] += __popc(peers);
    __syncwarp();
    if (e >= 0) {
      const int within = hist_prefix[(size_t)blockIdx.x * E + e] + local;
      const int p = offsets[e] + within;
      const int pp = poff[e] + within;
      perm[p] = r;
      inv[r] = p;
      pos_pad[r] = pp;
      row_of_pad[pp] = r;
      g_pad[pp] = wts[r];
    }
  }
  // padding rows of the experts this block owns
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int c = counts[e];
    const int pc = (c + kBM - 1) / kBM * kBM;
    for (int i = c + tid; i < pc; i += blockDim.x) {
      row_of_pad[poff[e] + i] = -1;
      g_pad[poff[e] + i] = 0.f;
    }
  }
}

}  // namespace

namespace {
cudaError_t launch_scatter(const moe_config& c, const moe_sched& s, const Ws& ws, cudaStream_t st) {
  const int R = c.T * c.k;
  TraceScope ts("sched_scatter", st);
  sched_scatter_kernel<<<(int)ws.L.nblk, kSchedThreads, 0, st>>>(
      s.topk_ids, s.topk_w, R, c.E, ws.hist(), s.counts, s.offsets, ws.poff(), s.perm, s.inv,
      ws.pos_pad(), ws.row_of_pad(), ws.g_pad(), sched_chunk_tokens(c.T, c.k) * c.k);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_schedule_tail(const moe_config& c, const moe_sched& s, const Ws& ws,
                                 cudaStream_t st) {
  const int R = c.T * c.k;
  cudaError_t err;
  {
    TraceScope ts("sched_hist", st);
    sched_hist_kernel<<<(int)ws.L.nblk, kSchedThreads, 0, st>>>(
        s.topk_ids, R, c.E, sched_chunk_tokens(c.T, c.k) * c.k, ws.hist(), ws.hdr(), s.counts, s.offsets,
        ws.poff(), ws.mt_off(), ws.pt_off());
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) return err;
  return launch_scatter(c, s, ws, st);
}

cudaError_t launch_schedule_from_logits(const moe_config& c, const float* logits, const moe_sched& s,
                                        const Ws& ws, cudaStream_t st) {
  const int nb = (int)ws.L.nblk, tb = sched_chunk_tokens(c.T, c.k);
  cudaError_t err;
  {
    TraceScope ts("sched_topk_hist", st);
    auto args = [&](auto kern) {
      kern<<<nb, kSchedThreads, 0, st>>>(logits, c.T, c.E, c.k, tb, s.topk_ids, s.topk_w, ws.hist(),
                                         ws.hdr(), s.counts, s.offsets, ws.poff(), ws.mt_off(),
                                         ws.pt_off());
    };
    if (c.E <= 32) args(sched_topk_hist_kernel<1>);
    else if (c.E <= 64) args(sched_topk_hist_kernel<2>);
    else if (c.E <= 128) args(sched_topk_hist_kernel<4>);
    else if (c.E <= 256) args(sched_topk_hist_kernel<8>);
    else args(sched_topk_hist_kernel<kMaxE / 32>);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) return err;
  return launch_scatter(c, s, ws, st);
}

cudaError_t launch_schedule(const moe_config& c, const float* logits, const moe_sched& s,
                            const Ws& ws, cudaStream_t st) {
  cudaError_t err = cudaMemsetAsync(ws.hdr(), 0, kHdrWords * sizeof(int), st);
  if (err == cudaSuccess) err = launch_schedule_from_logits(c, logits, s, ws, st);
  return err;
}

}  // namespace moe
