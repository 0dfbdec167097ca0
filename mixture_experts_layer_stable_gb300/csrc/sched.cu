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
#include "ptx.cuh"

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

// Top-k of chunk b's tokens (one warp per token) with the chunk's
// histogram written to hist row b; true in the block that finishes last
// (atomic ticket), which then owns the table.  sh: kMaxE ints of shared memory.
template <int NCH>
__device__ __forceinline__ bool topk_hist_chunk(const float* __restrict__ logits, int T, int E, int k,
                                                int tb, int b, int nb, int* __restrict__ ids,
                                                float* __restrict__ wts, int* __restrict__ hist,
                                                int* __restrict__ hdr, int* sh, int* s_last) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int e = tid; e < E; e += blockDim.x) sh[e] = 0;
  __syncthreads();
  const int t0 = b * tb, t1 = min(T, t0 + tb);
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
  for (int e = tid; e < E; e += blockDim.x) hist[(size_t)b * E + e] = sh[e];
  __threadfence();
  __syncthreads();
  if (tid == 0) *s_last = (atomicAdd(hdr + kHdrDone, 1) == nb - 1);
  __syncthreads();
  const bool last = *s_last != 0;
  if (last) __threadfence();
  return last;
}

// Top-k with the per-chunk histogram, then the table in the last block (see
// the file comment).
template <int NCH>
__global__ void __launch_bounds__(kSchedThreads) sched_topk_hist_kernel(
    const float* __restrict__ logits, int T, int E, int k, int tb, int* __restrict__ ids,
    float* __restrict__ wts, int* __restrict__ hist, int* __restrict__ hdr, int* __restrict__ counts,
    int* __restrict__ offsets, int* __restrict__ poff, int* __restrict__ mt_off,
    int* __restrict__ pt_off) {
  __shared__ int sh[kMaxE];
  __shared__ int aux[kSchedThreads];
  __shared__ int sh_last;
  if (topk_hist_chunk<NCH>(logits, T, E, k, tb, blockIdx.x, gridDim.x, ids, wts, hist, hdr, sh, &sh_last))
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

// Stable positions of chunk b's rows (rows [b cr, (b+1) cr)): ranks within
// the chunk by warp match and per-warp prefixes, offset by the chunk's
// exclusive prefix; the padding rows of the experts this block owns (every
// nb-th from b).  wcnt: kWarps x kMaxE ints of shared memory.
__device__ __forceinline__ void scatter_chunk(
    const int* __restrict__ ids, const float* __restrict__ wts, int R, int E,
    const int* __restrict__ hist_prefix, const int* __restrict__ counts,
    const int* __restrict__ offsets, const int* __restrict__ poff, int* __restrict__ perm,
    int* __restrict__ inv, int* __restrict__ pos_pad, int* __restrict__ row_of_pad,
    float* __restrict__ g_pad, int cr, int b, int nb, int (*wcnt)[kMaxE]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int r_begin = b * cr;
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
      const int within = hist_prefix[(size_t)b * E + e] + local;
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
  for (int e = b; e < E; e += nb) {
    const int c = counts[e];
    const int pc = (c + kBM - 1) / kBM * kBM;
    for (int i = c + tid; i < pc; i += blockDim.x) {
      row_of_pad[poff[e] + i] = -1;
      g_pad[poff[e] + i] = 0.f;
    }
  }
}

__global__ void __launch_bounds__(kSchedThreads) sched_scatter_kernel(
    const int* __restrict__ ids, const float* __restrict__ wts, int R, int E,
    const int* __restrict__ hist_prefix, const int* __restrict__ counts,
    const int* __restrict__ offsets, const int* __restrict__ poff, int* __restrict__ perm,
    int* __restrict__ inv, int* __restrict__ pos_pad, int* __restrict__ row_of_pad,
    float* __restrict__ g_pad, int cr) {
  __shared__ int wcnt[kWarps][kMaxE];
  scatter_chunk(ids, wts, R, E, hist_prefix, counts, offsets, poff, perm, inv, pos_pad, row_of_pad, g_pad,
                cr, blockIdx.x, gridDim.x, wcnt);
}

// The whole schedule in one cooperative launch (every block co-resident):
// each block's top-k and histogram, the table in the last block to finish,
// which then releases the others (a header flag, waited on with a bound),
// and every block's scatter of its own chunk.  Saves the second launch.
template <int NCH>
__global__ void __launch_bounds__(kSchedThreads) sched_fused_kernel(
    const float* __restrict__ logits, int T, int E, int k, int tb, int* __restrict__ ids,
    float* __restrict__ wts, int* __restrict__ hist, int* __restrict__ hdr, int* __restrict__ counts,
    int* __restrict__ offsets, int* __restrict__ poff, int* __restrict__ mt_off,
    int* __restrict__ pt_off, int* __restrict__ perm, int* __restrict__ inv, int* __restrict__ pos_pad,
    int* __restrict__ row_of_pad, float* __restrict__ g_pad) {
  __shared__ int sh[kMaxE];
  __shared__ int aux[kSchedThreads];
  __shared__ int wcnt[kWarps][kMaxE];
  __shared__ int sh_last, s_ok;
  const int nb = gridDim.x;
  const bool last = topk_hist_chunk<NCH>(logits, T, E, k, tb, blockIdx.x, nb, ids, wts, hist, hdr, sh, &sh_last);
  if (last) {
    finish_histograms(hist, nb, E, hdr, counts, offsets, poff, mt_off, pt_off, sh, aux);
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      red_release_add(hdr + kHdrSchedGo, 1);
    }
  }
  if (threadIdx.x == 0) {
    bool ok = true;
    if (!last && ld_acquire(hdr + kHdrSchedGo) == 0) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire(hdr + kHdrSchedGo) == 0) {
        __nanosleep(64);
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          report_status(hdr + kHdrStatus, kStatusTimeout, 950);
          ok = false;
          break;
        }
      }
    }
    s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  if (!s_ok) return;
  scatter_chunk(ids, wts, T * k, E, hist, counts, offsets, poff, perm, inv, pos_pad, row_of_pad, g_pad,
                tb * k, blockIdx.x, nb, wcnt);
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

namespace {
// Blocks of sched_fused_kernel<NCH> that fit on the GPU at once (0 if unknown).
template <int NCH>
int fused_capacity() {
  static int cap = -1;
  if (cap < 0) {
    int per_sm = 0;
    cap = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sched_fused_kernel<NCH>, kSchedThreads, 0) ==
                  cudaSuccess
              ? per_sm * num_sms()
              : 0;
  }
  return cap;
}

template <int NCH>
cudaError_t schedule_chunks(const moe_config& c, const float* logits, const moe_sched& s, const Ws& ws,
                            cudaStream_t st) {
  const int nb = (int)ws.L.nblk, tb = sched_chunk_tokens(c.T, c.k);
  if (nb <= fused_capacity<NCH>()) {
    // one cooperative launch: every block is resident while the others wait
    TraceScope ts("sched_fused", st);
    const float* lg = logits;
    int T = c.T, E = c.E, k = c.k, tbv = tb;
    int* ids = s.topk_ids;
    float* wts = s.topk_w;
    int* hist = ws.hist();
    int* hdr = ws.hdr();
    int* counts = s.counts;
    int* offsets = s.offsets;
    int* poff = ws.poff();
    int* mt_off = ws.mt_off();
    int* pt_off = ws.pt_off();
    int* perm = s.perm;
    int* inv = s.inv;
    int* pos_pad = ws.pos_pad();
    int* row_of_pad = ws.row_of_pad();
    float* g_pad = ws.g_pad();
    void* args[] = {&lg, &T, &E, &k, &tbv, &ids, &wts, &hist, &hdr, &counts, &offsets, &poff,
                    &mt_off, &pt_off, &perm, &inv, &pos_pad, &row_of_pad, &g_pad};
    const cudaError_t e = cudaLaunchCooperativeKernel((const void*)sched_fused_kernel<NCH>, dim3(nb),
                                                      dim3(kSchedThreads), args, 0, st);
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    (void)cudaGetLastError();  // not resident after all: the two-launch form below
  }
  cudaError_t err;
  {
    TraceScope ts("sched_topk_hist", st);
    sched_topk_hist_kernel<NCH><<<nb, kSchedThreads, 0, st>>>(logits, c.T, c.E, c.k, tb, s.topk_ids, s.topk_w,
                                                              ws.hist(), ws.hdr(), s.counts, s.offsets,
                                                              ws.poff(), ws.mt_off(), ws.pt_off());
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) return err;
  return launch_scatter(c, s, ws, st);
}
}  // namespace

// The header must have been cleared (launch_schedule and moe_route do).
cudaError_t launch_schedule_from_logits(const moe_config& c, const float* logits, const moe_sched& s,
                                        const Ws& ws, cudaStream_t st) {
  if (c.E <= 32) return schedule_chunks<1>(c, logits, s, ws, st);
  if (c.E <= 64) return schedule_chunks<2>(c, logits, s, ws, st);
  if (c.E <= 128) return schedule_chunks<4>(c, logits, s, ws, st);
  if (c.E <= 256) return schedule_chunks<8>(c, logits, s, ws, st);
  return schedule_chunks<kMaxE / 32>(c, logits, s, ws, st);
}

cudaError_t launch_schedule(const moe_config& c, const float* logits, const moe_sched& s,
                            const Ws& ws, cudaStream_t st) {
  cudaError_t err = cudaMemsetAsync(ws.hdr(), 0, kHdrWords * sizeof(int), st);
  if (err == cudaSuccess) err = launch_schedule_from_logits(c, logits, s, ws, st);
  return err;
}

}  // namespace moe
