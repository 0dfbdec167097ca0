// bulk_rows.cuh -- one warp's share of a row gather staged through shared
// memory with bulk copies (the TMA engine's untiled global <-> shared copies).
//
// Each warp owns nbw row buffers (one mbarrier each).  Lane 0 loads up to
// nbw rows ahead; a row leaves by a bulk store once its load has landed, and
// the buffer of the row `depth` items back is refilled as soon as that row's
// store has read it, so loads and stores of one warp overlap.  The source
// rows of 32 items at a time are read by the 32 lanes and shuffled to lane 0.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace moe {

constexpr int kRowZero = -1;  // item code: write a zero row
constexpr int kRowSkip = -2;  // item code: nothing to write

struct RowPipe {
  uint32_t wbuf;    // shared address of this warp's first row buffer
  uint32_t zrow;    // shared address of a zero row
  uint32_t rb;      // bytes per row (multiple of 16)
  uint64_t* bars;   // nbw mbarriers
  int nbw, depth;   // buffers, stores in flight before a refill waits (< nbw, <= 8)
  uint32_t ph;      // lane 0: phase parity per buffer
  uint32_t pend;    // lane 0: buffers with a load in flight
};

// Copies items 0..n-1 (warp-uniform call).  code_of(i), called per lane for
// any i < n, returns the item's code: >= 0 a source row, kRowZero, kRowSkip.
// src_of(code) and dst_of(i) give global addresses (16-byte aligned).
// Returns false when a bounded wait gave up; the caller then waits for the
// buffers in rp.pend before leaving.  Lane 0 still has stores in flight on
// return: a bulk_wait<0>() makes them visible.
template <class Code, class Src, class Dst>
__device__ __forceinline__ bool bulk_rows(RowPipe& rp, int n, Code code_of, Src src_of, Dst dst_of,
                                          volatile int* abort_flag, int* status, int where) {
  const int lane = threadIdx.x & 31;
  int c0 = 0;
  int ia = lane < n ? code_of(lane) : kRowSkip;
  int ib = 32 + lane < n ? code_of(32 + lane) : kRowSkip;
  auto code_at = [&](int i) { return __shfl_sync(0xffffffffu, (i - c0) < 32 ? ia : ib, (i - c0) & 31); };
  auto issue = [&](int i) {
    const int r = code_at(i);
    if (lane == 0 && r >= 0) {
      const int b = i % rp.nbw;
      mbar_arrive_expect_tx(&rp.bars[b], rp.rb);
      bulk_load(rp.wbuf + (uint32_t)b * rp.rb, src_of(r), rp.rb, smem_u32(&rp.bars[b]));
      rp.pend |= 1u << b;
    }
  };
  for (int i = 0; i < min(rp.nbw, n); ++i) issue(i);
  uint32_t stored = 0, frombuf = 0;  // lane 0: bit j set when item i - j committed a store / read its buffer
  for (int i = 0; i < n; ++i) {
    if (i - c0 == 32) {
      c0 += 32;
      ia = ib;
      ib = c0 + 32 + lane < n ? code_of(c0 + 32 + lane) : kRowSkip;
    }
    const int r = code_at(i);
    int ok = 1;
    if (lane == 0) {
      const int b = i % rp.nbw;
      uint32_t src = rp.zrow;
      if (r >= 0) {
        ok = mbar_wait(&rp.bars[b], (rp.ph >> b) & 1u, abort_flag, status, where);
        if (ok) {
          rp.ph ^= 1u << b;
          rp.pend &= ~(1u << b);
          src = rp.wbuf + (uint32_t)b * rp.rb;
        }
      }
      stored <<= 1;
      frombuf <<= 1;
      if (ok && r != kRowSkip) {
        bulk_store(dst_of(i), src, rp.rb);
        bulk_commit();
        stored |= 1u;
        frombuf |= r >= 0 ? 1u : 0u;
      }
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
    // refill the buffer of item i - depth with item i - depth + nbw
    const int j = i - rp.depth;
    if (j >= 0 && j + rp.nbw < n) {
      if (lane == 0 && ((frombuf >> rp.depth) & 1u))
        bulk_wait_read_n(__popc(stored & ((1u << rp.depth) - 1u)));  // stores committed after item j's
      issue(j + rp.nbw);
    }
  }
  return true;
}

}  // namespace moe
