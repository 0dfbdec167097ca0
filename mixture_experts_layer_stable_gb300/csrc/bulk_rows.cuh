// bulk_rows.cuh -- one warp's share of a row gather staged through shared
// memory with bulk copies (the TMA engine's untiled global <-> shared copies).
//
// Each warp owns nbw row buffers (one mbarrier each).  Lane 0 loads up to
// nbw rows ahead; a row leaves by one or more bulk stores (one per
// destination) once its load has landed, and the buffer of the row `depth`
// items back is refilled as soon as that row's stores have read it, so loads
// and stores of one warp overlap.  The codes of 32 items at a time are read
// by the 32 lanes and shuffled to lane 0.
#pragma once

#include <stdint.h>

#include <type_traits>

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
  uint32_t ph;      // lane 0 (every lane with a transformation): phase parity per buffer
  uint32_t pend;    // lane 0: buffers with a load in flight
  // L2 cache policies (createpolicy) of the loads and stores, each used when
  // its bit of `hints` is set (bit 0: loads, bit 1: stores)
  uint64_t ld_pol, st_pol;
  uint32_t hints;
};

// No transformation of a landed row: its rb bytes are stored as loaded.
struct RowAsIs {
  __device__ __forceinline__ void operator()(int, int, uint32_t) const {}
};

// Copies items 0..n-1 (warp-uniform call).  code_of(i), called per lane for
// any i < n, returns the item's code: >= 0 a source row, kRowZero, kRowSkip.
// src_of(code) gives the source address; dst_of(i, j), called by lane j for
// j < fan, the item's j-th destination, or nullptr for none (all 16-byte
// aligned).  xform(i, code, buf), called by every lane once the item's row
// (code >= 0) has landed in the buffer at shared address buf, may rewrite
// the buffer in place; then st_bytes (<= rb, a multiple of 16) bytes of it
// (of the zero row for kRowZero) go to every destination.
// Returns false when a bounded wait gave up; the caller then waits for the
// buffers in rp.pend before leaving.  Lane 0 still has stores in flight on
// return: a bulk_wait<0>() makes them visible.
template <class Code, class Src, class Dst, class Xform>
__device__ __forceinline__ bool bulk_rows_fan(RowPipe& rp, int n, int fan, uint32_t st_bytes,
                                              Code code_of, Src src_of, Dst dst_of, Xform xform,
                                              volatile int* abort_flag, int* status, int where) {
  // a transformation reads the landed row in every lane: every lane then
  // waits on the buffer's barrier itself (acquiring the copy's bytes)
  constexpr bool kAllWait = !std::is_same<Xform, RowAsIs>::value;
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
      if (rp.hints & 1u)
        bulk_load_hint(rp.wbuf + (uint32_t)b * rp.rb, src_of(r), rp.rb, smem_u32(&rp.bars[b]), rp.ld_pol);
      else
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
    const int b = i % rp.nbw;
    int ok = 1;
    if (r >= 0 && (kAllWait || lane == 0)) {
      ok = mbar_wait(&rp.bars[b], (rp.ph >> b) & 1u, abort_flag, status, where);
      if (ok) {
        rp.ph ^= 1u << b;
        rp.pend &= ~(1u << b);
      }
    }
    if (kAllWait ? !__all_sync(0xffffffffu, ok) : !__shfl_sync(0xffffffffu, ok, 0)) return false;
    const uint32_t src = r >= 0 ? rp.wbuf + (uint32_t)b * rp.rb : rp.zrow;
    if (r != kRowSkip) xform(i, r, src);
    // destinations: lane j holds the j-th
    const uint64_t dl = (r != kRowSkip && lane < fan) ? reinterpret_cast<uint64_t>(dst_of(i, lane)) : 0ull;
    int nst = 0;
    for (int j = 0; j < fan; ++j) {
      const uint64_t dp = __shfl_sync(0xffffffffu, dl, j);
      if (lane == 0 && dp != 0ull) {
        if (rp.hints & 2u)
          bulk_store_hint(reinterpret_cast<void*>(dp), src, st_bytes, rp.st_pol);
        else
          bulk_store(reinterpret_cast<void*>(dp), src, st_bytes);
        ++nst;
      }
    }
    if (lane == 0) {
      stored <<= 1;
      frombuf <<= 1;
      if (nst > 0) {
        bulk_commit();
        stored |= 1u;
        frombuf |= r >= 0 ? 1u : 0u;
      }
    }
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

// One destination per item: dst_of(i).
template <class Code, class Src, class Dst>
__device__ __forceinline__ bool bulk_rows(RowPipe& rp, int n, Code code_of, Src src_of, Dst dst_of,
                                          volatile int* abort_flag, int* status, int where) {
  return bulk_rows_fan(
      rp, n, 1, rp.rb, code_of, src_of, [&](int i, int) { return dst_of(i); }, RowAsIs(), abort_flag,
      status, where);
}

}  // namespace moe
