// rowops.cuh -- row-level memory operations shared by the stand-alone
// gather / merge kernels (gather_merge.cu) and the persistent ring forward
// kernel (ring.cu).
//
// merge_token: the final weighted merge of one token (leiphone "MoK..."
// section 03, last step of the benchmarked layer): out[t] = sum over slots j
// (in slot order, fp32, fma) of w[t,j] * rows[pos_pad[t*k+j]], rounded once to
// bf16.  With w == nullptr the plain sum (the backward's reverse dispatch).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Coherent (L2) load: for data written earlier in the same kernel by other CTAs.
__device__ __forceinline__ uint4 ldcg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void stg_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// The same store with an L2 cache policy (createpolicy) for the line.
__device__ __forceinline__ void stg_v4_hint(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// Merge token t with threads [tid0, tid0 + nthr) of the block, each owning
// 8-column vectors.  sp / sw hold the token's k padded row positions and
// weights.  COHERENT selects L2 loads for rows written in the same kernel.
template <bool COHERENT>
__device__ __forceinline__ void merge_token(const __nv_bfloat16* __restrict__ rows, const int* sp,
                                            const float* sw, bool weighted, int t, int k, int d,
                                            __nv_bfloat16* __restrict__ out, int tid0, int nthr) {
  const int nvec = d >> 3;
  for (int v = tid0; v < nvec; v += nthr) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    // the slots' rows 8 at a time: loads first (in flight together), then
    // the sums in slot order
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint4 y[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u < k) {
          const void* src = rows + (size_t)sp[j0 + u] * d + (size_t)v * 8;
          y[u] = COHERENT ? ldcg_v4(src) : ldg_nc_v4(src);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u >= k) break;
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&y[u]);
        const float g = sw[j0 + u];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(h[i]);
          if (weighted) {
            acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
          } else {
            acc[2 * i] += f.x;
            acc[2 * i + 1] += f.y;
          }
        }
      }
    }
    uint4 o;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0], acc[1]);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2], acc[3]);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[4], acc[5]);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(acc[6], acc[7]);
    o.x = *reinterpret_cast<uint32_t*>(&p0);
    o.y = *reinterpret_cast<uint32_t*>(&p1);
    o.z = *reinterpret_cast<uint32_t*>(&p2);
    o.w = *reinterpret_cast<uint32_t*>(&p3);
    stg_v4(out + (size_t)t * d + (size_t)v * 8, o);
  }
}

}  // namespace moe
