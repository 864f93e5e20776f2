// argmax.cuh -- greedy-argmax reduction shared by the fused decode epilogue
// and the stand-alone argmax kernel.
//
// The order: a NaN logit ranks above every number (the first NaN wins, as a
// NaN-propagating argmax reports it); otherwise the larger value wins, and
// equal values go to the lower index ("Pushing the limits of legacy
// hardware", section "Build the execution path, then share the weights": the
// fused greedy head keeps each tile's maximum with its original index, so the
// reduction must not depend on which tile finishes first).  The order is a
// total order on (value, index) pairs, so any reduction tree gives the same
// winner.
#pragma once
#include <cstdint>

#include "qmm_launch.h"

namespace qmm {

__device__ __forceinline__ bool am_better(float v1, int i1, float v2, int i2) {
  const bool n1 = isnan(v1), n2 = isnan(v2);
  if (n1 != n2) return n1;
  if (!n1 && v1 != v2) return v1 > v2;
  return i1 < i2;
}

__device__ __forceinline__ void am_warp_reduce(float &v, int &i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (am_better(ov, oi, v, i)) v = ov, i = oi;
  }
}

// Called by every thread of `nwarps` consecutive full warps starting at warp
// `warp0` of the CTA, each with its own candidate (v, i).  `scratch` holds
// 2 * nwarps words of shared memory; `bar_id` / `nthreads` name a barrier
// those warps (and only they) use.  The CTA's winner goes to the work
// arrays; the last CTA to finish combines all CTAs' winners, writes the
// result and resets the counter, so the work area is ready for the next call.
__device__ __forceinline__ void am_cta_finish(float v, int i, int warp0, int nwarps, uint32_t *scratch,
                                              int bar_id, int nthreads, const ArgmaxWork &w) {
  const int warp = (threadIdx.x >> 5) - warp0, lane = threadIdx.x & 31;
  am_warp_reduce(v, i);
  if (lane == 0) {
    scratch[2 * warp] = __float_as_uint(v);
    scratch[2 * warp + 1] = (uint32_t)i;
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(nthreads) : "memory");
  if (warp != 0) return;
  v = lane < nwarps ? __uint_as_float(scratch[2 * lane]) : __int_as_float(0xFF800000);   // -inf
  i = lane < nwarps ? (int)scratch[2 * lane + 1] : 0x7FFFFFFF;
  am_warp_reduce(v, i);
  unsigned done = 0;
  if (lane == 0) {
    w.part_val[blockIdx.x] = v;
    w.part_idx[blockIdx.x] = i;
    __threadfence();                                   // the winner is visible before the count
    done = atomicAdd(w.counter, 1u);
  }
  done = __shfl_sync(0xffffffffu, done, 0);
  if (done != gridDim.x - 1) return;
  // the last CTA: every other CTA's winner is visible (fence before each count)
  __threadfence();
  float bv = __int_as_float(0xFF800000);
  int bi = 0x7FFFFFFF;
  for (int c = lane; c < (int)gridDim.x; c += 32) {
    const float cv = __ldcg(w.part_val + c);
    const int ci = __ldcg(w.part_idx + c);
    if (am_better(cv, ci, bv, bi)) bv = cv, bi = ci;
  }
  am_warp_reduce(bv, bi);
  if (lane == 0) {
    *w.out_idx = bi;
    if (w.out_val) *w.out_val = bv;
    *w.counter = 0u;
  }
}

}  // namespace qmm
