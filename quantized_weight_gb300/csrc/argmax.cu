// argmax.cu -- greedy argmax over rows of float32 logits (the unfused path of
// qmm_gemv_argmax, used when the fused decode epilogue does not apply).
//
// One CTA per row: 1024 threads stride over the row, then warp shuffles and
// one warp combine the candidates under the order of argmax.cuh.
#include "argmax.cuh"
#include "qmm_launch.h"

namespace qmm {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads) argmax_rows_kernel(const float *__restrict__ logits, int64_t N,
                                                                int32_t *__restrict__ idx,
                                                                float *__restrict__ val) {
  __shared__ uint32_t scratch[2 * (kThreads / 32)];
  const int m = blockIdx.x;
  const float *row = logits + (int64_t)m * N;
  float bv = __int_as_float(0xFF800000);
  int bi = 0x7FFFFFFF;
  for (int64_t n = threadIdx.x; n < N; n += kThreads) {
    const float v = row[n];
    if (am_better(v, (int)n, bv, bi)) bv = v, bi = (int)n;
  }
  am_warp_reduce(bv, bi);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    scratch[2 * warp] = __float_as_uint(bv);
    scratch[2 * warp + 1] = (uint32_t)bi;
  }
  __syncthreads();
  if (warp != 0) return;
  bv = __uint_as_float(scratch[2 * lane]);
  bi = (int)scratch[2 * lane + 1];
  am_warp_reduce(bv, bi);
  if (lane == 0) {
    idx[m] = bi;
    if (val) val[m] = bv;
  }
}

}  // namespace

cudaError_t launch_argmax_rows(const float *logits, int M, int64_t N, int32_t *idx, float *val, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  argmax_rows_kernel<<<M, kThreads, 0, s>>>(logits, N, idx, val);
  return cudaGetLastError();
}

}  // namespace qmm
