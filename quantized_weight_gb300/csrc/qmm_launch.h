// qmm_launch.h -- internal launchers behind the C ABI (include/qmm.h).
//
// The ABI layer (api.cu) validates every argument before calling one of
// these; each launcher only picks a kernel configuration and enqueues it on
// the given stream, returning the cudaError_t of the launch.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace qmm {

// Work area of a fused greedy-argmax decode product (device memory).
struct ArgmaxWork {
  unsigned *counter;      // CTAs finished in this call: 0 before a call, reset to 0 by its last CTA
  float *part_val;        // [grid] per-CTA winners
  int32_t *part_idx;
  int32_t *out_idx;       // the result (one token)
  float *out_val;         // may be null
};
constexpr int kArgmaxMaxCtas = 1024;

cudaError_t launch_pack(const uint8_t *codes, uint32_t *packed, int64_t N, int64_t K, int bits,
                        cudaStream_t s);
cudaError_t launch_unpack(const uint32_t *packed, uint8_t *codes, int64_t N, int64_t K, int bits,
                          cudaStream_t s);
cudaError_t launch_dequant(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                           float *w, int64_t N, int64_t K, int bits, int group, cudaStream_t s);

// out[t, :] = dequant(W[ids[t], :]) for t < T; ids outside [0, N) give NaN rows.
cudaError_t launch_gather_dequant(const int32_t *ids, int64_t T, const uint32_t *packed, const uint16_t *scales,
                                  const uint16_t *biases, float *out, int64_t N, int64_t K, int bits, int group,
                                  cudaStream_t s);
// INT4 affine quantization of float32 w [N, K] (group in {32, 64, 128}).
cudaError_t launch_quantize(const float *w, uint32_t *packed, uint16_t *scales, uint16_t *biases, int64_t N,
                            int64_t K, int group, cudaStream_t s);

// Decode product, 1 <= M <= 8, K > 0, N > 0.
cudaError_t launch_gemv(const float *x, const uint32_t *codes, const uint16_t *scales,
                        const uint16_t *biases, float *y, int M, int64_t N, int64_t K, int bits,
                        int group, cudaStream_t s);

// Decode product for M == 1 (any format) or 2 <= M <= 4 (INT8) streamed
// through shared memory by bulk copies; returns cudaErrorNotSupported
// (nothing launched) for shapes outside its layout.
cudaError_t launch_gemv_stream(const float *x, const uint32_t *codes, const uint16_t *scales,
                               const uint16_t *biases, float *y, int M, int64_t N, int64_t K, int bits,
                               int group, cudaStream_t s);

// M == 1 decode product whose epilogue keeps only the argmax of y (no y is
// written); cudaErrorNotSupported (nothing launched) outside the streaming layout.
cudaError_t launch_gemv_stream_argmax(const float *x, const uint32_t *codes, const uint16_t *scales,
                                      const uint16_t *biases, int64_t N, int64_t K, int bits, int group,
                                      const ArgmaxWork &w, cudaStream_t s);
// The fused M == 1 greedy head: the tensor-core kernel for INT4 (as
// launch_gemv), the streamed kernel first for INT8 and Q1, then the
// tensor-core kernel.  cudaErrorNotSupported if none takes the shape.
cudaError_t launch_gemv_argmax_fused(const float *x, const uint32_t *codes, const uint16_t *scales,
                                     const uint16_t *biases, int64_t N, int64_t K, int bits, int group,
                                     const ArgmaxWork &w, cudaStream_t s);
// Per row m < M of logits [M, N]: idx[m] = argmax (NaN first, ties to the lower index), val[m] its value.
cudaError_t launch_argmax_rows(const float *logits, int M, int64_t N, int32_t *idx, float *val, cudaStream_t s);

// Decode product on the warp-level tensor cores (mma.sync), 1 <= M <= 8, every
// format; returns cudaErrorNotSupported (nothing launched) for shapes outside
// its layout (groups per row not a multiple of 8, or a lane split the
// instantiated kernels do not cover).
cudaError_t launch_gemv_tc(const float *x, const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                           float *y, int M, int64_t N, int64_t K, int bits, int group, cudaStream_t s);
// The same for M == 1 with the greedy-argmax epilogue (no y written).
cudaError_t launch_gemv_tc_argmax(const float *x, const uint32_t *codes, const uint16_t *scales,
                                  const uint16_t *biases, int64_t N, int64_t K, int bits, int group,
                                  const ArgmaxWork &w, cudaStream_t s);

// Binary (Q1) decode product for M == 1 through per-chunk lookup tables;
// returns cudaErrorNotSupported (nothing launched) for shapes outside its layout.
cudaError_t launch_gemv_q1(const float *x, const uint32_t *codes, const uint16_t *scales, float *y, int64_t N,
                           int64_t K, int group, cudaStream_t s);

// Small-batch decode product, 2 <= M <= 8, bits 4 or 8, codes streamed into
// shared memory; returns cudaErrorNotSupported (nothing launched) for shapes
// outside its layout.
cudaError_t launch_gemv_batch(const float *x, const uint32_t *codes, const uint16_t *scales,
                              const uint16_t *biases, float *y, int M, int64_t N, int64_t K, int bits,
                              int group, cudaStream_t s);

// Prefill product, bits in {1, 4, 8}, group in {64, 128}, K % 64 == 0 (K % 128
// for bits 1), M >= 1, N >= 1.
cudaError_t launch_gemm(const uint16_t *x_bf16, const uint32_t *codes, const uint16_t *scales,
                        const uint16_t *biases, float *y, int64_t M, int64_t N, int64_t K, int bits,
                        int group, cudaStream_t s);

// Device status words written by kernels whose bounded waits ran out (one per
// translation unit); each call synchronizes `s`, returns the word and clears it.
cudaError_t read_clear_gemm_status(int *status, cudaStream_t s);
cudaError_t read_clear_gemv_status(int *status, cudaStream_t s);
cudaError_t read_clear_q1_status(int *status, cudaStream_t s);
cudaError_t read_clear_batch_status(int *status, cudaStream_t s);
// Test hook: the next tensor-core decode launch makes one wait on a barrier
// that never completes, limited to limit_ns, and so reports a device timeout.
void set_tc_test_wait(unsigned long long limit_ns);
cudaError_t read_clear_tc_status(int *status, cudaStream_t s);

}  // namespace qmm
