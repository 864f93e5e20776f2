// api.cu -- the extern "C" entry points declared in include/qmm.h.
//
// Every entry point checks all of its arguments on the host before it
// enqueues anything, so a rejected call leaves every buffer untouched; only
// then does it call one launcher of qmm_launch.h on the caller's stream.  No
// entry point allocates or frees device memory.
#include <cstdint>
#include <cuda_runtime.h>

#include "qmm.h"
#include "qmm_launch.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool bits_ok(int bits) { return bits == 1 || bits == 4 || bits == 8; }
bool group_ok(int group) { return group == 32 || group == 64 || group == 128; }
constexpr int64_t kMaxDim = (int64_t)1 << 31;   // N, K, M each fit in int for the kernels

int cuda_status(cudaError_t e) { return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA; }

// Argmax workspace: a 16-byte counter slot, then per-CTA winners (values,
// indices), then room for logits when the unfused path runs.
constexpr size_t kArgmaxHead = 16 + 8 * (size_t)qmm::kArgmaxMaxCtas;

// Shared checks for the entries that take codes + coefficients.
int check_coeffs(const uint16_t *scales, const uint16_t *biases, int bits) {
  if (!scales) return QMM_ERR_ARG;
  if (bits == 4 && !biases) return QMM_ERR_ARG;
  if (bits != 4 && biases) return QMM_ERR_ARG;
  if (!aligned16(scales) || (biases && !aligned16(biases))) return QMM_ERR_ALIGN;
  return QMM_OK;
}

}  // namespace

extern "C" {

int qmm_abi_version(void) { return 1; }

const char *qmm_status_string(int status) {
  switch (status) {
    case QMM_OK: return "QMM_OK";
    case QMM_ERR_ARG: return "QMM_ERR_ARG: null pointer or biases pointer inconsistent with bits";
    case QMM_ERR_SHAPE: return "QMM_ERR_SHAPE: size out of range or not a multiple of 32 / group";
    case QMM_ERR_ALIGN: return "QMM_ERR_ALIGN: device pointer not aligned (16 bytes; idx and val: 4 bytes)";
    case QMM_ERR_UNSUPPORTED: return "QMM_ERR_UNSUPPORTED: bits/group combination not implemented";
    case QMM_ERR_CUDA: return "QMM_ERR_CUDA: a CUDA call or kernel launch failed";
    case QMM_ERR_DEVICE_TIMEOUT: return "QMM_ERR_DEVICE_TIMEOUT: a bounded device-side wait ran out";
    default: return "unknown qmm status";
  }
}

int qmm_pack(const uint8_t *codes, uint32_t *packed, int64_t N, int64_t K, int bits, qmm_stream_t stream) {
  if (!bits_ok(bits)) return QMM_ERR_UNSUPPORTED;
  if (N < 0 || K < 0 || K % 32 != 0 || N >= kMaxDim || K >= kMaxDim) return QMM_ERR_SHAPE;
  if (N == 0 || K == 0) return QMM_OK;
  if (!codes || !packed) return QMM_ERR_ARG;
  if (!aligned16(codes) || !aligned16(packed)) return QMM_ERR_ALIGN;
  return cuda_status(qmm::launch_pack(codes, packed, N, K, bits, stream));
}

int qmm_unpack(const uint32_t *packed, uint8_t *codes, int64_t N, int64_t K, int bits, qmm_stream_t stream) {
  if (!bits_ok(bits)) return QMM_ERR_UNSUPPORTED;
  if (N < 0 || K < 0 || K % 32 != 0 || N >= kMaxDim || K >= kMaxDim) return QMM_ERR_SHAPE;
  if (N == 0 || K == 0) return QMM_OK;
  if (!codes || !packed) return QMM_ERR_ARG;
  if (!aligned16(codes) || !aligned16(packed)) return QMM_ERR_ALIGN;
  return cuda_status(qmm::launch_unpack(packed, codes, N, K, bits, stream));
}

int qmm_dequant(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases, float *w,
                int64_t N, int64_t K, int bits, int group, qmm_stream_t stream) {
  if (!bits_ok(bits) || !group_ok(group)) return QMM_ERR_UNSUPPORTED;
  if (N < 0 || K < 0 || K % 32 != 0 || K % group != 0 || N >= kMaxDim || K >= kMaxDim) return QMM_ERR_SHAPE;
  if (N == 0 || K == 0) return QMM_OK;
  if (!packed || !w) return QMM_ERR_ARG;
  int st = check_coeffs(scales, biases, bits);
  if (st != QMM_OK) return st;
  if (!aligned16(packed) || !aligned16(w)) return QMM_ERR_ALIGN;
  return cuda_status(qmm::launch_dequant(packed, scales, biases, w, N, K, bits, group, stream));
}

int qmm_gemv(const float *x, const uint32_t *codes, const uint16_t *scales, const uint16_t *biases, float *y,
             int64_t M, int64_t N, int64_t K, int bits, int group, qmm_stream_t stream) {
  if (!bits_ok(bits) || !group_ok(group)) return QMM_ERR_UNSUPPORTED;
  if (M < 0 || M > 8 || N < 0 || K < 0 || K % 32 != 0 || K % group != 0 || N >= kMaxDim || K >= kMaxDim)
    return QMM_ERR_SHAPE;
  if (bits == 1 && K % 128 != 0) return QMM_ERR_SHAPE;
  if (M == 0 || N == 0) return QMM_OK;
  if (!y) return QMM_ERR_ARG;
  if (!aligned16(y)) return QMM_ERR_ALIGN;
  if (K == 0) return cuda_status(cudaMemsetAsync(y, 0, sizeof(float) * (size_t)(M * N), stream));
  if (!x || !codes) return QMM_ERR_ARG;
  int st = check_coeffs(scales, biases, bits);
  if (st != QMM_OK) return st;
  if (!aligned16(x) || !aligned16(codes)) return QMM_ERR_ALIGN;
  return cuda_status(qmm::launch_gemv(x, codes, scales, biases, y, (int)M, N, K, bits, group, stream));
}

int qmm_gemm(const uint16_t *x_bf16, const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
             float *y, int64_t M, int64_t N, int64_t K, int bits, int group, qmm_stream_t stream) {
  if (!bits_ok(bits) || !group_ok(group)) return QMM_ERR_UNSUPPORTED;
  if (M < 0 || N < 0 || K < 64 || K % 64 != 0 || K % group != 0 || M >= kMaxDim || N >= kMaxDim ||
      K >= kMaxDim)
    return QMM_ERR_SHAPE;
  if (bits == 1 && K % 128 != 0) return QMM_ERR_SHAPE;
  if (M == 0 || N == 0) return QMM_OK;
  if (!x_bf16 || !codes || !y) return QMM_ERR_ARG;
  int st = check_coeffs(scales, biases, bits);
  if (st != QMM_OK) return st;
  if (!aligned16(x_bf16) || !aligned16(codes) || !aligned16(y)) return QMM_ERR_ALIGN;
  return cuda_status(qmm::launch_gemm(x_bf16, codes, scales, biases, y, M, N, K, bits, group, stream));
}

size_t qmm_gemv_argmax_workspace_size(int64_t M, int64_t N) {
  if (M < 0 || N < 0) return 0;
  return (size_t)kArgmaxHead + (size_t)M * (size_t)N * sizeof(float);
}

int qmm_gemv_argmax(const float *x, const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                    int32_t *idx, float *val, int64_t M, int64_t N, int64_t K, int bits, int group,
                    void *workspace, size_t workspace_bytes, qmm_stream_t stream) {
  if (!bits_ok(bits) || !group_ok(group)) return QMM_ERR_UNSUPPORTED;
  if (M < 1 || M > 8 || N < 1 || K < 32 || K % 32 != 0 || K % group != 0 || N >= kMaxDim || K >= kMaxDim)
    return QMM_ERR_SHAPE;
  if (bits == 1 && K % 128 != 0) return QMM_ERR_SHAPE;
  if (!x || !codes || !idx || !workspace) return QMM_ERR_ARG;
  int st = check_coeffs(scales, biases, bits);
  if (st != QMM_OK) return st;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(workspace) || !aligned4(idx) || (val && !aligned4(val)))
    return QMM_ERR_ALIGN;
  if (workspace_bytes < qmm_gemv_argmax_workspace_size(M, N)) return QMM_ERR_SHAPE;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  if (M == 1) {
    qmm::ArgmaxWork w{reinterpret_cast<unsigned *>(ws), reinterpret_cast<float *>(ws + 16),
                      reinterpret_cast<int32_t *>(ws + 16 + 4 * qmm::kArgmaxMaxCtas), idx, val};
    cudaError_t e = qmm::launch_gemv_argmax_fused(x, codes, scales, biases, N, K, bits, group, w, stream);
    if (e != cudaErrorNotSupported) return cuda_status(e);
  }
  float *logits = reinterpret_cast<float *>(ws + kArgmaxHead);
  cudaError_t e = qmm::launch_gemv(x, codes, scales, biases, logits, (int)M, N, K, bits, group, stream);
  if (e != cudaSuccess) return QMM_ERR_CUDA;
  return cuda_status(qmm::launch_argmax_rows(logits, (int)M, N, idx, val, stream));
}

int qmm_quantize(const float *w, uint32_t *packed, uint16_t *scales, uint16_t *biases, int64_t N,
                 int64_t K, int group, qmm_stream_t stream) {
  if (!group_ok(group)) return QMM_ERR_UNSUPPORTED;
  if (N < 0 || K < 0 || K % 32 != 0 || K % group != 0 || N >= kMaxDim || K >= kMaxDim) return QMM_ERR_SHAPE;
  if (N == 0 || K == 0) return QMM_OK;
  if (!w || !packed || !scales || !biases) return QMM_ERR_ARG;
  if (!aligned16(w) || !aligned16(packed) || !aligned16(scales) || !aligned16(biases)) return QMM_ERR_ALIGN;
  return cuda_status(qmm::launch_quantize(w, packed, scales, biases, N, K, group, stream));
}

int qmm_gather_dequant(const int32_t *ids, int64_t T, const uint32_t *packed, const uint16_t *scales,
                       const uint16_t *biases, float *out, int64_t N, int64_t K, int bits, int group,
                       qmm_stream_t stream) {
  if (!bits_ok(bits) || !group_ok(group)) return QMM_ERR_UNSUPPORTED;
  if (T < 0 || N < 0 || K < 0 || K % 32 != 0 || K % group != 0 || T >= kMaxDim || N >= kMaxDim ||
      K >= kMaxDim)
    return QMM_ERR_SHAPE;
  if (T == 0 || K == 0) return QMM_OK;
  if (!ids || !packed || !out) return QMM_ERR_ARG;
  int st = check_coeffs(scales, biases, bits);
  if (st != QMM_OK) return st;
  if (!aligned16(ids) || !aligned16(packed) || !aligned16(out)) return QMM_ERR_ALIGN;
  return cuda_status(qmm::launch_gather_dequant(ids, T, packed, scales, biases, out, N, K, bits, group, stream));
}

int qmm_test_timeout_next_decode(int64_t limit_ns) {
  if (limit_ns < 1000 || limit_ns > 100000000) return QMM_ERR_ARG;
  qmm::set_tc_test_wait((unsigned long long)limit_ns);
  return QMM_OK;
}

int qmm_check(qmm_stream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return QMM_ERR_CUDA;
  int st[5] = {0, 0, 0, 0, 0};
  if (qmm::read_clear_gemm_status(&st[0], stream) != cudaSuccess) return QMM_ERR_CUDA;
  if (qmm::read_clear_gemv_status(&st[1], stream) != cudaSuccess) return QMM_ERR_CUDA;
  if (qmm::read_clear_q1_status(&st[2], stream) != cudaSuccess) return QMM_ERR_CUDA;
  if (qmm::read_clear_batch_status(&st[3], stream) != cudaSuccess) return QMM_ERR_CUDA;
  if (qmm::read_clear_tc_status(&st[4], stream) != cudaSuccess) return QMM_ERR_CUDA;
  return (st[0] | st[1] | st[2] | st[3] | st[4]) != 0 ? QMM_ERR_DEVICE_TIMEOUT : QMM_OK;
}

}  // extern "C"
