// noalloc.cu -- the greedy argmax head without a caller-provided work area.
//
// qmm_gemv_argmax needs a small device work area (a CTA counter and the
// per-CTA winners) that the caller allocates.  Some callers cannot allocate
// device memory at the point of the call: a decode loop that must not enter
// the device allocator between tokens (an allocation can synchronize the
// device or fail under memory pressure), or a C host that links only this
// library and has no allocator of its own.  This entry point keeps that work
// area in a fixed, file-scope device array instead, so it allocates nothing.
//
// Limits and rules (also stated in include/qmm.h):
//   * the array holds a 16-byte counter slot and the winners of at most
//     kArgmaxMaxCtas (1024) CTAs: 8208 bytes; shapes whose fused launch would
//     need more CTAs, and shapes the fused M == 1 kernel does not take, are
//     rejected with QMM_ERR_UNSUPPORTED (there is no unfused fallback here,
//     since that would need room for the logits);
//   * the counter must be zero when a call starts: the array is zero when the
//     module loads, and every call's last CTA sets it back to zero;
//   * the address of the array is looked up with cudaGetSymbolAddress and
//     cached per device together with the context that was current at the
//     lookup; a call made in another context (after cudaDeviceReset, or once
//     the primary context was destroyed and created again) looks it up anew.
//     Make the first call in each context before any stream capture begins;
//   * all calls on a device share the array, so two calls must never be in
//     flight at the same time (for instance on two streams): they would race
//     on the counter and the winners.  Calls issued one after another on one
//     stream are fine.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "qmm.h"
#include "qmm_launch.h"

namespace {

constexpr size_t kScratchBytes = 16 + 8 * (size_t)qmm::kArgmaxMaxCtas;   // 8208 bytes
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_argmax_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// cuCtxGetCurrent through the runtime's driver entry point (no link to libcuda).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  return fn;
}

// The device address of g_argmax_scratch in the current context.  The cached
// address is reused only while the context it was looked up in is current.
cudaError_t scratch_address(void **addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!ctx || ctx != g_scratch_ctx[dev] || !g_scratch_addr[dev]) {
    // The lookup makes the device's primary context current if none is.
    e = cudaGetSymbolAddress(&g_scratch_addr[dev], g_argmax_scratch);
    if (e != cudaSuccess) return e;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
    g_scratch_ctx[dev] = ctx;
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" int qmm_gemv_argmax_noalloc(const float *x, const uint32_t *codes, const uint16_t *scales,
                                       const uint16_t *biases, int32_t *idx, float *val, int64_t N, int64_t K,
                                       int bits, int group, qmm_stream_t stream) {
  if ((bits != 1 && bits != 4 && bits != 8) || (group != 32 && group != 64 && group != 128))
    return QMM_ERR_UNSUPPORTED;
  if (N < 1 || K < 32 || K % 32 != 0 || K % group != 0 || N >= ((int64_t)1 << 31) || K >= ((int64_t)1 << 31))
    return QMM_ERR_SHAPE;
  if (bits == 1 && K % 128 != 0) return QMM_ERR_SHAPE;
  if (!x || !codes || !scales || !idx) return QMM_ERR_ARG;
  if ((bits == 4) != (biases != nullptr)) return QMM_ERR_ARG;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || (biases && !aligned16(biases)) ||
      !aligned4(idx) || (val && !aligned4(val)))
    return QMM_ERR_ALIGN;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return QMM_ERR_CUDA;
  uint8_t *ws = static_cast<uint8_t *>(scratch);
  qmm::ArgmaxWork w{reinterpret_cast<unsigned *>(ws), reinterpret_cast<float *>(ws + 16),
                    reinterpret_cast<int32_t *>(ws + 16 + 4 * qmm::kArgmaxMaxCtas), idx, val};
  const cudaError_t e = qmm::launch_gemv_argmax_fused(x, codes, scales, biases, N, K, bits, group, w, stream);
  if (e == cudaErrorNotSupported) return QMM_ERR_UNSUPPORTED;
  return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}
