// pack.cu -- format kernels: pack / unpack / dequantize, row gather, quantize.
//
// Packing convention (the pages fix no bit order): element k of a row sits in
// 32-bit word k / (32/bits) of that row, at bit offset bits * (k mod (32/bits)),
// lowest k in the lowest bits -- the order a shift-and-mask decoder of
// group-64 4-bit codes reads ("Pushing the limits of legacy hardware", section
// "Half a billion values, and one negative zero").  Rows are K*bits/32 words
// long with no padding, so word i of the whole matrix holds the codes of
// elements [i*(32/bits), (i+1)*(32/bits)) of the flattened [N, K] array: the
// pack and unpack kernels need no row arithmetic.
//
// One thread handles one 32-bit word in a grid-stride loop; reads and writes
// are contiguous across consecutive threads.  The same file holds the other
// format kernels: row gather with dequantization and the INT4 quantizer.
#include <cuda_fp16.h>

#include "qmm_device.cuh"
#include "qmm_launch.h"

namespace qmm {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t items) {
  int64_t blocks = (items + kThreads - 1) / kThreads;
  if (blocks > 152 * 16) blocks = 152 * 16;   // grid-stride beyond 16 blocks per SM
  return (int)(blocks < 1 ? 1 : blocks);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) pack_kernel(const uint8_t *__restrict__ codes,
                                                         uint32_t *__restrict__ packed,
                                                         int64_t words) {
  constexpr int PER = 32 / BITS;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint8_t *c = codes + i * PER;
    uint32_t w = 0;
    if (BITS == 8) {
      w = *reinterpret_cast<const uint32_t *>(c);          // already 4 bytes in k order
    } else if (BITS == 4) {
      uint2 b = *reinterpret_cast<const uint2 *>(c);        // 8 codes, one per byte
#pragma unroll
      for (int j = 0; j < 4; j++) {
        w |= ((b.x >> (8 * j)) & MASK) << (4 * j);
        w |= ((b.y >> (8 * j)) & MASK) << (4 * (j + 4));
      }
    } else {
      const uint4 *c4 = reinterpret_cast<const uint4 *>(c);  // 32 codes, one per byte
      uint4 lo = c4[0], hi = c4[1];
      uint32_t b[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
      for (int q = 0; q < 8; q++)
#pragma unroll
        for (int j = 0; j < 4; j++) w |= ((b[q] >> (8 * j)) & 1u) << (4 * q + j);
    }
    packed[i] = w;
  }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) unpack_kernel(const uint32_t *__restrict__ packed,
                                                           uint8_t *__restrict__ codes,
                                                           int64_t words) {
  constexpr int PER = 32 / BITS;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint32_t w = packed[i];
    uint8_t *c = codes + i * PER;
    if (BITS == 8) {
      *reinterpret_cast<uint32_t *>(c) = w;
    } else if (BITS == 4) {
      uint2 b = make_uint2(0, 0);
#pragma unroll
      for (int j = 0; j < 4; j++) {
        b.x |= ((w >> (4 * j)) & MASK) << (8 * j);
        b.y |= ((w >> (4 * (j + 4))) & MASK) << (8 * j);
      }
      *reinterpret_cast<uint2 *>(c) = b;
    } else {
      uint32_t b[8];
#pragma unroll
      for (int q = 0; q < 8; q++) {
        b[q] = 0;
#pragma unroll
        for (int j = 0; j < 4; j++) b[q] |= ((w >> (4 * q + j)) & 1u) << (8 * j);
      }
      uint4 *c4 = reinterpret_cast<uint4 *>(c);
      c4[0] = make_uint4(b[0], b[1], b[2], b[3]);
      c4[1] = make_uint4(b[4], b[5], b[6], b[7]);
    }
  }
}

// w = s*q + b (bits 4), s*q (bits 8), s*(2b-1) (bits 1), in float32 with
// round-to-nearest.  s*q is exact in float32 (at most 11 + 8 significant
// bits), so a single rounded add gives the correctly rounded weight; the
// explicit _rn intrinsics keep the compiler from contracting or reordering.
template <int BITS>
__device__ __forceinline__ void dequant_word(uint32_t w, float s, float b, float (&v)[32 / BITS]) {
#pragma unroll
  for (int j = 0; j < 32 / BITS; j++) {
    uint32_t u = (w >> (BITS * j)) & ((1u << BITS) - 1u);
    if (BITS == 4) {
      v[j] = __fadd_rn(__fmul_rn(s, (float)u), b);
    } else if (BITS == 8) {
      v[j] = __fmul_rn(s, (float)(int)(int8_t)(uint8_t)u);
    } else {
      v[j] = u ? s : -s;                            // s * (2b - 1), exact
    }
  }
}

template <int PER>
__device__ __forceinline__ void store_vec(float *out, const float (&v)[PER]) {
  float4 *o = reinterpret_cast<float4 *>(out);
#pragma unroll
  for (int j = 0; j < PER / 4; j++) o[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

template <int BITS>
__global__ void __launch_bounds__(kThreads) dequant_kernel(
    const uint32_t *__restrict__ packed, const uint16_t *__restrict__ scales,
    const uint16_t *__restrict__ biases, float *__restrict__ out, int64_t words,
    int64_t words_per_row, int64_t groups_per_row, int group) {
  constexpr int PER = 32 / BITS;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t n = i / words_per_row;
    int64_t k0 = (i % words_per_row) * PER;
    int64_t gi = n * groups_per_row + k0 / group;   // a word never straddles a group
    float v[PER];
    dequant_word<BITS>(packed[i], h2f(scales[gi]), (BITS == 4) ? h2f(biases[gi]) : 0.0f, v);
    store_vec<PER>(out + i * PER, v);
  }
}

// Row gather with dequantization: out[t, :] = dequant(W[ids[t], :]), the
// embedding lookup of a tied INT4 table ("Pushing the limits of legacy
// hardware", section "Half a billion values, and one negative zero": token ids
// select rows that are decoded exactly).  Same element rule as dequant_kernel;
// an id outside [0, N) yields a row of quiet NaNs (nothing is read for it).
template <int BITS>
__global__ void __launch_bounds__(kThreads) gather_dequant_kernel(
    const int32_t *__restrict__ ids, const uint32_t *__restrict__ packed, const uint16_t *__restrict__ scales,
    const uint16_t *__restrict__ biases, float *__restrict__ out, int64_t items, int64_t N,
    int64_t words_per_row, int64_t groups_per_row, int group) {
  constexpr int PER = 32 / BITS;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < items;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / words_per_row, j = i % words_per_row;
    const int64_t n = ids[t];
    float v[PER];
    if (n < 0 || n >= N) {
#pragma unroll
      for (int e = 0; e < PER; e++) v[e] = __int_as_float(0x7FC00000);
    } else {
      const int64_t gi = n * groups_per_row + j * PER / group;
      dequant_word<BITS>(packed[n * words_per_row + j], h2f(scales[gi]), (BITS == 4) ? h2f(biases[gi]) : 0.0f,
                         v);
    }
    store_vec<PER>(out + i * PER, v);
  }
}

// ---------------------------------------------------------------- quantizer

// The group's range takes NaN-free values in a total order with -0 below
// +0, so the stored bias does not depend on the order of the reduction.  The
// order is that of these integer keys (the sign-magnitude bits with the
// magnitude flipped for negative values), compared with one integer min/max.
__device__ __forceinline__ int order_key(float f) {
  const int b = __float_as_int(f);
  return b ^ ((b >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float from_order_key(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7FFFFFFF)); }

// Approximate reciprocal (relative error within a few units in the last place).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// binary16 bits of f, round to nearest even; any NaN becomes 0x7E00.
__device__ __forceinline__ uint16_t half_bits_rn(float f) {
  return isnan(f) ? (uint16_t)0x7E00u : __half_as_ushort(__float2half_rn(f));
}

// INT4 affine quantization of float32 weights to the stored format, after
// the quantization section of "I Built an LLM Inference Engine on a 15 year
// old GPU and the Math was the Easy Part": per group of consecutive k, the
// range [min, max] is cut into 15 steps, scale = (max - min) / 15 and
// bias = min are stored as binary16 (round to nearest even), and each weight
// becomes q = clamp(round((w - bias) / scale), 0, 15) computed in float32
// with the stored coefficients (halves away from zero; q = 0 for a NaN weight
// or a scale that is not positive and finite).  One thread per 8 weights (one
// code word); the GT = group/8 threads of a group are adjacent lanes of one
// warp and reduce the range with shuffles.
template <int GT>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const float *__restrict__ w,
                                                             uint32_t *__restrict__ packed,
                                                             uint16_t *__restrict__ scales,
                                                             uint16_t *__restrict__ biases, int64_t words) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // the next word's 32 bytes are loaded before the current word is worked on
  // (two loads in flight per thread)
  const float4 *w4 = reinterpret_cast<const float4 *>(w);
  const float4 nan4 = make_float4(__int_as_float(0x7FC00000), __int_as_float(0x7FC00000),
                                  __int_as_float(0x7FC00000), __int_as_float(0x7FC00000));
  int64_t base = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) - lane;
  float4 na = nan4, nc = nan4;
  if (base + lane < words) na = w4[2 * (base + lane)], nc = w4[2 * (base + lane) + 1];
  // the loop bound is uniform per warp so that every lane takes part in the shuffles
  for (; base < words; base += stride) {
    const int64_t i = base + lane;
    const bool active = i < words;
    const float4 a = na, c = nc;
    if (i + stride < words) na = w4[2 * (i + stride)], nc = w4[2 * (i + stride) + 1];
    else na = nan4, nc = nan4;
    float v[8];
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = c.x, v[5] = c.y, v[6] = c.z, v[7] = c.w;
    int kmin = 0x7FFFFFFF, kmax = (int)0x80000000;            // no value yet (NaN weights are skipped)
#pragma unroll
    for (int j = 0; j < 8; j++)
      if (!isnan(v[j])) {
        const int k = order_key(v[j]);
        kmin = min(kmin, k);
        kmax = max(kmax, k);
      }
#pragma unroll
    for (int o = 1; o < GT; o <<= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
    }
    if (!active) continue;
    const float nan = __int_as_float(0x7FC00000);
    const float lo = kmin == 0x7FFFFFFF ? nan : from_order_key(kmin);   // an all-NaN group has a NaN range
    const float hi = kmax == (int)0x80000000 ? nan : from_order_key(kmax);
    const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    const uint16_t sh = half_bits_rn(s32), bh = half_bits_rn(lo);
    const float s = h2f(sh), b = h2f(bh);
    uint32_t word = 0;
    if (s > 0.0f && isfinite(s)) {
      // The quotient (w - b) / s, correctly rounded, decides q only through
      // roundf, i.e. only where it lies next to a half-integer.  A product
      // with the approximate reciprocal is within a few units in the last
      // place of it; where that product is farther than 1e-5 (relative) from
      // the nearest half-integer both round alike, elsewhere the correctly
      // rounded division is taken.
      // A NaN weight gives a NaN quotient, which clamps to 0; an infinite one
      // takes the division and clamps to 0 or 15.
      const float inv = rcp_approx(s);
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const float d = __fsub_rn(v[j], b);
        const float qf = __fmul_rn(d, inv);
        const float fl = floorf(qf);
        const float fr = qf - fl;                 // exact, except just below 0 where only the check needs it
        float r;
        if (fabsf(fr - 0.5f) > 1e-5f * fmaxf(1.0f, fabsf(qf))) r = fr > 0.5f ? fl + 1.0f : fl;   // = roundf(qf)
        else r = roundf(__fdiv_rn(d, s));
        r = fminf(fmaxf(r, 0.0f), 15.0f);
        word |= (__float_as_uint(r + 8388608.0f) & 0xFu) << (4 * j);   // the integer r in the low mantissa bits
      }
    }
    packed[i] = word;
    if (lane % GT == 0) {
      scales[i / GT] = sh;
      biases[i / GT] = bh;
    }
  }
}

}  // namespace

cudaError_t launch_pack(const uint8_t *codes, uint32_t *packed, int64_t N, int64_t K, int bits,
                        cudaStream_t s) {
  int64_t words = N * K * bits / 32;
  if (words == 0) return cudaSuccess;
  int g = grid_for(words);
  if (bits == 4) pack_kernel<4><<<g, kThreads, 0, s>>>(codes, packed, words);
  else if (bits == 8) pack_kernel<8><<<g, kThreads, 0, s>>>(codes, packed, words);
  else pack_kernel<1><<<g, kThreads, 0, s>>>(codes, packed, words);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t *packed, uint8_t *codes, int64_t N, int64_t K, int bits,
                          cudaStream_t s) {
  int64_t words = N * K * bits / 32;
  if (words == 0) return cudaSuccess;
  int g = grid_for(words);
  if (bits == 4) unpack_kernel<4><<<g, kThreads, 0, s>>>(packed, codes, words);
  else if (bits == 8) unpack_kernel<8><<<g, kThreads, 0, s>>>(packed, codes, words);
  else unpack_kernel<1><<<g, kThreads, 0, s>>>(packed, codes, words);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                           float *w, int64_t N, int64_t K, int bits, int group, cudaStream_t s) {
  int64_t words = N * K * bits / 32;
  if (words == 0) return cudaSuccess;
  int64_t wpr = K * bits / 32, gpr = K / group;
  int g = grid_for(words);
  if (bits == 4) dequant_kernel<4><<<g, kThreads, 0, s>>>(packed, scales, biases, w, words, wpr, gpr, group);
  else if (bits == 8) dequant_kernel<8><<<g, kThreads, 0, s>>>(packed, scales, biases, w, words, wpr, gpr, group);
  else dequant_kernel<1><<<g, kThreads, 0, s>>>(packed, scales, biases, w, words, wpr, gpr, group);
  return cudaGetLastError();
}

cudaError_t launch_gather_dequant(const int32_t *ids, int64_t T, const uint32_t *packed, const uint16_t *scales,
                                  const uint16_t *biases, float *out, int64_t N, int64_t K, int bits, int group,
                                  cudaStream_t s) {
  const int64_t wpr = K * bits / 32, gpr = K / group, items = T * wpr;
  if (items == 0) return cudaSuccess;
  int g = grid_for(items);
  if (bits == 4)
    gather_dequant_kernel<4><<<g, kThreads, 0, s>>>(ids, packed, scales, biases, out, items, N, wpr, gpr, group);
  else if (bits == 8)
    gather_dequant_kernel<8><<<g, kThreads, 0, s>>>(ids, packed, scales, biases, out, items, N, wpr, gpr, group);
  else
    gather_dequant_kernel<1><<<g, kThreads, 0, s>>>(ids, packed, scales, biases, out, items, N, wpr, gpr, group);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const float *w, uint32_t *packed, uint16_t *scales, uint16_t *biases, int64_t N,
                            int64_t K, int group, cudaStream_t s) {
  const int64_t words = N * K / 8;
  if (words == 0) return cudaSuccess;
  int g = grid_for(words);
  if (group == 32) quantize_kernel<4><<<g, kThreads, 0, s>>>(w, packed, scales, biases, words);
  else if (group == 64) quantize_kernel<8><<<g, kThreads, 0, s>>>(w, packed, scales, biases, words);
  else quantize_kernel<16><<<g, kThreads, 0, s>>>(w, packed, scales, biases, words);
  return cudaGetLastError();
}

}  // namespace qmm
