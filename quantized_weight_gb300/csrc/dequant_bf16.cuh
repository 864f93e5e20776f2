// dequant_bf16.cuh -- codes to bfloat16 for the tensor-core prefill kernel:
// the weight in float32 (INT4: s*q + b with the product exact and one
// rounding; INT8: s*q, exact; Q1: +-s, exact), then round-to-nearest-even to
// bfloat16, two values per 32-bit word with the lower k in the lower half.
#pragma once
#include <cstdint>

#include "qmm_device.cuh"

namespace qmm {

// Dequantize 8 codes (one 32-bit word, k = 8c .. 8c+7) into 8 bf16 packed as
// four 32-bit words, k order low-to-high within each word.
//   w_j = s*q_j + b, evaluated as fma(s*16^-cls, q_j*16^cls, b): the nibble is
//   masked in place and OR-ed into the bits of 2^23 (an exact float
//   2^23 + q*16^cls), 2^23 is subtracted exactly, and the power-of-two
//   pre-scaled s makes the product exact, so the FMA rounds s*q + b once.
__device__ __forceinline__ uint4 dequant_word_bf16(uint32_t w, const f2 (&sp)[4], f2 b2) {
  const f2 magic2 = f2_make(8388608.0f, 8388608.0f);
  const uint32_t wh = w >> 12;
  const uint32_t M0 = 0x4B000000u;
  f2 q01 = f2_sub(f2_bits(and_or(w, 0xFu, M0), and_or(w, 0xF0u, M0)), magic2);
  f2 q23 = f2_sub(f2_bits(and_or(w, 0xF00u, M0), and_or(w, 0xF000u, M0)), magic2);
  f2 q45 = f2_sub(f2_bits(and_or(w, 0xF0000u, M0), and_or(wh, 0xF00u, M0)), magic2);
  f2 q67 = f2_sub(f2_bits(and_or(wh, 0xF000u, M0), and_or(wh, 0xF0000u, M0)), magic2);
  // sp[0] = (s, s/16), sp[1] = (s/256, s/4096), sp[2] = (s/65536, s/256), sp[3] = (s/4096, s/65536)
  f2 v01 = f2_fma(q01, sp[0], b2);
  f2 v23 = f2_fma(q23, sp[1], b2);
  f2 v45 = f2_fma(q45, sp[2], b2);
  f2 v67 = f2_fma(q67, sp[3], b2);
  float a, c;
  uint4 o;
  f2_split(v01, a, c);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.x) : "f"(c), "f"(a));
  f2_split(v23, a, c);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.y) : "f"(c), "f"(a));
  f2_split(v45, a, c);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.z) : "f"(c), "f"(a));
  f2_split(v67, a, c);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.w) : "f"(c), "f"(a));
  return o;
}

__device__ __forceinline__ void scale_pairs(float s, f2 (&sp)[4]) {
  const float s1 = s * 0.0625f, s2 = s * 0.00390625f, s3 = s * 0.000244140625f,
              s4 = s * 1.52587890625e-05f;   // exact: powers of two, no underflow for binary16 s
  sp[0] = f2_make(s, s1);
  sp[1] = f2_make(s2, s3);
  sp[2] = f2_make(s4, s2);
  sp[3] = f2_make(s3, s4);
}

// Half i (0..7) of eight binary16 values held in a uint4.
__device__ __forceinline__ uint16_t half_at(const uint4 v, int i) {
  const uint32_t w = (i & 4) ? ((i & 2) ? v.w : v.z) : ((i & 2) ? v.y : v.x);
  return (uint16_t)((i & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// INT8: 8 codes (two words, k order) -> 8 bf16 of s*q.  After XOR 0x80 per
// byte one prmt builds the float 2^23 + (q + 128), a packed subtract gives q,
// a packed multiply by s gives s*q exactly (at most 11 + 8 significant bits).
__device__ __forceinline__ uint4 dequant_int8x8_bf16(uint32_t w0, uint32_t w1, f2 s2) {
  const f2 off2 = f2_make(8388736.0f, 8388736.0f);   // 2^23 + 128
  const uint32_t M0 = 0x4B000000u;
  const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
  const f2 v01 = f2_mul(f2_sub(f2_bits(prmt(u0, M0, 0x7540u), prmt(u0, M0, 0x7541u)), off2), s2);
  const f2 v23 = f2_mul(f2_sub(f2_bits(prmt(u0, M0, 0x7542u), prmt(u0, M0, 0x7543u)), off2), s2);
  const f2 v45 = f2_mul(f2_sub(f2_bits(prmt(u1, M0, 0x7540u), prmt(u1, M0, 0x7541u)), off2), s2);
  const f2 v67 = f2_mul(f2_sub(f2_bits(prmt(u1, M0, 0x7542u), prmt(u1, M0, 0x7543u)), off2), s2);
  uint4 o;
  float a, c;
  f2_split(v01, a, c);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.x) : "f"(c), "f"(a));
  f2_split(v23, a, c);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.y) : "f"(c), "f"(a));
  f2_split(v45, a, c);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.z) : "f"(c), "f"(a));
  f2_split(v67, a, c);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o.w) : "f"(c), "f"(a));
  return o;
}

// bf16 bits of s (round to nearest even), in both halves of a word.
__device__ __forceinline__ uint32_t bf16_pair(float s) {
  uint32_t o;
  asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(o) : "f"(s));
  return o;
}

// Q1: 8 sign bits (bit j = k j; set: +1, clear: -1) -> 8 bf16 of +-s, where
// sp holds bf16(s) in both halves: a clear bit sets that half's sign bit.
__device__ __forceinline__ uint4 signs8_bf16(uint32_t bits8, uint32_t sp) {
  const uint32_t nb = ~bits8;
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const uint32_t m = ((nb >> (2 * i)) & 1u) << 15 | ((nb >> (2 * i + 1)) & 1u) << 31;
    o[i] = sp ^ m;
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace qmm
