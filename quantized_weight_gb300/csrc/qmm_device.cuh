// qmm_device.cuh -- small device-side helpers shared by the qmm kernels (sm_103a).
//
// Inline PTX wrappers for the instructions the kernels are built from: streaming
// 128-bit loads that do not allocate in L1, packed f32x2 arithmetic, lop3/prmt
// bit manipulation, programmatic-dependent-launch control and IEEE binary16
// decoding.  Nothing here is specific to one format.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace qmm {

// ---------------------------------------------------------------- loads

// Read-only 16-byte load that streams through L2 without allocating in L1:
// every packed code is read exactly once, so caching it in L1 only evicts x.
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_nc_u16(const void *p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float4 ld_nc_f4(const void *p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// binary16 bits -> float32, exact (subnormals kept: cvt does not flush).
__device__ __forceinline__ float h2f(uint16_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}

// ---------------------------------------------------------------- f32x2
// Blackwell executes two float32 lanes per instruction with the .f32x2 forms;
// a pair lives in one 64-bit register.

struct f2 { unsigned long long v; };

__device__ __forceinline__ f2 f2_make(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r.v) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ f2 f2_bits(uint32_t a, uint32_t b) {
  f2 r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r.v) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ void f2_split(f2 p, float &a, float &b) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(a), "=f"(b) : "l"(p.v));
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
  f2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r.v) : "l"(a.v), "l"(b.v));
  return r;
}
// a * b + c, one rounding per lane
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r.v) : "l"(a.v), "l"(b.v), "l"(c.v));
  return r;
}
__device__ __forceinline__ f2 f2_zero() { return f2_bits(0u, 0u); }

// ---------------------------------------------------------------- bit ops

// (a & b) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// a ^ (~b & c)
__device__ __forceinline__ uint32_t xor_andnot(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xD2;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// byte permute: d.byte[i] = ({b,a} bytes)[sel nibble i]
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// ---------------------------------------------------------------- launch control

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (a no-op when the kernel
// was launched without the programmatic-serialization attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace qmm
