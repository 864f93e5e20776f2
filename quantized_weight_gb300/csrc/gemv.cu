// gemv.cu -- the decode product y[M, N] = x[M, K] * dequant(W)^T for 1 <= M <= 8.
//
// Decode reads every weight exactly once and is bound by HBM bandwidth ("...
// Tesla C2075 ..." paper, section 3.3 "Decode, and why 4-bit is slower"), so
// the kernel is built around one 16-byte coalesced, L1-bypassing load per lane
// per chunk of codes (32 INT4 / 16 INT8 / 128 Q1 weights).  The same section
// reports that on Fermi the nibble-unpacking shifts pushed the 4-bit kernel off
// its bandwidth bound; on GB300 the analogous risk is the issue rate (about 5
// lane-instructions per byte of HBM traffic per SM), so every per-weight step is
// one instruction or less:
//
//   INT4  q*16^c comes out of ONE lop3: OR-ing the masked nibble (left where it
//         sits in the word, c = its position class) into the bit pattern of
//         2^23 gives the float 2^23 + q*16^c exactly; a packed f32x2 subtract
//         removes 2^23 and a packed f32x2 FMA multiplies by x.  The 16^c factors
//         are exact powers of two, taken out once per chunk.  The group bias is
//         factored out:  sum_k (s q_k + b) x_k = s * sum_k q_k x_k + b * sum_k x_k,
//         with sum_k x_k computed once per chunk per CTA while staging x.
//   INT8  after XOR 0x80 per byte, one prmt builds the float 2^23 + (q + 128);
//         a packed subtract of 2^23 + 128 gives q exactly.
//   Q1    w*x = +x or -x: one shift and one lop3 move the sign bit, a packed add
//         accumulates; the group scale multiplies the word's sum.
//
// Work layout: a warp's 32 lanes are LK lanes along K times (32/LK) lanes
// along N; each lane owns R rows.  The activations of one K-tile are staged in
// shared memory once per CTA (swizzled so that the LK distinct 16-byte reads
// of one instruction hit distinct banks) and reused by every row of the CTA.
// Partial sums are reduced across the LK lanes with shuffles in a fixed order:
// no atomics, the result is identical on every run.
//
// The codes of the first K-tile are requested before the kernel waits on the
// previous kernel in the stream (programmatic dependent launch), so in a chain
// of decode products the weight stream of one layer overlaps the tail of the
// previous one; x is read only after that wait.
#include "qmm_device.cuh"
#include "qmm_launch.h"

namespace qmm {
namespace {

constexpr uint32_t kMagic = 0x4B000000u;       // bit pattern of 2^23
constexpr float kTwo23 = 8388608.0f;           // 2^23
constexpr float kTwo23p128 = 8388736.0f;       // 2^23 + 128

struct GemvParams {
  const float *x;
  const uint4 *codes;
  const uint16_t *scales;
  const uint16_t *biases;
  float *y;
  int M, N, K;
  int gshift;            // log2(group)
  int chunks_per_row;    // K / CW
  int groups_per_row;    // K / group
};

template <int BITS>
struct Fmt {
  static constexpr int CW = 128 / BITS;   // weights per 16-byte chunk
  static constexpr int CU = CW / 4;       // float4 units of x per chunk
  static constexpr int SPAN = CU > 8 ? CU : 8;
  // one x-sum per 32 weights for INT4 (per chunk) and Q1 (per word); none for INT8
  static constexpr bool SUMS = (BITS != 8);
};

// Physical float4 slot of logical x unit u (one x row of the tile): XOR the
// low three bits with the chunk index so that lanes reading the same unit of
// consecutive chunks land in different 16-byte bank groups.
template <int BITS>
__device__ __forceinline__ int swz(int u) {
  return u ^ ((u / Fmt<BITS>::SPAN) & 7);
}

// ---------------------------------------------------------------- per-format chunk math

// INT4: returns sum_k q_k x_k over the 32 weights of one chunk (4 words).
__device__ __forceinline__ float dot_int4(const uint4 c, const f2 (&xp)[16]) {
  const f2 magic2 = f2_make(kTwo23, kTwo23);
  f2 a01 = f2_zero(), a23 = f2_zero(), a45 = f2_zero(), a67 = f2_zero();
  const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int wi = 0; wi < 4; wi++) {
    const uint32_t w = wv[wi];
    const uint32_t wh = w >> 12;
    f2 q01 = f2_sub(f2_bits(and_or(w, 0xFu, kMagic), and_or(w, 0xF0u, kMagic)), magic2);
    f2 q23 = f2_sub(f2_bits(and_or(w, 0xF00u, kMagic), and_or(w, 0xF000u, kMagic)), magic2);
    f2 q45 = f2_sub(f2_bits(and_or(w, 0xF0000u, kMagic), and_or(wh, 0xF00u, kMagic)), magic2);
    f2 q67 = f2_sub(f2_bits(and_or(wh, 0xF000u, kMagic), and_or(wh, 0xF0000u, kMagic)), magic2);
    a01 = f2_fma(q01, xp[4 * wi + 0], a01);
    a23 = f2_fma(q23, xp[4 * wi + 1], a23);
    a45 = f2_fma(q45, xp[4 * wi + 2], a45);
    a67 = f2_fma(q67, xp[4 * wi + 3], a67);
  }
  float c0, c1, c2, c3, c4, c5, c6, c7;
  f2_split(a01, c0, c1);   // position classes 16^0, 16^1
  f2_split(a23, c2, c3);   // 16^2, 16^3
  f2_split(a45, c4, c5);   // 16^4, 16^2
  f2_split(a67, c6, c7);   // 16^3, 16^4
  float d = c0;
  d = fmaf(c1, 0.0625f, d);
  d = fmaf(c2 + c5, 0.00390625f, d);
  d = fmaf(c3 + c6, 0.000244140625f, d);
  d = fmaf(c4 + c7, 1.52587890625e-05f, d);
  return d;
}

// INT8: sum_k q_k x_k over the 16 weights of one chunk.
__device__ __forceinline__ float dot_int8(const uint4 c, const f2 (&xp)[8]) {
  const f2 off2 = f2_make(kTwo23p128, kTwo23p128);
  f2 a0 = f2_zero(), a1 = f2_zero();
  const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int wi = 0; wi < 4; wi++) {
    const uint32_t w = wv[wi] ^ 0x80808080u;        // q + 128 as an unsigned byte
    f2 q01 = f2_sub(f2_bits(prmt(w, kMagic, 0x7540u), prmt(w, kMagic, 0x7541u)), off2);
    f2 q23 = f2_sub(f2_bits(prmt(w, kMagic, 0x7542u), prmt(w, kMagic, 0x7543u)), off2);
    a0 = f2_fma(q01, xp[2 * wi + 0], a0);
    a1 = f2_fma(q23, xp[2 * wi + 1], a1);
  }
  float c0, c1, c2, c3;
  f2_split(a0, c0, c1);
  f2_split(a1, c2, c3);
  return (c0 + c1) + (c2 + c3);
}

// Q1: sum_k (2 b_k - 1) x_k over the 32 weights of one word.
__device__ __forceinline__ float dot_q1(const uint32_t w, const f2 (&xp)[16]) {
  f2 a[4] = {f2_zero(), f2_zero(), f2_zero(), f2_zero()};
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float xa, xb;
    f2_split(xp[j / 2], xa, xb);
    // bit j of w moved to bit 31; a clear bit flips the sign of x
    uint32_t sa = xor_andnot(__float_as_uint(xa), w << (31 - j), 0x80000000u);
    uint32_t sb = xor_andnot(__float_as_uint(xb), w << (30 - j), 0x80000000u);
    a[(j / 2) & 3] = f2_add(a[(j / 2) & 3], f2_bits(sa, sb));
  }
  float t[8];
  f2_split(a[0], t[0], t[1]);
  f2_split(a[1], t[2], t[3]);
  f2_split(a[2], t[4], t[5]);
  f2_split(a[3], t[6], t[7]);
  return ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
}

// ---------------------------------------------------------------- the kernel

template <int BITS, int MT, int LK, int R, int CH>
__global__ void __launch_bounds__(256) gemv_kernel(const GemvParams p) {
  using F = Fmt<BITS>;
  constexpr int CW = F::CW, CU = F::CU;
  constexpr int LR = 32 / LK;
  constexpr int KT = LK * CH * CW;             // weights per K-tile
  constexpr int TU = KT / 4;                   // float4 units per x row of a tile
  constexpr int NSUM = F::SUMS ? KT / 32 : 1;  // x sums per x row of a tile

  extern __shared__ float4 smem[];
  float4 *xs = smem;                                              // [MT][TU]
  float *xsum = reinterpret_cast<float *>(smem + MT * TU);       // [MT][NSUM]

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int kq = lane % LK, rr = lane / LK;
  const int rows_per_cta = (blockDim.x >> 5) * LR * R;
  const int row0 = blockIdx.x * rows_per_cta + (warp * LR + rr) * R;

  pdl_launch_dependents();

  float acc[R][MT];
#pragma unroll
  for (int r = 0; r < R; r++)
#pragma unroll
    for (int m = 0; m < MT; m++) acc[r][m] = 0.0f;

  for (int t0 = 0; t0 < p.K; t0 += KT) {
    const int tchunks = min(KT, p.K - t0) / CW;
    const int c0 = t0 / CW;

    // 1. request this tile's codes and coefficients
    uint4 c[R][CH];
    float s[R][CH][BITS == 1 ? 4 : 1];
    float b[R][CH];
#pragma unroll
    for (int r = 0; r < R; r++) {
      const int row = row0 + r;
      const bool row_ok = row < p.N;
      const uint4 *crow = p.codes + (int64_t)row * p.chunks_per_row + c0;
      const int64_t grow = (int64_t)row * p.groups_per_row;
#pragma unroll
      for (int i = 0; i < CH; i++) {
        const int ch = kq + LK * i;
        const bool ok = row_ok && ch < tchunks;
        c[r][i] = ok ? ld_stream_u4(crow + ch) : make_uint4(0u, 0u, 0u, 0u);
        const int k = t0 + ch * CW;
        if (BITS == 1) {
#pragma unroll
          for (int wi = 0; wi < 4; wi++) {
            const int g = (k + 32 * wi) >> p.gshift;
            s[r][i][wi] = ok ? h2f(ld_nc_u16(p.scales + grow + g)) : 0.0f;
          }
          b[r][i] = 0.0f;
        } else {
          const int g = k >> p.gshift;
          s[r][i][0] = ok ? h2f(ld_nc_u16(p.scales + grow + g)) : 0.0f;
          b[r][i] = (BITS == 4 && ok) ? h2f(ld_nc_u16(p.biases + grow + g)) : 0.0f;
        }
      }
    }

    // 2. stage x[:, t0 : t0 + KT] (and its 32-element sums) in shared memory
    if (t0 == 0) pdl_wait();        // x is written by the previous kernel
    __syncthreads();                // readers of the previous tile are done
    {
      const int tu = tchunks * CU;                 // units per x row in this tile
      const int total = p.M * tu;                  // multiple of 8
      const int span = (total + blockDim.x - 1) / blockDim.x * blockDim.x;
      for (int idx = threadIdx.x; idx < span; idx += blockDim.x) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        const int m = idx / tu, u = idx - m * tu;
        if (idx < total) {
          v = ld_nc_f4(p.x + (int64_t)m * p.K + t0 + 4 * u);
          xs[m * TU + swz<BITS>(u)] = v;
        }
        if (F::SUMS) {
          float part = (v.x + v.y) + (v.z + v.w);
          part += __shfl_xor_sync(0xffffffffu, part, 1);
          part += __shfl_xor_sync(0xffffffffu, part, 2);
          part += __shfl_xor_sync(0xffffffffu, part, 4);
          if (idx < total && (u & 7) == 0) xsum[m * NSUM + (u >> 3)] = part;
        }
      }
    }
    __syncthreads();

    // 3. multiply-accumulate
#pragma unroll
    for (int i = 0; i < CH; i++) {
      const int ch = kq + LK * i;
      if (ch >= tchunks) continue;
#pragma unroll
      for (int m = 0; m < MT; m++) {
        if (m >= p.M) continue;
        const float4 *xrow = xs + m * TU;
        if (BITS == 4) {
          f2 xp[16];
#pragma unroll
          for (int j = 0; j < 8; j++) {
            float4 v = xrow[swz<BITS>(ch * CU + j)];
            xp[2 * j] = f2_make(v.x, v.y);
            xp[2 * j + 1] = f2_make(v.z, v.w);
          }
          const float xsumv = xsum[m * NSUM + ch];
#pragma unroll
          for (int r = 0; r < R; r++) {
            const float d = dot_int4(c[r][i], xp);
            acc[r][m] = fmaf(s[r][i][0], d, fmaf(b[r][i], xsumv, acc[r][m]));
          }
        } else if (BITS == 8) {
          f2 xp[8];
#pragma unroll
          for (int j = 0; j < 4; j++) {
            float4 v = xrow[swz<BITS>(ch * CU + j)];
            xp[2 * j] = f2_make(v.x, v.y);
            xp[2 * j + 1] = f2_make(v.z, v.w);
          }
#pragma unroll
          for (int r = 0; r < R; r++) acc[r][m] = fmaf(s[r][i][0], dot_int8(c[r][i], xp), acc[r][m]);
        } else {
#pragma unroll
          for (int wi = 0; wi < 4; wi++) {
            f2 xp[16];
#pragma unroll
            for (int j = 0; j < 8; j++) {
              float4 v = xrow[swz<BITS>(ch * CU + 8 * wi + j)];
              xp[2 * j] = f2_make(v.x, v.y);
              xp[2 * j + 1] = f2_make(v.z, v.w);
            }
            (void)xsum;
#pragma unroll
            for (int r = 0; r < R; r++) {
              const uint32_t w = wi == 0 ? c[r][i].x : wi == 1 ? c[r][i].y : wi == 2 ? c[r][i].z : c[r][i].w;
              acc[r][m] = fmaf(s[r][i][wi], dot_q1(w, xp), acc[r][m]);
            }
          }
        }
      }
    }
  }

  // 4. reduce over the LK lanes of each row (fixed butterfly order), store
#pragma unroll
  for (int r = 0; r < R; r++)
#pragma unroll
    for (int m = 0; m < MT; m++) {
      float v = acc[r][m];
#pragma unroll
      for (int off = LK / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[r][m] = v;
    }
  if (kq == 0) {
#pragma unroll
    for (int r = 0; r < R; r++) {
      const int row = row0 + r;
      if (row < p.N) {
#pragma unroll
        for (int m = 0; m < MT; m++)
          if (m < p.M) p.y[(int64_t)m * p.N + row] = acc[r][m];
      }
    }
  }
}

// ---------------------------------------------------------------- dispatch

template <int BITS, int MT, int LK, int R, int CH>
cudaError_t launch_cfg(const GemvParams &p, int warps, cudaStream_t s) {
  using F = Fmt<BITS>;
  constexpr int KT = LK * CH * F::CW;
  constexpr int NSUM = F::SUMS ? KT / 32 : 1;
  const size_t smem = sizeof(float4) * MT * (KT / 4) + sizeof(float) * MT * NSUM;
  const int rows_per_cta = warps * (32 / LK) * R;
  const int grid = (p.N + rows_per_cta - 1) / rows_per_cta;
  auto kern = gemv_kernel<BITS, MT, LK, R, CH>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

// Warps per CTA: as many as keep at least ~2 CTAs per SM busy, at most 8.
int pick_warps(int64_t N, int rows_per_warp) {
  const int64_t target = 2LL * sm_count();
  int w = 8;
  while (w > 1 && (N + (int64_t)w * rows_per_warp - 1) / ((int64_t)w * rows_per_warp) < target) w >>= 1;
  return w;
}

template <int BITS, int MT>
cudaError_t launch_bits_m(const GemvParams &p, cudaStream_t s) {
  if (BITS == 4) {
    if (MT == 1) return launch_cfg<4, 1, 8, 2, 4>(p, pick_warps(p.N, 4 * 2), s);
    return launch_cfg<4, MT, 8, 1, 4>(p, pick_warps(p.N, 4 * 1), s);
  } else if (BITS == 8) {
    if (MT == 1) return launch_cfg<8, 1, 8, 2, 8>(p, pick_warps(p.N, 4 * 2), s);
    return launch_cfg<8, MT, 8, 2, 8>(p, pick_warps(p.N, 4 * 2), s);
  } else {
    return launch_cfg<1, MT, 8, 2, 2>(p, pick_warps(p.N, 4 * 2), s);
  }
}

template <int BITS>
cudaError_t launch_bits(const GemvParams &p, cudaStream_t s) {
  if (p.M == 1) return launch_bits_m<BITS, 1>(p, s);
  if (p.M == 2) return launch_bits_m<BITS, 2>(p, s);
  if (p.M <= 4) return launch_bits_m<BITS, 4>(p, s);
  return launch_bits_m<BITS, 8>(p, s);
}

}  // namespace

cudaError_t launch_gemv(const float *x, const uint32_t *codes, const uint16_t *scales,
                        const uint16_t *biases, float *y, int M, int64_t N, int64_t K, int bits,
                        int group, cudaStream_t s) {
  GemvParams p;
  p.x = x;
  p.codes = reinterpret_cast<const uint4 *>(codes);
  p.scales = scales;
  p.biases = biases;
  p.y = y;
  p.M = M;
  p.N = (int)N;
  p.K = (int)K;
  p.gshift = __builtin_ctz((unsigned)group);
  p.chunks_per_row = (int)(K * bits / 128);
  p.groups_per_row = (int)(K / group);
  if (bits == 4 && !(M == 1 && N * K <= ((int64_t)1 << 21))) {
    // INT4: the tensor-core kernel first (measured faster for every shape it
    // takes, except one-token products of at most 2 M weights: 1024 x 1024
    // took 2.94 us there against 2.32 us on the streamed kernel, whose rows
    // need no 16-row tiles)
    cudaError_t e = launch_gemv_tc(x, codes, scales, biases, y, M, N, K, bits, group, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (M == 1 && bits == 1) {
    cudaError_t e = launch_gemv_q1(x, codes, scales, y, N, K, group, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (M >= 2 && ((bits == 8 && M >= 3) || bits == 1)) {
    // 8-bit codes with 3 to 8 tokens and binary codes with 2 to 8 tokens: the
    // tensor-core kernel with K split over a cluster (measured faster)
    cudaError_t e = launch_gemv_tc(x, codes, scales, biases, y, M, N, K, bits, group, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (M >= 2 && M <= 8 && bits == 8) {
    // INT8, 2-8 tokens: the streamed kernel unpacks each code once per pass of up to four
    cudaError_t e = launch_gemv_stream(x, codes, scales, biases, y, M, N, K, bits, group, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (M >= 2) {
    cudaError_t e = launch_gemv_batch(x, codes, scales, biases, y, M, N, K, bits, group, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (M == 1) {
    cudaError_t e = launch_gemv_stream(x, codes, scales, biases, y, 1, N, K, bits, group, s);
    if (e != cudaErrorNotSupported) return e;
  }
  {
    // shapes the kernels above do not take (the same order as the fused
    // argmax head for one token)
    cudaError_t e = launch_gemv_tc(x, codes, scales, biases, y, M, N, K, bits, group, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (bits == 4) return launch_bits<4>(p, s);
  if (bits == 8) return launch_bits<8>(p, s);
  return launch_bits<1>(p, s);
}

cudaError_t launch_gemv_argmax_fused(const float *x, const uint32_t *codes, const uint16_t *scales,
                                     const uint16_t *biases, int64_t N, int64_t K, int bits, int group,
                                     const ArgmaxWork &w, cudaStream_t s) {
  // the same kernel order as launch_gemv for one token (so that the winner's
  // value equals that logit bit for bit)
  if (bits == 4 && N * K > ((int64_t)1 << 21)) {
    const cudaError_t e = launch_gemv_tc_argmax(x, codes, scales, biases, N, K, bits, group, w, s);
    if (e != cudaErrorNotSupported) return e;
  }
  cudaError_t e = launch_gemv_stream_argmax(x, codes, scales, biases, N, K, bits, group, w, s);
  if (e != cudaErrorNotSupported) return e;
  return launch_gemv_tc_argmax(x, codes, scales, biases, N, K, bits, group, w, s);
}

}  // namespace qmm
