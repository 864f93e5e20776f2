// gemv_stream.cu -- decode product y[1, N] = x[1, K] * dequant(W)^T, fed by the TMA engine.
//
// Decode reads each weight once and is bound by memory bandwidth ("... Tesla
// C2075 ..." paper, section 3.3 "Decode, and why 4-bit is slower").  At GB300's
// bandwidth a decode-sized matrix (a few MB) must be almost entirely in flight
// at once to keep HBM busy, which registers cannot hold.  So each CTA (one per
// SM) owns a contiguous slab of rows and one producer thread streams the slab
// into shared memory with a handful of large bulk async copies (the TMA
// engine; completion counted on mbarriers): the coefficients of all the slab's
// rows, then the codes in stages of up to 16 rows (for slabs over 128 rows,
// the wide layout: each stage's coefficient rows come with its codes).  The
// weights do not depend on the previous kernel in the stream, so the producer
// runs before the programmatic-dependent-launch wait; where two CTAs fit on an
// SM, a chain of decode products keeps HBM streaming across kernel
// boundaries, and the consumers also wait for the coefficients and first code
// stages before that wait.
//
// After that wait, the consumer warps load x once per CTA (INT4: coalesced
// loads into a transposed shared-memory layout; INT8: each lane's 16 values
// straight into registers); each warp then owns one
// K-segment (32 lanes x 16 bytes of codes: 1024 INT4, 512 INT8 or, with 4-byte
// lanes, 1024 Q1 weights) and keeps that segment's activations in registers.
// A warp takes every wps-th group of 4 rows of the slab; per group the lanes
// form partial dot products with exact bit tricks (below), a transposing
// butterfly reduces the 4 rows over the warp (6 shuffles), and the totals go to
// a per-row, per-segment slot in shared memory.  When every warp is done (a
// named barrier among the consumer warps), one
// thread per row adds the segment slots in segment order and stores y: no
// atomics, the same bits on every run.
//
//   INT4  q*16^c comes out of one lop3 (the masked nibble, left where it sits
//         in the word, OR-ed into the bits of 2^23) and one packed f32x2
//         subtract; nibble pairs of equal position class share a packed FMA
//         accumulator; the group bias is factored out as b * sum(x).
//   INT8  after XOR 0x80 per byte, one prmt builds the float 2^23 + (q + 128).
//   Q1    w*x = +-x: one shift and one lop3 move the sign bit.
//
// Every mbarrier wait is bounded (bounded_wait.cuh); a wait that runs out
// aborts the CTA, drains its outstanding copies and records
// QMM_ERR_DEVICE_TIMEOUT for qmm_check().
#include "argmax.cuh"
#include "bounded_wait.cuh"
#include "qmm_device.cuh"
#include "qmm_launch.h"
#include "sm100_ptx.cuh"

namespace qmm {

__device__ int g_gemv_status = 0;

namespace {

using namespace sm100;

constexpr uint32_t kMagic = 0x4B000000u;   // bit pattern of 2^23
constexpr int RG = 4;                      // rows per group (one butterfly)
constexpr int STAGE_ROWS_MAX = 16;         // rows per code stage
constexpr int kSmemBudget = 200 * 1024;
constexpr int kSmemPair = 108 * 1024;      // leaves room for two CTAs per SM
constexpr int kAmScratch = 8 * 32;         // argmax scratch: two words per consumer warp
constexpr int kMaxConsumerWarps = 15;
constexpr int kMaxConsumerWarpsWide = 27;  // long slabs: one CTA per SM, 28 warps
constexpr int kWideRows = 128;             // slabs longer than this take the wide layout

template <int BITS>
struct Lane {
  static constexpr int BYTES = BITS == 1 ? 4 : 16;     // codes per lane per row
  static constexpr int W = BYTES * 8 / BITS;           // weights per lane per row
  static constexpr int SEG_W = 32 * W;                 // weights per warp segment
  static constexpr int SEG_BYTES = 32 * BYTES;
  static constexpr int PAIRS = W / 2;                  // x register pairs per lane
};

struct StreamParams {
  const float *x;
  const uint8_t *codes;
  const uint16_t *scales;
  const uint16_t *biases;
  float *y;
  int N, K, G, gshift;
  int row_bytes;       // K * bits / 8
  int segs;            // K / SEG_W
  int wps;             // consumer warps per K-segment
  int stage_rows;      // rows per code stage (multiple of RG)
  int stages;          // ring depth
  int rows_per_cta;
  int two_per_sm;      // two CTAs fit on an SM (so the next product's copies start early)
  int wide;            // long slab: wide layout (see the kernel)
  int stage_bytes;     // bytes per ring stage (codes, then in the wide layout the stage's coefficients)
  // shared-memory layout (bytes from the 128-byte-aligned base)
  int off_coef, off_x, off_red, off_bar, off_am;
  ArgmaxWork am;       // used by the argmax epilogue only
  int M;               // tokens: 1, or 2..8 for INT8
  int red_tokens;      // token slots of the partial sums: MT per pass (all tokens, a pass of MT at a time)
};

// INT4, two rows at once; see the file comment.  x pairs per word:
// (x0,x1) (x2,x3) (x5,x6) (x4,x7).
__device__ __forceinline__ void dot2_int4(const uint4 ca, const uint4 cb, const f2 (&xp)[16], float &da,
                                          float &db) {
  const f2 magic2 = f2_make(8388608.0f, 8388608.0f);
  f2 aA = f2_zero(), aB = f2_zero(), aC = f2_zero();
  f2 bA = f2_zero(), bB = f2_zero(), bC = f2_zero();
  const uint32_t wa[4] = {ca.x, ca.y, ca.z, ca.w};
  const uint32_t wb[4] = {cb.x, cb.y, cb.z, cb.w};
#pragma unroll
  for (int wi = 0; wi < 4; wi++) {
    const uint32_t w = wa[wi], wh = w >> 12;
    const uint32_t v = wb[wi], vh = v >> 12;
    const f2 x01 = xp[4 * wi + 0], x23 = xp[4 * wi + 1], x56 = xp[4 * wi + 2], x47 = xp[4 * wi + 3];
    aA = f2_fma(f2_sub(f2_bits(and_or(w, 0xFu, kMagic), and_or(w, 0xF0u, kMagic)), magic2), x01, aA);
    bA = f2_fma(f2_sub(f2_bits(and_or(v, 0xFu, kMagic), and_or(v, 0xF0u, kMagic)), magic2), x01, bA);
    aB = f2_fma(f2_sub(f2_bits(and_or(w, 0xF00u, kMagic), and_or(w, 0xF000u, kMagic)), magic2), x23, aB);
    bB = f2_fma(f2_sub(f2_bits(and_or(v, 0xF00u, kMagic), and_or(v, 0xF000u, kMagic)), magic2), x23, bB);
    aC = f2_fma(f2_sub(f2_bits(and_or(w, 0xF0000u, kMagic), and_or(wh, 0xF0000u, kMagic)), magic2), x47, aC);
    bC = f2_fma(f2_sub(f2_bits(and_or(v, 0xF0000u, kMagic), and_or(vh, 0xF0000u, kMagic)), magic2), x47, bC);
    aB = f2_fma(f2_sub(f2_bits(and_or(wh, 0xF00u, kMagic), and_or(wh, 0xF000u, kMagic)), magic2), x56, aB);
    bB = f2_fma(f2_sub(f2_bits(and_or(vh, 0xF00u, kMagic), and_or(vh, 0xF000u, kMagic)), magic2), x56, bB);
  }
  float t0, t1;
  f2_split(aA, t0, t1);
  float d = fmaf(t1, 0.0625f, t0);
  f2_split(aB, t0, t1);
  d = fmaf(t0, 0.00390625f, d);
  d = fmaf(t1, 0.000244140625f, d);
  f2_split(aC, t0, t1);
  da = fmaf(t0 + t1, 1.52587890625e-05f, d);
  f2_split(bA, t0, t1);
  d = fmaf(t1, 0.0625f, t0);
  f2_split(bB, t0, t1);
  d = fmaf(t0, 0.00390625f, d);
  d = fmaf(t1, 0.000244140625f, d);
  f2_split(bC, t0, t1);
  db = fmaf(t0 + t1, 1.52587890625e-05f, d);
}

__device__ __forceinline__ float dot_int8(const uint4 c, const f2 (&xp)[8]) {
  const f2 off2 = f2_make(8388736.0f, 8388736.0f);     // 2^23 + 128
  f2 a0 = f2_zero(), a1 = f2_zero();
  const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int wi = 0; wi < 4; wi++) {
    const uint32_t w = wv[wi] ^ 0x80808080u;
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

// INT8, tokens 0 .. NQ: each code word unpacked once, multiplied into every
// token's activations (token 0 in xp, tokens 1 .. NQ in xq).
template <int NQ>
__device__ __forceinline__ void dot_int8_mt(const uint4 c, const f2 (&xp)[8], const f2 (&xq)[NQ][8], float &d0,
                                            float (&dq)[NQ]) {
  const f2 off2 = f2_make(8388736.0f, 8388736.0f);     // 2^23 + 128
  f2 a0 = f2_zero(), a1 = f2_zero(), b0[NQ], b1[NQ];
#pragma unroll
  for (int m = 0; m < NQ; m++) b0[m] = f2_zero(), b1[m] = f2_zero();
  const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int wi = 0; wi < 4; wi++) {
    const uint32_t w = wv[wi] ^ 0x80808080u;
    const f2 q01 = f2_sub(f2_bits(prmt(w, kMagic, 0x7540u), prmt(w, kMagic, 0x7541u)), off2);
    const f2 q23 = f2_sub(f2_bits(prmt(w, kMagic, 0x7542u), prmt(w, kMagic, 0x7543u)), off2);
    a0 = f2_fma(q01, xp[2 * wi + 0], a0);
    a1 = f2_fma(q23, xp[2 * wi + 1], a1);
#pragma unroll
    for (int m = 0; m < NQ; m++) {
      b0[m] = f2_fma(q01, xq[m][2 * wi + 0], b0[m]);
      b1[m] = f2_fma(q23, xq[m][2 * wi + 1], b1[m]);
    }
  }
  float c0, c1, c2, c3;
  f2_split(a0, c0, c1);
  f2_split(a1, c2, c3);
  d0 = (c0 + c1) + (c2 + c3);
#pragma unroll
  for (int m = 0; m < NQ; m++) {
    f2_split(b0[m], c0, c1);
    f2_split(b1[m], c2, c3);
    dq[m] = (c0 + c1) + (c2 + c3);
  }
}

__device__ __forceinline__ float dot_q1(const uint32_t w, const f2 (&xp)[16]) {
  f2 a[4] = {f2_zero(), f2_zero(), f2_zero(), f2_zero()};
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    float xa, xb;
    f2_split(xp[j / 2], xa, xb);
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

// Register pair (0 .. PAIRS-1) and slot (0: .x, 1: .y) of activation j
// (0 .. W-1) of a lane.
template <int BITS>
__device__ __forceinline__ int pair_of(int j, int &slot) {
  if constexpr (BITS == 4) {
    // per word: (x0,x1) (x2,x3) (x5,x6) (x4,x7)
    const int o = j & 7;
    const int pidx = (o < 4) ? (o >> 1) : (o == 4 || o == 7) ? 3 : 2;
    slot = (o == 1 || o == 3 || o == 6 || o == 7) ? 1 : 0;
    return 4 * (j >> 3) + pidx;
  } else {
    slot = j & 1;
    return j >> 1;
  }
}

// ARGMAX: instead of storing y, the epilogue reduces this CTA's rows to their
// greedy argmax and the last CTA combines the CTAs' winners (argmax.cuh).
// Stages x (K floats) into shared memory as each lane's register pairs:
// coalesced float4 loads, XU of them in flight per thread before its stores.
template <int BITS, int XU>
__device__ __forceinline__ void stage_x(const float *__restrict__ x, int K, f2 *xs, int ct, int nthreads) {
  using L = Lane<BITS>;
  const int units = K / 4;
  for (int u0 = ct; u0 < units; u0 += XU * nthreads) {
    float4 v[XU];
#pragma unroll
    for (int i = 0; i < XU; i++) {
      const int u = u0 + i * nthreads;
      v[i] = u < units ? ld_nc_f4(x + 4 * u) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < XU; i++) {
      const int u = u0 + i * nthreads;
      if (u >= units) break;
      const int k = 4 * u;
      const int sg = k / L::SEG_W, l = (k % L::SEG_W) / L::W, jj = k % L::W;
      const float vv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int e = 0; e < 4; e++) {
        int slot;
        const int pi = pair_of<BITS>(jj + e, slot);
        float *dst = reinterpret_cast<float *>(&xs[(sg * L::PAIRS + pi) * 32 + l]);
        dst[slot] = vv[e];
      }
    }
  }
}

// WIDE (slabs longer than kWideRows rows, e.g. a vocabulary head): up to 27
// consumer warps (72 registers each: measured faster than 31 at 64), a deep
// ring, and the coefficients of each stage's rows copied with its codes (a
// whole slab's coefficients would crowd out the ring).  Otherwise: up to 15
// consumer warps, two CTAs per SM where they fit, the slab's coefficients
// copied once.
// MT (INT8 only): tokens per pass, each code unpacked once for all of them
// (more tokens: passes over a slab kept resident); the extra activation
// registers leave room for one CTA per SM.
template <int BITS, bool ARGMAX, bool WIDE, int MT>
__global__ void __launch_bounds__(WIDE ? 896 : 512, (WIDE || MT > 1) ? 1 : 2)
    gemv_stream_kernel(const StreamParams p) {
  static_assert(MT == 1 || (BITS == 8 && !ARGMAX && !WIDE), "several tokens: INT8 products only");
  constexpr int NQ = MT > 1 ? MT - 1 : 1;                        // tokens after the first (array extent)
  using L = Lane<BITS>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = p.stages;
  const uint32_t sbase = smem_addr(smem);
  const int code_stage_bytes = p.stage_rows * p.row_bytes;
  const int cbytes_row = p.G * 2;                                 // one coefficient row (scales or biases)
  const uint16_t *sc = reinterpret_cast<const uint16_t *>(smem + p.off_coef);
  const uint16_t *bi = sc + p.rows_per_cta * p.G;
  f2 *xs = reinterpret_cast<f2 *>(smem + p.off_x);                 // [segs][PAIRS][32 lanes]
  float *red = reinterpret_cast<float *>(smem + p.off_red);        // [rows_per_cta][segs][MT]
  const uint32_t bars = sbase + p.off_bar;
  auto full = [&](int s) { return bars + 8 * s; };
  auto empty = [&](int s) { return bars + 8 * (S + s); };
  const uint32_t coef_full = bars + 8 * (2 * S);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.off_bar + 8 * (2 * S + 2));
  const WaitCtl ctl{abort_flag, &g_gemv_status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int consumers = p.segs * p.wps;
  // rows split evenly over the grid (one CTA per SM): every SM gets the
  // same work, and under programmatic dependent launch an SM with room for a
  // second CTA takes one of the next product
  const int n_begin = (int)((int64_t)blockIdx.x * p.N / gridDim.x);
  const int rows = (int)((int64_t)(blockIdx.x + 1) * p.N / gridDim.x) - n_begin;   // <= rows_per_cta
  const int nst = (rows + p.stage_rows - 1) / p.stage_rows;
  const int groups_per_stage = p.stage_rows / RG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), groups_per_stage * p.segs);   // one arrival per (group, segment)
    }
    mbar_init(coef_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      if constexpr (!WIDE) {
        const uint32_t gbytes = (uint32_t)rows * p.G * 2;
        mbar_arrive_expect_tx(coef_full, gbytes * (BITS == 4 ? 2 : 1));
        bulk_load(sbase + p.off_coef, p.scales + (int64_t)n_begin * p.G, gbytes, coef_full, pol);
        if (BITS == 4)
          bulk_load(sbase + p.off_coef + p.rows_per_cta * p.G * 2, p.biases + (int64_t)n_begin * p.G, gbytes,
                    coef_full, pol);
      } else {
        mbar_arrive(coef_full);                                  // the coefficients come with the stages
      }
      int j = 0;
      for (; j < nst; j++) {
        const int s = j % S;
        const uint32_t ph = (j / S) & 1;
        if (!wait_bounded(empty(s), ph ^ 1, ctl)) break;
        const int r0 = j * p.stage_rows;
        const int nr = min(p.stage_rows, rows - r0);
        const uint32_t cbytes = (uint32_t)nr * p.row_bytes;
        const uint32_t gbytes = (uint32_t)(nr * cbytes_row);
        const uint32_t dst = sbase + s * p.stage_bytes;
        mbar_arrive_expect_tx(full(s), cbytes + (WIDE ? gbytes * (BITS == 4 ? 2 : 1) : 0));
        bulk_load(dst, p.codes + (int64_t)(n_begin + r0) * p.row_bytes, cbytes, full(s), pol);
        if constexpr (WIDE) {
          // the stage's scale (and bias) rows, after its codes
          bulk_load(dst + code_stage_bytes, p.scales + (int64_t)(n_begin + r0) * p.G, gbytes, full(s), pol);
          if (BITS == 4)
            bulk_load(dst + code_stage_bytes + p.stage_rows * cbytes_row, p.biases + (int64_t)(n_begin + r0) * p.G,
                      gbytes, full(s), pol);
        }
      }
      // every copy this thread issued lands before it exits, also when the
      // consumers give up later (after a normal run these waits end at once)
      const int first = j > S ? j - S : 0;
      for (int i = first; i < j; i++) wait_drain(full(i % S), (i / S) & 1);
      wait_drain(coef_full, 0);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int ct = cw * 32 + lane;                                // consumer thread index
  const int nthreads = consumers * 32;
  const int seg = cw % p.segs, t0 = cw / p.segs;
  const int ngroups = (rows + RG - 1) / RG;
  // The coefficients and the first S stages of codes (first use of every
  // ring slot) do not depend on the previous kernel: wait for them before the
  // dependent-launch wait, where the waits' latency (a few hundred ns each,
  // even for copies that landed long ago) overlaps the previous product's tail.
  // This pays only when two CTAs share an SM: this CTA's copies were then
  // issued while the previous product ran.  With one CTA per SM the copies
  // start with this kernel, and the x staging below overlaps their transfer.
  bool ok = true;
  int prewaited = -1;                                            // stages < S waited for already
  if (p.two_per_sm) {
    ok = __all_sync(0xffffffffu, wait_bounded(coef_full, 0, ctl));
    for (int grp = t0; ok && grp < ngroups; grp += p.wps) {
      const int j = grp / groups_per_stage;
      if (j >= S) break;
      if (j > prewaited) {
        if (!__all_sync(0xffffffffu, wait_bounded(full(j), 0, ctl))) ok = false;
        prewaited = j;
      }
    }
  }
  pdl_wait();                                                    // x is written by the previous kernel
  // INT8 with more tokens than MT: passes of MT tokens over the same resident
  // slab (plan() then keeps every stage of the slab in shared memory at once)
  const int npass = MT == 4 ? p.red_tokens / MT : 1;           // (two tokens never take a second pass)
  const int rtok = MT == 4 ? p.red_tokens : MT;                  // token slots per partial-sum row
  for (int pass = 0; pass < npass; pass++) {
    const int tok0 = pass * MT;                                    // first token of the pass
    f2 xp[L::PAIRS];
    f2 xq[NQ][L::PAIRS];                                           // tokens 1 .. MT-1 (MT > 1 only)
    if constexpr (BITS == 8) {
      // INT8: this lane's 16 activations (64 contiguous bytes), loaded
      // straight into its register pairs (measured faster than staging)
      const float *src = p.x + (int64_t)(MT == 1 ? 0 : min(tok0, p.M - 1)) * p.K + seg * L::SEG_W + lane * L::W;
#pragma unroll
      for (int i = 0; i < L::W / 4; i++) {
        const float4 v = ld_nc_f4(src + 4 * i);
        xp[2 * i] = f2_make(v.x, v.y);
        xp[2 * i + 1] = f2_make(v.z, v.w);
      }
      if constexpr (MT > 1) {
        // the other tokens; past M the last one repeats (its sums are not stored)
#pragma unroll
        for (int m = 0; m < NQ; m++) {
          const float *sq = p.x + (int64_t)min(tok0 + m + 1, p.M - 1) * p.K + seg * L::SEG_W + lane * L::W;
#pragma unroll
          for (int i = 0; i < L::W / 4; i++) {
            const float4 v = ld_nc_f4(sq + 4 * i);
            xq[m][2 * i] = f2_make(v.x, v.y);
            xq[m][2 * i + 1] = f2_make(v.z, v.w);
          }
        }
      }
    } else {
      // INT4: x once per CTA, coalesced, staged in shared memory as each lane's
      // register pairs (a lane's 128 contiguous bytes load slowly from L1)
      if (p.two_per_sm) stage_x<BITS, 4>(p.x, p.K, xs, ct, nthreads);
      else stage_x<BITS, 1>(p.x, p.K, xs, ct, nthreads);
      // consumer warps only; every consumer thread reaches it (no exit before)
      asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
#pragma unroll
      for (int i = 0; i < L::PAIRS; i++) xp[i] = xs[(seg * L::PAIRS + i) * 32 + lane];
    }
    float xsum = 0.0f;
    if constexpr (BITS == 4) {
#pragma unroll
      for (int i = 0; i < L::PAIRS; i++) {
        float a, b;
        f2_split(xp[i], a, b);
        xsum += a + b;
      }
    }
    const int g = (seg * L::SEG_W + lane * L::W) >> p.gshift;    // a lane chunk lies in one group
    const int lane_off = seg * L::SEG_BYTES + lane * L::BYTES;
    if (!p.two_per_sm && pass == 0) ok = ok && __all_sync(0xffffffffu, wait_bounded(coef_full, 0, ctl));

    // the group's stage j, ring slot s and phase ph (where a warp walks many
    // groups, a wide slab or INT8 with one warp per segment, they advance
    // without a division; measured slower for the short INT4 slabs)
    int j = t0 / groups_per_stage, jrem = t0 - j * groups_per_stage;
    int s = j % S;
    uint32_t ph = (j / S) & 1;
    for (int grp = t0; ok && grp < ngroups; grp += p.wps) {
      if constexpr (WIDE || BITS != 4) {
        if (grp != t0) {
          jrem += p.wps;
          while (jrem >= groups_per_stage) {
            jrem -= groups_per_stage;
            j++;
            if (++s == S) s = 0, ph ^= 1u;
          }
        }
      } else {
        j = grp / groups_per_stage;
        s = j % S;
        ph = (j / S) & 1;
      }
      if (j > prewaited && !__all_sync(0xffffffffu, wait_bounded(full(s), ph, ctl))) { ok = false; break; }
      const int rbase = grp * RG;                                  // first row (within the CTA)
      const int nr = min(RG, rows - rbase);
      const uint8_t *st = smem + s * p.stage_bytes + (rbase - j * p.stage_rows) * p.row_bytes;
      // this group's coefficient rows: in the stage (wide layout), or in the slab
      const uint16_t *scg = sc, *big = bi;
      int crow = rbase;
      if constexpr (WIDE) {
        scg = reinterpret_cast<const uint16_t *>(smem + s * p.stage_bytes + code_stage_bytes);
        big = scg + p.stage_rows * p.G;
        crow = rbase - j * p.stage_rows;
      }
      float part[RG];
      float partq[RG][NQ];                                         // tokens 1 .. MT-1 (MT > 1 only)
      if constexpr (BITS == 4) {
#pragma unroll
        for (int rr = 0; rr < RG; rr += 2) {
          const int ra = rr < nr ? rr : 0, rb = rr + 1 < nr ? rr + 1 : 0;
          float da, db;
          dot2_int4(*reinterpret_cast<const uint4 *>(st + ra * p.row_bytes + lane_off),
                    *reinterpret_cast<const uint4 *>(st + rb * p.row_bytes + lane_off), xp, da, db);
          const int ia = (crow + ra) * p.G + g, ib = (crow + rb) * p.G + g;
          part[rr] = fmaf(h2f(scg[ia]), da, h2f(big[ia]) * xsum);
          part[rr + 1] = fmaf(h2f(scg[ib]), db, h2f(big[ib]) * xsum);
        }
      } else {
#pragma unroll
        for (int rr = 0; rr < RG; rr++) {
          const int r = rr < nr ? rr : 0;
          const uint8_t *cp = st + r * p.row_bytes + lane_off;
          const float sv = h2f(scg[(crow + r) * p.G + g]);
          if constexpr (BITS == 8 && MT > 1) {
            float d0, dq[NQ];
            dot_int8_mt<NQ>(*reinterpret_cast<const uint4 *>(cp), xp, xq, d0, dq);
            part[rr] = sv * d0;
#pragma unroll
            for (int m = 0; m < NQ; m++) partq[rr][m] = sv * dq[m];
          } else if constexpr (BITS == 8) {
            part[rr] = sv * dot_int8(*reinterpret_cast<const uint4 *>(cp), xp);
          } else {
            part[rr] = sv * dot_q1(*reinterpret_cast<const uint32_t *>(cp), xp);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && pass + 1 == npass) mbar_arrive(empty(s));  // this group's codes are consumed
      // transposing butterfly: 4 row partials over 32 lanes in 6 shuffles;
      // afterwards lane l holds the warp total of row 2*bit4(l) + bit3(l)
      const bool h16 = lane & 16, h8 = lane & 8;
      float k0 = h16 ? part[2] : part[0], k1 = h16 ? part[3] : part[1];
      const float s0 = h16 ? part[0] : part[2], s1 = h16 ? part[1] : part[3];
      k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
      k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
      float k = h8 ? k1 : k0;
      const float sk = h8 ? k0 : k1;
      k += __shfl_xor_sync(0xffffffffu, sk, 8);
      k += __shfl_xor_sync(0xffffffffu, k, 4);
      k += __shfl_xor_sync(0xffffffffu, k, 2);
      k += __shfl_xor_sync(0xffffffffu, k, 1);
      const int rr = (h16 ? 2 : 0) + (h8 ? 1 : 0);
      if ((lane & 7) == 0 && rr < nr) red[((rbase + rr) * p.segs + seg) * rtok + tok0] = k;
      if constexpr (MT > 1) {
        // the same butterfly for the other tokens
#pragma unroll
        for (int m = 0; m < NQ; m++) {
          float q0 = h16 ? partq[2][m] : partq[0][m], q1 = h16 ? partq[3][m] : partq[1][m];
          const float t0 = h16 ? partq[0][m] : partq[2][m], t1 = h16 ? partq[1][m] : partq[3][m];
          q0 += __shfl_xor_sync(0xffffffffu, t0, 16);
          q1 += __shfl_xor_sync(0xffffffffu, t1, 16);
          float kq = h8 ? q1 : q0;
          const float tk = h8 ? q0 : q1;
          kq += __shfl_xor_sync(0xffffffffu, tk, 8);
          kq += __shfl_xor_sync(0xffffffffu, kq, 4);
          kq += __shfl_xor_sync(0xffffffffu, kq, 2);
          kq += __shfl_xor_sync(0xffffffffu, kq, 1);
          if ((lane & 7) == 0 && rr < nr) red[((rbase + rr) * p.segs + seg) * rtok + tok0 + 1 + m] = kq;
        }
      }
    }
    prewaited = 0x7FFFFFFF;                                        // a later pass finds every stage waited for
  }
  // every consumer warp gets here (the loop above only ends or breaks), so
  // the named barrier completes; after it, one thread per row adds the
  // segment totals in segment order, unless some wait of the CTA ran out
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  const bool fin = ok && !*abort_flag;
  if constexpr (ARGMAX) {
    // every consumer warp takes part, also after an abort (with no candidate),
    // so the CTA barrier inside completes and the CTA is counted
    float bv = __int_as_float(0xFF800000);
    int bi = 0x7FFFFFFF;
    if (fin) {
      for (int r = ct; r < rows; r += nthreads) {
        float acc = 0.0f;
        for (int q = 0; q < p.segs; q++) acc += red[r * p.segs + q];
        if (am_better(acc, n_begin + r, bv, bi)) bv = acc, bi = n_begin + r;
      }
    }
    am_cta_finish(bv, bi, 1, consumers, reinterpret_cast<uint32_t *>(smem + p.off_am), 1, nthreads, p.am);
    return;
  }
  if (!fin) return;
  if constexpr (MT == 1) {
    for (int r = ct; r < rows; r += nthreads) {
      float acc = 0.0f;
      for (int q = 0; q < p.segs; q++) acc += red[r * p.segs + q];
      p.y[n_begin + r] = acc;
    }
  } else {
    const int rt = rtok;
    for (int idx = ct; idx < rows * rt; idx += nthreads) {
      const int r = idx / rt, m = idx - r * rt;
      if (m >= p.M) continue;
      float acc = 0.0f;
      for (int q = 0; q < p.segs; q++) acc += red[(r * p.segs + q) * rt + m];
      p.y[(int64_t)m * p.N + n_begin + r] = acc;
    }
  }
}

int sm_count_stream() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

template <int BITS>
bool plan(int64_t N, int64_t K, int group, StreamParams &p, int &grid, int &threads, size_t &smem) {
  using L = Lane<BITS>;
  if (K % L::SEG_W != 0) return false;
  const int G = (int)(K / group);
  if ((G * 2) % 16 != 0) return false;                   // coefficient rows must be 16-byte multiples
  p.N = (int)N;
  p.K = (int)K;
  p.G = G;
  p.gshift = __builtin_ctz((unsigned)group);
  p.row_bytes = (int)(K * BITS / 8);
  p.segs = (int)(K / L::SEG_W);
  grid = (int)((N + RG - 1) / RG);
  if (grid > sm_count_stream()) grid = sm_count_stream();
  p.rows_per_cta = (int)((N + grid - 1) / grid);            // the largest slab of the even split
  p.wide = p.rows_per_cta > kWideRows ? 1 : 0;
  if (p.wide && p.M > 1) return false;                          // 32 warps leave too few registers for several tokens
  const int max_warps = p.wide ? kMaxConsumerWarpsWide : kMaxConsumerWarps;
  if (p.segs > max_warps) return false;
  const int coef_row = G * 2 * (BITS == 4 ? 2 : 1);              // coefficient bytes per row
  const int coef = p.wide ? 0 : p.rows_per_cta * coef_row;      // the slab's, copied once
  const int srow = p.row_bytes + (p.wide ? coef_row : 0);        // ring bytes per row
  const int xbytes = BITS == 8 ? 0 : (int)K * 4;               // INT8 loads x into registers
  const int mt = p.M <= 1 ? 1 : p.M <= 2 ? 2 : 4;              // tokens per pass
  const int npass = (p.M + mt - 1) / mt;
  p.red_tokens = mt * npass;
  const int redb = p.rows_per_cta * p.segs * 4 * p.red_tokens;
  const int fixed = coef + xbytes + redb + 8 * 64 + kAmScratch;
  int stage_rows0 = STAGE_ROWS_MAX;
  while (stage_rows0 > RG && stage_rows0 / 2 >= p.rows_per_cta) stage_rows0 /= 2;
  // Prefer a ring small enough for two CTAs per SM (the next product's CTA
  // then starts, and its first copies land, while this one still runs), as
  // long as it keeps two stages in flight; else the deepest ring that fits.
  // A wide slab takes the deepest ring that fits.
  int S = 0;
  for (int sr = stage_rows0; !p.wide && npass == 1 && sr >= RG && S == 0; sr /= 2) {
    const int nst = (p.rows_per_cta + sr - 1) / sr;
    int s2 = (kSmemPair - fixed) / (sr * srow);
    if (s2 > nst) s2 = nst;
    if (s2 >= 2 || s2 == nst) S = s2, p.stage_rows = sr;
  }
  if (S < 1) {
    p.stage_rows = stage_rows0;
    const int nst = (p.rows_per_cta + p.stage_rows - 1) / p.stage_rows;
    S = (kSmemBudget - fixed) / (p.stage_rows * srow);
    if (S > nst) S = nst;
  }
  if (S < 1) return false;
  // several passes read the slab again: all of it must stay resident
  if (npass > 1 && S < (p.rows_per_cta + p.stage_rows - 1) / p.stage_rows) return false;
  const int stage_bytes = p.stage_rows * srow;
  p.stage_bytes = stage_bytes;
  p.stages = S;
  p.off_coef = S * stage_bytes;
  p.off_x = (p.off_coef + coef + 15) & ~15;
  p.off_red = p.off_x + xbytes;
  p.off_bar = (p.off_red + redb + 7) & ~7;
  p.off_am = (p.off_bar + 8 * (2 * S + 2) + 16 + 15) & ~15;
  smem = (size_t)p.off_am + kAmScratch;
  p.two_per_sm = 2 * (smem + 1024) <= 228 * 1024 ? 1 : 0;   // 1 KB reserved per CTA
  int wps = max_warps / p.segs;
  const int ngroups = (p.rows_per_cta + RG - 1) / RG;
  if (wps > ngroups) wps = ngroups;
  if (wps < 1) wps = 1;
  p.wps = wps;
  threads = 32 * (1 + p.segs * wps);
  return true;
}

template <int BITS, bool ARGMAX, bool WIDE, int MT = 1>
cudaError_t launch_stream_as(const StreamParams &p0, int grid, int threads, size_t smem, cudaStream_t s) {
  auto kern = gemv_stream_kernel<BITS, ARGMAX, WIDE, MT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // Every instantiation asks for the same (largest) shared-memory carveout, so
  // that a CTA of the next decode product can join an SM that still runs one
  // of the previous product (programmatic dependent launch overlap).
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p0);
}

template <int BITS, bool ARGMAX>
cudaError_t launch_stream(const StreamParams &p0, int grid, int threads, size_t smem, cudaStream_t s) {
  if constexpr (BITS == 8 && !ARGMAX) {
    if (p0.M > 1) {   // (plan() keeps several tokens out of the wide layout)
      if (p0.M <= 2) return launch_stream_as<BITS, ARGMAX, false, 2>(p0, grid, threads, smem, s);
      return launch_stream_as<BITS, ARGMAX, false, 4>(p0, grid, threads, smem, s);
    }
  }
  return p0.wide ? launch_stream_as<BITS, ARGMAX, true>(p0, grid, threads, smem, s)
                 : launch_stream_as<BITS, ARGMAX, false>(p0, grid, threads, smem, s);
}

}  // namespace

// Returns cudaErrorNotSupported when the shape does not fit this kernel's
// layout (K not a whole number of warp segments, more segments than consumer warps,
// coefficient rows not 16-byte multiples, or a slab too large for shared
// memory); the caller then uses the register-fed kernel.
cudaError_t launch_gemv_stream(const float *x, const uint32_t *codes, const uint16_t *scales,
                               const uint16_t *biases, float *y, int M, int64_t N, int64_t K, int bits, int group,
                               cudaStream_t s) {
  if (M < 1 || M > 8 || (M > 1 && bits != 8)) return cudaErrorNotSupported;
  StreamParams p{};
  p.M = M;
  p.x = x;
  p.codes = reinterpret_cast<const uint8_t *>(codes);
  p.scales = scales;
  p.biases = biases;
  p.y = y;
  int grid = 0, threads = 0;
  size_t smem = 0;
  bool ok = bits == 4 ? plan<4>(N, K, group, p, grid, threads, smem)
            : bits == 8 ? plan<8>(N, K, group, p, grid, threads, smem)
                        : plan<1>(N, K, group, p, grid, threads, smem);
  if (!ok) return cudaErrorNotSupported;
  if (bits == 4) return launch_stream<4, false>(p, grid, threads, smem, s);
  if (bits == 8) return launch_stream<8, false>(p, grid, threads, smem, s);
  return launch_stream<1, false>(p, grid, threads, smem, s);
}

cudaError_t launch_gemv_stream_argmax(const float *x, const uint32_t *codes, const uint16_t *scales,
                                      const uint16_t *biases, int64_t N, int64_t K, int bits, int group,
                                      const ArgmaxWork &w, cudaStream_t s) {
  StreamParams p{};
  p.x = x;
  p.codes = reinterpret_cast<const uint8_t *>(codes);
  p.scales = scales;
  p.biases = biases;
  p.y = nullptr;
  p.M = 1;
  p.am = w;
  int grid = 0, threads = 0;
  size_t smem = 0;
  bool ok = bits == 4 ? plan<4>(N, K, group, p, grid, threads, smem)
            : bits == 8 ? plan<8>(N, K, group, p, grid, threads, smem)
                        : plan<1>(N, K, group, p, grid, threads, smem);
  if (!ok || grid > kArgmaxMaxCtas) return cudaErrorNotSupported;
  if (bits == 4) return launch_stream<4, true>(p, grid, threads, smem, s);
  if (bits == 8) return launch_stream<8, true>(p, grid, threads, smem, s);
  return launch_stream<1, true>(p, grid, threads, smem, s);
}

cudaError_t read_clear_gemv_status(int *status, cudaStream_t s) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_gemv_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_gemv_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace qmm
