// gemv_tc.cu -- decode product y[M, N] = x[M, K] * dequant(W)^T (M = 1..8) on
// the warp-level tensor-core path (mma.sync m16n8k16, f16 inputs, f32
// accumulation).
//
// Decode reads every weight once and is bound by memory bandwidth ("... Tesla
// C2075 ..." paper, section 3.3 "Decode, and why 4-bit is slower"); what
// decides whether a kernel reaches that bound is the instruction cost of
// turning packed codes into products.  Here the tensor cores take the
// multiply-add and the reduction across k, and the only per-weight work left
// on the integer pipes is moving codes into MMA operand registers:
//
//   * A binary16 bit pattern whose bits 11..15 are zero is the integer it
//     spells times 2^-24 (subnormals and the first normal binade share one
//     spacing), and the MMA multiplies such subnormal operands exactly.  So a
//     code masked in place is already an exact operand: INT4 nibbles at bits
//     0..3 and 4..7 of each 16-bit half give q * 2^-24 and 16 q * 2^-24 (one
//     AND each; one shift per word brings the other two nibbles down), INT8
//     bytes (XOR 0x80 makes them q + 128) are spread into 16-bit halves by one
//     byte permute, and a Q1 sign bit i of a half (i <= 10) is 2^i * 2^-24.
//   * The k-dependent factors (1/16 for the upper nibble, 2^-i for a sign
//     bit) are folded into the activation operand, which is built once per
//     CTA: x of each token is scaled by a power of two 2^S (so that its largest
//     magnitude lies in [2^14, 2^15)), split into two binary16 terms hi + lo
//     (22 significant bits, the dropped part at most 2^-22 |x|), and stored in
//     shared memory in the B-fragment order the MMAs read.
//   * Each MMA gives D = 2^-24 * sum(code * x'); per (row, group) the kernel
//     adds s * D and, once per group, the x-only correction (b * sum x' for the
//     INT4 bias, -128 s * sum x' for the INT8 offset, -s * sum x' for Q1's
//     w = s (2 bit - 1)), all in FP32; the sums of x' per group come from the
//     same preparation pass.  y = total * 2^(24 - S), exactly.
//
// Operand layout.  A = 16 weight rows x 16 k (rows g and g + 8 of a lane's
// quad), B = 16 k x 8 columns.  Each lane quad t = 0..3 contributes the k of
// its own code words; a column is non-zero only at the k of the lanes whose
// words belong to the column's group, so one MMA can keep several groups
// apart: with one token the 8 columns are (group of lane t, hi/lo) for the
// four lanes' four different groups, with two tokens (group pair, token,
// hi/lo), and from three tokens on (token, hi/lo) over one group.  The D
// registers of lane t then hold exactly the (group, token) it applies the
// coefficients of, so the per-group epilogue costs a few FMAs per lane.
//
// Layout of the work.  Each CTA (one per SM, or two where a CTA's shared
// memory allows, so that the next product's CTA streams its weights while
// this one computes) owns a contiguous slab of up to 256 rows.  TMA tensor
// copies of eight rows each bring the slab's codes into shared memory as
// 128-byte columns of those rows (the 128-byte swizzle puts the eight rows
// one warp instruction reads in eight different bank groups), and one more
// per coefficient array and box brings the scales (and biases) as 8-group
// blocks; the engine's cost is per copy, so a few large copies replace one
// per row.  The copies do not depend on the previous kernel in the stream,
// so they are issued before the programmatic-dependent-launch wait.  The 16
// warps then take runs of (16-row tile, k-step) work (for 4-bit codes in
// groups of 64 with one token, of whole group sets: a lane quad's four
// groups, two k-steps), the first (units % 16) warps one unit more, so that
// the four warp schedulers get equal shares.  Longer slabs (a vocabulary
// head) stream through a ring of 16-row stages fed by a producer warp, and
// their work units (tile, K slice) go to 15 or 16 consumer warps, each ring
// slot's own.  Partial sums land in per-(unit, row, token) shared-memory
// slots; after a barrier one thread per output adds them in a fixed order:
// no atomics, the same bits on every run.
//
// K split over a cluster (two to eight tokens).  The activation operand of
// eight tokens over the whole K does not fit beside a slab, so these products
// can split K over a thread-block cluster of ks CTAs: every CTA of a cluster
// streams one K slice (whole 128-byte code columns and whole 8-group
// coefficient blocks) of the cluster's rows through the ring and prepares
// the activation operand of its slice only; ranks 1 .. ks-1 write their row
// totals into rank 0's shared memory (distributed shared memory) and rank 0
// adds them in rank order after a cluster barrier.  These are separate
// kernel instantiations, so the one-CTA kernels carry none of it; those for
// 8-bit codes or five to eight tokens may run a 17th warp (16 consumers),
// which the plan takes where it gives each tile its own ring slot.
//
// Every mbarrier wait is bounded (bounded_wait.cuh); a wait that runs out
// aborts the CTA, drains its outstanding copies and records
// QMM_ERR_DEVICE_TIMEOUT for qmm_check().
#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "argmax.cuh"
#include "bounded_wait.cuh"
#include "qmm_device.cuh"
#include "qmm_launch.h"
#include "sm100_ptx.cuh"

namespace qmm {

__device__ int g_tc_status = 0;

// Test hook: the limit the next launch's test wait gets (0: no test wait).
std::atomic<unsigned long long> g_tc_test_wait_ns{0};

namespace {

using namespace sm100;

constexpr int kThreads = 512;              // 16 warps
constexpr int kThreadsRing = 544;          // one-token ring and K split: a producer warp and 16 consumer warps
constexpr int kTileRows = 16;              // rows per MMA tile and per stage
constexpr int kSmemMax = 225 * 1024;
constexpr int kSmemPair = 113 * 1024;      // at most this much shared memory: two CTAs per SM
constexpr int kAmScratch = 2 * 4 * 32;

// Per code format: k per 32-bit word.
template <int FMT> struct Fmt;
template <> struct Fmt<4> { static constexpr int WPK = 8; };
template <> struct Fmt<8> { static constexpr int WPK = 4; };
template <> struct Fmt<1> { static constexpr int WPK = 32; };

struct TcParams {
  const float *x;
  float *y;
  int M, N, K, G, NG;
  int row_bytes, row_words;
  int ncoef;                 // coefficient arrays (2: scales and biases; 1: scales)
  int gpm, lg_gpm;           // groups per MMA (4, 2, 1) and its log2
  int lg_lpg;                // log2 of the lanes per group (4 / gpm)
  int wpg, lg_wpg;           // code words per group row
  int wl, lg_wl;             // words per lane per group
  int npos, spt;             // lane word positions per tile row; UW-steps per tile
  int R;                     // rows of the largest CTA slab (not wide) or of a ring stage (wide: 16)
  int BH;                    // rows per copy box: 8 (not wide: a slab is copied as 8-row boxes) or 16
  int noct;                  // not wide: 8-row blocks of the N rows (split evenly over the CTAs)
  int wide, nks, lg_nks;     // ring + round-robin units of nks K slices per tile
  int stages;                // ring depth (1 when not wide)
  int code_bytes;            // codes of one slab / stage: R * row_bytes (boxes of BH rows one after another)
  int coef_bytes;            // one coefficient array of one slab / stage: R * NG * 2
  int stage_bytes;           // slab / stage: codes, then the coefficient arrays (1024-byte multiple)
  int warp0, nwarps;         // first consumer warp, consumer warps
  int nj2;                   // MMA pairs per tile row (B fragments)
  int nact0, nact1;          // active B lanes per MMA in column blocks 0 and 1
  int pstr0, pstr1;          // bytes per MMA pair of B in column blocks 0 and 1 (16 * nact + 16)
  int off_b, off_xs, off_red, off_zero, off_bar, off_am, off_tw;
  int gs;                    // INT4 group 64, one token, resident slab: k-loop in whole group sets (1) or k-steps (0)
  ArgmaxWork am;
  // K split over a cluster of ks CTAs (wide only; 1: no split).  Rank r of a
  // cluster takes the slice of row_words words (NG groups) starting at word
  // r * row_words of every row of the cluster's rows: all the sizes above
  // are those of one slice.  K is the full length (x's row stride).
  int ks;
  int rmax;                  // rows of the largest cluster row block (its reduction buffer's stride)
  int off_cl;                // shared offset of the reduction buffer (rank 0's is used)
  // Test hook, 0 in every normal launch: > 0 makes the first consumer warp
  // wait on a barrier that never completes, with this limit in nanoseconds,
  // so that the wait runs out and the launch reports a device timeout.
  unsigned long long test_wait_ns;
};

// ---------------------------------------------------------------- helpers

// The test hook's wait (out of line: it runs only when the hook is set).
__device__ __noinline__ void test_wait(uint32_t never_bar, WaitCtl ctl, unsigned long long limit_ns) {
  wait_bounded(never_bar, 0, ctl, limit_ns);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with C = 0 (the first MMA of an accumulator chain).
__device__ __forceinline__ void mma_f16_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Two floats -> two binary16 (round to nearest even): low half from `lo`.
__device__ __forceinline__ uint32_t f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ void f16x2_to_f32(uint32_t v, float &lo, float &hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(v));
}
// The pair (a, b) of activation values as two binary16 terms each:
// hi = f16(a), f16(b); lo = f16 of the exact float residuals.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
  hi = f16x2(a, b);
  float ha, hb;
  f16x2_to_f32(hi, ha, hb);
  lo = f16x2(a - ha, b - hb);
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }   // -126 <= e <= 127

// Exponent S of the activation scale 2^S from the largest |x| bit pattern:
// max |x| * 2^S lies in [2^14, 2^15).  Zero or non-finite maxima take S = 0.
__device__ __forceinline__ int scale_exp(uint32_t mbits) {
  if (mbits == 0u || mbits >= 0x7F800000u) return 0;
  const int e = (int)(mbits >> 23) - 127;
  const int S = 14 - e;
  return S > 126 ? 126 : S;
}

__device__ __forceinline__ uint32_t absbits(float v) { return __float_as_uint(v) & 0x7FFFFFFFu; }

// Code words [word0, word0 + UW) of one row.  A copy box of BH rows holds
// 128-byte columns of its rows (column stride BH * 128 bytes), each 16-byte
// chunk swizzled within its 128-byte line (chunk ^= row & 7, the TMA 128-byte
// swizzle on a 1024-byte-aligned base); `rowb` is the row's line in column 0,
// `sw` its swizzle.  word0 is a multiple of UW.  Plain loads, so that the
// compiler may schedule them early.
template <int UW>
__device__ __forceinline__ void lds_codes(const uint8_t *smem, int rowb, int colstride, int sw, int word0,
                                          uint32_t (&w)[UW]) {
  const uint8_t *lb = smem + (rowb + (word0 >> 5) * colstride);
  const int ch = (word0 >> 2) & 7;
  if constexpr (UW == 1) {
    w[0] = *reinterpret_cast<const uint32_t *>(lb + ((ch ^ sw) << 4) + (word0 & 3) * 4);
  } else if constexpr (UW == 2) {
    const uint2 v = *reinterpret_cast<const uint2 *>(lb + ((ch ^ sw) << 4) + (word0 & 3) * 4);
    w[0] = v.x;
    w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < UW; i += 4) {
      const uint4 v = *reinterpret_cast<const uint4 *>(lb + (((ch + (i >> 2)) ^ sw) << 4));
      w[i] = v.x;
      w[i + 1] = v.y;
      w[i + 2] = v.z;
      w[i + 3] = v.w;
    }
  }
}
__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ uint16_t lds16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

// B column (and its column block) of token m's term tau for the words of lane t.
__device__ __forceinline__ void b_lane(int gpm, int m, int t, int tau, int &cb, int &ai) {
  if (gpm == 4) {
    cb = 0;
    ai = 2 * t + tau;                        // lanes (g = 2t + tau, t), index g
  } else if (gpm == 2) {
    cb = 0;
    ai = 4 * t + 2 * m + tau;                // lanes (g = 4 (t / 2) + 2m + tau, t)
  } else {
    cb = m >> 2;
    ai = 4 * (2 * (m & 3) + tau) + t;        // lanes (g = 2 (m % 4) + tau, t), index = lane id
  }
}

// ---------------------------------------------------------------- kernel

// Not wide: with W working warps (W = min(16, units)), warp w takes the
// work units [run(w), run(w + 1)) of the slab's tiles, in (tile, unit) order;
// every run is non-empty.  The first total % W warps take one unit more, so
// that the four warp schedulers of an SM (warp w on scheduler w % 4) get
// equal shares to within one unit: the loop is bound by each scheduler's issue.
__host__ __device__ __forceinline__ int run_begin(int w, int W, int total) {
  const int q = total / W, r = total - q * W;
  return w * q + (w < r ? w : r);
}

// LAY: 0 resident slab (one-token kernels; the others also take a ring at
// run time), 1 ring (one-token kernels for long slabs, whose shared memory
// holds one CTA per SM: up to 128 registers), 2 ring with K split over a
// cluster.  Separate instantiations keep each kernel's code to the
// layout it runs (code a kernel carries but never runs measured 2 % slower).
template <int FMT, int UW, int MT, int GPM, bool ARGMAX, int LAY>
__global__ void __launch_bounds__(LAY == 1 || (LAY == 2 && (MT == 2 || FMT == 8)) ? kThreadsRing : kThreads,
                                  MT == 1 && LAY != 1 && !(LAY == 2 && FMT == 8) ? 2 : 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
                   const __grid_constant__ CUtensorMap tm_biases, const TcParams p) {
  using F = Fmt<FMT>;
  constexpr int LPG = 4 / GPM;                     // lanes per group
  constexpr int LG_LPG = LPG == 4 ? 2 : LPG == 2 ? 1 : 0;
  constexpr int LG_GPM = GPM == 4 ? 2 : GPM == 2 ? 1 : 0;
  // MMA pairs per code word (INT4: the word's P and Q MMAs; INT8: half a
  // pair; Q1: four pairs), counted in quarter pairs
  // the parameters the loops use, in registers
  const int M = p.M, NG = p.NG, row_words = p.row_words;
  const int wpg = p.wpg, lg_wpg = p.lg_wpg, wl = p.wl, lg_wl = p.lg_wl, npos = p.npos, spt = p.spt;
  constexpr bool SPLIT = LAY == 2;
  const bool wide = LAY != 0 || (GPM != 4 && p.wide != 0);
  const int nks = p.nks, lg_nks = p.lg_nks, S = p.stages, stage_bytes = p.stage_bytes;
  const int code_bytes = p.code_bytes, coef_bytes = p.coef_bytes;
  const int nj2 = p.nj2, nwarps = p.nwarps, warp0 = p.warp0;
  const int BH = p.BH, lg_bh = BH == 16 ? 4 : 3, row_bytes = p.row_bytes, pstr0 = p.pstr0, pstr1 = p.pstr1;

  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the swizzled code columns need a 1024-byte-aligned base (the launch adds
  // 1 KB); pointer arithmetic keeps the shared address space visible
  const uint32_t sraw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (sraw & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bars = sbase + p.off_bar;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.off_bar + 8 * (2 * S));
  const float4 *xgc = reinterpret_cast<const float4 *>(smem + p.off_xs);   // [NG][M] per-(group, token) constants
  int *tw = reinterpret_cast<int *>(smem + p.off_tw);                       // not wide: [tile] first and last warp
  float *red = reinterpret_cast<float *>(smem + p.off_red);
  const WaitCtl ctl{abort_flag, &g_tc_status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // not wide: 8-row blocks split over the CTAs; wide: the CTA's share of the rows
  // (a cluster of ks CTAs shares one row block, each CTA a K slice)
  const int ks = SPLIT ? p.ks : 1;
  const int crank = SPLIT ? (int)cluster_ctarank() : 0;
  int n_begin, rows;
  if (wide) {
    const int ncl = gridDim.x / ks, cl = blockIdx.x / ks;
    n_begin = (int)((int64_t)cl * p.N / ncl);
    rows = (int)((int64_t)(cl + 1) * p.N / ncl) - n_begin;
  } else {
    const int o0 = (int)((int64_t)blockIdx.x * p.noct / gridDim.x);
    const int o1 = (int)((int64_t)(blockIdx.x + 1) * p.noct / gridDim.x);
    n_begin = 8 * o0;
    rows = min(8 * (o1 - o0), p.N - n_begin);
  }
  const int ntiles = (rows + kTileRows - 1) / kTileRows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(bars + 8 * s, 1);
      mbar_init(bars + 8 * (S + s), nks);
    }
    mbar_init(bars + 8 * (2 * S) + 8, 1);      // test hook: initialised, never arrived on
    *abort_flag = 0;
    fence_mbar_init();
  }
  // B of inactive lanes: 16 zero bytes, or 1 KB in the group-set loop (which
  // reads them at the immediate offsets of an active lane's eight fragments)
  if (threadIdx.x < (p.gs ? 64 : 1))
    reinterpret_cast<uint4 *>(smem + p.off_zero)[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  pdl_launch_dependents();

  // Copies: codes as 128-byte swizzled columns, coefficients as 8-group
  // blocks, one box of BH rows each; rows past N are zero-filled.
  const uint32_t box_bytes = (uint32_t)(BH * row_bytes + p.ncoef * BH * NG * 2);
  if (wide) {
    if (warp == 0) {
      // ------------------------------------------------ producer (ring of 16-row stages)
      if (lane == 0) {
        const uint64_t pol = policy_evict_first();
        int j = 0;
        for (int s = 0, ph = 0; j < ntiles; j++) {
          if (j >= S && !wait_bounded(bars + 8 * (S + s), ph ^ 1, ctl)) break;
          const uint32_t st = sbase + s * stage_bytes, fb = bars + 8 * s;
          mbar_arrive_expect_tx(fb, box_bytes);
          tma_load_3d_hint(st, &tm_codes, 0, n_begin + j * kTileRows, crank * (row_words >> 5), fb, pol);
          tma_load_3d_hint(st + code_bytes, &tm_scales, 0, n_begin + j * kTileRows, crank * (NG >> 3), fb, pol);
          if (FMT == 4)
            tma_load_3d_hint(st + code_bytes + coef_bytes, &tm_biases, 0, n_begin + j * kTileRows, crank * (NG >> 3),
                             fb, pol);
          if (++s == S) s = 0, ph ^= 1;
        }
        // the last copies of every slot land before this thread exits (so
        // that a CTA whose consumers gave up never exits with a copy in
        // flight); after a normal run these waits end at once
        const int first = j > S ? j - S : 0;
        for (int i = first; i < j; i++) wait_drain(bars + 8 * (i % S), (i / S) & 1);
      }
      if constexpr (SPLIT) {
        __syncwarp();
        cluster_sync();            // the consumers' cluster reduction (every thread takes part)
      }
      return;
    }
  } else if (threadIdx.x == 0) {
    // the whole slab, resident, as 8-row boxes
    const uint64_t pol = policy_evict_first();
    const int nbox = (rows + 7) >> 3;
    mbar_arrive_expect_tx(bars, (uint32_t)nbox * box_bytes);
    for (int i = 0; i < nbox; i++) {
      tma_load_3d_hint(sbase + i * 8 * row_bytes, &tm_codes, 0, n_begin + 8 * i, 0, bars, pol);
      tma_load_3d_hint(sbase + code_bytes + i * 8 * NG * 2, &tm_scales, 0, n_begin + 8 * i, 0, bars, pol);
      if (FMT == 4)
        tma_load_3d_hint(sbase + code_bytes + coef_bytes + i * 8 * NG * 2, &tm_biases, 0, n_begin + 8 * i, 0, bars,
                         pol);
    }
  }

  // ------------------------------------------------------------ consumers
  const int cw = warp - warp0;
  const int nthreads = nwarps * 32;
  const int ct = cw * 32 + lane;
  const int g = lane >> 2, t = lane & 3;
  // INT4 group 64 with one token (the MLP shapes): the resident-slab loop
  // takes whole group sets (the lane quad's four groups, two k-steps) as its
  // work units, with addresses advanced by constants
  constexpr bool GS_T = FMT == 4 && GPM == 4 && MT == 1 && UW == 4 && LAY == 0;
  const bool gs = GS_T && p.gs != 0;
  const int upt = gs ? (spt >> 1) : spt;                   // work units per tile
  const int total_steps = ntiles * upt;
  const int W = total_steps < 16 ? total_steps : 16;    // not wide: working warps
  // not wide: wait for the slab before the dependent-launch wait (its copies
  // were issued at the start; the wait overlaps the previous kernel's tail)
  const int sb = (wide || cw >= W) ? 0 : run_begin(cw, W, total_steps);
  const int se = (wide || cw >= W) ? 0 : run_begin(cw + 1, W, total_steps);
  // (warp 0 holds the thread that issued the slab's copies: its wait does not
  // stop at an abort, so the CTA never exits with a copy in flight)
  bool ok = true;
  if (!wide) ok = __all_sync(0xffffffffu, wait_bounded(bars, 0, ctl, kWaitLimitNs, warp != 0));

  // ------------------------------------------- products: setup and helpers
  // (none of it depends on x, so it runs before the dependent-launch wait)
  // B fragments of this lane: byte offset and stride per MMA pair (inactive
  // lanes read 16 zero bytes)
  // The tile rows of MMA rows g and g + 8.  A quarter-warp (lanes 8i .. 8i + 7)
  // holds MMA rows 2i and 2i + 1; where each lane of a row reads its own
  // 16-byte chunk (one or two groups per MMA: four chunks of a row per
  // quarter-warp), rows 2i and 2i + 1 would read the same chunks after the
  // 128-byte swizzle (2-way bank conflicts), so those MMA rows map to tile
  // rows i and i + 4, whose swizzles differ in the chunk's bit 2.
  const int gr = GPM == 4 ? g : ((g >> 1) | ((g & 1) << 2));
  int bofs0[MT], bstr[MT], tokv[MT];
#pragma unroll
  for (int cb = 0; cb < MT; cb++) {
    int active, ai;
    if constexpr (GPM == 4) {
      active = (g >> 1) == t;
      ai = g;
    } else if constexpr (GPM == 2) {
      active = (g >> 2) == (t >> 1);
      ai = 4 * t + (g & 3);
    } else {
      active = 4 * cb + (g >> 1) < M;
      ai = 4 * g + t;
    }
    bstr[cb] = active ? (cb ? pstr1 : pstr0) : 0;
    bofs0[cb] = active ? p.off_b + cb * nj2 * pstr0 + ai * 16 : p.off_zero;
    // token whose results lane t holds in column block cb
    tokv[cb] = GPM == 4 ? 0 : GPM == 2 ? (t & 1) : min(4 * cb + t, M - 1);
  }
  const int gsel_lane = t >> LG_LPG;                               // group of this lane within a group set
  const int wofs_lane = (t & (LPG - 1)) << lg_wl;                  // first word of this lane within its group
  const int colstride = BH * 128, kblk = BH * 16;

  float acc[MT][2];
#pragma unroll
  for (int cb = 0; cb < MT; cb++) acc[cb][0] = acc[cb][1] = 0.0f;

  // partial sums of this lane's rows to slot `slot` (lane-quad reduction first)
  auto flush = [&](int slot) {
#pragma unroll
    for (int cb = 0; cb < MT; cb++) {
      float a0 = acc[cb][0], a1 = acc[cb][1];
      if constexpr (GPM == 4) {
        a0 += __shfl_xor_sync(0xffffffffu, a0, 1);
        a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
        a0 += __shfl_xor_sync(0xffffffffu, a0, 2);
        a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
      } else if constexpr (GPM == 2) {
        a0 += __shfl_xor_sync(0xffffffffu, a0, 2);
        a1 += __shfl_xor_sync(0xffffffffu, a1, 2);
      }
      const bool writer = GPM == 4 ? t == 0 : GPM == 2 ? t < 2 : 4 * cb + t < M;
      if (writer) {
        float *dst = red + (slot * M + tokv[cb]) * kTileRows;
        dst[gr] = a0;
        dst[gr + 8] = a1;
      }
      acc[cb][0] = acc[cb][1] = 0.0f;
    }
  };

  // Per-tile row state of this lane: code line of column 0 and swizzle of
  // rows ra and rb, coefficient rows (16-byte blocks of 8 groups, block
  // stride BH * 16 bytes); byte offsets from the shared-memory base.
  int ca = 0, cb8 = 0, swa = 0, swb = 0, ka = 0, kb8 = 0;
  const int box_code = BH * row_bytes, box_coef = BH * NG * 2;
  auto set_rows = [&](int st, int ra, int rb) {
    ca = st + (ra >> lg_bh) * box_code + (ra & (BH - 1)) * 128;
    cb8 = st + (rb >> lg_bh) * box_code + (rb & (BH - 1)) * 128;
    ka = st + code_bytes + (ra >> lg_bh) * box_coef + (ra & (BH - 1)) * 16;
    kb8 = st + code_bytes + (rb >> lg_bh) * box_coef + (rb & (BH - 1)) * 16;
    swa = ra & 7;
    swb = rb & 7;
  };

  // B fragments of the UW words at lane position pst: one 16-byte quarter of
  // an MMA pair per quad (INT4: a word's P and Q; INT8: two words; Q1: a
  // quarter of a word), for each column block.
  constexpr int NQ = FMT == 4 ? UW : FMT == 8 ? UW / 2 : 4 * UW;
  auto load_b = [&](int pst, uint4 (&bf)[MT][NQ]) {
    const int q0 = FMT == 4 ? pst : FMT == 8 ? (pst >> 1) : 4 * pst;
#pragma unroll
    for (int cb = 0; cb < MT; cb++)
#pragma unroll
      for (int q = 0; q < NQ; q++) bf[cb][q] = lds128(smem + bofs0[cb] + (q0 + q) * bstr[cb]);
  };

  // One k-step: UW words per lane starting at word0, with B fragments bf,
  // accumulated into d (zero: d starts from zero).  In the resident-slab
  // layout the k-steps of a group accumulate into one d and step_epi applies
  // the group's coefficients once: at the group's last step, or where a
  // warp's run ends inside the group (the epilogue is linear in d; the x-only
  // term goes with the part that holds the group's first step).  The ring
  // layout, throughput-bound with many warps, keeps one epilogue per k-step
  // (each step's MMA chains independent: measured faster there); `fresh`
  // (a std::integral_constant) selects that at compile time.
  auto step_mma = [&](int word0, const uint4 (&bf)[MT][NQ], float (&d)[2][MT][4], bool zero, auto fresh) {
    constexpr bool FRESH = decltype(fresh)::value;
    if (!FRESH && zero) {
#pragma unroll
      for (int h = 0; h < 2; h++)
#pragma unroll
        for (int cb = 0; cb < MT; cb++) d[h][cb][0] = d[h][cb][1] = d[h][cb][2] = d[h][cb][3] = 0.0f;
    }
    uint32_t wa[UW], wb[UW];
    lds_codes<UW>(smem, ca, colstride, swa, word0, wa);
    lds_codes<UW>(smem, cb8, colstride, swb, word0, wb);
#pragma unroll
    for (int u = 0; u < UW; u++) {
      if constexpr (FMT == 4) {
        const uint32_t w = wa[u], v = wb[u], w8 = w >> 8, v8 = v >> 8;
#pragma unroll
        for (int cb = 0; cb < MT; cb++) {
          const uint4 b = bf[cb][u];
          if (FRESH && u == 0) {
            mma_f16_z(d[0][cb], w & 0x000F000Fu, v & 0x000F000Fu, w & 0x00F000F0u, v & 0x00F000F0u, b.x, b.y);
            mma_f16_z(d[1][cb], w8 & 0x000F000Fu, v8 & 0x000F000Fu, w8 & 0x00F000F0u, v8 & 0x00F000F0u, b.z, b.w);
          } else {
            mma_f16(d[0][cb], w & 0x000F000Fu, v & 0x000F000Fu, w & 0x00F000F0u, v & 0x00F000F0u, b.x, b.y);
            mma_f16(d[1][cb], w8 & 0x000F000Fu, v8 & 0x000F000Fu, w8 & 0x00F000F0u, v8 & 0x00F000F0u, b.z, b.w);
          }
        }
      } else if constexpr (FMT == 8) {
        if ((u & 1) == 0) {
          const uint32_t w0 = wa[u] ^ 0x80808080u, v0 = wb[u] ^ 0x80808080u;
          const uint32_t w1 = wa[u + 1] ^ 0x80808080u, v1 = wb[u + 1] ^ 0x80808080u;
#pragma unroll
          for (int cb = 0; cb < MT; cb++) {
            const uint4 b = bf[cb][u >> 1];
            if (FRESH && u == 0) {
              mma_f16_z(d[0][cb], prmt(w0, 0u, 0x4140u), prmt(v0, 0u, 0x4140u), prmt(w0, 0u, 0x4342u),
                        prmt(v0, 0u, 0x4342u), b.x, b.y);
              mma_f16_z(d[1][cb], prmt(w1, 0u, 0x4140u), prmt(v1, 0u, 0x4140u), prmt(w1, 0u, 0x4342u),
                        prmt(v1, 0u, 0x4342u), b.z, b.w);
            } else {
              mma_f16(d[0][cb], prmt(w0, 0u, 0x4140u), prmt(v0, 0u, 0x4140u), prmt(w0, 0u, 0x4342u),
                      prmt(v0, 0u, 0x4342u), b.x, b.y);
              mma_f16(d[1][cb], prmt(w1, 0u, 0x4140u), prmt(v1, 0u, 0x4140u), prmt(w1, 0u, 0x4342u),
                      prmt(v1, 0u, 0x4342u), b.z, b.w);
            }
          }
        }
      } else {
        const uint32_t w = wa[u], v = wb[u], w11 = w >> 11, v11 = v >> 11;
#pragma unroll
        for (int jp = 0; jp < 4; jp++) {
          uint32_t aw[4], av[4];
#pragma unroll
          for (int q = 0; q < 4; q++) {
            const int i = 4 * jp + q;
            const uint32_t mask = 0x00010001u << (i <= 10 ? i : i - 11);
            aw[q] = (i <= 10 ? w : w11) & mask;
            av[q] = (i <= 10 ? v : v11) & mask;
          }
#pragma unroll
          for (int cb = 0; cb < MT; cb++) {
            const uint4 b = bf[cb][4 * u + jp];
            if (FRESH && u == 0 && jp == 0) {
              mma_f16_z(d[0][cb], aw[0], av[0], aw[1], av[1], b.x, b.y);
              mma_f16_z(d[1][cb], aw[2], av[2], aw[3], av[3], b.z, b.w);
            } else {
              mma_f16(d[0][cb], aw[0], av[0], aw[1], av[1], b.x, b.y);
              mma_f16(d[1][cb], aw[2], av[2], aw[3], av[3], b.z, b.w);
            }
          }
        }
      }
    }
  };

  // The coefficients of group grp applied to its accumulated d, into acc:
  // (s' D + e X) * 2^(24 - S) per (row, group, token), the x-only
  // correction e X only when withx.
  auto step_epi = [&](int grp, bool withx, const float (&d)[2][MT][4]) {
    const int kofs = (grp >> 3) * kblk + (grp & 7) * 2;
    const uint16_t sah = lds16(smem + ka + kofs), sbh = lds16(smem + kb8 + kofs);
    float4 xc[MT];
#pragma unroll
    for (int cb = 0; cb < MT; cb++) xc[cb] = xgc[grp * M + tokv[cb]];
    float sa = h2f(sah), sbv = h2f(sbh);
    float ea = 0.0f, eb = 0.0f;
    if (withx) {
      if constexpr (FMT == 4) {
        ea = h2f(lds16(smem + ka + coef_bytes + kofs));
        eb = h2f(lds16(smem + kb8 + coef_bytes + kofs));
      } else if constexpr (FMT == 8) {
        ea = -128.0f * sa;
        eb = -128.0f * sbv;
      } else {
        ea = -sa;
        eb = -sbv;
      }
    }
    if constexpr (FMT == 1) {
      sa *= 2.0f;
      sbv *= 2.0f;
    }
#pragma unroll
    for (int cb = 0; cb < MT; cb++) {
      const float d0 = (d[0][cb][0] + d[0][cb][1]) + (d[1][cb][0] + d[1][cb][1]);
      const float d1 = (d[0][cb][2] + d[0][cb][3]) + (d[1][cb][2] + d[1][cb][3]);
      const float ta = fmaf(sa, d0, ea * xc[cb].x), tb = fmaf(sbv, d1, eb * xc[cb].x);
      acc[cb][0] = fmaf(ta * xc[cb].y, xc[cb].z, acc[cb][0]);
      acc[cb][1] = fmaf(tb * xc[cb].y, xc[cb].z, acc[cb][1]);
    }
  };


  // Group-set loop (INT4 group 64, one token): per-lane state and the MMAs of
  // four code words of rows g and g + 8 (two k-steps make a group set)
  const int bstep = bstr[0] * 8;                 // B bytes per group set: 1152, or 0 for an inactive lane
  int oa0 = 0, ob0 = 0;                          // chunk 2t of rows g and g + 8 in column 0 (after the swizzle)
  auto tile_rows = [&](int tl) {
    set_rows(0, min(tl * kTileRows + gr, rows - 1), min(tl * kTileRows + gr + 8, rows - 1));
    oa0 = ca + (((2 * t) ^ swa) << 4);
    ob0 = cb8 + (((2 * t) ^ swb) << 4);
  };
  auto mma_words = [&](const uint4 &wa4, const uint4 &wb4, const uint8_t *b8, float (&e)[2][MT][4]) {
    const uint32_t wa[4] = {wa4.x, wa4.y, wa4.z, wa4.w}, wb[4] = {wb4.x, wb4.y, wb4.z, wb4.w};
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const uint4 b = lds128(b8 + u * 144);
      const uint32_t w = wa[u], v = wb[u], w8 = w >> 8, v8 = v >> 8;
      if (u == 0) {
        mma_f16_z(e[0][0], w & 0x000F000Fu, v & 0x000F000Fu, w & 0x00F000F0u, v & 0x00F000F0u, b.x, b.y);
        mma_f16_z(e[1][0], w8 & 0x000F000Fu, v8 & 0x000F000Fu, w8 & 0x00F000F0u, v8 & 0x00F000F0u, b.z, b.w);
      } else {
        mma_f16(e[0][0], w & 0x000F000Fu, v & 0x000F000Fu, w & 0x00F000F0u, v & 0x00F000F0u, b.x, b.y);
        mma_f16(e[1][0], w8 & 0x000F000Fu, v8 & 0x000F000Fu, w8 & 0x00F000F0u, v8 & 0x00F000F0u, b.z, b.w);
      }
    }
  };

  {
    // one MMA on zeros while the previous kernel finishes: the first MMA of a
    // CTA is slow, and this moves its cost off the dependent path (measured
    // 60-70 ns less per chained product)
    float dz[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    mma_f16(dz, 0u, 0u, 0u, 0u, 0u, 0u);
    asm volatile("" ::"f"(dz[0]), "f"(dz[1]), "f"(dz[2]), "f"(dz[3]));
  }
  pdl_wait();                                                  // x is written by the previous kernel

  // ---------------------------------------------- activation preparation
  // One pass, a thread per (token, code word), 16 floats of x per thread
  // per round: per group g of token m the scale 2^S (largest |x| of the group
  // in [2^14, 2^15)); x' = x * 2^S split into binary16 hi + lo and stored as
  // B fragments; per (m, g) the constants {2^-24 sum x', f1, f2} with
  // f1 * f2 = 2^(24 - S).  A warp's 32 words lie in one token (row_words is a
  // multiple of 32) and a group's words in wpg adjacent lanes.
  {
    constexpr int NB = F::WPK >= 16 ? 1 : 16 / F::WPK;        // words per thread per round
    const int total_words = M * row_words;
    float4 *xgw = reinterpret_cast<float4 *>(smem + p.off_xs);
    for (int base0 = cw * 32; base0 < total_words; base0 += NB * nthreads) {
      float xv[NB][F::WPK];
#pragma unroll
      for (int b = 0; b < NB; b++) {
        // word u of the (token, slice word) sequence; a warp's 32 words lie in
        // one token, whose slice starts at word crank * row_words of x's row
        const int ub = base0 + b * nthreads;
        int64_t xo = 0;                                            // float offset of word ub + lane
        if (ub < total_words) {
          xo = (int64_t)(ub + lane) * F::WPK;
          if constexpr (SPLIT) {
            const int mu = ub / row_words;
            xo += (int64_t)mu * (p.K - row_words * F::WPK) + (int64_t)crank * row_words * F::WPK;
          }
        }
        const float4 *src = reinterpret_cast<const float4 *>(p.x + xo);
#pragma unroll
        for (int i = 0; i < F::WPK / 4; i++) {
          const float4 v = __ldg(src + i);
          xv[b][4 * i] = v.x;
          xv[b][4 * i + 1] = v.y;
          xv[b][4 * i + 2] = v.z;
          xv[b][4 * i + 3] = v.w;
        }
      }
#pragma unroll
      for (int b = 0; b < NB; b++) {
        const int ubase = base0 + b * nthreads;
        if (ubase >= total_words) break;                       // warp-uniform
        const int u = ubase + lane;
        const bool valid = u < total_words;
        const int m = ubase / row_words;
        const int wd = u - m * row_words;
        // the group's largest |x| and its sum, reduced in the same shuffle
        // rounds; the sum of x' = 2^S x is the sum of x times 2^S (scaling by
        // a power of two commutes with rounding away from over- and underflow)
        uint32_t mx = 0u;
        float rsum = 0.0f;
#pragma unroll
        for (int e = 0; e < F::WPK; e++) {
          mx = max(mx, absbits(xv[b][e]));
          rsum += xv[b][e];
        }
        if (!valid) mx = 0u, rsum = 0.0f;
        for (int o = 1; o < wpg; o <<= 1) {
          const uint32_t om = __shfl_xor_sync(0xffffffffu, mx, o);
          const float os = __shfl_xor_sync(0xffffffffu, rsum, o);
          mx = max(mx, om);
          rsum += os;
        }
        const int Sx = scale_exp(mx);
        const float sc = pow2f(Sx);
#pragma unroll
        for (int e = 0; e < F::WPK; e++) xv[b][e] *= sc;
        const float wsum = rsum * sc;
        if (!valid) continue;
        const int grp = wd >> lg_wpg, wig = wd & (wpg - 1);
        if (wig == 0) {
          const int ex = 24 - Sx, e1 = ex > 127 ? 127 : ex;
          xgw[grp * M + m] = make_float4(wsum * 5.9604644775390625e-08f, pow2f(e1), pow2f(ex - e1), 0.0f);
        }
        // this word's lane and position in the MMA sequence
        const int gq = grp >> LG_GPM, gsel = grp & (GPM - 1);
        const int lt = (gsel << LG_LPG) + (wig >> lg_wl);
        const int pos = (gq << lg_wl) + (wig & (wl - 1));
        // the hi terms go to the B lane of term 0, the lo terms to that of term 1
        uint8_t *bb[2];
        int ps[2];
#pragma unroll
        for (int tau = 0; tau < 2; tau++) {
          int cb, ai;
          b_lane(GPM, m, lt, tau, cb, ai);
          ps[tau] = cb ? pstr1 : pstr0;
          bb[tau] = smem + p.off_b + cb * nj2 * pstr0 + ai * 16;
        }
        if constexpr (FMT == 4) {
          // MMA pair (P, Q) of this word: P (e0, e4 | e1, e5), Q (e2, e6 | e3, e7)
          uint32_t h[4], l[4];
          split_pair(xv[b][0], xv[b][4], h[0], l[0]);
          split_pair(xv[b][1] * 0.0625f, xv[b][5] * 0.0625f, h[1], l[1]);
          split_pair(xv[b][2], xv[b][6], h[2], l[2]);
          split_pair(xv[b][3] * 0.0625f, xv[b][7] * 0.0625f, h[3], l[3]);
          *reinterpret_cast<uint4 *>(bb[0] + pos * ps[0]) = make_uint4(h[0], h[1], h[2], h[3]);
          *reinterpret_cast<uint4 *>(bb[1] + pos * ps[1]) = make_uint4(l[0], l[1], l[2], l[3]);
        } else if constexpr (FMT == 8) {
          uint32_t h[2], l[2];
          split_pair(xv[b][0], xv[b][1], h[0], l[0]);
          split_pair(xv[b][2], xv[b][3], h[1], l[1]);
          *reinterpret_cast<uint2 *>(bb[0] + (pos >> 1) * ps[0] + 8 * (pos & 1)) = make_uint2(h[0], h[1]);
          *reinterpret_cast<uint2 *>(bb[1] + (pos >> 1) * ps[1] + 8 * (pos & 1)) = make_uint2(l[0], l[1]);
        } else {
          // MMA j of the word: (e_2j, e_16+2j | e_2j+1, e_17+2j), element e of a
          // half at bit position e (e <= 10) or e - 11, so divided by that power
#pragma unroll
          for (int jp = 0; jp < 4; jp++) {
            uint32_t hh[4], ll[4];
#pragma unroll
            for (int q = 0; q < 4; q++) {
              const int i = 4 * jp + q;                    // register index 0..15 (= 2j or 2j + 1)
              const float f = 1.0f / (float)(1 << (i <= 10 ? i : i - 11));
              split_pair(xv[b][i] * f, xv[b][16 + i] * f, hh[q], ll[q]);
            }
            *reinterpret_cast<uint4 *>(bb[0] + (pos * 4 + jp) * ps[0]) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
            *reinterpret_cast<uint4 *>(bb[1] + (pos * 4 + jp) * ps[1]) = make_uint4(ll[0], ll[1], ll[2], ll[3]);
          }
        }
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");

  uint4 bf[MT][NQ];
  float d[2][MT][4];
  if (gs) {
    if constexpr (GS_T) {
      // Group-set units.  Unit j of a tile is group set j: lane t takes group
      // 4j + t, whose 8 code words of a row are the 16-byte chunks 2t and
      // 2t + 1 of 128-byte column j (before the swizzle; the two differ in
      // address bit 4 after it), and whose B fragments are the 8 MMA pairs
      // from 8j on (144 bytes apart: 8 active lanes plus the padding).
      // Inactive B lanes read a 1 KB zero block at the same offsets.
      if (ok && se > sb) {
        int tile = sb / upt;
        int j = sb - tile * upt;
        bool first = j == 0;                                   // this warp took the tile's first unit
        tile_rows(tile);
        const uint8_t *bp = smem + bofs0[0] + j * bstep;
        for (int s = sb; s < se; s++) {
          const int cofs = j << 10;                            // column j (8-row boxes: 1 KB columns)
          float e1[2][MT][4];
          mma_words(lds128(smem + oa0 + cofs), lds128(smem + ob0 + cofs), bp, d);
          mma_words(lds128(smem + (oa0 ^ 16) + cofs), lds128(smem + (ob0 ^ 16) + cofs), bp + 4 * 144, e1);
#pragma unroll
          for (int h = 0; h < 2; h++)
#pragma unroll
            for (int i = 0; i < 4; i++) d[h][0][i] += e1[h][0][i];
          step_epi(4 * j + t, true, d);
          bp += bstep;
          j++;
          if (j == upt || s + 1 == se) {
            flush(cw + tile);                                  // (warp, tile) -> warp + tile is one-to-one
            if (lane == 0 && first) tw[2 * tile] = cw;
            if (lane == 0 && j == upt) tw[2 * tile + 1] = cw;
            if (s + 1 == se) break;
            tile++;
            j = 0;
            first = true;
            bp = smem + bofs0[0];
            tile_rows(tile);
          }
        }
      }
    }
  } else if (!wide) {
    if (ok && se > sb) {
      int tile = sb / spt;
      int pst = (sb - tile * spt) * UW;                        // lane word position in the tile row
      int pst0 = pst;                                          // position of the run's first step in this tile
      int wi = pst & (wl - 1);
      int grp = ((pst >> lg_wl) << LG_GPM) + gsel_lane;
      int word0 = grp * wpg + wofs_lane + wi;
      bool withx = wi == 0, zero = true;
      set_rows(0, min(tile * kTileRows + gr, rows - 1), min(tile * kTileRows + gr + 8, rows - 1));
      for (int s = sb; s < se; s++) {
        load_b(pst, bf);
        step_mma(word0, bf, d, zero, std::false_type{});
        zero = false;
        pst += UW;
        wi += UW;
        word0 += UW;
        if (wi == wl || s + 1 == se) {                          // the group's last step here
          step_epi(grp, withx, d);
          zero = true;
        }
        if (wi == wl) {
          wi = 0;
          grp += GPM;
          word0 += GPM * wpg - wl;
          withx = true;
        }
        if (pst == npos || s + 1 == se) {
          flush(cw + tile);                           // (warp, tile) -> warp + tile is one-to-one
          // the warps that took the tile's first and last k-step record
          // themselves for the final sums
          if (lane == 0 && pst0 == 0) tw[2 * tile] = cw;
          if (lane == 0 && pst == npos) tw[2 * tile + 1] = cw;
          if (s + 1 == se) break;
          tile++;
          pst = 0;
          pst0 = 0;
          wi = 0;
          grp = gsel_lane;
          word0 = grp * wpg + wofs_lane;
          set_rows(0, min(tile * kTileRows + gr, rows - 1), min(tile * kTileRows + gr + 8, rows - 1));
        }
      }
    }
  } else {
    // Each ring slot has its own nks consumer warps (S * nks <= 15 or 16), and a
    // warp takes its slot's tiles in order, so every wait is for the next
    // phase of its own slot: a phase parity can never be taken for another
    // lap (copies may land out of order)
    const int spu = spt >> lg_nks;                   // steps per unit
    const int slot = cw >> lg_nks, kq = cw & (nks - 1);   // the warp's slot and K slice
    for (int tile = slot, lap = 0; ok && cw < S * nks && tile < ntiles; tile += S, lap ^= 1) {
      const int u = tile * nks + kq;
      if (!__all_sync(0xffffffffu, wait_bounded(bars + 8 * slot, lap, ctl))) { ok = false; break; }
      set_rows(slot * stage_bytes, gr, gr + 8);
      int pst = kq * spu * UW;
      int wi = pst & (wl - 1);
      int grp = ((pst >> lg_wl) << LG_GPM) + gsel_lane;
      int word0 = grp * wpg + wofs_lane + wi;
      if (GPM == 4 && wl == 2 * UW && wi == 0 && (spu & 1) == 0) {
        // a group is two k-steps: each into its own accumulators (two
        // independent MMA chains, as with an epilogue per step), added once,
        // and one epilogue per group
        float d2[2][MT][4];
        for (int s = 0; s < spu; s += 2) {
          load_b(pst, bf);
          step_mma(word0, bf, d, true, std::true_type{});
          load_b(pst + UW, bf);
          step_mma(word0 + UW, bf, d2, true, std::true_type{});
#pragma unroll
          for (int h = 0; h < 2; h++)
#pragma unroll
            for (int cb = 0; cb < MT; cb++)
#pragma unroll
              for (int i = 0; i < 4; i++) d[h][cb][i] += d2[h][cb][i];
          step_epi(grp, true, d);
          pst += 2 * UW;
          grp += GPM;
          word0 += GPM * wpg;
        }
      } else {
        for (int s = 0; s < spu; s++) {
          load_b(pst, bf);
          step_mma(word0, bf, d, true, std::true_type{});
          step_epi(grp, wi == 0, d);
          pst += UW;
          wi += UW;
          word0 += UW;
          if (wi == wl) {
            wi = 0;
            grp += GPM;
            word0 += GPM * wpg - wl;
          }
        }
      }
      flush(u);
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * (S + slot));
    }
  }

  // test hook: the first consumer warp waits on the barrier nothing completes;
  // the wait runs out and raises the CTA's abort flag, so no output is written
  if (p.test_wait_ns && cw == 0) test_wait(bars + 8 * (2 * S) + 8, ctl, p.test_wait_ns);
  // every consumer warp gets here; then one thread per output adds the
  // partial sums in a fixed order
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  const bool fin = ok && !*abort_flag;
  auto total = [&](int r, int m) {
    const int tile = r >> 4, rr = r & (kTileRows - 1);
    float sum = 0.0f;
    if (!wide) {
      const int w1 = tw[2 * tile + 1];
      for (int w = tw[2 * tile]; w <= w1; w++) sum += red[((w + tile) * M + m) * kTileRows + rr];
    } else {
      for (int q = 0; q < nks; q++) sum += red[((tile * nks + q) * M + m) * kTileRows + rr];
    }
    return sum;
  };
  if constexpr (ARGMAX) {
    float bv = __int_as_float(0xFF800000);
    int bi = 0x7FFFFFFF;
    if (fin) {
      for (int r = ct; r < rows; r += nthreads) {
        const float v = total(r, 0);
        if (am_better(v, n_begin + r, bv, bi)) bv = v, bi = n_begin + r;
      }
    }
    am_cta_finish(bv, bi, warp0, nwarps, reinterpret_cast<uint32_t *>(smem + p.off_am), 1, nthreads, p.am);
    return;
  }
  float *__restrict__ y = p.y;
  const int N = p.N;
  if constexpr (SPLIT) {
    // K split over the cluster: ranks 1 .. ks-1 hand their row totals to
    // rank 0 through distributed shared memory, with a flag saying whether
    // they finished; rank 0 adds them in rank order (a fixed order) and stores
    const uint32_t cbuf = sbase + p.off_cl;                 // [ks - 1][M][rmax] floats, then [ks - 1] flags
    const int nbuf = (ks - 1) * M * p.rmax;
    if (crank != 0) {
      const uint32_t rb = mapa_shared(cbuf, 0);
      for (int idx = ct; idx < rows * M; idx += nthreads) {
        const int m = idx / rows, r = idx - m * rows;
        st_cluster_f32(rb + 4u * (uint32_t)(((crank - 1) * M + m) * p.rmax + r), fin ? total(r, m) : 0.0f);
      }
      if (ct == 0) st_cluster_u32(rb + 4u * (uint32_t)(nbuf + crank - 1), fin ? 1u : 0u);
    }
    __syncwarp();
    cluster_sync();
    if (crank != 0) return;
    const float *cb = reinterpret_cast<const float *>(smem + p.off_cl);
    const uint32_t *cf = reinterpret_cast<const uint32_t *>(cb + nbuf);
    bool all = fin;
    for (int q = 1; q < ks; q++) all = all && cf[q - 1] != 0u;
    if (!all) return;
    for (int idx = ct; idx < rows * M; idx += nthreads) {
      const int m = idx / rows, r = idx - m * rows;
      float v = total(r, m);
      for (int q = 1; q < ks; q++) v += cb[((q - 1) * M + m) * p.rmax + r];
      y[(int64_t)m * N + n_begin + r] = v;
    }
    return;
  }
  if (!fin) return;
  if (M == 1) {
    for (int r = ct; r < rows; r += nthreads) y[n_begin + r] = total(r, 0);
  } else {
    for (int idx = ct; idx < rows * M; idx += nthreads) {
      const int m = idx / rows, r = idx - m * rows;
      y[(int64_t)m * N + n_begin + r] = total(r, m);
    }
  }
}

// ---------------------------------------------------------------- host plan

int sm_count_tc() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool have_variant(int fmt, int uw, int mt, int gpm, bool argmax);

int ilog2(int v) {
  int l = 0;
  while ((1 << l) < v) l++;
  return l;
}

size_t align1k(size_t v) { return (v + 1023) & ~(size_t)1023; }

bool plan_tc(int fmt, int M, int64_t N, int64_t K, int group, bool argmax, TcParams &p, int &uw_out, int &grid,
             size_t &smem) {
  const int WPK = fmt == 4 ? 8 : fmt == 8 ? 4 : 32;
  const int MPW = fmt == 4 ? 2 : fmt == 8 ? 1 : 8;
  if (K % WPK != 0 || K % group != 0 || group % WPK != 0) return false;
  const int NG = (int)(K / group);
  if (NG % 8 != 0 || NG / 8 > 256) return false;       // coefficient rows in 16-byte blocks, one box
  const int wpg = group / WPK;
  const int row_words = (int)(K / WPK);
  if (row_words % 32 != 0 || row_words / 32 > 256 || wpg > 32) return false;   // 128-byte code columns, one box
  int gpm = 0;
  const int cand[3] = {4, 2, 1};
  for (int i = 0; i < 3 && !gpm; i++) {
    const int c = cand[i];
    if (M == 2 && c == 4) continue;
    if (M >= 3 && c != 1) continue;
    if (NG % c == 0 && (wpg * c) % 4 == 0) gpm = c;
  }
  if (!gpm) return false;
  const int mt = M > 4 ? 2 : 1;
  if (mt == 2 && gpm != 1) return false;
  if (argmax && mt != 1) return false;
  const int wl = wpg * gpm / 4;
  const int npos = row_words / 4;
  const int sms = sm_count_tc();
  const int row_bytes = (int)(K * (fmt == 4 ? 4 : fmt == 8 ? 8 : 1) / 8);
  const int ncoef = fmt == 4 ? 2 : 1;
  int nact0, nact1 = 0;
  if (gpm == 4) nact0 = 8;
  else if (gpm == 2) nact0 = 16;
  else {
    nact0 = 8 * (M < 4 ? M : 4);
    nact1 = M > 4 ? 8 * (M - 4) : 0;
  }
  const int nj2 = npos * MPW / 2;
  // B pair stride, padded by 16 bytes (conflict-free stores in the
  // preparation) unless that costs a slab two CTAs per SM
  int pstr0 = nact0 * 16 + 16, pstr1 = nact1 ? nact1 * 16 + 16 : 0;
  size_t bbytes = (size_t)nj2 * (pstr0 + pstr1);
  const size_t xsbytes = (size_t)M * NG * 16;              // {2^-24 sum x', f1, f2} per (group, token)
  const size_t misc = 16 + 256 + kAmScratch + 16 + 1024;  // zero block, tile table, argmax scratch, abort, alignment
  // INT4 group 64 with one token: the slab loop in group sets, whose inactive
  // B lanes read a 1 KB zero block (1008 bytes more than the 16 above)
  const bool gs_fmt = fmt == 4 && gpm == 4 && mt == 1 && wpg == 8;
  const size_t gs_extra = gs_fmt ? 1008 : 0;

  // rows per CTA: the 8-row blocks of N split evenly over one CTA per SM (so
  // that no SM holds two CTAs of one product); a slab is copied as 8-row
  // boxes, each of whose 128-byte code columns (1 KB) and 16-byte coefficient
  // block columns (128 B) starts on a 1024- and 128-byte boundary
  const int noct = (int)((N + 7) / 8);
  const int grid_nw = noct < sms ? noct : sms;
  const int R = 8 * ((noct + grid_nw - 1) / grid_nw);
  const int ntiles = (R + kTileRows - 1) / kTileRows;

  int best_uw = 0, best_wide = 0, best_S = 1, best_nks = 1, best_spt = 0;
  double best_cost = 1e30;
  for (int uw = 8; uw >= 1; uw >>= 1) {
    if (wl % uw != 0 || !have_variant(fmt, uw, mt, gpm, argmax)) continue;
    const int spt = npos / uw;
    const double step_cost = uw * (1.0 + 0.15 * 8 / (uw * MPW));   // relative cost of one k-step
    // resident slab (up to 256 rows): warps take runs of k-steps
    if (R <= 256) {
      const size_t slab = align1k((size_t)R * row_bytes + (size_t)ncoef * R * NG * 2);
      const size_t rest = xsbytes + (size_t)(15 + ntiles) * M * kTileRows * 4 + misc + gs_extra + 16;
      if (slab + bbytes + rest > (size_t)kSmemPair && slab + (size_t)nj2 * (nact0 + nact1) * 16 + rest <= (size_t)kSmemPair) {
        pstr0 = nact0 * 16;
        pstr1 = nact1 * 16;
        bbytes = (size_t)nj2 * (pstr0 + pstr1);
      }
      // partial sums: one slot per (warp, tile) of the runs, warp + tile
      const size_t sm = slab + bbytes + xsbytes + (size_t)(15 + ntiles) * M * kTileRows * 4 + misc + gs_extra + 16;
      if (sm <= (size_t)kSmemMax) {
        const double cost = (double)((ntiles * spt + 15) / 16) * step_cost;
        if (cost < best_cost) {
          best_cost = cost, best_uw = uw, best_wide = 0, best_S = 1, best_nks = 1, best_spt = spt;
        }
        continue;
      }
    }
    // ring of 16-row stages with a producer warp; each of the S slots has
    // nks consumer warps (S * nks <= 16 with one token, else 15) taking its tiles in order, one K
    // slice each
    if (mt != 1) continue;
    const int rows_w = (int)((N + sms - 1) / sms);
    const int nt_w = (rows_w + kTileRows - 1) / kTileRows;
    const size_t stage = align1k((size_t)kTileRows * row_bytes + (size_t)ncoef * kTileRows * NG * 2);
    const int consumers = gpm == 4 ? 16 : 15;     // one-token rings run with a 17th warp
    for (int nks = 1; nks <= 8 && nks <= spt; nks <<= 1) {
      if (spt % nks) break;
      const int ring = std::min(consumers / nks, nt_w);
      const size_t smw = (size_t)ring * stage + bbytes + xsbytes + (size_t)nt_w * nks * M * kTileRows * 4 + misc +
                         16 * (size_t)ring;
      if (smw > (size_t)kSmemMax) continue;
      // the longest warp: ceil(tiles / S) units of spt / nks steps
      const double c = (double)((nt_w + ring - 1) / ring) * (spt / nks) * step_cost *
                       ((double)nt_w / std::max(1, ntiles));
      if (c < best_cost) {
        best_cost = c, best_uw = uw, best_wide = 1, best_S = ring, best_nks = nks, best_spt = spt;
      }
    }
  }
  if (!best_uw) return false;

  p.ks = 1;
  p.M = M;
  p.N = (int)N;
  p.K = (int)K;
  p.G = group;
  p.NG = NG;
  p.row_bytes = row_bytes;
  p.row_words = row_words;
  p.ncoef = ncoef;
  p.gpm = gpm;
  p.lg_gpm = ilog2(gpm);
  p.lg_lpg = ilog2(4 / gpm);
  p.wpg = wpg;
  p.lg_wpg = ilog2(wpg);
  p.wl = wl;
  p.lg_wl = ilog2(wl);
  p.npos = npos;
  p.spt = best_spt;
  p.wide = best_wide;
  p.nks = best_nks;
  p.lg_nks = ilog2(best_nks);
  p.stages = best_S;
  p.R = best_wide ? kTileRows : R;
  p.BH = best_wide ? kTileRows : 8;
  p.noct = noct;
  p.code_bytes = p.R * row_bytes;
  p.coef_bytes = p.R * NG * 2;
  p.stage_bytes = (int)align1k((size_t)p.code_bytes + (size_t)ncoef * p.coef_bytes);
  p.warp0 = best_wide ? 1 : 0;
  p.nwarps = best_wide ? (gpm == 4 ? 16 : 15) : 16;
  p.nj2 = nj2;
  p.nact0 = nact0;
  p.nact1 = nact1;
  p.pstr0 = pstr0;
  p.pstr1 = pstr1;
  p.gs = gs_fmt && !best_wide && best_uw == 4 && pstr0 == 144 && best_spt % 2 == 0 ? 1 : 0;
  if (best_wide) grid = sms < (N + 7) / 8 ? sms : (int)((N + 7) / 8);
  else grid = grid_nw;
  const int nt_red = best_wide ? (int)((N + grid - 1) / grid + kTileRows - 1) / kTileRows : ntiles;
  size_t off = (size_t)p.stages * p.stage_bytes;
  p.off_b = (int)off;
  off += bbytes;
  p.off_xs = (int)off;
  off += xsbytes;
  p.off_red = (int)off;
  off += (best_wide ? (size_t)nt_red * best_nks : (size_t)(15 + ntiles)) * M * kTileRows * 4;
  p.off_zero = (int)off;
  off += p.gs ? 1024 : 16;
  p.off_tw = (int)off;
  off += 8 * 32;
  p.off_bar = (int)off;
  off += 8 * 2 * p.stages + 16;
  off = (off + 15) & ~(size_t)15;
  p.off_am = (int)off;
  off += kAmScratch;
  smem = off + 1024;                                       // room to align the base to 1024 bytes
  if (smem > (size_t)kSmemMax) return false;
  uw_out = best_uw;
  return true;
}

// Two to eight tokens with K split over a cluster of ks CTAs: each CTA of a
// cluster streams one K slice of the cluster's rows through a ring of 16-row
// stages (wide layout, the sizes in p those of one slice); ncl clusters.
bool plan_tc_split(int fmt, int M, int64_t N, int64_t K, int group, int ks, int ncl, TcParams &p, int &uw_out,
                   int &grid, size_t &smem) {
  const int WPK = fmt == 4 ? 8 : fmt == 8 ? 4 : 32;
  const int MPW = fmt == 4 ? 2 : fmt == 8 ? 1 : 8;
  if (M < 2 || M > 8 || ks < 2 || ks > 8 || ncl < 1) return false;
  if (K % WPK != 0 || K % group != 0 || group % WPK != 0) return false;
  const int NGf = (int)(K / group), rwf = (int)(K / WPK);
  if (rwf % (32 * ks) != 0 || NGf % (8 * ks) != 0) return false;   // whole 128-byte columns and 8-group blocks
  const int NG = NGf / ks, row_words = rwf / ks, wpg = group / WPK;
  if (NG / 8 > 256 || row_words / 32 > 256 || wpg > 32) return false;
  int gpm = 0;
  if (M == 2 && NG % 2 == 0 && (wpg * 2) % 4 == 0) gpm = 2;
  else if (wpg % 4 == 0) gpm = 1;
  if (!gpm) return false;
  const int mt = M > 4 ? 2 : 1;
  if (mt == 2 && gpm != 1) return false;
  const int wl = wpg * gpm / 4;
  const int npos = row_words / 4;
  const int row_bytes = (int)(K * (fmt == 4 ? 4 : fmt == 8 ? 8 : 1) / 8) / ks;
  const int ncoef = fmt == 4 ? 2 : 1;
  const int nact0 = gpm == 2 ? 16 : 8 * (M < 4 ? M : 4);
  const int nact1 = M > 4 ? 8 * (M - 4) : 0;
  const int nj2 = npos * MPW / 2;
  const int pstr0 = nact0 * 16 + 16, pstr1 = nact1 ? nact1 * 16 + 16 : 0;
  const size_t bbytes = (size_t)nj2 * (pstr0 + pstr1);
  const size_t xsbytes = (size_t)M * NG * 16;
  const int rmax = (int)((N + ncl - 1) / ncl);
  const int nt_w = (rmax + kTileRows - 1) / kTileRows;
  int uw = 0;
  for (int c = 8; c >= 1 && !uw; c >>= 1)
    if (wl % c == 0 && have_variant(fmt, c, mt, gpm, false)) uw = c;
  if (!uw) return false;
  const int spt = npos / uw;
  // each of the S ring slots has nks consumer warps (S * nks <= the
  // consumer warps) taking its tiles in order; nks is chosen for the shortest
  // longest warp.  Kernels for 8-bit codes and for 5 to 8 tokens may run 16
  // consumer warps instead of 15 (a 17th warp) with one or two per slot,
  // taken only where that shortens the longest warp: measured 25-30 % faster
  // with 8-bit codes (a ring slot per tile), and 18 % slower for 4-bit codes
  // with eight warps per slot (a two-stage ring); the Q1 kernels for 2 to 4
  // tokens keep 16 warps with two CTAs' registers (25 % slower with 17)
  const size_t stage = align1k((size_t)kTileRows * row_bytes + (size_t)ncoef * kTileRows * NG * 2);
  const size_t cl = ((size_t)(ks - 1) * M * rmax * 4 + 4 * (size_t)(ks - 1) + 15) & ~(size_t)15;
  int nks = 0, S = 0, consumers = 15;
  size_t red = 0;
  long best = 0;
  for (int cons = 15; cons <= (mt == 2 || fmt == 8 ? 16 : 15); cons++)
  for (int c = 1; c <= 8 && c <= spt && spt % c == 0; c <<= 1) {
    if (cons == 16 && c > 2) break;
    const int sc = std::min(nt_w, cons / c);
    const size_t rc = (size_t)nt_w * c * M * kTileRows * 4;
    const size_t fixed = bbytes + xsbytes + rc + 16 + 256 + kAmScratch + cl + 1024 + 64;
    if (sc * stage + fixed + 16 * (size_t)sc > (size_t)kSmemMax) continue;
    const long cost = (long)((nt_w + sc - 1) / sc) * (spt / c);
    if (!nks || cost < best) nks = c, S = sc, red = rc, best = cost, consumers = cons;
  }
  if (!nks) return false;

  p = TcParams{};
  p.ks = ks;
  p.rmax = rmax;
  p.M = M;
  p.N = (int)N;
  p.K = (int)K;
  p.G = group;
  p.NG = NG;
  p.row_bytes = row_bytes;
  p.row_words = row_words;
  p.ncoef = ncoef;
  p.gpm = gpm;
  p.lg_gpm = ilog2(gpm);
  p.lg_lpg = ilog2(4 / gpm);
  p.wpg = wpg;
  p.lg_wpg = ilog2(wpg);
  p.wl = wl;
  p.lg_wl = ilog2(wl);
  p.npos = npos;
  p.spt = spt;
  p.wide = 1;
  p.nks = nks;
  p.lg_nks = ilog2(nks);
  p.stages = S;
  p.R = kTileRows;
  p.BH = kTileRows;
  p.noct = (int)((N + 7) / 8);
  p.code_bytes = kTileRows * row_bytes;
  p.coef_bytes = kTileRows * NG * 2;
  p.stage_bytes = (int)stage;
  p.warp0 = 1;
  p.nwarps = consumers;
  p.nj2 = nj2;
  p.nact0 = nact0;
  p.nact1 = nact1;
  p.pstr0 = pstr0;
  p.pstr1 = pstr1;
  p.gs = 0;
  size_t off = (size_t)S * stage;
  p.off_b = (int)off;
  off += bbytes;
  p.off_xs = (int)off;
  off += xsbytes;
  p.off_red = (int)off;
  off += red;
  p.off_zero = (int)off;
  off += 16;
  p.off_tw = (int)off;
  off += 8 * 32;
  p.off_bar = (int)off;
  off += 8 * 2 * S + 16;
  off = (off + 15) & ~(size_t)15;
  p.off_am = (int)off;
  off += kAmScratch;
  p.off_cl = (int)off;
  off += cl;
  smem = off + 1024;
  if (smem > (size_t)kSmemMax) return false;
  grid = ncl * ks;
  uw_out = uw;
  return true;
}

// Tensor maps of the codes (128-byte columns of R rows, 128-byte swizzle)
// and of one coefficient array (8-group blocks of R rows).
bool encode_maps(const TcParams &p, const void *codes, const void *scales, const void *biases, CUtensorMap &tc,
                 CUtensorMap &ts, CUtensorMap &tb) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tc_encode();
  if (!enc) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  {
    // (a K split copies one slice of every row: the box spans a slice, the
    // tensor the full rows)
    cuuint64_t dims[3] = {32, (cuuint64_t)p.N, (cuuint64_t)(p.ks * p.row_words / 32)};
    cuuint64_t strides[2] = {(cuuint64_t)p.ks * p.row_bytes, 128};
    cuuint32_t box[3] = {32, (cuuint32_t)p.BH, (cuuint32_t)(p.row_words / 32)};
    if (enc(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(codes), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  cuuint64_t dims[3] = {8, (cuuint64_t)p.N, (cuuint64_t)(p.ks * p.NG / 8)};
  cuuint64_t strides[2] = {(cuuint64_t)p.ks * p.NG * 2, 16};
  cuuint32_t box[3] = {8, (cuuint32_t)p.BH, (cuuint32_t)(p.NG / 8)};
  if (enc(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(scales), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  if (!biases) {
    tb = ts;
    return true;
  }
  return enc(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(biases), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int UW, int MT, int GPM, bool ARGMAX, int LAY>
cudaError_t launch_tc_as(const CUtensorMap &tc, const CUtensorMap &ts, const CUtensorMap &tb, const TcParams &p,
                         int grid, size_t smem, cudaStream_t s) {
  constexpr bool SPLIT = LAY == 2;
  auto kern = gemv_tc_kernel<FMT, UW, MT, GPM, ARGMAX, LAY>;
  // the attributes are set once per instantiation and device (and again for
  // a larger shared-memory size): a launch then costs no attribute calls
  static std::atomic<uint64_t> set_for{0};           // (device + 1) << 32 | bytes of the last setting
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t cur = set_for.load(std::memory_order_relaxed);
  if ((cur >> 32) != (uint64_t)(dev + 1) || (cur & 0xFFFFFFFFu) < smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    set_for.store(((uint64_t)(dev + 1) << 32) | (uint64_t)smem, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * (p.warp0 + p.nwarps));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (SPLIT) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.ks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, kern, tc, ts, tb, p);
  if (e == cudaErrorInvalidValue) {
    // the attributes may have been lost with the context (a device reset):
    // set them again and retry once
    (void)cudaGetLastError();
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    set_for.store(((uint64_t)(dev + 1) << 32) | (uint64_t)smem, std::memory_order_relaxed);
    e = cudaLaunchKernelEx(&cfg, kern, tc, ts, tb, p);
  }
  return e;
}

// Clusters of ks CTAs of one kernel variant that fit on the GPU at once.
template <int FMT, int UW, int MT, int GPM>
int max_clusters_as(int ks, size_t smem, int threads) {
  auto kern = gemv_tc_kernel<FMT, UW, MT, GPM, false, 2>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ks);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// The instantiated kernels: (format, k-step UW, column blocks MT, groups per
// MMA GPM); the greedy-argmax variants mirror the one-token ones, so that a
// fused argmax sums exactly as the plain product.
template <bool ARGMAX>
cudaError_t launch_tc(int fmt, int uw, int mt, int gpm, const CUtensorMap &tc, const CUtensorMap &ts,
                      const CUtensorMap &tb, const TcParams &p, int grid, size_t smem, cudaStream_t s) {
  if (gpm == 4 && p.wide) {
#define QMM_TC(F_, U_, T_, G_)                                                        \
  if (fmt == F_ && uw == U_ && mt == T_ && gpm == G_)                                 \
    return launch_tc_as<F_, U_, T_, G_, ARGMAX, 1>(tc, ts, tb, p, grid, smem, s);
    QMM_TC(4, 4, 1, 4) QMM_TC(4, 2, 1, 4)
    QMM_TC(8, 8, 1, 4) QMM_TC(8, 4, 1, 4)
    QMM_TC(1, 2, 1, 4)
#undef QMM_TC
    return cudaErrorNotSupported;
  }
#define QMM_TC(F_, U_, T_, G_)                                                        \
  if (fmt == F_ && uw == U_ && mt == T_ && gpm == G_)                                 \
    return launch_tc_as<F_, U_, T_, G_, ARGMAX, 0>(tc, ts, tb, p, grid, smem, s);
  QMM_TC(4, 4, 1, 4) QMM_TC(4, 2, 1, 4)
  QMM_TC(8, 8, 1, 4) QMM_TC(8, 4, 1, 4)
  QMM_TC(1, 2, 1, 4)
  if constexpr (!ARGMAX) {
    QMM_TC(4, 4, 1, 2) QMM_TC(4, 2, 1, 2)
    QMM_TC(8, 8, 1, 2) QMM_TC(8, 4, 1, 2)
    QMM_TC(4, 4, 1, 1) QMM_TC(4, 2, 1, 1) QMM_TC(4, 4, 2, 1) QMM_TC(4, 2, 2, 1)
    QMM_TC(8, 8, 1, 1) QMM_TC(8, 4, 1, 1) QMM_TC(8, 8, 2, 1) QMM_TC(8, 4, 2, 1)
    QMM_TC(1, 2, 1, 2) QMM_TC(1, 1, 1, 2) QMM_TC(1, 1, 1, 1) QMM_TC(1, 1, 2, 1)
  }
#undef QMM_TC
  return cudaErrorNotSupported;
}

// The K-split kernels (clusters of ks CTAs, two to eight tokens).
cudaError_t launch_tc_split(int fmt, int uw, int mt, int gpm, const CUtensorMap &tc, const CUtensorMap &ts,
                            const CUtensorMap &tb, const TcParams &p, int grid, size_t smem, cudaStream_t s) {
#define QMM_TC(F_, U_, T_, G_) \
  if (fmt == F_ && uw == U_ && mt == T_ && gpm == G_) return launch_tc_as<F_, U_, T_, G_, false, 2>(tc, ts, tb, p, grid, smem, s);
  QMM_TC(4, 4, 1, 2) QMM_TC(4, 2, 1, 2)
  QMM_TC(8, 8, 1, 2) QMM_TC(8, 4, 1, 2)
  QMM_TC(4, 4, 1, 1) QMM_TC(4, 2, 1, 1) QMM_TC(4, 4, 2, 1) QMM_TC(4, 2, 2, 1)
  QMM_TC(8, 8, 1, 1) QMM_TC(8, 4, 1, 1) QMM_TC(8, 8, 2, 1) QMM_TC(8, 4, 2, 1)
  QMM_TC(1, 2, 1, 2) QMM_TC(1, 1, 1, 2) QMM_TC(1, 1, 1, 1) QMM_TC(1, 1, 2, 1)
#undef QMM_TC
  return cudaErrorNotSupported;
}

int max_clusters(int fmt, int uw, int mt, int gpm, int ks, size_t smem, int threads) {
#define QMM_TC(F_, U_, T_, G_) \
  if (fmt == F_ && uw == U_ && mt == T_ && gpm == G_) return max_clusters_as<F_, U_, T_, G_>(ks, smem, threads);
  QMM_TC(4, 4, 1, 2) QMM_TC(4, 2, 1, 2)
  QMM_TC(8, 8, 1, 2) QMM_TC(8, 4, 1, 2)
  QMM_TC(4, 4, 1, 1) QMM_TC(4, 2, 1, 1) QMM_TC(4, 4, 2, 1) QMM_TC(4, 2, 2, 1)
  QMM_TC(8, 8, 1, 1) QMM_TC(8, 4, 1, 1) QMM_TC(8, 8, 2, 1) QMM_TC(8, 4, 2, 1)
  QMM_TC(1, 2, 1, 2) QMM_TC(1, 1, 1, 2) QMM_TC(1, 1, 1, 1) QMM_TC(1, 1, 2, 1)
#undef QMM_TC
  return 0;
}

bool have_variant(int fmt, int uw, int mt, int gpm, bool argmax) {
  if (gpm == 4) return mt == 1 && ((fmt == 4 && (uw == 4 || uw == 2)) || (fmt == 8 && (uw == 8 || uw == 4)) ||
                                   (fmt == 1 && uw == 2));
  if (argmax) return false;
  if (fmt == 4) return (uw == 4 || uw == 2) && (gpm == 1 || mt == 1);
  if (fmt == 8) return (uw == 8 || uw == 4) && (gpm == 1 || mt == 1);
  if (fmt == 1) return gpm == 2 ? mt == 1 && (uw == 2 || uw == 1) : uw == 1;
  return false;
}

}  // namespace

namespace {

// Plans and tensor maps of recent calls, keyed by the weight pointers, the
// shape, the format and the device: a repeated call (a decode loop issuing
// the same projections every token) skips planning, the cluster occupancy
// query and the three tensor-map encodings.  A tensor map holds addresses,
// sizes and strides only, so the weights' contents may change freely.
struct PlanKey {
  const void *codes, *scales, *biases;
  int64_t N, K;
  int M, bits, group, argmax, dev;
  bool operator==(const PlanKey &o) const {
    return codes == o.codes && scales == o.scales && biases == o.biases && N == o.N && K == o.K && M == o.M &&
           bits == o.bits && group == o.group && argmax == o.argmax && dev == o.dev;
  }
};
struct PlanVal {
  bool ok;                       // false: the kernel does not take this call
  TcParams p;
  int uw, grid;
  size_t smem;
  CUtensorMap tc, ts, tb;
};
constexpr int kPlanCache = 64;
std::mutex g_plan_mutex;
PlanKey g_plan_keys[kPlanCache];
PlanVal g_plan_vals[kPlanCache];
int g_plan_count = 0, g_plan_next = 0;

bool plan_lookup(const PlanKey &k, PlanVal &v) {
  std::lock_guard<std::mutex> lock(g_plan_mutex);
  for (int i = 0; i < g_plan_count; i++)
    if (g_plan_keys[i] == k) {
      v = g_plan_vals[i];
      return true;
    }
  return false;
}
void plan_store(const PlanKey &k, const PlanVal &v) {
  std::lock_guard<std::mutex> lock(g_plan_mutex);
  g_plan_keys[g_plan_next] = k;
  g_plan_vals[g_plan_next] = v;
  g_plan_next = (g_plan_next + 1) % kPlanCache;
  if (g_plan_count < kPlanCache) g_plan_count++;
}

// The plan of a decode product on the tensor-core kernel (false: not taken).
bool plan_gemv_tc(int M, int64_t N, int64_t K, int bits, int group, TcParams &p, int &uw, int &grid,
                  size_t &smem) {
  bool planned = false;
  // the K split is measured faster for 8-bit codes with 3 to 8 tokens, for
  // binary codes, and for 4-bit codes with 3 or more tokens over K >= 4096
  // (whose activation operand leaves the slab one CTA per SM: the down
  // projection K = 6144 at 4 tokens 8.1 -> 7.5 us; at 2 tokens the slab is
  // faster); otherwise it is the fallback of the resident-slab plan
  const bool split_first = (bits == 8 && M >= 3) || (bits == 1 && M >= 2) || (bits == 4 && M >= 3 && K >= 4096);
  if (M >= 2 && !split_first) planned = plan_tc(bits, M, N, K, group, false, p, uw, grid, smem);
  if (M >= 2 && !planned) {
    // K split over a cluster, slices of about 1024 k (the smallest split
    // that gets there), on as many clusters as fit at once
    const int sms = sm_count_tc();
    for (int ks = 2; ks <= 8 && !planned; ks++) {
      if (K / ks > 1024 && ks < 8) continue;
      int ncl = sms / ks;
      if (!plan_tc_split(bits, M, N, K, group, ks, ncl, p, uw, grid, smem)) continue;
      const int fit = max_clusters(bits, uw, M > 4 ? 2 : 1, p.gpm, ks, smem, 32 * (p.warp0 + p.nwarps));
      if (fit < 1) continue;
      if (fit < ncl) {
        ncl = fit;
        if (!plan_tc_split(bits, M, N, K, group, ks, ncl, p, uw, grid, smem)) continue;
        if (max_clusters(bits, uw, M > 4 ? 2 : 1, p.gpm, ks, smem, 32 * (p.warp0 + p.nwarps)) < ncl) continue;
      }
      planned = true;
    }
  }
  if (!planned && (M >= 2 && !split_first)) return false;
  if (!planned && !plan_tc(bits, M, N, K, group, false, p, uw, grid, smem)) return false;
  return true;
}

}  // namespace

cudaError_t launch_gemv_tc(const float *x, const uint32_t *codes, const uint16_t *scales, const uint16_t *biases,
                           float *y, int M, int64_t N, int64_t K, int bits, int group, cudaStream_t s) {
  if (M < 1 || M > 8) return cudaErrorNotSupported;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorNotSupported;
  const PlanKey key{codes, scales, biases, N, K, M, bits, group, 0, dev};
  PlanVal v;
  if (!plan_lookup(key, v)) {
    v = PlanVal{};
    v.ok = plan_gemv_tc(M, N, K, bits, group, v.p, v.uw, v.grid, v.smem) &&
           encode_maps(v.p, codes, scales, biases, v.tc, v.ts, v.tb);
    plan_store(key, v);
  }
  if (!v.ok) return cudaErrorNotSupported;
  TcParams p = v.p;
  p.x = x;
  p.y = y;
  p.test_wait_ns = g_tc_test_wait_ns.exchange(0);
  if (p.ks > 1) return launch_tc_split(bits, v.uw, M > 4 ? 2 : 1, p.gpm, v.tc, v.ts, v.tb, p, v.grid, v.smem, s);
  return launch_tc<false>(bits, v.uw, M > 4 ? 2 : 1, p.gpm, v.tc, v.ts, v.tb, p, v.grid, v.smem, s);
}

cudaError_t launch_gemv_tc_argmax(const float *x, const uint32_t *codes, const uint16_t *scales,
                                  const uint16_t *biases, int64_t N, int64_t K, int bits, int group,
                                  const ArgmaxWork &w, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorNotSupported;
  const PlanKey key{codes, scales, biases, N, K, 1, bits, group, 1, dev};
  PlanVal v;
  if (!plan_lookup(key, v)) {
    v = PlanVal{};
    v.ok = plan_tc(bits, 1, N, K, group, true, v.p, v.uw, v.grid, v.smem) && v.grid <= kArgmaxMaxCtas &&
           encode_maps(v.p, codes, scales, biases, v.tc, v.ts, v.tb);
    plan_store(key, v);
  }
  if (!v.ok) return cudaErrorNotSupported;
  TcParams p = v.p;
  p.x = x;
  p.y = nullptr;
  p.am = w;
  p.test_wait_ns = g_tc_test_wait_ns.exchange(0);
  return launch_tc<true>(bits, v.uw, 1, p.gpm, v.tc, v.ts, v.tb, p, v.grid, v.smem, s);
}

void set_tc_test_wait(unsigned long long limit_ns) { g_tc_test_wait_ns.store(limit_ns); }

cudaError_t read_clear_tc_status(int *status, cudaStream_t s) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace qmm
