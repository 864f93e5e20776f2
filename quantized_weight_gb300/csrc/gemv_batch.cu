// gemv_batch.cu -- small-batch decode product y[M, N] = x[M, K] * dequant(W)^T
// for 2 <= M <= 8 and INT4 / INT8 codes.
//
// Batched decode reads each weight once for all M sequences (the Polaris
// page, "Pushing the limits of legacy hardware", section "Use short context to
// change the state cost", batches decode so the weights are shared).  Each
// code is therefore unpacked once and used M times, and each activation
// loaded is used for several rows: a lane owns R rows (8R-row block: lane =
// 8 row slots x 4 k lanes; R = 4, or 2 for the single-pass INT8 path) and,
// per step, one 32-bit code word of each of its rows and the matching
// activations of MT tokens.
// Per step a lane issues 4 code loads and MT (INT8) or 2*MT (INT4) 16-byte
// activation loads for 4 * MT * (32/bits) multiply-adds.
//
// Layout.  One CTA per SM owns a contiguous slab of rows.  One producer
// thread bulk-copies the slab's coefficients and its codes (row by row, at a
// stride of row_bytes + 16, so the 8 row slots x 4 k lanes of one code load
// hit 32 distinct banks) into shared memory, before the
// programmatic-dependent-launch wait.  The activations of MT tokens are
// staged in shared memory per pass (M > MT takes two passes), except for
// INT8 with 5 to 8 tokens: eight tokens of x do not fit beside the slab, so
// that path reads them from global memory (L1-cached) at each step and takes
// all tokens in one pass.  Consumer warps
// take (32-row block, K part) work items; a lane's 4 k lanes are reduced with
// two shuffles, the K parts of a row in part order: no atomics, the same bits
// on every run.
//
//   INT8  w = s*q: after XOR 0x80 per byte one prmt builds 2^23 + (q + 128),
//         a packed subtract gives q, a packed multiply by s gives w exactly
//         (s*q has at most 18 significant bits).
//   INT4  w = s*q + b: the nibble is masked in place and OR-ed into the bits
//         of 2^23 (2^23 + q*16^c exactly), 2^23 is subtracted, and a packed FMA
//         with the power-of-two pre-scaled s and with b rounds s*q + b once.
//         The activations of each 8-k word are stored in the order
//         (0,1,2,3,5,6,4,7) so that they pair with the nibble classes.
//
// Every mbarrier wait is bounded (bounded_wait.cuh).
#include "bounded_wait.cuh"
#include "qmm_device.cuh"
#include "qmm_launch.h"
#include "sm100_ptx.cuh"

namespace qmm {

__device__ int g_batch_status = 0;

namespace {

using namespace sm100;

constexpr uint32_t kMagic = 0x4B000000u;   // bit pattern of 2^23
constexpr int kMaxConsumerWarps = 15;   // 16 warps: 4 per scheduler, up to 128 registers each
constexpr int kThreads = 32 * (kMaxConsumerWarps + 1);
constexpr int kSmemBudget = 220 * 1024;
constexpr int kMaxRowBlocks = 8;

struct BatchParams {
  const float *x;
  const uint8_t *codes;
  const uint16_t *scales;
  const uint16_t *biases;
  float *y;
  int M, N, K, G, gshift;
  int row_bytes, row_stride;
  int quads;             // 16-byte code quads per row
  int parts, row_blocks;
  int off_x, off_coef, off_red, off_bar;
};

// R rows per lane (row block of 8 * R rows); MT tokens per pass; XG: the
// activations are read from global memory (L1-cached) at each step instead
// of being staged in shared memory (INT8, all tokens in one pass).
template <int BITS, int MT, int R, bool XG>
__global__ void __launch_bounds__(kThreads, 1) gemv_batch_kernel(const BatchParams p) {
  static_assert(!XG || BITS == 8, "global activations only for INT8");
  constexpr int KW = 32 / BITS;                 // weights per code word
  constexpr int kRowsPerBlock = 8 * R;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  float *xs = reinterpret_cast<float *>(smem + p.off_x);                       // [MT][K]
  const uint16_t *sc = reinterpret_cast<const uint16_t *>(smem + p.off_coef);  // [rows][G]
  float *red = reinterpret_cast<float *>(smem + p.off_red);                    // [rows][MT][parts]
  const uint32_t bars = sbase + p.off_bar;
  auto full = [&](int b) { return bars + 8 * b; };
  const uint32_t coef_full = bars + 8 * kMaxRowBlocks;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.off_bar + 8 * (kMaxRowBlocks + 1));
  const WaitCtl ctl{abort_flag, &g_batch_status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int consumers = p.row_blocks * p.parts;
  const int n_begin = (int)((int64_t)blockIdx.x * p.N / gridDim.x);
  const int rows = (int)((int64_t)(blockIdx.x + 1) * p.N / gridDim.x) - n_begin;
  const int nrb = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const int rows_max = p.row_blocks * kRowsPerBlock;

  if (threadIdx.x == 0) {
    for (int b = 0; b <= kMaxRowBlocks; b++) mbar_init(bars + 8 * b, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint32_t gbytes = (uint32_t)rows * p.G * 2;
      mbar_arrive_expect_tx(coef_full, gbytes * (BITS == 4 ? 2 : 1));
      bulk_load(sbase + p.off_coef, p.scales + (int64_t)n_begin * p.G, gbytes, coef_full, pol);
      if (BITS == 4)
        bulk_load(sbase + p.off_coef + (uint32_t)rows_max * p.G * 2, p.biases + (int64_t)n_begin * p.G, gbytes,
                  coef_full, pol);
      for (int b = 0; b < nrb; b++) {
        const int r0 = kRowsPerBlock * b, nr = min(kRowsPerBlock, rows - r0);
        mbar_arrive_expect_tx(full(b), (uint32_t)(nr * p.row_bytes));
        for (int i = 0; i < nr; i++)
          bulk_load(sbase + (uint32_t)((r0 + i) * p.row_stride),
                    p.codes + (int64_t)(n_begin + r0 + i) * p.row_bytes, (uint32_t)p.row_bytes, full(b), pol);
      }
      for (int b = 0; b < nrb; b++) wait_drain(full(b), 0);
      wait_drain(coef_full, 0);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int ct = cw * 32 + lane;
  const int nthreads = consumers * 32;
  const int blk = cw / p.parts, part = cw % p.parts;
  const int rs = lane >> 2, ks = lane & 3;
  const uint16_t *bi = sc + rows_max * p.G;
  pdl_wait();                                                    // x is written by the previous kernel

  bool ok = true;
  bool waited = false;
  for (int m0 = 0; m0 < p.M; m0 += MT) {
    // 1. activations of tokens m0 .. m0+MT-1 (zeros past M), coalesced
    if constexpr (!XG) {
      const int units = MT * (p.K / 4);
      for (int u = ct; u < units; u += nthreads) {
        const int m = u / (p.K / 4), k4 = u - m * (p.K / 4);
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m0 + m < p.M) v = ld_nc_f4(p.x + (int64_t)(m0 + m) * p.K + 4 * k4);
        if (BITS == 4 && (k4 & 1)) v = make_float4(v.y, v.z, v.x, v.w);   // (4,5,6,7) -> (5,6,4,7)
        *reinterpret_cast<float4 *>(xs + m * p.K + 4 * k4) = v;
      }
      asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
    }
    // 2. products of this warp's rows over its K part
    if (blk < nrb) {
      if (!waited) {
        ok = __all_sync(0xffffffffu, wait_bounded(coef_full, 0, ctl)) &&
             __all_sync(0xffffffffu, wait_bounded(full(blk), 0, ctl));
        waited = true;
      }
      if (ok) {
        int row[R];
        bool valid[R];
#pragma unroll
        for (int i = 0; i < R; i++) {
          row[i] = kRowsPerBlock * blk + rs + 8 * i;
          valid[i] = row[i] < rows;
          if (!valid[i]) row[i] = kRowsPerBlock * blk;           // a valid row of the block
        }
        f2 acc[R][MT];
#pragma unroll
        for (int i = 0; i < R; i++)
#pragma unroll
          for (int m = 0; m < MT; m++) acc[i][m] = f2_zero();
        const int q0 = part * p.quads / p.parts, q1 = (part + 1) * p.quads / p.parts;
        int gcur = -1;
        // per row, the group's scale pairs (INT4: s * 16^-c per nibble class) and bias
        f2 sA[R], sB[R], sC[R], bb[R];
        for (int q = q0; q < q1; q++) {
          const int wi = 4 * q + ks;                             // this lane's code word
          const int g = (wi * KW) >> p.gshift;
          if (g != gcur) {
            gcur = g;
#pragma unroll
            for (int i = 0; i < R; i++) {
              const float sv = h2f(sc[row[i] * p.G + g]);
              if constexpr (BITS == 4) {
                const float bv = h2f(bi[row[i] * p.G + g]);
                // exact: powers of two, no underflow for binary16 s
                sA[i] = f2_make(sv, sv * 0.0625f);
                sB[i] = f2_make(sv * 0.00390625f, sv * 0.000244140625f);
                sC[i] = f2_make(sv * 1.52587890625e-05f, sv * 1.52587890625e-05f);
                bb[i] = f2_make(bv, bv);
              } else {
                sA[i] = f2_make(sv, sv);
              }
            }
          }
          if constexpr (BITS == 8) {
            f2 x01[MT], x23[MT];
#pragma unroll
            for (int m = 0; m < MT; m++) {
              float4 v;
              if constexpr (XG)   // tokens past M repeat the last one (their sums are not stored)
                v = ld_nc_f4(p.x + (int64_t)min(m0 + m, p.M - 1) * p.K + 4 * wi);
              else
                v = *reinterpret_cast<const float4 *>(xs + m * p.K + 4 * wi);
              x01[m] = f2_make(v.x, v.y);
              x23[m] = f2_make(v.z, v.w);
            }
            const f2 off2 = f2_make(8388736.0f, 8388736.0f);   // 2^23 + 128
#pragma unroll
            for (int i = 0; i < R; i++) {
              const uint32_t w = *reinterpret_cast<const uint32_t *>(smem + row[i] * p.row_stride + 4 * wi) ^
                                 0x80808080u;
              const f2 w01 = f2_mul(f2_sub(f2_bits(prmt(w, kMagic, 0x7540u), prmt(w, kMagic, 0x7541u)), off2), sA[i]);
              const f2 w23 = f2_mul(f2_sub(f2_bits(prmt(w, kMagic, 0x7542u), prmt(w, kMagic, 0x7543u)), off2), sA[i]);
#pragma unroll
              for (int m = 0; m < MT; m++) {
                acc[i][m] = f2_fma(w01, x01[m], acc[i][m]);
                acc[i][m] = f2_fma(w23, x23[m], acc[i][m]);
              }
            }
          } else {
            f2 xa[MT], xb[MT], xc[MT], xd[MT];                   // (x0,x1) (x2,x3) (x5,x6) (x4,x7)
#pragma unroll
            for (int m = 0; m < MT; m++) {
              const float4 v = *reinterpret_cast<const float4 *>(xs + m * p.K + 8 * wi);
              const float4 u = *reinterpret_cast<const float4 *>(xs + m * p.K + 8 * wi + 4);
              xa[m] = f2_make(v.x, v.y);
              xb[m] = f2_make(v.z, v.w);
              xc[m] = f2_make(u.x, u.y);
              xd[m] = f2_make(u.z, u.w);
            }
            const f2 magic2 = f2_make(8388608.0f, 8388608.0f);
#pragma unroll
            for (int i = 0; i < R; i++) {
              const uint32_t w = *reinterpret_cast<const uint32_t *>(smem + row[i] * p.row_stride + 4 * wi);
              const uint32_t wh = w >> 12;
              const f2 wa = f2_fma(f2_sub(f2_bits(and_or(w, 0xFu, kMagic), and_or(w, 0xF0u, kMagic)), magic2), sA[i], bb[i]);
              const f2 wb = f2_fma(f2_sub(f2_bits(and_or(w, 0xF00u, kMagic), and_or(w, 0xF000u, kMagic)), magic2), sB[i], bb[i]);
              const f2 wc = f2_fma(f2_sub(f2_bits(and_or(wh, 0xF00u, kMagic), and_or(wh, 0xF000u, kMagic)), magic2), sB[i], bb[i]);
              const f2 wd = f2_fma(f2_sub(f2_bits(and_or(w, 0xF0000u, kMagic), and_or(wh, 0xF0000u, kMagic)), magic2), sC[i], bb[i]);
#pragma unroll
              for (int m = 0; m < MT; m++) {
                acc[i][m] = f2_fma(wa, xa[m], acc[i][m]);
                acc[i][m] = f2_fma(wb, xb[m], acc[i][m]);
                acc[i][m] = f2_fma(wc, xc[m], acc[i][m]);
                acc[i][m] = f2_fma(wd, xd[m], acc[i][m]);
              }
            }
          }
        }
        // the 4 k lanes of each row slot, then this part's slot
#pragma unroll
        for (int i = 0; i < R; i++)
#pragma unroll
          for (int m = 0; m < MT; m++) {
            float lo, hi;
            f2_split(acc[i][m], lo, hi);
            float v = lo + hi;
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            if (ks == 0 && valid[i]) red[((kRowsPerBlock * blk + rs + 8 * i) * MT + m) * p.parts + part] = v;
          }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
    // 3. one thread per (row, token) adds the parts in part order
    if (!*abort_flag) {
      for (int idx = ct; idx < rows * MT; idx += nthreads) {
        const int r = idx / MT, m = idx - r * MT;
        if (m0 + m >= p.M) continue;
        float v = 0.0f;
        for (int q = 0; q < p.parts; q++) v += red[idx * p.parts + q];
        p.y[(int64_t)(m0 + m) * p.N + n_begin + r] = v;
      }
    }
    // the activations and partial sums of this pass are no longer read
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  }
}

int sm_count_batch() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

template <int BITS, int MT, int R, bool XG>
cudaError_t launch_mt(const BatchParams &p, int grid, int threads, size_t smem, cudaStream_t s) {
  auto kern = gemv_batch_kernel<BITS, MT, R, XG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
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
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Shared-memory layout for MT tokens per pass and row blocks of rb rows
// (activations staged unless xg); 0 if it does not fit.
size_t layout(BatchParams &p, int MT, int bits, int rb, bool xg) {
  const int rows_max = p.row_blocks * rb;
  const int code_bytes = rows_max * p.row_stride;
  p.off_x = (code_bytes + 127) & ~127;
  p.off_coef = p.off_x + (xg ? 0 : MT * p.K * 4);
  const int coef_bytes = rows_max * p.G * 2 * (bits == 4 ? 2 : 1);
  p.off_red = (p.off_coef + coef_bytes + 15) & ~15;
  const int red_bytes = rows_max * MT * p.parts * 4;
  p.off_bar = (p.off_red + red_bytes + 7) & ~7;
  const size_t smem = (size_t)p.off_bar + 8 * (kMaxRowBlocks + 1) + 16;
  return smem <= (size_t)kSmemBudget ? smem : 0;
}

}  // namespace

// Returns cudaErrorNotSupported (nothing launched) when the slab of rows and
// the activations do not fit in shared memory or the rows are not whole
// 16-byte quads; the caller then uses the register-fed kernel.
cudaError_t launch_gemv_batch(const float *x, const uint32_t *codes, const uint16_t *scales,
                              const uint16_t *biases, float *y, int M, int64_t N, int64_t K, int bits,
                              int group, cudaStream_t s) {
  if ((bits != 4 && bits != 8) || M < 2 || M > 8) return cudaErrorNotSupported;
  BatchParams p{};
  p.x = x;
  p.codes = reinterpret_cast<const uint8_t *>(codes);
  p.scales = scales;
  p.biases = biases;
  p.y = y;
  p.M = M;
  p.N = (int)N;
  p.K = (int)K;
  p.G = (int)(K / group);
  p.gshift = __builtin_ctz((unsigned)group);
  p.row_bytes = (int)(K * bits / 8);
  if (p.row_bytes % 16 != 0 || (p.G * 2) % 16 != 0) return cudaErrorNotSupported;
  p.row_stride = p.row_bytes + 16;
  p.quads = p.row_bytes / 16;
  int grid = sm_count_batch();
  if (N < grid) grid = (int)N;
  const int rows_max = (int)((N + grid - 1) / grid);
  // row blocks of rb rows; the K parts share the consumer warps
  auto setup = [&](int rb) {
    p.row_blocks = (rows_max + rb - 1) / rb;
    if (p.row_blocks > kMaxRowBlocks) return false;
    int parts = kMaxConsumerWarps / p.row_blocks;
    if (parts > p.quads) parts = p.quads;
    p.parts = parts < 1 ? 1 : parts;
    return true;
  };
  auto threads = [&]() { return 32 * (1 + p.row_blocks * p.parts); };
  if (bits == 8 && M > 4 && setup(16)) {
    // INT8, 5..8 tokens: one pass over all of them, 2 rows per lane, the
    // activations read at each step (8 tokens of x do not fit beside the slab)
    const size_t smem = layout(p, 8, bits, 16, true);
    if (smem != 0) return launch_mt<8, 8, 2, true>(p, grid, threads(), smem, s);
  }
  if (!setup(32)) return cudaErrorNotSupported;
  // tokens per pass: all M (rounded up to 2 or 4) when they fit, else 4 or 2
  const int want = M <= 2 ? 2 : 4;
  for (int mt = want; mt >= 2; mt /= 2) {
    const size_t smem = layout(p, mt, bits, 32, false);
    if (smem == 0) continue;
    if (bits == 8)
      return mt == 4 ? launch_mt<8, 4, 4, false>(p, grid, threads(), smem, s)
                     : launch_mt<8, 2, 4, false>(p, grid, threads(), smem, s);
    return mt == 4 ? launch_mt<4, 4, 4, false>(p, grid, threads(), smem, s)
                   : launch_mt<4, 2, 4, false>(p, grid, threads(), smem, s);
  }
  return cudaErrorNotSupported;
}

cudaError_t read_clear_batch_status(int *status, cudaStream_t s) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_batch_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_batch_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace qmm
