// gemv_q1.cu -- binary (Q1) decode product y[1, N] = x[1, K] * dequant(W)^T
// through per-chunk lookup tables.
//
// A Q1 weight is s * (+1 or -1), so a row's product over four consecutive k
// only ever takes one of 16 values: the signed sums +-x0 +-x1 +-x2 +-x3.
// Those 16 sums depend on x alone, so each CTA builds them once for every
// 4-k chunk (K/4 tables of 16 floats) and every 4 weights of every row then
// cost one table lookup and one add, instead of a sign flip and an add per
// weight.  This is the lookup-table idea that the Maxwell Q1 page ("A 27B
// model on two 4GB Maxwell GPUs: inference tuning", section "A packed Q1
// prefill kernel with a narrow dispatch window") points to for binary
// weights.
//
// Layout.  One CTA per SM owns a contiguous slab of rows; one producer
// thread bulk-copies the slab's fp16 scales and its codes into shared memory
// (codes row by row, at a stride of row_bytes + 16 so that the 32 rows read by
// one warp instruction fall in distinct bank groups), before the
// programmatic-dependent-launch wait.  Consumer warps then build the tables
// from x and take (32-row block, K part) work items: lane i walks row
// 32*block + i over the part's k range.  All 32 lanes of an instruction read
// the same 64-byte table, so a lookup is one shared-memory wavefront (equal
// nibbles broadcast, distinct nibbles hit distinct banks).  Per group the
// lookups are summed in k order and scaled by the group's scale; the parts
// of a row are added in part order at the end: no atomics, the same bits on
// every run.
//
// Every mbarrier wait is bounded (bounded_wait.cuh).
#include "bounded_wait.cuh"
#include "qmm_device.cuh"
#include "qmm_launch.h"
#include "sm100_ptx.cuh"

namespace qmm {

__device__ int g_q1_status = 0;

namespace {

using namespace sm100;

constexpr int kMaxConsumerWarps = 28;
constexpr int kThreadsMax = 32 * (kMaxConsumerWarps + 1);
constexpr int kSmemBudget = 220 * 1024;
constexpr int kMaxRowBlocks = 8;

struct Q1Params {
  const float *x;
  const uint8_t *codes;
  const uint16_t *scales;
  float *y;
  int N, K, G;            // G = groups per row
  int group_words;        // 32-bit code words per group (1, 2 or 4); selects the kernel
  int row_bytes, row_stride;
  int units;              // 128-k units per row
  int parts;              // K parts per row block
  int row_blocks;         // 32-row blocks of the largest slab
  int off_tab, off_coef, off_red, off_bar;
};

// The 16 signed sums of x[4c .. 4c+3] (bit j of the index set: +x_j, clear: -x_j),
// added as (+-x0 +-x1) + (+-x2 +-x3).
__device__ __forceinline__ void build_table(const float4 v, float (&t)[16]) {
  const float a[4] = {-v.x - v.y, v.x - v.y, -v.x + v.y, v.x + v.y};
  const float b[4] = {-v.z - v.w, v.z - v.w, -v.z + v.w, v.z + v.w};
#pragma unroll
  for (int i = 0; i < 16; i++) t[i] = a[i & 3] + b[i >> 2];
}

// GW: 32-bit code words per group (group / 32).
template <int GW>
__global__ void __launch_bounds__(kThreadsMax, 1) gemv_q1_kernel(const Q1Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_addr(smem);
  const uint16_t *sc = reinterpret_cast<const uint16_t *>(smem + p.off_coef);
  float *red = reinterpret_cast<float *>(smem + p.off_red);
  const uint32_t bars = sbase + p.off_bar;
  auto full = [&](int b) { return bars + 8 * b; };
  const uint32_t coef_full = bars + 8 * kMaxRowBlocks;
  const uint32_t done_bar = coef_full + 8;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.off_bar + 8 * (kMaxRowBlocks + 2));
  const WaitCtl ctl{abort_flag, &g_q1_status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int consumers = p.row_blocks * p.parts;
  const int n_begin = (int)((int64_t)blockIdx.x * p.N / gridDim.x);
  const int rows = (int)((int64_t)(blockIdx.x + 1) * p.N / gridDim.x) - n_begin;
  const int nrb = (rows + 31) / 32;

  if (threadIdx.x == 0) {
    for (int b = 0; b < kMaxRowBlocks; b++) mbar_init(full(b), 1);
    mbar_init(coef_full, 1);
    mbar_init(done_bar, consumers);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint32_t cbytes = (uint32_t)rows * p.G * 2;
      mbar_arrive_expect_tx(coef_full, cbytes);
      bulk_load(sbase + p.off_coef, p.scales + (int64_t)n_begin * p.G, cbytes, coef_full, pol);
      for (int b = 0; b < nrb; b++) {
        const int r0 = 32 * b, nr = min(32, rows - r0);
        mbar_arrive_expect_tx(full(b), (uint32_t)(nr * p.row_bytes));
        for (int i = 0; i < nr; i++)
          bulk_load(sbase + (uint32_t)((r0 + i) * p.row_stride),
                    p.codes + (int64_t)(n_begin + r0 + i) * p.row_bytes, (uint32_t)p.row_bytes, full(b), pol);
      }
      // every copy lands before this thread (and so the CTA) can finish
      for (int b = 0; b < nrb; b++) wait_drain(full(b), 0);
      wait_drain(coef_full, 0);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int ct = cw * 32 + lane;
  const int nthreads = consumers * 32;
  pdl_wait();                                                    // x is written by the previous kernel
  {
    const int chunks = p.K / 4;
    for (int c = ct; c < chunks; c += nthreads) {
      float t[16];
      build_table(ld_nc_f4(p.x + 4 * c), t);
      float4 *dst = reinterpret_cast<float4 *>(smem + p.off_tab + c * 64);
      dst[0] = make_float4(t[0], t[1], t[2], t[3]);
      dst[1] = make_float4(t[4], t[5], t[6], t[7]);
      dst[2] = make_float4(t[8], t[9], t[10], t[11]);
      dst[3] = make_float4(t[12], t[13], t[14], t[15]);
    }
    // consumer warps only; every consumer thread reaches it (no exit before)
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  }
  const int blk = cw / p.parts, part = cw % p.parts;
  bool ok = true;
  if (blk < nrb) {
    ok = __all_sync(0xffffffffu, wait_bounded(coef_full, 0, ctl)) &&
         __all_sync(0xffffffffu, wait_bounded(full(blk), 0, ctl));
    if (ok) {
      const int r = 32 * blk + lane;
      const bool valid = r < rows;
      const int rr = valid ? r : 32 * blk;                       // a valid row of the block
      const int u0 = part * p.units / p.parts, u1 = (part + 1) * p.units / p.parts;
      const uint8_t *crow = smem + rr * p.row_stride;
      const uint16_t *srow = sc + rr * p.G;
      float acc = 0.0f, gacc = 0.0f;
      for (int u = u0; u < u1; u++) {
        const uint4 cw4 = *reinterpret_cast<const uint4 *>(crow + 16 * u);
        const uint32_t words[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
        const uint32_t tu = (uint32_t)p.off_tab + (uint32_t)u * 32 * 64;   // this unit's 32 tables (64-byte aligned)
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const uint32_t w = words[j];
#pragma unroll
          for (int i = 0; i < 8; i++) {
            // nibble i times 4 (the byte offset of the entry), OR-ed into the
            // 64-byte-aligned table base; the chunk offset is an immediate
            const uint32_t off = (i == 0 ? (w << 2) : (w >> (4 * i - 2))) & 0x3Cu;
            gacc += *reinterpret_cast<const float *>(smem + ((tu | off) + (j * 8 + i) * 64));
          }
          if ((j + 1) % GW == 0) {
            acc = fmaf(h2f(srow[(u * 4 + j) / GW]), gacc, acc);
            gacc = 0.0f;
          }
        }
      }
      if (valid) red[r * p.parts + part] = acc;
    }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(done_bar);
  if (!__all_sync(0xffffffffu, ok)) return;
  if (!__all_sync(0xffffffffu, wait_bounded(done_bar, 0, ctl))) return;
  for (int r = ct; r < rows; r += nthreads) {
    float s = 0.0f;
    for (int q = 0; q < p.parts; q++) s += red[r * p.parts + q];
    p.y[n_begin + r] = s;
  }
}

int sm_count_q1() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

}  // namespace

// Returns cudaErrorNotSupported (nothing launched) when the slab of rows or
// the tables do not fit in shared memory or the coefficient rows are not
// 16-byte multiples; the caller then uses another decode kernel.
cudaError_t launch_gemv_q1(const float *x, const uint32_t *codes, const uint16_t *scales, float *y, int64_t N,
                           int64_t K, int group, cudaStream_t s) {
  if (K % 128 != 0 || group % 32 != 0) return cudaErrorNotSupported;
  Q1Params p{};
  p.x = x;
  p.codes = reinterpret_cast<const uint8_t *>(codes);
  p.scales = scales;
  p.y = y;
  p.N = (int)N;
  p.K = (int)K;
  p.G = (int)(K / group);
  if ((p.G * 2) % 16 != 0) return cudaErrorNotSupported;
  p.group_words = group / 32;
  p.row_bytes = (int)(K / 8);
  p.row_stride = p.row_bytes + 16;
  p.units = (int)(K / 128);
  int grid = sm_count_q1();
  if (N < grid) grid = (int)N;
  const int rows_max = (int)((N + grid - 1) / grid);
  p.row_blocks = (rows_max + 31) / 32;
  if (p.row_blocks > kMaxRowBlocks) return cudaErrorNotSupported;
  int parts = kMaxConsumerWarps / p.row_blocks;
  if (parts > p.units) parts = p.units;
  p.parts = parts < 1 ? 1 : parts;
  const int code_bytes = rows_max * p.row_stride;
  p.off_tab = (code_bytes + 127) & ~127;
  const int tab_bytes = (int)(K / 4) * 64;
  p.off_coef = p.off_tab + tab_bytes;
  const int coef_bytes = rows_max * p.G * 2;
  p.off_red = (p.off_coef + coef_bytes + 15) & ~15;
  const int red_bytes = rows_max * p.parts * 4;
  p.off_bar = (p.off_red + red_bytes + 7) & ~7;
  const size_t smem = (size_t)p.off_bar + 8 * (kMaxRowBlocks + 2) + 16;
  if (smem > (size_t)kSmemBudget) return cudaErrorNotSupported;
  const int threads = 32 * (1 + p.row_blocks * p.parts);

  auto kern = p.group_words == 1 ? gemv_q1_kernel<1> : p.group_words == 2 ? gemv_q1_kernel<2> : gemv_q1_kernel<4>;
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

cudaError_t read_clear_q1_status(int *status, cudaStream_t s) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_q1_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_q1_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace qmm
