// gemv_q1.cu -- binary (Q1) decode product y[1, N] = x[1, K] * dequant(W)^T
// through per-chunk lookup tables.
//
// A Q1 weight is s * (+1 or -1), so a row's product over four consecutive k
// only ever takes one of 16 values: the signed sums +-x0 +-x1 +-x2 +-x3.
// Those 16 sums depend on x alone, so each CTA builds them for the 4-k chunks
// of x and every 4 weights of every row then cost one table lookup and one
// add, instead of a sign flip and an add per weight.  This is the
// lookup-table idea that the Maxwell Q1 page ("A 27B model on two 4GB Maxwell
// GPUs: inference tuning", section "A packed Q1 prefill kernel with a narrow
// dispatch window") points to for binary weights.
//
// Layout.  Each CTA owns a contiguous slab of rows (whole 8-row blocks).
// Before the programmatic-dependent-launch wait, one producer thread copies
// the slab's codes as TMA tensor boxes of eight rows (128-byte columns with
// the 128-byte swizzle, so the 32 rows one warp instruction reads fall in
// distinct bank groups) and its fp16 scales with one bulk copy.  The tables
// are built a phase at a time, for eight 128-k units (1024 k, 16 KB of
// tables), so that the shared memory of a CTA stays under half an SM's and
// the next product's CTA can copy its codes while this one computes.  Sixteen
// consumer warps: four per 32-row block, each taking two of the phase's
// units, lane i walking row 32 * block + i.  All 32 lanes of a lookup read the
// same 64-byte table: one shared-memory wavefront (equal nibbles broadcast,
// distinct nibbles hit distinct banks).  Per group the lookups are summed in
// k order and scaled by the group's scale; a row's four parts are added in
// part order at the end: no atomics, the same bits on every run.
//
// Every mbarrier wait is bounded (bounded_wait.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "bounded_wait.cuh"
#include "qmm_device.cuh"
#include "qmm_launch.h"
#include "sm100_ptx.cuh"

namespace qmm {

__device__ int g_q1_status = 0;

namespace {

using namespace sm100;

constexpr int kConsumerWarps = 16;
constexpr int kThreads = 32 * (kConsumerWarps + 1);   // a producer warp and the consumers
constexpr int kParts = 4;                             // consumer warps per 32-row block
constexpr int kUnitsPerPart = 2;                      // 128-k units per part and phase
constexpr int kPhaseUnits = kParts * kUnitsPerPart;   // units of one phase's tables
constexpr int kPhaseChunks = kPhaseUnits * 32;        // 4-k chunks (tables) per phase
constexpr int kSmemMax = 225 * 1024;

struct Q1Params {
  const float *x;
  const uint16_t *scales;
  float *y;
  int N, K, G;            // G = groups per row
  int units;              // 128-k units per row
  int phases;             // ceil(units / kPhaseUnits)
  int noct;               // 8-row blocks of the N rows (split evenly over the CTAs)
  int row_bytes;
  int off_tab, off_coef, off_red, off_bar;
};

// The signed sums of x[4c .. 4c+3] with entry i = a[i & 3] + b[i >> 2]
// (bit j of i set: +x_j, clear: -x_j), entries 8h .. 8h + 7 of the 16.
__device__ __forceinline__ void build_half(const float4 v, int h, float (&t)[8]) {
  const float a[4] = {-v.x - v.y, v.x - v.y, -v.x + v.y, v.x + v.y};
  const float b0 = h ? (-v.z + v.w) : (-v.z - v.w);
  const float b1 = h ? (v.z + v.w) : (v.z - v.w);
#pragma unroll
  for (int i = 0; i < 4; i++) {
    t[i] = a[i] + b0;
    t[4 + i] = a[i] + b1;
  }
}

// GW: 32-bit code words per group (group / 32).
template <int GW>
__global__ void __launch_bounds__(kThreads, 2) gemv_q1_kernel(const __grid_constant__ CUtensorMap tm_codes,
                                                                const Q1Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // the swizzled code columns need a 1024-byte-aligned base (the launch adds 1 KB)
  const uint32_t sraw = smem_addr(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (sraw & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const uint16_t *sc = reinterpret_cast<const uint16_t *>(smem + p.off_coef);
  float *red = reinterpret_cast<float *>(smem + p.off_red);
  const uint32_t codes_full = sbase + p.off_bar, coef_full = codes_full + 8;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.off_bar + 16);
  const WaitCtl ctl{abort_flag, &g_q1_status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o0 = (int)((int64_t)blockIdx.x * p.noct / gridDim.x);
  const int o1 = (int)((int64_t)(blockIdx.x + 1) * p.noct / gridDim.x);
  const int n_begin = 8 * o0;
  const int rows = min(8 * (o1 - o0), p.N - n_begin);
  const int row_bytes = p.row_bytes, G = p.G;

  if (threadIdx.x == 0) {
    mbar_init(codes_full, 1);
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
      const int nbox = (rows + 7) >> 3;
      mbar_arrive_expect_tx(codes_full, (uint32_t)(nbox * 8 * row_bytes));
      for (int i = 0; i < nbox; i++)
        tma_load_3d_hint(sbase + (uint32_t)(i * 8 * row_bytes), &tm_codes, 0, n_begin + 8 * i, 0, codes_full, pol);
      const uint32_t cbytes = (uint32_t)rows * G * 2;
      mbar_arrive_expect_tx(coef_full, cbytes);
      bulk_load(sbase + p.off_coef, p.scales + (int64_t)n_begin * G, cbytes, coef_full, pol);
      // every copy lands before this thread (and so the CTA) can finish
      wait_drain(codes_full, 0);
      wait_drain(coef_full, 0);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int ct = cw * 32 + lane;
  constexpr int nthreads = kConsumerWarps * 32;
  const int blk = cw / kParts, part = cw % kParts;
  const int r = 32 * blk + lane;
  const bool valid = r < rows;
  const int rr = valid ? r : 0;
  // the slab was requested at the start: wait for it before the dependent-launch wait
  bool ok = __all_sync(0xffffffffu, wait_bounded(codes_full, 0, ctl)) &&
            __all_sync(0xffffffffu, wait_bounded(coef_full, 0, ctl));
  pdl_wait();                                                    // x is written by the previous kernel

  // this thread's table half: chunk ct / 2 of each phase, entries 8 (ct & 1) ..
  const int nchunks = p.K >> 2;
  const int hsel = ct & 1;
  auto load_x = [&](int ph) {
    const int c = ph * kPhaseChunks + (ct >> 1);
    return c < nchunks ? ld_nc_f4(p.x + 4 * c) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  };
  float4 xnext = load_x(0);
  // row r's code line in box r / 8, and its swizzle
  const int rbase = (rr >> 3) * 8 * row_bytes + (rr & 7) * 128, rsw = rr & 7;
  const uint16_t *srow = sc + rr * G;
  float acc = 0.0f;
  for (int ph = 0; ph < p.phases; ph++) {
    const float4 xv = xnext;
    if (ph + 1 < p.phases) xnext = load_x(ph + 1);
    {
      float t[8];
      build_half(xv, hsel, t);
      float4 *dst = reinterpret_cast<float4 *>(smem + p.off_tab + (ct >> 1) * 64 + hsel * 32);
      dst[0] = make_float4(t[0], t[1], t[2], t[3]);
      dst[1] = make_float4(t[4], t[5], t[6], t[7]);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");       // the phase's tables are complete
    if (ok && valid) {
#pragma unroll
      for (int uu = 0; uu < kUnitsPerPart; uu++) {
        const int ul = part * kUnitsPerPart + uu;                  // unit within the phase
        const int u = ph * kPhaseUnits + ul;
        if (u < p.units) {
          // 16 code bytes of unit u: 128-byte column u / 8, 16-byte piece u % 8
          const uint4 cw4 = *reinterpret_cast<const uint4 *>(smem + rbase + (u >> 3) * 1024 +
                                                              ((((u & 7) ^ rsw)) << 4));
          const uint32_t words[4] = {cw4.x, cw4.y, cw4.z, cw4.w};
          const uint32_t tu = (uint32_t)p.off_tab + (uint32_t)ul * 32 * 64;   // the unit's 32 tables (2 KB aligned)
          float gacc = 0.0f;
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
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");       // before the next phase's tables
  }
  if (valid) red[r * kParts + part] = acc;
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  if (!ok || *abort_flag) return;
  for (int q = ct; q < rows; q += nthreads) {
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kParts; k++) s += red[q * kParts + k];
    p.y[n_begin + q] = s;
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

PFN_cuTensorMapEncodeTiled_v12000 q1_encode() {
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

}  // namespace

// Returns cudaErrorNotSupported (nothing launched) when K is not a whole
// number of 1024-k code columns, the coefficient rows are not 16-byte
// multiples or the slab does not fit in shared memory; the caller then uses
// another decode kernel.
cudaError_t launch_gemv_q1(const float *x, const uint32_t *codes, const uint16_t *scales, float *y, int64_t N,
                           int64_t K, int group, cudaStream_t s) {
  if (K % 1024 != 0 || group % 32 != 0 || group > 128 || K > 256 * 1024) return cudaErrorNotSupported;
  Q1Params p{};
  p.x = x;
  p.scales = scales;
  p.y = y;
  p.N = (int)N;
  p.K = (int)K;
  p.G = (int)(K / group);
  if ((p.G * 2) % 16 != 0) return cudaErrorNotSupported;
  p.row_bytes = (int)(K / 8);
  p.units = (int)(K / 128);
  p.phases = (p.units + kPhaseUnits - 1) / kPhaseUnits;
  p.noct = (int)((N + 7) / 8);
  const int sms = sm_count_q1();
  const int grid = p.noct < sms ? p.noct : sms;
  const int R = 8 * ((p.noct + grid - 1) / grid);
  if (R > 4 * 32) return cudaErrorNotSupported;            // four 32-row blocks of consumer warps
  size_t off = (size_t)R * p.row_bytes;                    // codes: boxes of 8 rows, 1024-byte multiples
  p.off_tab = (int)off;
  off += (size_t)kPhaseChunks * 64;
  p.off_coef = (int)off;
  off += ((size_t)R * p.G * 2 + 15) & ~(size_t)15;
  p.off_red = (int)off;
  off += (size_t)R * kParts * 4;
  p.off_bar = (int)((off + 15) & ~(size_t)15);
  const size_t smem = (size_t)p.off_bar + 32 + 1024;       // room to align the base to 1024 bytes
  if (smem > (size_t)kSmemMax) return cudaErrorNotSupported;

  PFN_cuTensorMapEncodeTiled_v12000 enc = q1_encode();
  if (!enc) return cudaErrorNotSupported;
  CUtensorMap tm;
  const cuuint32_t es[3] = {1, 1, 1};
  cuuint64_t dims[3] = {32, (cuuint64_t)N, (cuuint64_t)(K / 1024)};
  cuuint64_t strides[2] = {(cuuint64_t)p.row_bytes, 128};
  cuuint32_t box[3] = {32, 8, (cuuint32_t)(K / 1024)};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t *>(codes), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorNotSupported;

  const int gw = group / 32;
  auto kern = gw == 1 ? gemv_q1_kernel<1> : gw == 2 ? gemv_q1_kernel<2> : gemv_q1_kernel<4>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm, p);
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
