// gemm.cu -- the prefill product y[M, N] = x[M, K] * dequant(W)^T on tcgen05.
//
// The "... Tesla C2075 ..." paper (section 3.1 "Prefill projections: dequantize,
// then call the vendor") dequantizes every 8-bit weight into an FP32 scratch
// matrix and then calls the vendor GEMM; the Maxwell Q1 page ("A 27B model on
// two 4GB Maxwell GPUs", section "A packed Q1 prefill kernel with a narrow
// dispatch window") expands Q1 weights to FP32 before SGEMM.  Here the
// dequantization is fused into the tensor-core pipeline instead: codes travel
// from HBM to shared memory by TMA, eight warps turn each 128-row x 64-k code
// tile into bf16 directly in the 128-byte-swizzled K-major layout the tensor
// core reads, and no dequantized weight ever reaches global memory.  The
// kernel is instantiated per code format (INT4 affine, INT8 symmetric, Q1
// signs); only the code tile width and the dequantization differ.
//
// Roles of one persistent CTA per SM (14 warps):
//   warp 0      TMA producer: per K-step, the x tile (bf16, BN tokens x 64 k,
//               128-byte swizzle) and the code tile (128 rows x 32 / 64 / 16
//               bytes for INT4 / INT8 / Q1; a Q1 chunk holds two K-steps)
//   warp 1      TMEM allocation and the single-thread tcgen05.mma issuer
//   warps 2-9   dequantization, two threads per weight row (32 k each): the
//               weight in float32 (INT4 s*q + b with an exact product and one
//               rounding; INT8 s*q and Q1 +-s, exact), then round-to-nearest-
//               even bf16, stored swizzled, proxy-fenced; the row's scales
//               (and biases) come eight groups at a time with 16-byte loads,
//               one chunk ahead (group 64: K-steps eight at a time, unrolled);
//               with wide tiles they also help drain the accumulator
//   warps 10-13 epilogue: tcgen05.ld of the f32 accumulator, y stored with
//               32 consecutive n per warp-wide store
//
// The MMA computes D[128 weight rows, BN tokens] = A * B^T with A = the
// dequantized weight tile and B = the x tile, i.e. the transpose of a y tile;
// putting the weights on the M side lets one dequantized tile serve BN tokens.
// BN (a multiple of 16 up to 256, or for INT4 / INT8 of 32 up to 512) is
// chosen per call (pick_bn).  Up to 256, two accumulators of 256 columns live
// in TMEM so the epilogue of one tile overlaps the main loop of the next;
// wider tiles are two MMAs per k-slice (two x boxes of BN/2 rows) into one
// accumulator of BN columns, which dequantizes each weight tile for more
// tokens: on the M = 1024 shapes one wave of 3 x 48 tiles instead of two
// waves of 6 x 48.  Stage buffers (as many as shared memory holds, up to
// eight) are guarded by mbarriers (TMA -> full, dequant -> afull, MMA commit
// -> empty).
//
// Every wait is bounded by wall time (bounded_wait.cuh).  A wait that runs out
// records QMM_ERR_DEVICE_TIMEOUT in a device status word, raises a CTA-wide
// abort flag that the other roles poll, drains this CTA's outstanding TMA
// copies and MMAs (again with bounded waits), frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "bounded_wait.cuh"
#include "dequant_bf16.cuh"
#include "qmm_device.cuh"
#include "qmm_launch.h"
#include "sm100_ptx.cuh"

namespace qmm {

__device__ int g_gemm_status = 0;   // QMM_OK or QMM_ERR_DEVICE_TIMEOUT (-6)

namespace {

using namespace sm100;

constexpr int BM = 128;                // weight rows per tile (MMA M)
constexpr int BK = 64;                 // k per stage: one 128-byte swizzle atom of bf16
constexpr int BN_MAX = 256;            // tokens per MMA (N), at most
constexpr int BN_WIDE_MAX = 512;       // tokens per tile, as two MMAs of up to 256 into one accumulator
constexpr int MAX_STAGES = 8;           // ring depth: as many stages as shared memory holds
constexpr int SMEM_LIMIT = 227 * 1024;    // dynamic shared memory per CTA
constexpr int UMMA_K = 16;
constexpr int DQ_WARP0 = 2, DQ_WARPS = 8, EPI_WARP0 = DQ_WARP0 + DQ_WARPS;
constexpr int NUM_THREADS = 32 * (EPI_WARP0 + 4);
constexpr int DQ_THREADS = 32 * DQ_WARPS;
static_assert(DQ_THREADS == 2 * BM, "two dequantization threads per weight row, 32 k each");

// Code bytes per weight row loaded per K-step: INT4 32, INT8 64; Q1 16 (the
// 16-byte chunk holding 128 k, loaded for each of its two K-steps, since a
// TMA copy cannot start inside a 16-byte unit).
template <int BITS>
constexpr int code_bytes_per_row() { return BITS == 4 ? 32 : BITS == 8 ? 64 : 16; }

// One ring stage: the dequantized weight tile, the x tile (BN rows of 128
// bytes) and the code tile, each a multiple of 1024 bytes (swizzle atoms).
// The stage size depends on BN, so the ring depth is chosen per call.
template <int BITS>
struct Smem {
  static constexpr int CB = code_bytes_per_row<BITS>();
  static constexpr int A_BYTES = BM * BK * 2;        // 16 KB dequantized weights (bf16)
  static constexpr int C_BYTES = BM * CB;            // codes: 4 KB (INT4), 8 KB (INT8), 2 KB (Q1)
  static constexpr int BARS = 3 * MAX_STAGES + 4 + 1;  // full, afull, empty, acc_full[2], acc_empty[2], drain
  static constexpr int TAIL = BARS * 8 + 16 /* tmem slot + abort flag */ + 1024 /* base alignment slack */;
  static constexpr uint32_t TMEM_COLS = 2 * BN_MAX;  // two accumulators
  static constexpr int stage_bytes(int bn) { return A_BYTES + bn * BK * 2 + C_BYTES; }
  static constexpr int stages(int bn) {
    const int n = (SMEM_LIMIT - TAIL) / stage_bytes(bn);
    return n > MAX_STAGES ? MAX_STAGES : n;
  }
  static constexpr int alloc(int bn) { return stages(bn) * stage_bytes(bn) + TAIL; }
};

// Position in the stage ring: slot and phase parity, advanced without a
// division (the ring depth is a runtime value).
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int stages) {
    if (++s == stages) s = 0, ph ^= 1u;
  }
};

struct GemmParams {
  const uint16_t *scales;
  const uint16_t *biases;
  float *y;
  int M, N, K;
  int gshift;
  int groups_per_row;
  int coef_vec;          // coefficient rows load as 16-byte vectors
  int bn;
  int nsub, bn_sub;      // MMAs per k-slice (1, or 2 for tiles wider than 256) and tokens per MMA
  int stages;            // ring depth
  int m_blocks, n_blocks, tiles;
};

template <int BITS, bool G64, int NSUB>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    qmm_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                    const __grid_constant__ CUtensorMap tmap_codes, const GemmParams p) {
  using S = Smem<BITS>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // align the working area to 1024 bytes (128-byte swizzle atoms)
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int STAGES = p.stages;
  const int stage_bytes = S::stage_bytes(p.bn);
  const int b_off = S::A_BYTES, c_off = S::A_BYTES + p.bn * BK * 2;
  auto a_buf = [&](int s) { return sbase + s * stage_bytes; };
  auto b_buf = [&](int s) { return sbase + s * stage_bytes + b_off; };
  auto c_ptr = [&](int s) { return smem + s * stage_bytes + c_off; };
  auto c_buf = [&](int s) { return sbase + s * stage_bytes + c_off; };
  const int bar_off = STAGES * stage_bytes;
  const uint32_t bars = sbase + bar_off;
  auto full = [&](int s) { return bars + 8 * s; };
  auto afull = [&](int s) { return bars + 8 * (MAX_STAGES + s); };
  auto empty = [&](int s) { return bars + 8 * (2 * MAX_STAGES + s); };
  auto acc_full = [&](int b) { return bars + 8 * (3 * MAX_STAGES + b); };
  auto acc_empty = [&](int b) { return bars + 8 * (3 * MAX_STAGES + 2 + b); };
  const uint32_t drain_bar = bars + 8 * (3 * MAX_STAGES + 4);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + bar_off + S::BARS * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + bar_off + S::BARS * 8 + 4);
  const WaitCtl ctl{abort_flag, &g_gemm_status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ksteps = p.K / BK;
  const int bn = p.bn;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; s++) {
      mbar_init(full(s), 1);
      mbar_init(afull(s), DQ_THREADS);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), NSUB == 1 ? 128 : 128 + DQ_THREADS);   // wide: the dequantization warps help
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), S::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // The y rows of a finished accumulator: this warp's TMEM lane quarter, the
  // 32-column chunks c with c % nroles == role (one role per epilogue warp; a
  // wide tile's single accumulator is shared with the dequantization warps).
  auto store_tile = [&](int tile, int buf, int role, int nroles) {
    const int q = warp & 3;                          // TMEM lane quarter this warp may read
    const int r = q * 32 + lane;                     // weight row within the tile
    const int mb = tile % p.m_blocks, nb = tile / p.m_blocks;
    tc_fence_after();
    const int n = nb * BM + r;
    const int m0 = mb * bn;
    const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + buf * BN_MAX;
#pragma unroll 1
    for (int c0 = 32 * role; c0 < bn; c0 += 32 * nroles) {
      if (c0 + 32 <= bn) {
        uint32_t v[32];
        __syncwarp();                  // tcgen05.ld is .sync.aligned: the whole warp, converged
        tmem_ld_32x32b_x32(tbase + c0, v);
        tmem_ld_wait();
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 32; j++) {
            const int m = m0 + c0 + j;
            if (m < p.M) __stcs(p.y + (int64_t)m * p.N + n, __uint_as_float(v[j]));
          }
        }
      } else {
        uint32_t v[16];
        __syncwarp();
        tmem_ld_32x32b_x16(tbase + c0, v);
        tmem_ld_wait();
        if (n < p.N) {
#pragma unroll
          for (int j = 0; j < 16; j++) {
            const int m = m0 + c0 + j;
            if (m < p.M) __stcs(p.y + (int64_t)m * p.N + n, __uint_as_float(v[j]));
          }
        }
      }
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_x);
      tma_prefetch_desc(&tmap_codes);
      const uint32_t tx = (uint32_t)bn * BK * 2 + S::C_BYTES;
      int it = 0;                   // global K-step counter of this CTA
      Ring ring;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
        const int mb = tile % p.m_blocks, nb = tile / p.m_blocks;
        for (int kb = 0; kb < ksteps; kb++, it++, ring.next(STAGES)) {
          const int s = ring.s;
          const uint32_t ph = ring.ph;
          if (!wait_bounded(empty(s), ph ^ 1, ctl)) { ok = false; break; }
          mbar_arrive_expect_tx(full(s), tx);
#pragma unroll
          for (int h = 0; h < NSUB; h++)     // the x tile in boxes of bn_sub rows
            tma_load_2d(b_buf(s) + h * p.bn_sub * (BK * 2), &tmap_x, kb * BK, mb * bn + h * p.bn_sub, full(s));
          const int cx = BITS == 1 ? (kb >> 1) * S::CB : kb * S::CB;   // byte column of the code chunk
          tma_load_2d(c_buf(s), &tmap_codes, cx, nb * BM, full(s));
        }
      }
      // drain: every copy this thread issued lands before it exits, also when
      // the consumers give up later (after a normal run these waits end at once)
      const int first = it > STAGES ? it - STAGES : 0;
      for (int j = first; j < it; j++) wait_drain(full(j % STAGES), (j / STAGES) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, p.bn_sub);
      constexpr int nbuf = NSUB == 1 ? 2 : 1;   // a tile wider than 256 fills TMEM: one accumulator
      int it = 0, local = 0;
      Ring ring;
      bool ok = true;
      // Readiness of stage `it` tested while the previous stage's MMAs were
      // being issued, so the ~180-cycle latency of the test is hidden; only a
      // stage found not ready takes the blocking (bounded) wait.
      bool ready = false;
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, local++) {
        const int buf = local % nbuf;
        const uint32_t use = (local / nbuf) & 1;
        if (!wait_bounded(acc_empty(buf), use ^ 1, ctl)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN_MAX;
        for (int kb = 0; kb < ksteps; kb++, it++, ring.next(STAGES)) {
          const int s = ring.s;
          const uint32_t ph = ring.ph;
          if (!ready) {
            const bool f = mbar_test(full(s), ph), a = mbar_test(afull(s), ph);
            if (!(f || wait_bounded(full(s), ph, ctl)) || !(a || wait_bounded(afull(s), ph, ctl))) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint64_t ad = smem_desc_sw128(a_buf(s));
          const uint64_t bd = smem_desc_sw128(b_buf(s));
#pragma unroll
          for (int h = 0; h < NSUB; h++) {
            // sub-tile h: tokens h*bn_sub.., rows of 128 bytes (address field in 16-byte units)
            const uint64_t bdh = bd + (uint64_t)(h * p.bn_sub * (BK * 2 / 16));
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; kk++) {
              // +32 bytes per 16 k inside the swizzle atom: +2 in the encoded address
              umma_bf16(d_tmem + h * p.bn_sub, ad + 2 * kk, bdh + 2 * kk, idesc, (kb | kk) != 0);
            }
          }
          umma_commit(empty(s));          // stage free once these MMAs have read it
          // Test the next stage only now: a test (acquire) holds back this
          // thread's later operations until it returns (~250 cycles), which
          // then overlaps the MMAs just issued instead of delaying them.
          Ring nx = ring;
          nx.next(STAGES);
          const int sn = nx.s;
          const uint32_t phn = nx.ph;
          const bool fn = mbar_test(full(sn), phn), an = mbar_test(afull(sn), phn);
          ready = fn && an;
        }
        if (!ok) break;
        umma_commit(acc_full(buf));       // accumulator complete
      }
      if (!ok) {
        umma_commit(drain_bar);           // wait for every MMA issued so far
        wait_drain(drain_bar, 0);
      }
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ dequantization
    const int t = threadIdx.x - DQ_WARP0 * 32;      // 0 .. DQ_THREADS - 1
    const int r = t >> 1, part = t & 1;             // weight row within the tile, k half
    const int G = p.groups_per_row;
    Ring ring;
    int dq_local = 0;         // tiles of this CTA so far
    bool ok = true;
    bool ready = false;       // the current stage seen complete by a test issued one K-step early
    for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
      const int nb = tile / p.m_blocks;
      const int row = nb * BM + r;
      const bool row_ok = row < p.N;
      const uint16_t *srow = p.scales + (int64_t)(row_ok ? row : 0) * G;
      const uint16_t *brow = BITS == 4 ? p.biases + (int64_t)(row_ok ? row : 0) * G : nullptr;
      // coefficients: eight groups per 16-byte load, current and next chunk
      uint4 sc_cur = make_uint4(0, 0, 0, 0), bc_cur = sc_cur, sc_nxt = sc_cur, bc_nxt = sc_cur;
      int cur_chunk = 0;
      if (p.coef_vec && row_ok) {
        sc_cur = ld_stream_u4(srow);
        if (BITS == 4) bc_cur = ld_stream_u4(brow);
        if (G > 8) {
          sc_nxt = ld_stream_u4(srow + 8);
          if (BITS == 4) bc_nxt = ld_stream_u4(brow + 8);
        }
      }
      // G64 (group 64 = one K-step, 16-byte coefficient loads): the K-steps
      // go eight at a time, unrolled, so each step's half of the chunk's
      // 16-byte coefficient vector is picked out at compile time
      constexpr int UN = G64 ? 8 : 1;
      for (int kb0 = 0; kb0 < ksteps && ok; kb0 += UN) {
#pragma unroll
      for (int u = 0; u < UN; u++) {
        const int kb = kb0 + u;
        if (UN > 1 && kb >= ksteps) break;
        const int s = ring.s;
        const uint32_t ph = ring.ph;
        const int g = (kb * BK + 32 * part) >> p.gshift;  // this thread's 32 k lie in one group
        uint16_t sb = 0, bb = 0;
        if (G64) {
          if (row_ok) {
            if (u == 0 && kb0 > 0) {                    // the next chunk of eight groups
              sc_cur = sc_nxt;
              bc_cur = bc_nxt;
              if (kb0 + 8 < G) {
                sc_nxt = ld_stream_u4(srow + kb0 + 8);
                if (BITS == 4) bc_nxt = ld_stream_u4(brow + kb0 + 8);
              }
            }
            sb = half_at(sc_cur, u);
            if (BITS == 4) bb = half_at(bc_cur, u);
          }
        } else if (row_ok) {
          if (p.coef_vec) {
            if ((g >> 3) != cur_chunk) {
              cur_chunk = g >> 3;
              sc_cur = sc_nxt;
              bc_cur = bc_nxt;
              if ((cur_chunk + 1) * 8 < G) {
                sc_nxt = ld_stream_u4(srow + (cur_chunk + 1) * 8);
                if (BITS == 4) bc_nxt = ld_stream_u4(brow + (cur_chunk + 1) * 8);
              }
            }
            sb = half_at(sc_cur, g & 7);
            if (BITS == 4) bb = half_at(bc_cur, g & 7);
          } else {
            sb = ld_nc_u16(srow + g);
            if (BITS == 4) bb = ld_nc_u16(brow + g);
          }
        }
        const float sf = row_ok ? h2f(sb) : 0.0f;
        const float bf = row_ok ? h2f(bb) : 0.0f;
        f2 sp[4], b2, s2;
        uint32_t sbf = 0;
        if constexpr (BITS == 4) {
          scale_pairs(sf, sp);
          b2 = f2_make(bf, bf);
        } else if constexpr (BITS == 8) {
          s2 = f2_make(sf, sf);
        } else {
          sbf = bf16_pair(sf);
        }
        if (!ready && !__all_sync(0xffffffffu, wait_bounded(full(s), ph, ctl))) { ok = false; break; }
        // this thread's 32 k of row r (k = 32 * part ..)
        uint32_t words[8];
        if constexpr (BITS == 4) {
          const uint4 cw = *reinterpret_cast<const uint4 *>(c_ptr(s) + r * 32 + part * 16);
          words[0] = cw.x, words[1] = cw.y, words[2] = cw.z, words[3] = cw.w;
        } else if constexpr (BITS == 8) {
          const uint4 c0 = *reinterpret_cast<const uint4 *>(c_ptr(s) + r * 64 + part * 32);
          const uint4 c1 = *reinterpret_cast<const uint4 *>(c_ptr(s) + r * 64 + part * 32 + 16);
          words[0] = c0.x, words[1] = c0.y, words[2] = c0.z, words[3] = c0.w;
          words[4] = c1.x, words[5] = c1.y, words[6] = c1.z, words[7] = c1.w;
        } else {
          words[0] = *reinterpret_cast<const uint32_t *>(c_ptr(s) + r * 16 + (kb & 1) * 8 + part * 4);
        }
        // the next stage's readiness, tested early: its result is read after
        // this stage's stores (measured faster than testing after them)
        Ring nx = ring;
        nx.next(STAGES);
        const bool next_ready = mbar_test(full(nx.s), nx.ph);
        const uint32_t arow = a_buf(s) + r * 128;
#pragma unroll
        for (int i = 0; i < 4; i++) {
          const int c = 4 * part + i;                                      // 16-byte chunk: k = 8c..8c+7
          uint4 v;
          if constexpr (BITS == 4) v = dequant_word_bf16(words[i], sp, b2);
          else if constexpr (BITS == 8) v = dequant_int8x8_bf16(words[2 * i], words[2 * i + 1], s2);
          else v = signs8_bf16(words[0] >> (8 * i), sbf);
          const uint32_t dst = arow + ((c ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                       "r"(v.w)
                       : "memory");
        }
        fence_proxy_async_smem();
        mbar_arrive(afull(s));
        ready = __all_sync(0xffffffffu, next_ready);
        ring.next(STAGES);
      }
      }
      if constexpr (NSUB == 2) {
        // a wide tile's accumulator is the only one: help drain it
        if (!ok) break;
        if (!__all_sync(0xffffffffu, wait_bounded(acc_full(0), dq_local & 1, ctl))) { ok = false; break; }
        store_tile(tile, 0, 1 + (warp - DQ_WARP0) / 4, 3);
        tc_fence_before();
        mbar_arrive(acc_empty(0));
      }
      dq_local++;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    int local = 0;
    bool ok = true;
    constexpr int nbuf = NSUB == 1 ? 2 : 1;
    for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, local++) {
      const int buf = local % nbuf;
      const uint32_t use = (local / nbuf) & 1;
      if (!__all_sync(0xffffffffu, wait_bounded(acc_full(buf), use, ctl))) { ok = false; break; }
      store_tile(tile, buf, 0, NSUB == 1 ? 1 : 3);
      tc_fence_before();
      mbar_arrive(acc_empty(buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

int sm_count_gemm() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

// Token-tile width: a multiple of 16 up to 256, or of 32 up to 512 (two MMAs
// per k-slice, where allowed and a ring of three stages still fits), that
// minimizes waves * (C0 + BN): a wave is one tile per SM,
// and a tile's time was measured to grow only slowly with BN (one wave of
// INT4 tiles: 20.0 us at BN = 64, 24.3 us at 256), the per-K-step
// dequantization of the 128-row weight tile being the fixed part C0 (in
// token units).  Ties go to the wider tile.
int pick_bn(int64_t M, int64_t N, int sms, int code_tile_bytes, bool allow_wide) {
  const int64_t nblk = (N + BM - 1) / BM;
  const int64_t c0 = 850;
  int best = 16;
  int64_t best_cost = -1;
  for (int bn = 16; bn <= BN_WIDE_MAX; bn += bn < BN_MAX ? 16 : 32) {
    // a wide tile only with a ring of at least three stages (measured: two are too shallow)
    const int stage = BM * BK * 2 + bn * BK * 2 + code_tile_bytes;
    if (bn > BN_MAX && (!allow_wide || (SMEM_LIMIT - 2048) / stage < 3)) break;
    // the last token tile of a wide width must reach into its second x box
    if (bn > BN_MAX && M - ((M + bn - 1) / bn - 1) * bn <= bn / 2) continue;
    const int64_t tiles = ((M + bn - 1) / bn) * nblk;
    const int64_t waves = (tiles + sms - 1) / sms;
    const int64_t cost = waves * (c0 + bn);
    if (best_cost < 0 || cost <= best_cost) {
      best_cost = cost;
      best = bn;
    }
    if (bn >= M) break;            // wider tiles only add padding
  }
  return best;
}

}  // namespace

namespace {

template <int BITS>
cudaError_t launch_bits(const uint16_t *x_bf16, const uint32_t *codes, const GemmParams &p, int64_t M, int64_t N,
                        int64_t K, cudaStream_t s) {
  using S = Smem<BITS>;
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tx, tc;
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {BK, (cuuint32_t)p.bn_sub};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x_bf16), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // codes as bytes: [N, K*BITS/8], box of CB bytes x 128 rows
    cuuint64_t dims[2] = {(cuuint64_t)(K * BITS / 8), (cuuint64_t)N};
    cuuint64_t strides[1] = {(cuuint64_t)(K * BITS / 8)};
    cuuint32_t box[2] = {(cuuint32_t)S::CB, BM};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t *>(codes), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  GemmParams pp = p;
  pp.stages = S::stages(p.bn);
  if (pp.stages < 2) return cudaErrorNotSupported;
  const int alloc = S::alloc(p.bn);
  const bool g64 = p.gshift == 6 && p.coef_vec;
  auto kern = p.nsub == 2 ? (g64 ? qmm_gemm_kernel<BITS, true, 2> : qmm_gemm_kernel<BITS, false, 2>)
                          : (g64 ? qmm_gemm_kernel<BITS, true, 1> : qmm_gemm_kernel<BITS, false, 1>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, alloc);
  if (e != cudaSuccess) return e;
  const int grid = p.tiles < sm_count_gemm() ? p.tiles : sm_count_gemm();
  kern<<<grid, NUM_THREADS, alloc, s>>>(tx, tc, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const uint16_t *x_bf16, const uint32_t *codes, const uint16_t *scales,
                        const uint16_t *biases, float *y, int64_t M, int64_t N, int64_t K, int bits, int group,
                        cudaStream_t s) {
  GemmParams p{};
  p.scales = scales;
  p.biases = biases;
  p.y = y;
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.gshift = __builtin_ctz((unsigned)group);
  p.groups_per_row = (int)(K / group);
  p.coef_vec = (p.groups_per_row % 8 == 0) ? 1 : 0;   // rows are then 16-byte multiples (bases are 16-aligned)
  // (Q1, whose per-K-step dequantization is the lightest, measured slower with wide tiles)
  p.bn = pick_bn(M, N, sm_count_gemm(), BM * (bits == 4 ? 32 : bits == 8 ? 64 : 16), bits != 1);
  p.nsub = p.bn > BN_MAX ? 2 : 1;
  p.bn_sub = p.bn / p.nsub;
  p.m_blocks = (int)((M + p.bn - 1) / p.bn);
  p.n_blocks = (int)((N + BM - 1) / BM);
  p.tiles = p.m_blocks * p.n_blocks;
  if (bits == 4) return launch_bits<4>(x_bf16, codes, p, M, N, K, s);
  if (bits == 8) return launch_bits<8>(x_bf16, codes, p, M, N, K, s);
  if (bits == 1) return launch_bits<1>(x_bf16, codes, p, M, N, K, s);
  return cudaErrorNotSupported;
}

cudaError_t read_clear_gemm_status(int *status, cudaStream_t s) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_gemm_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_gemm_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
  }
  *status = v;
  return cudaSuccess;
}

}  // namespace qmm
