/*
 * qmm.h -- C ABI of libqmm.so: weight-only quantized matrix products on GB300.
 *
 *   y = x * dequant(W)^T
 *
 * over weights W[N, K] stored as packed low-bit codes with one coefficient
 * set per group of `group` consecutive elements along K:
 *
 *   bits = 4  affine:     w = s * q + b,   q in 0..15
 *             (group-64 affine INT4 codes with 16-bit scale and bias:
 *              "Pushing the limits of legacy hardware", section "Start with the
 *              machine that actually exists"; the formula  q * scale + min  is on
 *              "I Built an LLM Inference Engine on a 15 year old GPU ...",
 *              section "Quantization: The Model Doesn't Run on INT4")
 *   bits = 8  symmetric:  w = s * q,       q a two's-complement int8
 *             (8-bit group-wise symmetric weights, one scale per group of 64:
 *              "... Tesla C2075 ..." paper, section 2.3 "Quantization and residency")
 *   bits = 1  sign:       w = s * (2b - 1), bit b = 1 means +1, b = 0 means -1
 *             (binary Q1 weights with FP16 scales: "A 27B model on two 4GB
 *              Maxwell GPUs: inference tuning", section "Why this machine is awkward")
 *
 * Layouts (all row-major, all sizes in elements unless stated):
 *   x       [M, K]  float32 (qmm_gemv) or bfloat16 bit patterns (qmm_gemm)
 *   codes   [N, K*bits/32] 32-bit words.  Element k of row n sits in word
 *           k / (32/bits) of that row at bit offset bits * (k mod (32/bits)):
 *           the lowest nibble / byte / bit holds the lowest k.
 *   scales  [N, K/group] IEEE binary16 bit patterns
 *   biases  [N, K/group] IEEE binary16 bit patterns (bits == 4 only, else NULL)
 *   y       [M, N]  float32, y[m, n] = sum_k x[m, k] * w[n, k]
 *
 * Memory and ownership.  Every array argument is device memory owned by the
 * caller (for instance a torch tensor's storage); the library never keeps a
 * pointer past the call, and never allocates or frees device memory in any
 * call (the residency rule of the "15 year old GPU" page, section "Cost 2:
 * memory is allocated and freed on every layer").  Device pointers must be
 * 16-byte aligned, except the idx and val outputs of the argmax heads, which
 * need only their element's 4-byte alignment (so a decode loop can write the
 * token straight into tokens[t]).
 *
 * Asynchrony.  Every call validates its arguments on the host and then only
 * enqueues kernels on `stream` (a cudaStream_t; NULL is the legacy default
 * stream) and returns; results are valid once the stream has reached that
 * point.  On any validation failure nothing is enqueued and no output is
 * touched ("fail before changing live state": "Pushing the limits of legacy
 * hardware", section "Build the execution path, then share the weights").
 *
 * Errors.  Each call returns a qmm_status.  Launch failures are QMM_ERR_CUDA.
 * Every wait inside a kernel is bounded; if one runs out the kernel records
 * a device status word, waits (bounded) for its own copies in flight, and
 * exits without writing its output, and qmm_check() reports
 * QMM_ERR_DEVICE_TIMEOUT.  No exception crosses this interface.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qmm_stream_t;   /* the same type as cudaStream_t */

typedef enum {
    QMM_OK = 0,
    QMM_ERR_ARG = -1,             /* NULL pointer, or a biases pointer that contradicts bits */
    QMM_ERR_SHAPE = -2,           /* negative size, K % 32, K % group, M outside the entry's range */
    QMM_ERR_ALIGN = -3,           /* a device pointer not 16-byte aligned (idx, val: 4-byte) */
    QMM_ERR_UNSUPPORTED = -4,     /* bits / group combination this entry does not implement */
    QMM_ERR_CUDA = -5,            /* a CUDA runtime call or launch failed */
    QMM_ERR_DEVICE_TIMEOUT = -6   /* a bounded device-side wait ran out (see qmm_check) */
} qmm_status;

/*
 * qmm_pack -- codes one-per-byte -> packed 32-bit words.
 *   codes  [N, K] uint8: 0..15 (bits 4), the int8 bit pattern (bits 8), 0/1 (bits 1).
 *          Bits above the format's width are ignored (masked off).
 *   packed [N, K*bits/32] uint32, written.
 *   Requires N >= 0, K >= 0, K % 32 == 0, bits in {1, 4, 8}.
 * Layout: "bits" above.  The pages fix no bit order; this one puts the lowest
 * k in the lowest bits, as the 4-bit, group-64 shift-and-mask decoder of
 * "Pushing the limits of legacy hardware" (section "Half a billion values, and
 * one negative zero") reads codes by shifts and masks.
 */
int qmm_pack(const uint8_t *codes, uint32_t *packed, int64_t N, int64_t K, int bits,
             qmm_stream_t stream);

/*
 * qmm_unpack -- the inverse of qmm_pack: packed words -> one code per byte
 * (int8 bit patterns for bits 8, 0/1 for bits 1).  Same requirements.
 */
int qmm_unpack(const uint32_t *packed, uint8_t *codes, int64_t N, int64_t K, int bits,
               qmm_stream_t stream);

/*
 * qmm_dequant -- dense float32 weights w[N, K] from packed codes.
 *   w[n, k] = s*q + b (bits 4), s*q (bits 8), s*(2b-1) (bits 1), evaluated in
 *   float32 with round-to-nearest; s*q is exact in float32, so w is the
 *   correctly rounded value of the exact weight.  Signed zeros and binary16
 *   subnormal coefficients are kept (no flush to zero), as the exact-decoder
 *   work of "Pushing the limits of legacy hardware", section "Half a billion
 *   values, and one negative zero", requires.
 *   Requires K % 32 == 0, group > 0, K % group == 0; biases non-NULL iff bits == 4.
 */
int qmm_dequant(const uint32_t *packed, const uint16_t *scales, const uint16_t *biases,
                float *w, int64_t N, int64_t K, int bits, int group, qmm_stream_t stream);

/*
 * qmm_gemv -- decode product y[M, N] = x[M, K] * dequant(W)^T, 1 <= M <= 8.
 *   float32 activations, float32 accumulation; bandwidth-bound: every code
 *   is read once from HBM ("... Tesla C2075 ..." paper, section 3.3 "Decode,
 *   and why 4-bit is slower": decode is a bandwidth-bound matrix-vector
 *   product reading each weight once).  The reduction order is fixed, so the
 *   result is the same on every run.  NaN or Inf in x propagate.
 *   Supported: bits 4 and 8 with group in {32, 64, 128}; bits 1 with group in
 *   {32, 64, 128} and K % 128 == 0.  K == 0 writes y = 0.
 *   M == 0 or N == 0 is a no-op.
 *   Weight reads start early.  The decode kernels are launched as dependents
 *   of the kernel before them on the stream (programmatic dependent launch):
 *   they start copying codes, scales and biases while that kernel may still
 *   run, and wait for it only before reading x.  A run of decode calls
 *   (qmm_gemv, qmm_gemv_argmax, qmm_gemv_argmax_noalloc) back to back on one
 *   stream can therefore overlap.  So the weights of a decode call must not
 *   be written by the operation right before it on the stream, nor be the y
 *   or argmax outputs of an earlier call of the same run.  Weights written on
 *   the stream (qmm_pack, qmm_quantize, a copy) are safe once one operation
 *   that is not a decode call (any other kernel or copy) or a host
 *   synchronization lies between the write and the decode call.  x and y
 *   follow plain stream order.
 */
int qmm_gemv(const float *x, const uint32_t *codes, const uint16_t *scales,
             const uint16_t *biases, float *y, int64_t M, int64_t N, int64_t K, int bits,
             int group, qmm_stream_t stream);

/*
 * qmm_gemm -- prefill product y[M, N] = x[M, K] * dequant(W)^T for any M >= 1.
 *   x holds bfloat16 bit patterns.  Each weight is dequantized in float32,
 *   rounded to bfloat16 (nearest even) in shared memory, and multiplied on
 *   the tensor cores with float32 accumulation: the fused replacement of
 *   "dequantize each weight once into an FP32 scratch buffer, then call the
 *   vendor GEMM" ("... Tesla C2075 ..." paper, section 3.1 "Prefill
 *   projections: dequantize, then call the vendor"), and of the Q1 page's
 *   expand-to-FP32 prefill ("A 27B model on two 4GB Maxwell GPUs", section "A
 *   packed Q1 prefill kernel with a narrow dispatch window").
 *   Supported: bits 4, 8 and 1, group in {32, 64, 128}, K % 64 == 0 (K % 128 == 0
 *   for bits 1), K >= 64.  M == 0 or N == 0 is a no-op.
 */
int qmm_gemm(const uint16_t *x_bf16, const uint32_t *codes, const uint16_t *scales,
             const uint16_t *biases, float *y, int64_t M, int64_t N, int64_t K, int bits,
             int group, qmm_stream_t stream);

/*
 * qmm_gemv_argmax -- greedy decode head: idx[m] = argmax_n y[m, n] of the
 *   decode product y = x * dequant(W)^T (qmm_gemv's arithmetic and shape
 *   rules, 1 <= M <= 8), and val[m] = y[m, idx[m]] if val is not NULL.  The
 *   fused greedy head of "Pushing the limits of legacy hardware", section
 *   "Build the execution path, then share the weights": each tile keeps its
 *   maximum with the original index and the tiles are reduced to one winner,
 *   so the logits need not be written (at M == 1 the product's epilogue does
 *   this and no logit is stored; otherwise the logits go to the workspace and
 *   a reduction kernel follows).  Order: a NaN logit ranks first, then the
 *   larger value, equal values to the lower index; the result is the same on
 *   every run.
 *   workspace: device memory of at least qmm_gemv_argmax_workspace_size(M, N)
 *   bytes, 16-byte aligned, owned by the caller, whose first 16 bytes are zero
 *   before the first call (for instance from cudaMemset); every call leaves
 *   them zero again.  Two calls in flight at the same time must not share a
 *   workspace.  idx: int32 [M]; val: float32 [M] or NULL (both 4-byte
 *   aligned; QMM_ERR_ALIGN otherwise).
 */
size_t qmm_gemv_argmax_workspace_size(int64_t M, int64_t N);
int qmm_gemv_argmax(const float *x, const uint32_t *codes, const uint16_t *scales,
                    const uint16_t *biases, int32_t *idx, float *val, int64_t M, int64_t N, int64_t K,
                    int bits, int group, void *workspace, size_t workspace_bytes, qmm_stream_t stream);

/*
 * qmm_gemv_argmax_noalloc -- qmm_gemv_argmax for M == 1 without a work area:
 *   the same fused kernel and the same result (idx[0], and val[0] if val is
 *   not NULL), with the CTA counter and per-CTA winners kept in a fixed
 *   static device array of this library (8208 bytes: a 16-byte counter slot
 *   and the winners of at most 1024 CTAs) instead of caller memory.  The pages
 *   have no counterpart of this entry point: it exists for callers that cannot
 *   allocate device memory at the call (a decode loop that must stay out of
 *   the allocator between tokens, or a C host without an allocator).
 *   Rules: the array's counter is zero when the library loads and every call
 *   leaves it zero; the first call on each device looks the array's address
 *   up (cudaGetSymbolAddress) and caches it with the current context, so make
 *   the first call in each context before any stream capture begins; a call
 *   in another context than the cached one (after cudaDeviceReset, or after
 *   the primary context was released and created again) looks the address up
 *   anew; all calls on a device share the array, so no
 *   two calls may be in flight at once (calls in order on one stream are
 *   fine).  Shapes that the fused M == 1 kernel does not take, or that would
 *   need more than 1024 CTAs, return QMM_ERR_UNSUPPORTED.  Other argument
 *   rules as qmm_gemv_argmax.
 */
int qmm_gemv_argmax_noalloc(const float *x, const uint32_t *codes, const uint16_t *scales,
                            const uint16_t *biases, int32_t *idx, float *val, int64_t N, int64_t K,
                            int bits, int group, qmm_stream_t stream);

/*
 * qmm_quantize -- INT4 affine quantization of float32 weights w[N, K] into the
 *   stored format (packed codes, binary16 scales and biases per group), after
 *   the quantization section of "I Built an LLM Inference Engine on a 15 year
 *   old GPU and the Math was the Easy Part" ("Quantization: The Model Doesn't
 *   Run on INT4": a block's min and max define the range, scale =
 *   (max - min) / 15, q = round((w - min) / scale), dequantized = q * scale + min).
 *   Per group, in float32: lo / hi = min / max of the group (NaN values
 *   skipped, -0 ordered below +0), scale = binary16(RNE((hi - lo) / 15)),
 *   bias = binary16(RNE(lo)), and q = clamp(round((w - bias) / scale), 0, 15)
 *   with the stored coefficients, halves away from zero; q = 0 for a NaN
 *   weight or when the stored scale is not positive and finite.  A NaN scale or
 *   bias is stored as 0x7E00.  The result is the same on every run.
 *   Layout: w [N, K] float32; packed, scales, biases as for the products.
 *   Requires K % 32 == 0, group in {32, 64, 128}, K % group == 0.
 */
int qmm_quantize(const float *w, uint32_t *packed, uint16_t *scales, uint16_t *biases, int64_t N,
                 int64_t K, int group, qmm_stream_t stream);

/*
 * qmm_gather_dequant -- out[t, :] = dequant(W[ids[t], :]) for t < T: rows of a
 *   quantized table selected by token ids and decoded exactly (the embedding
 *   lookup of a tied INT4 table, "Pushing the limits of legacy hardware",
 *   section "Half a billion values, and one negative zero").  Each element is
 *   computed as in qmm_dequant, so signed zeros and subnormal coefficients are
 *   kept.  ids are int32 in device memory; an id outside [0, N) is not read
 *   through and yields a row of quiet NaNs.
 *   Layout: ids [T] int32, out [T, K] float32; packed, scales, biases as above.
 *   Requires K % 32 == 0, K % group == 0; biases non-NULL iff bits == 4.
 *   T == 0 is a no-op.
 */
int qmm_gather_dequant(const int32_t *ids, int64_t T, const uint32_t *packed, const uint16_t *scales,
                       const uint16_t *biases, float *out, int64_t N, int64_t K, int bits, int group,
                       qmm_stream_t stream);

/*
 * qmm_check -- synchronize `stream`, then report QMM_ERR_CUDA if a kernel
 * failed, QMM_ERR_DEVICE_TIMEOUT if a bounded wait in any kernel ran out
 * since the last qmm_check (and clear that record), else QMM_OK.
 */
int qmm_check(qmm_stream_t stream);

/*
 * qmm_test_timeout_next_decode -- test hook for the failure path above.  The
 *   next decode launch that runs on the tensor-core decode kernel (qmm_gemv
 *   or the argmax heads: INT4 products of more than 2^21 weights or of two
 *   or more tokens, INT8 with 3 to 8 tokens, Q1 with 2 to 8 tokens) has its first
 *   consumer warp wait on a barrier that is never completed, with a limit of
 *   limit_ns instead of the normal 2 s.  That wait runs out: the launch
 *   writes no output (an argmax head writes idx = 2147483647 and val =
 *   -inf, no valid winner, and leaves its workspace ready), waits for its
 *   copies in flight, and the next qmm_check() returns QMM_ERR_DEVICE_TIMEOUT;
 *   the call after it runs normally.  One-shot: the launch that takes the
 *   hook clears it.  limit_ns must be in [1000, 100000000] (QMM_ERR_ARG
 *   otherwise).  Not for production use: it exists so that the timeout path
 *   can be exercised without faulting or hanging a GPU.
 */
int qmm_test_timeout_next_decode(int64_t limit_ns);

/* A static, human-readable name for a qmm_status value. */
const char *qmm_status_string(int status);

/* The ABI version: bumps on any incompatible change of the declarations above. */
int qmm_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* QMM_H */
