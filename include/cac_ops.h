/*
 * cac_ops.h — op-level entry points of the GB300 cache-aware Conformer
 * library, for kernel-level parity tests and microbenchmarks.  Same
 * conventions as cac.h (status codes, device pointers owned by the caller,
 * asynchronous on `stream`).
 */
#ifndef CAC_OPS_H_
#define CAC_OPS_H_

#include "cac.h"

#ifdef __cplusplus
extern "C" {
#endif

/* C[M][N] = A[M][K] * B[N][K]^T (+ bias[N]) on the tcgen05/TMEM tensor-core
 * GEMM that every projection of the encoder step uses (feed-forward, Q/K/V,
 * out-projection, pointwise convolutions, joint projection: "True streaming
 * encode", §Per-chunk flow step 3).  A and B bf16, row-major (K contiguous);
 * C fp32 row-major; bias fp32 or NULL.  K % 64 == 0, N % 64 == 0, M >= 1;
 * 16-byte aligned pointers.  splits: 1..4 K-splits per output tile (reduced
 * in a thread-block cluster), 0 = the library's choice.
 * a_split != 0: A is a split operand [M][2K] — row r holds hi[r][0..K) then
 * lo[r][0..K), two bf16 terms of one higher-precision activation — and the
 * product is (hi + lo) * B^T (the form in which the encoder's LayerNorm
 * outputs enter their projections). */
int cac_op_gemm_bf16(int M, int N, int K, const void* A, const void* B, const float* bias, float* C, int splits,
                     int a_split, void* stream);

/* C = A W^T (+ bias) with palette weights ("Fast Accuracy-Preserving RNNT Beam
 * Search on Apple Silicon", §1.3: 64-entry lookup tables, 6-bit palettes) on
 * the tensor cores (bf16 x bf16, fp32 accumulation).
 *   A       device bf16 [M][K], row-major, 16-byte aligned
 *   packed  device bytes [N][3K/4]: row n's indices as a little-endian bit
 *           stream, index k in bits [6k, 6k + 6); 16-byte aligned
 *   table   device bf16 [64]: W[n][k] = table[index]
 *   bias    device fp32 [N] or NULL;  C  device fp32 [M][N], 16-byte aligned
 *   status  device int or NULL: a bounded wait that gave up latches
 *           CAC_E_TIMEOUT there (first error wins)
 * N and K multiples of 64.  Asynchronous on `stream`.  CAC_E_INVAL for bad
 * sizes or NULL operands, CAC_E_ALIGN for misaligned pointers. */
int cac_op_gemm_palette(int M, int N, int K, const void* A, const void* packed, const void* table,
                        const float* bias, float* C, int* status, void* stream);

/* Failure-path self-test of the library's bounded device waits: runs the
 * wait the library uses with nothing that can satisfy it and returns the
 * status the device latched — CAC_E_TIMEOUT when the wait gave up as designed.
 *   which 0: an mbarrier wait (the TMA / tensor-core pipelines' wait) on a
 *            barrier no thread arrives at; gives up after about 2 s;
 *   which 1: the decoder's grid-wide barrier in a cooperative launch whose
 *            first block never arrives; the others give up after about 1 s,
 *            raise the abort word and return.
 * Synchronous; the kernels exit normally, so the context stays usable.
 * CAC_E_INVAL for another `which`, CAC_E_CUDA if a launch failed. */
int cac_op_wait_selftest(int which, void* stream);

/* Self-test of the checked build (cac_build_checked() == 1): a kernel whose
 * threads index past a 32-float buffer runs with the library's index check,
 * which keeps every access in bounds; returns the status it latched —
 * CAC_E_BOUNDS as designed.  Synchronous.  CAC_E_UNSUPPORTED in the default
 * build (nothing is launched). */
int cac_op_bounds_selftest(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CAC_OPS_H_ */
