/*
 * attention.h: C ABI of the attention forward pass of libdtgemm.so (sm_103a).
 *
 * "Two Waves, One Stage Apart: Warp-Pipelining Triton GEMMs on AMD Instinct"
 * (section "Beyond GEMM: FlashAttention") carries the GEMM's stage-offset
 * schedule over to the FlashAttention inner loop: QK and PV products
 * alternate with an online softmax, and the QK product of the next key block
 * overlaps the PV product of the current one. This entry point computes that
 * loop's result,
 *
 *     O = softmax(scale * Q K^T) V,    LSE = log(sum_k exp(scale * q . k))
 *
 * per (batch, head), with FP32 accumulation (scores, probabilities' sum and
 * output) and the output cast to the operand type, rounding to nearest even.
 * The probabilities enter the PV product rounded to the operand type; their
 * FP32 row sum is taken before that rounding.
 * Status codes are gemm.h's gemm_status_t.
 */
#ifndef DENSE_TILED_GEMM_ATTENTION_H
#define DENSE_TILED_GEMM_ATTENTION_H

#include <stdint.h>

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attention_fwd: O = softmax(scale * Q K^T) V on the current device,
 * asynchronously on `stream`.
 *
 *   Q       device pointer, [B][H][Lq][d] row-major, dtype.
 *   K, V    device pointers, [B][H][Lk][d] row-major, dtype.
 *   O       device pointer, [B][H][Lq][d] row-major, dtype (written).
 *   LSE     device pointer, [B][H][Lq] FP32 natural-log row log-sum-exp
 *           (written), or NULL. A row with no visible key gets -inf and an
 *           all-zero O row.
 *   B, H, Lq, Lk  sizes >= 1, B * H <= 2^31 - 1 (GEMM_ERR_UNSUPPORTED otherwise).
 *   d       head dimension; must be 128 (otherwise GEMM_ERR_UNSUPPORTED).
 *   dtype   GEMM_F16 or GEMM_BF16 for Q, K, V and O.
 *   causal  0: every key is visible; 1: key k is visible to query row i iff
 *           k <= i + (Lk - Lq) (the diagonal ends at the last query row).
 *   scale   the score scale, usually 1/sqrt(d); must be finite and > 0.
 *   stream  cudaStream_t as void*.
 *
 * Base addresses must be 16-byte aligned (GEMM_ERR_UNSUPPORTED otherwise).
 * The caller owns all memory; nothing is allocated. The call may be captured
 * into a CUDA graph once one call on the device has run outside the capture. Errors: host-side
 * argument checks return before launch; a kernel wait past its limit (2 s)
 * is reported through gemm_last_device_status.
 */
gemm_status_t attention_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                            int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t d,
                            int dtype, int causal, float scale, void *stream);

/*
 * attention_fwd_ex: attention_fwd with a cap on the persistent grid.
 *
 * The kernel runs one CTA per SM (never more than one per row block of 256
 * query rows of one head); each CTA takes one row block per round of G (the
 * grid size), rounds alternating in direction. max_ctas > 0 caps G, so that
 * each CTA takes more row blocks (the tests use it to reach that path on
 * small problems); max_ctas <= 0 means no cap. Arguments, results and errors are
 * attention_fwd's; max_ctas changes neither the result nor its bits.
 */
gemm_status_t attention_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE,
                               int64_t B, int64_t H, int64_t Lq, int64_t Lk, int64_t d,
                               int dtype, int causal, float scale, int max_ctas, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_TILED_GEMM_ATTENTION_H */
