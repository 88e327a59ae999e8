/*
 * gqa_qk.h -- C ABI of the GB300 (sm_103a) decode score step: the softmax-
 * normalised query-key products that the AV reduction (gqa_av.h) consumes.
 *
 * Operation: for every b < B, q_h < Hq and c < L_b,
 *
 *     s[b, c, q_h]    = scale * sum_d q[b, q_h, d] * K[b, c, kv_h, d],
 *     attn[b, c, q_h] = exp(s[b, c, q_h] - M) / sum_{c' < L_b} exp(s[b, c', q_h] - M),
 *     kv_h = q_h / G,   G = Hq / Hkv,   M = max_{c' < L_b} s[b, c', q_h],
 *     L_b = clamp(seq_lens[b], 0, Cmax).
 *
 * It is the step before the AV coop-GEMV of LLM decode (page "pytorch/
 * executorch pull 21063", summary paragraph), with the same grouping of
 * query heads onto KV heads: in GQA-reuse mode each K row is read from HBM
 * once for the G query heads of its group, in per-head mode once per query
 * head. The mode switch follows the AV call's: -1 auto, 0 per-head, 1 GQA.
 *
 * Layouts (all contiguous, row-major, caller-owned DEVICE memory, 16-byte
 * aligned):
 *     q         [B, Hq, D]          float32
 *     k_cache   [B, Cmax, Hkv, D]   bf16 (GQA_AV_BF16) or fp16 (GQA_AV_FP16)
 *     seq_lens  [B]                 int32, or NULL meaning every L_b = Cmax
 *     attn      [B, Cmax, Hq]       float32: rows c < L_b are written;
 *                                   rows c >= L_b are left untouched
 * attn is the layout gqa_av_decode takes, so the two calls chain directly.
 *
 * Numerics. K is widened exactly (bf16/fp16 -> fp32). The CUDA-core FMA
 * kernel (engine 1) forms the products and sums over d in fp32. The tcgen05
 * tensor-core kernels (engines 2 and 3, the defaults) split each fp32 query value
 * into two 16-bit values of K's type, hi = round(q) and lo = round(q - hi),
 * so the query keeps about 16 (bf16) or 22 (fp16) significant bits; K x hi
 * and K x lo are exact in fp32 and accumulated over d in fp32 in tensor
 * memory. The softmax runs in fp32 from per-split (max, sum of exp) pairs
 * merged in a fixed order, so repeated calls with the same shape give
 * bitwise-identical attn. Every written probability stays within 1e-4 of the
 * exact value relative to that value, and every row sums to 1 within 1e-5, on
 * the tested shapes.
 *
 * Limits (GQA_AV_ERR_UNSUPPORTED otherwise): D = 64, 128 or 256;
 * at most 64 query heads per KV head in GQA mode, and a head count per CTA
 * that splits into at most 8 chunks of at most 16 heads; Hq <= 2048.
 *
 * Execution: asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 * default stream), no host synchronisation. The call keeps its own
 * per-device workspace (per-split or per-segment softmax pairs and a status
 * word), grown on
 * demand with cudaMalloc outside stream capture; calls that may overlap on the
 * GPU must not be issued concurrently. Errors: a status code from gqa_av.h;
 * on error nothing is launched and gqa_qk_last_error() holds a message.
 */
#ifndef GQA_QK_H
#define GQA_QK_H

#include <stdint.h>

#include "gqa_av.h"

#ifdef __cplusplus
extern "C" {
#endif

int gqa_qk_softmax_decode(const float *q, const void *k_cache, const int32_t *seq_lens,
                          float *attn, int B, int Cmax, int Hq, int Hkv, int D, int k_dtype,
                          float scale, int mode, void *stream);

/* The same with the kernel chosen: engine 0 lets the library pick (the
 * streamed tensor-core kernel for at most 2048 sequences, except on short
 * streams -- fewer tiles (sequences x head groups) than SMs, D <= 128 and at
 * most 2 x 2048 x SMs rows over all tiles -- and on larger batches, where it
 * takes the fixed-split one), 1 forces the CUDA-core FMA kernel, 2 the tcgen05 tensor-core kernel
 * with fixed context splits (K rows as the A operand in place, the queries
 * split into 16-bit hi and lo halves as B), 3 the streamed tcgen05 kernel
 * (the same products; persistent CTAs, two an SM where they fit, each taking
 * an equal run of its head group's 128-row stages across sequences; at most
 * 2048 sequences). All give results within the stated tolerance. */
int gqa_qk_softmax_decode_tuned(const float *q, const void *k_cache, const int32_t *seq_lens,
                                float *attn, int B, int Cmax, int Hq, int Hkv, int D,
                                int k_dtype, float scale, int mode, int engine, void *stream);

/* Synchronise `stream`, then read this call's device status word (set when a
 * bounded wait inside a kernel runs out): GQA_AV_OK or
 * GQA_AV_ERR_DEVICE_TIMEOUT; with clear != 0 the word is reset. */
int gqa_qk_device_status(void *stream, int clear);

/* Message of the calling thread's last score-step error ("" if none). */
const char *gqa_qk_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_QK_H */
