/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) fused decode attention: the
 * score step (gqa_qk.h) and the AV reduction (gqa_av.h) in one pass over the
 * KV cache, the softmax weights made and used on chip.
 *
 * Operation: for every b < B, q_h < Hq and d < D,
 *
 *     s[b, c, q_h]   = scale * sum_d' q[b, q_h, d'] * K[b, c, kv_h, d'],
 *     out[b, q_h, d] = sum_{c < L_b} exp(s[b, c, q_h] - M) / Z * V[b, c, kv_h, d],
 *     M = max_{c < L_b} s[b, c, q_h],   Z = sum_{c < L_b} exp(s[b, c, q_h] - M),
 *     kv_h = q_h / G,   G = Hq / Hkv,   L_b = clamp(seq_lens[b], 0, Cmax);
 *
 * an empty context (L_b = 0) gives out = 0. The AV coop-GEMV of LLM decode
 * (page "pytorch/executorch pull 21063", summary paragraph) consumes softmax
 * weights; this call computes them from the same step's query-key products
 * with the same grouping of query heads onto KV heads. In GQA-reuse mode each
 * K and V row is read from HBM once for the G query heads of its group (for
 * G > 16, once per chunk of at most 16 of them); in per-head mode once per
 * query head. mode: -1 auto (GQA if G > 1), 0 per-head, 1 GQA.
 *
 * Layouts (all contiguous, row-major, caller-owned DEVICE memory, 16-byte
 * aligned):
 *     q         [B, Hq, D]          float32
 *     k_cache   [B, Cmax, Hkv, D]   bf16 (GQA_AV_BF16) or fp16 (GQA_AV_FP16)
 *     v_cache   [B, Cmax, Hkv, D]   the same type as k_cache
 *     seq_lens  [B]                 int32, or NULL meaning every L_b = Cmax
 *     out       [B, Hq, D]          float32, fully overwritten
 * Rows c >= L_b of the caches are never used (they may hold anything).
 *
 * Numerics: the query-key and weight-value products run on the tensor cores
 * with fp32 accumulation; the fp32 query (times scale * log2 e) and the fp32
 * weights are each split into two 16-bit halves of the cache's type, so the
 * products carry about 16 (bf16) or 22 (fp16) significant bits of them.
 * The running softmax and the output sums are fp32. Repeated calls with the
 * same shape give bitwise-identical out. For fp16 caches |q * scale| must stay
 * below 2^15 (the 16-bit halves must not overflow).
 *
 * Limits (GQA_AV_ERR_UNSUPPORTED otherwise): D = 64, 128 or 256.
 *
 * Execution: asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 * default stream), no host synchronisation. The call keeps its own
 * per-device workspace (split partials and a status word), grown on demand
 * with cudaMalloc outside stream capture; calls that may overlap on the GPU
 * must not be issued concurrently. Errors: a status code from gqa_av.h; on
 * error nothing is launched and gqa_attn_last_error() holds a message.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stdint.h>

#include "gqa_av.h"

#ifdef __cplusplus
extern "C" {
#endif

int gqa_attn_decode(const float *q, const void *k_cache, const void *v_cache,
                    const int32_t *seq_lens, float *out, int B, int Cmax, int Hq, int Hkv, int D,
                    int kv_dtype, float scale, int mode, void *stream);

/* The same with the launch shape chosen: consumer_warps (1..8; 1..6 at
 * D = 256) warps stream the context in each CTA; nsplit is the number of
 * context splits per tile (rounded so each split is a whole number of 32-row
 * stages); split_mode 1 cuts each sequence into those fixed splits, 2 spreads
 * the batch's context rows evenly over tiles x nsplit CTAs whatever the
 * lengths (each CTA reads all of seq_lens to find its split); column_blocks
 * 1 lets one CTA write all D output columns of its heads, 2 (D = 256 only)
 * gives each of two CTAs 128 of them (both compute all the scores). 0 lets
 * the library choose any of them: balanced splits when seq_lens is given and
 * B > 1, two column blocks at D = 256. Any choice gives results within the
 * stated bounds. */
int gqa_attn_decode_tuned(const float *q, const void *k_cache, const void *v_cache,
                          const int32_t *seq_lens, float *out, int B, int Cmax, int Hq, int Hkv,
                          int D, int kv_dtype, float scale, int mode, int consumer_warps,
                          int nsplit, int split_mode, int column_blocks, void *stream);

/* The launch plan of a call without launching it (ragged != 0: seq_lens will
 * be given): info[0..10] = resolved mode, query heads per CTA, consumer
 * warps, ring stages, rows per fixed split, splits per tile, tiles, dynamic
 * shared memory bytes, split mode (1 fixed, 2 balanced), CTAs launched,
 * column blocks (the first n_info of them). */
int gqa_attn_plan(int B, int Cmax, int Hq, int Hkv, int D, int kv_dtype, int mode,
                  int consumer_warps, int nsplit, int split_mode, int column_blocks, int ragged,
                  int *info, int n_info);

/* Synchronise `stream`, then read the call's device status word (set when a
 * bounded wait inside a kernel runs out): GQA_AV_OK or
 * GQA_AV_ERR_DEVICE_TIMEOUT; with clear != 0 the word is reset. */
int gqa_attn_device_status(void *stream, int clear);

/* Message of the calling thread's last attention error ("" if none). */
const char *gqa_attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
