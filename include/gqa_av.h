/*
 * gqa_av.h -- C ABI of the GB300 (sm_103a) grouped-query-attention AV decode
 * reduction.
 *
 * Operation (page "pytorch/executorch pull 21063", summary paragraph): in
 * grouped-query attention Hq = G * Hkv query heads share each KV head, and the
 * decode-step output of query head q_h is
 *
 *     out[b, q_h, d] = sum_{c < L_b} attn[b, c, q_h] * V[b, c, kv_h, d],
 *     kv_h = q_h / G,   G = Hq / Hkv,   L_b = clamp(seq_lens[b], 0, Cmax).
 *
 * The GQA-reuse variant (same page, paragraph on the GQA-reuse AV variant)
 * reads each V-cache row once and reuses it for all G query heads of its
 * group; the per-head variant reads it once per query head (G times). Both
 * compute the same sums. The mode switch follows the page's test-only override
 * knob (bullet on `gqa_override`): -1 auto-select, 0 force per-head,
 * 1 force GQA-reuse, so both kernels can be measured on one shape.
 *
 * Layouts (all contiguous, row-major, caller-owned DEVICE memory):
 *     attn      [B, Cmax, Hq]       float32
 *     v_cache   [B, Cmax, Hkv, D]   bf16 (GQA_AV_BF16) or fp16 (GQA_AV_FP16)
 *     seq_lens  [B]                 int32, or NULL meaning every L_b = Cmax
 *     out       [B, Hq, D]          float32, fully overwritten (never accumulated)
 * Entries at c >= L_b are never used. Values outside [0, Cmax] in seq_lens
 * are clamped to that range on the device.
 *
 * Numerics. V is widened exactly (bf16/fp16 -> fp32); which arithmetic runs
 * depends on the kernel the plan picks (gqa_av_plan_info.engine):
 *   - CUDA-core FMA kernel (engine 1: the default for D % 8 == 0 calls with
 *     fewer than 8 heads per CTA that stream fewer than 2^18 tile rows) and
 *     the generic kernel (engine 3: D % 8 != 0 or misaligned pointers):
 *     fp32 products and sums, every multiply-add rounded like fmaf.
 *   - tcgen05 tensor-core kernel (engine 2: the default where it applies --
 *     head groups of at most 64 heads, D >= 64 with D <= 128 or D % 128 == 0
 *     -- and the CTA has 8 or more heads or the call streams 2^18 tile rows
 *     or more): each fp32 weight w is split into two 16-bit values of V's
 *     type, hi = round(w) and lo = round(w - hi) (fp16 weights scaled by 2^12
 *     first, exactly, and unscaled at the end), so the weights keep about 16
 *     (bf16) or 22 (fp16) significant bits; V x hi and V x lo are exact in
 *     fp32; the tensor core accumulates them in fp32 over one pipeline stage
 *     (at most R / 16 products a value), and stages are added in fp32
 *     registers.
 * Both stay within max|out - exact| <= 1e-4 * max(1, max|exact|) on the
 * tested workloads. Context splits are combined in a fixed order, so repeated
 * calls with the same shape and lengths give bitwise-identical out.
 *
 * Execution: every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and performs no host synchronisation. Calls
 * share one per-device workspace, so calls that may overlap on the GPU (on
 * different streams) must not be issued concurrently; calls on one stream are
 * always safe. The workspace grows on demand with cudaMalloc; during stream
 * capture it cannot grow, so make one call with the largest shape first (or
 * supply a workspace with gqa_av_set_workspace).
 *
 * Errors: every entry point returns a status code. On any error nothing is
 * launched and gqa_av_last_error() holds a message for the calling thread.
 */
#ifndef GQA_AV_H
#define GQA_AV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define GQA_AV_OK                  0
#define GQA_AV_ERR_INVALID         1 /* NULL pointer, size <= 0, Hq % Hkv != 0, bad mode or dtype */
#define GQA_AV_ERR_UNSUPPORTED     2 /* outside a variant's limits (see each call), shape too large */
#define GQA_AV_ERR_CUDA            3 /* a CUDA runtime/driver call or a launch failed */
#define GQA_AV_ERR_NOMEM           4 /* workspace could not be allocated (or not during capture) */
#define GQA_AV_ERR_DEVICE_TIMEOUT  5 /* a bounded wait inside a kernel ran out (device status word) */

/* V-cache element types. */
#define GQA_AV_BF16 0
#define GQA_AV_FP16 1

/* Modes (the page's gqa_override knob). */
#define GQA_AV_MODE_AUTO     (-1) /* GQA-reuse when G > 1, per-head when G == 1 (MHA) */
#define GQA_AV_MODE_PER_HEAD   0  /* one CTA per (b, q_h, d-tile, split): V read G times */
#define GQA_AV_MODE_GQA        1  /* one CTA per (b, kv_h, d-tile, split): V read once */

/*
 * The reduction. Arguments as in the layouts above; B, Cmax, Hq, Hkv, D > 0,
 * Hq % Hkv == 0; attn and out 4-byte aligned, v_cache 2-byte aligned (their
 * element types), seq_lens 4-byte aligned. With D % 8 == 0 and attn, v_cache
 * and out 16-byte aligned the TMA kernels run (the FMA or the tensor-core
 * engine); any other D or alignment runs the generic kernel (plain loads, any
 * D >= 1; the page's 4-wide texel granularity and below), with the same
 * results within the stated gate and the same determinism. Forcing a mode on
 * a shape it cannot run is an error (never a silent fallback): with
 * Hq % Hkv != 0 every mode returns GQA_AV_ERR_INVALID.
 */
int gqa_av_decode(const float *attn, const void *v_cache, const int32_t *seq_lens,
                  float *out, int B, int Cmax, int Hq, int Hkv, int D,
                  int v_dtype, int mode, void *stream);

/* Per-head baseline: identical to gqa_av_decode(..., GQA_AV_MODE_PER_HEAD, stream). */
int gqa_av_decode_per_head(const float *attn, const void *v_cache, const int32_t *seq_lens,
                           float *out, int B, int Cmax, int Hq, int Hkv, int D,
                           int v_dtype, void *stream);

/*
 * Launch-shape overrides for sweeps and tests. A field <= 0 keeps the
 * library's choice.
 *   nsplit: context splits per tile (of a full-length sequence); with
 *     balanced splits the batch's context is spread over tiles x nsplit
 *     CTAs; with streamed splits it is the CTAs per SM (1..4, default 2).
 *   dtile: output columns per CTA (a multiple of 8 dividing D, <= 256).
 *   rows_per_stage: V rows per pipeline stage (8..256).
 *   stages: pipeline depth (2..8).
 *   early_stages: stages each CTA issues before it has read its sequence
 *     length (1..stages). With fixed splits the library issues one: rows past
 *     a length are read for nothing and the first stage lands later behind
 *     the others. Balanced and streamed splits issue none (a CTA finds its
 *     range from the lengths), though the value is still checked against
 *     stages.
 *   engine: 0 lets the library pick, 1 forces the CUDA-core packed-FMA
 *     kernel, 2 the tcgen05 tensor-core kernel (head groups of <= 64 heads
 *     and D >= 64 with D <= 128 or D % 128 == 0; dtile must then be
 *     min(D, 128) or unset and rows_per_stage a multiple of 16). The library
 *     picks the tensor-core kernel where it applies and the CTA has 8 or more
 *     heads or the call streams 2^18 tile rows or more (there the FMA kernel
 *     is bound by its own arithmetic issue), else the FMA kernel (short calls
 *     with few heads are latency-bound); setting dtile selects the FMA kernel.
 *   split_mode: 1 fixed splits (split s of each sequence covers rows
 *     [s, s + 1) x rows_per_split, and splits past a sequence's length have
 *     no work); 2 balanced splits (tensor-core engine only: every CTA reads
 *     all lengths and the batch's context rows are cut into equal splits of
 *     whole stages); 3 streamed splits (tensor-core engine only, contiguous V,
 *     B <= 2048: persistent CTAs, nsplit CTAs an SM, each take an equal run
 *     of one column of the call's stage list across sequence boundaries);
 *     0 lets the library pick: fixed for the FMA kernel; streamed for the
 *     tensor-core kernel, except where streaming does not apply (paged V,
 *     B > 2048) or nsplit or early_stages is set, where it takes balanced
 *     splits on shapes with at least as many tiles as SMs and fixed splits on
 *     the others.
 * Results stay within the stated tolerance for every choice, and are bitwise
 * reproducible for a fixed choice and fixed lengths. Tunings apply to the TMA
 * kernels only: a call that would run the generic kernel (D % 8 != 0 or a
 * pointer not 16-byte aligned) with any field set returns
 * GQA_AV_ERR_UNSUPPORTED. The paged and no-allocation variants keep the TMA
 * kernels' limits (D % 8 == 0, 16-byte aligned attn, V and out).
 */
typedef struct gqa_av_tuning {
    int nsplit;
    int dtile;
    int rows_per_stage;
    int stages;
    int early_stages;
    int engine;
    int split_mode;
} gqa_av_tuning;

int gqa_av_decode_tuned(const float *attn, const void *v_cache, const int32_t *seq_lens,
                        float *out, int B, int Cmax, int Hq, int Hkv, int D,
                        int v_dtype, int mode, const gqa_av_tuning *tuning, void *stream);

/*
 * Paged V cache (a block table, as serving engines keep their KV cache):
 * the same reduction, with V row c of sequence b at
 *     v_pool[block_table[b * max_blocks + c / block_size]][c % block_size][kv_h][:],
 *     v_pool [num_blocks, block_size, Hkv, D] (bf16/fp16), block_table [B, max_blocks] int32.
 * attn, seq_lens and out are as in gqa_av_decode, with Cmax <= max_blocks * block_size.
 * block_size is a positive multiple of 8; a stage is whole blocks or a divisor of one.
 * Table entries of blocks past a sequence's length are never used for the sum and may
 * hold anything; an entry outside [0, num_blocks) reads zeros. tuning may be NULL.
 */
int gqa_av_decode_paged(const float *attn, const void *v_pool, const int32_t *block_table,
                        const int32_t *seq_lens, float *out, int B, int Cmax, int Hq, int Hkv,
                        int D, int v_dtype, int block_size, int num_blocks, int max_blocks,
                        int mode, const gqa_av_tuning *tuning, void *stream);

/* The launch shape a call with these arguments would use (no launch, no allocation). */
typedef struct gqa_av_plan_info {
    int mode;            /* resolved mode: 0 per-head, 1 GQA-reuse */
    int heads_per_cta;   /* query heads each CTA accumulates (G or 1) */
    int head_chunk;      /* query heads per thread (a divisor of heads_per_cta) */
    int dtile;           /* output columns per CTA */
    int rows_per_stage;
    int stages;
    int early_stages;    /* stages issued before the sequence length is read (0: none) */
    int engine;          /* 1 CUDA-core packed FMA, 2 tcgen05 tensor cores, 3 generic
                            (D % 8 != 0; a call with misaligned pointers also runs it) */
    int split_mode;      /* 1 fixed, 2 balanced over the batch's lengths, 3 streamed */
    int nsplit;          /* context splits per tile (of a full-length sequence);
                            streamed: CTAs per SM */
    int combine_ctas;    /* CTAs of the split-combine kernel (0: not launched) */
    int rows_per_split;  /* of a full-length sequence */
    int tiles;           /* (head groups) x B x (D / dtile) */
    int ctas;            /* tiles x nsplit; tiles x (nsplit + 1) with balanced splits;
                            streamed: (head groups x D / dtile) x the groups that fit
                            nsplit CTAs on every SM */
    int threads_per_cta;
    int smem_bytes;
    int ctas_per_sm;     /* occupancy of this kernel at this shared-memory size */
    size_t workspace_bytes;
} gqa_av_plan_info;

int gqa_av_plan(int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode,
                const gqa_av_tuning *tuning, gqa_av_plan_info *info);

/* Device workspace bytes a call with these arguments needs (0 when none). */
size_t gqa_av_workspace_bytes(int B, int Cmax, int Hq, int Hkv, int D, int v_dtype, int mode);

/*
 * Hand the library a caller-owned device workspace for the current device
 * (at least gqa_av_workspace_bytes of the largest call, 256-byte aligned).
 * The library zeroes its status word here (synchronously) and never frees it.
 * ptr == NULL
 * returns to a library-owned workspace. The caller keeps the memory alive
 * until it calls gqa_av_set_workspace(NULL, 0) or the process ends.
 */
int gqa_av_set_workspace(void *ptr, size_t bytes);

/*
 * Synchronise `stream`, then read the current device's status words, which
 * kernels set when a bounded wait runs out: the one in the workspace of
 * gqa_av_decode and its variants, and the one in the fixed array of
 * gqa_av_decode_noalloc (once that call has run on the device). A word stays
 * set until it is cleared here, so a timeout in any earlier call is reported.
 * Returns GQA_AV_OK or GQA_AV_ERR_DEVICE_TIMEOUT; with clear != 0 both words
 * are reset.
 */
int gqa_av_device_status(void *stream, int clear);

/*
 * No-allocation variant of gqa_av_decode. The source pages have no
 * counterpart to it; it exists for callers that may not allocate device memory when they run the
 * reduction: engine plug-ins whose host owns all device memory, latency-
 * critical loops that must not risk the implicit synchronisation of
 * cudaMalloc/cudaFree, processes with a fixed up-front memory budget.
 *
 * Same arguments, layouts, launch shape and results as gqa_av_decode on the
 * calls the TMA kernels take: D % 8 == 0 and 16-byte aligned attn, v_cache
 * and out (anything else returns GQA_AV_ERR_UNSUPPORTED; gqa_av_decode runs
 * it on the generic kernel). The scratch it needs (status word, split
 * partials) lives in one fixed array of GQA_AV_NOALLOC_SCRATCH_BYTES in this
 * library's device globals, held on every GPU that loads the library until
 * the process exits. No call allocates or frees memory. Set-up: the first
 * call on each device looks up that array's device address
 * (cudaGetSymbolAddress) and zeroes its status word (synchronously), so make
 * that first call before any stream capture. A shape whose split partials
 * need more than the array holds (8 MiB less its 256-byte status word) is
 * rejected with GQA_AV_ERR_UNSUPPORTED and a message; gqa_av_decode handles
 * it. All calls on a device share the array, which keeps the last call's
 * contents: every partial is written before it is read, and the status word
 * stays set until gqa_av_device_status reads and clears it (that call reports
 * this array's word together with gqa_av_decode's). Calls that may overlap on
 * the GPU (unordered streams) race on the array and must not be issued.
 */
#define GQA_AV_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB */

int gqa_av_decode_noalloc(const float *attn, const void *v_cache, const int32_t *seq_lens,
                          float *out, int B, int Cmax, int Hq, int Hkv, int D,
                          int v_dtype, int mode, void *stream);

/*
 * Self-test of the failure path (the pages have no counterpart: it checks
 * this library's bounded waits). Runs the CUDA-core FMA kernel on the given
 * call (same arguments and limits as gqa_av_decode's TMA kernels, mode auto)
 * with the producer withholding the last pipeline stage of every context
 * split of at least two stages -- nothing of that stage is ever issued, so no
 * copy is in flight when a CTA leaves -- and the consumers' wait for a stage
 * bounded by wait_ns (1 us to 2 s) instead of 2 s. Their wait for the
 * withheld stage runs out, they set the device status word and leave through
 * the same barriers as on any timeout; no GPU fault, trap or hang is caused.
 * scratch 0 puts the status word and partials in gqa_av_decode's workspace,
 * 1 in gqa_av_decode_noalloc's fixed array. Returns GQA_AV_OK once launched;
 * gqa_av_device_status then reports GQA_AV_ERR_DEVICE_TIMEOUT. `out` is left
 * unspecified. GQA_AV_ERR_UNSUPPORTED when the call's splits are shorter than
 * two stages.
 */
int gqa_av_selftest_wait_timeout(const float *attn, const void *v_cache, const int32_t *seq_lens,
                                 float *out, int B, int Cmax, int Hq, int Hkv, int D,
                                 int v_dtype, long long wait_ns, int scratch, void *stream);

/* Name of a status code; never NULL. */
const char *gqa_av_status_string(int status);

/* Message of the calling thread's last error ("" if none). */
const char *gqa_av_last_error(void);

/* Library version, for the Python binding's load check. */
int gqa_av_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GQA_AV_H */
