/*
 * CPU oracle for the grouped-query-attention AV decode reduction.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. It shares no code with the CUDA path.
 *
 * Definition (page "pytorch/executorch pull 21063", summary paragraph): in
 * grouped-query attention Hq = G * Hkv query heads share each KV head, and the
 * decode-step output of query head q_h is the attention-weighted sum of the V
 * cache rows of its KV head,
 *
 *     out[b, q_h, d] = sum_{c = 0}^{L_b - 1} attn[b, c, q_h] * V[b, c, kv_h, d],
 *     kv_h = q_h / G (contiguous groups),  G = Hq / Hkv,
 *     L_b  = clamp(seq_lens[b], 0, Cmax)   (Cmax for every b when seq_lens is NULL).
 *
 * The batch index b and the per-sequence lengths are added in front of the
 * page's formula; positions c >= L_b are never read. The weights are taken as
 * given (no softmax here). Every product and the whole sum are done in binary64;
 * each product of an fp32 weight with a bf16/fp16 value is exact in binary64,
 * so the only rounding is the L-term sum, in increasing c.
 *
 * Layouts, all contiguous row-major:
 *     attn     [B, Cmax, Hq]      binary32
 *     v_bits   [B, Cmax, Hkv, D]  raw 16-bit patterns, bf16 (v_dtype 0) or fp16 (1)
 *     seq_lens [B]                int32, may be NULL
 *     out      [B, Hq, D]         binary64, fully overwritten
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bfloat16 is the upper half of an IEEE-754 binary32 pattern. */
double oracle_decode_bf16(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE-754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_fp16(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int m = bits & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
    else if (e == 31)
        mag = m ? NAN : INFINITY;
    else
        mag = ldexp((double)(m + 1024), e - 25);  /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -mag : mag;
}

typedef struct {
    const float *attn;
    const uint16_t *v_bits;
    const int32_t *seq_lens;
    double *out;
    int64_t B, Cmax, Hq, Hkv, D;
    int v_dtype;
    int64_t unit_begin, unit_step;
} job_t;

static double decode(uint16_t bits, int v_dtype)
{
    return v_dtype == 0 ? oracle_decode_bf16(bits) : oracle_decode_fp16(bits);
}

/* One unit of work is one (b, q_h) pair: all D outputs of that query head. */
static void *worker(void *arg)
{
    const job_t *j = (const job_t *)arg;
    const int64_t G = j->Hq / j->Hkv;
    double *acc = (double *)malloc((size_t)j->D * sizeof(double));
    if (!acc)
        return (void *)1;
    for (int64_t u = j->unit_begin; u < j->B * j->Hq; u += j->unit_step) {
        const int64_t b = u / j->Hq;
        const int64_t q_h = u % j->Hq;
        const int64_t kv_h = q_h / G;
        int64_t L = j->seq_lens ? (int64_t)j->seq_lens[b] : j->Cmax;
        if (L < 0) L = 0;
        if (L > j->Cmax) L = j->Cmax;
        for (int64_t d = 0; d < j->D; ++d)
            acc[d] = 0.0;
        for (int64_t c = 0; c < L; ++c) {
            const double w = (double)j->attn[(b * j->Cmax + c) * j->Hq + q_h];
            const uint16_t *row = j->v_bits + ((b * j->Cmax + c) * j->Hkv + kv_h) * j->D;
            for (int64_t d = 0; d < j->D; ++d)
                acc[d] += w * decode(row[d], j->v_dtype);
        }
        double *o = j->out + (b * j->Hq + q_h) * j->D;
        for (int64_t d = 0; d < j->D; ++d)
            o[d] = acc[d];
    }
    free(acc);
    return NULL;
}

/*
 * Returns 0 on success, -1 on invalid arguments (NULL pointer, negative size,
 * Hkv == 0, Hq not a multiple of Hkv, unknown v_dtype), -2 if a thread could
 * not be started or ran out of memory. nthreads <= 0 means one thread.
 */
int oracle_gqa_av(const float *attn, const uint16_t *v_bits, int v_dtype,
                  const int32_t *seq_lens, double *out,
                  int64_t B, int64_t Cmax, int64_t Hq, int64_t Hkv, int64_t D,
                  int nthreads)
{
    if (B < 0 || Cmax < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0)
        return -1;
    if (v_dtype != 0 && v_dtype != 1)
        return -1;
    if (B == 0)
        return 0;
    if (!out || (Cmax > 0 && (!attn || !v_bits)))
        return -1;
    if (nthreads <= 0)
        nthreads = 1;
    if ((int64_t)nthreads > B * Hq)
        nthreads = (int)(B * Hq);

    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    int rc = 0, started = 0;
    for (int t = 0; t < nthreads; ++t) {
        job_t j = {attn, v_bits, seq_lens, out, B, Cmax, Hq, Hkv, D, v_dtype,
                   t, nthreads};
        jobs[t] = j;
        if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) {
            rc = -2;
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(tids[t], &ret);
        if (ret)
            rc = -2;
    }
    free(jobs);
    free(tids);
    return rc;
}
