/*
 * oracle.c -- plain, slow CPU oracle for the FP8 KV-cache write and for
 * attention over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant generator with the CUDA library: everything here is written
 * from the method's definition, in float64 where the method leaves the precision
 * open, with no blocking, fusion or reordering.
 *
 * Sources (web pages; cited by title and section):
 *   [KO]  "vLLM FP8 KV-Cache 및 Attention 양자화 업데이트" (agentlenshq.com, ko):
 *         storing K/V as FP8 e4m3 halves KV storage and attention runs in FP8
 *         (opening paragraph); per-KV-head scale arrays ("커널 및 퓨전 최적화");
 *         uncalibrated scale = 1.0 ("정확도 및 검증"); sliding-window layers kept
 *         in BF16 ("하이브리드 Attention 및 레이어 스킵").
 *   [KVQ] "[vLLM] KV Cache Quantization: KV 캐시 FP8/INT8 양자화"
 *         (blog.secrett2633.cloud): per-token-head scales computed by the kernel at
 *         cache-store time, per-tensor scale from a checkpoint or 1.0
 *         ("Per-Token-Head vs Per-Tensor 양자화").
 *   [PR]  "vLLM Qwen3.8-Flash-Next: QSA Indexer 캐시를 위한 FP8 지원 ..."
 *         (blog.secrett2633.cloud): the dtype is torch.float8_e4m3fn, e4m3 is
 *         sign-magnitude, and the absolute grid step at denormal magnitudes is
 *         2^-9 ("코드 분석", the assert_fp8_within_one_ulp helper).
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *   - e4m3 variant is e4m3fn: bias 7, no infinities, NaN = S.1111.111, largest
 *     finite 448.  Encoding rounds to nearest, ties to even, and saturates to
 *     +-448 (satfinite); NaN stays NaN.
 *   - per-token-head scale = fp32(amax / 448) with amax = max |x| over the head's
 *     D channels of one token; codes are e4m3(fp32(x / scale)).  A zero scale
 *     (an all-zero row) stores scale 0 and codes 0.
 *   - page size 16; slot = block * 16 + offset; a negative slot is skipped.
 *   - query head hq reads KV head hq / (Hq / Hkv).
 *   - a window w > 0 keeps the keys at positions >= ctx - w.
 *   - prefill query i of a chunk of n queries sits at position ctx - n + i and
 *     sees keys 0 .. that position.
 *
 * Numeric conventions shared with callers (interface values, not code):
 *   kv_dtype   0 = e4m3 cache, 1 = bf16 cache
 *   scale_mode 0 = per tensor, 1 = per KV head, 2 = per token and KV head
 * Return codes: 0 ok, -1 invalid argument, -6 bad block id / slot.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PAGE 16

/* ------------------------------------------------------------------------ */
/* e4m3fn codec                                                              */
/* ------------------------------------------------------------------------ */

/*
 * Encode one fp32 value as an e4m3fn byte: round to nearest, ties to even,
 * saturating to +-448.  Works on the integer bits of the float: the value is
 * significand * 2^(exponent - 150) with a 24-bit significand, and the e4m3
 * quantum at that magnitude is 2^(max(e, -6) - 3), so the code's integer
 * mantissa is the significand shifted right with guard/sticky rounding.
 */
uint8_t oracle_e4m3_encode(float x)
{
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    uint8_t sign = (uint8_t)((bits >> 24) & 0x80u);
    uint32_t mag = bits & 0x7FFFFFFFu;

    if (mag > 0x7F800000u)            /* NaN stays NaN (S.1111.111) */
        return (uint8_t)(sign | 0x7Fu);
    if (mag >= 0x43E00000u)           /* |x| >= 448 (also +-inf): saturate */
        return (uint8_t)(sign | 0x7Eu);

    int32_t biased = (int32_t)(mag >> 23);
    if (biased == 0)                  /* fp32 subnormal: far below 2^-10 */
        return sign;
    uint32_t signif = (mag & 0x7FFFFFu) | 0x800000u;   /* 24-bit significand */
    int32_t e = biased - 127;                          /* |x| in [2^e, 2^(e+1)) */

    /* Exponent of the e4m3 quantum: 2^(e-3) for normals (e >= -6), 2^-9 below. */
    int32_t quantum_exp = (e >= -6 ? e : -6) - 3;
    /* |x| / 2^quantum_exp = signif * 2^(e - 23 - quantum_exp) */
    int32_t shift = quantum_exp - (e - 23);            /* >= 20 */
    if (shift >= 26)                                   /* |x| / quantum < 1/2 */
        return sign;

    uint32_t n = signif >> shift;
    uint32_t rem = signif & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (n & 1u)))
        n += 1u;

    /* |x| ~= n * 2^quantum_exp. */
    uint32_t code;
    if (e < -6) {
        /* Subnormal quantum 2^-9: code is the mantissa itself.  n == 8 is the
         * smallest normal 2^-6, whose code (exponent field 1, mantissa 0) is 8. */
        code = n;
    } else {
        /* n in [8, 16]; n == 16 means the rounding carried into the next binade. */
        int32_t exp_field = e + 7;
        if (n == 16u) {
            n = 8u;
            exp_field += 1;
        }
        code = ((uint32_t)exp_field << 3) | (n - 8u);
    }
    return (uint8_t)(sign | code);
}

/* Exact value of an e4m3fn byte. */
double oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int ef = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (ef == 0xF && m == 7)
        v = NAN;
    else if (ef == 0)
        v = ldexp((double)m, -9);                  /* subnormal: m * 2^-9 */
    else
        v = ldexp(1.0 + (double)m / 8.0, ef - 7);  /* normal: (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

void oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

/* bf16 bit pattern -> float (exact: bf16 is the top half of an fp32). */
static float bf16_to_float(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* KV cache write                                                            */
/* ------------------------------------------------------------------------ */

/* Quantize one token-head row of D values into e4m3 codes with scale s. */
static void quantize_row(const uint16_t* x, int D, float s, uint8_t* codes)
{
    for (int d = 0; d < D; ++d) {
        if (s == 0.0f) {
            codes[d] = 0;
        } else {
            float q = bf16_to_float(x[d]) / s;   /* IEEE fp32 divide */
            codes[d] = oracle_e4m3_encode(q);
        }
    }
}

/* fp32 amax / 448 of one row (the dynamic per-token-head scale). */
static float row_scale(const uint16_t* x, int D)
{
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(bf16_to_float(x[d]));
        if (a > amax)
            amax = a;
    }
    return amax / 448.0f;
}

/*
 * Write T new tokens of K and V (bf16 [T][Hkv][D]) into the paged cache
 * [num_blocks][Hkv][16][D] at slot_mapping[t] (block * 16 + offset).
 * kv_dtype 1 copies the bf16 bytes; kv_dtype 0 stores e4m3 codes under the
 * scale mode and, for per-token-head scales, the fp32 scale of every
 * (token, head) row into k/v_scale_cache [num_blocks][Hkv][16].
 */
int oracle_kv_cache_write(const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                          int64_t T, int Hkv, int D, int kv_dtype, int scale_mode,
                          const float* k_scale, const float* v_scale,
                          void* k_cache, void* v_cache,
                          float* k_scale_cache, float* v_scale_cache, int64_t num_blocks)
{
    if (T < 0 || Hkv <= 0 || D <= 0 || (kv_dtype != 0 && kv_dtype != 1))
        return -1;
    if (kv_dtype == 0 && (scale_mode < 0 || scale_mode > 2))
        return -1;
    int status = 0;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / PAGE, off = slot % PAGE;
        if (blk >= num_blocks) {
            status = -6;
            continue;
        }
        for (int h = 0; h < Hkv; ++h) {
            const uint16_t* xk = k + ((size_t)t * Hkv + h) * D;
            const uint16_t* xv = v + ((size_t)t * Hkv + h) * D;
            size_t row = ((size_t)blk * Hkv + h) * PAGE + (size_t)off;
            if (kv_dtype == 1) {
                memcpy((uint16_t*)k_cache + row * D, xk, (size_t)D * 2);
                memcpy((uint16_t*)v_cache + row * D, xv, (size_t)D * 2);
                continue;
            }
            float sk, sv;
            if (scale_mode == 0) {
                sk = k_scale[0];
                sv = v_scale[0];
            } else if (scale_mode == 1) {
                sk = k_scale[h];
                sv = v_scale[h];
            } else {
                sk = row_scale(xk, D);
                sv = row_scale(xv, D);
                k_scale_cache[row] = sk;
                v_scale_cache[row] = sv;
            }
            quantize_row(xk, D, sk, (uint8_t*)k_cache + row * D);
            quantize_row(xv, D, sv, (uint8_t*)v_cache + row * D);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Attention over the dequantized paged cache (float64)                      */
/* ------------------------------------------------------------------------ */

typedef struct {
    const void* k_cache;
    const void* v_cache;
    int kv_dtype, scale_mode;
    const float *k_scale, *v_scale, *k_scale_cache, *v_scale_cache;
    const int32_t* block_table;
    int max_blocks_per_seq;
    int Hkv, D;
    int64_t num_blocks;
} cache_view;

/* Dequantized value of cache element (row, d) and its scale, in double. */
static double cache_value(const cache_view* c, const void* base, const float* tensor_scale,
                          const float* token_scale, size_t row, int h, int d)
{
    if (c->kv_dtype == 1)
        return (double)bf16_to_float(((const uint16_t*)base)[row * c->D + d]);
    double s;
    if (c->scale_mode == 0)
        s = tensor_scale[0];
    else if (c->scale_mode == 1)
        s = tensor_scale[h];
    else
        s = token_scale[row];
    return oracle_e4m3_decode(((const uint8_t*)base)[row * c->D + d]) * s;
}

/*
 * One query head of one sequence attends to key positions [lo, hi) of that
 * sequence: z_t = softmax_scale * sum_d q_d k_hat_{t,d}; w = softmax(z) (max,
 * then exponentials and their sum); o = sum_t w_t v_hat_t.  An empty range
 * gives zeros.  Returns 0 or -6 on a block id outside the cache.
 */
static int attend(const cache_view* c, const uint16_t* q, int seq, int h, int lo, int hi,
                  double softmax_scale, double* out)
{
    int D = c->D;
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (hi <= lo)
        return 0;
    int n = hi - lo;
    double* z = (double*)malloc(sizeof(double) * (size_t)n);
    size_t* rows = (size_t*)malloc(sizeof(size_t) * (size_t)n);
    if (!z || !rows) {
        free(z);
        free(rows);
        return -1;
    }
    for (int j = 0; j < n; ++j) {
        int t = lo + j;
        int32_t blk = c->block_table[(size_t)seq * c->max_blocks_per_seq + t / PAGE];
        if (blk < 0 || blk >= c->num_blocks) {
            free(z);
            free(rows);
            return -6;
        }
        rows[j] = ((size_t)blk * c->Hkv + h) * PAGE + (size_t)(t % PAGE);
    }
    /* logits */
    for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) {
            double qd = (double)bf16_to_float(q[d]);
            double kd = cache_value(c, c->k_cache, c->k_scale, c->k_scale_cache, rows[j], h, d);
            dot += qd * kd;
        }
        z[j] = softmax_scale * dot;
    }
    /* softmax: max, exponentials, sum */
    double m = z[0];
    for (int j = 1; j < n; ++j)
        if (z[j] > m)
            m = z[j];
    double sum = 0.0;
    for (int j = 0; j < n; ++j) {
        z[j] = exp(z[j] - m);
        sum += z[j];
    }
    /* weighted sum of values */
    for (int j = 0; j < n; ++j) {
        double w = z[j] / sum;
        for (int d = 0; d < D; ++d)
            out[d] += w * cache_value(c, c->v_cache, c->v_scale, c->v_scale_cache, rows[j], h, d);
    }
    free(z);
    free(rows);
    return 0;
}

typedef struct {
    const cache_view* c;
    const uint16_t* q;           /* decode: [B][Hq][D]; prefill: [Tq][Hq][D] */
    const int32_t* context_lens;
    const int32_t* cu_seqlens_q; /* prefill only */
    int B, Hq, window, prefill;
    double softmax_scale;
    const int32_t* units;        /* (seq or token, hq) pairs */
    int64_t begin, end;
    double* out;                 /* [n_units][D] */
    int status;
} work_slice;

static int run_unit(const work_slice* w, int64_t u)
{
    const cache_view* c = w->c;
    int a = w->units[2 * u], hq = w->units[2 * u + 1];
    int G = w->Hq / c->Hkv;
    int h = hq / G;
    double* out = w->out + (size_t)u * c->D;
    if (!w->prefill) {
        int seq = a;
        if (seq < 0 || seq >= w->B || hq < 0 || hq >= w->Hq)
            return -1;
        int ctx = w->context_lens[seq];
        if (ctx < 0 || ctx > c->max_blocks_per_seq * PAGE)
            return -1;
        int lo = (w->window > 0 && ctx > w->window) ? ctx - w->window : 0;
        const uint16_t* q = w->q + ((size_t)seq * w->Hq + hq) * c->D;
        return attend(c, q, seq, h, lo, ctx, w->softmax_scale, out);
    }
    /* prefill: a is the query token's row in the packed chunk */
    int tok = a, seq = -1;
    for (int b = 0; b < w->B; ++b)
        if (tok >= w->cu_seqlens_q[b] && tok < w->cu_seqlens_q[b + 1]) {
            seq = b;
            break;
        }
    if (seq < 0 || hq < 0 || hq >= w->Hq)
        return -1;
    int nq = w->cu_seqlens_q[seq + 1] - w->cu_seqlens_q[seq];
    int ctx = w->context_lens[seq];
    int pos = ctx - nq + (tok - w->cu_seqlens_q[seq]);
    if (pos < 0 || ctx > c->max_blocks_per_seq * PAGE)
        return -1;
    const uint16_t* q = w->q + ((size_t)tok * w->Hq + hq) * c->D;
    return attend(c, q, seq, h, 0, pos + 1, w->softmax_scale, out);
}

static void* run_slice(void* arg)
{
    work_slice* w = (work_slice*)arg;
    w->status = 0;
    for (int64_t u = w->begin; u < w->end; ++u) {
        int s = run_unit(w, u);
        if (s != 0 && w->status == 0)
            w->status = s;
    }
    return NULL;
}

static int run_units(const work_slice* proto, int64_t n_units, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((int64_t)nthreads > n_units)
        nthreads = n_units > 0 ? (int)n_units : 1;
    work_slice slices[256];
    pthread_t tids[256];
    int started[256];
    for (int i = 0; i < nthreads; ++i) {
        slices[i] = *proto;
        slices[i].begin = n_units * i / nthreads;
        slices[i].end = n_units * (i + 1) / nthreads;
        started[i] = 0;
    }
    for (int i = 1; i < nthreads; ++i)
        started[i] = pthread_create(&tids[i], NULL, run_slice, &slices[i]) == 0;
    run_slice(&slices[0]);
    int status = slices[0].status;
    for (int i = 1; i < nthreads; ++i) {
        if (started[i])
            pthread_join(tids[i], NULL);
        else
            run_slice(&slices[i]);
        if (slices[i].status != 0 && status == 0)
            status = slices[i].status;
    }
    return status;
}

/*
 * Decode attention: for every listed unit (seq, hq), the query q[seq][hq]
 * attends to the sequence's keys [lo, ctx) (lo = ctx - window when a window is
 * set).  units is n_units (seq, hq) int32 pairs; out is [n_units][D] float64.
 */
int oracle_decode_attn(const uint16_t* q, const void* k_cache, const void* v_cache,
                       int kv_dtype, int scale_mode,
                       const float* k_scale, const float* v_scale,
                       const float* k_scale_cache, const float* v_scale_cache,
                       const int32_t* block_table, int max_blocks_per_seq,
                       const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                       int64_t num_blocks, double softmax_scale, int window,
                       const int32_t* units, int64_t n_units, double* out, int nthreads)
{
    if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || D <= 0 || n_units < 0)
        return -1;
    if (kv_dtype != 0 && kv_dtype != 1)
        return -1;
    if (kv_dtype == 0 && (scale_mode < 0 || scale_mode > 2))
        return -1;
    cache_view c = {k_cache, v_cache, kv_dtype, scale_mode, k_scale, v_scale,
                    k_scale_cache, v_scale_cache, block_table, max_blocks_per_seq,
                    Hkv, D, num_blocks};
    work_slice w;
    memset(&w, 0, sizeof w);
    w.c = &c;
    w.q = q;
    w.context_lens = context_lens;
    w.B = B;
    w.Hq = Hq;
    w.window = window;
    w.prefill = 0;
    w.softmax_scale = softmax_scale;
    w.units = units;
    w.out = out;
    return run_units(&w, n_units, nthreads);
}

/*
 * Chunked-prefill attention: q is [Tq][Hq][D] holding each sequence's new
 * queries back to back (cu_seqlens_q[b] .. cu_seqlens_q[b+1]); context_lens[b]
 * counts all keys of sequence b including the chunk, which is already in the
 * cache.  Query i of sequence b sits at position ctx_b - n_b + i and attends
 * causally to keys 0 .. that position.  Q and P are not quantized here: this is
 * the exact result the FP8 tensor-core path approximates.  units is (token, hq)
 * pairs; out is [n_units][D] float64.
 */
int oracle_prefill_attn(const uint16_t* q, const int32_t* cu_seqlens_q,
                        const void* k_cache, const void* v_cache, int kv_dtype, int scale_mode,
                        const float* k_scale, const float* v_scale,
                        const float* k_scale_cache, const float* v_scale_cache,
                        const int32_t* block_table, int max_blocks_per_seq,
                        const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                        int64_t num_blocks, double softmax_scale,
                        const int32_t* units, int64_t n_units, double* out, int nthreads)
{
    if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0 || D <= 0 || n_units < 0 || B < 0)
        return -1;
    if (kv_dtype != 0 && kv_dtype != 1)
        return -1;
    if (kv_dtype == 0 && (scale_mode < 0 || scale_mode > 2))
        return -1;
    cache_view c = {k_cache, v_cache, kv_dtype, scale_mode, k_scale, v_scale,
                    k_scale_cache, v_scale_cache, block_table, max_blocks_per_seq,
                    Hkv, D, num_blocks};
    work_slice w;
    memset(&w, 0, sizeof w);
    w.c = &c;
    w.q = q;
    w.context_lens = context_lens;
    w.cu_seqlens_q = cu_seqlens_q;
    w.B = B;
    w.Hq = Hq;
    w.window = 0;
    w.prefill = 1;
    w.softmax_scale = softmax_scale;
    w.units = units;
    w.out = out;
    return run_units(&w, n_units, nthreads);
}
