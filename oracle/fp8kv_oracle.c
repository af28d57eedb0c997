/*
 * fp8kv_oracle.c -- plain, slow CPU oracle for the fp8 e4m3 KV cache path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference leg may load this library.  It shares no code,
 * header, table or constant generator with the CUDA library; the two meet
 * only through the seeded input generators.
 *
 * Sources (web pages, cited by title and section):
 *   [PR]  vLLM pull request 54705, "fp8 e4m3 KV cache for Inkling on SM100":
 *         section "Purpose" (gate, query quantization, quant-on-store,
 *         descale handling, cache plumbing), "Accuracy", "Evidence document"
 *         (Tier 0, Tier 2 table), "Scale calibration" and the calibration
 *         paragraph of the evidence document (rule max(1, max|x|*1.3/448)).
 *   [CAL] model card "Qwen3.8-27B-FP8-KVcal": section "What it fixes"
 *         (scale table: amax/448, prob_scale 1/448) and section
 *         "Rebuild / reproduce" (ceil_to_bfloat16(amax/448)).
 *   [OCP] OCP 8-bit floating point specification, E4M3 format (bias 7,
 *         no infinities, S.1111.111 is NaN, max normal 448) -- the format the
 *         pages call "e4m3" with its 448 ceiling.
 *
 * Everything here is the plain definition: no blocking, no fusion, float64
 * attention.  Readings of points the pages leave open are marked READING.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define OR_E4M3_MAX 448.0

/* ------------------------------------------------------------------ */
/* E4M3 codec                                                          */
/* ------------------------------------------------------------------ */

/* Exact value of an E4M3 byte [OCP]: sign, 4 exponent bits (bias 7),
 * 3 mantissa bits; exponent field 0 is subnormal m * 2^-9; S.1111.111 is NaN;
 * there are no infinities. */
double or_e4m3_decode(uint8_t b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);               /* subnormal: m/8 * 2^(1-7) */
    else
        mag = ldexp((double)(8 + m), e - 10);     /* (1 + m/8) * 2^(e-7)      */
    return sign ? -mag : mag;
}

/* Round an fp32 value to E4M3, nearest with ties to the even code, with
 * saturation to +-448 [PR "Purpose", quant-on-store: values are clamped to
 * the e4m3 finite range].
 * READING: NaN keeps its sign and becomes the NaN code; +-Inf saturates to
 * +-448 (a saturating conversion); -0.0 keeps its sign (0x80).
 * The search runs over the 127 non-negative codes 0x00..0x7E, whose values
 * increase with the code: find the largest code not above |x|, then pick the
 * nearer of it and the next code, a tie going to the even code. */
uint8_t or_e4m3_encode(float x)
{
    uint8_t s;
    double a;
    int lo, hi, c;
    if (isnan(x))
        return signbit(x) ? 0xFF : 0x7F;
    s = signbit(x) ? 0x80 : 0x00;
    a = fabs((double)x);
    if (a >= OR_E4M3_MAX)
        return (uint8_t)(s | 0x7E);
    lo = 0;
    hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (or_e4m3_decode((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    c = lo;
    if (c < 0x7E) {
        double below = a - or_e4m3_decode((uint8_t)c);
        double above = or_e4m3_decode((uint8_t)(c + 1)) - a;
        if (above < below || (above == below && ((c + 1) & 1) == 0))
            c = c + 1;
    }
    return (uint8_t)(s | c);
}

/* bf16 bit pattern -> float (exact: bf16 is the top half of fp32). */
static float bf16_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

double or_bf16_to_double(uint16_t bits) { return (double)bf16_to_float(bits); }

/* Quantize one bf16 element on store [PR "Purpose", quant-on-store]:
 * divide by the per-tensor scale in fp32, clamp to +-448, convert to e4m3.
 * READING: the division is the IEEE fp32 quotient x/s (correctly rounded).
 * (float)((double)x/(double)s) is that quotient: double carries more than
 * 2*24+2 significand bits, so rounding twice gives the single rounding. */
uint8_t or_quantize(uint16_t x_bf16, float scale)
{
    float x = bf16_to_float(x_bf16);
    float q = (float)((double)x / (double)scale);
    return or_e4m3_encode(q);
}

/* Elementwise quantize of n bf16 values (query rows, or one sequence's keys
 * and values in token order). */
void or_quantize_array(const uint16_t *x, int64_t n, float scale, uint8_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_quantize(x[i], scale);
}

void or_decode_array(const uint8_t *x, int64_t n, double *out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_e4m3_decode(x[i]);
}

/* Store into the paged cache [PR "Purpose", quant-on-store and cache
 * plumbing: caches are byte arrays, written at each token's slot].
 * READING: each cache is uint8[num_blocks][num_kv_heads][block_size][head_dim]
 * (the pages fix no layout; head-major blocks keep one head's block rows
 * contiguous); token t goes to block slot/block_size, row slot%block_size of
 * every head; a negative slot means the token is not stored.
 * k, v: bf16 [num_tokens] rows of num_kv_heads*head_dim, rows k_stride /
 * v_stride elements apart.  Returns 0, or -1 when a slot is out of range. */
int or_kv_store(uint8_t *cache_k, uint8_t *cache_v, int64_t num_blocks,
                int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                const uint16_t *k, const uint16_t *v, int64_t k_stride,
                int64_t v_stride, const int64_t *slot_mapping,
                int64_t num_tokens, float k_scale, float v_scale)
{
    int64_t t;
    int32_t h, d;
    for (t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t], blk, off;
        if (slot < 0)
            continue;
        blk = slot / block_size;
        off = slot % block_size;
        if (blk >= num_blocks)
            return -1;
        for (h = 0; h < num_kv_heads; ++h) {
            int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
            int64_t src = (int64_t)h * head_dim;
            for (d = 0; d < head_dim; ++d) {
                cache_k[dst + d] = or_quantize(k[t * k_stride + src + d], k_scale);
                cache_v[dst + d] = or_quantize(v[t * v_stride + src + d], v_scale);
            }
        }
    }
    return 0;
}

/* Running absolute maximum over the stored tokens [CAL "What it fixes":
 * amax measured at the cache-write point; PR "Evidence document", Tier 2:
 * gather exactly the values stored at each call's slot mapping].
 * slot_mapping may be NULL (all tokens count); tokens with slot < 0 are
 * skipped.  READING: NaN elements do not take part in the maximum.
 * Returns max(amax_in, max |x|). */
float or_amax(const uint16_t *x, int64_t tok_stride, const int64_t *slot_mapping,
              int64_t num_tokens, int32_t num_heads, int32_t head_dim, float amax_in)
{
    int64_t t, i, row = (int64_t)num_heads * head_dim;
    float m = amax_in;
    for (t = 0; t < num_tokens; ++t) {
        if (slot_mapping && slot_mapping[t] < 0)
            continue;
        for (i = 0; i < row; ++i) {
            float a = fabsf(bf16_to_float(x[t * tok_stride + i]));
            if (a > m)
                m = a;
        }
    }
    return m;
}

/* Band counters of quantizing the stored values at one scale [PR "Evidence
 * document", Tier 2: exact e4m3 band counters at scale 1.0 and 3.0 over
 * exactly the values stored at each call's slot mapping, giving the clip
 * rate, the flush-to-zero rate and the round-trip error of its table].
 * READING: an element is counted when it is finite; it is clipped when its
 * quotient |x/s| is above 448 (e4m3 saturates it); it is flushed when it is
 * not zero but its code is +-0 (it lies below the smallest e4m3 magnitude
 * after rounding); its round-trip error is |s*dec(enc(x/s)) - x| / |x|, over
 * the non-zero elements, clipped and flushed ones included.  The quotient
 * and the code are those of or_quantize.
 * Adds into counts[0..3] = (finite, non-zero, clipped, flushed) and into
 * *err_sum. */
void or_band_counts(const uint16_t *x, int64_t tok_stride, const int64_t *slot_mapping,
                    int64_t num_tokens, int32_t row, float scale, int64_t *counts,
                    double *err_sum)
{
    int64_t t, i;
    for (t = 0; t < num_tokens; ++t) {
        if (slot_mapping && slot_mapping[t] < 0)
            continue;
        for (i = 0; i < row; ++i) {
            uint16_t bits = x[t * tok_stride + i];
            float xf = bf16_to_float(bits);
            float q;
            uint8_t c;
            double back;
            if (!isfinite(xf))
                continue;
            counts[0] += 1;
            if (xf == 0.0f)
                continue;
            counts[1] += 1;
            q = (float)((double)xf / (double)scale);
            if (fabsf(q) > 448.0f)
                counts[2] += 1;
            c = or_e4m3_encode(q);
            if ((c & 0x7F) == 0)
                counts[3] += 1;
            back = or_e4m3_decode(c) * (double)scale;
            *err_sum += fabs(back - (double)xf) / fabs((double)xf);
        }
    }
}

/* Scale from a measured amax.
 *  rule 0: amax/448                 [CAL "What it fixes", scale table]
 *  rule 1: ceil_to_bfloat16(amax/448), kept as fp32
 *                                   [CAL "Rebuild / reproduce"]
 *  rule 2: max(1, amax*1.3/448)     [PR calibration paragraph, safety rule]
 * Scales must be finite and positive [PR "Purpose", unity-scale warning
 * bullet: loaded scales are validated finite and positive]; returns 0 on
 * success and -1 when the result would not be (e.g. amax = 0). */
int or_scale_from_amax(float amax, int rule, float *scale)
{
    float s;
    if (!(amax >= 0.0f) || isinf(amax))
        return -1;
    if (rule == 0) {
        s = (float)((double)amax / OR_E4M3_MAX);
    } else if (rule == 1) {
        float q = (float)((double)amax / OR_E4M3_MAX);
        uint32_t u;
        memcpy(&u, &q, sizeof u);
        if (u & 0xFFFFu)
            u = (u & 0xFFFF0000u) + 0x10000u;   /* smallest bf16 >= q (q > 0) */
        memcpy(&s, &u, sizeof s);
    } else if (rule == 2) {
        double r = (double)amax * 1.3 / OR_E4M3_MAX;
        s = (float)(r > 1.0 ? r : 1.0);
    } else {
        return -1;
    }
    if (!(s > 0.0f) || isinf(s))
        return -1;
    *scale = s;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Attention over the e4m3 cache                                       */
/* ------------------------------------------------------------------ */

/* One query row, float64 [PR "Purpose", descale handling: scores are
 * descaled (softmax_scale * q_scale * k_scale) before the exact bf16 relative
 * bias is added; the output is multiplied by v_scale].
 *
 * q8:     e4m3 query row, head_dim bytes (the query after quantization).
 * k8, v8: e4m3 keys / values of this sequence and KV head in token order:
 *         key j's row starts at k8 + j*ld.
 * len_k:  keys in the sequence; pos_q: the query's position (0-based).
 * bias:   NULL, or the bf16 relative-bias vector of this query token and
 *         head, indexed by distance d = pos_q - j, d in [0, rel_extent).
 * window: 0 = full causal; else key j is visible iff pos_q - j < window.
 * form 4: z_j = (sigma*s_q*s_k) * sum_d q8_d k8_jd + bias, o = s_v * P.v8
 *         (the fold of the descales into the softmax scale and output);
 * form 5: explicit dequantize-then-attend: qh = s_q q8, kh = s_k k8,
 *         vh = s_v v8, z_j = sigma * qh.kh_j + bias, o = P.vh.
 * READINGS: causal visibility is j <= pos_q; the bias is zero outside
 * [0, rel_extent) and is not multiplied by sigma; a row with no visible key
 * returns zeros.  out: head_dim doubles. */
void or_attend_row(int32_t head_dim, const uint8_t *q8, const uint8_t *k8,
                   const uint8_t *v8, int64_t ld, int64_t len_k, int64_t pos_q,
                   double sigma, double s_q, double s_k, double s_v,
                   const uint16_t *bias, int32_t rel_extent, int32_t window,
                   int form, double *out)
{
    int64_t j, lo = 0, hi, n;
    int32_t d;
    double *z, zmax = -INFINITY, wsum = 0.0;
    double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);

    for (d = 0; d < head_dim; ++d) {
        out[d] = 0.0;
        qd[d] = or_e4m3_decode(q8[d]);
    }
    hi = pos_q + 1 < len_k ? pos_q + 1 : len_k;   /* causal: j <= pos_q */
    if (window > 0 && pos_q - window + 1 > lo)
        lo = pos_q - window + 1;                  /* pos_q - j < window */
    n = hi - lo;
    if (n <= 0) {
        free(qd);
        return;
    }
    z = (double *)malloc(sizeof(double) * (size_t)n);
    for (j = lo; j < hi; ++j) {
        const uint8_t *kr = k8 + j * ld;
        double dot = 0.0, zj;
        int64_t dist = pos_q - j;
        if (form == 5) {
            for (d = 0; d < head_dim; ++d)
                dot += (s_q * qd[d]) * (s_k * or_e4m3_decode(kr[d]));
            zj = sigma * dot;
        } else {
            for (d = 0; d < head_dim; ++d)
                dot += qd[d] * or_e4m3_decode(kr[d]);
            zj = (sigma * s_q * s_k) * dot;
        }
        if (bias && dist >= 0 && dist < rel_extent)
            zj += or_bf16_to_double(bias[dist]);
        z[j - lo] = zj;
        if (zj > zmax)
            zmax = zj;
    }
    for (j = 0; j < n; ++j) {
        z[j] = exp(z[j] - zmax);
        wsum += z[j];
    }
    for (j = lo; j < hi; ++j) {
        const uint8_t *vr = v8 + j * ld;
        double w = z[j - lo] / wsum;
        if (form == 5) {
            for (d = 0; d < head_dim; ++d)
                out[d] += w * (s_v * or_e4m3_decode(vr[d]));
        } else {
            for (d = 0; d < head_dim; ++d)
                out[d] += w * or_e4m3_decode(vr[d]);
        }
    }
    if (form != 5)
        for (d = 0; d < head_dim; ++d)
            out[d] *= s_v;
    free(z);
    free(qd);
}

/* ------------------------------------------------------------------ */
/* Per-token scales                                                    */
/* ------------------------------------------------------------------ */

/* Per-token dynamic scale [local-inference-lab/vllm PR 189, per-token scale:
 * each cached token carries its own scale beside its codes, so no calibrated
 * per-tensor scale is needed].
 * READING: one scale per token and KV head (one row of head_dim values):
 * s = max |x| / 448 over the row's finite elements (NaN and +-Inf do not take
 * part), as the correctly rounded fp32 quotient, and s = 1 for a row whose
 * finite elements are all zero; each element is then quantized with
 * or_quantize at that scale. */
float or_row_scale(const uint16_t *x, int32_t n)
{
    int32_t i;
    float m = 0.0f;
    for (i = 0; i < n; ++i) {
        float a = fabsf(bf16_to_float(x[i]));
        if (isfinite(a) && a > m)
            m = a;
    }
    return m > 0.0f ? (float)((double)m / (double)OR_E4M3_MAX) : 1.0f;
}

/* n_rows rows of row_len bf16 values -> codes (same shape) and one scale per
 * row. */
void or_quantize_per_token(const uint16_t *x, int64_t n_rows, int32_t row_len, uint8_t *codes,
                           float *scales)
{
    int64_t r;
    int32_t i;
    for (r = 0; r < n_rows; ++r) {
        float s = or_row_scale(x + r * row_len, row_len);
        scales[r] = s;
        for (i = 0; i < row_len; ++i)
            codes[r * row_len + i] = or_quantize(x[r * row_len + i], s);
    }
}

/* One query row over keys with per-token scales: key j is k_j = sk[j] *
 * dec(k8_j) and v_j = sv[j] * dec(v8_j) (dequantize-then-attend); z_j =
 * sigma * (s_q q8) . k_j + bias, o = softmax(z) . v.  Visibility, bias and
 * the empty row as in or_attend_row. */
void or_attend_row_pt(int32_t head_dim, const uint8_t *q8, const uint8_t *k8,
                      const uint8_t *v8, int64_t ld, const float *sk, const float *sv,
                      int64_t len_k, int64_t pos_q, double sigma, double s_q,
                      const uint16_t *bias, int32_t rel_extent, int32_t window, double *out)
{
    int64_t j, lo = 0, hi, n;
    int32_t d;
    double *z, zmax = -INFINITY, wsum = 0.0;
    for (d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    hi = pos_q + 1 < len_k ? pos_q + 1 : len_k;
    if (window > 0 && pos_q - window + 1 > lo)
        lo = pos_q - window + 1;
    n = hi - lo;
    if (n <= 0)
        return;
    z = (double *)malloc(sizeof(double) * (size_t)n);
    for (j = lo; j < hi; ++j) {
        const uint8_t *kr = k8 + j * ld;
        double dot = 0.0, zj;
        int64_t dist = pos_q - j;
        for (d = 0; d < head_dim; ++d)
            dot += (s_q * or_e4m3_decode(q8[d])) * ((double)sk[j] * or_e4m3_decode(kr[d]));
        zj = sigma * dot;
        if (bias && dist >= 0 && dist < rel_extent)
            zj += or_bf16_to_double(bias[dist]);
        z[j - lo] = zj;
        if (zj > zmax)
            zmax = zj;
    }
    for (j = 0; j < n; ++j) {
        z[j] = exp(z[j] - zmax);
        wsum += z[j];
    }
    for (j = lo; j < hi; ++j) {
        const uint8_t *vr = v8 + j * ld;
        double w = z[j - lo] / wsum;
        for (d = 0; d < head_dim; ++d)
            out[d] += w * ((double)sv[j] * or_e4m3_decode(vr[d]));
    }
    free(z);
}

/* Many rows, one per (sequence, query, head) the caller lists.  Row r reads
 * q8 + q_off[r], k8 + kv_off[r], v8 + kv_off[r] (rows ld apart), bias +
 * bias_off[r] (bias_off < 0: no bias), and writes head_dim doubles at
 * out + r*head_dim.  Rows are independent; OpenMP spreads them over the host
 * cores when the library is built with it. */
void or_attend_rows(int64_t n_rows, int32_t head_dim, const uint8_t *q8,
                    const int64_t *q_off, const uint8_t *k8, const uint8_t *v8,
                    const int64_t *kv_off, int64_t ld, const int64_t *len_k,
                    const int64_t *pos_q, double sigma, double s_q, double s_k,
                    double s_v, const uint16_t *bias, const int64_t *bias_off,
                    int32_t rel_extent, int32_t window, int form, double *out)
{
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < n_rows; ++r) {
        const uint16_t *b = (bias && bias_off[r] >= 0) ? bias + bias_off[r] : NULL;
        or_attend_row(head_dim, q8 + q_off[r], k8 + kv_off[r], v8 + kv_off[r], ld,
                      len_k[r], pos_q[r], sigma, s_q, s_k, s_v, b, rel_extent,
                      window, form, out + r * head_dim);
    }
}

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
