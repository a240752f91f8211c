/*
 * kvc_oracle.c - plain, slow, CPU reference for the decode-attention KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library under kv_cache_decode_flash_gb300/) never calls it, and
 * the two share no source, header, table or helper.
 *
 * Everything here is written from the definitions, in double precision
 * unless a definition fixes single precision:
 *
 *   - fp16 (IEEE-754 binary16) encode/decode, round to nearest even, with
 *     subnormals and overflow to infinity.
 *   - q4_0 block quantisation (V): 32 4-bit codes plus one fp16 scale per
 *     block, a reading stated at orc_q4_0_quantize_block.
 *   - q8_0 block quantisation: 32 int8 codes plus one fp16 scale per block.
 *     The pages only name the type ("-ctk q8_0", F5 - Advanced KV Cache
 *     Techniques, section M6 - PolyKV; "q8_0 K/V", sched: pipeline the
 *     delivery of a host-resident KV cache (R4), section Measurements).
 *     The reading used: d = max|x| / 127 and q = round(x * (1/d)), rounded
 *     half away from zero, all in fp32, the scale stored as fp16(d).  The
 *     step order is fixed because codes must match bit for bit.
 *   - single-query attention softmax(s) V with s = kq_scale * q.k over the
 *     dequantised cache, grouped-query heads in contiguous groups
 *     (F5 - Advanced KV Cache Techniques, section M2/M3: the GQA-clamped
 *     gpu_heads * gqa_ratio head split).
 *   - RoPE re-rotation of a stored key by a position delta
 *     (Plan: lossless long context - derived hot/cold sizing + host-RAM KV
 *     cold store, section OpenVINO - KV-byte offload: shifted imports
 *     rotate RoPE-positioned keys by the destination/source delta).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 * (no FMA contraction: the fp32 quantiser is a fixed op sequence).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_QK 32 /* elements per q8_0 block */

/* ------------------------------------------------------------------ */
/* fp16 from the IEEE-754 binary16 definition                          */
/* ------------------------------------------------------------------ */

/* Decode: sign * 2^(e-15) * (1 + m/1024) for 1 <= e <= 30,
 *         sign * 2^-14 * (m/1024) for e == 0, inf/nan for e == 31. */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return sign ? -v : v;
}

/* Round half to even of a non-negative double that is exactly known. */
static double orc_round_half_even(double a) {
    double n = floor(a);
    double f = a - n; /* exact: a and n share the binade or n is smaller */
    if (f > 0.5) return n + 1.0;
    if (f < 0.5) return n;
    return (fmod(n, 2.0) == 0.0) ? n : n + 1.0;
}

/* Encode any double as the nearest binary16, ties to even. */
uint16_t orc_f64_to_f16(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2); /* a in [2^(e2-1), 2^e2) */
    int e = e2 - 1;      /* a = 1.f * 2^e */
    if (e < -14) {
        /* subnormal range: quantum 2^-24 */
        double n = orc_round_half_even(ldexp(a, 24));
        /* n == 1024 rolls over to the smallest normal, which has the same bits */
        return (uint16_t)(sign | (uint16_t)n);
    }
    double n = orc_round_half_even(ldexp(a, 10 - e)); /* in [1024, 2048] */
    if (n >= 2048.0) {
        n = 1024.0;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(n - 1024.0));
}

uint16_t orc_f32_to_f16(float x) { return orc_f64_to_f16((double)x); }

void orc_f32_to_f16_array(const float *x, uint16_t *h, int64_t n) {
    for (int64_t i = 0; i < n; ++i) h[i] = orc_f32_to_f16(x[i]);
}

void orc_f16_to_f64_array(const uint16_t *h, double *x, int64_t n) {
    for (int64_t i = 0; i < n; ++i) x[i] = orc_f16_to_f64(h[i]);
}

/* ------------------------------------------------------------------ */
/* q8_0                                                                */
/* ------------------------------------------------------------------ */

/* One block of 32 fp32 values -> 32 codes + fp16 scale bits.
 * fp32 steps, in this order: a = max |x_i|; d = a / 127; id = 1/d (0 if
 * d == 0); q_i = roundf(x_i * id) (half away from zero); scale = fp16(d). */
void orc_q8_0_quantize_block(const float *x, int8_t *q, uint16_t *scale) {
    float a = 0.0f;
    for (int i = 0; i < ORC_QK; ++i) {
        float ax = fabsf(x[i]);
        if (ax > a) a = ax;
    }
    volatile float d = a / 127.0f;
    volatile float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int i = 0; i < ORC_QK; ++i) {
        volatile float v = x[i] * id;
        q[i] = (int8_t)roundf(v);
    }
    *scale = orc_f32_to_f16(d);
}

/* n values (n a multiple of 32) -> n codes and n/32 scales. */
void orc_q8_0_quantize_row(const float *x, int64_t n, int8_t *q, uint16_t *scale) {
    for (int64_t b = 0; b < n / ORC_QK; ++b)
        orc_q8_0_quantize_block(x + b * ORC_QK, q + b * ORC_QK, scale + b);
}

/* Dequantised value of one element: fp16(d) * q, exact in double. */
double orc_q8_0_value(int8_t q, uint16_t scale) { return orc_f16_to_f64(scale) * (double)q; }

void orc_q8_0_dequantize_row(const int8_t *q, const uint16_t *scale, int64_t n, double *x) {
    for (int64_t i = 0; i < n; ++i) x[i] = orc_q8_0_value(q[i], scale[i / ORC_QK]);
}

/* ------------------------------------------------------------------ */
/* q4_0 (V only)                                                       */
/* ------------------------------------------------------------------ */

/* The pages name "-ctv q4_0" (F5 - Advanced KV Cache Techniques, section
 * M6 - PolyKV: asymmetric K/V compression) but do not define it.  The
 * reading used, the plainest 4-bit counterpart of q8_0 with one fp16 scale
 * per block of 32:
 *   m = the element of largest magnitude, sign kept (the first one on ties);
 *   d = m / -8; id = 1/d (0 if d == 0); code_i = min(15, trunc(x_i * id + 8.5))
 *   with the product and the sum each rounded to fp32; scale = fp16(d).
 *   Value of a code: (code - 8) * fp16(d)  (m itself maps to code 0).
 *   Packing: byte j (0..15) of a block holds code j in its low four bits
 *   and code j + 16 in its high four bits. */
void orc_q4_0_quantize_block(const float *x, uint8_t *packed, uint16_t *scale) {
    float amax = 0.0f, m = 0.0f;
    for (int i = 0; i < ORC_QK; ++i) {
        float ax = fabsf(x[i]);
        if (ax > amax) {
            amax = ax;
            m = x[i];
        }
    }
    volatile float d = m / -8.0f;
    volatile float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    int code[ORC_QK];
    for (int i = 0; i < ORC_QK; ++i) {
        volatile float t = x[i] * id;
        volatile float u = t + 8.5f;
        int c = (int)u; /* u > 0: truncation is the floor */
        code[i] = c > 15 ? 15 : c;
    }
    for (int j = 0; j < ORC_QK / 2; ++j) packed[j] = (uint8_t)(code[j] | (code[j + ORC_QK / 2] << 4));
    *scale = orc_f32_to_f16(d);
}

/* n values (n a multiple of 32) -> n/2 packed bytes and n/32 scales. */
void orc_q4_0_quantize_row(const float *x, int64_t n, uint8_t *packed, uint16_t *scale) {
    for (int64_t b = 0; b < n / ORC_QK; ++b)
        orc_q4_0_quantize_block(x + b * ORC_QK, packed + b * (ORC_QK / 2), scale + b);
}

/* Code of element i of a row of packed blocks. */
static int orc_q4_0_code(const uint8_t *packed, int64_t i) {
    const uint8_t *blk = packed + (i / ORC_QK) * (ORC_QK / 2);
    int k = (int)(i % ORC_QK);
    return k < ORC_QK / 2 ? (blk[k] & 15) : (blk[k - ORC_QK / 2] >> 4);
}

/* Dequantised values of n elements: (code - 8) * fp16(d), exact in double. */
void orc_q4_0_dequantize_row(const uint8_t *packed, const uint16_t *scale, int64_t n, double *x) {
    for (int64_t i = 0; i < n; ++i) x[i] = (double)(orc_q4_0_code(packed, i) - 8) * orc_f16_to_f64(scale[i / ORC_QK]);
}

/* ------------------------------------------------------------------ */
/* Attention                                                           */
/* ------------------------------------------------------------------ */

/* KV storage description used by the attention and rope routines.
 * type 8 = q8_0: codes int8 [n][Hk][D], scales fp16 bits [n][Hk][D/32].
 * type 2 = q4_0: packed bytes [n][Hk][D/2], scales fp16 bits [n][Hk][D/32].
 * type 1 = f16 : values fp16 bits [n][Hk][D] (codes pointer), scales NULL. */
typedef struct {
    int type;
    const void *data;       /* int8 codes (q8_0) or uint16 halves (f16) */
    const uint16_t *scales; /* q8_0 only */
} orc_kv;

/* Dequantise the head-row (token j, kv head g) of a cache tensor into out[D]. */
static void orc_load_row(const orc_kv *t, int64_t j, int g, int Hk, int D, double *out) {
    int64_t base = (j * Hk + g) * (int64_t)D;
    if (t->type == 8) {
        const int8_t *c = (const int8_t *)t->data + base;
        const uint16_t *s = t->scales + (j * Hk + g) * (int64_t)(D / ORC_QK);
        for (int i = 0; i < D; ++i) out[i] = orc_f16_to_f64(s[i / ORC_QK]) * (double)c[i];
    } else if (t->type == 2) {
        const uint8_t *c = (const uint8_t *)t->data + (j * Hk + g) * (int64_t)(D / 2);
        const uint16_t *s = t->scales + (j * Hk + g) * (int64_t)(D / ORC_QK);
        orc_q4_0_dequantize_row(c, s, D, out);
    } else {
        const uint16_t *h = (const uint16_t *)t->data + base;
        for (int i = 0; i < D; ++i) out[i] = orc_f16_to_f64(h[i]);
    }
}

/* Single-query attention over n rows for the query heads [h0, h1).
 * q: fp32 [H][D]; out: double [H][D] (only rows h0..h1-1 written).
 * Query head h reads kv head g = h / (H/Hk) (contiguous groups).
 * s_j = kq_scale * sum_i q[h][i] * k[j][g][i]; p = softmax(s) (two-pass,
 * max-subtracted, fp64); o = sum_j p_j v[j][g].  n == 0 gives o = 0. */
int orc_attn(const float *q, int H, int Hk, int D, int64_t n, int type_k, const void *k,
             const uint16_t *ks, int type_v, const void *v, const uint16_t *vs, double kq_scale,
             int h0, int h1, double *out) {
    if (H % Hk) return -1;
    int r = H / Hk;
    orc_kv K = {type_k, k, ks}, V = {type_v, v, vs};
    double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *row = (double *)malloc(sizeof(double) * (size_t)D);
    if (!s || !row) {
        free(s);
        free(row);
        return -2;
    }
    for (int h = h0; h < h1; ++h) {
        int g = h / r;
        double *o = out + (int64_t)h * D;
        for (int i = 0; i < D; ++i) o[i] = 0.0;
        if (n == 0) continue;
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            orc_load_row(&K, j, g, Hk, D, row);
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += (double)q[(int64_t)h * D + i] * row[i];
            s[j] = kq_scale * acc;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        for (int64_t j = 0; j < n; ++j) {
            orc_load_row(&V, j, g, Hk, D, row);
            double p = s[j] / l;
            for (int i = 0; i < D; ++i) o[i] += p * row[i];
        }
    }
    free(s);
    free(row);
    return 0;
}

/* A second, deliberately different formulation for tiny inputs: per token,
 * in long double, no max subtraction:  o = sum_j e^{s_j} v_j / sum_j e^{s_j}. */
int orc_attn_bruteforce(const float *q, int H, int Hk, int D, int64_t n, int type_k,
                        const void *k, const uint16_t *ks, int type_v, const void *v,
                        const uint16_t *vs, double kq_scale, double *out) {
    if (H % Hk) return -1;
    int r = H / Hk;
    orc_kv K = {type_k, k, ks}, V = {type_v, v, vs};
    double *kr = (double *)malloc(sizeof(double) * (size_t)D);
    double *vr = (double *)malloc(sizeof(double) * (size_t)D);
    long double *num = (long double *)malloc(sizeof(long double) * (size_t)D);
    if (!kr || !vr || !num) {
        free(kr);
        free(vr);
        free(num);
        return -2;
    }
    for (int h = 0; h < H; ++h) {
        int g = h / r;
        long double den = 0.0L;
        for (int i = 0; i < D; ++i) num[i] = 0.0L;
        for (int64_t j = 0; j < n; ++j) {
            orc_load_row(&K, j, g, Hk, D, kr);
            orc_load_row(&V, j, g, Hk, D, vr);
            long double dot = 0.0L;
            for (int i = 0; i < D; ++i) dot += (long double)q[(int64_t)h * D + i] * (long double)kr[i];
            long double w = expl((long double)kq_scale * dot);
            den += w;
            for (int i = 0; i < D; ++i) num[i] += w * (long double)vr[i];
        }
        for (int i = 0; i < D; ++i) out[(int64_t)h * D + i] = n ? (double)(num[i] / den) : 0.0;
    }
    free(kr);
    free(vr);
    free(num);
    return 0;
}

/* ------------------------------------------------------------------ */
/* RoPE shift                                                          */
/* ------------------------------------------------------------------ */

/* Rotate one head-row in place by the angle delta * theta_i per rotary pair,
 * theta_i = base^(-2i/D), i in [0, D/2).  mode 0 (NEOX): pair (i, i + D/2);
 * mode 1 (NORM): pair (2i, 2i+1).  (a, b) -> (a cos - b sin, a sin + b cos). */
void orc_rope_rotate(double *x, int D, int mode, double base, int64_t delta) {
    for (int i = 0; i < D / 2; ++i) {
        double theta = pow(base, -2.0 * (double)i / (double)D);
        double phi = (double)delta * theta;
        int ia = mode == 0 ? i : 2 * i;
        int ib = mode == 0 ? i + D / 2 : 2 * i + 1;
        double a = x[ia], b = x[ib];
        double c = cos(phi), s = sin(phi);
        x[ia] = a * c - b * s;
        x[ib] = a * s + b * c;
    }
}

/* Shift n stored q8_0 head-rows (each D codes + D/32 scales, rows contiguous)
 * by delta: dequantise exactly, rotate in fp64, round each value to fp32,
 * requantise every block with the quantiser above. */
int orc_rope_shift_q8_0(int8_t *codes, uint16_t *scales, int64_t n_rows, int D, int mode,
                        double base, int64_t delta) {
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    float *xf = (float *)malloc(sizeof(float) * (size_t)D);
    if (!x || !xf) {
        free(x);
        free(xf);
        return -2;
    }
    for (int64_t j = 0; j < n_rows; ++j) {
        int8_t *c = codes + j * D;
        uint16_t *s = scales + j * (D / ORC_QK);
        orc_q8_0_dequantize_row(c, s, D, x);
        orc_rope_rotate(x, D, mode, base, delta);
        for (int i = 0; i < D; ++i) xf[i] = (float)x[i];
        orc_q8_0_quantize_row(xf, D, c, s);
    }
    free(x);
    free(xf);
    return 0;
}

/* Shift n stored f16 head-rows by delta: decode, rotate in fp64, re-encode
 * with a single round to nearest even. */
int orc_rope_shift_f16(uint16_t *h, int64_t n_rows, int D, int mode, double base, int64_t delta) {
    double *x = (double *)malloc(sizeof(double) * (size_t)D);
    if (!x) return -2;
    for (int64_t j = 0; j < n_rows; ++j) {
        uint16_t *r = h + j * D;
        for (int i = 0; i < D; ++i) x[i] = orc_f16_to_f64(r[i]);
        orc_rope_rotate(x, D, mode, base, delta);
        for (int i = 0; i < D; ++i) r[i] = orc_f64_to_f16(x[i]);
    }
    free(x);
    return 0;
}

/* ------------------------------------------------------------------ */
/* KeyDiff distinctiveness ("F5 - Advanced KV Cache Techniques", M1:   */
/* retention-aware context shift)                                     */
/* ------------------------------------------------------------------ */

/* Cosine of two D-vectors; 0 when either norm is 0 (a reading: the page
 * does not define the degenerate case). */
static double orc_cos(const double *a, const double *b, int D) {
    double ab = 0.0, aa = 0.0, bb = 0.0;
    for (int i = 0; i < D; ++i) {
        ab += a[i] * b[i];
        aa += a[i] * a[i];
        bb += b[i] * b[i];
    }
    if (aa == 0.0 || bb == 0.0) return 0.0;
    return ab / (sqrt(aa) * sqrt(bb));
}

/* Per-row KeyDiff score of n rows of one layer's K, in the order given:
 * mean_g = (1/n) sum_j K[j][g] for every KV head g, and
 * score[j] = (1/Hk) sum_g (1 - cos(K[j][g], mean_g)).
 * K as in orc_kv (q8_0 dequantised exactly, f16 decoded). */
int orc_keydiff_scores(int type_k, const void *k, const uint16_t *ks, int64_t n, int Hk, int D, double *score) {
    if (n <= 0) return 0;
    orc_kv t = {type_k, k, ks};
    double *mean = (double *)calloc((size_t)Hk * D, sizeof(double));
    double *row = (double *)malloc((size_t)D * sizeof(double));
    if (!mean || !row) {
        free(mean);
        free(row);
        return -1;
    }
    for (int64_t j = 0; j < n; ++j)
        for (int g = 0; g < Hk; ++g) {
            orc_load_row(&t, j, g, Hk, D, row);
            for (int i = 0; i < D; ++i) mean[(int64_t)g * D + i] += row[i];
        }
    for (int64_t i = 0; i < (int64_t)Hk * D; ++i) mean[i] /= (double)n;
    for (int64_t j = 0; j < n; ++j) {
        double s = 0.0;
        for (int g = 0; g < Hk; ++g) {
            orc_load_row(&t, j, g, Hk, D, row);
            s += 1.0 - orc_cos(row, mean + (int64_t)g * D, D);
        }
        score[j] = s / (double)Hk;
    }
    free(mean);
    free(row);
    return 0;
}

/* Start w0 of the width-w window of consecutive entries of score[0..n)
 * lying inside [lo, hi) whose sum is smallest (prefix sums in fp64; the
 * first such window on ties).  -1 when no window fits. */
int64_t orc_min_window(const double *score, int64_t n, int64_t lo, int64_t hi, int64_t w) {
    if (lo < 0) lo = 0;
    if (hi > n) hi = n;
    if (w <= 0 || hi - lo < w) return -1;
    double *pre = (double *)malloc((size_t)(n + 1) * sizeof(double));
    if (!pre) return -1;
    pre[0] = 0.0;
    for (int64_t j = 0; j < n; ++j) pre[j + 1] = pre[j] + score[j];
    int64_t best = lo;
    double best_sum = pre[lo + w] - pre[lo];
    for (int64_t s = lo + 1; s + w <= hi; ++s) {
        const double sum = pre[s + w] - pre[s];
        if (sum < best_sum) {
            best_sum = sum;
            best = s;
        }
    }
    free(pre);
    return best;
}
