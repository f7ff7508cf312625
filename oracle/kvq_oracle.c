/*
 * kvq_oracle.c -- CPU oracle for the quantized KV cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the GPU library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or constant with the CUDA library, and the CUDA library never
 * calls it.
 *
 * What it follows:
 *   - The Q4_G64 codec: 4-bit signed codes, an fp16 scale for each group of 64 values,
 *     4.25 bits per value (den_llama.cpp, "What this fork is", quantized KV
 *     cache bullet; "build3 (working engine) -- additions" table, Q4_G64 row,
 *     whose footnote says the CUDA quantizer is byte-identical to a CPU
 *     reference and the dequantizer bit-identical).  The pages give no rounding
 *     rule; the rule used is scale = fp16(absmax / 7), q = clamp(rne(x / scale),
 *     -8, 7), with the division by the fp16-rounded scale widened to fp32.
 *   - Q4_G32: the "q4_0" V cache of the shipped pair "-ctk q8_0 -ctv q4_0"
 *     (den_llama.cpp, "What's in the fork": the q8_0-q4_0 FlashAttention pair;
 *     "Results": the 65K serve run) is not defined on the pages; it is read as
 *     the Q4_G64 rule and nibble layout with groups of 32 values (4.5 bits per
 *     value).
 *   - NVFP4, the pages' KV type of the matched "-ctk nvfp4 -ctv nvfp4" and
 *     mixed "-ctk q8_0 -ctv nvfp4" runs (den_llama.cpp, "What this fork is",
 *     quantized KV cache bullet; "build3 (working engine) -- additions" table,
 *     NVFP4 KV row; "Build3" command block), whose format the pages do not
 *     give: read as NVIDIA's published NVFP4 -- FP4 E2M1 values in blocks of
 *     16, each block with one FP8 E4M3 scale -- without the per-tensor second
 *     scale (a cache is appended to row by row, so no tensor-wide absmax
 *     exists when a row is written): scale = e4m3(absmax / 6), code =
 *     e2m1(x / (float)scale), both round-to-nearest-even on their format's
 *     grid and held at the largest finite value (448, 6); 4.5 bits per value.
 *   - The q8_0-style K codec of the mixed pair "-ctk q8_0 -ctv q4_g64"
 *     (den_llama.cpp, "Build3 (working engine)" command block): 32 int8 values
 *     with one FP16 scale, scale = fp16(absmax / 127), q = clamp(rne(x/scale),
 *     -127, 127).
 *   - Decode attention over the dequantized cache: plain softmax attention,
 *     one (or 1 + 2 draft) query tokens per sequence, grouped-query heads,
 *     causal among the new query tokens (den_llama.cpp, "What's in the fork",
 *     the fattn-vec-instance-q4_g64 row; the MTP n-max 2 runs in "Results").
 *   - The KV-cache append stage that writes new K/V rows (Llaminar, "Graphs
 *     and Compute Stages": KV-cache append and attention are separate stages).
 *   - Split-then-merge by log-sum-exp, the plain identity
 *     softmax over a union = exp-weighted combination of per-part softmaxes.
 *
 * Floating point: the codec works in fp32 exactly as stated above (IEEE
 * division, round-to-nearest-even); attention works in fp64.  Build with
 * -ffp-contract=off and without -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_Q4 1
#define ORC_Q8 2
#define ORC_Q4_32 3
#define ORC_NVFP4 4

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 <-> binary32, written from the format definition.      */
/* ------------------------------------------------------------------------ */

/* binary32 -> binary16, round to nearest, ties to even.  Subnormal results
 * are produced exactly; magnitudes that round past the largest finite half
 * (65504) become infinity; NaN stays NaN (quiet). */
uint16_t orc_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;

    if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);       /* NaN */
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);      /* >= 65520: rounds to inf */

    if (ax >= 0x38800000u) {                                        /* >= 2^-14: normal half */
        uint32_t e = (ax >> 23) - 127u + 15u;                       /* half biased exponent */
        uint32_t m = ax & 0x7FFFFFu;
        uint32_t h = (e << 10) | (m >> 13);
        uint32_t rem = m & 0x1FFFu;                                 /* 13 dropped bits */
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;  /* carry may step the exponent */
        return (uint16_t)(sign | h);
    }
    if (ax < 0x33000000u) return (uint16_t)sign;                   /* < 2^-25: rounds to zero */

    /* subnormal half: value in units of 2^-24 is m * 2^(e - 126) */
    uint32_t e = ax >> 23;                                          /* biased, 102..112 */
    uint32_t m = (ax & 0x7FFFFFu) | 0x800000u;
    uint32_t shift = 126u - e;                                      /* 14..24 */
    uint32_t h = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (h & 1u))) h += 1u;          /* 1024 becomes the smallest normal */
    return (uint16_t)(sign | h);
}

/* binary16 -> binary32 (exact). */
float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0) v = ldexp((double)m, -24);                          /* zero / subnormal */
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(1024 + m), e - 25);                     /* (1.m) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

void orc_f32_to_f16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}

void orc_f16_to_f32_array(const uint16_t *h, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(h[i]);
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 and FP4 E2M1, written from their format definitions.            */
/* ------------------------------------------------------------------------ */

/* E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
 * holds the subnormals m * 2^-9; no infinities; S.1111.111 is NaN, so the
 * largest finite magnitude is 1.75 * 2^8 = 448. */
float orc_e4m3_to_f32(uint8_t b)
{
    int e = (b >> 3) & 15, m = b & 7;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = (float)m * ldexpf(1.0f, -9);
    else v = (1.0f + (float)m / 8.0f) * ldexpf(1.0f, e - 7);
    return (b & 0x80) ? -v : v;
}

/* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0
 * holds the subnormal m * 0.5.  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
float orc_e2m1_to_f32(uint8_t n)
{
    int e = (n >> 1) & 3, m = n & 1;
    float v = (e == 0) ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * ldexpf(1.0f, e - 1);
    return (n & 8) ? -v : v;
}

/* Nearest of the n_codes non-negative finite values of a small format to |f|:
 * at or past the largest value, the largest (the saturation the formats are
 * used with); otherwise the code whose value is closest (exact: every
 * candidate and |f| are floats below the largest value, their differences
 * are formed in double), ties to the even code (even mantissa). */
static int orc_nearest_code(float a, int n_codes, float (*decode)(uint8_t))
{
    if (a >= decode((uint8_t)(n_codes - 1))) return n_codes - 1;
    int best = 0;
    double bd = fabs((double)a - (double)decode(0));
    for (int c = 1; c < n_codes; ++c) {
        double d = fabs((double)a - (double)decode((uint8_t)c));
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bd = d;
        }
    }
    return best;
}

/* binary32 -> E4M3 / E2M1: round to nearest, ties to even, saturating; the
 * sign bit is the input's (so a negative value that rounds to zero is -0).
 * Finite inputs. */
uint8_t orc_f32_to_e4m3(float f)
{
    int c = orc_nearest_code(fabsf(f), 127, orc_e4m3_to_f32);      /* 0x00 .. 0x7E */
    return (uint8_t)(c | (signbit(f) ? 0x80 : 0));
}

uint8_t orc_f32_to_e2m1(float f)
{
    int c = orc_nearest_code(fabsf(f), 8, orc_e2m1_to_f32);
    return (uint8_t)(c | (signbit(f) ? 8 : 0));
}

void orc_f32_to_e4m3_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(x[i]);
}

void orc_f32_to_e2m1_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e2m1(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Codec                                                                    */
/* ------------------------------------------------------------------------ */

/* Integer 4-bit codecs: Q4_G64 and Q4_G32 (the same rule and nibble layout with 32-value groups). */
static int orc_is4(int codec) { return codec == ORC_Q4 || codec == ORC_Q4_32; }
static int orc_group(int codec) { return codec == ORC_Q4 ? 64 : codec == ORC_NVFP4 ? 16 : 32; }
static int orc_qmax(int codec) { return orc_is4(codec) ? 7 : 127; }
static int orc_qmin(int codec) { return orc_is4(codec) ? -8 : -127; }

/* Bytes of the code plane per row of head_dim values. */
int orc_row_bytes(int codec, int head_dim)
{
    return (orc_is4(codec) || codec == ORC_NVFP4) ? head_dim / 2 : head_dim;
}

int orc_scales_per_row(int codec, int head_dim) { return head_dim / orc_group(codec); }

/* Bytes of one scale: fp16 bit patterns, except NVFP4's E4M3 bytes. */
int orc_scale_bytes(int codec) { return codec == ORC_NVFP4 ? 1 : 2; }

/* Scale of one group: fp16(absmax / qmax), the fp32 quotient rounded once to
 * fp16; a result past the largest finite half is held at 65504. */
static uint16_t orc_group_scale(const float *x, int n, int qmax)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s = amax / (float)qmax;
    uint16_t d = orc_f32_to_f16(s);
    if (d == 0x7C00u) d = 0x7BFFu;
    return d;
}

/* Code of one value: nearest integer to x / d (fp32 IEEE quotient, ties to
 * even), clamped to [qmin, qmax]; zero when the scale is zero. */
static int orc_code(float x, float d, int qmin, int qmax)
{
    if (d == 0.0f) return 0;
    float r = nearbyintf(x / d);
    if (r < (float)qmin) r = (float)qmin;
    if (r > (float)qmax) r = (float)qmax;
    return (int)r;
}

/* NVFP4 block: scale = e4m3(absmax / 6) with the fp32 quotient; codes
 * e2m1(x / (float)scale), all 0 when the scale is 0.  Codes go to c[0..n). */
static uint8_t orc_nvfp4_block(const float *x, int n, uint8_t *c)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    uint8_t sb = orc_f32_to_e4m3(amax / 6.0f);
    float d = orc_e4m3_to_f32(sb);
    for (int i = 0; i < n; ++i) c[i] = (d == 0.0f) ? 0 : orc_f32_to_e2m1(x[i] / d);
    return sb;
}

/* Quantize n_rows rows of head_dim fp32 values.
 * Q4_G64: qs row = head_dim/2 bytes; byte j holds value 2j in its low nibble
 *         and value 2j+1 in its high nibble, each as a 4-bit two's complement
 *         code; scales row = head_dim/64 fp16 bit patterns, group order.
 * Q4_G32: the same with groups of 32 values (head_dim/32 scales).
 * Q8_0:   qs row = head_dim int8 codes; scales row = head_dim/32 fp16.
 * NVFP4:  qs row as Q4_G64 with E2M1 codes; scales row = head_dim/16 E4M3
 *         bytes (scales is a byte array for this codec). */
void orc_quantize(int codec, const float *x, int64_t n_rows, int head_dim,
                  uint8_t *qs, void *scales)
{
    int gs = orc_group(codec), rb = orc_row_bytes(codec, head_dim), ng = head_dim / gs;
    if (codec == ORC_NVFP4) {
        uint8_t *sc = (uint8_t *)scales, c[16];
        for (int64_t r = 0; r < n_rows; ++r)
            for (int g = 0; g < ng; ++g) {
                sc[r * ng + g] = orc_nvfp4_block(x + r * head_dim + g * gs, gs, c);
                for (int i = 0; i < gs; ++i) {
                    int v = g * gs + i;
                    uint8_t *b = qs + r * rb + (v >> 1);
                    if (v & 1) *b = (uint8_t)((*b & 0x0F) | (c[i] << 4));
                    else       *b = (uint8_t)((*b & 0xF0) | c[i]);
                }
            }
        return;
    }
    uint16_t *sc16 = (uint16_t *)scales;
    int qmax = orc_qmax(codec), qmin = orc_qmin(codec);
    for (int64_t r = 0; r < n_rows; ++r) {
        const float *xr = x + r * head_dim;
        uint8_t *qr = qs + r * rb;
        for (int g = 0; g < ng; ++g) {
            const float *xg = xr + g * gs;
            uint16_t dh = orc_group_scale(xg, gs, qmax);
            float d = orc_f16_to_f32(dh);
            sc16[r * ng + g] = dh;
            for (int i = 0; i < gs; ++i) {
                int q = orc_code(xg[i], d, qmin, qmax);
                int v = g * gs + i;
                if (orc_is4(codec)) {
                    uint8_t nib = (uint8_t)(q & 0xF);
                    if (v & 1) qr[v >> 1] = (uint8_t)((qr[v >> 1] & 0x0F) | (nib << 4));
                    else       qr[v >> 1] = (uint8_t)((qr[v >> 1] & 0xF0) | nib);
                } else {
                    qr[v] = (uint8_t)(int8_t)q;
                }
            }
        }
    }
}

/* Code of value v of a row, as a signed integer. */
static int orc_get_code(int codec, const uint8_t *qr, int v)
{
    if (orc_is4(codec)) {
        int nib = (v & 1) ? (qr[v >> 1] >> 4) : (qr[v >> 1] & 0xF);
        return nib >= 8 ? nib - 16 : nib;
    }
    return (int)(int8_t)qr[v];
}

/* Dequantize rows: x_hat = (float)scale * (float)code, exact in fp32 (NVFP4:
 * e4m3 scale times e2m1 value, 4 x 2 significant bits). */
void orc_dequantize(int codec, const uint8_t *qs, const void *scales,
                    int64_t n_rows, int head_dim, float *out)
{
    int gs = orc_group(codec), rb = orc_row_bytes(codec, head_dim), ng = head_dim / gs;
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int v = 0; v < head_dim; ++v) {
            const uint8_t *qr = qs + r * rb;
            if (codec == ORC_NVFP4) {
                float d = orc_e4m3_to_f32(((const uint8_t *)scales)[r * ng + v / gs]);
                uint8_t nib = (v & 1) ? (qr[v >> 1] >> 4) : (qr[v >> 1] & 0xF);
                out[r * head_dim + v] = d * orc_e2m1_to_f32(nib);
            } else {
                float d = orc_f16_to_f32(((const uint16_t *)scales)[r * ng + v / gs]);
                out[r * head_dim + v] = d * (float)orc_get_code(codec, qr, v);
            }
        }
    }
}

/* Quantize-on-append.  src is [n_seq][n_new][n_kv_heads][head_dim] fp32;
 * the cache planes are [n_seq][n_kv_heads][capacity][row].  Token i of
 * sequence s goes to cache position pos0[s] + i.  A sequence whose positions
 * fall outside [0, capacity) is skipped and bit 0 of the return value set. */
int orc_quantize_append(int codec, const float *src, int n_seq, int n_new, int n_kv_heads,
                        int head_dim, int capacity, const int32_t *pos0,
                        uint8_t *qs, void *scales)
{
    int err = 0;
    int rb = orc_row_bytes(codec, head_dim);
    int64_t sb = (int64_t)orc_scales_per_row(codec, head_dim) * orc_scale_bytes(codec);
    for (int s = 0; s < n_seq; ++s) {
        if (pos0[s] < 0 || (int64_t)pos0[s] + n_new > capacity) { err |= 1; continue; }
        for (int i = 0; i < n_new; ++i)
            for (int h = 0; h < n_kv_heads; ++h) {
                const float *x = src + (((int64_t)s * n_new + i) * n_kv_heads + h) * head_dim;
                int64_t row = ((int64_t)s * n_kv_heads + h) * capacity + pos0[s] + i;
                orc_quantize(codec, x, 1, head_dim, qs + row * rb, (uint8_t *)scales + row * sb);
            }
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Attention (fp64)                                                          */
/* ------------------------------------------------------------------------ */

/* Keys visible to query token i of a sequence whose last query token sees
 * kv_len keys: the n_q new tokens are the last n_q cache positions and attend
 * causally to each other. */
static int64_t orc_visible(int32_t kv_len, int n_q, int i)
{
    int64_t n = (int64_t)kv_len - n_q + i + 1;
    return n < 0 ? 0 : n;
}

typedef struct {
    int k_codec, v_codec;
    const uint8_t *k_qs, *v_qs;
    const uint8_t *k_sc, *v_sc;     /* scale planes as bytes (fp16 or E4M3 elements) */
    int n_seq, n_kv_heads, head_dim, capacity;
    const float *q;            /* [n_seq][n_q][n_heads][head_dim] */
    int n_q, n_heads;
    const int32_t *kv_len;     /* [n_seq] */
    double scale;
} orc_attn_args;

/* Softmax attention of the query rows [r_lo, r_hi) of (s, kv head kh) over
 * the tokens [t_lo, t_hi) intersected with each row's visible range.  Writes,
 * for each of those rows r, the output normalised over that range and its
 * log-sum-exp at o + r * stride and lse + r * stride (rows outside the range
 * are not touched); a row with no token in range gets o = 0 and lse = -inf.
 * Query head h uses kv head h / (n_heads / n_kv_heads).  Two passes: scores
 * and their maximum, then exp, sum and the weighted sum of V rows.  Each row's
 * arithmetic depends on that row alone, so any row range gives the same
 * values for its rows. */
static void orc_attend_rows(const orc_attn_args *a, int s, int kh, int64_t t_lo, int64_t t_hi, int r_lo,
                            int r_hi, double *o, double *lse, int64_t o_row_stride_elems, int64_t lse_row_stride)
{
    int D = a->head_dim, G = a->n_heads / a->n_kv_heads, R = a->n_q * G;
    int64_t span = t_hi > t_lo ? t_hi - t_lo : 0;
    double *z = (double *)malloc(sizeof(double) * (size_t)(R * (span > 0 ? span : 1)));
    float *kr = (float *)malloc(sizeof(float) * (size_t)D);
    float *vr = (float *)malloc(sizeof(float) * (size_t)D);
    double *qd = (double *)malloc(sizeof(double) * (size_t)(R * D));
    int64_t *nv = (int64_t *)malloc(sizeof(int64_t) * (size_t)R);
    int krb = orc_row_bytes(a->k_codec, D), vrb = orc_row_bytes(a->v_codec, D);
    int64_t ksb = (int64_t)orc_scales_per_row(a->k_codec, D) * orc_scale_bytes(a->k_codec);
    int64_t vsb = (int64_t)orc_scales_per_row(a->v_codec, D) * orc_scale_bytes(a->v_codec);

    /* row r = i * G + j is query token i, query head kh * G + j */
    for (int i = 0; i < a->n_q; ++i)
        for (int j = 0; j < G; ++j) {
            int r = i * G + j, h = kh * G + j;
            if (r < r_lo || r >= r_hi) continue;
            const float *qv = a->q + (((int64_t)s * a->n_q + i) * a->n_heads + h) * D;
            for (int d = 0; d < D; ++d) qd[r * D + d] = (double)qv[d];
            int64_t vis = orc_visible(a->kv_len[s], a->n_q, i);
            int64_t hi = vis < t_hi ? vis : t_hi;
            nv[r] = hi > t_lo ? hi - t_lo : 0;       /* tokens of the range this row sees */
        }

    int64_t plane = ((int64_t)s * a->n_kv_heads + kh) * a->capacity;
    /* pass 1: scores */
    for (int64_t t = 0; t < span; ++t) {
        int64_t row = plane + t_lo + t;
        orc_dequantize(a->k_codec, a->k_qs + row * krb, a->k_sc + row * ksb, 1, D, kr);
        for (int r = r_lo; r < r_hi; ++r) {
            if (t >= nv[r]) continue;
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[r * D + d] * (double)kr[d];
            z[r * span + t] = acc * a->scale;
        }
    }
    double *m = (double *)malloc(sizeof(double) * (size_t)R);
    double *l = (double *)malloc(sizeof(double) * (size_t)R);
    for (int r = r_lo; r < r_hi; ++r) {
        m[r] = -INFINITY;
        for (int64_t t = 0; t < nv[r]; ++t) if (z[r * span + t] > m[r]) m[r] = z[r * span + t];
        l[r] = 0.0;
        for (int64_t t = 0; t < nv[r]; ++t) {
            z[r * span + t] = exp(z[r * span + t] - m[r]);
            l[r] += z[r * span + t];
        }
        double *orow = o + (int64_t)r * o_row_stride_elems;
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
    }
    /* pass 2: weighted sum of V rows */
    for (int64_t t = 0; t < span; ++t) {
        int64_t row = plane + t_lo + t;
        int need = 0;
        for (int r = r_lo; r < r_hi; ++r) need |= (t < nv[r]);
        if (!need) continue;
        orc_dequantize(a->v_codec, a->v_qs + row * vrb, a->v_sc + row * vsb, 1, D, vr);
        for (int r = r_lo; r < r_hi; ++r) {
            if (t >= nv[r]) continue;
            double p = z[r * span + t];
            double *orow = o + (int64_t)r * o_row_stride_elems;
            for (int d = 0; d < D; ++d) orow[d] += p * (double)vr[d];
        }
    }
    for (int r = r_lo; r < r_hi; ++r) {
        double *orow = o + (int64_t)r * o_row_stride_elems;
        if (nv[r] == 0) { lse[(int64_t)r * lse_row_stride] = -INFINITY; continue; }
        for (int d = 0; d < D; ++d) orow[d] /= l[r];
        lse[(int64_t)r * lse_row_stride] = m[r] + log(l[r]);
    }
    free(z); free(kr); free(vr); free(qd); free(nv); free(m); free(l);
}

/* Output row offsets: out is [n_seq][n_q][n_heads][head_dim], so row r = i*G + j
 * of (s, kh) is at ((s*n_q + i)*n_heads + kh*G + j).  The unit writes rows with
 * a stride; query token i of the unit starts G rows further in the unit but
 * n_heads rows further in the output, so the unit is run per query token. */
static void orc_attend_unit_to_output(const orc_attn_args *a, int s, int kh, int64_t t_lo,
                                      int64_t t_hi, int r_lo, int r_hi, double *out, double *out_lse)
{
    int D = a->head_dim, G = a->n_heads / a->n_kv_heads, R = a->n_q * G;
    double *o = (double *)malloc(sizeof(double) * (size_t)(R * D));
    double *l = (double *)malloc(sizeof(double) * (size_t)R);
    orc_attend_rows(a, s, kh, t_lo, t_hi, r_lo, r_hi, o, l, D, 1);
    for (int i = 0; i < a->n_q; ++i)
        for (int j = 0; j < G; ++j) {
            if (i * G + j < r_lo || i * G + j >= r_hi) continue;
            int64_t orow = ((int64_t)s * a->n_q + i) * a->n_heads + kh * G + j;
            memcpy(out + orow * D, o + (int64_t)(i * G + j) * D, sizeof(double) * (size_t)D);
            out_lse[orow] = l[i * G + j];
        }
    free(o); free(l);
}

/* Full decode attention: out [n_seq][n_q][n_heads][head_dim] fp64,
 * out_lse [n_seq][n_q][n_heads] fp64 (natural log).  q is fp32 (the fp16 or
 * fp32 inputs widened exactly).  n_threads > 1 spreads (seq, kv head, query
 * row) items over OpenMP threads; the arithmetic of each row is the same
 * whichever thread computes it. */
void orc_decode_attention(int k_codec, const uint8_t *k_qs, const void *k_sc,
                          int v_codec, const uint8_t *v_qs, const void *v_sc,
                          int n_seq, int n_kv_heads, int head_dim, int capacity,
                          const float *q, int n_q, int n_heads, const int32_t *kv_len,
                          double scale, double *out, double *out_lse, int n_threads)
{
    orc_attn_args a = {k_codec, v_codec, k_qs, v_qs, (const uint8_t *)k_sc, (const uint8_t *)v_sc, n_seq, n_kv_heads, head_dim,
                       capacity, q, n_q, n_heads, kv_len, scale};
    int R = n_q * (n_heads / n_kv_heads);
    if (n_threads <= 1) {
        /* one thread: every row of a (seq, kv head) unit in one pass */
        for (int u = 0; u < n_seq * n_kv_heads; ++u) {
            int s = u / n_kv_heads, kh = u % n_kv_heads;
            int64_t hi = kv_len[s] < 0 ? 0 : kv_len[s];
            orc_attend_unit_to_output(&a, s, kh, 0, hi, 0, R, out, out_lse);
        }
        return;
    }
    int64_t items = (int64_t)n_seq * n_kv_heads * R;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int64_t it = 0; it < items; ++it) {
        int u = (int)(it / R), r = (int)(it % R);
        int s = u / n_kv_heads, kh = u % n_kv_heads;
        int64_t hi = kv_len[s] < 0 ? 0 : kv_len[s];
        orc_attend_unit_to_output(&a, s, kh, 0, hi, r, r + 1, out, out_lse);
    }
    (void)n_threads;
}

/* Split attention: the last query token's visible range [0, kv_len[s]) is cut
 * into n_splits contiguous chunks of ceil(kv_len[s] / n_splits) tokens
 * (trailing chunks may be empty); each query row attends to its visible part
 * of each chunk.  part_o is [n_splits][n_seq][n_q][n_heads][head_dim],
 * part_lse [n_splits][n_seq][n_q][n_heads]; an empty part has o = 0 and
 * lse = -inf. */
void orc_decode_attention_split(int k_codec, const uint8_t *k_qs, const void *k_sc,
                                int v_codec, const uint8_t *v_qs, const void *v_sc,
                                int n_seq, int n_kv_heads, int head_dim, int capacity,
                                const float *q, int n_q, int n_heads, const int32_t *kv_len,
                                double scale, int n_splits, double *part_o, double *part_lse)
{
    orc_attn_args a = {k_codec, v_codec, k_qs, v_qs, (const uint8_t *)k_sc, (const uint8_t *)v_sc, n_seq, n_kv_heads, head_dim,
                       capacity, q, n_q, n_heads, kv_len, scale};
    int64_t rows = (int64_t)n_seq * n_q * n_heads;
    for (int sp = 0; sp < n_splits; ++sp)
        for (int s = 0; s < n_seq; ++s) {
            int64_t len = kv_len[s] < 0 ? 0 : kv_len[s];
            int64_t chunk = (len + n_splits - 1) / n_splits;
            int64_t lo = sp * chunk, hi = lo + chunk < len ? lo + chunk : len;
            if (lo > hi) lo = hi;
            for (int kh = 0; kh < n_kv_heads; ++kh)
                orc_attend_unit_to_output(&a, s, kh, lo, hi, 0, n_q * (n_heads / n_kv_heads),
                                          part_o + sp * rows * head_dim, part_lse + sp * rows);
        }
}

/* Log-sum-exp merge of n_splits partial results per row:
 * M = max_s lse_s, w_s = exp(lse_s - M), o = sum_s w_s o_s / sum_s w_s,
 * lse = M + ln sum_s w_s.  Parts with lse = -inf carry no weight; a row whose
 * parts are all -inf gets o = 0 and lse = -inf.  part_o is
 * [n_splits][rows][head_dim] and part_lse [n_splits][rows], as fp64. */
void orc_merge_splits(const double *part_o, const double *part_lse, int n_splits, int64_t rows,
                      int head_dim, double *out, double *out_lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < n_splits; ++s)
            if (part_lse[s * rows + r] > M) M = part_lse[s * rows + r];
        double *o = out + r * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (M == -INFINITY) { out_lse[r] = -INFINITY; continue; }
        double wsum = 0.0;
        for (int s = 0; s < n_splits; ++s) {
            double ls = part_lse[s * rows + r];
            if (ls == -INFINITY) continue;
            double w = exp(ls - M);
            wsum += w;
            const double *os = part_o + (s * rows + r) * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] += w * os[d];
        }
        for (int d = 0; d < head_dim; ++d) o[d] /= wsum;
        out_lse[r] = M + log(wsum);
    }
}

int orc_omp_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
