/*
 * thinmx CPU oracle — TEST INFRASTRUCTURE, not part of the product.
 * See thinmx_oracle.h for the sources followed and the rules on its use.
 *
 * Everything is plain C99, single-threaded, fp64, written so that each
 * step can be checked by eye against the definitions it follows:
 *   - no blocking, no fusion, no reordering of the sums beyond k = 0..K-1;
 *   - scalar formats decoded from their bit fields;
 *   - rounding done on exact quantities with rint() (round to nearest,
 *     ties to even, the C default rounding mode).
 */
#include "thinmx_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ===================================================================== */
/* Scalar formats                                                         */
/* ===================================================================== */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
   exponent 0 is subnormal: value = m/2; otherwise 2^(e-1) * (1 + m/2). */
double orc_e2m1_value(unsigned code)
{
    unsigned s = (code >> 3) & 1u;
    unsigned e = (code >> 1) & 3u;
    unsigned m = code & 1u;
    double v;
    if (e == 0)
        v = 0.5 * (double)m;
    else
        v = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -v : v;
}

/* E8M0: an unsigned biased exponent, value 2^(b-127); 0xFF encodes NaN. */
double orc_e8m0_value(unsigned byte)
{
    if (byte == 255u) return NAN;
    return ldexp(1.0, (int)byte - 127);
}

/* Nearest E2M1 magnitude to |t|; at an exact midpoint the candidate whose
   mantissa bit is 0 wins; magnitudes above 6 saturate to 6 (the largest
   code).  The sign bit is copied from t, so a negative value that rounds
   to zero gives code 0x8. */
unsigned orc_e2m1_encode(double t)
{
    unsigned sign = signbit(t) ? 8u : 0u;
    double a = fabs(t);
    if (a > 6.0) a = 6.0; /* saturate first: far above 6, the distances to
                             4 and 6 are equal in fp64 */
    unsigned best = 0;
    double best_d = INFINITY;
    for (unsigned c = 0; c < 8; ++c) {
        double d = fabs(a - orc_e2m1_value(c));
        if (d < best_d || (d == best_d && (c & 1u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    return sign | best;
}

/* floor(log2 a) for finite a > 0, read off the binary exponent:
   frexp gives a = f * 2^e with f in [0.5, 1), so floor(log2 a) = e - 1.
   (A library log2 rounds values just below a power of two up to it.) */
int orc_floor_log2(float a)
{
    int e = 0;
    (void)frexp((double)a, &e);
    return e - 1;
}

double orc_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round v to the nearest value with p significant bits whose exponent is
   at least emin (subnormals below that), ties to even.  Returns the
   rounded value as a double (exact).  Used by both 16-bit formats. */
static double round_to_format(double a /* >= 0, finite */, int p, int emin)
{
    if (a == 0.0) return 0.0;
    int e2 = 0;
    (void)frexp(a, &e2);
    int e = e2 - 1;                 /* floor(log2 a) */
    if (e < emin) e = emin;
    double q = ldexp(1.0, e - (p - 1)); /* spacing of the binade */
    double r = rint(a / q);         /* a/q is exact: scaling by 2^k */
    return r * q;
}

uint16_t orc_bf16_round(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    /* bf16: 8 significant bits, exponent range of fp32 */
    double r = round_to_format(a, 8, -126);
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    float f = (float)r; /* exact: every bf16 value is an fp32 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

double orc_f16_value(uint16_t h)
{
    unsigned s = (h >> 15) & 1u;
    unsigned e = (h >> 10) & 31u;
    unsigned m = h & 1023u;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)m / 1024.0, (int)e - 15);
    return s ? -v : v;
}

uint16_t orc_f16_round(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    /* binary16: 11 significant bits, min normal exponent -14 */
    double r = round_to_format(a, 11, -14);
    if (r >= 65536.0) return (uint16_t)(sign | 0x7C00u);
    if (r < ldexp(1.0, -14)) /* subnormal (or zero): mantissa = r / 2^-24 */
        return (uint16_t)(sign | (uint16_t)ldexp(r, 24));
    int e2 = 0;
    double f = frexp(r, &e2); /* r = f * 2^e2, f in [0.5,1) */
    int ex = e2 - 1;
    unsigned mant = (unsigned)((2.0 * f - 1.0) * 1024.0);
    return (uint16_t)(sign | (unsigned)((ex + 15) << 10) | mant);
}

/* ===================================================================== */
/* MXFP4                                                                  */
/* ===================================================================== */

static unsigned get_nibble(const uint8_t* row, int64_t i)
{
    return (row[i / 2] >> (4 * (i & 1))) & 15u;
}

static void put_nibble(uint8_t* row, int64_t i, unsigned v)
{
    uint8_t* b = &row[i / 2];
    if (i & 1)
        *b = (uint8_t)((*b & 0x0Fu) | (v << 4));
    else
        *b = (uint8_t)((*b & 0xF0u) | v);
}

/* Per block of 32 weights along k:
     amax = max |w|;  X = floor(log2 amax) - 2 clamped to [-127, 127]
     (X = -127 when amax = 0);  scale byte = X + 127;
     code = E2M1 round-to-nearest-even of w / 2^X, saturating at 6. */
int orc_mxfp4_quantize(const float* w, int64_t n, int64_t k,
                       uint8_t* codes, uint8_t* scales)
{
    if (n < 0 || k < 0 || k % 32 != 0) return ORC_ERR_SHAPE;
    int status = ORC_OK;
    const int64_t nb = k / 32;
    for (int64_t r = 0; r < n; ++r) {
        const float* wr = w + r * k;
        uint8_t* cr = codes + r * (k / 2);
        for (int64_t b = 0; b < nb; ++b) {
            int finite = 1;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double v = (double)wr[b * 32 + i];
                if (!isfinite(v)) finite = 0;
                else if (fabs(v) > amax) amax = fabs(v);
            }
            if (!finite) {
                scales[r * nb + b] = 0xFF;
                for (int i = 0; i < 32; ++i) put_nibble(cr, b * 32 + i, 0);
                status = ORC_ERR_NONFINITE;
                continue;
            }
            int X;
            if (amax == 0.0) {
                X = -127;
            } else {
                X = orc_floor_log2((float)amax) - 2;
                if (X < -127) X = -127;
                if (X > 127) X = 127;
            }
            scales[r * nb + b] = (uint8_t)(X + 127);
            for (int i = 0; i < 32; ++i) {
                double t = ldexp((double)wr[b * 32 + i], -X);
                put_nibble(cr, b * 32 + i, orc_e2m1_encode(t));
            }
        }
    }
    return status;
}

static double mxfp4_weight(const uint8_t* codes, const uint8_t* scales,
                           int64_t k, int64_t r, int64_t kk)
{
    unsigned c = get_nibble(codes + r * (k / 2), kk);
    unsigned s = scales[r * (k / 32) + kk / 32];
    return orc_e2m1_value(c) * orc_e8m0_value(s);
}

void orc_mxfp4_dequantize(const uint8_t* codes, const uint8_t* scales,
                          int64_t n, int64_t k, double* out)
{
    for (int64_t r = 0; r < n; ++r)
        for (int64_t kk = 0; kk < k; ++kk)
            out[r * k + kk] = mxfp4_weight(codes, scales, k, r, kk);
}

void orc_mxfp4_matvec(const uint8_t* codes, const uint8_t* scales,
                      const float* postscale, int64_t n, int64_t k,
                      const uint16_t* x_bf16, int64_t m, double* y)
{
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t r = 0; r < n; ++r) {
            double acc = 0.0;
            for (int64_t kk = 0; kk < k; ++kk)
                acc += mxfp4_weight(codes, scales, k, r, kk) *
                       orc_bf16_value(x_bf16[i * k + kk]);
            if (postscale) acc *= (double)postscale[r];
            y[i * n + r] = acc;
        }
    }
}

void orc_bf16_matvec(const uint16_t* w_bf16, int64_t n, int64_t k,
                     const uint16_t* x_bf16, int64_t m, double* y)
{
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t r = 0; r < n; ++r) {
            double acc = 0.0;
            for (int64_t kk = 0; kk < k; ++kk)
                acc += orc_bf16_value(w_bf16[r * k + kk]) *
                       orc_bf16_value(x_bf16[i * k + kk]);
            y[i * n + r] = acc;
        }
    }
}

/* SwiGLU, the gated activation: h = silu(g) * u = g / (1 + e^-g) * u. */
void orc_swiglu(const double* g, const double* u, int64_t len, double* h)
{
    for (int64_t i = 0; i < len; ++i)
        h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

void orc_mxfp4_swiglu_matvec(const uint8_t* g_codes, const uint8_t* g_scales,
                             const float* g_post,
                             const uint8_t* u_codes, const uint8_t* u_scales,
                             const float* u_post, int64_t n, int64_t k,
                             const uint16_t* x_bf16, int64_t m, double* h)
{
    double* g = (double*)malloc(sizeof(double) * (size_t)(m * n + 1));
    double* u = (double*)malloc(sizeof(double) * (size_t)(m * n + 1));
    orc_mxfp4_matvec(g_codes, g_scales, g_post, n, k, x_bf16, m, g);
    orc_mxfp4_matvec(u_codes, u_scales, u_post, n, k, x_bf16, m, u);
    orc_swiglu(g, u, m * n, h);
    free(g);
    free(u);
}

void orc_bf16_swiglu_matvec(const uint16_t* wg, const uint16_t* wu,
                            int64_t n, int64_t k, const uint16_t* x_bf16,
                            int64_t m, double* h)
{
    double* g = (double*)malloc(sizeof(double) * (size_t)(m * n + 1));
    double* u = (double*)malloc(sizeof(double) * (size_t)(m * n + 1));
    orc_bf16_matvec(wg, n, k, x_bf16, m, g);
    orc_bf16_matvec(wu, n, k, x_bf16, m, u);
    orc_swiglu(g, u, m * n, h);
    free(g);
    free(u);
}

/* ===================================================================== */
/* MoE: router -> top-k -> softmax over the selected -> expert MLPs      */
/* ===================================================================== */

void orc_router_logits(const uint16_t* x_bf16, const uint16_t* wr_bf16,
                       int32_t n_experts, int64_t hidden, double* logits)
{
    for (int32_t e = 0; e < n_experts; ++e) {
        double acc = 0.0;
        for (int64_t kk = 0; kk < hidden; ++kk)
            acc += orc_bf16_value(x_bf16[kk]) *
                   orc_bf16_value(wr_bf16[(int64_t)e * hidden + kk]);
        logits[e] = acc;
    }
}

/* top_k rounds of "largest remaining logit, lower index on ties". */
void orc_topk(const float* logits, int32_t n_experts, int32_t top_k,
              int32_t* idx)
{
    char* taken = (char*)calloc((size_t)n_experts + 1, 1);
    for (int32_t j = 0; j < top_k; ++j) {
        int32_t best = -1;
        for (int32_t e = 0; e < n_experts; ++e) {
            if (taken[e]) continue;
            if (best < 0 || logits[e] > logits[best]) best = e;
        }
        idx[j] = best;
        if (best >= 0) taken[best] = 1;
    }
    free(taken);
}

void orc_softmax_selected(const float* logits, const int32_t* idx,
                          int32_t top_k, double* p)
{
    double mx = -INFINITY;
    for (int32_t j = 0; j < top_k; ++j)
        if ((double)logits[idx[j]] > mx) mx = (double)logits[idx[j]];
    double den = 0.0;
    for (int32_t j = 0; j < top_k; ++j) {
        p[j] = exp((double)logits[idx[j]] - mx);
        den += p[j];
    }
    for (int32_t j = 0; j < top_k; ++j) p[j] /= den;
}

/* y[r] = sum_k deq[r][k] * v[k] with an fp64 vector v. */
static void mxfp4_matvec_f64(const uint8_t* codes, const uint8_t* scales,
                             int64_t n, int64_t k, const double* v,
                             double* y)
{
    for (int64_t r = 0; r < n; ++r) {
        double acc = 0.0;
        for (int64_t kk = 0; kk < k; ++kk)
            acc += mxfp4_weight(codes, scales, k, r, kk) * v[kk];
        y[r] = acc;
    }
}

int orc_moe_mlp(const uint16_t* x_bf16, int64_t hidden, int64_t inter,
                const uint16_t* wr_bf16, int32_t n_experts, int32_t top_k,
                const uint8_t* gu_codes, const uint8_t* gu_scales,
                const uint8_t* dn_codes, const uint8_t* dn_scales,
                double* out, int32_t* idx, double* p, float* logits32)
{
    if (top_k < 1 || top_k > n_experts || hidden % 32 || inter % 32)
        return ORC_ERR_SHAPE;
    double* logits = (double*)malloc(sizeof(double) * (size_t)n_experts);
    orc_router_logits(x_bf16, wr_bf16, n_experts, hidden, logits);
    /* The selection is taken on the fp32 rounding of each exact logit. */
    for (int32_t e = 0; e < n_experts; ++e) logits32[e] = (float)logits[e];
    orc_topk(logits32, n_experts, top_k, idx);
    orc_softmax_selected(logits32, idx, top_k, p);

    double* xv = (double*)malloc(sizeof(double) * (size_t)hidden);
    double* g = (double*)malloc(sizeof(double) * (size_t)inter);
    double* u = (double*)malloc(sizeof(double) * (size_t)inter);
    double* h = (double*)malloc(sizeof(double) * (size_t)inter);
    double* y = (double*)malloc(sizeof(double) * (size_t)hidden);
    for (int64_t kk = 0; kk < hidden; ++kk) xv[kk] = orc_bf16_value(x_bf16[kk]);
    for (int64_t r = 0; r < hidden; ++r) out[r] = 0.0;

    const int64_t gu_rows = 2 * inter;
    for (int32_t j = 0; j < top_k; ++j) {
        int64_t e = idx[j];
        const uint8_t* gc = gu_codes + e * gu_rows * (hidden / 2);
        const uint8_t* gs = gu_scales + e * gu_rows * (hidden / 32);
        /* gate = rows [0, inter), up = rows [inter, 2*inter) */
        mxfp4_matvec_f64(gc, gs, inter, hidden, xv, g);
        mxfp4_matvec_f64(gc + inter * (hidden / 2), gs + inter * (hidden / 32),
                         inter, hidden, xv, u);
        orc_swiglu(g, u, inter, h);
        const uint8_t* dc = dn_codes + e * hidden * (inter / 2);
        const uint8_t* ds = dn_scales + e * hidden * (inter / 32);
        mxfp4_matvec_f64(dc, ds, hidden, inter, h, y);
        for (int64_t r = 0; r < hidden; ++r) out[r] += p[j] * y[r];
    }
    free(logits); free(xv); free(g); free(u); free(h); free(y);
    return ORC_OK;
}

/* ===================================================================== */
/* Grouped affine INT4                                                    */
/* ===================================================================== */

/* Per (row, group): mn/mx over the group's own elements (the last group
   may be partial); s = fp16(RNE((mx - mn) / 15)); zp = clamp(rint(-mn/s),
   0, 15); q = clamp(rint(w/s) + zp, 0, 15); deq = (q - zp) * s.
   A group with s == 0 (constant group, or a range below fp16's
   resolution) stores zp = 0 and q = 0.  A group holding a NaN/Inf, or
   whose scale overflows fp16, stores zp = 0, q = 0 and flags the call. */
int orc_int4_quantize(const float* w, int64_t n, int64_t k, int32_t group,
                      uint8_t* codes, uint16_t* scales_f16, uint8_t* zp)
{
    if (n < 0 || k < 0 || k % 2 != 0 || group < 1) return ORC_ERR_SHAPE;
    int status = ORC_OK;
    const int64_t ng = (k + group - 1) / group;
    const int64_t zb = (ng + 1) / 2;
    for (int64_t r = 0; r < n; ++r) {
        const float* wr = w + r * k;
        uint8_t* cr = codes + r * (k / 2);
        uint8_t* zr = zp + r * zb;
        memset(zr, 0, (size_t)zb);
        for (int64_t g = 0; g < ng; ++g) {
            int64_t lo = g * group;
            int64_t hi = lo + group < k ? lo + group : k;
            int finite = 1;
            float mn = wr[lo], mx = wr[lo];
            for (int64_t kk = lo; kk < hi; ++kk) {
                if (!isfinite(wr[kk])) finite = 0;
                if (wr[kk] < mn) mn = wr[kk];
                if (wr[kk] > mx) mx = wr[kk];
            }
            uint16_t s16;
            if (!finite) {
                s16 = 0x7E00u;
            } else {
                double range = (double)mx - (double)mn;
                s16 = orc_f16_round(range / 15.0);
            }
            scales_f16[r * ng + g] = s16;
            double s = orc_f16_value(s16);
            if (!finite || isinf(s)) {
                status = ORC_ERR_NONFINITE;
                for (int64_t kk = lo; kk < hi; ++kk) put_nibble(cr, kk, 0);
                continue;
            }
            if (s == 0.0) {
                for (int64_t kk = lo; kk < hi; ++kk) put_nibble(cr, kk, 0);
                continue;
            }
            double z = rint(-(double)mn / s);
            if (z < 0) z = 0;
            if (z > 15) z = 15;
            put_nibble(zr, g, (unsigned)z);
            for (int64_t kk = lo; kk < hi; ++kk) {
                double q = rint((double)wr[kk] / s) + z;
                if (q < 0) q = 0;
                if (q > 15) q = 15;
                put_nibble(cr, kk, (unsigned)q);
            }
        }
    }
    return status;
}

static double int4_weight(const uint8_t* codes, const uint16_t* scales_f16,
                          const uint8_t* zp, int64_t k, int32_t group,
                          int64_t r, int64_t kk)
{
    const int64_t ng = (k + group - 1) / group;
    const int64_t zb = (ng + 1) / 2;
    int64_t g = kk / group;
    double q = (double)get_nibble(codes + r * (k / 2), kk);
    double z = (double)get_nibble(zp + r * zb, g);
    double s = orc_f16_value(scales_f16[r * ng + g]);
    return (q - z) * s;
}

void orc_int4_dequantize(const uint8_t* codes, const uint16_t* scales_f16,
                         const uint8_t* zp, int64_t n, int64_t k,
                         int32_t group, double* out)
{
    for (int64_t r = 0; r < n; ++r)
        for (int64_t kk = 0; kk < k; ++kk)
            out[r * k + kk] = int4_weight(codes, scales_f16, zp, k, group, r, kk);
}

void orc_int4_matvec(const uint8_t* codes, const uint16_t* scales_f16,
                     const uint8_t* zp, int64_t n, int64_t k, int32_t group,
                     const uint16_t* x_bf16, int64_t m, double* y)
{
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t r = 0; r < n; ++r) {
            double acc = 0.0;
            for (int64_t kk = 0; kk < k; ++kk)
                acc += int4_weight(codes, scales_f16, zp, k, group, r, kk) *
                       orc_bf16_value(x_bf16[i * k + kk]);
            y[i * n + r] = acc;
        }
    }
}

/* ===================================================================== */
/* FP8 (E4M3) with one fp32 scale per row                                 */
/* ===================================================================== */

/* E4M3 without infinities: bit 7 sign, bits 6..3 exponent (bias 7), bits
   2..0 mantissa.  Exponent 0 is subnormal: (m/8) * 2^-6; exponent 15 with
   mantissa 7 is NaN; otherwise 2^(e-7) * (1 + m/8).  The largest finite
   magnitude is 448 (e = 15, m = 6). */
double orc_e4m3_value(unsigned code)
{
    unsigned s = (code >> 7) & 1u;
    unsigned e = (code >> 3) & 15u;
    unsigned m = code & 7u;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -v : v;
}

/* Nearest finite E4M3 magnitude to |t|; at an exact midpoint the code
   whose mantissa bit 0 is clear wins (ties to even); magnitudes above 448
   saturate to 448.  The sign is copied from t, so a negative value that
   rounds to zero gives 0x80; NaN gives 0x7F. */
unsigned orc_e4m3_encode(double t)
{
    if (isnan(t)) return 0x7Fu;
    unsigned sign = signbit(t) ? 0x80u : 0u;
    double a = fabs(t);
    if (a > 448.0) a = 448.0;
    unsigned best = 0;
    double best_d = INFINITY;
    for (unsigned c = 0; c < 0x7Fu; ++c) { /* the 127 finite magnitudes */
        double d = fabs(a - orc_e4m3_value(c));
        if (d < best_d || (d == best_d && (c & 1u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    return sign | best;
}

/* Per row: amax = max |w|; scale = fp32(amax / 448); code = E4M3 of
   w / scale (the division in fp64 with the stored fp32 scale). */
int orc_fp8_quantize(const float* w, int64_t n, int64_t k, uint8_t* codes,
                     float* scales)
{
    if (n < 0 || k < 0) return ORC_ERR_SHAPE;
    int status = ORC_OK;
    for (int64_t r = 0; r < n; ++r) {
        const float* wr = w + r * k;
        uint8_t* cr = codes + r * k;
        int finite = 1;
        double amax = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            double v = (double)wr[i];
            if (!isfinite(v)) finite = 0;
            else if (fabs(v) > amax) amax = fabs(v);
        }
        if (!finite) {
            scales[r] = NAN;
            for (int64_t i = 0; i < k; ++i) cr[i] = 0;
            status = ORC_ERR_NONFINITE;
            continue;
        }
        float s = (float)(amax / 448.0);
        scales[r] = s;
        if (s == 0.0f) { /* amax = 0, or below what an fp32 scale can hold */
            for (int64_t i = 0; i < k; ++i) cr[i] = 0;
            continue;
        }
        for (int64_t i = 0; i < k; ++i)
            cr[i] = (uint8_t)orc_e4m3_encode((double)wr[i] / (double)s);
    }
    return status;
}

void orc_fp8_dequantize(const uint8_t* codes, const float* scales, int64_t n,
                        int64_t k, double* out)
{
    for (int64_t r = 0; r < n; ++r)
        for (int64_t i = 0; i < k; ++i)
            out[r * k + i] = orc_e4m3_value(codes[r * k + i]) * (double)scales[r];
}

/* The row sum of code values times x, then times the row's scale. */
void orc_fp8_matvec(const uint8_t* codes, const float* scales, int64_t n,
                    int64_t k, const uint16_t* x_bf16, int64_t m, double* y)
{
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t r = 0; r < n; ++r) {
            double acc = 0.0;
            for (int64_t kk = 0; kk < k; ++kk)
                acc += orc_e4m3_value(codes[r * k + kk]) *
                       orc_bf16_value(x_bf16[i * k + kk]);
            y[i * n + r] = acc * (double)scales[r];
        }
    }
}

void orc_fp8_swiglu_matvec(const uint8_t* g_codes, const float* g_scales,
                           const uint8_t* u_codes, const float* u_scales,
                           int64_t n, int64_t k, const uint16_t* x_bf16,
                           int64_t m, double* h)
{
    double* g = (double*)malloc(sizeof(double) * (size_t)(m * n));
    double* u = (double*)malloc(sizeof(double) * (size_t)(m * n));
    orc_fp8_matvec(g_codes, g_scales, n, k, x_bf16, m, g);
    orc_fp8_matvec(u_codes, u_scales, n, k, x_bf16, m, u);
    orc_swiglu(g, u, m * n, h);
    free(g);
    free(u);
}

/* ===================================================================== */
/* Single-token grouped-query attention over a bf16 KV cache             */
/* ===================================================================== */

/* For query head h, kv_head = h / (heads / kv_heads); over the cached
   tokens t < len of that kv head: s_t = scale * sum_i q[h][i] * k[t][i],
   p = softmax(s) over t (with the max subtracted), o[h][i] = sum_t p_t *
   v[t][i].  q bf16 [heads][d]; k, v bf16 [kv_heads][cap][d] (token t of kv
   head j at (j * cap + t) * d); o fp64 [heads][d].  Everything in fp64. */
int orc_gqa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                   int32_t heads, int32_t kv_heads, int32_t d, int64_t cap,
                   int64_t len, double scale, double* o)
{
    if (heads < 1 || kv_heads < 1 || heads % kv_heads != 0 || d < 1 ||
        len < 1 || cap < len)
        return ORC_ERR_SHAPE;
    const int32_t group = heads / kv_heads;
    double* s = (double*)malloc(sizeof(double) * (size_t)len);
    for (int32_t h = 0; h < heads; ++h) {
        const int32_t j = h / group;
        const uint16_t* kh = k + (int64_t)j * cap * d;
        const uint16_t* vh = v + (int64_t)j * cap * d;
        double mx = -INFINITY;
        for (int64_t t = 0; t < len; ++t) {
            double acc = 0.0;
            for (int32_t i = 0; i < d; ++i)
                acc += orc_bf16_value(q[(int64_t)h * d + i]) *
                       orc_bf16_value(kh[t * d + i]);
            s[t] = acc * scale;
            if (s[t] > mx) mx = s[t];
        }
        double sum = 0.0;
        for (int64_t t = 0; t < len; ++t) {
            s[t] = exp(s[t] - mx);
            sum += s[t];
        }
        for (int32_t i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int64_t t = 0; t < len; ++t)
                acc += s[t] * orc_bf16_value(vh[t * d + i]);
            o[(int64_t)h * d + i] = acc / sum;
        }
    }
    free(s);
    return ORC_OK;
}

/* ===================================================================== */
/* Q1 / Q2 packed low-bit experts                                         */
/* ===================================================================== */

/* Layout of one matrix [n][k] (n rows = outputs, k = reduction), written
   as one buffer:
     plane 0 [n][P], then (Q2 only) plane 1 [n][P], then scales [n][S];
   P = ceil(k/8) rounded up to 16 bytes, S = ceil(k/128) rounded up to 16.
   Bit (kk mod 8) of byte kk/8 of a row's plane p holds bit p of the code
   of element kk; padding bytes are zero.  Scale byte: E8M0 of the block's
   step 2^X. */
#define LB_BLOCK 128

static int64_t round_up16(int64_t v) { return (v + 15) / 16 * 16; }

int64_t orc_lowbit_plane_bytes(int64_t k) { return round_up16((k + 7) / 8); }
int64_t orc_lowbit_scale_bytes(int64_t k)
{
    return round_up16((k + LB_BLOCK - 1) / LB_BLOCK);
}
int64_t orc_lowbit_matrix_bytes(int32_t bits, int64_t n, int64_t k)
{
    return n * ((int64_t)bits * orc_lowbit_plane_bytes(k) +
                orc_lowbit_scale_bytes(k));
}

/* The block's step exponent X: m = (sum of |w| in order, in fp64) / count;
   X = floor(log2 m) + (m's mantissa in [1, 2) above 1.5), so that 2^X is
   the power of two nearest m (ties to the lower one); clamped to
   [-127, 127].  An all-zero block gives -127; a block holding a NaN/Inf
   gives 128 (no valid exponent). */
static int lowbit_block_exponent(const float* w, int64_t cnt)
{
    double s = 0.0;
    for (int64_t i = 0; i < cnt; ++i) {
        if (!isfinite(w[i])) return 128;
        s += fabs((double)w[i]);
    }
    if (s == 0.0) return -127;
    const double m = s / (double)cnt;
    int e;
    const double f = frexp(m, &e); /* m = f * 2^e, f in [0.5, 1) */
    int x = (e - 1) + (2.0 * f > 1.5 ? 1 : 0);
    if (x < -127) x = -127;
    if (x > 127) x = 127;
    return x;
}

/* Q1: code 1 for w < 0, else 0 (value (1 - 2c) * 2^X).
   Q2: code q = clamp(floor(w / 2^X) + 2, 0, 3) (value (q - 1.5) * 2^X:
   the nearest of the levels -1.5, -0.5, 0.5, 1.5 steps, a tie at a
   multiple of the step going up). */
int orc_lowbit_quantize(int32_t bits, const float* w, int64_t n, int64_t k,
                        uint8_t* buf)
{
    if ((bits != 1 && bits != 2) || n < 0 || k < 1) return ORC_ERR_SHAPE;
    const int64_t P = orc_lowbit_plane_bytes(k), S = orc_lowbit_scale_bytes(k);
    memset(buf, 0, (size_t)orc_lowbit_matrix_bytes(bits, n, k));
    int status = ORC_OK;
    for (int64_t r = 0; r < n; ++r) {
        const float* row = w + r * k;
        for (int64_t b0 = 0; b0 < k; b0 += LB_BLOCK) {
            const int64_t cnt = (k - b0 < LB_BLOCK) ? k - b0 : LB_BLOCK;
            const int x = lowbit_block_exponent(row + b0, cnt);
            uint8_t* sc = buf + (int64_t)bits * n * P + r * S + b0 / LB_BLOCK;
            if (x == 128) { /* NaN/Inf: NaN scale, zero codes */
                *sc = 0xFF;
                status = ORC_ERR_NONFINITE;
                continue;
            }
            *sc = (uint8_t)(x + 127);
            const double t = ldexp(1.0, x);
            for (int64_t i = 0; i < cnt; ++i) {
                const int64_t kk = b0 + i;
                unsigned code;
                if (bits == 1) {
                    code = row[kk] < 0.0f ? 1u : 0u;
                } else {
                    double q = floor((double)row[kk] / t) + 2.0;
                    if (q < 0.0) q = 0.0;
                    if (q > 3.0) q = 3.0;
                    code = (unsigned)q;
                }
                for (int32_t p = 0; p < bits; ++p)
                    if ((code >> p) & 1u)
                        buf[p * n * P + r * P + kk / 8] |= (uint8_t)(1u << (kk % 8));
            }
        }
    }
    return status;
}

static double lowbit_weight(int32_t bits, const uint8_t* buf, int64_t n,
                            int64_t k, int64_t r, int64_t kk)
{
    const int64_t P = orc_lowbit_plane_bytes(k), S = orc_lowbit_scale_bytes(k);
    unsigned code = 0;
    for (int32_t p = 0; p < bits; ++p)
        code |= ((buf[p * n * P + r * P + kk / 8] >> (kk % 8)) & 1u) << p;
    const double t =
        orc_e8m0_value(buf[(int64_t)bits * n * P + r * S + kk / LB_BLOCK]);
    if (bits == 1) return (code ? -1.0 : 1.0) * t;
    return ((double)code - 1.5) * t;
}

void orc_lowbit_dequantize(int32_t bits, const uint8_t* buf, int64_t n,
                           int64_t k, double* out)
{
    for (int64_t r = 0; r < n; ++r)
        for (int64_t kk = 0; kk < k; ++kk)
            out[r * k + kk] = lowbit_weight(bits, buf, n, k, r, kk);
}

/* y[r] = sum_k deq[r][k] * v[k] with an fp64 vector v. */
static void lowbit_matvec_f64(int32_t bits, const uint8_t* buf, int64_t n,
                              int64_t k, const double* v, double* y)
{
    for (int64_t r = 0; r < n; ++r) {
        double acc = 0.0;
        for (int64_t kk = 0; kk < k; ++kk)
            acc += lowbit_weight(bits, buf, n, k, r, kk) * v[kk];
        y[r] = acc;
    }
}

/* The MoE layer with Q1 / Q2 experts: router logits, top-k on their fp32
   roundings, softmax over the selected, then for each selected expert j
   h_j = silu(gate_j x) * up_j x (gate = rows [0, inter) of the expert's
   gate/up matrix [2 inter][hidden], up = rows [inter, 2 inter)), and
   out = sum_j p_j down_j h_j (down [hidden][inter]).  gu / dn hold the E
   experts' buffers back to back; h [top_k][inter] returns the h_j. */
int orc_moe_lowbit_mlp(int32_t bits, const uint16_t* x_bf16, int64_t hidden,
                       int64_t inter, const uint16_t* wr_bf16,
                       int32_t n_experts, int32_t top_k, const uint8_t* gu,
                       const uint8_t* dn, double* out, int32_t* idx, double* p,
                       float* logits32, double* h)
{
    if ((bits != 1 && bits != 2) || top_k < 1 || top_k > n_experts ||
        hidden < 1 || inter < 1)
        return ORC_ERR_SHAPE;
    double* logits = (double*)malloc(sizeof(double) * (size_t)n_experts);
    orc_router_logits(x_bf16, wr_bf16, n_experts, hidden, logits);
    for (int32_t e = 0; e < n_experts; ++e) logits32[e] = (float)logits[e];
    orc_topk(logits32, n_experts, top_k, idx);
    orc_softmax_selected(logits32, idx, top_k, p);

    double* xv = (double*)malloc(sizeof(double) * (size_t)hidden);
    double* g = (double*)malloc(sizeof(double) * (size_t)(2 * inter));
    double* y = (double*)malloc(sizeof(double) * (size_t)hidden);
    for (int64_t kk = 0; kk < hidden; ++kk) xv[kk] = orc_bf16_value(x_bf16[kk]);
    for (int64_t r = 0; r < hidden; ++r) out[r] = 0.0;
    const int64_t gu_bytes = orc_lowbit_matrix_bytes(bits, 2 * inter, hidden);
    const int64_t dn_bytes = orc_lowbit_matrix_bytes(bits, hidden, inter);
    for (int32_t j = 0; j < top_k; ++j) {
        const int64_t e = idx[j];
        /* gate and up rows of one matrix: g[0, inter) and g[inter, 2 inter) */
        lowbit_matvec_f64(bits, gu + e * gu_bytes, 2 * inter, hidden, xv, g);
        double* hj = h + (int64_t)j * inter;
        orc_swiglu(g, g + inter, inter, hj);
        lowbit_matvec_f64(bits, dn + e * dn_bytes, hidden, inter, hj, y);
        for (int64_t r = 0; r < hidden; ++r) out[r] += p[j] * y[r];
    }
    free(logits); free(xv); free(g); free(y);
    return ORC_OK;
}

