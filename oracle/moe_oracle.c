/*
 * moe_oracle.c -- plain CPU reference of one MoE FFN layer's forward pass.
 *
 * TEST INFRASTRUCTURE ONLY (see moe_oracle.h): used by the tests, the smoke
 * check and the benchmark's CPU-baseline leg, never by the product path.
 * Build with -O2 -ffp-contract=off so that no fused multiply-add changes the
 * fp32 score arithmetic.
 *
 * The steps follow the pages in order:
 *   0. optional router front end: LayerNorm or L2 normalisation of h
 *      ([2kiu] §5.2), a two-layer router silu(x W1) W2 ([cnnetsun] §3.1)
 *   1. logits z = h . W_router (+ bias)          [coreui] §3.1, [csdn] §3.1
 *      (scores divided by a temperature tau      [cnnetsun] §3.1 step 3)
 *   2. penalty s_i = z_i - lambda * usage_i       [mhpn] §2.3 (second layer),
 *      applied before top-k                       [cnnetsun] §3.1 step 4
 *   3. softmax over experts and top-k picks      [coreui] §3.1
 *   4. f_i (top-k counts / T) and P_i (mean p_i) [cnnetsun] §4.2, [coreui] §3.1
 *   5. capacity-capped dispatch with reroute     [mhpn] §2.3 (third layer),
 *      capacity ceil(T*k/E*cf)                   [coreui] §5.2, [2kiu] §2
 *   6. SwiGLU experts W2(silu(W1 x) * W3 x)      [mhpn] §3.1, [2kiu] §1
 *   7. weighted combine, weights renormalised    [mhpn] §4.3
 *      over the experts actually used
 *   (8. expert weights stored as 8-bit codes with one scale per row, the
 *      bytes-moved concern of [cnnetsun] §3.2 and [2kiu] §5.1: decoded here
 *      from the e4m3 format's definition and used in double precision.)
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* e4m3 ("E4M3" 8-bit float): bit 7 sign, bits 6..3 exponent with bias 7, bits
 * 2..0 mantissa; exponent field 0 holds subnormals m/8 * 2^-6; the codes with
 * every exponent and mantissa bit set (0x7F, 0xFF) are NaN; there is no
 * infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_value(uint8_t b)
{
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* The e4m3 code nearest to v, ties to the even code; magnitudes above 448
 * (the largest finite value) give +-448; NaN gives 0x7F. */
uint8_t oracle_e4m3_encode(float v)
{
    if (isnan(v)) return 0x7F;
    const uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {   /* subnormal range: steps of 2^-9 */
        double q = a / ldexp(1.0, -9);
        double f = floor(q);
        double m = (q - f > 0.5 || (q - f == 0.5 && fmod(f, 2.0) != 0.0)) ? f + 1.0 : f;
        return sign | (uint8_t)m;   /* m == 8 is the code of 2^-6 */
    }
    int e;
    double fr = frexp(a, &e);   /* a = fr * 2^e, fr in [0.5, 1) */
    e -= 1;                     /* a = (2 fr) * 2^e, 2 fr in [1, 2) */
    double q = (2.0 * fr - 1.0) * 8.0;
    double f = floor(q);
    double m = (q - f > 0.5 || (q - f == 0.5 && fmod(f, 2.0) != 0.0)) ? f + 1.0 : f;
    if (m == 8.0) {
        m = 0.0;
        e += 1;
    }
    if (e + 7 > 15 || (e + 7 == 15 && m == 7.0)) return sign | 0x7E;
    return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

/* Row-wise e4m3 quantisation: s = max |x| / 448 (fp32; 1 for an all-zero
 * row), code_i = e4m3(x_i / s) with the quotient rounded to fp32. */
void oracle_quantize_row(int n, const float* x, uint8_t* codes, float* scale)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int i = 0; i < n; ++i) codes[i] = oracle_e4m3_encode(x[i] / s);
    *scale = s;
}

/* e2m1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0
 * is the subnormal 0.5 * m. */
double oracle_e2m1_value(uint8_t code)
{
    const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* Nearest e2m1 code by the distance to each of the eight magnitudes, ties to
 * the code whose mantissa bit is 0; beyond 6 the largest magnitude. */
uint8_t oracle_e2m1_encode(float v)
{
    if (isnan(v)) return 0;
    const uint8_t sign = signbit(v) ? 8 : 0;
    const double a = fabs((double)v);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        const double dd = fabs(a - oracle_e2m1_value((uint8_t)c));
        if (dd < bd || (dd == bd && (c & 1) == 0 && (best & 1) == 1)) {
            bd = dd;
            best = c;
        }
    }
    return sign | (uint8_t)best;
}

void oracle_quantize_row_nvfp4(int n, const float* x, uint8_t* codes, uint8_t* bscale, float* scale)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const float s = amax > 0.0f ? amax / 2688.0f : 1.0f;
    for (int i = 0; i < n / 2; ++i) codes[i] = 0;
    for (int j = 0; j < n / 16; ++j) {
        float bmax = 0.0f;
        for (int i = 16 * j; i < 16 * j + 16; ++i) bmax = fmaxf(bmax, fabsf(x[i]));
        const float t = bmax / s;
        const float u = t / 6.0f;
        const uint8_t b = oracle_e4m3_encode(u);
        bscale[j] = b;
        const float den = (float)oracle_e4m3_value(b) * s;
        for (int i = 16 * j; i < 16 * j + 16; ++i) {
            const uint8_t c = den > 0.0f ? oracle_e2m1_encode(x[i] / den) : 0;
            codes[i / 2] |= (uint8_t)(c << (4 * (i & 1)));
        }
    }
    *scale = s;
}

static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* One expert's weight matrix: bf16 bits, e4m3 codes with one scale per row,
 * or packed e2m1 codes with e4m3 scales per 16 elements and one per row. */
typedef struct {
    const uint16_t* bf;
    const uint8_t* q;
    const float* s;
    size_t cols;
    const uint8_t* q4;
    const uint8_t* bs;
} Wmat;

/* The values of all 16 e2m1 and all 256 e4m3 codes, filled from the two
 * decoders (oracle_init_tables), so that a quantised weight costs table reads
 * instead of a decode. */
static double e2m1_tab[16], e4m3_tab[256];
static int tabs_ready = 0;

static void fill_tabs(void)
{
    if (tabs_ready) return;
    for (int c = 0; c < 16; ++c) e2m1_tab[c] = oracle_e2m1_value((uint8_t)c);
    for (int c = 0; c < 256; ++c) e4m3_tab[c] = oracle_e4m3_value((uint8_t)c);
    tabs_ready = 1;
}

void oracle_init_tables(void) { fill_tabs(); }

static double wval(const Wmat* w, size_t r, size_t c)
{
    if (w->bf) return (double)bf16_to_f32(w->bf[r * w->cols + c]);
    if (w->q4) {
        const size_t i = r * w->cols + c;
        const uint8_t code = (uint8_t)((w->q4[i / 2] >> (4 * (i & 1))) & 15);
        return e2m1_tab[code] * e4m3_tab[w->bs[(r * w->cols + c) / 16]] * (double)w->s[r];
    }
    return e4m3_tab[w->q[r * w->cols + c]] * (double)w->s[r];
}

int64_t oracle_capacity(int64_t T, int k, int E, double cf, int64_t explicit_cap)
{
    if (explicit_cap > 0) return explicit_cap;
    if (T <= 0 || k <= 0 || E <= 0 || !(cf > 0.0)) return 0;
    /* cf as an exact decimal: cf = cf_micro / 10^6. */
    int64_t cf_micro = llround(cf * 1e6);
    int64_t num = T * (int64_t)k * cf_micro;
    int64_t den = (int64_t)E * 1000000;
    return (num + den - 1) / den;
}

/* Score order used everywhere: a ranks before b when s_a > s_b, or when the
 * scores are equal and a has the lower index.  -0.0 and +0.0 compare equal. */
static int ranks_before(float sa, int a, float sb, int b)
{
    if (sa > sb) return 1;
    if (sa < sb) return 0;
    return a < b;
}

int oracle_preference(int E, const float* s_row, int32_t* order)
{
    for (int e = 0; e < E; ++e)
        if (isnan(s_row[e])) return 5;
    /* insertion sort by the score order */
    for (int e = 0; e < E; ++e) {
        int pos = e;
        while (pos > 0 && ranks_before(s_row[e], e, s_row[order[pos - 1]], order[pos - 1])) {
            order[pos] = order[pos - 1];
            --pos;
        }
        order[pos] = e;
    }
    return 0;
}

/* Softmax of one row of scores, in double.  Limits: when the largest score is
 * +inf the mass is shared equally by the +inf entries; when every score is
 * -inf the distribution is uniform. */
static void softmax_row(int E, const float* s, double* p)
{
    double m = -INFINITY;
    for (int e = 0; e < E; ++e)
        if ((double)s[e] > m) m = (double)s[e];
    if (isinf(m)) {
        int n = 0;
        for (int e = 0; e < E; ++e) n += ((double)s[e] == m);
        for (int e = 0; e < E; ++e) p[e] = ((double)s[e] == m) ? 1.0 / n : 0.0;
        return;
    }
    double z = 0.0;
    for (int e = 0; e < E; ++e) {
        p[e] = exp((double)s[e] - m);
        z += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= z;
}

int oracle_route(int T, int d, int E, int k, const uint16_t* h, const uint16_t* wr,
                 const float* bias, const float* usage, float lambda, float tau,
                 const float* logits_in, float* logits, float* scores, int32_t* ids,
                 float* topk_p, int32_t* counts_pre, float* f, float* P)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E) return 1;
    if (!(tau > 0.0f) || isinf(tau)) return 1;
    if (!logits_in && (d <= 0 || !h || !wr)) return 1;

    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double* psum = (double*)calloc((size_t)E, sizeof(double));
    int status = 0;
    for (int e = 0; e < E; ++e) counts_pre[e] = 0;

    for (int t = 0; t < T && status == 0; ++t) {
        float* z = logits + (size_t)t * E;
        float* s = scores + (size_t)t * E;
        /* step 1: z = h_t . W_router (+ b) */
        for (int e = 0; e < E; ++e) {
            if (logits_in) {
                z[e] = logits_in[(size_t)t * E + e];
            } else {
                double acc = 0.0;
                const uint16_t* ht = h + (size_t)t * d;
                const uint16_t* we = wr + (size_t)e * d;
                for (int i = 0; i < d; ++i)
                    acc += (double)bf16_to_f32(ht[i]) * (double)bf16_to_f32(we[i]);
                if (bias) acc += (double)bias[e];
                z[e] = (float)acc;
            }
        }
        /* step 2: s = fl(z / tau) - fl(lambda * usage), fp32, no FMA; the
         * temperature divides the scores before the penalty is taken off */
        for (int e = 0; e < E; ++e) {
            volatile float zt = z[e] / tau;
            if (!usage || lambda == 0.0f) {
                s[e] = zt;
            } else {
                volatile float pen = lambda * usage[e];
                s[e] = zt - pen;
            }
        }
        /* step 3: preference order, top-k ids, softmax probabilities */
        if (oracle_preference(E, s, order)) { status = 5; break; }
        softmax_row(E, s, p);
        for (int r = 0; r < k; ++r) {
            ids[(size_t)t * k + r] = order[r];
            topk_p[(size_t)t * k + r] = (float)p[order[r]];
            counts_pre[order[r]] += 1;
        }
        for (int e = 0; e < E; ++e) psum[e] += p[e];
    }
    /* step 4: f_i = counts_pre_i / T, P_i = mean over tokens of p_i */
    for (int e = 0; e < E; ++e) {
        f[e] = T > 0 ? (float)((double)counts_pre[e] / (double)T) : 0.0f;
        P[e] = T > 0 ? (float)(psum[e] / (double)T) : 0.0f;
    }
    free(order);
    free(p);
    free(psum);
    return status;
}

int oracle_router_logits(int T, int d, int E, int hidden, int norm, float eps,
                         const uint16_t* h, const float* gamma, const float* beta,
                         const uint16_t* w, const uint16_t* w2, const float* bias,
                         float* logits)
{
    if (T < 0 || d <= 0 || E <= 0 || hidden < 0 || norm < 0 || norm > 2 || !(eps >= 0.0f)) return 1;
    if (!h || !w || !logits || (hidden > 0 && !w2)) return 1;
    double* x = (double*)malloc(sizeof(double) * (size_t)d);
    double* a = (double*)malloc(sizeof(double) * (size_t)(hidden > 0 ? hidden : 1));
    for (int t = 0; t < T; ++t) {
        const uint16_t* ht = h + (size_t)t * d;
        for (int i = 0; i < d; ++i) x[i] = (double)bf16_to_f32(ht[i]);
        if (norm == 1) {
            /* LayerNorm over the row: mean, mean squared deviation */
            double mean = 0.0, var = 0.0;
            for (int i = 0; i < d; ++i) mean += x[i];
            mean /= (double)d;
            for (int i = 0; i < d; ++i) var += (x[i] - mean) * (x[i] - mean);
            var /= (double)d;
            const double inv = 1.0 / sqrt(var + (double)eps);
            for (int i = 0; i < d; ++i)
                x[i] = (x[i] - mean) * inv * (gamma ? (double)gamma[i] : 1.0) + (beta ? (double)beta[i] : 0.0);
        } else if (norm == 2) {
            double ss = 0.0;
            for (int i = 0; i < d; ++i) ss += x[i] * x[i];
            double nrm = sqrt(ss);
            if (nrm < (double)eps) nrm = (double)eps;
            for (int i = 0; i < d; ++i) x[i] = nrm > 0.0 ? x[i] / nrm : 0.0;
        }
        float* zt = logits + (size_t)t * E;
        if (hidden == 0) {
            for (int e = 0; e < E; ++e) {
                double acc = 0.0;
                const uint16_t* we = w + (size_t)e * d;
                for (int i = 0; i < d; ++i) acc += x[i] * (double)bf16_to_f32(we[i]);
                if (bias) acc += (double)bias[e];
                zt[e] = (float)acc;
            }
        } else {
            for (int j = 0; j < hidden; ++j) {
                double u = 0.0;
                const uint16_t* wj = w + (size_t)j * d;
                for (int i = 0; i < d; ++i) u += x[i] * (double)bf16_to_f32(wj[i]);
                a[j] = u / (1.0 + exp(-u));
            }
            for (int e = 0; e < E; ++e) {
                double acc = 0.0;
                const uint16_t* we = w2 + (size_t)e * hidden;
                for (int j = 0; j < hidden; ++j) acc += a[j] * (double)bf16_to_f32(we[j]);
                if (bias) acc += (double)bias[e];
                zt[e] = (float)acc;
            }
        }
    }
    free(x);
    free(a);
    return 0;
}

int oracle_dispatch(int T, int E, int k, int64_t C, const float* scores,
                    int32_t* assign, int32_t* slot, uint8_t* flags, int32_t* counts,
                    int32_t* offsets, int32_t* perm, float* cw,
                    int32_t* n_rerouted, int32_t* n_dropped)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E || C < 0) return 1;
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)T * (size_t)E);
    int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    int status = 0;

    for (int t = 0; t < T; ++t)
        if (oracle_preference(E, scores + (size_t)t * E, order + (size_t)t * E)) { status = 5; break; }

    int32_t nre = 0, ndrop = 0;
    if (status == 0) {
        /* Rank-major, token-minor: every rank-0 choice before any rank-1 choice. */
        for (int r = 0; r < k; ++r) {
            for (int t = 0; t < T; ++t) {
                const int32_t* pi = order + (size_t)t * E;
                int32_t chosen = -1;
                /* The token's own pick is pi[r]; when that expert is full (or
                 * already serves this token) walk on to the next candidate. */
                for (int j = r; j < E && chosen < 0; ++j) {
                    int32_t e = pi[j];
                    if (fill[e] >= C) continue;
                    int held = 0;
                    for (int q = 0; q < r; ++q) held |= (assign[(size_t)t * k + q] == e);
                    if (held) continue;
                    chosen = e;
                }
                size_t idx = (size_t)t * k + r;
                if (chosen < 0) {
                    assign[idx] = -1;
                    slot[idx] = -1;
                    flags[idx] = 2;
                    ++ndrop;
                } else {
                    assign[idx] = chosen;
                    slot[idx] = (int32_t)fill[chosen];
                    fill[chosen] += 1;
                    flags[idx] = (chosen != pi[r]) ? 1 : 0;
                    nre += (chosen != pi[r]);
                }
            }
        }
        offsets[0] = 0;
        for (int e = 0; e < E; ++e) {
            counts[e] = (int32_t)fill[e];
            offsets[e + 1] = offsets[e] + counts[e];
        }
        for (int t = 0; t < T; ++t)
            for (int r = 0; r < k; ++r) {
                size_t idx = (size_t)t * k + r;
                if (assign[idx] >= 0) perm[offsets[assign[idx]] + slot[idx]] = (int32_t)idx;
            }
        /* Combine weights: softmax probability of the expert actually used,
         * renormalised over the token's kept experts. */
        for (int t = 0; t < T; ++t) {
            softmax_row(E, scores + (size_t)t * E, p);
            double tot = 0.0;
            for (int r = 0; r < k; ++r) {
                int32_t e = assign[(size_t)t * k + r];
                if (e >= 0) tot += p[e];
            }
            for (int r = 0; r < k; ++r) {
                int32_t e = assign[(size_t)t * k + r];
                cw[(size_t)t * k + r] = (e >= 0 && tot > 0.0) ? (float)(p[e] / tot) : 0.0f;
            }
        }
        *n_rerouted = nre;
        *n_dropped = ndrop;
    }
    free(order);
    free(fill);
    free(p);
    return status;
}

static double silu(double x) { return x / (1.0 + exp(-x)); }

/* A row replaced by its NVFP4 representation (oracle_quantize_row_nvfp4). */
static void nvfp4_row(int n, float* x, double* out)
{
    uint8_t* codes = (uint8_t*)malloc((size_t)n / 2 + 1);
    uint8_t* bs = (uint8_t*)malloc((size_t)n / 16 + 1);
    float sc = 1.0f;
    oracle_quantize_row_nvfp4(n, x, codes, bs, &sc);
    for (int i = 0; i < n; ++i)
        out[i] = oracle_e2m1_value((uint8_t)((codes[i / 2] >> (4 * (i & 1))) & 15)) *
                 oracle_e4m3_value(bs[i / 16]) * (double)sc;
    free(codes);
    free(bs);
}

/* y = W2 (silu(W1 x) * W3 x) in double; W1, W3 [F][d], W2 [d][F]. */
/* quant_act 1: x and a = silu(g)*u enter their products as per-row e4m3 codes
 * times the row scale (a first rounded to bf16, as it is stored); 2: as their
 * NVFP4 representation (a again rounded to bf16 first). */
static void expert_row_w(int d, int F, const uint16_t* x, const Wmat* w1, const Wmat* w3,
                         const Wmat* w2, int quant_act, double* y)
{
    double* xf = (double*)malloc(sizeof(double) * (size_t)d);
    double* a = (double*)malloc(sizeof(double) * (size_t)F);
    float* tmp = (float*)calloc((size_t)(d > F ? d : F), sizeof(float));
    uint8_t* codes = (uint8_t*)malloc((size_t)(d > F ? d : F));
    float sc = 1.0f;
    for (int i = 0; i < d; ++i) xf[i] = (double)bf16_to_f32(x[i]);
    if (quant_act == 1) {
        for (int i = 0; i < d; ++i) tmp[i] = (float)xf[i];
        oracle_quantize_row(d, tmp, codes, &sc);
        for (int i = 0; i < d; ++i) xf[i] = oracle_e4m3_value(codes[i]) * (double)sc;
    } else if (quant_act == 2) {
        for (int i = 0; i < d; ++i) tmp[i] = (float)xf[i];
        nvfp4_row(d, tmp, xf);
    }
    for (int j = 0; j < F; ++j) {
        double g = 0.0, u = 0.0;
        for (int i = 0; i < d; ++i) {
            g += wval(w1, (size_t)j, (size_t)i) * xf[i];
            u += wval(w3, (size_t)j, (size_t)i) * xf[i];
        }
        a[j] = silu(g) * u;
    }
    if (quant_act == 1) {
        for (int j = 0; j < F; ++j) tmp[j] = bf16_to_f32(f32_to_bf16_rne((float)a[j]));
        oracle_quantize_row(F, tmp, codes, &sc);
        for (int j = 0; j < F; ++j) a[j] = oracle_e4m3_value(codes[j]) * (double)sc;
    } else if (quant_act == 2) {
        for (int j = 0; j < F; ++j) tmp[j] = bf16_to_f32(f32_to_bf16_rne((float)a[j]));
        nvfp4_row(F, tmp, a);
    }
    free(tmp);
    free(codes);
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < F; ++j) acc += wval(w2, (size_t)i, (size_t)j) * a[j];
        y[i] = acc;
    }
    free(xf);
    free(a);
}

void oracle_expert_row(int d, int F, const uint16_t* x, const uint16_t* w1,
                       const uint16_t* w3, const uint16_t* w2, double* y)
{
    const Wmat m1 = {w1, NULL, NULL, (size_t)d, NULL, NULL}, m3 = {w3, NULL, NULL, (size_t)d, NULL, NULL},
               m2 = {w2, NULL, NULL, (size_t)F, NULL, NULL};
    expert_row_w(d, F, x, &m1, &m3, &m2, 0, y);
}

/* The weight matrices of expert e: bf16 (q1 == NULL), e4m3 codes + row
 * scales (b1 == NULL), or packed e2m1 codes + e4m3 block scales + row scales. */
typedef struct {
    const uint16_t *w1, *w3, *w2;
    const uint8_t *q1, *q3, *q2;
    const float *s1, *s3, *s2;
    int quant_act;
    const uint8_t *b1, *b3, *b2;
} ExpertSet;

static void expert_mats(const ExpertSet* x, int e, int d, int F, Wmat* m1, Wmat* m3, Wmat* m2)
{
    const size_t wsz = (size_t)F * d;
    if (!x->q1) {
        *m1 = (Wmat){x->w1 + (size_t)e * wsz, NULL, NULL, (size_t)d, NULL, NULL};
        *m3 = (Wmat){x->w3 + (size_t)e * wsz, NULL, NULL, (size_t)d, NULL, NULL};
        *m2 = (Wmat){x->w2 + (size_t)e * wsz, NULL, NULL, (size_t)F, NULL, NULL};
    } else if (x->b1) {
        *m1 = (Wmat){NULL, NULL, x->s1 + (size_t)e * F, (size_t)d, x->q1 + (size_t)e * wsz / 2, x->b1 + (size_t)e * wsz / 16};
        *m3 = (Wmat){NULL, NULL, x->s3 + (size_t)e * F, (size_t)d, x->q3 + (size_t)e * wsz / 2, x->b3 + (size_t)e * wsz / 16};
        *m2 = (Wmat){NULL, NULL, x->s2 + (size_t)e * d, (size_t)F, x->q2 + (size_t)e * wsz / 2, x->b2 + (size_t)e * wsz / 16};
    } else {
        *m1 = (Wmat){NULL, x->q1 + (size_t)e * wsz, x->s1 + (size_t)e * F, (size_t)d, NULL, NULL};
        *m3 = (Wmat){NULL, x->q3 + (size_t)e * wsz, x->s3 + (size_t)e * F, (size_t)d, NULL, NULL};
        *m2 = (Wmat){NULL, x->q2 + (size_t)e * wsz, x->s2 + (size_t)e * d, (size_t)F, NULL, NULL};
    }
}

static int combine_rows_x(int T, int d, int E, int k, int F, const uint16_t* h, const ExpertSet* W,
                          const int32_t* assign, const float* cw, const int32_t* tokens, int ntok,
                          float* out_rows)
{
    if (d <= 0 || F <= 0 || E <= 0 || k <= 0) return 1;
    double* y = (double*)malloc(sizeof(double) * (size_t)d);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < ntok; ++i) {
        int t = tokens[i];
        if (t < 0 || t >= T) { free(y); free(acc); return 1; }
        for (int c = 0; c < d; ++c) acc[c] = 0.0;
        for (int r = 0; r < k; ++r) {
            int32_t e = assign[(size_t)t * k + r];
            if (e < 0) continue;
            if (e >= E) { free(y); free(acc); return 1; }
            Wmat m1, m3, m2;
            expert_mats(W, e, d, F, &m1, &m3, &m2);
            expert_row_w(d, F, h + (size_t)t * d, &m1, &m3, &m2, W->quant_act, y);
            double w = (double)cw[(size_t)t * k + r];
            for (int c = 0; c < d; ++c) acc[c] += w * y[c];
        }
        for (int c = 0; c < d; ++c) out_rows[(size_t)i * d + c] = (float)acc[c];
    }
    free(y);
    free(acc);
    return 0;
}

int oracle_combine_rows(int T, int d, int E, int k, int F, const uint16_t* h,
                        const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                        const int32_t* assign, const float* cw,
                        const int32_t* tokens, int ntok, float* out_rows)
{
    const ExpertSet W = {w1, w3, w2, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL, NULL};
    return combine_rows_x(T, d, E, k, F, h, &W, assign, cw, tokens, ntok, out_rows);
}

int oracle_combine_rows_q8(int T, int d, int E, int k, int F, const uint16_t* h,
                           const uint8_t* q1, const float* s1, const uint8_t* q3, const float* s3,
                           const uint8_t* q2, const float* s2, int quant_act, const int32_t* assign,
                           const float* cw, const int32_t* tokens, int ntok, float* out_rows)
{
    const ExpertSet W = {NULL, NULL, NULL, q1, q3, q2, s1, s3, s2, quant_act ? 1 : 0, NULL, NULL, NULL};
    fill_tabs();
    return combine_rows_x(T, d, E, k, F, h, &W, assign, cw, tokens, ntok, out_rows);
}

static int expert_slots_x(int T, int d, int E, int k, int F, const uint16_t* h, const ExpertSet* W,
                          const int32_t* assign, const int32_t* perm, int row0, int row1, float* y_slots)
{
    if (d <= 0 || F <= 0 || E <= 0 || k <= 0 || row0 < 0 || row1 < row0) return 1;
    double* y = (double*)malloc(sizeof(double) * (size_t)d);
    for (int i = row0; i < row1; ++i) {
        int32_t idx = perm[i];
        int t = idx / k;
        if (t < 0 || t >= T) { free(y); return 1; }
        int32_t e = assign[idx];
        if (e < 0 || e >= E) { free(y); return 1; }
        Wmat m1, m3, m2;
        expert_mats(W, e, d, F, &m1, &m3, &m2);
        expert_row_w(d, F, h + (size_t)t * d, &m1, &m3, &m2, W->quant_act, y);
        for (int c = 0; c < d; ++c) y_slots[(size_t)(i - row0) * d + c] = (float)y[c];
    }
    free(y);
    return 0;
}

int oracle_expert_slots(int T, int d, int E, int k, int F, const uint16_t* h,
                        const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                        const int32_t* assign, const int32_t* perm,
                        int row0, int row1, float* y_slots)
{
    const ExpertSet W = {w1, w3, w2, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL, NULL};
    return expert_slots_x(T, d, E, k, F, h, &W, assign, perm, row0, row1, y_slots);
}

int oracle_expert_slots_q8(int T, int d, int E, int k, int F, const uint16_t* h,
                           const uint8_t* q1, const float* s1, const uint8_t* q3, const float* s3,
                           const uint8_t* q2, const float* s2, int quant_act, const int32_t* assign,
                           const int32_t* perm, int row0, int row1, float* y_slots)
{
    const ExpertSet W = {NULL, NULL, NULL, q1, q3, q2, s1, s3, s2, quant_act ? 1 : 0, NULL, NULL, NULL};
    fill_tabs();
    return expert_slots_x(T, d, E, k, F, h, &W, assign, perm, row0, row1, y_slots);
}

int oracle_combine_rows_q4(int T, int d, int E, int k, int F, const uint16_t* h,
                           const uint8_t* q1, const uint8_t* b1, const float* s1,
                           const uint8_t* q3, const uint8_t* b3, const float* s3,
                           const uint8_t* q2, const uint8_t* b2, const float* s2, int quant_act,
                           const int32_t* assign, const float* cw, const int32_t* tokens, int ntok,
                           float* out_rows)
{
    if (d % 16 != 0 || F % 16 != 0) return 1;
    const ExpertSet W = {NULL, NULL, NULL, q1, q3, q2, s1, s3, s2, quant_act ? 2 : 0, b1, b3, b2};
    fill_tabs();
    return combine_rows_x(T, d, E, k, F, h, &W, assign, cw, tokens, ntok, out_rows);
}

int oracle_expert_slots_q4(int T, int d, int E, int k, int F, const uint16_t* h,
                           const uint8_t* q1, const uint8_t* b1, const float* s1,
                           const uint8_t* q3, const uint8_t* b3, const float* s3,
                           const uint8_t* q2, const uint8_t* b2, const float* s2, int quant_act,
                           const int32_t* assign, const int32_t* perm, int row0, int row1,
                           float* y_slots)
{
    if (d % 16 != 0 || F % 16 != 0) return 1;
    const ExpertSet W = {NULL, NULL, NULL, q1, q3, q2, s1, s3, s2, quant_act ? 2 : 0, b1, b3, b2};
    fill_tabs();
    return expert_slots_x(T, d, E, k, F, h, &W, assign, perm, row0, row1, y_slots);
}

/* The layer's backward pass, in the order of the forward run backwards:
 * combine -> down projection -> SwiGLU -> gate and up projections for each
 * kept (t, r), then the combine weights -> renormalisation -> softmax ->
 * temperature -> router GEMM for each token. */
int oracle_layer_backward(int T, int d, int E, int k, int F, float tau, const uint16_t* h,
                          const uint16_t* wr, const uint16_t* w1, const uint16_t* w3,
                          const uint16_t* w2, const float* scores, const int32_t* assign,
                          const float* dout, const float* dP, double* dh, double* dwr,
                          double* dbias, double* dw1, double* dw3, double* dw2)
{
    if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || F <= 0) return 1;
    if (!(tau > 0.0f) || isinf(tau)) return 1;
    const size_t wsz = (size_t)F * d;
    memset(dh, 0, sizeof(double) * (size_t)T * d);
    memset(dwr, 0, sizeof(double) * (size_t)E * d);
    memset(dbias, 0, sizeof(double) * (size_t)E);
    memset(dw1, 0, sizeof(double) * E * wsz);
    memset(dw3, 0, sizeof(double) * E * wsz);
    memset(dw2, 0, sizeof(double) * E * wsz);
    double* x = (double*)malloc(sizeof(double) * (size_t)d);
    double* g = (double*)malloc(sizeof(double) * (size_t)F);
    double* u = (double*)malloc(sizeof(double) * (size_t)F);
    double* a = (double*)malloc(sizeof(double) * (size_t)F);
    double* da = (double*)malloc(sizeof(double) * (size_t)F);
    double* dy = (double*)malloc(sizeof(double) * (size_t)d);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double* dp = (double*)malloc(sizeof(double) * (size_t)E);
    double* cw = (double*)malloc(sizeof(double) * (size_t)k);
    double* dcw = (double*)malloc(sizeof(double) * (size_t)k);
    int status = 0;
    for (int t = 0; t < T && status == 0; ++t) {
        const uint16_t* ht = h + (size_t)t * d;
        const float* gt = dout + (size_t)t * d;
        for (int i = 0; i < d; ++i) x[i] = (double)bf16_to_f32(ht[i]);
        softmax_row(E, scores + (size_t)t * E, p);
        /* the renormalised combine weights of t's kept ranks */
        double S = 0.0;
        for (int r = 0; r < k; ++r) {
            const int32_t e = assign[(size_t)t * k + r];
            if (e < -1 || e >= E) { status = 1; break; }
            if (e >= 0) S += p[e];
        }
        if (status) break;
        for (int r = 0; r < k; ++r) {
            const int32_t e = assign[(size_t)t * k + r];
            cw[r] = (e >= 0 && S > 0.0) ? p[e] / S : 0.0;
            dcw[r] = 0.0;
            if (e < 0) continue;
            const uint16_t* W1 = w1 + (size_t)e * wsz;
            const uint16_t* W3 = w3 + (size_t)e * wsz;
            const uint16_t* W2 = w2 + (size_t)e * wsz;
            /* forward of the expert: g, u, a = silu(g) * u, then dcw = dout . y */
            for (int j = 0; j < F; ++j) {
                double gg = 0.0, uu = 0.0;
                for (int i = 0; i < d; ++i) {
                    gg += (double)bf16_to_f32(W1[(size_t)j * d + i]) * x[i];
                    uu += (double)bf16_to_f32(W3[(size_t)j * d + i]) * x[i];
                }
                g[j] = gg;
                u[j] = uu;
                a[j] = silu(gg) * uu;
            }
            for (int c = 0; c < d; ++c) {
                double y = 0.0;
                for (int j = 0; j < F; ++j) y += (double)bf16_to_f32(W2[(size_t)c * F + j]) * a[j];
                dcw[r] += (double)gt[c] * y;
                dy[c] = cw[r] * (double)gt[c];
            }
            /* down projection: da = W2^T dy, dW2 += dy a^T */
            for (int j = 0; j < F; ++j) da[j] = 0.0;
            double* DW2 = dw2 + (size_t)e * wsz;
            for (int c = 0; c < d; ++c) {
                for (int j = 0; j < F; ++j) {
                    da[j] += (double)bf16_to_f32(W2[(size_t)c * F + j]) * dy[c];
                    DW2[(size_t)c * F + j] += dy[c] * a[j];
                }
            }
            /* SwiGLU: a = silu(g) u, silu'(g) = sig(g) (1 + g (1 - sig(g))) */
            double* DW1 = dw1 + (size_t)e * wsz;
            double* DW3 = dw3 + (size_t)e * wsz;
            for (int j = 0; j < F; ++j) {
                const double sg = 1.0 / (1.0 + exp(-g[j]));
                const double dg = da[j] * u[j] * sg * (1.0 + g[j] * (1.0 - sg));
                const double du = da[j] * silu(g[j]);
                for (int i = 0; i < d; ++i) {
                    dh[(size_t)t * d + i] += (double)bf16_to_f32(W1[(size_t)j * d + i]) * dg +
                                             (double)bf16_to_f32(W3[(size_t)j * d + i]) * du;
                    DW1[(size_t)j * d + i] += dg * x[i];
                    DW3[(size_t)j * d + i] += du * x[i];
                }
            }
        }
        /* combine weights -> probabilities: cw_r = p_{e_r} / S over the kept ranks */
        for (int e = 0; e < E; ++e) dp[e] = dP ? (double)dP[e] / (double)T : 0.0;
        if (S > 0.0) {
            double m = 0.0;
            for (int r = 0; r < k; ++r) m += dcw[r] * cw[r];
            for (int r = 0; r < k; ++r) {
                const int32_t e = assign[(size_t)t * k + r];
                if (e >= 0) dp[e] += (dcw[r] - m) / S;
            }
        }
        /* softmax, then s = z / tau - lambda * usage */
        double pd = 0.0;
        for (int e = 0; e < E; ++e) pd += p[e] * dp[e];
        for (int e = 0; e < E; ++e) {
            const double dz = p[e] * (dp[e] - pd) / (double)tau;
            dbias[e] += dz;
            const uint16_t* we = wr + (size_t)e * d;
            for (int i = 0; i < d; ++i) {
                dh[(size_t)t * d + i] += dz * (double)bf16_to_f32(we[i]);
                dwr[(size_t)e * d + i] += dz * x[i];
            }
        }
    }
    free(x); free(g); free(u); free(a); free(da); free(dy); free(p); free(dp); free(cw); free(dcw);
    return status;
}
