/*
 * CPU oracle of the LatentMoE layer forward pass -- TEST INFRASTRUCTURE ONLY.
 * (Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * use this file; see lmoe_oracle.h for the sources and formats.)
 *
 * Everything is evaluated in double precision, one thread, in the order the
 * layer is defined.  Rounding happens only where the definition quantises:
 * router logits are fp32, the gate weights are fp32, activations entering an
 * expert GEMM are MXFP8 (x and the gated product h), and the layer output is
 * bf16.
 */
#include "lmoe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* element codecs                                                            */
/* ------------------------------------------------------------------------ */

/* e2m1 magnitude grid, codes 0..7 (OCP microscaling FP4: 2 exponent bits with
 * bias 1, 1 mantissa bit; code 1 is the subnormal 0.5). */
double oracle_e2m1_value(uint8_t code)
{
    int sgn = (code >> 3) & 1, ex = (code >> 1) & 3, man = code & 1;
    double mag = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);
    return sgn ? -mag : mag;
}

/* e4m3 (OCP FP8 E4M3, "fn" variant): bias 7, subnormals for exponent 0,
 * S.1111.111 is NaN, no infinities. */
double oracle_e4m3_value(uint8_t code)
{
    int sgn = (code >> 7) & 1, ex = (code >> 3) & 15, man = code & 7;
    double mag;
    if (ex == 15 && man == 7) return NAN;
    if (ex == 0) mag = ldexp((double)man / 8.0, -6);
    else mag = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return sgn ? -mag : mag;
}

double oracle_e8m0_value(uint8_t s) { return s == 255 ? NAN : ldexp(1.0, (int)s - 127); }

/* Round-to-nearest-even onto an ascending magnitude grid indexed by code:
 * the nearest grid point; on an exact tie the point with the even code
 * (= even mantissa, since the mantissa is the low code bits); beyond the
 * last point, saturate to it. */
static int nearest_even_on_grid(double a, const double *grid, int n)
{
    if (a >= grid[n - 1]) return n - 1;
    int lo = 0, hi = n - 1; /* grid[lo] <= a < grid[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (grid[mid] <= a) lo = mid;
        else hi = mid;
    }
    double dl = a - grid[lo], dh = grid[hi] - a;
    if (dl < dh) return lo;
    if (dh < dl) return hi;
    return (lo % 2 == 0) ? lo : hi;
}

static double g_e2m1_grid[8];
static double g_e4m3_grid[127]; /* codes 0x00..0x7E */
static int g_grids_ready = 0;

static void init_grids(void)
{
    if (g_grids_ready) return;
    for (int c = 0; c < 8; ++c) g_e2m1_grid[c] = oracle_e2m1_value((uint8_t)c);
    for (int c = 0; c < 127; ++c) g_e4m3_grid[c] = oracle_e4m3_value((uint8_t)c);
    g_grids_ready = 1;
}

uint8_t oracle_e2m1_encode(double v)
{
    init_grids();
    int sgn = signbit(v) ? 1 : 0;
    int c = nearest_even_on_grid(fabs(v), g_e2m1_grid, 8);
    return (uint8_t)((sgn << 3) | c);
}

uint8_t oracle_e4m3_encode(double v)
{
    init_grids();
    int sgn = signbit(v) ? 1 : 0;
    int c = nearest_even_on_grid(fabs(v), g_e4m3_grid, 127);
    return (uint8_t)((sgn << 7) | c);
}

/* Shared exponent of a block (OCP MX): X = floor(log2 amax) - emax, where emax
 * is the exponent of the element format's largest normal (2 for e2m1, 8 for
 * e4m3); stored as the e8m0 byte X + 127, clamped to [0, 254]. */
uint8_t oracle_scale_byte(double amax, int emax)
{
    if (amax == 0.0) return 0;
    int e;
    frexp(amax, &e); /* amax = m * 2^e, m in [0.5, 1) => floor(log2 amax) = e - 1 */
    int X = (e - 1) - emax;
    int b = X + 127;
    if (b < 0) b = 0;
    if (b > 254) b = 254;
    return (uint8_t)b;
}

/* ------------------------------------------------------------------------ */
/* block quantisation                                                        */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static uint16_t double_to_bf16(double v)
{
    /* bf16 round-to-nearest-even of the exact value v: first to the nearest
     * bf16 directly from double (no double rounding through fp32). */
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int sgn = signbit(v) ? 1 : 0;
    double a = fabs(v);
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e) */
    int ulp_exp = (e - 1) - 7;           /* 8 significant bits */
    if (ulp_exp < -133) ulp_exp = -133;  /* bf16 subnormal spacing 2^-133 */
    double q = a / ldexp(1.0, ulp_exp);  /* exact */
    double fl = floor(q), fr = q - fl;
    double r = fl;
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) != 0.0)) r = fl + 1.0;
    double res = r * ldexp(1.0, ulp_exp);
    float f = (float)res; /* exact: res is a bf16 value (or overflows to inf) */
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t out = (uint16_t)(u >> 16);
    if (sgn) out |= 0x8000;
    return out;
}

void oracle_round_bf16(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(v[i]);
}

void oracle_quant_mxfp4(const float *w, int64_t rows, int K, uint8_t *q, uint8_t *s)
{
    const int nb = K / 32;
    for (int64_t r = 0; r < rows; ++r) {
        memset(q + r * (K / 2), 0, (size_t)(K / 2));
        for (int b = 0; b < nb; ++b) {
            const float *blk = w + r * K + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs((double)blk[i]));
            uint8_t sb = oracle_scale_byte(amax, 2);
            s[r * nb + b] = sb;
            for (int i = 0; i < 32; ++i) {
                double v = ldexp((double)blk[i], 127 - (int)sb); /* blk[i] / 2^(sb-127), exact */
                uint8_t c = oracle_e2m1_encode(v);
                int col = b * 32 + i;
                q[r * (K / 2) + col / 2] |= (uint8_t)(c << (4 * (col & 1)));
            }
        }
    }
}

void oracle_quant_mxfp8_f64(const double *x, int64_t rows, int K, uint8_t *q, uint8_t *s)
{
    const int nb = K / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            const double *blk = x + r * K + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(blk[i]));
            uint8_t sb = oracle_scale_byte(amax, 8);
            s[r * nb + b] = sb;
            for (int i = 0; i < 32; ++i) q[r * K + b * 32 + i] = oracle_e4m3_encode(ldexp(blk[i], 127 - (int)sb));
        }
}

void oracle_quant_mxfp4_f64(const double *x, int64_t rows, int K, uint8_t *q, uint8_t *s)
{
    const int nb = K / 32;
    for (int64_t r = 0; r < rows; ++r) {
        memset(q + r * (K / 2), 0, (size_t)(K / 2));
        for (int b = 0; b < nb; ++b) {
            const double *blk = x + r * K + b * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs(blk[i]));
            uint8_t sb = oracle_scale_byte(amax, 2);
            s[r * nb + b] = sb;
            for (int i = 0; i < 32; ++i) {
                uint8_t c = oracle_e2m1_encode(ldexp(blk[i], 127 - (int)sb));
                int col = b * 32 + i;
                q[r * (K / 2) + col / 2] |= (uint8_t)(c << (4 * (col & 1)));
            }
        }
    }
}

void oracle_quant_mxfp8(const uint16_t *x_bf16, int64_t rows, int K, uint8_t *q, uint8_t *s)
{
    double *tmp = (double *)malloc(sizeof(double) * (size_t)K);
    for (int64_t r = 0; r < rows; ++r) {
        for (int c = 0; c < K; ++c) tmp[c] = bf16_to_double(x_bf16[r * K + c]);
        oracle_quant_mxfp8_f64(tmp, 1, K, q + r * K, s + r * (K / 32));
    }
    free(tmp);
}

void oracle_dequant_mxfp4(const uint8_t *q, const uint8_t *s, int64_t rows, int K, double *out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int c = 0; c < K; ++c) {
            uint8_t code = (q[r * (K / 2) + c / 2] >> (4 * (c & 1))) & 15;
            out[r * K + c] = oracle_e2m1_value(code) * oracle_e8m0_value(s[r * (K / 32) + c / 32]);
        }
}

void oracle_dequant_mxfp8(const uint8_t *q, const uint8_t *s, int64_t rows, int K, double *out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int c = 0; c < K; ++c)
            out[r * K + c] = oracle_e4m3_value(q[r * K + c]) * oracle_e8m0_value(s[r * (K / 32) + c / 32]);
}

/* ------------------------------------------------------------------------ */
/* routing  [P2-MoE]                                                         */
/* ------------------------------------------------------------------------ */

/* logits[t][e] = fp32( sum_c x[t][c] * Wr[e][c] ) (+ bias[e] in fp32). */
void oracle_router_logits(const uint16_t *x_bf16, const float *Wr, const float *bias, int T, int d, int E,
                          float *logits)
{
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += bf16_to_double(x_bf16[(int64_t)t * d + c]) * (double)Wr[(int64_t)e * d + c];
            float l = (float)acc;
            if (bias) l = l + bias[e];
            logits[(int64_t)t * E + e] = l;
        }
}

/* Slot j holds the best expert not chosen in slots 0..j-1, "best" meaning the
 * larger logit, and on equal logits the smaller expert id.  The gate weights
 * are the softmax over the k chosen logits. */
void oracle_topk_softmax(const float *logits, int T, int E, int k, int32_t *idx, float *w)
{
    char *taken = (char *)malloc((size_t)E);
    double *ex = (double *)malloc(sizeof(double) * (size_t)k);
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (int64_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict: equal keeps the smaller id */
            }
            taken[best] = 1;
            idx[(int64_t)t * k + j] = best;
        }
        double l0 = (double)l[idx[(int64_t)t * k]], sum = 0.0;
        for (int j = 0; j < k; ++j) {
            ex[j] = exp((double)l[idx[(int64_t)t * k + j]] - l0);
            sum += ex[j];
        }
        for (int j = 0; j < k; ++j) w[(int64_t)t * k + j] = (float)(ex[j] / sum);
    }
    free(taken);
    free(ex);
}

/* Counting sort of the pair ids p = t*k + j by expert [P3-EP dispatch]:
 * counts[e], offsets = exclusive prefix sum (E+1 entries), perm lists the
 * pairs of expert 0, then expert 1, ..., each group in ascending p, and
 * inv[p] is the position of pair p in perm. */
void oracle_permute(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                    int32_t *inv)
{
    const int64_t P = (int64_t)T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) counts[idx[p]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int64_t p = 0; p < P; ++p) {
        int e = idx[p];
        int32_t pos = offsets[e] + fill[e]++;
        perm[pos] = (int32_t)p;
        inv[p] = pos;
    }
    free(fill);
}

/* ------------------------------------------------------------------------ */
/* experts and combine  [P1-A], [P1-L1], [P2-MX], [P3-EP combine]            */
/* ------------------------------------------------------------------------ */

static double mxfp4_elem(const uint8_t *q, const uint8_t *s, int64_t row, int K, int c)
{
    uint8_t code = (q[row * (K / 2) + c / 2] >> (4 * (c & 1))) & 15;
    return oracle_e2m1_value(code) * oracle_e8m0_value(s[row * (K / 32) + c / 32]);
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* xhat: the token's MXFP8-decoded activation (d values). */
static void expert_ffn(const double *xhat, const oracle_experts *W, int e, int d, int I, double *out)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    uint8_t *hq = (uint8_t *)malloc((size_t)I);
    uint8_t *hs = (uint8_t *)malloc((size_t)(I / 32));
    double *hhat = (double *)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        int64_t row = (int64_t)e * I + i;
        double g = 0.0, u = 0.0;
        for (int c = 0; c < d; ++c) {
            g += mxfp4_elem(W->gate_q, W->gate_s, row, d, c) * xhat[c];
            u += mxfp4_elem(W->up_q, W->up_s, row, d, c) * xhat[c];
        }
        h[i] = silu(g) * u;
    }
    oracle_quant_mxfp8_f64(h, 1, I, hq, hs);
    oracle_dequant_mxfp8(hq, hs, 1, I, hhat);
    for (int o = 0; o < d; ++o) {
        int64_t row = (int64_t)e * d + o;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += mxfp4_elem(W->down_q, W->down_s, row, I, i) * hhat[i];
        out[o] = acc;
    }
    free(h);
    free(hq);
    free(hs);
    free(hhat);
}

static void token_xhat(const uint16_t *x_row, int d, double *xhat)
{
    uint8_t *xq = (uint8_t *)malloc((size_t)d);
    uint8_t *xs = (uint8_t *)malloc((size_t)(d / 32));
    oracle_quant_mxfp8(x_row, 1, d, xq, xs);
    oracle_dequant_mxfp8(xq, xs, 1, d, xhat);
    free(xq);
    free(xs);
}

void oracle_expert_ffn_token(const uint16_t *x_bf16_row, const oracle_experts *W, int e, int d, int I, double *out)
{
    double *xhat = (double *)malloc(sizeof(double) * (size_t)d);
    token_xhat(x_bf16_row, d, xhat);
    expert_ffn(xhat, W, e, d, I, out);
    free(xhat);
}

void oracle_moe_tokens(const uint16_t *x_bf16, const int32_t *idx, const float *w, const oracle_experts *W, int T,
                       int d, int E, int k, int I, const int32_t *tokens, int ntok, uint16_t *y_bf16, double *y_f64)
{
    (void)E;
    if (!tokens) ntok = T;
    double *xhat = (double *)malloc(sizeof(double) * (size_t)d);
    double *f = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int n = 0; n < ntok; ++n) {
        int t = tokens ? tokens[n] : n;
        token_xhat(x_bf16 + (int64_t)t * d, d, xhat);
        for (int o = 0; o < d; ++o) y[o] = 0.0;
        for (int j = 0; j < k; ++j) { /* slot order */
            int e = idx[(int64_t)t * k + j];
            double wj = (double)w[(int64_t)t * k + j];
            expert_ffn(xhat, W, e, d, I, f);
            for (int o = 0; o < d; ++o) y[o] += wj * f[o];
        }
        for (int o = 0; o < d; ++o) {
            if (y_bf16) y_bf16[(int64_t)n * d + o] = double_to_bf16(y[o]);
            if (y_f64) y_f64[(int64_t)n * d + o] = y[o];
        }
    }
    free(xhat);
    free(f);
    free(y);
}

/* The activation rounding of the FP4 mode: values -> MXFP4 -> decoded. */
static void round_mxfp4(const double *v, int K, double *out)
{
    uint8_t *q = (uint8_t *)malloc((size_t)(K / 2));
    uint8_t *s = (uint8_t *)malloc((size_t)(K / 32));
    oracle_quant_mxfp4_f64(v, 1, K, q, s);
    oracle_dequant_mxfp4(q, s, 1, K, out);
    free(q);
    free(s);
}

/* One expert's FFN on a decoded activation, FP4 mode: h rounded to MXFP4. */
static void expert_ffn_fp4(const double *xhat, const oracle_experts *W, int e, int d, int I, double *out)
{
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    double *hhat = (double *)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        int64_t row = (int64_t)e * I + i;
        double g = 0.0, u = 0.0;
        for (int c = 0; c < d; ++c) {
            g += mxfp4_elem(W->gate_q, W->gate_s, row, d, c) * xhat[c];
            u += mxfp4_elem(W->up_q, W->up_s, row, d, c) * xhat[c];
        }
        h[i] = silu(g) * u;
    }
    round_mxfp4(h, I, hhat);
    for (int o = 0; o < d; ++o) {
        int64_t row = (int64_t)e * d + o;
        double acc = 0.0;
        for (int i = 0; i < I; ++i) acc += mxfp4_elem(W->down_q, W->down_s, row, I, i) * hhat[i];
        out[o] = acc;
    }
    free(h);
    free(hhat);
}

void oracle_moe_tokens_act(const uint16_t *x_bf16, const int32_t *idx, const float *w, const oracle_experts *W,
                           int T, int d, int E, int k, int I, const int32_t *tokens, int ntok, int act,
                           uint16_t *y_bf16, double *y_f64)
{
    if (act != ORACLE_ACT_MXFP4) {
        oracle_moe_tokens(x_bf16, idx, w, W, T, d, E, k, I, tokens, ntok, y_bf16, y_f64);
        return;
    }
    if (!tokens) ntok = T;
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *xhat = (double *)malloc(sizeof(double) * (size_t)d);
    double *f = (double *)malloc(sizeof(double) * (size_t)d);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int n = 0; n < ntok; ++n) {
        int t = tokens ? tokens[n] : n;
        for (int c = 0; c < d; ++c) xv[c] = bf16_to_double(x_bf16[(int64_t)t * d + c]);
        round_mxfp4(xv, d, xhat);
        for (int o = 0; o < d; ++o) y[o] = 0.0;
        for (int j = 0; j < k; ++j) { /* slot order */
            int e = idx[(int64_t)t * k + j];
            double wj = (double)w[(int64_t)t * k + j];
            expert_ffn_fp4(xhat, W, e, d, I, f);
            for (int o = 0; o < d; ++o) y[o] += wj * f[o];
        }
        for (int o = 0; o < d; ++o) {
            if (y_bf16) y_bf16[(int64_t)n * d + o] = double_to_bf16(y[o]);
            if (y_f64) y_f64[(int64_t)n * d + o] = y[o];
        }
    }
    (void)E;
    free(xv);
    free(xhat);
    free(f);
    free(y);
}

void oracle_moe_dense(const uint16_t *x_bf16, const int32_t *idx, const float *w, const oracle_experts *W, int T,
                      int d, int E, int k, int I, const int32_t *tokens, int ntok, double *y_f64)
{
    if (!tokens) ntok = T;
    double *xhat = (double *)malloc(sizeof(double) * (size_t)d);
    double *f = (double *)malloc(sizeof(double) * (size_t)d);
    double *gate = (double *)malloc(sizeof(double) * (size_t)E);
    for (int n = 0; n < ntok; ++n) {
        int t = tokens ? tokens[n] : n;
        token_xhat(x_bf16 + (int64_t)t * d, d, xhat);
        for (int e = 0; e < E; ++e) gate[e] = 0.0;
        for (int j = 0; j < k; ++j) gate[idx[(int64_t)t * k + j]] = (double)w[(int64_t)t * k + j];
        double *y = y_f64 + (int64_t)n * d;
        for (int o = 0; o < d; ++o) y[o] = 0.0;
        for (int e = 0; e < E; ++e) {
            expert_ffn(xhat, W, e, d, I, f);
            for (int o = 0; o < d; ++o) y[o] += gate[e] * f[o];
        }
    }
    free(xhat);
    free(f);
    free(gate);
}

void oracle_linear_bf16(const uint16_t *x, const uint16_t *W, int64_t rows, int K, int N, uint16_t *out)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += bf16_to_double(x[r * K + c]) * bf16_to_double(W[(int64_t)n * K + c]);
            out[r * N + n] = double_to_bf16(acc);
        }
}
