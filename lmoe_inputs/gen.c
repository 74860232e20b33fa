/*
 * Seeded synthetic inputs for the LatentMoE layer (test and benchmark data).
 *
 * This module produces the input tensors only: Gaussian activations and
 * weights of the shapes the layer is run on, and the expert-popularity logit
 * bias of the skewed-routing workload.  It holds none of the layer's own
 * arithmetic (no quantisation, routing, GEMM or combine), so both the CUDA
 * path and the CPU oracle can be fed byte-identical inputs from it.
 *
 * Generator: counter-based.  Element i of stream s under seed S is derived
 * from the SplitMix64 output function (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014; constants as
 * published by Vigna) applied to key(S, s) + (i + 1) * golden-gamma, so any
 * slice of any tensor can be generated independently and in parallel.
 * Normals come from the Box-Muller transform.  The logarithm, sine and cosine
 * it needs are evaluated here with plain series in IEEE double arithmetic
 * (compiled without FMA contraction), so every host architecture produces
 * the same bits.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return mix64(mix64(seed * GOLDEN_GAMMA + 0x632BE59BD9B4E019ULL) ^ (stream * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t ctr) { return mix64(key + (ctr + 1) * GOLDEN_GAMMA); }

/* Series coefficients, computed once by exact-as-possible double division
 * (the same IEEE operations on every host, so the same bits). */
static double g_inv_odd[16];     /* 1/(2j+1)          */
static double g_sin_c[13];       /* (-1)^k/(2k+1)!    */
static double g_cos_c[13];       /* (-1)^k/(2k)!      */
static pthread_once_t g_once = PTHREAD_ONCE_INIT;

static void init_tables(void)
{
    for (int j = 0; j < 16; ++j) g_inv_odd[j] = 1.0 / (double)(2 * j + 1);
    double f = 1.0; /* running factorial */
    for (int k = 0; k < 13; ++k) {
        double f_even = f;                      /* (2k)!   */
        double f_odd = f * (double)(2 * k + 1); /* (2k+1)! */
        g_cos_c[k] = ((k & 1) ? -1.0 : 1.0) / f_even;
        g_sin_c[k] = ((k & 1) ? -1.0 : 1.0) / f_odd;
        f = f_odd * (double)(2 * k + 2);
    }
}

/* Natural logarithm of a positive finite x: x = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * ln x = e ln 2 + 2 atanh((m-1)/(m+1)), atanh by its odd power series
 * (|s| <= 0.1716, 16 terms leave < 1e-24). */
static double det_log(double x)
{
    int e;
    double m = frexp(x, &e); /* m in [0.5, 1) */
    if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
    double s = (m - 1.0) / (m + 1.0);
    double s2 = s * s;
    double p = g_inv_odd[15];
    for (int j = 14; j >= 0; --j) p = p * s2 + g_inv_odd[j];
    return (double)e * 0.69314718055994530942 + 2.0 * s * p;
}

/* sin and cos of phi in [0, pi/2] by their Taylor polynomials (to phi^25 / phi^24). */
static void det_sincos_quarter(double phi, double *s, double *c)
{
    double p2 = phi * phi;
    double ps = g_sin_c[12], pc = g_cos_c[12];
    for (int k = 11; k >= 0; --k) {
        ps = ps * p2 + g_sin_c[k];
        pc = pc * p2 + g_cos_c[k];
    }
    *s = phi * ps;
    *c = pc;
}

/* sin and cos of 2*pi*u for u in [0, 1), reduced to a quarter turn exactly. */
static void det_sincos_turn(double u, double *s, double *c)
{
    double u4 = u * 4.0;
    int q = (int)u4;
    double f = u4 - (double)q; /* exact */
    double sq, cq;
    det_sincos_quarter(f * 1.57079632679489661923, &sq, &cq);
    switch (q & 3) {
    case 0: *s = sq; *c = cq; break;
    case 1: *s = cq; *c = -sq; break;
    case 2: *s = -sq; *c = -cq; break;
    default: *s = -cq; *c = sq; break;
    }
}

/* The Box-Muller pair number `pair` of a stream: standard normals 2*pair
 * (cosine branch) and 2*pair+1 (sine branch). */
static void normal_pair(uint64_t key, uint64_t pair, double *z0, double *z1)
{
    uint64_t r1 = draw(key, 2 * pair), r2 = draw(key, 2 * pair + 1);
    double u1 = ((double)(r1 >> 11) + 0.5) * (1.0 / 9007199254740992.0); /* (0,1) */
    double u2 = (double)(r2 >> 11) * (1.0 / 9007199254740992.0);         /* [0,1) */
    double rad = sqrt(-2.0 * det_log(u1));
    double s, c;
    det_sincos_turn(u2, &s, &c);
    *z0 = rad * c;
    *z1 = rad * s;
}

static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

typedef struct {
    uint64_t key, start, n;
    double sigma;
    int kind; /* 0 = f32, 1 = bf16 */
    void *out;
} job_t;

static void put(job_t *j, uint64_t i, double z)
{
    if (j->kind == 0) ((float *)j->out)[i] = (float)(j->sigma * z);
    else ((uint16_t *)j->out)[i] = f32_to_bf16_rne((float)(j->sigma * z));
}

static void *run_job(void *arg)
{
    job_t *j = (job_t *)arg;
    uint64_t i = 0;
    double z0, z1;
    if (j->n && (j->start & 1)) { /* leading odd element: sine branch of its pair */
        normal_pair(j->key, j->start >> 1, &z0, &z1);
        put(j, 0, z1);
        i = 1;
    }
    for (; i + 1 < j->n; i += 2) {
        normal_pair(j->key, (j->start + i) >> 1, &z0, &z1);
        put(j, i, z0);
        put(j, i + 1, z1);
    }
    if (i < j->n) {
        normal_pair(j->key, (j->start + i) >> 1, &z0, &z1);
        put(j, i, z0);
    }
    return NULL;
}

static void run_parallel(uint64_t key, uint64_t start, uint64_t n, double sigma, int kind, void *out, int threads)
{
    pthread_once(&g_once, init_tables);
    if (threads < 1) threads = 1;
    if (threads > 64) threads = 64;
    if (n < (1u << 16)) threads = 1;
    pthread_t tid[64];
    job_t jobs[64];
    uint64_t chunk = (n + (uint64_t)threads - 1) / (uint64_t)threads;
    int launched = 0;
    for (int t = 0; t < threads; ++t) {
        uint64_t b = (uint64_t)t * chunk;
        if (b >= n) break;
        uint64_t e = b + chunk < n ? b + chunk : n;
        size_t esz = kind == 0 ? 4 : 2;
        jobs[t] = (job_t){key, start + b, e - b, sigma, kind, (char *)out + b * esz};
        if (threads == 1 || pthread_create(&tid[t], NULL, run_job, &jobs[t]) != 0) {
            run_job(&jobs[t]);
            tid[t] = 0;
        }
        launched = t + 1;
    }
    for (int t = 0; t < launched; ++t)
        if (threads > 1 && tid[t]) pthread_join(tid[t], NULL);
}

/* out[i] = float(sigma * N_(start+i)) for i in [0, n). */
void lmoe_gen_normal_f32(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n, double sigma, float *out,
                         int threads)
{
    run_parallel(stream_key(seed, stream), start, n, sigma, 0, out, threads);
}

/* out[i] = bf16_rne(float(sigma * N_(start+i))) as raw bf16 bits. */
void lmoe_gen_normal_bf16(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n, double sigma, uint16_t *out,
                          int threads)
{
    run_parallel(stream_key(seed, stream), start, n, sigma, 1, out, threads);
}

/* Raw 64-bit draws (for tests of the generator itself). */
void lmoe_gen_raw_u64(uint64_t seed, uint64_t stream, uint64_t start, uint64_t n, uint64_t *out)
{
    uint64_t key = stream_key(seed, stream);
    for (uint64_t i = 0; i < n; ++i) out[i] = draw(key, start + i);
}

/* The deterministic log / sincos used by Box-Muller, exposed for tests. */
double lmoe_gen_det_log(double x)
{
    pthread_once(&g_once, init_tables);
    return det_log(x);
}

void lmoe_gen_det_sincos_turn(double u, double *s, double *c)
{
    pthread_once(&g_once, init_tables);
    det_sincos_turn(u, s, c);
}

/* exp(y) for finite y: y = n ln2 + f with |f| <= ln2/2, exp(f) by Taylor series,
 * then an exact power-of-two scaling. */
static double det_exp(double y)
{
    /* ln 2 split in a high part with trailing zero bits (n * hi is exact) and a
     * low correction (Cody and Waite's reduction). */
    double n = floor(y / 0.69314718055994530942 + 0.5);
    double f = (y - n * 6.93147180369123816490e-01) - n * 1.90821492927058770002e-10;
    double term = 1.0, sum = 0.0;
    for (int k = 1; k <= 24; ++k) { sum += term; term *= f / (double)k; }
    return ldexp(sum, (int)n);
}

/* Expert-popularity logit bias of the skewed-routing workload:
 * bias[e] = beta * ln p(e), p(e) = (e+1)^-s / sum_r r^-s over the E experts
 * (Zipf law with exponent s; expert e has popularity rank e+1). */
void lmoe_gen_zipf_bias(int E, double s, double beta, float *bias)
{
    pthread_once(&g_once, init_tables);
    double z = 0.0;
    for (int r = 1; r <= E; ++r) z += det_exp(-s * det_log((double)r));
    double lnz = det_log(z);
    for (int e = 0; e < E; ++e) bias[e] = (float)(beta * (-s * det_log((double)(e + 1)) - lnz));
}

double lmoe_gen_det_exp(double y) { return det_exp(y); }
