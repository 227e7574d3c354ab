/*
 * Seeded synthetic inputs for the split GEMV + one-shot all-reduce workloads.
 *
 * This module only produces input values.  It holds none of the arithmetic of
 * the method (no products, no reductions, no output rounding); both the CPU
 * oracle and the GPU path receive the bf16 words written here.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast Splittable Pseudorandom
 * Number Generators", OOPSLA 2014), used in counter form: the i-th output of a
 * stream whose state starts at `base` is mix(base + (i + 1) * GAMMA).  Every
 * element is therefore a pure function of (base, i) and threads may split the
 * index range freely without changing any value.
 *
 * Normals: Box-Muller transform (Box & Muller, 1958) on consecutive pairs of
 * 53-bit uniforms; element 2j takes the cosine branch of pair j, element 2j+1
 * the sine branch.
 *
 * Every value is formed in fp64 and rounded once to bf16, round to nearest,
 * ties to even.  Compile with -ffp-contract=off so that fp64 values do not
 * depend on whether the host contracts a*b+c into a fused multiply-add.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t sm64_at(uint64_t base, uint64_t i) {
    return sm64_mix(base + (i + 1) * SM64_GAMMA);
}

/* Start state of the stream for (seed, tag).  Tags separate the tensors of
 * one workload (W, x, the two SiLU operands, the outlier permutation, ...). */
uint64_t synth_stream_base(uint64_t seed, uint32_t tag) {
    return sm64_mix(seed * 0x100000001B3ULL ^ ((uint64_t)tag << 40) ^ 0x5851F42D4C957F2DULL);
}

uint64_t synth_u64(uint64_t base, uint64_t i) { return sm64_at(base, i); }

/* [0, 1) with 53 random bits. */
static inline double u53(uint64_t z) { return (double)(z >> 11) * 0x1.0p-53; }

/* Pair j of standard normals (Box-Muller); u1 is moved into (0, 1]. */
static inline void normal_pair(uint64_t base, uint64_t j, double *c, double *s) {
    double u1 = 1.0 - u53(sm64_at(base, 2 * j));
    double u2 = u53(sm64_at(base, 2 * j + 1));
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586476925286766559 * u2;
    *c = rad * cos(ang);
    *s = rad * sin(ang);
}

/* fp64 -> bf16 bits, round to nearest even, by scaling onto the integer grid
 * of the bf16 quantum and calling nearbyint (default rounding mode: ties to
 * even).  The scaling is by powers of two and therefore exact. */
uint16_t synth_round_bf16(double d) {
    uint16_t sign = signbit(d) ? 0x8000u : 0u;
    double a = fabs(d);
    if (isnan(d)) return (uint16_t)(sign | 0x7FC0u);
    if (isinf(d)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);            /* a = f * 2^e, 0.5 <= f < 1 */
    int q = e - 8;           /* bf16 keeps 8 significant bits */
    if (q < -133) q = -133;  /* quantum of the bf16 subnormals */
    double v = ldexp(nearbyint(ldexp(a, -q)), q);
    if (v >= 0x1.0p128) return (uint16_t)(sign | 0x7F80u);
    float f = (float)v;      /* exact: v has <= 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return (uint16_t)(sign | (bits >> 16));
}

/* ---------------------------------------------------------------- threads */

typedef struct {
    int kind;               /* 0 normal, 1 uniform */
    uint64_t base;
    double p0, p1;          /* normal: mean, std; uniform: lo, hi */
    size_t rows, cols;      /* logical row-major (rows x cols) tensor */
    int shards;             /* column shards; out is [shards][rows][cols/shards] */
    uint16_t *out_bf16;
    double *out_f64;
    uint64_t pair_lo, pair_hi;
} gen_job;

static void put(const gen_job *g, uint64_t i, double v) {
    if (i >= (uint64_t)g->rows * g->cols) return;
    size_t r = (size_t)(i / g->cols), c = (size_t)(i % g->cols);
    size_t cs = g->cols / (size_t)g->shards;
    size_t s = c / cs, cc = c % cs;
    size_t dst = (s * g->rows + r) * cs + cc;
    if (g->out_bf16) g->out_bf16[dst] = synth_round_bf16(v);
    else g->out_f64[dst] = v;
}

static void *gen_worker(void *arg) {
    const gen_job *g = (const gen_job *)arg;
    for (uint64_t j = g->pair_lo; j < g->pair_hi; ++j) {
        double a, b;
        if (g->kind == 0) {
            normal_pair(g->base, j, &a, &b);
            a = g->p0 + g->p1 * a;
            b = g->p0 + g->p1 * b;
        } else {
            a = g->p0 + (g->p1 - g->p0) * u53(sm64_at(g->base, 2 * j));
            b = g->p0 + (g->p1 - g->p0) * u53(sm64_at(g->base, 2 * j + 1));
        }
        put(g, 2 * j, a);
        put(g, 2 * j + 1, b);
    }
    return NULL;
}

static int run_jobs(gen_job proto, int threads) {
    uint64_t n = (uint64_t)proto.rows * proto.cols;
    uint64_t pairs = (n + 1) / 2;
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if ((uint64_t)threads > pairs) threads = pairs ? (int)pairs : 1;
    pthread_t tid[256];
    int live[256];
    gen_job jobs[256];
    for (int t = 0; t < threads; ++t) {
        jobs[t] = proto;
        jobs[t].pair_lo = pairs * (uint64_t)t / (uint64_t)threads;
        jobs[t].pair_hi = pairs * (uint64_t)(t + 1) / (uint64_t)threads;
        live[t] = 0;
        if (t < threads - 1 && pthread_create(&tid[t], NULL, gen_worker, &jobs[t]) == 0)
            live[t] = 1;
        else
            gen_worker(&jobs[t]);   /* last share, or no thread available */
    }
    for (int t = 0; t < threads; ++t)
        if (live[t]) pthread_join(tid[t], NULL);
    return 0;
}

/* Normal(mean, std) values of a row-major rows x cols tensor, element i of
 * the stream at row-major index i, written in column-sharded layout
 * out[s][r][c'] with c = s * (cols / shards) + c'.  shards must divide cols.
 * Exactly one of out_bf16 / out_f64 is non-NULL. */
int synth_normal(uint64_t seed, uint32_t tag, double mean, double std,
                 size_t rows, size_t cols, int shards,
                 uint16_t *out_bf16, double *out_f64, int threads) {
    if (shards < 1 || cols % (size_t)shards) return -1;
    if (!out_bf16 == !out_f64) return -1;
    gen_job g;
    memset(&g, 0, sizeof g);
    g.kind = 0; g.base = synth_stream_base(seed, tag); g.p0 = mean; g.p1 = std;
    g.rows = rows; g.cols = cols; g.shards = shards;
    g.out_bf16 = out_bf16; g.out_f64 = out_f64;
    return run_jobs(g, threads);
}

/* Uniform on [lo, hi) values, same layout rules as synth_normal. */
int synth_uniform(uint64_t seed, uint32_t tag, double lo, double hi,
                  size_t rows, size_t cols, int shards,
                  uint16_t *out_bf16, double *out_f64, int threads) {
    if (shards < 1 || cols % (size_t)shards) return -1;
    if (!out_bf16 == !out_f64) return -1;
    gen_job g;
    memset(&g, 0, sizeof g);
    g.kind = 1; g.base = synth_stream_base(seed, tag); g.p0 = lo; g.p1 = hi;
    g.rows = rows; g.cols = cols; g.shards = shards;
    g.out_bf16 = out_bf16; g.out_f64 = out_f64;
    return run_jobs(g, threads);
}

/* The first `count` entries of a seeded Fisher-Yates shuffle of 0..n-1
 * (Durstenfeld's in-place form, drawing j uniformly from i..n-1 by
 * multiply-shift of a 64-bit word).  `scratch` holds n ints. */
int synth_choose(uint64_t seed, uint32_t tag, int n, int count, int *scratch, int *out) {
    if (n < 0 || count < 0 || count > n) return -1;
    uint64_t base = synth_stream_base(seed, tag);
    for (int i = 0; i < n; ++i) scratch[i] = i;
    for (int i = 0; i < count; ++i) {
        uint64_t span = (uint64_t)(n - i);
        uint64_t z = sm64_at(base, (uint64_t)i);
        uint64_t j = (uint64_t)i + (uint64_t)(((unsigned __int128)z * span) >> 64);
        int tmp = scratch[i]; scratch[i] = scratch[j]; scratch[j] = tmp;
        out[i] = scratch[i];
    }
    return 0;
}

/* Round an fp64 array to bf16 words (used for inputs formed in fp64 from
 * several streams, e.g. SiLU(g)*u or outlier-scaled channels). */
void synth_round_array(const double *in, size_t n, uint16_t *out) {
    for (size_t i = 0; i < n; ++i) out[i] = synth_round_bf16(in[i]);
}
