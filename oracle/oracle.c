/*
 * CPU oracle for the tensor-parallel GEMV fused with a one-shot all-reduce.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's CPU
 * baseline leg are the only callers.  The CUDA path never loads this file and
 * this file includes nothing from it.
 *
 * What is computed, and where the pages define it:
 *
 *  - Row-parallel linear layer.  "Bay.Area.AI: Tensor and 2D Parallelism"
 *    (talk transcript, the Megatron-style column-then-row sharding passage):
 *    after a row-wise sharded linear each rank holds a partial output and the
 *    layer ends in one all-reduce.  Rank r holds the column block
 *    W_r = W[:, r*K_r : (r+1)*K_r] (N x K_r, row-major) and x_r = x[:, same
 *    columns] (B x K_r); its partial is P_r[b][n] = sum_k W_r[n][k] x_r[b][k],
 *    and y = sum_r P_r = W x.
 *
 *  - Fusing that GEMV with its all-reduce.  "Overlapping Collective
 *    Communication with Dependent Computation ... GPU-Initiated Intra-Kernel
 *    Networking" (linnk.ai summary of "Optimizing Distributed ML Communication
 *    with Fused Computation-Collective Operations"), Abstract: the fused
 *    GEMV + AllReduce operator.  Fusion changes when partials move, not what
 *    is summed, so the oracle is the unfused definition.
 *
 *  - One-shot all-reduce.  "PyTorch Symmetric Memory: A New Programming
 *    Paradigm for Distributed AI" (talk), the one-shot all-reduce segment, and
 *    the PyTorch Symmetric Memory documentation, op reference
 *    `one_shot_all_reduce` (reduce op "sum" only): every rank reads the inputs
 *    of all ranks and reduces locally; all ranks end with the same sum.
 *
 *  - Precision.  PyTorch Symmetric Memory documentation, "higher-precision
 *    reduction" of the NCCL symmetric kernels: bf16 in, wider accumulation,
 *    bf16 out.  The oracle accumulates in fp64: each rank's partial in
 *    ascending k, the partials in rank order 0..R-1 (or an explicit order),
 *    then rounds once, fp64 -> bf16, round to nearest, ties to even.
 *
 * Every rank's output slot receives the same rounded value; the oracle writes
 * all R replicas and checks that they are identical.
 *
 * Further collectives on the same slots, each defined where it is written
 * below: the reduce-scatter (flat, and along the batch rows of the fused
 * layer), the all-reduce followed by a bias and RMS normalisation (alone and
 * as the fused layer's epilogue), and the 2-D tile reduce to one or several
 * roots.  A two-shot all-reduce reaches exactly the all-reduce definition
 * (its two phases change where each sum is computed, not the sum), so its
 * oracle is oracle_one_shot_all_reduce.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------ bf16 words */

/* bf16 bits -> exact fp64 value, from the field definitions
 * (1 sign bit, 8 exponent bits with bias 127, 7 fraction bits). */
double oracle_bf16_value(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int m = h & 0x7F;
    double v;
    if (e == 0xFF) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -133);          /* m * 2^(1-127-7) */
    else v = ldexp((double)(128 + m), e - 134);             /* 1.m * 2^(e-127) */
    return s ? -v : v;
}

/* fp64 -> bf16 bits, round to nearest, ties to even, working on the fp64
 * bit fields: keep the significand bits down to the bf16 quantum 2^q, look at
 * the dropped bits, round, and re-encode.  With q the quantum exponent and
 * `keep` the rounded count of quanta, the bf16 word is ((q + 133) << 7) + keep
 * for normals and subnormals alike (a carry into the next binade lands in the
 * exponent field by itself); words >= 0x7F80 overflow to infinity. */
uint16_t oracle_bf16_round(double v) {
    uint64_t u;
    memcpy(&u, &v, 8);
    uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
    u &= 0x7FFFFFFFFFFFFFFFULL;
    int E = (int)(u >> 52);
    uint64_t frac = u & ((1ULL << 52) - 1);
    if (E == 0x7FF) return (uint16_t)(sign | (frac ? 0x7FC0u : 0x7F80u));
    if (E == 0) return sign;                  /* |v| < 2^-1022: far below half of 2^-133 */
    uint64_t S = (1ULL << 52) | frac;         /* v = S * 2^(E - 1075) */
    int e = E - 1023;                         /* v in [2^e, 2^(e+1)) */
    int q = e - 7;
    if (q < -133) q = -133;
    int shift = q - (E - 1075);               /* low bits of S below the quantum */
    uint64_t keep;
    if (shift >= 64) {
        keep = 0;
    } else {
        keep = S >> shift;
        uint64_t rem = S & ((1ULL << shift) - 1);
        uint64_t half = 1ULL << (shift - 1);
        if (rem > half || (rem == half && (keep & 1))) keep += 1;
    }
    long long word = ((long long)(q + 133) << 7) + (long long)keep;
    if (keep == 0) return sign;
    if (word >= 0x7F80) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)word);
}

/* Decoded value of every bf16 word, filled once from oracle_bf16_value; the
 * sums below look values up here instead of re-decoding each element. */
static double g_bf16_table[65536];
static pthread_once_t g_table_once = PTHREAD_ONCE_INIT;

static void fill_table(void) {
    for (uint32_t h = 0; h < 65536u; ++h) g_bf16_table[h] = oracle_bf16_value((uint16_t)h);
}

static const double *bf16_table(void) {
    pthread_once(&g_table_once, fill_table);
    return g_bf16_table;
}

/* ------------------------------------------------------ GEMV + all-reduce */

typedef struct {
    int R, N, Kr, B;
    const uint16_t *W;      /* [R][N][Kr] */
    const uint16_t *x;      /* [R][B][Kr] */
    const int *order;       /* rank summation order, length R */
    double *y_ref;          /* [B][N] */
    uint16_t *y_out;        /* [R][B][N] or NULL */
    int n_lo, n_hi;
} gemv_job;

/* Partial of rank r for output (b, n), fp64, ascending k. */
static double rank_partial(const gemv_job *g, int r, int b, int n) {
    const uint16_t *w = g->W + ((size_t)r * g->N + n) * g->Kr;
    const uint16_t *xv = g->x + ((size_t)r * g->B + b) * g->Kr;
    const double *val = bf16_table();
    double p = 0.0;
    for (int k = 0; k < g->Kr; ++k)
        p += val[w[k]] * val[xv[k]];
    return p;
}

static double reduce_ranks(const gemv_job *g, int b, int n) {
    double y = 0.0;
    for (int i = 0; i < g->R; ++i) y += rank_partial(g, g->order[i], b, n);
    return y;
}

static void *gemv_worker(void *arg) {
    gemv_job *g = (gemv_job *)arg;
    for (int n = g->n_lo; n < g->n_hi; ++n) {
        for (int b = 0; b < g->B; ++b) {
            double y = reduce_ranks(g, b, n);
            g->y_ref[(size_t)b * g->N + n] = y;
            if (g->y_out) {
                uint16_t h = oracle_bf16_round(y);
                for (int s = 0; s < g->R; ++s)
                    g->y_out[((size_t)s * g->B + b) * g->N + n] = h;
            }
        }
    }
    return NULL;
}

static int order_ok(int R, const int *order, int *buf) {
    int seen[64];
    if (R < 1 || R > 64) return 0;
    memset(seen, 0, sizeof seen);
    for (int i = 0; i < R; ++i) {
        int r = order ? order[i] : i;
        if (r < 0 || r >= R || seen[r]) return 0;
        seen[r] = 1;
        buf[i] = r;
    }
    return 1;
}

static int replicas_identical(const uint16_t *out, int R, size_t per_rank) {
    for (int s = 1; s < R; ++s)
        if (memcmp(out, out + (size_t)s * per_rank, per_rank * sizeof(uint16_t)) != 0) return 0;
    return 1;
}

/* y_ref[b][n] = sum over ranks (in `order`, NULL = 0..R-1) of the fp64
 * partial of that rank; y_out[s][b][n] = bf16 RNE of y_ref for every rank s.
 * Returns 0, -1 on bad arguments, -2 if the replicas differ. */
int oracle_gemv_all_reduce(int R, int N, int K, int B, const uint16_t *W, const uint16_t *x,
                           const int *order, double *y_ref, uint16_t *y_out, int threads) {
    int ord[64];
    if (N < 0 || K < 0 || B < 0 || !order_ok(R, order, ord) || K % R) return -1;
    gemv_job proto = {R, N, K / R, B, W, x, ord, y_ref, y_out, 0, 0};
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (threads > N) threads = N > 0 ? N : 1;
    pthread_t tid[256];
    int live[256];
    gemv_job jobs[256];
    for (int t = 0; t < threads; ++t) {
        jobs[t] = proto;
        jobs[t].n_lo = (int)((long long)N * t / threads);
        jobs[t].n_hi = (int)((long long)N * (t + 1) / threads);
        live[t] = 0;
        if (t < threads - 1 && pthread_create(&tid[t], NULL, gemv_worker, &jobs[t]) == 0)
            live[t] = 1;
        else
            gemv_worker(&jobs[t]);
    }
    for (int t = 0; t < threads; ++t)
        if (live[t]) pthread_join(tid[t], NULL);
    if (y_out && !replicas_identical(y_out, R, (size_t)B * N)) return -2;
    return 0;
}

/* One output of the definition above, for sampled checks at full size. */
double oracle_gemv_element(int R, int N, int K, int B, const uint16_t *W, const uint16_t *x,
                           int b, int n) {
    int ord[64];
    if (!order_ok(R, NULL, ord) || K % R || b < 0 || b >= B || n < 0 || n >= N) return NAN;
    gemv_job g = {R, N, K / R, B, W, x, ord, NULL, NULL, 0, 0};
    return reduce_ranks(&g, b, n);
}

/* Each rank's fp64 partial for output (b, n): partials[r], r = 0..R-1. */
int oracle_gemv_partials(int R, int N, int K, int B, const uint16_t *W, const uint16_t *x,
                         int b, int n, double *partials) {
    int ord[64];
    if (!order_ok(R, NULL, ord) || K % R || b < 0 || b >= B || n < 0 || n >= N) return -1;
    gemv_job g = {R, N, K / R, B, W, x, ord, NULL, NULL, 0, 0};
    for (int r = 0; r < R; ++r) partials[r] = rank_partial(&g, r, b, n);
    return 0;
}

/* ---------------------------------------------------- one-shot all-reduce */

typedef struct {
    int R;
    size_t n;
    const uint16_t *in;     /* [R][n] */
    const int *order;
    double *ref;            /* [n] */
    uint16_t *out;          /* [R][n] or NULL */
    size_t lo, hi;
} ar_job;

static void *ar_worker(void *arg) {
    ar_job *a = (ar_job *)arg;
    const double *val = bf16_table();
    for (size_t i = a->lo; i < a->hi; ++i) {
        double s = 0.0;
        for (int j = 0; j < a->R; ++j) s += val[a->in[(size_t)a->order[j] * a->n + i]];
        a->ref[i] = s;
        if (a->out) {
            uint16_t h = oracle_bf16_round(s);
            for (int r = 0; r < a->R; ++r) a->out[(size_t)r * a->n + i] = h;
        }
    }
    return NULL;
}

/* ref[i] = sum over ranks (in `order`) of in[r][i] in fp64;
 * out[s][i] = bf16 RNE of ref[i] for every rank s. */
int oracle_one_shot_all_reduce(int R, size_t n, const uint16_t *in, const int *order,
                               double *ref, uint16_t *out, int threads) {
    int ord[64];
    if (!order_ok(R, order, ord)) return -1;
    ar_job proto = {R, n, in, ord, ref, out, 0, 0};
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if ((size_t)threads > n) threads = n > 0 ? (int)n : 1;
    pthread_t tid[256];
    int live[256];
    ar_job jobs[256];
    for (int t = 0; t < threads; ++t) {
        jobs[t] = proto;
        jobs[t].lo = n * (size_t)t / (size_t)threads;
        jobs[t].hi = n * (size_t)(t + 1) / (size_t)threads;
        live[t] = 0;
        if (t < threads - 1 && pthread_create(&tid[t], NULL, ar_worker, &jobs[t]) == 0)
            live[t] = 1;
        else
            ar_worker(&jobs[t]);
    }
    for (int t = 0; t < threads; ++t)
        if (live[t]) pthread_join(tid[t], NULL);
    if (out && !replicas_identical(out, R, n)) return -2;
    return 0;
}

/* ------------------------------------------------------- reduce-scatter */

/* The sequence-parallel ending of the row-parallel layer: "Bay.Area.AI:
 * Tensor and 2D Parallelism" (talk, sequence-parallel passage) -- after the
 * row-wise sharded linear, a reduce-scatter instead of an all-reduce leaves
 * each rank one shard of the summed tensor.  The shards are the R equal
 * consecutive blocks of the flat tensor: rank s keeps elements
 * [s*n/R, (s+1)*n/R) of the sum (n % R == 0).
 *   ref[i]          fp64 sum over ranks in order 0..R-1, i < n
 *   out[s][j]       bf16 RNE of ref[s*(n/R) + j]
 * Returns 0, -1 on bad arguments. */
int oracle_reduce_scatter(int R, size_t n, const uint16_t *in, double *ref, uint16_t *out) {
    if (R < 1 || R > 64 || n % (size_t)R) return -1;
    const double *val = bf16_table();
    const size_t c = n / (size_t)R;
    for (int s = 0; s < R; ++s) {
        for (size_t j = 0; j < c; ++j) {
            const size_t i = (size_t)s * c + j;
            double acc = 0.0;
            for (int r = 0; r < R; ++r) acc += val[in[(size_t)r * n + i]];
            ref[i] = acc;
            out[(size_t)s * c + j] = oracle_bf16_round(acc);
        }
    }
    return 0;
}

/* Reduce-scatter of the fused layer's output along the token (batch)
 * dimension, the dimension sequence parallelism shards: rank s keeps rows
 * b in [s*B/R, (s+1)*B/R) of y = sum_r W_r x_r (B % R == 0).
 *   y_ref[b][n]     the fp64 sum, as oracle_gemv_all_reduce computes it
 *   out[s][i][n]    bf16 RNE of y_ref[s*B/R + i][n]
 * Returns 0, -1 on bad arguments. */
int oracle_gemv_reduce_scatter(int R, int N, int K, int B, const uint16_t *W, const uint16_t *x,
                               double *y_ref, uint16_t *out, int threads) {
    if (R < 1 || R > 64 || B % R) return -1;
    int rc = oracle_gemv_all_reduce(R, N, K, B, W, x, NULL, y_ref, NULL, threads);
    if (rc) return rc;
    const int Bs = B / R;
    for (int s = 0; s < R; ++s)
        for (int i = 0; i < Bs; ++i)
            for (int n = 0; n < N; ++n)
                out[((size_t)s * Bs + i) * N + n] = oracle_bf16_round(y_ref[(size_t)(s * Bs + i) * N + n]);
    return 0;
}

/* ------------------------------------------- all-reduce + bias + RMSNorm */

/* "PyTorch Symmetric Memory: A New Programming Paradigm for Distributed AI"
 * (talk, the fused kernel segment): an all-reduce, then a bias added to its
 * result, then RMS normalisation, in one kernel.  Per row of H elements:
 *     z[h]  = (sum_r in_r[h]) + bias[h]
 *     ms    = (1/H) sum_h z[h]^2
 *     y[h]  = z[h] / sqrt(ms + eps) * gamma[h]
 * (RMS normalisation with a per-element gain and eps inside the square root;
 * NULL bias means zeros, NULL gamma means ones).  Everything in fp64, one
 * rounding to bf16 at the end, the same value for every rank. */
static void bias_rmsnorm_row(double *z, int H, const uint16_t *bias, const uint16_t *gamma, double eps,
                             double *y) {
    const double *val = bf16_table();
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
        if (bias) z[h] += val[bias[h]];
        ss += z[h] * z[h];
    }
    const double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int h = 0; h < H; ++h) y[h] = z[h] * inv * (gamma ? val[gamma[h]] : 1.0);
}

/* in [R][rows][H]; ref [rows][H] (fp64 result before rounding);
 * out [R][rows][H] or NULL.  Returns 0, -1 on bad arguments, -2 if the
 * replicas differ. */
int oracle_all_reduce_bias_rmsnorm(int R, int rows, int H, const uint16_t *in, const uint16_t *bias,
                                   const uint16_t *gamma, double eps, double *ref, uint16_t *out) {
    if (R < 1 || R > 64 || rows < 0 || H < 1 || !(eps >= 0.0)) return -1;
    const double *val = bf16_table();
    double *z = (double *)malloc((size_t)H * sizeof(double));
    if (!z) return -1;
    for (int i = 0; i < rows; ++i) {
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int r = 0; r < R; ++r) acc += val[in[((size_t)r * rows + i) * H + h]];
            z[h] = acc;
        }
        bias_rmsnorm_row(z, H, bias, gamma, eps, ref + (size_t)i * H);
        if (out)
            for (int h = 0; h < H; ++h) {
                const uint16_t w = oracle_bf16_round(ref[(size_t)i * H + h]);
                for (int s = 0; s < R; ++s) out[((size_t)s * rows + i) * H + h] = w;
            }
    }
    free(z);
    if (out && !replicas_identical(out, R, (size_t)rows * H)) return -2;
    return 0;
}

/* The same epilogue on the fused layer: y[b] = RMSNorm(W x[b] + bias) over
 * the N outputs of each batch row, the GEMV sum as oracle_gemv_all_reduce
 * computes it.  y_ref [B][N]; out [R][B][N] or NULL. */
int oracle_gemv_bias_rmsnorm(int R, int N, int K, int B, const uint16_t *W, const uint16_t *x,
                             const uint16_t *bias, const uint16_t *gamma, double eps, double *y_ref,
                             uint16_t *out, int threads) {
    if (N < 1 || !(eps >= 0.0)) return -1;
    double *z = (double *)malloc((size_t)B * N * sizeof(double) + 1);
    if (!z) return -1;
    int rc = oracle_gemv_all_reduce(R, N, K, B, W, x, NULL, z, NULL, threads);
    if (rc == 0) {
        for (int b = 0; b < B; ++b) {
            bias_rmsnorm_row(z + (size_t)b * N, N, bias, gamma, eps, y_ref + (size_t)b * N);
            if (out)
                for (int n = 0; n < N; ++n) {
                    const uint16_t w = oracle_bf16_round(y_ref[(size_t)b * N + n]);
                    for (int s = 0; s < R; ++s) out[((size_t)s * B + b) * N + n] = w;
                }
        }
    }
    free(z);
    return rc;
}

/* ------------------------------------------------------------ tile reduce */

/* PyTorch Symmetric Memory documentation, op reference `tile_reduce` and
 * `multi_root_tile_reduce`, and the talk's tile-communication segment: a 2-D
 * tile (rows x cols elements of a row-major tensor with leading dimension
 * ld, i.e. not contiguous) is summed over all ranks and the sum is written
 * into the output tile of one root rank only; with several tiles each goes
 * to its own root, and no rank is root twice.
 *
 * The buffers are whole slots: in is [R][in_slot] and out is [R][out_slot]
 * bf16 words; tile i starts at element in_off[i] of every input slot, the
 * output tile at element out_off of an output slot.  For every tile i, element (a, c):
 *     ref[i][a][c] = sum_r in[r][in_off[i] + a*ld_in + c]   (fp64, rank order)
 *     out[roots[i]][out_off + a*ld_out + c] = bf16 RNE of ref[i][a][c]
 * and nothing else of out changes.  Returns 0, -1 on bad arguments (root
 * out of range or repeated, a tile outside the slot). */
int oracle_tile_reduce(int R, size_t in_slot, const uint16_t *in, size_t out_slot, uint16_t *out, int ntiles,
                       const size_t *in_off, size_t out_off, const int *roots, int rows, int cols,
                       size_t ld_in, size_t ld_out, double *ref) {
    if (R < 1 || R > 64 || ntiles < 1 || ntiles > R || rows < 0 || cols < 0) return -1;
    if (rows > 0 && cols > 0) {
        if ((size_t)cols > ld_in || (size_t)cols > ld_out) return -1;
        if (out_off + (size_t)(rows - 1) * ld_out + (size_t)cols > out_slot) return -1;
    }
    int used[64];
    memset(used, 0, sizeof used);
    for (int i = 0; i < ntiles; ++i) {
        if (roots[i] < 0 || roots[i] >= R || used[roots[i]]) return -1;
        used[roots[i]] = 1;
        if (rows > 0 && cols > 0 && in_off[i] + (size_t)(rows - 1) * ld_in + (size_t)cols > in_slot)
            return -1;
    }
    const double *val = bf16_table();
    for (int i = 0; i < ntiles; ++i) {
        for (int a = 0; a < rows; ++a) {
            for (int c = 0; c < cols; ++c) {
                double acc = 0.0;
                for (int r = 0; r < R; ++r)
                    acc += val[in[(size_t)r * in_slot + in_off[i] + (size_t)a * ld_in + (size_t)c]];
                if (ref) ref[((size_t)i * rows + a) * cols + c] = acc;
                out[(size_t)roots[i] * out_slot + out_off + (size_t)a * ld_out + (size_t)c] =
                    oracle_bf16_round(acc);
            }
        }
    }
    return 0;
}
