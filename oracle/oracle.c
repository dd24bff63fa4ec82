/*
 * CPU oracle for the MXFP4 grouped MoE path.  TEST INFRASTRUCTURE ONLY: only the
 * test-suite, the smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no code, header, table or constant generator with the CUDA library.
 *
 * Everything here is the plain definition, in double precision, with no blocking
 * or reordering beyond what the definition states.  Sources (page titles and the
 * section each rule comes from):
 *
 *  [TPU] "Running DeepSeek V4 Flash on TPU v6", section 1 "Four bits that v6e
 *        can't hold": tokens sorted by expert into one row band per expert; the
 *        grouped-matmul loop nest; 4-bit e2m1 codes decoded to their exact value
 *        (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6); per-32 block scales applied to
 *        the decoded tile before the matmul; bf16 activations, f32 accumulation;
 *        ragged groups including empty ones.
 *  [NVFP4] "DeepSeek-V4-Flash-0731-NVFP4", "The lossless weight cast": E8M0
 *        power-of-two scales per 32 elements; w1/w3 fused into one GEMM; E2M1 -0
 *        is canonicalised to +0; NVFP4's two scale levels (per-16 E4M3 block
 *        scales under a per-tensor weight_scale_2) and the cast into them.
 *  [Pocket] "DeepSeek-V4-Flash" (PocketLLM), "Correctness and precision":
 *        deterministic expert reduction without atomics.
 *
 * Readings where the pages leave a detail open:
 *  - nibble order: element 2j of a byte is the low nibble (bits 0-3);
 *  - nibble bits: bit 3 sign, bits 2-1 exponent, bit 0 mantissa, so the
 *    magnitude index 2e+m is the low three bits;
 *  - code 0x8 (-0) decodes to +0;
 *  - E8M0 bias 127; scale bytes 253..255 are rejected (253/254 would overflow
 *    bfloat16 for the larger codes, 255 is the E8M0 NaN);
 *  - stable sort: within an expert, slots keep ascending s = t*k + j;
 *  - w13 output columns [0, I) are the gate, [I, 2I) the up projection;
 *  - SwiGLU h = silu(g) * u, silu(g) = g / (1 + e^-g), rounded once to bf16;
 *  - "block 32" and "block 512" ([TPU] section 1, the two measured kernel
 *    variants) are read as the number of consecutive k sharing one E8M0 scale:
 *    the scale of weight (e, n, k) is scales[e, n, k / block], with K / block
 *    scale bytes per row.  MXFP4 proper is block 32.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* The e2m1 value of each 4-bit code.  Magnitudes from [TPU] section 1; the
 * upper eight codes carry the sign bit; code 8 (-0) is +0 per [NVFP4]. */
static const double E2M1_VALUE[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

double oracle_e2m1_value(int code) { return E2M1_VALUE[code & 15]; }

/* ------------------------------------------------------------------ bfloat16 */

static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to the nearest bfloat16 (ties to even), with bfloat16's
 * subnormals (quantum 2^-133) and overflow to infinity.  Returns the bits. */
uint16_t oracle_double_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                  /* a = f * 2^e, f in [0.5, 1): leading bit 2^(e-1) */
    int q = e - 8;                 /* quantum of an 8-bit significand */
    if (q < -133) q = -133;        /* subnormal range has a fixed quantum */
    double r = nearbyint(ldexp(a, -q));   /* default rounding mode: ties to even */
    double y = ldexp(r, q);
    if (y >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)y;            /* exact: y has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

double oracle_bf16_to_double(uint16_t b) { return bf16_bits_to_double(b); }

/* --------------------------------------------------------------- thread pool */

typedef struct {
    void (*fn)(void *ctx, long item);
    void *ctx;
    long n_items;
    long next;
    pthread_mutex_t mu;
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        long i = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (i >= p->n_items) break;
        p->fn(p->ctx, i);
    }
    return NULL;
}

static int g_threads_used = 1;
int oracle_threads_used(void) { return g_threads_used; }

static void run_parallel(void (*fn)(void *, long), void *ctx, long n_items, int n_threads) {
    if (n_threads <= 0) n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_items) n_threads = (int)(n_items > 0 ? n_items : 1);
    g_threads_used = n_threads;
    pool_t p = {fn, ctx, n_items, 0};
    pthread_mutex_init(&p.mu, NULL);
    if (n_threads == 1) {
        pool_worker(&p);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
        for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, pool_worker, &p);
        for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------ weight decode */

/* Exact value of weight (e, n, k): e2m1(code) * 2^(scale - 127), with one
 * scale byte per `block` consecutive k.  Returns 0 on success, -1 if the scale
 * byte is outside 0..252. */
static int weight_value_block(const uint8_t *codes, const uint8_t *scales, long N, long K,
                              long block, long e, long n, long k, double *w) {
    uint8_t byte = codes[(e * N + n) * (K / 2) + k / 2];
    int code = (k & 1) ? (byte >> 4) : (byte & 15);
    int s = scales[(e * N + n) * (K / block) + k / block];
    if (s > 252) return -1;
    *w = ldexp(E2M1_VALUE[code], s - 127);
    return 0;
}

/* MXFP4: one scale per 32 k. */
static int weight_value(const uint8_t *codes, const uint8_t *scales, long N, long K,
                        long e, long n, long k, double *w) {
    return weight_value_block(codes, scales, N, K, 32, e, n, k, w);
}

/* Decoded weights of expert e as bfloat16 bits [N, K].  Every e2m1 value times
 * 2^(s-127), s in 0..252, is a bfloat16 number, so the rounding is exact. */
int oracle_decode_expert_bf16(const uint8_t *codes, const uint8_t *scales, long E, long N, long K,
                              long e, uint16_t *out) {
    if (e < 0 || e >= E || K % 32) return -1;
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k) {
            double w;
            if (weight_value(codes, scales, N, K, e, n, k, &w)) return -1;
            out[n * K + k] = oracle_double_to_bf16(w);
        }
    return 0;
}

/* --------------------------------------------------------------- route sort */

/* Stable counting sort of the T*k routing slots by expert ([TPU] section 1:
 * rows are ordered by expert so each expert owns one contiguous band).  Outputs: group_sizes[E], group_offsets[E+1], sorted_slot[rows]
 * (row -> slot), slot_to_row[rows].  Returns -1 on an out-of-range id. */
int oracle_route_sort(const int32_t *ids, long T, long k, long E, int32_t *group_sizes,
                      int32_t *group_offsets, int32_t *sorted_slot, int32_t *slot_to_row) {
    if (T < 0 || k < 0 || E <= 0) return -1;
    long rows = T * k;
    for (long e = 0; e < E; ++e) group_sizes[e] = 0;
    for (long s = 0; s < rows; ++s) {
        if (ids[s] < 0 || ids[s] >= E) return -1;
        group_sizes[ids[s]] += 1;
    }
    group_offsets[0] = 0;
    for (long e = 0; e < E; ++e) group_offsets[e + 1] = group_offsets[e] + group_sizes[e];
    int32_t *cursor = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (long s = 0; s < rows; ++s) {           /* ascending s: stable */
        int32_t e = ids[s];
        int32_t row = group_offsets[e] + cursor[e]++;
        sorted_slot[row] = (int32_t)s;
        slot_to_row[s] = row;
    }
    free(cursor);
    return 0;
}

/* x_sorted[row, :] = x[sorted_slot[row] / k, :]  (bf16 bits copied). */
void oracle_gather(const uint16_t *x, long hidden, const int32_t *sorted_slot, long rows, long k,
                   uint16_t *x_sorted) {
    for (long r = 0; r < rows; ++r)
        memcpy(x_sorted + r * hidden, x + (long)(sorted_slot[r] / k) * hidden,
               (size_t)hidden * sizeof(uint16_t));
}

/* ------------------------------------------------------------- grouped GEMM */

typedef struct {
    const uint16_t *act;
    const uint8_t *codes, *scales;
    const int32_t *offsets;
    long K, N, n_block;
    long n_blocks_per_e;
    double *out, *abs_out;
    int bad_scale;
    long block;                                 /* k per scale byte */
} gemm_ctx;

#define N_BLOCK 32

static void gemm_item(void *vctx, long item) {
    gemm_ctx *c = (gemm_ctx *)vctx;
    long e = item / c->n_blocks_per_e;
    long n0 = (item % c->n_blocks_per_e) * N_BLOCK;
    long r0 = c->offsets[e], r1 = c->offsets[e + 1];
    if (r1 <= r0) return;                       /* empty group: no rows, no work */
    long K = c->K, N = c->N;
    double *w = (double *)malloc(sizeof(double) * (size_t)K);
    for (long n = n0; n < n0 + N_BLOCK && n < N; ++n) {
        for (long k = 0; k < K; ++k)
            if (weight_value_block(c->codes, c->scales, N, K, c->block, e, n, k, &w[k]))
                c->bad_scale = 1;
        for (long r = r0; r < r1; ++r) {
            const uint16_t *a = c->act + r * K;
            double acc = 0.0, mag = 0.0;
            for (long k = 0; k < K; ++k) {      /* ascending k */
                double p = bf16_bits_to_double(a[k]) * w[k];
                acc += p;
                mag += fabs(p);
            }
            c->out[r * N + n] = acc;
            if (c->abs_out) c->abs_out[r * N + n] = mag;
        }
    }
    free(w);
}

/* out[r, n] = sum_k act[r, k] * w_e[n, k] for every row r of band e ([TPU]
 * section 1, the grouped-matmul loop nest with the decode step).  The bands
 * are group_sizes in expert order.  abs_out (optional) receives
 * sum_k |act[r,k] * w_e[n,k]|, the scale of the accumulation error.  Returns -1
 * if sum(group_sizes) != rows, a size is negative, or a scale byte is > 252. */
int oracle_grouped_gemm(const uint16_t *act, long rows, long K, const uint8_t *codes,
                        const uint8_t *scales, const int32_t *group_sizes, long E, long N,
                        double *out, double *abs_out, int n_threads) {
    if (K % 32) return -1;
    int32_t *off = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    off[0] = 0;
    for (long e = 0; e < E; ++e) {
        if (group_sizes[e] < 0) { free(off); return -1; }
        off[e + 1] = off[e] + group_sizes[e];
    }
    if (off[E] != rows) { free(off); return -1; }
    gemm_ctx c = {act, codes, scales, off, K, N, N_BLOCK, (N + N_BLOCK - 1) / N_BLOCK, out, abs_out, 0,
                  32};
    run_parallel(gemm_item, &c, E * c.n_blocks_per_e, n_threads);
    free(off);
    return c.bad_scale ? -1 : 0;
}

/* The grouped GEMM with one scale byte per `block` consecutive k (scales
 * [E, N, K / block]); block 32 is oracle_grouped_gemm.  Returns -1 if block
 * is not 32 or 512, K is not a multiple of block, or as oracle_grouped_gemm. */
int oracle_grouped_gemm_block(const uint16_t *act, long rows, long K, long block,
                              const uint8_t *codes, const uint8_t *scales,
                              const int32_t *group_sizes, long E, long N, double *out,
                              double *abs_out, int n_threads) {
    if ((block != 32 && block != 512) || K % block) return -1;
    int32_t *off = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    off[0] = 0;
    for (long e = 0; e < E; ++e) {
        if (group_sizes[e] < 0) { free(off); return -1; }
        off[e + 1] = off[e] + group_sizes[e];
    }
    if (off[E] != rows) { free(off); return -1; }
    gemm_ctx c = {act, codes, scales, off, K, N, N_BLOCK, (N + N_BLOCK - 1) / N_BLOCK, out, abs_out, 0,
                  block};
    run_parallel(gemm_item, &c, E * c.n_blocks_per_e, n_threads);
    free(off);
    return c.bad_scale ? -1 : 0;
}

typedef struct {
    const uint16_t *act;
    const uint8_t *codes, *scales;
    const int32_t *offsets;
    long E, K, N;
    const int64_t *srow, *scol;
    double *out, *abs_out;
    int bad;
} sampled_ctx;

static void sampled_item(void *vctx, long i) {
    sampled_ctx *c = (sampled_ctx *)vctx;
    long r = (long)c->srow[i], n = (long)c->scol[i];
    /* The expert owning row r is the last e with off[e] <= r; then off[e+1] > r,
     * so that band is not empty. */
    long lo = 0, hi = c->E - 1;
    while (lo < hi) {
        long mid = (lo + hi + 1) / 2;
        if (c->offsets[mid] <= r) lo = mid; else hi = mid - 1;
    }
    long e = lo;
    double acc = 0.0, mag = 0.0;
    for (long k = 0; k < c->K; ++k) {
        double w;
        if (weight_value(c->codes, c->scales, c->N, c->K, e, n, k, &w)) c->bad = 1;
        double p = bf16_bits_to_double(c->act[r * c->K + k]) * w;
        acc += p;
        mag += fabs(p);
    }
    c->out[i] = acc;
    c->abs_out[i] = mag;
}

/* The same definition evaluated only at the listed (row, column) pairs. */
int oracle_grouped_gemm_sampled(const uint16_t *act, long rows, long K, const uint8_t *codes,
                                const uint8_t *scales, const int32_t *group_sizes, long E, long N,
                                const int64_t *srow, const int64_t *scol, long n_samples,
                                double *out, double *abs_out, int n_threads) {
    if (K % 32) return -1;
    int32_t *off = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    off[0] = 0;
    for (long e = 0; e < E; ++e) off[e + 1] = off[e] + group_sizes[e];
    if (off[E] != rows) { free(off); return -1; }
    for (long i = 0; i < n_samples; ++i)
        if (srow[i] < 0 || srow[i] >= rows || scol[i] < 0 || scol[i] >= N) { free(off); return -1; }
    sampled_ctx c = {act, codes, scales, off, E, K, N, srow, scol, out, abs_out, 0};
    run_parallel(sampled_item, &c, n_samples, n_threads);
    free(off);
    return c.bad ? -1 : 0;
}

/* ------------------------------------------------------------------- SwiGLU */

/* h[r, i] = bf16( silu(g) * u ), g = gu[r, i], u = gu[r, I + i], in double. */
void oracle_swiglu(const double *gu, long rows, long I, uint16_t *h) {
    for (long r = 0; r < rows; ++r)
        for (long i = 0; i < I; ++i) {
            double g = gu[r * 2 * I + i], u = gu[r * 2 * I + I + i];
            double silu = g / (1.0 + exp(-g));
            h[r * I + i] = oracle_double_to_bf16(silu * u);
        }
}

/* ------------------------------------------------------------------ combine */

/* out[t, n] = sum_{j=0..k-1} topk_w[t, j] * y[slot_to_row[t*k + j], n], summed
 * in ascending j ([Pocket], deterministic expert reduction).  abs_out
 * (optional) receives sum_j |w * y|. */
void oracle_combine(const double *y, long N, const int32_t *slot_to_row, const float *topk_w,
                    long T, long k, double *out, double *abs_out) {
    for (long t = 0; t < T; ++t)
        for (long n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (long j = 0; j < k; ++j) {
                double p = (double)topk_w[t * k + j] * y[(long)slot_to_row[t * k + j] * N + n];
                acc += p;
                mag += fabs(p);
            }
            out[t * N + n] = acc;
            if (abs_out) abs_out[t * N + n] = mag;
        }
}

/* ------------------------------------------------- MXFP4 -> NVFP4 weight cast */

/* E4M3 (sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no infinities,
 * exponent 15 with mantissa 7 is NaN) value of a byte, from the format's
 * definition. */
double oracle_e4m3_value(int byte) {
    const int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);              /* subnormal: m/8 * 2^-6 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* E4M3 byte of 2^p if it is exactly representable (p in -9..8), else -1. */
static int e4m3_of_power_of_two(int p) {
    if (p > 8 || p < -9) return -1;
    if (p >= -6) return (p + 7) << 3;                   /* normal, mantissa 0 */
    return 1 << (p + 9);                                /* subnormal: 2^p = m * 2^-9 */
}

/* The lossless cast of [NVFP4] "The lossless weight cast": for each expert e
 * (its whole [N, K/32] scale tensor, so the fused w1/w3 rows share it),
 * k_max = max over blocks of (scale byte - 127); the per-tensor scale is
 * 2^(k_max - 8) and block j's per-16 scale (written for both halves of the
 * 32-element block) is 2^(k_j - k_max + 8), so that per-16 scale times the
 * per-tensor scale is the block's own 2^(k_j).  The 4-bit codes are unchanged.
 * A block whose per-16 scale falls below E4M3's smallest power of two (2^-9)
 * cannot be cast exactly: it is counted in out_of_range[e] and written as 0.
 * Scale byte 255 (E8M0 NaN) is rejected (returns 1). */
int oracle_mxfp4_to_nvfp4(const uint8_t *scales, long E, long N, long K, uint8_t *e4m3,
                          double *weight_scale_2, int64_t *out_of_range) {
    const long nb = K / 32;
    for (long e = 0; e < E; ++e) {
        const uint8_t *s = scales + e * N * nb;
        int kmax = -1000;
        for (long i = 0; i < N * nb; ++i) {
            if (s[i] == 255) return 1;
            if ((int)s[i] - 127 > kmax) kmax = (int)s[i] - 127;
        }
        weight_scale_2[e] = ldexp(1.0, kmax - 8);
        int64_t bad = 0;
        for (long i = 0; i < N * nb; ++i) {
            int b = e4m3_of_power_of_two((int)s[i] - 127 - kmax + 8);
            if (b < 0) {
                ++bad;
                b = 0;
            }
            e4m3[(e * N * nb + i) * 2] = (uint8_t)b;
            e4m3[(e * N * nb + i) * 2 + 1] = (uint8_t)b;
        }
        out_of_range[e] = bad;
    }
    return 0;
}

/* ------------------------------------------------------ NVFP4 grouped GEMM */

/* Exact value of NVFP4 weight (e, n, k): e2m1(code) * e4m3(s16[e, n, k/16]) *
 * weight_scale_2[e].  [TPU] section 1 describes an NVFP4 kernel that decodes
 * the e2m1 weights and their per-16 E4M3 scales; [NVFP4] "The lossless weight
 * cast" gives the two scale levels (per-16 E4M3 under a per-tensor f32
 * weight_scale_2) whose product reconstructs each weight.  Every factor is
 * exact in double and so is their product (at most 2 + 4 + 24 significant
 * bits).  Returns -1 for a NaN scale byte (0x7F or 0xFF). */
static int nvfp4_weight_value(const uint8_t *codes, const uint8_t *s16, const float *ws2, long N,
                              long K, long e, long n, long k, double *w) {
    uint8_t byte = codes[(e * N + n) * (K / 2) + k / 2];
    int code = (k & 1) ? (byte >> 4) : (byte & 15);
    double s = oracle_e4m3_value(s16[(e * N + n) * (K / 16) + k / 16]);
    if (isnan(s)) return -1;
    *w = E2M1_VALUE[code] * s * (double)ws2[e];
    return 0;
}

typedef struct {
    const uint16_t *act;
    const uint8_t *codes, *s16;
    const float *ws2;
    const int32_t *offsets;
    long K, N, n_blocks_per_e;
    double *out, *abs_out;
    int bad_scale;
} nvfp4_ctx;

static void nvfp4_gemm_item(void *vctx, long item) {
    nvfp4_ctx *c = (nvfp4_ctx *)vctx;
    long e = item / c->n_blocks_per_e;
    long n0 = (item % c->n_blocks_per_e) * N_BLOCK;
    long r0 = c->offsets[e], r1 = c->offsets[e + 1];
    if (r1 <= r0) return;                       /* empty group: no rows, no work */
    long K = c->K, N = c->N;
    double *w = (double *)malloc(sizeof(double) * (size_t)K);
    for (long n = n0; n < n0 + N_BLOCK && n < N; ++n) {
        for (long k = 0; k < K; ++k)
            if (nvfp4_weight_value(c->codes, c->s16, c->ws2, N, K, e, n, k, &w[k])) c->bad_scale = 1;
        for (long r = r0; r < r1; ++r) {
            const uint16_t *a = c->act + r * K;
            double acc = 0.0, mag = 0.0;
            for (long k = 0; k < K; ++k) {      /* ascending k */
                double p = bf16_bits_to_double(a[k]) * w[k];
                acc += p;
                mag += fabs(p);
            }
            c->out[r * N + n] = acc;
            if (c->abs_out) c->abs_out[r * N + n] = mag;
        }
    }
    free(w);
}

/* out[r, n] = sum_k act[r, k] * w_e[n, k] with the NVFP4 weights above, for
 * every row r of band e (bands = group_sizes in expert order), summed in
 * ascending k.  codes [E, N, K/2] as for MXFP4; scales16 [E, N, K/16] E4M3
 * bytes; weight_scale_2 [E] f32.  abs_out (optional) receives sum_k |a * w|.
 * Returns -1 if K % 16 != 0, a group size is negative, sum(group_sizes) !=
 * rows, or a scale byte read is NaN. */
int oracle_nvfp4_grouped_gemm(const uint16_t *act, long rows, long K, const uint8_t *codes,
                              const uint8_t *scales16, const float *weight_scale_2,
                              const int32_t *group_sizes, long E, long N, double *out,
                              double *abs_out, int n_threads) {
    if (K % 16 || K <= 0) return -1;
    int32_t *off = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    off[0] = 0;
    for (long e = 0; e < E; ++e) {
        if (group_sizes[e] < 0) { free(off); return -1; }
        off[e + 1] = off[e] + group_sizes[e];
    }
    if (off[E] != rows) { free(off); return -1; }
    nvfp4_ctx c = {act, codes, scales16, weight_scale_2, off, K, N, (N + N_BLOCK - 1) / N_BLOCK,
                   out, abs_out, 0};
    run_parallel(nvfp4_gemm_item, &c, E * c.n_blocks_per_e, n_threads);
    free(off);
    return c.bad_scale ? -1 : 0;
}
