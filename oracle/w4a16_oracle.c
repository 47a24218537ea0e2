/*
 * w4a16_oracle.c -- plain, slow, obviously correct CPU oracle for the
 * group-wise INT4 weight-only linear layer (W4A16).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only tests/, the smoke check and the CPU-baseline leg of the
 * benchmark do.  It shares no code, header, table or constant generator with
 * the CUDA library: the two meet only through the seeded input generator.
 *
 * What it computes (the method, as the pages describe it):
 *   forum.sourcefind.cn thread "vLLM on Hygon Z100", section 四 (W4A16):
 *   INT4 weights carry a per-group scale and zero point; the kernel unpacks the
 *   packed INT4 words, reads scale and zero, restores each weight and
 *   multiply-accumulates it with the 16-bit activations.
 *   haowenji.com V100 decode article, paragraph on "groupwise-int": integers
 *   times a per-group scale.
 * Written out for m < M, n < N, k < K, g = floor(k / group):
 *     w[n,k] = (q[n,k] - z[n,g]) * s[n,g]
 *     y[m,n] = sum_k x[m,k] * w[n,k]
 * with q, z unsigned 4-bit, s and x IEEE binary16 or bfloat16 (the pages'
 * activations are "fp16 or bf16"; a bf16 layer keeps its scales in bf16 too),
 * y returned in binary64.
 *
 * Readings taken where the pages are silent:
 *   - packed layout [N, K/8] 32-bit words, rows = outputs (section 四 names
 *     "[N,K/8] int32"); element k sits in bits 4*(k%8)..4*(k%8)+3 of word k/8;
 *   - zeros are 4-bit too, packed 8 per word along the group axis with the
 *     same rule; a row has ceil(G/8) words, pad nibbles are written as 0;
 *   - the sum runs in binary64 in increasing k.  Every product x*(q-z)*s is
 *     exact in binary64 (11 + 4 + 11 significant bits), so the only rounding is
 *     in the additions.
 *
 * Parity pins (tests/test_oracle_pins.py, all CPU):
 *   half<->double conversions against numpy's IEEE binary16 conversion over
 *   every bit pattern and a tie/overflow/subnormal battery; pack against
 *   closed-form words; pack/unpack round trip over every nibble value in every
 *   position; dequant against exact rationals for all 256 (q, z) pairs and a
 *   set of scales; linear against exact-rational brute force on tiny shapes,
 *   q == z gives 0, one nonzero group, linearity, and an integer special case
 *   that reduces to an int64 matrix product; the epilogues against closed
 *   forms (sigmoid at ln 3), the odd-part identity and exact sums; the repack
 *   transpose against the pinned pack/unpack, a hand 8 x 8 block, ragged rows
 *   and a nibble-order permutation; bfloat16 conversions against numpy's
 *   binary32 decoder over every pattern, neighbours and ties; the bf16 linear
 *   against exact rationals and an int64 matrix product; the dense 16-bit
 *   linear against exact rationals, an int64 product and, bit for bit, the
 *   4-bit linear over its own exactly representable dequantised weights; the
 *   MoE alignment against a stable sort, the expert linears against the
 *   pinned linear of each slot's expert, the weighted sum exact.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16 <-> binary64, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent field 0
 * holds zero and subnormals (fraction * 2^-24), field 31 holds inf / NaN.
 * ------------------------------------------------------------------------- */
double w4o_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* Round to nearest, ties to even.  Exact: the value is scaled by a power of
 * two into units of the binary16 quantum at its binade, so the integer and
 * fractional parts below are exact in binary64. */
uint16_t w4o_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00u);
    /* 65504 is the largest finite value; 65520 is the midpoint to 2^16 and
     * rounds (to even) upward, i.e. to infinity. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;               /* a in [2^E, 2^(E+1)) */
    if (E < -14) E = -14;         /* subnormal range shares the 2^-24 quantum */
    double r = ldexp(a, 10 - E);  /* a / 2^(E-10), exact */
    double fl = floor(r);
    double frac = r - fl;
    uint64_t m = (uint64_t)fl;
    if (frac > 0.5 || (frac == 0.5 && (m & 1u))) m++;
    if (m == 0) return sign;
    if (m < 1024) {               /* only reachable with E == -14: subnormal */
        return (uint16_t)(sign | (uint16_t)m);
    }
    if (m == 2048) {              /* rounding carried into the next binade */
        m = 1024;
        E++;
    }
    int field = E + 15;
    if (field >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(field << 10) | (uint16_t)(m - 1024));
}

/* ---------------------------------------------------------------------------
 * bfloat16 <-> binary64 (the 16-bit activation type the pages name beside
 * fp16, "fp16 or bf16"), written from the format's definition: 1 sign bit,
 * 8 exponent bits (bias 127), 7 fraction bits -- the top half of an IEEE
 * binary32.  Exponent field 0 holds zero and subnormals (fraction * 2^-133),
 * field 255 holds inf / NaN.
 * ------------------------------------------------------------------------- */
double w4o_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134);
    }
    return sign ? -v : v;
}

/* Round to nearest, ties to even, by the same exact scaling as for binary16:
 * 8 significant bits, binades 2^-126 .. 2^127, subnormal quantum 2^-133. */
uint16_t w4o_double_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7fc0u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7f80u);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;               /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;       /* subnormal range shares the 2^-133 quantum */
    if (E > 127) return (uint16_t)(sign | 0x7f80u);
    double r = ldexp(a, 7 - E);   /* a / 2^(E-7), exact */
    double fl = floor(r);
    double frac = r - fl;
    uint64_t m = (uint64_t)fl;
    if (frac > 0.5 || (frac == 0.5 && (m & 1u))) m++;
    if (m == 0) return sign;
    if (m < 128) return (uint16_t)(sign | (uint16_t)m);  /* subnormal */
    if (m == 256) {               /* rounding carried into the next binade */
        m = 128;
        E++;
    }
    int field = E + 127;
    if (field >= 255) return (uint16_t)(sign | 0x7f80u);
    return (uint16_t)(sign | (uint16_t)(field << 7) | (uint16_t)(m - 128));
}

void w4o_round_to_bf16(const double *v, long n, uint16_t *out)
{
    for (long i = 0; i < n; i++) out[i] = w4o_double_to_bf16(v[i]);
}

void w4o_bf16_array_to_double(const uint16_t *b, long n, double *out)
{
    for (long i = 0; i < n; i++) out[i] = w4o_bf16_to_double(b[i]);
}

/* The 16-bit type of activations and scales: 0 = IEEE binary16, 1 = bfloat16. */
typedef double (*decode16_fn)(uint16_t);
static decode16_fn decoder_for(int dtype)
{
    return dtype == 1 ? w4o_bf16_to_double : w4o_half_to_double;
}

/* ---------------------------------------------------------------------------
 * Nibble access with the sequential little-endian rule.
 * ------------------------------------------------------------------------- */
static inline unsigned nibble_at(const uint32_t *row_words, long idx)
{
    return (row_words[idx / 8] >> (4 * (idx % 8))) & 0xfu;
}

static inline long zero_words_per_row(int G) { return (G + 7) / 8; }

/* q: [N, K] bytes 0..15, z: [N, G] bytes 0..15 ->
 * qweight: [N, K/8] words, zeros: [N, ceil(G/8)] words. */
void w4o_pack(const uint8_t *q, const uint8_t *z, int N, int K, int group,
              uint32_t *qweight, uint32_t *zeros)
{
    int G = K / group;
    long KW = K / 8, ZW = zero_words_per_row(G);
    for (long n = 0; n < N; n++) {
        for (long w = 0; w < KW; w++) {
            uint32_t word = 0;
            for (int j = 0; j < 8; j++) {
                uint32_t v = q[n * K + w * 8 + j] & 0xfu;
                word |= v << (4 * j);
            }
            qweight[n * KW + w] = word;
        }
        for (long w = 0; w < ZW; w++) {
            uint32_t word = 0;
            for (int j = 0; j < 8; j++) {
                long g = w * 8 + j;
                if (g < G) word |= (uint32_t)(z[n * G + g] & 0xfu) << (4 * j);
            }
            zeros[n * ZW + w] = word;
        }
    }
}

void w4o_unpack(const uint32_t *qweight, const uint32_t *zeros, int N, int K,
                int group, uint8_t *q, uint8_t *z)
{
    int G = K / group;
    long KW = K / 8, ZW = zero_words_per_row(G);
    for (long n = 0; n < N; n++) {
        for (long k = 0; k < K; k++) q[n * K + k] = (uint8_t)nibble_at(qweight + n * KW, k);
        for (long g = 0; g < G; g++) z[n * G + g] = (uint8_t)nibble_at(zeros + n * ZW, g);
    }
}

/* w[n,k] = (q - z) * s, exact in binary64. */
void w4o_dequant(const uint32_t *qweight, const uint16_t *scales,
                 const uint32_t *zeros, int N, int K, int group, double *w)
{
    int G = K / group;
    long KW = K / 8, ZW = zero_words_per_row(G);
    for (long n = 0; n < N; n++) {
        for (long k = 0; k < K; k++) {
            long g = k / group;
            int qv = (int)nibble_at(qweight + n * KW, k);
            int zv = (int)nibble_at(zeros + n * ZW, g);
            double s = w4o_half_to_double(scales[n * G + g]);
            w[n * K + k] = (double)(qv - zv) * s;
        }
    }
}

/* One output element, the definition written out: dequantise each weight,
 * multiply by the activation, add in increasing k. */
static double linear_one(const uint16_t *x_row, const uint32_t *q_row,
                         const uint16_t *s_row, const uint32_t *z_row, int K,
                         int group, decode16_fn dec)
{
    double acc = 0.0;
    for (long k = 0; k < K; k++) {
        long g = k / group;
        int qv = (int)nibble_at(q_row, k);
        int zv = (int)nibble_at(z_row, g);
        double w = (double)(qv - zv) * dec(s_row[g]);
        acc += dec(x_row[k]) * w;
    }
    return acc;
}

typedef struct {
    const uint16_t *x;
    const uint32_t *qweight;
    const uint16_t *scales;
    const uint32_t *zeros;
    const int64_t *rows; /* NULL: all rows */
    int M, N, K, group, nrows, dtype;
    double *y; /* [M, nrows] */
    int t, nthreads;
} linear_job;

static void *linear_worker(void *arg)
{
    linear_job *j = (linear_job *)arg;
    int G = j->K / j->group;
    long KW = j->K / 8, ZW = zero_words_per_row(G);
    for (long i = j->t; i < j->nrows; i += j->nthreads) {
        long n = j->rows ? (long)j->rows[i] : i;
        for (long m = 0; m < j->M; m++) {
            j->y[m * j->nrows + i] =
                linear_one(j->x + m * (long)j->K, j->qweight + n * KW,
                           j->scales + n * G, j->zeros + n * ZW, j->K, j->group,
                           decoder_for(j->dtype));
        }
    }
    return NULL;
}

static void run_linear(linear_job base, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if (nthreads == 1) {
        base.t = 0;
        base.nthreads = 1;
        linear_worker(&base);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    linear_job *jobs = (linear_job *)malloc(sizeof(linear_job) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = base;
        jobs[t].t = t;
        jobs[t].nthreads = nthreads;
        if (pthread_create(&th[t], NULL, linear_worker, &jobs[t]) == 0) {
            started++;
        } else {
            /* could not start a thread: do its share here */
            linear_worker(&jobs[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; t++)
        if (th[t]) pthread_join(th[t], NULL);
    (void)started;
    free(jobs);
    free(th);
}

/* y[M, N] in binary64, rows split over nthreads host threads; x and scales
 * are 16-bit bit patterns of type dtype (0 binary16, 1 bfloat16). */
void w4o_linear_dt(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                   const uint32_t *zeros, int M, int N, int K, int group, int dtype,
                   double *y, int nthreads)
{
    linear_job j = {x, qweight, scales, zeros, NULL, M, N, K, group, N, dtype, y, 0, 1};
    run_linear(j, nthreads);
}

/* Sampled outputs: y[M, nrows] for the listed output rows only.  The weight
 * arrays still describe all N rows (row n starts at n * K/8 words). */
void w4o_linear_rows_dt(const uint16_t *x, const uint32_t *qweight,
                        const uint16_t *scales, const uint32_t *zeros, int M, int N,
                        int K, int group, int dtype, const int64_t *rows, int nrows,
                        double *y, int nthreads)
{
    linear_job j = {x, qweight, scales, zeros, rows, M, N, K, group, nrows, dtype, y, 0, 1};
    run_linear(j, nthreads);
}

/* Elementwise binary64 -> binary16 (RNE) over an array. */
void w4o_round_to_half(const double *v, long n, uint16_t *out)
{
    for (long i = 0; i < n; i++) out[i] = w4o_double_to_half(v[i]);
}

void w4o_half_array_to_double(const uint16_t *h, long n, double *out)
{
    for (long i = 0; i < n; i++) out[i] = w4o_half_to_double(h[i]);
}

/* ---- epilogues: the steps right after the linear.  SiLU-and-mul follows
 * the fused gate+up projection (Z100 thread, section 二, which lists it among
 * the MLP operators); the residual add follows the output projections (V100
 * article, third round of changes: the MLP's add-back of its input merged into
 * the matmul's output stage).  TEST INFRASTRUCTURE ONLY.
 *
 * SiLU and multiply.  y is [M, 2I]: columns 0..I-1 are the gate g, columns
 * I..2I-1 the up projection u (the fused gate+up layout, gate rows first).
 * out[m, n] = silu(g) * u with silu(g) = g / (1 + exp(-g)), in binary64. */
void w4o_silu_mul(const double *y, int M, int I, double *out)
{
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < I; ++n) {
            const double g = y[(long)m * 2 * I + n];
            const double u = y[(long)m * 2 * I + I + n];
            out[(long)m * I + n] = g / (1.0 + exp(-g)) * u;
        }
}

/* Residual add: out[i] = y[i] + r[i], r given as 16-bit bit patterns of type
 * dtype (0 binary16, 1 bfloat16). */
void w4o_add_residual_dt(const double *y, const uint16_t *r, long n, int dtype, double *out)
{
    decode16_fn dec = decoder_for(dtype);
    for (long i = 0; i < n; ++i) out[i] = y[i] + dec(r[i]);
}

/* ---- load-time repack (Z100 thread, section 四: checkpoint INT4 layouts are
 * transposed and repacked at load time, now at nibble level in 8 x 8 blocks,
 * without unpacking the whole matrix to int32).  TEST INFRASTRUCTURE ONLY.
 *
 * Transpose of a packed 4-bit matrix A [rows, cols]:
 *   src [rows, cols/8] words, packed along cols; element (r, c) sits at nibble
 *       position ((order >> 4*(c%8)) & 7) of word src[r][c/8] (order: eight
 *       nibbles, entry j = the position holding element j of a word's group of
 *       eight; 0x76543210 is the sequential order used everywhere else);
 *   dst [cols, ceil(rows/8)] words, packed along rows in sequential order:
 *       element (c, r) of A^T at nibble r%8 of word dst[c][r/8]; pad nibbles 0.
 * Written element by element from that definition. */
void w4o_transpose_u4(const uint32_t *src, long rows, long cols, uint32_t order,
                      uint32_t *dst)
{
    const long sw = cols / 8, dw = (rows + 7) / 8;
    memset(dst, 0, sizeof(uint32_t) * (size_t)(cols * dw));
    for (long r = 0; r < rows; ++r)
        for (long c = 0; c < cols; ++c) {
            const unsigned pos = (order >> (4 * (c % 8))) & 7u;
            const unsigned v = (src[r * sw + c / 8] >> (4 * pos)) & 15u;
            dst[c * dw + r / 8] |= (uint32_t)v << (4 * (r % 8));
        }
}

/* Transpose of a binary16 matrix (the per-group scales of a checkpoint laid
 * out [G, N], to this layout's [N, G]): dst[c][r] = src[r][c]. */
void w4o_transpose_u16(const uint16_t *src, long rows, long cols, uint16_t *dst)
{
    for (long r = 0; r < rows; ++r)
        for (long c = 0; c < cols; ++c) dst[c * rows + r] = src[r * cols + c];
}

/* ---- dense 16-bit linear (Z100 thread, section 六: weights dequantised to
 * fp16/bf16 once at load time, then a large-K, small-M GEMV with fp32
 * products and sums).  TEST INFRASTRUCTURE ONLY.
 * y[m, n] = sum_k x[m, k] * w[n, k] in binary64, increasing k; x [M, K] and
 * w [N, K] are 16-bit bit patterns of type dtype (0 binary16, 1 bfloat16).
 * Each product is exact in binary64 (at most 11 + 11 significant bits). */
void w4o_dense_linear(const uint16_t *x, const uint16_t *w, int M, int N, int K, int dtype,
                      double *y)
{
    decode16_fn dec = decoder_for(dtype);
    for (long m = 0; m < M; ++m)
        for (long n = 0; n < N; ++n) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k) acc += dec(x[m * K + k]) * dec(w[n * K + k]);
            y[m * N + n] = acc;
        }
}

/* The same for the listed output rows only: y[M, nrows]. */
void w4o_dense_linear_rows(const uint16_t *x, const uint16_t *w, int M, int N, int K,
                           int dtype, const int64_t *rows, int nrows, double *y)
{
    decode16_fn dec = decoder_for(dtype);
    (void)N;
    for (long m = 0; m < M; ++m)
        for (long i = 0; i < nrows; ++i) {
            const long n = (long)rows[i];
            double acc = 0.0;
            for (long k = 0; k < K; ++k) acc += dec(x[m * K + k]) * dec(w[n * K + k]);
            y[m * nrows + i] = acc;
        }
}

/* ---- mixture of experts (Z100 thread, section 七: tokens rearranged by
 * expert, the W4A16 expert small-M GEMV over packed INT4 experts, and the
 * weighted sum of each token's expert outputs).  TEST INFRASTRUCTURE ONLY.
 *
 * Slots: token t's j-th choice is slot s = t*k + j, routed to expert
 * ids[s] (0 <= ids[s] < E).
 *
 * Alignment: the slots grouped by expert, in increasing slot order within
 * an expert (a stable counting sort).  offsets[e] is the first sorted
 * position of expert e (offsets[E] = T*k), sorted[p] the slot at position
 * p, pos[s] the position of slot s. */
void w4o_moe_align(const int32_t *ids, int n_slots, int E, int32_t *sorted, int32_t *pos,
                   int32_t *offsets)
{
    for (int e = 0; e <= E; ++e) offsets[e] = 0;
    for (int s = 0; s < n_slots; ++s) offsets[ids[s] + 1]++;
    for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int s = 0; s < n_slots; ++s) {
        const int p = fill[ids[s]]++;
        sorted[p] = s;
        pos[s] = p;
    }
    free(fill);
}

/* Expert linears: y[s, n] = sum_k xs[m(s), k] * w_e[n, k], e = ids[s], with
 * the experts' packed layers stacked ([E, N, K/8] words, [E, N, G] scales,
 * [E, N, ceil(G/8)] zeros words).  The input row m(s) is the slot's token
 * t = s / k when per_slot is 0 (the first linear of an expert MLP), the slot
 * itself when per_slot is 1 (a later linear, fed by the slot's own
 * activations).  y is [T*k, N] in slot order, binary64. */
void w4o_moe_linear(const uint16_t *x, int per_slot, const uint32_t *qweight,
                    const uint16_t *scales, const uint32_t *zeros, const int32_t *ids, int T,
                    int k, int E, int N, int K, int group, int dtype, double *y)
{
    const int G = K / group;
    const long KW = K / 8, ZW = zero_words_per_row(G);
    decode16_fn dec = decoder_for(dtype);
    (void)E;
    for (long s = 0; s < (long)T * k; ++s) {
        const long e = ids[s], m = per_slot ? s : s / k;
        for (long n = 0; n < N; ++n) {
            const long row = e * N + n;
            y[s * N + n] = linear_one(x + m * K, qweight + row * KW, scales + row * G,
                                      zeros + row * ZW, K, group, dec);
        }
    }
}

/* Weighted sum per token: out[t, n] = sum_j wts[t*k + j] * y[t*k + j, n],
 * in binary64, j increasing. */
void w4o_moe_sum(const double *y, const double *wts, int T, int k, int N, double *out)
{
    for (long t = 0; t < T; ++t)
        for (long n = 0; n < N; ++n) {
            double acc = 0.0;
            for (long j = 0; j < k; ++j) acc += wts[t * k + j] * y[(t * k + j) * N + n];
            out[t * N + n] = acc;
        }
}
