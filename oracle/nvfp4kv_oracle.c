/*
 * nvfp4kv_oracle.c -- plain, slow CPU oracle for the NVFP4 paged KV cache.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline / reference legs may load this library.  The product library
 * (nvfp4_quantised_paged_gb300/) never calls it, and the two share no code,
 * headers, tables or constants.
 *
 * What it computes (source: "Accelerating Long-Context and Agentic Inference
 * with NVFP4 KV Cache", sections A3 and A2, Fig. 1):
 *   - each run of 16 consecutive K or V values along head_dim gets one FP8
 *     E4M3 block scale; the values become 4-bit E2M1 codes; an FP32 tensor
 *     scale (1.0 in all of the page's experiments, section A7) multiplies both;
 *   - the quantised values are written into a paged cache through a slot
 *     mapping (section A2, paths 1 and 2);
 *   - decode attention reads them back, dequantises, and runs softmax
 *     attention (section A2, path 3), here in fp64;
 *   - chunked prefill / extend dequantises a cached prefix into a contiguous
 *     workspace (section A2, path 2), here BF16, and the new chunk attends to
 *     [that prefix || its own K/V], causally within the chunk;
 *   - the FP32 tensor scale, fixed at 1.0 by the page, can be calibrated
 *     (section A4, outlook): g = amax / (6 * 448), the two-level NVFP4 rule.
 * The FP8 E4M3 cache the page compares against (section A4, the fp8_e4m3
 * baseline) is provided too.
 *
 * Readings taken where the page is silent:
 *   E4M3 is the OCP FP8 "fn" variant (bias 7, no infinities, S.1111.111 NaN,
 *   max 448).  Both codecs round to nearest, ties to the even code, and
 *   saturate at their largest finite value.  A scale or code is the rounding
 *   of the exact quotient (amax / (6 g), x / (scale g), x / g): the oracle
 *   decides it by comparing the dividend with exact products of the divisor
 *   and the grid's values and midpoints, never by forming the quotient.  A
 *   dequantised value stored in BF16 (the prefix workspace) is the exact
 *   product e2m1 * e4m3 * g rounded to BF16 once.  The tensor scale g is a
 *   positive normal FP32 number.  A block whose scale rounds to zero stores
 *   zero magnitudes and keeps each element's sign, like every other element
 *   that rounds to zero.
 *   Nibble order: element 2i in the low nibble of byte i.  Query head h reads
 *   KV head h / G (G = query heads per KV head).
 *
 * Pool layout (one slab per (page, kv_head), slabs ordered page-major).  A
 * slab of P tokens is P/16 groups of 16 consecutive tokens, each group laid out
 * as (row r = 0..15 of the group):
 *   NVFP4 (2304 B): K codes [16][64] | K scales [16][8] | V codes [16][64] |
 *                   V scales [8][16] (block-major: block j of row r at [j][r])
 *   FP8   (4096 B): K codes [16][128] | V codes [16][128]
 * Token t of a sequence lives in page block_table[t / P] at row t % P.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC -pthread -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENONFINITE -2
#define ORACLE_ESLOT -3
#define ORACLE_EPAGE -4

#define ORACLE_DTYPE_NVFP4 0
#define ORACLE_DTYPE_FP8 1

#define HEAD_DIM 128
#define BLOCK 16

/* ------------------------------------------------------------------ */
/* Scalar formats                                                       */
/* ------------------------------------------------------------------ */

/* BF16 bit pattern -> exact double. */
double oracle_bf16_value(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Round a float to BF16, nearest-even (the value is finite). */
uint16_t oracle_bf16_from_float(float f)
{
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    if ((w & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((w >> 16) | 0x40u); /* NaN */
    uint32_t lower = w & 0xffffu;
    uint32_t upper = w >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* E4M3: sign bit, 4 exponent bits (bias 7), 3 mantissa bits. */
double oracle_e4m3_value(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -mag : mag;
}

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Magnitudes of codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_value(uint8_t code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[code & 7];
    return (code & 8) ? -v : v;
}

/* Round |a| to the nearest of the ascending magnitudes vals[0..n-1] (codes
 * 0..n-1, vals[0] = 0), ties to the even code, saturating at vals[n-1].
 * The bracketing pair and its midpoint are exact in double. */
static int round_to_table(double a, const double *vals, int n)
{
    if (a >= vals[n - 1]) return n - 1;
    int hi = 1;
    while (vals[hi] < a) hi++;
    int lo = hi - 1;
    if (vals[hi] == a) return hi;
    double mid = 0.5 * (vals[lo] + vals[hi]);
    if (a < mid) return lo;
    if (a > mid) return hi;
    return (lo % 2 == 0) ? lo : hi;
}

/* The same rounding applied to the exact quotient a / den (a >= 0, den > 0),
 * decided without forming it: a / den < v  <=>  a < v * den.  Every product
 * compared here is exact in double: den is 6 g, scale * g or g (at most 27
 * significant bits for a 24-bit g), a grid value or midpoint has at most 5,
 * and the exponents stay far inside double's range for a normal FP32 g. */
static int round_quotient_to_table(double a, double den, const double *vals, int n)
{
    if (a >= vals[n - 1] * den) return n - 1;
    int hi = 1;
    while (vals[hi] * den < a) hi++;
    int lo = hi - 1;
    if (vals[hi] * den == a) return hi;
    double mid = 0.5 * (vals[lo] + vals[hi]);
    if (a < mid * den) return lo;
    if (a > mid * den) return hi;
    return (lo % 2 == 0) ? lo : hi;
}

/* Round a finite double to BF16, nearest-even, once: 8 significant bits for
 * magnitudes from 2^-126 up, steps of 2^-133 below (subnormals), infinity
 * from 2^128 * (1 - 2^-9) up. */
uint16_t oracle_bf16_from_double(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                       /* a = m 2^e, m in [0.5, 1) */
    int step_exp = (e - 1 >= -126) ? e - 8 : -133;
    double q = ldexp(a, -step_exp);     /* a in units of the BF16 step: exact */
    double f = floor(q), r = q - f;
    if (r > 0.5 || (r == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;
    double v = ldexp(f, step_exp);      /* the rounded magnitude */
    if (v >= ldexp(1.0, 128)) return sign | 0x7f80u;
    if (v < ldexp(1.0, -126)) return sign | (uint16_t)f;      /* subnormal (or 0x0080 at the boundary) */
    int ve;
    double vm = frexp(v, &ve);          /* v = vm 2^ve, vm in [0.5, 1) */
    uint16_t mant = (uint16_t)(ldexp(vm, 8) - 128.0);
    return sign | (uint16_t)((ve - 1 + 127) << 7) | mant;
}

static double e4m3_mags[127]; /* codes 0x00..0x7E */
static double e2m1_mags[8];
static pthread_once_t tables_once = PTHREAD_ONCE_INIT;
static void build_tables(void)
{
    for (int c = 0; c < 127; c++) e4m3_mags[c] = oracle_e4m3_value((uint8_t)c);
    for (int c = 0; c < 8; c++) e2m1_mags[c] = oracle_e2m1_value((uint8_t)c);
}

/* Round-to-nearest-even, saturating, keeping the sign (so -0 -> 0x80). */
uint8_t oracle_e4m3_encode(float x)
{
    pthread_once(&tables_once, build_tables);
    int c = round_to_table(fabs((double)x), e4m3_mags, 127);
    return (uint8_t)(signbit(x) ? (0x80 | c) : c);
}

uint8_t oracle_e2m1_encode(float x)
{
    pthread_once(&tables_once, build_tables);
    int c = round_to_table(fabs((double)x), e2m1_mags, 8);
    return (uint8_t)(signbit(x) ? (8 | c) : c);
}

/* Batch form used by the brute-force tests: code_i = E2M1(fl32(x_i / d_i)). */
void oracle_e2m1_encode_quotients(const float *x, const float *d, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e2m1_encode(x[i] / d[i]);
}

void oracle_e4m3_encode_many(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------ */
/* NVFP4 block quantisation                                             */
/* ------------------------------------------------------------------ */

static int valid_tensor_scale(float g) { return isfinite(g) && g >= 0x1p-126f; }

/* Quantise 16 BF16 values with tensor scale g:
 *   amax  = max |x_i|
 *   scale = E4M3(amax / (6 g))           (6 = largest E2M1 magnitude)
 *   code_i = E2M1(x_i / (scale g)),  or a signed zero when scale is 0,
 * each the rounding of the exact quotient.  Codes are returned one per byte
 * (sign in bit 3). */
int oracle_quantize_block16(const uint16_t *x_bf16, float g, uint8_t *codes16, uint8_t *scale_code)
{
    pthread_once(&tables_once, build_tables);
    if (!valid_tensor_scale(g)) return ORACLE_EINVAL;
    double x[BLOCK];
    double amax = 0.0;
    for (int i = 0; i < BLOCK; i++) {
        x[i] = oracle_bf16_value(x_bf16[i]);
        if (!isfinite(x[i])) return ORACLE_ENONFINITE;
        if (fabs(x[i]) > amax) amax = fabs(x[i]);
    }
    uint8_t s = (uint8_t)round_quotient_to_table(amax, 6.0 * (double)g, e4m3_mags, 127);
    double sd = oracle_e4m3_value(s);
    for (int i = 0; i < BLOCK; i++) {
        int c = (sd == 0.0) ? 0 : round_quotient_to_table(fabs(x[i]), sd * (double)g, e2m1_mags, 8);
        codes16[i] = (uint8_t)(signbit(x[i]) ? (8 | c) : c);
    }
    *scale_code = s;
    return ORACLE_OK;
}

/* Dequantised value as stored by the cache: e2m1 * e4m3 * g (exact in double). */
/*
 * Per-tensor FP32 global scale (section A4, outlook: calibrating the tensor
 * scale that the page fixes at 1.0).  amax = the largest finite |x| over the
 * n BF16 values; g = amax / (6 * 448) in FP32, so that the block holding amax
 * gets E4M3's largest scale; 1.0 when amax is 0 (nothing to calibrate).
 */
float oracle_calibrate_global_scale(const uint16_t *x_bf16, int64_t n)
{
    double amax = 0.0;
    for (int64_t i = 0; i < n; i++) {
        const double a = fabs(oracle_bf16_value(x_bf16[i]));
        if (isfinite(a) && a > amax) amax = a;
    }
    if (amax == 0.0) return 1.0f;
    const float largest_e2m1 = 6.0f, largest_e4m3 = 448.0f;
    return (float)amax / (largest_e2m1 * largest_e4m3);
}

static double nvfp4_dequant(uint8_t code, uint8_t scale, float g)
{
    return oracle_e2m1_value(code) * oracle_e4m3_value(scale) * (double)g;
}

/* ------------------------------------------------------------------ */
/* Pool layout                                                          */
/* ------------------------------------------------------------------ */

int64_t oracle_slab_bytes(int dtype, int page_size)
{
    if (page_size < 16 || page_size % 16) return -1;
    if (dtype == ORACLE_DTYPE_NVFP4) return (int64_t)page_size * (64 + 8 + 64 + 8);
    if (dtype == ORACLE_DTYPE_FP8) return (int64_t)page_size * (128 + 128);
    return -1;
}

typedef struct {
    uint8_t *pool;
    int64_t num_pages;
    int page_size;
    int num_kv_heads;
    int dtype;
    float gk, gv;
} pool_t;

static uint8_t *slab_ptr(const pool_t *p, int64_t page, int kv)
{
    return p->pool + (page * p->num_kv_heads + kv) * oracle_slab_bytes(p->dtype, p->page_size);
}

/* Row `row` of K (which = 0) or V (which = 1) of one slab: its codes, and the
 * scale byte of block `blk` (16-token groups, see the header). */
static uint8_t *codes_row(const pool_t *p, uint8_t *slab, int which, int row)
{
    int grp = row / 16, r = row % 16;
    if (p->dtype == ORACLE_DTYPE_NVFP4) return slab + grp * 2304 + (which ? 1152 : 0) + r * 64;
    return slab + grp * 4096 + (which ? 2048 : 0) + r * 128;
}

static uint8_t *scale_ptr(const pool_t *p, uint8_t *slab, int which, int row, int blk)
{
    (void)p;
    int grp = row / 16, r = row % 16;
    if (which == 0) return slab + grp * 2304 + 1024 + r * 8 + blk;
    return slab + grp * 2304 + 2176 + blk * 16 + r;
}

/* Dequantise one head_dim row of K or V into out[128] (double). */
static void dequant_row(const pool_t *p, int64_t page, int kv, int which, int row, double *out)
{
    uint8_t *slab = slab_ptr(p, page, kv);
    uint8_t *c = codes_row(p, slab, which, row);
    float g = which ? p->gv : p->gk;
    if (p->dtype == ORACLE_DTYPE_NVFP4) {
        for (int d = 0; d < HEAD_DIM; d++) {
            uint8_t byte = c[d / 2];
            uint8_t code = (d % 2 == 0) ? (byte & 15) : (byte >> 4);
            out[d] = nvfp4_dequant(code, *scale_ptr(p, slab, which, row, d / BLOCK), g);
        }
    } else {
        for (int d = 0; d < HEAD_DIM; d++) out[d] = oracle_e4m3_value(c[d]) * (double)g;
    }
}

/* ------------------------------------------------------------------ */
/* Quantise-append (section A2, paths 1 and 2: new K/V written into pages) */
/* ------------------------------------------------------------------ */

/* Quantise one head_dim row of BF16 values and store it at (page, kv, row). */
static int store_row(const pool_t *p, int64_t page, int kv, int which, int row, const uint16_t *x)
{
    pthread_once(&tables_once, build_tables);
    uint8_t *slab = slab_ptr(p, page, kv);
    uint8_t *c = codes_row(p, slab, which, row);
    float g = which ? p->gv : p->gk;
    if (p->dtype == ORACLE_DTYPE_NVFP4) {
        for (int b = 0; b < HEAD_DIM / BLOCK; b++) {
            uint8_t codes[BLOCK];
            int rc = oracle_quantize_block16(x + b * BLOCK, g, codes, scale_ptr(p, slab, which, row, b));
            if (rc) return rc;
            for (int i = 0; i < BLOCK / 2; i++)
                c[b * 8 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
        }
    } else {
        if (!valid_tensor_scale(g)) return ORACLE_EINVAL;
        for (int d = 0; d < HEAD_DIM; d++) {
            double v = oracle_bf16_value(x[d]);
            if (!isfinite(v)) return ORACLE_ENONFINITE;
            int m = round_quotient_to_table(fabs(v), (double)g, e4m3_mags, 127);
            c[d] = (uint8_t)(signbit(v) ? (0x80 | m) : m);
        }
    }
    return ORACLE_OK;
}

/* k, v: BF16 [num_tokens][token_stride elements], head kv at offset kv*128.
 * slot_mapping[t] = page * P + row; a negative slot skips the token. */
int oracle_quantize_append(uint8_t *pool, int64_t num_pages, int page_size, int num_kv_heads, int dtype,
                           float gk, float gv, const uint16_t *k, const uint16_t *v, int64_t num_tokens,
                           int64_t token_stride, const int64_t *slot_mapping)
{
    pool_t p = {pool, num_pages, page_size, num_kv_heads, dtype, gk, gv};
    if (oracle_slab_bytes(dtype, page_size) < 0 || token_stride < (int64_t)num_kv_heads * HEAD_DIM)
        return ORACLE_EINVAL;
    for (int64_t t = 0; t < num_tokens; t++) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_pages * page_size) return ORACLE_ESLOT;
        int64_t page = slot / page_size;
        int row = (int)(slot % page_size);
        for (int kv = 0; kv < num_kv_heads; kv++) {
            int rc = store_row(&p, page, kv, 0, row, k + t * token_stride + kv * HEAD_DIM);
            if (!rc) rc = store_row(&p, page, kv, 1, row, v + t * token_stride + kv * HEAD_DIM);
            if (rc) return rc;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Decode attention in fp64 (section A2, path 3)                        */
/* ------------------------------------------------------------------ */

/* A source of dequantised rows: fills out[128] with row t of K (which = 0)
 * or V (which = 1) of one sequence and one KV head; returns non-zero when the
 * row cannot be read. */
typedef int (*row_fn)(void *ctx, int which, int64_t t, double *out);

/* out[h][:] = sum_t softmax_t(sm_scale * q_h . k_t) v_t over the n tokens of
 * one sequence, for the G query heads q[G][128] that share one KV head.
 * Two passes: the scores (max-shifted softmax needs all of them), then the
 * probability-weighted sum of V.  scores has room for G * n values.
 *
 * spread (may be NULL): spread[h][d] = sum_t w_t |v_t[d] - out[h][d]| with
 * w_t the softmax weights -- how far the values lie from the output on
 * average.  Not part of the method: the parity tests bound a kernel's error
 * by it (rounding each weight by a relative e moves the output by at most
 * e * spread, to first order), and a third pass over V computes it. */
static int attend_group(const double *q, int G, row_fn rows, void *ctx, int64_t n, double sm_scale, double *out,
                        double *scores, double *spread)
{
    double krow[HEAD_DIM], vrow[HEAD_DIM], m[16], l[16];
    for (int h = 0; h < G; h++) {
        for (int d = 0; d < HEAD_DIM; d++) out[h * HEAD_DIM + d] = 0.0;
        m[h] = -INFINITY;
        l[h] = 0.0;
    }
    if (spread)
        for (int i = 0; i < G * HEAD_DIM; i++) spread[i] = 0.0;
    if (n == 0) return ORACLE_OK;
    for (int64_t t = 0; t < n; t++) {
        if (rows(ctx, 0, t, krow)) return ORACLE_EPAGE;
        for (int h = 0; h < G; h++) {
            double s = 0.0;
            for (int d = 0; d < HEAD_DIM; d++) s += q[h * HEAD_DIM + d] * krow[d];
            s *= sm_scale;
            scores[h * n + t] = s;
            if (s > m[h]) m[h] = s;
        }
    }
    for (int64_t t = 0; t < n; t++) {
        if (rows(ctx, 1, t, vrow)) return ORACLE_EPAGE;
        for (int h = 0; h < G; h++) {
            double pt = exp(scores[h * n + t] - m[h]);
            l[h] += pt;
            for (int d = 0; d < HEAD_DIM; d++) out[h * HEAD_DIM + d] += pt * vrow[d];
        }
    }
    for (int h = 0; h < G; h++)
        for (int d = 0; d < HEAD_DIM; d++) out[h * HEAD_DIM + d] /= l[h];
    if (spread) {
        for (int i = 0; i < G * HEAD_DIM; i++) spread[i] = 0.0;
        for (int64_t t = 0; t < n; t++) {
            if (rows(ctx, 1, t, vrow)) return ORACLE_EPAGE;
            for (int h = 0; h < G; h++) {
                double wt = exp(scores[h * n + t] - m[h]) / l[h];
                for (int d = 0; d < HEAD_DIM; d++)
                    spread[h * HEAD_DIM + d] += wt * fabs(vrow[d] - out[h * HEAD_DIM + d]);
            }
        }
    }
    return ORACLE_OK;
}

/* Rows of a cached sequence, read through its block table. */
typedef struct {
    const pool_t *p;
    const int32_t *pages; /* this sequence's block-table row */
    int kv;
} paged_rows_t;

static int paged_row(void *ctx, int which, int64_t t, double *out)
{
    paged_rows_t *c = (paged_rows_t *)ctx;
    int64_t page = c->pages[t / c->p->page_size];
    if (page < 0 || page >= c->p->num_pages) return 1;
    dequant_row(c->p, page, c->kv, which, (int)(t % c->p->page_size), out);
    return 0;
}

typedef struct {
    const pool_t *p;
    const uint16_t *q;
    int batch, num_q_heads;
    const int32_t *block_table;
    int max_pages;
    const int32_t *seq_lens;
    double sm_scale;
    double *out, *spread;
    int64_t next_unit; /* shared work counter */
    pthread_mutex_t lock;
    int status;
} decode_job_t;

static int64_t take_unit(decode_job_t *j)
{
    pthread_mutex_lock(&j->lock);
    int64_t u = j->next_unit++;
    pthread_mutex_unlock(&j->lock);
    return u;
}

static void set_status(decode_job_t *j, int rc)
{
    pthread_mutex_lock(&j->lock);
    if (!j->status) j->status = rc;
    pthread_mutex_unlock(&j->lock);
}

/* One unit = one (sequence, kv_head). */
static void *decode_worker(void *arg)
{
    decode_job_t *j = (decode_job_t *)arg;
    const pool_t *p = j->p;
    int Hkv = p->num_kv_heads, G = j->num_q_heads / Hkv;
    int64_t units = (int64_t)j->batch * Hkv;
    double qd[16 * HEAD_DIM];
    for (;;) {
        int64_t u = take_unit(j);
        if (u >= units) break;
        int b = (int)(u / Hkv), kv = (int)(u % Hkv);
        int64_t n = j->seq_lens[b];
        if (n < 0 || n > (int64_t)j->max_pages * p->page_size) {
            set_status(j, ORACLE_EINVAL);
            continue;
        }
        for (int h = 0; h < G; h++)
            for (int d = 0; d < HEAD_DIM; d++)
                qd[h * HEAD_DIM + d] =
                    oracle_bf16_value(j->q[((int64_t)b * j->num_q_heads + kv * G + h) * HEAD_DIM + d]);
        double *scores = malloc(sizeof(double) * (size_t)G * (size_t)(n > 0 ? n : 1));
        paged_rows_t ctx = {p, j->block_table + (int64_t)b * j->max_pages, kv};
        const int64_t o = ((int64_t)b * j->num_q_heads + (int64_t)kv * G) * HEAD_DIM;
        int rc = attend_group(qd, G, paged_row, &ctx, n, j->sm_scale, j->out + o, scores,
                              j->spread ? j->spread + o : NULL);
        free(scores);
        if (rc) set_status(j, rc);
    }
    return NULL;
}

static int resolve_threads(int nthreads)
{
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* q: BF16 [batch][num_q_heads][128]; out and spread (may be NULL): double
 * [batch][num_q_heads][128].  nthreads <= 0 uses every online core; the units
 * are independent, so the thread count does not change any result. */
int oracle_decode_attention(const uint8_t *pool, int64_t num_pages, int page_size, int num_kv_heads, int dtype,
                            float gk, float gv, const uint16_t *q, int batch, int num_q_heads,
                            const int32_t *block_table, int max_pages, const int32_t *seq_lens, double sm_scale,
                            double *out, double *spread, int nthreads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 16 ||
        oracle_slab_bytes(dtype, page_size) < 0)
        return ORACLE_EINVAL;
    pool_t p = {(uint8_t *)pool, num_pages, page_size, num_kv_heads, dtype, gk, gv};
    decode_job_t j = {&p, q, batch, num_q_heads, block_table, max_pages, seq_lens, sm_scale, out, spread, 0,
                      PTHREAD_MUTEX_INITIALIZER, 0};
    int nt = resolve_threads(nthreads);
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nt);
    for (int i = 0; i < nt; i++) pthread_create(&th[i], NULL, decode_worker, &j);
    for (int i = 0; i < nt; i++) pthread_join(th[i], NULL);
    free(th);
    return j.status;
}

/* Rows of one sequence given as BF16 K/V: each row is quantised and
 * dequantised exactly as the cache would store it. */
typedef struct {
    const uint16_t *k, *v;
    int64_t row_stride;
    pool_t p; /* a one-page scratch pool */
    int status;
} bf16_rows_t;

static int bf16_row(void *ctx, int which, int64_t t, double *out)
{
    bf16_rows_t *c = (bf16_rows_t *)ctx;
    int rc = store_row(&c->p, 0, 0, which, 0, (which ? c->v : c->k) + t * c->row_stride);
    if (rc) {
        c->status = rc;
        return 1;
    }
    dequant_row(&c->p, 0, 0, which, 0, out);
    return 0;
}

/* Attention of one sequence straight from its BF16 K/V (no pool).
 * k, v: BF16 rows [n][row_stride] with the KV head's 128 values at the row
 * start; q: BF16 [G][128]; out: double [G][128].  Used for sampled checks of
 * very long sequences and for CPU timing. */
int oracle_sequence_attention(const uint16_t *q, int G, const uint16_t *k, const uint16_t *v, int64_t n,
                              int64_t row_stride, int dtype, float gk, float gv, double sm_scale, double *out,
                              double *spread)
{
    uint8_t slab[4096]; /* one 16-token group; rows are quantised into row 0 */
    if (G < 1 || G > 16 || oracle_slab_bytes(dtype, 16) < 0) return ORACLE_EINVAL;
    bf16_rows_t ctx = {k, v, row_stride, {slab, 1, 16, 1, dtype, gk, gv}, 0};
    double qd[16 * HEAD_DIM];
    for (int i = 0; i < G * HEAD_DIM; i++) qd[i] = oracle_bf16_value(q[i]);
    double *scores = malloc(sizeof(double) * (size_t)G * (size_t)(n > 0 ? n : 1));
    int rc = attend_group(qd, G, bf16_row, &ctx, n, sm_scale, out, scores, spread);
    free(scores);
    return ctx.status ? ctx.status : rc;
}

/* ------------------------------------------------------------------ */
/* Prefix dequant into a BF16 workspace (section A2, path 2)            */
/* ------------------------------------------------------------------ */

/* For request r and prefix token t < prefix_lens[r], row cu_prefix_lens[r] + t
 * of k_ws / v_ws ([total][num_kv_heads][128] BF16) receives the dequantised
 * token, the exact e2m1 * e4m3 * g rounded to BF16 once (exact when the
 * tensor scale is 1.0: every e2m1 x e4m3 product has at most 6 significant
 * bits). */
int oracle_prefix_dequant(const uint8_t *pool, int64_t num_pages, int page_size, int num_kv_heads, int dtype,
                          float gk, float gv, const int32_t *block_table, int max_pages, const int32_t *prefix_lens,
                          const int32_t *cu_prefix_lens, int num_reqs, uint16_t *k_ws, uint16_t *v_ws)
{
    pool_t p = {(uint8_t *)pool, num_pages, page_size, num_kv_heads, dtype, gk, gv};
    if (oracle_slab_bytes(dtype, page_size) < 0) return ORACLE_EINVAL;
    double row[HEAD_DIM];
    for (int r = 0; r < num_reqs; r++) {
        int64_t n = prefix_lens[r];
        if (n < 0 || n > (int64_t)max_pages * page_size) return ORACLE_EINVAL;
        for (int64_t t = 0; t < n; t++) {
            int64_t page = block_table[(int64_t)r * max_pages + t / page_size];
            if (page < 0 || page >= num_pages) return ORACLE_EPAGE;
            int64_t dst_row = (int64_t)cu_prefix_lens[r] + t;
            for (int kv = 0; kv < num_kv_heads; kv++) {
                for (int which = 0; which < 2; which++) {
                    uint16_t *dst = (which ? v_ws : k_ws) + (dst_row * num_kv_heads + kv) * HEAD_DIM;
                    dequant_row(&p, page, kv, which, (int)(t % page_size), row);
                    for (int d = 0; d < HEAD_DIM; d++) dst[d] = oracle_bf16_from_double(row[d]);
                }
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Extend attention (section A2, path 2)                                */
/* ------------------------------------------------------------------ */

/* Path 2's attention consumes two KV sources: the cached prefix as the
 * workspace holds it (BF16 rows, written by prefix dequant) and the current
 * chunk's own K/V.  Chunk token i of request r attends to all n_r prefix
 * tokens and to chunk tokens 0..i (causal), i.e. to the first n_r + i + 1
 * keys of [prefix || chunk]. */
typedef struct {
    const uint16_t *k_pre, *v_pre, *k_new, *v_new;
    int64_t pre0, new0, n_prefix; /* first workspace row, first chunk row, prefix length */
    int num_kv_heads, kv;
} extend_rows_t;

static int extend_row(void *ctx, int which, int64_t t, double *out)
{
    extend_rows_t *c = (extend_rows_t *)ctx;
    const uint16_t *src;
    if (t < c->n_prefix)
        src = (which ? c->v_pre : c->k_pre) + ((c->pre0 + t) * c->num_kv_heads + c->kv) * HEAD_DIM;
    else
        src = (which ? c->v_new : c->k_new) + ((c->new0 + t - c->n_prefix) * c->num_kv_heads + c->kv) * HEAD_DIM;
    for (int d = 0; d < HEAD_DIM; d++) out[d] = oracle_bf16_value(src[d]);
    return 0;
}

typedef struct {
    const uint16_t *q, *k_pre, *v_pre, *k_new, *v_new;
    const int32_t *cu_prefix, *cu_q;
    int num_reqs, num_q_heads, num_kv_heads;
    double sm_scale;
    double *out, *spread;
    int64_t total_units, next_unit;
    pthread_mutex_t lock;
    int status;
} extend_job_t;

/* One unit = one (chunk token, kv head) of the flattened chunk tokens. */
static void *extend_worker(void *arg)
{
    extend_job_t *j = (extend_job_t *)arg;
    const int Hkv = j->num_kv_heads, G = j->num_q_heads / Hkv;
    double qd[16 * HEAD_DIM];
    for (;;) {
        pthread_mutex_lock(&j->lock);
        int64_t u = j->next_unit++;
        pthread_mutex_unlock(&j->lock);
        if (u >= j->total_units) break;
        int64_t row = u / Hkv;
        int kv = (int)(u % Hkv);
        int r = 0;
        while (r + 1 < j->num_reqs && j->cu_q[r + 1] <= row) r++;
        int64_t i = row - j->cu_q[r];
        int64_t n_prefix = (int64_t)j->cu_prefix[r + 1] - j->cu_prefix[r];
        for (int h = 0; h < G; h++)
            for (int d = 0; d < HEAD_DIM; d++)
                qd[h * HEAD_DIM + d] = oracle_bf16_value(j->q[(row * j->num_q_heads + kv * G + h) * HEAD_DIM + d]);
        extend_rows_t ctx = {j->k_pre, j->v_pre, j->k_new, j->v_new, j->cu_prefix[r], j->cu_q[r], n_prefix, Hkv, kv};
        int64_t n = n_prefix + i + 1;
        double *scores = malloc(sizeof(double) * (size_t)G * (size_t)n);
        const int64_t o = (row * j->num_q_heads + (int64_t)kv * G) * HEAD_DIM;
        int rc = attend_group(qd, G, extend_row, &ctx, n, j->sm_scale, j->out + o, scores,
                              j->spread ? j->spread + o : NULL);
        free(scores);
        if (rc) {
            pthread_mutex_lock(&j->lock);
            if (!j->status) j->status = rc;
            pthread_mutex_unlock(&j->lock);
        }
    }
    return NULL;
}

/* q: BF16 [total_q][num_q_heads][128]; k_new, v_new: BF16 [total_q][num_kv_heads][128]
 * (request r's chunk = rows cu_q[r] .. cu_q[r+1]-1); k_pre, v_pre: BF16
 * [total_prefix][num_kv_heads][128] (request r's prefix = rows cu_prefix[r] ..
 * cu_prefix[r+1]-1, e.g. the output of oracle_prefix_dequant); out: double
 * [total_q][num_q_heads][128]. */
int oracle_extend_attention(const uint16_t *q, const uint16_t *k_pre, const uint16_t *v_pre, const int32_t *cu_prefix,
                            const uint16_t *k_new, const uint16_t *v_new, const int32_t *cu_q, int num_reqs,
                            int num_q_heads, int num_kv_heads, double sm_scale, double *out, double *spread,
                            int nthreads)
{
    if (num_reqs < 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || num_q_heads / num_kv_heads > 16)
        return ORACLE_EINVAL;
    for (int r = 0; r < num_reqs; r++)
        if (cu_q[r + 1] < cu_q[r] || cu_prefix[r + 1] < cu_prefix[r]) return ORACLE_EINVAL;
    int64_t total_q = num_reqs ? cu_q[num_reqs] - cu_q[0] : 0;
    if (num_reqs && cu_q[0] != 0) return ORACLE_EINVAL;
    extend_job_t j = {q, k_pre, v_pre, k_new, v_new, cu_prefix, cu_q, num_reqs, num_q_heads, num_kv_heads, sm_scale,
                      out, spread, total_q * num_kv_heads, 0, PTHREAD_MUTEX_INITIALIZER, 0};
    int nt = resolve_threads(nthreads);
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nt);
    for (int i = 0; i < nt; i++) pthread_create(&th[i], NULL, extend_worker, &j);
    for (int i = 0; i < nt; i++) pthread_join(th[i], NULL);
    free(th);
    return j.status;
}
