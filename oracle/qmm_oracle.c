/*
 * qmm_oracle.c -- plain, slow CPU oracle for the quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code with the CUDA path.
 *
 * What it computes (fp64 for floating point, int64 for integers):
 *
 *  1. Bitstream.  Column n of a b-bit weight matrix is its own byte string of
 *     K*b/8 bytes starting at packed + n*K*b/8.  Code k occupies stream bits
 *     [k*b, k*b+b); stream bit i is bit (i mod 8), LSB = 0, of byte i/8; bit
 *     j of the code is stream bit k*b+j.  This is the "little-endian
 *     bitstream along K" of the workloads; the pages themselves only say that
 *     arbitrary-width codes are loaded as raw bytes and reinterpreted
 *     (Tilus review, pith_extraction.core_discovery) and that INT4 is packed
 *     contiguously in bytes (BitLLM sec. 4.3, Fig. 8(a)).
 *  2. Dequantization, BitLLM Eq. (5): w = s * (q - z), with one scale s and
 *     one zero z per group of G consecutive codes along K (BitLLM sec. 2.2,
 *     per-group granularity).  q - z is exact in integers, then multiplied
 *     by the fp16 scale widened exactly to fp64.
 *  3. Matmul: y[m][n] = sum_k x[m][k] * w[n][k], fp64, k ascending.
 *  4. W4A8 (BitLLM sec. 4.3-4.4): signed int4 weights (two's complement
 *     nibbles, even k in the low nibble, no zero point) and int8
 *     activations; the integer core is the dp4a identity
 *     r + sum_i a_i*b_i accumulated per group of G into an integer; the
 *     epilogue is y = sa[m] * sum_g ws[n][g] * acc[m][n][g] in fp64.  The
 *     same core with signed 8-bit weights (two's-complement bytes) is the
 *     W8A8 precision BitLLM evaluates beside W4A8 (Experiment Setup).
 *  6. Signed b-bit weights (Tilus review: signed integer types of any width
 *     among the arbitrary low-precision types).  A code is b-bit two's
 *     complement, w = c * s with no zero point.  Flipping the top bit of
 *     every code (c xor 2^(b-1), "offset binary") turns such a stream into one
 *     whose unsigned codes u satisfy c = u - 2^(b-1): oracle_flip_sign flips
 *     stream bit k*b + b-1 of every code k, one bit at a time.
 *  7. Float b-bit weights (Tilus review: float3-float8 among the arbitrary
 *     low-precision types; the pages fix no exponent / mantissa split and no
 *     special values).  Reading: a code is 1 sign bit, e exponent bits and m
 *     mantissa bits (b = 1 + e + m, top to bottom), bias 2^(e-1) - 1, every
 *     encoding finite: E > 0 gives (-1)^s 2^(E - bias) (1 + M / 2^m), E = 0
 *     gives (-1)^s 2^(1 - bias) M / 2^m.  w = value * s per group.
 *  5. Per-token int8 quantization of fp16 activations (BitLLM sec. 2.2,
 *     Eq. (1), q = clip(round(x/s) + z, q_min, q_max), with the int8 range
 *     of Fig. 2(a)).  Reading: symmetric per token (z = 0), s = the token's
 *     largest |x| divided by 127 and stored as fp16, rounding half to even,
 *     q = 0 for a token whose stored scale is 0.  The quotients that decide
 *     the integers are single-precision IEEE divisions (the precision the
 *     GPU kernel uses too).
 *  8. Lane-interleaved int4 layout (BitLLM sec. 4.3, Fig. 6 and Fig. 8(b)):
 *     eight 4-bit codes per 32-bit little-endian word, with nibble slot s
 *     at bits [4s, 4s+4); slot 2j holds code j and slot 2j+1 code j+4 of the
 *     word's eight (j = 0..3), so the slots read 0 4 1 5 2 6 3 7, the order
 *     Fig. 6 prints.  Then the bytes of W & 0x0F0F0F0F are codes 0..3 and
 *     the bytes of (W & 0xF0F0F0F0) >> 4 are codes 4..7: one shift and two
 *     masks give four byte-aligned values each (Fig. 8(b); the page prints
 *     the first mask garbled as 0xF0F0F0F0 for both halves).
 *  9. Fragment-ordered ("tile16") layout, a reading of the pre-permuted,
 *     MMA-fragment-ordered bitstreams the pages point to (BitLLM sec. 4.3:
 *     weights are re-laid out offline so that each thread's loads are
 *     contiguous and need no reordering; the pages fix no order for a
 *     tensor-core fragment).  Rows are taken in tiles of 16 (the last tile
 *     padded with zero codes), K in blocks of 64 codes.  Unit (T, kb) holds
 *     rows 16T..16T+15 of codes 64kb..64kb+63 in 128*b bytes at byte
 *     (T*(K/64) + kb)*128*b.  Inside it, run r = (h*8 + g)*4 + t (h = 0..1,
 *     g = 0..7, t = 0..3) is codes 16t..16t+15 of the block for row
 *     16T + 8h + g, at bytes [2*b*r, 2*b*r + 2*b), code c of the run at bits
 *     [c*b, c*b + b) (LSB first).  Runs are the 16-code slices one
 *     tensor-core thread reads per row: thread (g, t) of a warp reads runs
 *     (0, g, t) and (1, g, t) of two 8-row halves.
 *
 * Every function follows the definition directly: per-bit loops, no word
 * tricks, no blocking.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>
#include <unistd.h>

/* ---- 1. bitstream ------------------------------------------------------- */

static int stream_bit(const uint8_t *row, long i)
{
    return (row[i >> 3] >> (i & 7)) & 1;
}

/* Code k of one column's bitstream: bit j of the code is stream bit k*b+j. */
int oracle_code(const uint8_t *row, long k, int bits)
{
    int q = 0;
    for (int j = 0; j < bits; ++j)
        q |= stream_bit(row, k * bits + j) << j;
    return q;
}

/* packed [N][K*bits/8] -> codes [N][K].  Requires K*bits % 8 == 0. */
void oracle_unpack(const uint8_t *packed, uint8_t *codes, long N, long K, int bits)
{
    long row_bytes = K * bits / 8;
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)oracle_code(packed + n * row_bytes, k, bits);
}

/* codes [N][K] -> packed [N][K*bits/8].  Only the low `bits` bits of each
 * code are stored; returns how many codes had bits set at or above `bits`. */
long oracle_pack(const uint8_t *codes, uint8_t *packed, long N, long K, int bits)
{
    long row_bytes = K * bits / 8;
    long bad = 0;
    memset(packed, 0, (size_t)(N * row_bytes));
    for (long n = 0; n < N; ++n) {
        uint8_t *row = packed + n * row_bytes;
        for (long k = 0; k < K; ++k) {
            int q = codes[n * K + k];
            if (q >> bits)
                ++bad;
            for (int j = 0; j < bits; ++j) {
                long i = k * bits + j;
                row[i >> 3] |= (uint8_t)(((q >> j) & 1) << (i & 7));
            }
        }
    }
    return bad;
}

/* ---- thread helper: split columns n over workers -------------------------- */

typedef void (*col_fn)(void *ctx, long n0, long n1);
typedef struct { col_fn fn; void *ctx; long n0, n1; } work_t;

static void *run_work(void *p)
{
    work_t *w = (work_t *)p;
    w->fn(w->ctx, w->n0, w->n1);
    return NULL;
}

static int resolve_threads(int nthreads, long N)
{
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > N) nthreads = (int)(N > 0 ? N : 1);
    if (nthreads > 256) nthreads = 256;
    return nthreads;
}

static void parallel_columns(col_fn fn, void *ctx, long N, int nthreads)
{
    int T = resolve_threads(nthreads, N);
    if (T <= 1) { fn(ctx, 0, N); return; }
    pthread_t th[256];
    work_t w[256];
    for (int t = 0; t < T; ++t) {
        w[t].fn = fn; w[t].ctx = ctx;
        w[t].n0 = N * t / T; w[t].n1 = N * (t + 1) / T;
        pthread_create(&th[t], NULL, run_work, &w[t]);
    }
    for (int t = 0; t < T; ++t) pthread_join(th[t], NULL);
}

int oracle_threads(int nthreads, long N) { return resolve_threads(nthreads, N); }

/* ---- 2 + 3. dequantize, then matmul in fp64 ----------------------------------- */

typedef struct {
    const double *x; const uint8_t *packed; int bits; int group;
    const double *scales; const uint8_t *zeros; int zero_const;
    double *y; long M, N, K;
} qmm_ctx;

static void qmm_cols(void *p, long n0, long n1)
{
    qmm_ctx *c = (qmm_ctx *)p;
    long K = c->K, ng = K / c->group, row_bytes = K * c->bits / 8;
    double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    for (long n = n0; n < n1; ++n) {
        const uint8_t *row = c->packed + n * row_bytes;
        for (long k = 0; k < K; ++k) {
            long g = k / c->group;
            long q = oracle_code(row, k, c->bits);
            long z = c->zeros ? c->zeros[n * ng + g] : c->zero_const;
            w[k] = (double)(q - z) * c->scales[n * ng + g];      /* Eq. (5) */
        }
        for (long m = 0; m < c->M; ++m) {
            double acc = 0.0;
            for (long k = 0; k < K; ++k)
                acc += c->x[m * K + k] * w[k];
            c->y[m * c->N + n] = acc;
        }
    }
    free(w);
}

/* y[M][N] = x[M][K] . W^T with W[n][k] = (q[n][k] - z[n][k/G]) * s[n][k/G].
 * x and scales are the stored fp16/bf16 values widened exactly to fp64;
 * zeros is [N][K/G] uint8 or NULL (then zero_const is used). */
void oracle_qmm(const double *x, const uint8_t *packed, int bits, int group,
                const double *scales, const uint8_t *zeros, int zero_const,
                double *y, long M, long N, long K, int nthreads)
{
    qmm_ctx c = { x, packed, bits, group, scales, zeros, zero_const, y, M, N, K };
    parallel_columns(qmm_cols, &c, N, nthreads);
}

/* ---- 4. W4A8 integer core and epilogue ---------------------------------------- */

/* Two's-complement value of a 4-bit code. */
int oracle_int4_value(int code)
{
    return (code & 8) ? (code & 15) - 16 : (code & 15);
}

/* Value of a b-bit two's-complement code: the top bit weighs -2^(b-1). */
int oracle_signed_value(int code, int bits)
{
    const int top = 1 << (bits - 1);
    code &= (1 << bits) - 1;
    return (code & top) ? code - 2 * top : code;
}

/* The dot-product primitive: r + sum_i a[i]*b[i] with int8 inputs and a wide
 * integer accumulator (dp4a is the n = 4 case). */
int64_t oracle_dot_i8(const int8_t *a, const int8_t *b, long n, int64_t r)
{
    for (long i = 0; i < n; ++i)
        r += (int64_t)a[i] * (int64_t)b[i];
    return r;
}

typedef struct {
    const int8_t *xq; const double *sa; const uint8_t *w4; const double *ws;
    int group; int64_t *acc; double *y; long M, N, K; int overflow; int bits;
} w4a8_ctx;

static void w4a8_cols(void *p, long n0, long n1)
{
    w4a8_ctx *c = (w4a8_ctx *)p;
    long K = c->K, ng = K / c->group, row_bytes = K * c->bits / 8;
    int8_t *w = (int8_t *)malloc((size_t)(K > 0 ? K : 1));
    for (long n = n0; n < n1; ++n) {
        const uint8_t *row = c->w4 + n * row_bytes;
        for (long k = 0; k < K; ++k)
            w[k] = (int8_t)oracle_signed_value(oracle_code(row, k, c->bits), c->bits);
        for (long m = 0; m < c->M; ++m) {
            double yy = 0.0;
            for (long g = 0; g < ng; ++g) {
                int64_t a = oracle_dot_i8(c->xq + m * K + g * c->group,
                                          w + g * c->group, c->group, 0);
                if (a > INT32_MAX || a < INT32_MIN) c->overflow = 1;
                if (c->acc) c->acc[(m * c->N + n) * ng + g] = a;
                yy += c->ws[n * ng + g] * (double)a;
            }
            c->y[m * c->N + n] = c->sa[m] * yy;
        }
    }
    free(w);
}

/* acc[m][n][g] = sum_{k in g} xq[m][k] * w4[n][k]   (int64, may be NULL)
 * y[m][n]      = sa[m] * sum_g ws[n][g] * acc[m][n][g]   (fp64)
 * Returns 1 if any accumulator falls outside the int32 range, else 0. */
int oracle_w4a8(const int8_t *xq, const double *sa, const uint8_t *w4,
                const double *ws, int group, int64_t *acc, double *y,
                long M, long N, long K, int nthreads)
{
    w4a8_ctx c = { xq, sa, w4, ws, group, acc, y, M, N, K, 0, 4 };
    parallel_columns(w4a8_cols, &c, N, nthreads);
    return c.overflow;
}

/* The same with signed b-bit weights (b = 8: W8A8, BitLLM's other integer
 * precision, Experiment Setup "Workloads": 8-bit weights and activations with
 * group-wise scaling): w[n][k] is the two's-complement value of code k of
 * column n's b-bit stream. */
int oracle_wxa8(const int8_t *xq, const double *sa, const uint8_t *w, int bits,
                const double *ws, int group, int64_t *acc, double *y,
                long M, long N, long K, int nthreads)
{
    w4a8_ctx c = { xq, sa, w, ws, group, acc, y, M, N, K, 0, bits };
    parallel_columns(w4a8_cols, &c, N, nthreads);
    return c.overflow;
}

/* ---- 5. per-token int8 activation quantization ------------------------- */

static float f16_bits_to_float(uint16_t h)
{
    _Float16 v;
    memcpy(&v, &h, sizeof(v));
    return (float)v;   /* exact */
}

static uint16_t float_to_f16_bits(float f)
{
    _Float16 v = (_Float16)f;   /* round to nearest even */
    uint16_t h;
    memcpy(&h, &v, sizeof(h));
    return h;
}

/* x: fp16 bit patterns [M][K]; writes xq int8 [M][K] and sa fp16 bits [M]. */
void oracle_quantize_act(const uint16_t *x, int8_t *xq, uint16_t *sa, long M, long K)
{
    for (long m = 0; m < M; ++m) {
        const uint16_t *row = x + m * K;
        float amax = 0.0f;
        for (long k = 0; k < K; ++k) {
            const float a = fabsf(f16_bits_to_float(row[k]));
            if (a > amax)
                amax = a;
        }
        sa[m] = float_to_f16_bits(amax / 127.0f);
        const float s = f16_bits_to_float(sa[m]);
        for (long k = 0; k < K; ++k) {
            float q = 0.0f;
            if (s > 0.0f) {
                q = rintf(f16_bits_to_float(row[k]) / s);   /* ties to even */
                if (q < -128.0f)
                    q = -128.0f;
                if (q > 127.0f)
                    q = 127.0f;
            }
            xq[m * K + k] = (int8_t)q;
        }
    }
}

/* ---- 6. signed weights: flip the top bit of every code ------------------ */

void oracle_flip_sign(uint8_t *packed, long N, long K, int bits)
{
    const long row_bytes = K * bits / 8;
    for (long n = 0; n < N; ++n) {
        uint8_t *row = packed + n * row_bytes;
        for (long k = 0; k < K; ++k) {
            const long i = k * bits + bits - 1;   /* the code's top stream bit */
            row[i >> 3] ^= (uint8_t)(1u << (i & 7));
        }
    }
}

/* ---- 7. float weights ---------------------------------------------------- */

double oracle_float_value(int code, int ebits, int mbits)
{
    const int b = 1 + ebits + mbits;
    const int sign = (code >> (b - 1)) & 1;
    const int E = (code >> mbits) & ((1 << ebits) - 1);
    const int M = code & ((1 << mbits) - 1);
    const int bias = (1 << (ebits - 1)) - 1;
    double v;
    if (E > 0)
        v = ldexp(1.0 + (double)M / (double)(1 << mbits), E - bias);
    else
        v = ldexp((double)M / (double)(1 << mbits), 1 - bias);
    return sign ? -v : v;
}

/* ---- 8. lane-interleaved int4 layout ------------------------------------ */

/* The nibble slot (0..7) of code r (0..7) within its 32-bit word. */
static int interleave4_slot(int r) { return r < 4 ? 2 * r : 2 * (r - 4) + 1; }

void oracle_interleave4(const uint8_t *codes, uint8_t *out, long N, long K)
{
    for (long n = 0; n < N; ++n) {
        const uint8_t *c = codes + n * K;
        uint8_t *row = out + n * (K / 2);
        memset(row, 0, (size_t)(K / 2));
        for (long k = 0; k < K; ++k) {
            const long slot = 8 * (k / 8) + interleave4_slot((int)(k % 8));
            row[slot / 2] |= (uint8_t)((c[k] & 15u) << (4 * (slot % 2)));
        }
    }
}

void oracle_deinterleave4(const uint8_t *in, uint8_t *codes, long N, long K)
{
    for (long n = 0; n < N; ++n) {
        const uint8_t *row = in + n * (K / 2);
        for (long k = 0; k < K; ++k) {
            const long slot = 8 * (k / 8) + interleave4_slot((int)(k % 8));
            codes[n * K + k] = (uint8_t)((row[slot / 2] >> (4 * (slot % 2))) & 15u);
        }
    }
}

/* ---- 9. fragment-ordered (tile16) layout ---------------------------------- */

/* Bit position, in the tile16 stream, of bit j of code k of row n. */
static long tile16_bit(long n, long k, int j, long K, int bits)
{
    const long T = n / 16, kb = k / 64;
    const long h = (n % 16) / 8, g = n % 8, t = (k % 64) / 16, c = k % 16;
    const long unit = T * (K / 64) + kb;
    const long run = (h * 8 + g) * 4 + t;
    return unit * 128L * bits * 8 + run * 16L * bits + c * bits + j;
}

/* Bytes of the tile16 stream of N rows: ceil(N/16) tiles of 16 rows. */
long oracle_tile16_bytes(long N, long K, int bits)
{
    return (N + 15) / 16 * 16 * K * bits / 8;
}

/* codes [N][K] (K % 64 == 0) -> tile16 stream; padding rows hold code 0. */
void oracle_tile16(const uint8_t *codes, uint8_t *out, long N, long K, int bits)
{
    memset(out, 0, (size_t)oracle_tile16_bytes(N, K, bits));
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k)
            for (int j = 0; j < bits; ++j)
                if ((codes[n * K + k] >> j) & 1u) {
                    const long i = tile16_bit(n, k, j, K, bits);
                    out[i / 8] |= (uint8_t)(1u << (i % 8));
                }
}

/* tile16 stream -> codes [N][K]. */
void oracle_untile16(const uint8_t *in, uint8_t *codes, long N, long K, int bits)
{
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k) {
            unsigned q = 0;
            for (int j = 0; j < bits; ++j) {
                const long i = tile16_bit(n, k, j, K, bits);
                q |= (unsigned)((in[i / 8] >> (i % 8)) & 1u) << j;
            }
            codes[n * K + k] = (uint8_t)q;
        }
}
