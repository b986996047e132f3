/*
 * qbw_oracle.c -- the plain, slow CPU oracle for block-quantized weight
 * matrix-vector products (GGUF Q8_0 / Q4_0).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA path: it has its own fp16/bf16 decoders, its own nibble unpacking
 * and its own GELU.
 *
 * Everything is scalar C, accumulated in double precision in ascending k, with
 * no SIMD intrinsics and no reordering beyond the textbook definition.  Built
 * with OpenMP (for the all-core CPU baseline only), the independent rows of a
 * product are split over threads; each row's arithmetic is unchanged.
 *
 * What is computed, and where the pages define it:
 *  - Q8_0 block: w = d * q, d an IEEE binary16 scale, q a signed byte
 *    (jouleclaw-loader-gguf BENCHMARKS, "Matmul throughput -- Q8_0 scalar vs
 *    NEON"; gem architecture, "M4 Max operating assumptions").
 *  - Q4_0 block: w = d * (q - 8), q a 4-bit code, 32 codes + scale in
 *    18 bytes (gem architecture, "M4 Max operating assumptions").  Nibble
 *    order follows the GGUF block_q4_0 record: code j in the low nibble of
 *    byte j, code j+16 in the high nibble.
 *  - Q4_K super-block: 256 weights in 144 bytes, w = d_sub * q - m_sub with
 *    d_sub = d * sc_j and m_sub = dmin * m_j for sub-block j (32 weights),
 *    q a 4-bit code (jouleclaw-loader-gguf BENCHMARKS, "Q4_K matmul --
 *    scalar fused vs AMX-tiled" and its NEON follow-up, which computes
 *    sum(a * (d_sub * q - m_sub)) = d_sub * sum(a * q) - m_sub * sum(a)).
 *    The byte layout follows the GGUF block_q4_K record: fp16 d, fp16 dmin,
 *    12 bytes of 6-bit (sc, m) pairs, 128 bytes of nibbles; each 64-weight
 *    chunk i keeps its first 32 codes in the low nibbles of bytes
 *    32i .. 32i + 31 and its last 32 in their high nibbles.
 *  - Matrix-vector product y = W x with W stored [out, in] row-major
 *    (SafeC Gemma 4 design notes, "Math primitives implementation status").
 *  - Gated FFN projection out = gelu_tanh(Wg x) * (Wu x) with the tanh form
 *    of GELU (SafeC Gemma 4 design notes, "Gated FFN").
 *  - Small-M product Y = X W^T for a few token rows (gem architecture,
 *    "Ownership boundaries": prompt tiles up to 32 tokens).
 *  - Mixed-bit matrices (int2-symmetric, int4-affine, int8) of a QAT
 *    checkpoint's hand-written decode loop (Core AI model zoo, Gemma-4-E2B
 *    raw-Metal port, "What shipped"); their layout is described above
 *    mixbit_field.
 *
 * Error scale: next to every output the oracle also returns
 * S = sum_k |w_k * x_k| (fp64), the scale the parity tolerances use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_QK 32
#define ORACLE_QK_K 256
#define ORACLE_PI 3.14159265358979323846

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_fp16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);              /* subnormal: m * 2^-133 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + m), e - 134);   /* (1 + m/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a double to the nearest bfloat16 (ties to even), return its bits. */
uint16_t oracle_round_bf16(double v)
{
    if (isnan(v))
        return 0x7fc0;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    uint16_t s = (uint16_t)(neg << 15);
    if (a == 0.0)
        return s;
    if (isinf(a))
        return (uint16_t)(s | 0x7f80);
    int ex;
    frexp(a, &ex);                     /* a in [2^(ex-1), 2^ex) */
    int q = ex - 8;                    /* quantum of 8 significant bits */
    if (q < -133)
        q = -133;                      /* subnormal quantum */
    double r = ldexp(a, -q);           /* exact: power-of-two scaling */
    double fl = floor(r);
    double frac = r - fl;
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))
        fl += 1.0;
    double res = ldexp(fl, q);
    /* largest finite bf16 is (2 - 2^-7) * 2^127 */
    if (res > ldexp(255.0, 120))
        return (uint16_t)(s | 0x7f80);
    if (res == 0.0)
        return s;
    /* encode: res = M * 2^E with M in [128, 256) for normals */
    int er;
    frexp(res, &er);                   /* res in [2^(er-1), 2^er) */
    int E = er - 1;                    /* unbiased exponent */
    if (E < -126) {                    /* subnormal: res = m * 2^-133 */
        int m = (int)ldexp(res, 133);
        return (uint16_t)(s | (uint16_t)m);
    }
    int m = (int)ldexp(res, 7 - E) - 128;
    return (uint16_t)(s | (uint16_t)((E + 127) << 7) | (uint16_t)m);
}

void oracle_round_bf16_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_round_bf16(v[i]);
}

void oracle_fp16_to_f64_array(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_fp16_to_f64(h[i]);
}

void oracle_bf16_to_f64_array(const uint16_t *b, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_bf16_to_f64(b[i]);
}

/* Activation dtype codes: 0 = fp32 values, 1 = bf16 bit patterns. */
static double *widen_activations(const void *x, int xdtype, int64_t n)
{
    double *out = (double *)malloc((size_t)n * sizeof(double));
    if (!out)
        return NULL;
    for (int64_t i = 0; i < n; i++) {
        if (xdtype == 0)
            out[i] = (double)((const float *)x)[i];
        else
            out[i] = oracle_bf16_to_f64(((const uint16_t *)x)[i]);
    }
    return out;
}

/* ------------------------------------------------------------ block decode */

static uint16_t read_u16le(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

/* fmt: 0 = Q8_0, 1 = Q4_0, 2 = Q4_K */
static int block_size(int fmt) { return fmt == 0 ? 34 : (fmt == 1 ? 18 : 144); }
static int block_elems(int fmt) { return fmt == 2 ? ORACLE_QK_K : ORACLE_QK; }

/* The 6-bit scale sc and min m of sub-block j (0..7) of a Q4_K super-block,
 * from its 12 scale bytes s[]: sub-blocks 0..3 keep sc and m in the low six
 * bits of s[j] and s[j + 4]; sub-blocks 4..7 keep the low four bits of sc and
 * of m in the low and high nibble of s[j + 4], and their top two bits in the
 * top two bits of s[j - 4] (sc) and s[j] (m). */
void oracle_q4k_scale_min(const uint8_t *s, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 0x0f) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* The code (0..15) of weight e (0..255) of a Q4_K super-block's 128 nibble
 * bytes: chunk e / 64, low nibble for its first 32 weights, high for the rest. */
static int q4k_code(const uint8_t *qs, int e)
{
    int chunk = e / 64, l = e % 64;
    uint8_t byte = qs[32 * chunk + (l % 32)];
    return (l < 32) ? (byte & 0x0f) : (byte >> 4);
}

/* Decode the weights of one block into w[0 .. block_elems(fmt) - 1]. */
static void decode_block(int fmt, const uint8_t *blk, double *w)
{
    if (fmt == 2) {
        double d = oracle_fp16_to_f64(read_u16le(blk));
        double dmin = oracle_fp16_to_f64(read_u16le(blk + 2));
        for (int e = 0; e < ORACLE_QK_K; e++) {
            int sc, m;
            oracle_q4k_scale_min(blk + 4, e / 32, &sc, &m);
            w[e] = d * (double)sc * (double)q4k_code(blk + 16, e) - dmin * (double)m;
        }
        return;
    }
    double d = oracle_fp16_to_f64(read_u16le(blk));
    for (int k = 0; k < ORACLE_QK; k++) {
        if (fmt == 0) {
            w[k] = d * (double)(int)(int8_t)blk[2 + k];
        } else {
            uint8_t byte = blk[2 + (k % 16)];
            int code = (k < 16) ? (byte & 0x0f) : (byte >> 4);
            w[k] = d * (double)(code - 8);
        }
    }
}

/* Dequantize a whole matrix to fp32.  Q8_0 / Q4_0: every d*q fits in 24 bits
 * of significand (11-bit scale times a code of at most 8 bits), so the double
 * product converts to float exactly.  Q4_K: d*sc*q and dmin*m are exact in
 * double, and their difference is rounded to float once (nearest even). */
int oracle_dequant(int fmt, const uint8_t *w, int64_t N, int64_t K, float *out)
{
    int be = block_elems(fmt);
    if (K % be)
        return -1;
    int64_t nb = K / be;
    double wb[ORACLE_QK_K];
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++) {
            decode_block(fmt, w + (n * nb + b) * block_size(fmt), wb);
            for (int k = 0; k < be; k++)
                out[n * K + b * be + k] = (float)wb[k];
        }
    return 0;
}

/* ------------------------------------------------------------- products */

/* y[n] = sum_k w[n,k] * x[k], S[n] = sum_k |w[n,k] * x[k]|, k ascending. */
static void matvec_rows(int fmt, const uint8_t *w, const double *x,
                        int64_t n0, int64_t n1, int64_t K, double *y, double *S)
{
    int be = block_elems(fmt);
    int64_t nb = K / be;
    /* rows are independent: the OpenMP build of this file (the all-core CPU
     * baseline) splits them over threads, each row computed as above */
#pragma omp parallel for schedule(static)
    for (int64_t n = n0; n < n1; n++) {
        double wb[ORACLE_QK_K];
        double acc = 0.0, sabs = 0.0;
        for (int64_t b = 0; b < nb; b++) {
            decode_block(fmt, w + (n * nb + b) * block_size(fmt), wb);
            for (int k = 0; k < be; k++) {
                double p = wb[k] * x[b * be + k];
                acc += p;
                sabs += fabs(p);
            }
        }
        y[n - n0] = acc;
        if (S)
            S[n - n0] = sabs;
    }
}

int oracle_qmv(int fmt, const uint8_t *w, const void *x, int xdtype,
               int64_t N, int64_t K, double *y, double *S)
{
    if (K % block_elems(fmt))
        return -1;
    double *xd = widen_activations(x, xdtype, K);
    if (!xd)
        return -2;
    matvec_rows(fmt, w, xd, 0, N, K, y, S);
    free(xd);
    return 0;
}

/* Same product for a subset of rows [n0, n1): used to time and to sample. */
int oracle_qmv_rows(int fmt, const uint8_t *w, const void *x, int xdtype,
                    int64_t n0, int64_t n1, int64_t K, double *y, double *S)
{
    if (K % block_elems(fmt))
        return -1;
    double *xd = widen_activations(x, xdtype, K);
    if (!xd)
        return -2;
    matvec_rows(fmt, w, xd, n0, n1, K, y, S);
    free(xd);
    return 0;
}

/* gelu_tanh(v) = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) */
double oracle_gelu_tanh(double v)
{
    const double c = sqrt(2.0 / ORACLE_PI);
    return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));
}

/* d/dv gelu_tanh(v); used only to scale the gate+up tolerance. */
double oracle_gelu_tanh_deriv(double v)
{
    const double c = sqrt(2.0 / ORACLE_PI);
    double z = c * (v + 0.044715 * v * v * v);
    double t = tanh(z);
    return 0.5 * (1.0 + t) + 0.5 * v * (1.0 - t * t) * c * (1.0 + 3.0 * 0.044715 * v * v);
}

void oracle_gelu_tanh_array(const double *v, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_gelu_tanh(v[i]);
}

void oracle_gelu_tanh_deriv_array(const double *v, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = oracle_gelu_tanh_deriv(v[i]);
}

/* g = Wg x, u = Wu x, out = gelu_tanh(g) * u (both matrices Q4_0). */
int oracle_gateup_q4_0(const uint8_t *wg, const uint8_t *wu, const void *x, int xdtype,
                       int64_t N, int64_t K, double *g, double *u, double *out,
                       double *Sg, double *Su)
{
    if (K % ORACLE_QK)
        return -1;
    double *xd = widen_activations(x, xdtype, K);
    if (!xd)
        return -2;
    matvec_rows(1, wg, xd, 0, N, K, g, Sg);
    matvec_rows(1, wu, xd, 0, N, K, u, Su);
    for (int64_t n = 0; n < N; n++)
        out[n] = oracle_gelu_tanh(g[n]) * u[n];
    free(xd);
    return 0;
}

/* Y[m, n] = sum_k X[m, k] * W[n, k] for m < M (W is Q4_0, X row-major). */
int oracle_qmm_q4_0(const uint8_t *w, const void *X, int xdtype,
                    int64_t M, int64_t N, int64_t K, double *Y, double *S)
{
    if (K % ORACLE_QK)
        return -1;
    double *xd = widen_activations(X, xdtype, M * K);
    if (!xd)
        return -2;
    for (int64_t m = 0; m < M; m++)
        matvec_rows(1, w, xd + m * K, 0, N, K, Y + m * N, S + m * N);
    free(xd);
    return 0;
}

/* The error scale of the algebraic split the Q4_K kernels compute,
 * d_sub * sum(q x) - m_sub * sum(x) per sub-block: S2[n] = sum over
 * sub-blocks j and their weights k of (|d_sub q_k| + |m_sub|) |x_k|.  Its two
 * sums are formed separately, so their rounding scales with this, not with
 * sum |w x| (which is 0 where d_sub q_k = m_sub exactly). */
int oracle_q4k_split_scale(const uint8_t *w, const void *x, int xdtype,
                           int64_t N, int64_t K, double *S2)
{
    if (K % ORACLE_QK_K)
        return -1;
    double *xd = widen_activations(x, xdtype, K);
    if (!xd)
        return -2;
    int64_t nb = K / ORACLE_QK_K;
    for (int64_t n = 0; n < N; n++) {
        double s2 = 0.0;
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = w + (n * nb + b) * 144;
            double d = oracle_fp16_to_f64(read_u16le(blk));
            double dmin = oracle_fp16_to_f64(read_u16le(blk + 2));
            for (int e = 0; e < ORACLE_QK_K; e++) {
                int sc, m;
                oracle_q4k_scale_min(blk + 4, e / 32, &sc, &m);
                double t = fabs(d * (double)sc * (double)q4k_code(blk + 16, e)) + fabs(dmin * (double)m);
                s2 += t * fabs(xd[b * ORACLE_QK_K + e]);
            }
        }
        S2[n] = s2;
    }
    free(xd);
    return 0;
}

/* ------------------------------------------------------- mixed-bit formats */

/* The mixed-bit matrices of a QAT checkpoint driven by hand-written
 * matrix-vector kernels (Core AI model zoo, Gemma-4-E2B raw-Metal port, "What
 * shipped" and "Architecture": int2-symmetric, int4-affine and int8 matvecs
 * over quantized words qp, scales sc and biases bi).  The page gives no byte
 * layout; this oracle reads the one the library documents:
 *  - qp: 32-bit little-endian words, row after row; weight k of a row holds
 *    bits [(k * b) % 32, (k * b) % 32 + b) of word (k * b) / 32 of that row
 *    (b = 2, 4 or 8 bits, lowest bits first);
 *  - sc, bi: IEEE binary16, one per group of G consecutive weights of a row,
 *    [N][K / G] row-major;
 *  - b = 2: q = the two's-complement value of the field (-2 .. 1), w = sc * q;
 *    b = 4: c = the unsigned field (0 .. 15), w = sc * c + bi;
 *    b = 8: q = the two's-complement byte (-128 .. 127), w = sc * q. */
static int mixbit_field(const uint32_t *row, int bits, int64_t k)
{
    int64_t bit = k * bits;
    uint32_t word = row[bit / 32];
    int v = (int)((word >> (bit % 32)) & ((1u << bits) - 1u));
    if (bits != 4 && v >= (1 << (bits - 1)))
        v -= 1 << bits;                        /* two's complement */
    return v;
}

/* The exact weight of row n, input k (fp64). */
static double mixbit_weight(int bits, const uint32_t *qp, const uint16_t *sc, const uint16_t *bi,
                            int64_t group, int64_t K, int64_t n, int64_t k)
{
    const uint32_t *row = qp + n * (K * bits / 32);
    int64_t g = n * (K / group) + k / group;
    double s = oracle_fp16_to_f64(sc[g]);
    double v = s * (double)mixbit_field(row, bits, k);
    if (bits == 4)
        v += oracle_fp16_to_f64(bi[g]);
    return v;
}

static int mixbit_shape_ok(int bits, int64_t group, int64_t K)
{
    if (bits != 2 && bits != 4 && bits != 8)
        return 0;
    if (K <= 0 || group <= 0 || K % group || (K * bits) % 32)
        return 0;
    return 1;
}

/* Dequantize to fp32: the exact weight (fp64) rounded to float once. */
int oracle_mixbit_dequant(int bits, const uint32_t *qp, const uint16_t *sc, const uint16_t *bi,
                          int64_t group, int64_t N, int64_t K, float *out)
{
    if (!mixbit_shape_ok(bits, group, K))
        return -1;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++)
            out[n * K + k] = (float)mixbit_weight(bits, qp, sc, bi, group, K, n, k);
    return 0;
}

/* y[n] = sum_k w[n,k] x[k] in fp64, k ascending; S[n] = sum_k |w x|; and
 * S2[n] = sum_k (|sc q| + |bi|) |x|, the scale of the affine split
 * sc * sum(c x) + bi * sum(x), whose two sums are formed apart (S2 = S for
 * the symmetric formats, which have no bias). */
int oracle_qmv_mixbit(int bits, const uint32_t *qp, const uint16_t *sc, const uint16_t *bi,
                      int64_t group, const void *x, int xdtype, int64_t N, int64_t K,
                      double *y, double *S, double *S2)
{
    if (!mixbit_shape_ok(bits, group, K))
        return -1;
    double *xd = widen_activations(x, xdtype, K);
    if (!xd)
        return -2;
    for (int64_t n = 0; n < N; n++) {
        double acc = 0.0, sabs = 0.0, s2 = 0.0;
        const uint32_t *row = qp + n * (K * bits / 32);
        for (int64_t k = 0; k < K; k++) {
            double w = mixbit_weight(bits, qp, sc, bi, group, K, n, k);
            double p = w * xd[k];
            acc += p;
            sabs += fabs(p);
            int64_t g = n * (K / group) + k / group;
            double t = fabs(oracle_fp16_to_f64(sc[g]) * (double)mixbit_field(row, bits, k));
            if (bits == 4)
                t += fabs(oracle_fp16_to_f64(bi[g]));
            s2 += t * fabs(xd[k]);
        }
        y[n] = acc;
        if (S)
            S[n] = sabs;
        if (S2)
            S2[n] = s2;
    }
    free(xd);
    return 0;
}
