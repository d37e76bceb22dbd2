/*
 * CPU oracle for the fused GPTQ W4A16 linear layer  y = x . W + bias.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the timed CPU
 * baseline can say what the right answer is.  It shares no code, header,
 * table or constant with the CUDA library.
 *
 * What it computes, and where that comes from:
 *
 *  - "GPTQ's 'Exllama Kernel Not Installed' Warning", section "Why the kernel
 *    is missing": a GPTQ checkpoint holds 4-bit integers packed into 32-bit
 *    words, with a scale and a zero point per group.
 *  - The same page, "What the fallback actually does": the fused kernel and
 *    the fallback reach the same answer; the fallback rebuilds the full
 *    weight matrix and runs an ordinary matmul.  That plain route is what
 *    this oracle is: unpack, dequantize, then a dense product.
 *  - "Implementation: Predibase Lorax GPTQ Exllama V1", section "I/O
 *    Contract": qweight/qzeros int32, scales fp16 per group, g_idx optional
 *    (None or trivial indices mean no act-order), bits must be 4, output
 *    fp16.
 *  - "Inference Backends", section "Concepts": GPTQ and GPTQ_V2 are distinct
 *    checkpoint formats.  This oracle implements the GPTQ (v1) storage
 *    convention: qweight [K/8][N] holds eight codes per word along K with
 *    the lowest nibble first; qzeros [G][N/8] holds eight zero points per
 *    word along N, lowest nibble first; scales [G][N] fp16; the effective
 *    zero point is the stored value plus one, so
 *        w[k][n] = scales[g][n] * (q[k][n] - (z[g][n] + 1)),  g = g_idx[k].
 *    The same page names GPTQ_V2 as a distinct format; read here as the same
 *    layout with the effective zero point stored as is, so
 *        w[k][n] = scales[g][n] * (q[k][n] - z[g][n])
 *    (oracle_dequant takes the offset, 1 or 0, as its last argument).
 *  - "Inference Backends", section "Numeric epilogues and input gradients":
 *    bias joins the wide accumulator before the single final cast.  Here
 *    everything is fp64, bias is added after the k-sum.
 *
 * Precision: fp64 throughout.  The dequantized weight is formed exactly in
 * fp64 (an 11-bit significand times an integer in [-16, 15], or [-256, 255]
 * for 8-bit codes, fits easily)
 * and then rounded once, to nearest-even, to fp16: that fp16 matrix (w16)
 * is the value a GPU dequantizer must reproduce bit for bit, and y_ref is
 * the fp64 product of the fp16 activations with w16.
 *
 * fp16 <-> double conversion is written here from the IEEE-754 binary16
 * definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits,
 * subnormals with quantum 2^-24) so that the oracle does not borrow a
 * converter from the code it checks.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- fp16 */

double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* zero or subnormal */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a non-negative double that is already scaled so that one unit is
 * one fp16 quantum: nearest integer, ties to the even one. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double d = q - fl;                             /* exact: q has few bits */
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t oracle_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs(v);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: quantum 2^-24; a count of 1024 lands exactly on
         * the smallest normal number, whose encoding is also 1024. */
        double r = round_half_even(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)r);
    }
    int e;
    frexp(a, &e);                                  /* a in [2^(e-1), 2^e) */
    double r = round_half_even(ldexp(a, 11 - e));  /* in [1024, 2048] */
    int E = e - 1 + 15;
    if (r == 2048.0) { r = 1024.0; E += 1; }
    if (E >= 31) return (uint16_t)(sign | 0x7c00u);   /* overflow -> inf */
    return (uint16_t)(sign | (uint16_t)(E << 10) | (uint16_t)((int)r - 1024));
}

void oracle_half_to_double_array(const uint16_t *h, size_t n, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = oracle_half_to_double(h[i]);
}

void oracle_double_to_half_array(const double *v, size_t n, uint16_t *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = oracle_double_to_half(v[i]);
}

/* bf16 activations ("Inference Backends": backends keep the activation and
 * output dtype, fp16 or bf16): a bf16 value is the upper 16 bits of an IEEE
 * binary32, so it converts to double exactly. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void oracle_bf16_to_double_array(const uint16_t *b, size_t n, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(b[i]);
}

/* fp32 activations ("Inference Backends", "Hardware, dependency, and format
 * requirements": the ExLlama v2 row declares FP16/BF16/FP32 activation
 * dtypes).  An IEEE binary32 bit pattern to its exact double, from the
 * format's definition: sign, 8-bit exponent with bias 127, 23-bit fraction;
 * exponent 0 is zero or subnormal (f 2^-149), 255 is infinity or NaN. */
double oracle_f32_to_double(uint32_t u)
{
    int sign = (int)(u >> 31);
    int e = (int)((u >> 23) & 0xffu);
    uint32_t f = u & 0x7fffffu;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -149);                /* zero or subnormal */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(0x800000u + f), e - 150);   /* (1 + f/2^23) 2^(e-127) */
    }
    return sign ? -v : v;
}

void oracle_f32_to_double_array(const uint32_t *u, size_t n, double *out)
{
    for (size_t i = 0; i < n; ++i) out[i] = oracle_f32_to_double(u[i]);
}

/* ------------------------------------------------------------- unpack */

/* q[k][n] = nibble (k mod 8) of qweight[k/8][n], lowest nibble first.
 * The word is read as unsigned so that the top nibble of a negative int32
 * comes out as 8..15. */
void oracle_unpack_qweight(const int32_t *qweight, int K, int N, uint8_t *q)
{
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            uint32_t word = (uint32_t)qweight[(size_t)(k / 8) * N + n];
            q[(size_t)k * N + n] = (uint8_t)((word >> (4 * (k % 8))) & 0xFu);
        }
}

/* z[i][n] = nibble (n mod 8) of qzeros[i][n/8], lowest nibble first. */
void oracle_unpack_qzeros(const int32_t *qzeros, int G, int N, uint8_t *z)
{
    for (int i = 0; i < G; ++i)
        for (int n = 0; n < N; ++n) {
            uint32_t word = (uint32_t)qzeros[(size_t)i * (N / 8) + n / 8];
            z[(size_t)i * N + n] = (uint8_t)((word >> (4 * (n % 8))) & 0xFu);
        }
}

/* 8-bit checkpoints.  "Inference Backends" declares GPTQ with 4 and 8 bits
 * (GPTQ Marlin, Swordfish) without printing the 8-bit layout; read here as the
 * same GPTQ packing with 32 / 8 = 4 codes per int32: qweight [K/4][N] holds
 * four codes per word along K, lowest byte first, and qzeros [G][N/4] four
 * zero points per word along N, lowest byte first.  oracle_dequant then
 * applies unchanged (q and z up to 255). */
void oracle_unpack_qweight8(const int32_t *qweight, int K, int N, uint8_t *q)
{
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            uint32_t word = (uint32_t)qweight[(size_t)(k / 4) * N + n];
            q[(size_t)k * N + n] = (uint8_t)((word >> (8 * (k % 4))) & 0xFFu);
        }
}

void oracle_unpack_qzeros8(const int32_t *qzeros, int G, int N, uint8_t *z)
{
    for (int i = 0; i < G; ++i)
        for (int n = 0; n < N; ++n) {
            uint32_t word = (uint32_t)qzeros[(size_t)i * (N / 4) + n / 4];
            z[(size_t)i * N + n] = (uint8_t)((word >> (8 * (n % 4))) & 0xFFu);
        }
}

/* Group of each row.  groupsize -1 means one group over all of K.
 * Without g_idx the group of row k is k / groupsize ("None or trivial
 * indices indicate no act-order", Lorax page, I/O Contract).
 * Returns G, or -1 when the arguments are invalid or an index is out of
 * [0, G). */
int oracle_row_groups(const int32_t *g_idx, int K, int groupsize, int32_t *gr)
{
    if (K <= 0) return -1;
    if (groupsize != -1 && (groupsize <= 0 || K % groupsize != 0)) return -1;
    int geff = (groupsize == -1) ? K : groupsize;
    int G = K / geff;
    for (int k = 0; k < K; ++k) {
        int g = g_idx ? g_idx[k] : k / geff;
        if (g < 0 || g >= G) return -1;
        gr[k] = g;
    }
    return G;
}

/* w64[k][n] = s * (q - (z + zero_offset)) exactly (zero_offset 1: GPTQ,
 * 0: GPTQ_V2); w16 = that value rounded once to fp16, nearest-even.  w64 may
 * be NULL. */
void oracle_dequant(const uint8_t *q, const uint8_t *z, const uint16_t *scales,
                    const int32_t *gr, int K, int N, uint16_t *w16, double *w64, int zero_offset)
{
    for (int k = 0; k < K; ++k) {
        int g = gr[k];
        for (int n = 0; n < N; ++n) {
            double s = oracle_half_to_double(scales[(size_t)g * N + n]);
            int iq = (int)q[(size_t)k * N + n] - ((int)z[(size_t)g * N + n] + zero_offset);
            double v = s * (double)iq;
            if (w64) w64[(size_t)k * N + n] = v;
            w16[(size_t)k * N + n] = oracle_double_to_half(v);
        }
    }
}

/* ------------------------------------------------------------- packing */

/* Pack float weights into a GPTQ checkpoint ("Inference Backends",
 * "Packing, conversion, and runtime initialization": packing takes the
 * original linear layer's weights with the quantizer's scales, zeros and
 * optional activation-order index; symmetric modules without zeros use
 * 2^(bits-1)).  Reading: the code of w is the nearest integer to w / s
 * (quotient of the fp16 values in IEEE binary32, ties to even) plus the
 * effective zero point, clamped to [0, 15]:
 *     q[k][n] = clamp(rint((float)w[k][n] / (float)s[g][n]) + z[g][n], 0, 15)
 * with g = g_idx[k] (or k / groupsize).  qweight [K/8][N] holds q along K,
 * lowest nibble first; qzeros [G][N/8] holds the stored zero along N,
 * lowest nibble first: z - 1 for GPTQ (zero_offset 1; taken mod 16, so an
 * effective zero of 0 is stored as 15), z for GPTQ_V2 (zero_offset 0).
 * zeros may be NULL: every effective zero is then 8.
 * Returns G, or -1 for an invalid groupsize / g_idx. */
int oracle_pack(const uint16_t *w, const uint16_t *scales, const int32_t *zeros, const int32_t *g_idx,
                int K, int N, int groupsize, int zero_offset, int32_t *qweight, int32_t *qzeros)
{
    int32_t *gr = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
    if (!gr) return -1;
    int G = oracle_row_groups(g_idx, K, groupsize, gr);
    if (G < 0) { free(gr); return -1; }
    memset(qweight, 0, sizeof(int32_t) * (size_t)(K / 8) * N);
    for (int k = 0; k < K; ++k) {
        int g = gr[k];
        for (int n = 0; n < N; ++n) {
            float wf = (float)oracle_half_to_double(w[(size_t)k * N + n]);
            float sf = (float)oracle_half_to_double(scales[(size_t)g * N + n]);
            float qf = rintf(wf / sf);
            int z = zeros ? zeros[(size_t)g * N + n] : 8;
            /* clamp in float (an infinite quotient clamps too); 0/0 gives the zero point */
            float v = (qf != qf) ? (float)z : qf + (float)z;
            if (v < 0.0f) v = 0.0f;
            if (v > 15.0f) v = 15.0f;
            long q = (long)v;
            uint32_t *word = (uint32_t *)&qweight[(size_t)(k / 8) * N + n];
            *word |= (uint32_t)q << (4 * (k % 8));
        }
    }
    memset(qzeros, 0, sizeof(int32_t) * (size_t)G * (N / 8));
    for (int g = 0; g < G; ++g)
        for (int n = 0; n < N; ++n) {
            int z = zeros ? zeros[(size_t)g * N + n] : 8;
            uint32_t stored = (uint32_t)(z - zero_offset) & 0xFu;
            uint32_t *word = (uint32_t *)&qzeros[(size_t)g * (N / 8) + n / 8];
            *word |= stored << (4 * (n % 8));
        }
    free(gr);
    return G;
}

/* ------------------------------------------------------------- linear */

struct linear_job {
    const double *x, *w, *bias;
    double *y;
    int M, K, N, n0, n1;
};

/* y[m][n] = (sum over k = 0, 1, ..., K-1 of x[m][k] * w[k][n]) + bias[n],
 * each sum taken in ascending k.  A worker owns the columns [n0, n1). */
static void *linear_worker(void *arg)
{
    const struct linear_job *j = (const struct linear_job *)arg;
    for (int m = 0; m < j->M; ++m) {
        double *yrow = j->y + (size_t)m * j->N;
        for (int n = j->n0; n < j->n1; ++n) yrow[n] = 0.0;
        for (int k = 0; k < j->K; ++k) {
            double xv = j->x[(size_t)m * j->K + k];
            const double *wrow = j->w + (size_t)k * j->N;
            for (int n = j->n0; n < j->n1; ++n) yrow[n] += xv * wrow[n];
        }
        if (j->bias)
            for (int n = j->n0; n < j->n1; ++n) yrow[n] += j->bias[n];
    }
    return NULL;
}

/* Dense fp64 product on nthreads host threads split by output columns.
 * Returns the number of threads used. */
int oracle_linear_f64(const double *x, const double *w, const double *bias,
                      int M, int K, int N, double *y, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = N > 0 ? N : 1;
    if (nthreads > 256) nthreads = 256;
    struct linear_job jobs[256];
    pthread_t tid[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].x = x; jobs[t].w = w; jobs[t].bias = bias; jobs[t].y = y;
        jobs[t].M = M; jobs[t].K = K; jobs[t].N = N;
        jobs[t].n0 = (int)((long long)N * t / nthreads);
        jobs[t].n1 = (int)((long long)N * (t + 1) / nthreads);
        started[t] = (t > 0) && pthread_create(&tid[t], NULL, linear_worker, &jobs[t]) == 0;
        if (t > 0 && !started[t]) linear_worker(&jobs[t]);
    }
    linear_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (started[t]) pthread_join(tid[t], NULL);
    return nthreads;
}
