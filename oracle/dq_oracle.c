/*
 * dq_oracle.c -- plain, slow, obviously-correct CPU oracle for the decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library, its Python
 * binding) may include, link, load or call this file.  Only the tests, the smoke
 * check and the bench's CPU-baseline leg use it.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * Arithmetic: every sum is accumulated in IEEE double, in the natural index order,
 * with no blocking, fusion or reordering.  Outputs are double unless a storage
 * format fixes otherwise (the fp16 KV cache).  An outer "omp parallel for" over
 * independent output rows is the only parallelism; it never changes a result.
 *
 * What each function follows (pages: "one-serial-kernel" = vocodex.ai,
 * "The Mountain Runs" = coderlegion S-MoE diary #5, "The roofline holds on a
 * second GPU" = research.arkey.ai):
 *   - RMSNorm / LayerNorm: "one-serial-kernel", section "One thread" (the norm
 *     run twice per layer and once at the end; layer norm reduced in two passes).
 *     The formulas themselves are not printed on the pages; the standard ones are
 *     used: RMSNorm y = x * (mean(x^2) + eps)^-1/2 * gamma, LayerNorm with the
 *     population variance, eps inside the root.
 *   - Q4_K / Q6_K super-blocks: "The roofline holds on a second GPU", section
 *     "The Math" (4.5 and 6.5625 bits per weight, 256 weights per 144 / 210 bytes;
 *     "The search space": Q4_K packs 256 weights into 144 bytes, Q6_K into 210).
 *     The pages do not give a bit layout, so this library defines one with the
 *     same field sizes (see the FORMAT comment below).
 *   - GEMV: "The Mountain Runs", section 3 (one output per weight row, the same
 *     product whatever the thread layout); fp32-or-better accumulation per
 *     "The roofline holds on a second GPU", section "Hiding, fusing..." (Dtypes).
 *   - Decode block: the Qwen3-8B tensor census of "The Math" (attention
 *     4096x4096 + K,V 1024x4096, gate/up 12288x4096, down 4096x12288, vocabulary
 *     151936x4096), pre-norm residual block, SwiGLU, grouped-query attention over
 *     an fp16 KV cache ("Said before the run": 512 tokens add 75.5 MB).
 *
 * FORMAT (this library's canonical little-endian layouts)
 *
 *   Q4_K super-block, 144 bytes, 256 weights n = 32*j + i (sub-block j = 0..7):
 *     [0,2)    d     IEEE binary16
 *     [2,4)    dmin  IEEE binary16
 *     [4,16)   a 96-bit little-endian bit string (bit b is bit b%8 of byte 4+b/8):
 *              bits [6j, 6j+6)      = sc_j, unsigned 6-bit sub-block scale
 *              bits [48+6j, 54+6j)  = m_j,  unsigned 6-bit sub-block min
 *     [16,144) codes: byte 16 + 16*j + i (i = 0..15) holds the 4-bit code of
 *              weight 32j+i in its low nibble and of weight 32j+16+i in its high nibble
 *     weight n = d * sc_j * q_n - dmin * m_j
 *
 *   Q6_K super-block, 210 bytes, 256 weights n = 32*g + r (group g = 0..7):
 *     [0,128)   ql: byte 16*g + i (i = 0..15) holds the low 4 bits of weight 32g+i
 *               in its low nibble and of weight 32g+16+i in its high nibble
 *     [128,192) qh: the high 2 bits of weight 32g + 16h + 4t + e (h in {0,1},
 *               t, e in 0..3) are bits 2t, 2t+1 of byte 128 + 8g + 4h + e
 *     [192,208) sc[16]: int8, sc[s] scales weights 16s .. 16s+15
 *     [208,210) d: IEEE binary16
 *     q_n = low4 | high2 << 4 (0..63); weight n = d * sc[n/16] * (q_n - 32)
 *
 *   Q2_K super-block, 84 bytes, 256 weights n = 16*j + i (sub-block j = 0..15):
 *     [0,2)    d     IEEE binary16
 *     [2,4)    dmin  IEEE binary16
 *     [4,20)   byte 4 + j: sc_j in its low nibble, m_j in its high nibble (unsigned 4-bit)
 *     [20,84)  codes: byte 20 + 4*j + b (b = 0..3) holds the 2-bit codes of
 *              weights 16j + 4k + b (k = 0..3) at bits [2k, 2k+2)
 *     weight n = d * sc_j * q_n - dmin * m_j
 *   (The pages name 2-bit codes as the next bytes-halving step -- "The Mountain
 *   Runs", its closing section: expert kernels that dequantise 2/4-bit codes in
 *   registers -- without a layout; this one is Q4_K's scale/min scheme with
 *   2-bit codes and 4-bit scales over 16-weight sub-blocks: 2.625 bits/weight.)
 *
 *   bf16 matrix: row-major, K contiguous, bfloat16 = top 16 bits of an fp32.
 *   fp16 KV cache: [layer][2 (k, v)][kv_head][max_ctx][head_dim] binary16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))

/* ---------------------------------------------------------------- scalars -- */

/* IEEE 754 binary16 -> double, from the definition:
 * exponent field 0 -> subnormal m * 2^-24; 31 -> inf/nan; else (1024 + m) * 2^(e-25). */
ORACLE_API double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* double -> binary16, round to nearest, ties to even (the rounding the fp16 KV
 * cache store uses).  Works on the exact value: a / quantum is exact because the
 * quantum is a power of two. */
ORACLE_API uint16_t oracle_double_to_half(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (isnan(v))
        return 0x7e00;
    double a = fabs(v);
    if (a >= 65520.0) /* halfway between 65504 and 2^16 rounds to even = inf */
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);      /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;     /* floor(log2 a) */
    if (E < -14)
        E = -14;        /* subnormal range shares the 2^-24 quantum */
    double n = nearbyint(ldexp(a, 10 - E)); /* default rounding mode: ties to even */
    /* n in [0, 2048]; value = n * 2^(E-10) */
    if (n >= 2048.0) {  /* carried into the next binade */
        n /= 2.0;
        E += 1;
    }
    if (n < 1024.0)     /* subnormal (only possible when E == -14) */
        return sign | (uint16_t)n;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)n - 1024));
}

/* bfloat16 -> double: the 16 bits are the top half of an IEEE binary32. */
ORACLE_API double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static inline uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ------------------------------------------------------------ Q4_K / Q6_K -- */

/* Bit b of the little-endian bit string that starts at p. */
static inline int bit_at(const uint8_t *p, int b) { return (p[b >> 3] >> (b & 7)) & 1; }

static int field6(const uint8_t *bits, int first_bit)
{
    int v = 0;
    for (int k = 0; k < 6; k++)
        v |= bit_at(bits, first_bit + k) << k;
    return v;
}

/* Unpack every field of one Q4_K block (used by the dequantiser and the tests). */
ORACLE_API void oracle_unpack_q4k(const uint8_t *blk, double *d, double *dmin, int sc[8], int m[8], int q[256])
{
    *d = oracle_half_to_double(rd16(blk + 0));
    *dmin = oracle_half_to_double(rd16(blk + 2));
    for (int j = 0; j < 8; j++) {
        sc[j] = field6(blk + 4, 6 * j);
        m[j] = field6(blk + 4, 48 + 6 * j);
    }
    for (int j = 0; j < 8; j++)
        for (int i = 0; i < 16; i++) {
            uint8_t byte = blk[16 + 16 * j + i];
            q[32 * j + i] = byte & 15;
            q[32 * j + 16 + i] = byte >> 4;
        }
}

/* Pack fields into one Q4_K block: the inverse of oracle_unpack_q4k. */
ORACLE_API void oracle_pack_q4k(uint16_t d_bits, uint16_t dmin_bits, const int sc[8], const int m[8], const int q[256], uint8_t *blk)
{
    memset(blk, 0, 144);
    blk[0] = d_bits & 255;    blk[1] = d_bits >> 8;
    blk[2] = dmin_bits & 255; blk[3] = dmin_bits >> 8;
    for (int j = 0; j < 8; j++)
        for (int k = 0; k < 6; k++) {
            int b = 6 * j + k;
            blk[4 + (b >> 3)] |= (uint8_t)(((sc[j] >> k) & 1) << (b & 7));
            b = 48 + 6 * j + k;
            blk[4 + (b >> 3)] |= (uint8_t)(((m[j] >> k) & 1) << (b & 7));
        }
    for (int j = 0; j < 8; j++)
        for (int i = 0; i < 16; i++)
            blk[16 + 16 * j + i] = (uint8_t)((q[32 * j + i] & 15) | ((q[32 * j + 16 + i] & 15) << 4));
}

/* weight n = d * sc_j * q_n - dmin * m_j, evaluated in double. */
static void dequant_q4k_block(const uint8_t *blk, double *w)
{
    double d, dmin;
    int sc[8], m[8], q[256];
    oracle_unpack_q4k(blk, &d, &dmin, sc, m, q);
    for (int n = 0; n < 256; n++) {
        int j = n / 32;
        w[n] = d * sc[j] * q[n] - dmin * m[j];
    }
}

ORACLE_API void oracle_unpack_q6k(const uint8_t *blk, double *d, int sc[16], int q[256])
{
    for (int s = 0; s < 16; s++)
        sc[s] = (int)(int8_t)blk[192 + s];
    *d = oracle_half_to_double(rd16(blk + 208));
    for (int g = 0; g < 8; g++) {
        for (int i = 0; i < 16; i++) {
            uint8_t byte = blk[16 * g + i];
            q[32 * g + i] = byte & 15;
            q[32 * g + 16 + i] = byte >> 4;
        }
        for (int h = 0; h < 2; h++)
            for (int t = 0; t < 4; t++)
                for (int e = 0; e < 4; e++) {
                    int hi = (blk[128 + 8 * g + 4 * h + e] >> (2 * t)) & 3;
                    q[32 * g + 16 * h + 4 * t + e] |= hi << 4;
                }
    }
}

ORACLE_API void oracle_pack_q6k(uint16_t d_bits, const int sc[16], const int q[256], uint8_t *blk)
{
    memset(blk, 0, 210);
    for (int g = 0; g < 8; g++) {
        for (int i = 0; i < 16; i++)
            blk[16 * g + i] = (uint8_t)((q[32 * g + i] & 15) | ((q[32 * g + 16 + i] & 15) << 4));
        for (int h = 0; h < 2; h++)
            for (int t = 0; t < 4; t++)
                for (int e = 0; e < 4; e++) {
                    int hi = (q[32 * g + 16 * h + 4 * t + e] >> 4) & 3;
                    blk[128 + 8 * g + 4 * h + e] |= (uint8_t)(hi << (2 * t));
                }
    }
    for (int s = 0; s < 16; s++)
        blk[192 + s] = (uint8_t)(int8_t)sc[s];
    blk[208] = d_bits & 255;
    blk[209] = d_bits >> 8;
}

/* weight n = d * sc[n/16] * (q_n - 32), evaluated in double. */
static void dequant_q6k_block(const uint8_t *blk, double *w)
{
    double d;
    int sc[16], q[256];
    oracle_unpack_q6k(blk, &d, sc, q);
    for (int n = 0; n < 256; n++)
        w[n] = d * sc[n / 16] * (q[n] - 32);
}

ORACLE_API void oracle_unpack_q2k(const uint8_t *blk, double *d, double *dmin, int sc[16], int m[16], int q[256])
{
    *d = oracle_half_to_double(rd16(blk + 0));
    *dmin = oracle_half_to_double(rd16(blk + 2));
    for (int j = 0; j < 16; j++) {
        sc[j] = blk[4 + j] & 15;
        m[j] = blk[4 + j] >> 4;
    }
    for (int j = 0; j < 16; j++)
        for (int k = 0; k < 4; k++)
            for (int b = 0; b < 4; b++)
                q[16 * j + 4 * k + b] = (blk[20 + 4 * j + b] >> (2 * k)) & 3;
}

ORACLE_API void oracle_pack_q2k(uint16_t d_bits, uint16_t dmin_bits, const int sc[16], const int m[16], const int q[256], uint8_t *blk)
{
    memset(blk, 0, 84);
    blk[0] = d_bits & 255;    blk[1] = d_bits >> 8;
    blk[2] = dmin_bits & 255; blk[3] = dmin_bits >> 8;
    for (int j = 0; j < 16; j++)
        blk[4 + j] = (uint8_t)((sc[j] & 15) | ((m[j] & 15) << 4));
    for (int j = 0; j < 16; j++)
        for (int k = 0; k < 4; k++)
            for (int b = 0; b < 4; b++)
                blk[20 + 4 * j + b] |= (uint8_t)((q[16 * j + 4 * k + b] & 3) << (2 * k));
}

/* weight n = d * sc[n/16] * q_n - dmin * m[n/16], evaluated in double. */
static void dequant_q2k_block(const uint8_t *blk, double *w)
{
    double d, dmin;
    int sc[16], m[16], q[256];
    oracle_unpack_q2k(blk, &d, &dmin, sc, m, q);
    for (int n = 0; n < 256; n++)
        w[n] = d * sc[n / 16] * q[n] - dmin * m[n / 16];
}

ORACLE_API void oracle_dequant_q2k(const uint8_t *blocks, long long nblocks, double *out)
{
#pragma omp parallel for schedule(static)
    for (long long b = 0; b < nblocks; b++)
        dequant_q2k_block(blocks + 84 * b, out + 256 * b);
}

ORACLE_API void oracle_dequant_q4k(const uint8_t *blocks, long long nblocks, double *out)
{
#pragma omp parallel for schedule(static)
    for (long long b = 0; b < nblocks; b++)
        dequant_q4k_block(blocks + 144 * b, out + 256 * b);
}

ORACLE_API void oracle_dequant_q6k(const uint8_t *blocks, long long nblocks, double *out)
{
#pragma omp parallel for schedule(static)
    for (long long b = 0; b < nblocks; b++)
        dequant_q6k_block(blocks + 210 * b, out + 256 * b);
}

/* ----------------------------------------------------------------- GEMV -- */

enum { FMT_BF16 = 0, FMT_Q4K = 1, FMT_Q6K = 2, FMT_Q2K = 3 };

static size_t row_bytes(int fmt, int K)
{
    if (fmt == FMT_BF16)
        return (size_t)K * 2;
    if (fmt == FMT_Q4K)
        return (size_t)(K / 256) * 144;
    if (fmt == FMT_Q2K)
        return (size_t)(K / 256) * 84;
    return (size_t)(K / 256) * 210;
}

/* y[r] = sum_k W[r][k] * x[k], one double accumulator per row, k ascending. */
static void gemv_any(int fmt, const uint8_t *W, const double *x, double *y, int rows, int K)
{
    size_t rb = row_bytes(fmt, K);
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; r++) {
        const uint8_t *row = W + rb * (size_t)r;
        double w[256];
        double acc = 0.0;
        if (fmt == FMT_BF16) {
            for (int k = 0; k < K; k++)
                acc += oracle_bf16_to_double(rd16(row + 2 * (size_t)k)) * x[k];
        } else {
            for (int b = 0; b < K / 256; b++) {
                if (fmt == FMT_Q4K)
                    dequant_q4k_block(row + 144 * (size_t)b, w);
                else if (fmt == FMT_Q2K)
                    dequant_q2k_block(row + 84 * (size_t)b, w);
                else
                    dequant_q6k_block(row + 210 * (size_t)b, w);
                for (int n = 0; n < 256; n++)
                    acc += w[n] * x[256 * b + n];
            }
        }
        y[r] = acc;
    }
}

ORACLE_API void oracle_gemv_bf16(const uint16_t *W, const uint16_t *x, double *y, int rows, int K)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; k++)
        xd[k] = oracle_bf16_to_double(x[k]);
    gemv_any(FMT_BF16, (const uint8_t *)W, xd, y, rows, K);
    free(xd);
}

ORACLE_API void oracle_gemv_q4k(const uint8_t *W, const float *x, double *y, int rows, int K)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; k++)
        xd[k] = x[k];
    gemv_any(FMT_Q4K, W, xd, y, rows, K);
    free(xd);
}

ORACLE_API void oracle_gemv_q6k(const uint8_t *W, const float *x, double *y, int rows, int K)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; k++)
        xd[k] = x[k];
    gemv_any(FMT_Q6K, W, xd, y, rows, K);
    free(xd);
}

ORACLE_API void oracle_gemv_q2k(const uint8_t *W, const float *x, double *y, int rows, int K)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int k = 0; k < K; k++)
        xd[k] = x[k];
    gemv_any(FMT_Q2K, W, xd, y, rows, K);
    free(xd);
}

/* Y[m][r] = sum_k W[r][k] * X[m][k] for M token vectors (the M-sweep). */
ORACLE_API void oracle_matmul_q4k(const uint8_t *W, const float *X, double *Y, int M, int rows, int K)
{
    double *xd = (double *)malloc(sizeof(double) * (size_t)K);
    for (int m = 0; m < M; m++) {
        for (int k = 0; k < K; k++)
            xd[k] = X[(size_t)m * K + k];
        gemv_any(FMT_Q4K, W, xd, Y + (size_t)m * rows, rows, K);
    }
    free(xd);
}

/* ---------------------------------------------------------------- norms -- */

static void rmsnorm_row(const double *x, const float *gamma, double *y, int n, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < n; i++)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / n + eps);
    for (int i = 0; i < n; i++)
        y[i] = x[i] * inv * (double)gamma[i];
}

ORACLE_API void oracle_rmsnorm(const float *x, const float *gamma, double *y, int rows, int n, double eps)
{
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; r++) {
        double *xd = (double *)malloc(sizeof(double) * (size_t)n);
        for (int i = 0; i < n; i++)
            xd[i] = x[(size_t)r * n + i];
        rmsnorm_row(xd, gamma, y + (size_t)r * n, n, eps);
        free(xd);
    }
}

/* Two passes: the mean first, then the variance of (x - mean). */
ORACLE_API void oracle_layernorm(const float *x, const float *gamma, const float *beta, double *y, int rows, int n, double eps)
{
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; r++) {
        const float *xr = x + (size_t)r * n;
        double s = 0.0;
        for (int i = 0; i < n; i++)
            s += xr[i];
        double mean = s / n;
        double v = 0.0;
        for (int i = 0; i < n; i++)
            v += (xr[i] - mean) * (xr[i] - mean);
        double inv = 1.0 / sqrt(v / n + eps);
        for (int i = 0; i < n; i++)
            y[(size_t)r * n + i] = (xr[i] - mean) * inv * (double)gamma[i] + (double)beta[i];
    }
}

/* ------------------------------------------------------------ attention -- */

/* Grouped-query decode attention for one layer.  q: [n_q][hd]; kc/vc: this
 * layer's fp16 K and V planes [n_kv][max_ctx][hd]; keys 0 .. n_keys-1.
 * Query head h reads KV head h / (n_q / n_kv).  Softmax is max-subtracted. */
ORACLE_API void oracle_attention(const double *q, const uint16_t *kc, const uint16_t *vc, double *out,
                                 int n_q, int n_kv, int hd, int max_ctx, int n_keys)
{
    int group = n_q / n_kv;
    double scale = 1.0 / sqrt((double)hd);
#pragma omp parallel for schedule(static)
    for (int h = 0; h < n_q; h++) {
        int g = h / group;
        double *s = (double *)malloc(sizeof(double) * (size_t)n_keys);
        double mx = -INFINITY;
        for (int j = 0; j < n_keys; j++) {
            const uint16_t *kr = kc + ((size_t)g * max_ctx + j) * hd;
            double dot = 0.0;
            for (int dd = 0; dd < hd; dd++)
                dot += q[h * hd + dd] * oracle_half_to_double(kr[dd]);
            s[j] = dot * scale;
            if (s[j] > mx)
                mx = s[j];
        }
        double l = 0.0;
        for (int j = 0; j < n_keys; j++) {
            s[j] = exp(s[j] - mx);
            l += s[j];
        }
        for (int dd = 0; dd < hd; dd++) {
            double o = 0.0;
            for (int j = 0; j < n_keys; j++)
                o += s[j] * oracle_half_to_double(vc[((size_t)g * max_ctx + j) * hd + dd]);
            out[h * hd + dd] = o / l;
        }
        free(s);
    }
}

ORACLE_API double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------ Qwen3 attention inputs -- */
/* The pages name the model (Qwen3-8B) but not its attention's input transforms;
 * these are the model family's own, written from their definitions:
 *   - per-head RMSNorm ("QK-norm"): each head's vector v (hd values) becomes
 *     v / sqrt(mean(v^2) + eps) * w, with one weight vector w[hd] per layer for
 *     all query heads and one for all key heads;
 *   - rotary position embedding, rotate-half pairing: for i < hd/2 the pair
 *     (v[i], v[i + hd/2]) turns by the angle pos * theta^(-2i/hd). */

ORACLE_API void oracle_head_rmsnorm(double *v, const float *w, int hd, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < hd; i++)
        ss += v[i] * v[i];
    double r = 1.0 / sqrt(ss / hd + eps);
    for (int i = 0; i < hd; i++)
        v[i] = v[i] * r * (double)w[i];
}

ORACLE_API void oracle_rope(double *v, int hd, int pos, double theta)
{
    int half = hd / 2;
    for (int i = 0; i < half; i++) {
        double ang = (double)pos * pow(theta, -2.0 * i / hd);
        double c = cos(ang), sn = sin(ang);
        double a = v[i], b = v[i + half];
        v[i] = a * c - b * sn;
        v[i + half] = b * c + a * sn;
    }
}

/* ---------------------------------------------------------- decode step -- */

typedef struct {
    int n_layers, hidden, ffn, n_q_heads, n_kv_heads, head_dim, vocab, max_ctx;
    double eps;
    const float *const *attn_norm;  /* [L] -> fp32[hidden] */
    const uint8_t *const *wqkv;     /* [L] -> Q4_K [(n_q + 2 n_kv) hd][hidden], rows q | k | v */
    const uint8_t *const *wo;       /* [L] -> Q4_K [hidden][n_q hd] */
    const float *const *ffn_norm;   /* [L] */
    const uint8_t *const *wgate;    /* [L] -> Q4_K [ffn][hidden] */
    const uint8_t *const *wup;      /* [L] -> Q4_K [ffn][hidden] */
    const uint8_t *const *wdown;    /* [L] -> Q4_K or Q6_K [hidden][ffn] */
    const int *down_fmt;            /* [L] 1 = Q4_K, 2 = Q6_K */
    const float *out_norm;          /* fp32[hidden] */
    const uint8_t *wvocab;          /* Q6_K [vocab][hidden] */
    uint16_t *kv_cache;             /* fp16 [L][2][n_kv][max_ctx][hd] */
    /* Qwen3 attention inputs; q_norm NULL: plain attention on the projections */
    const float *const *q_norm;     /* [L] -> fp32[hd] */
    const float *const *k_norm;     /* [L] -> fp32[hd] */
    double rope_theta;
} oracle_model;

/* One token: x_in (fp32 hidden) at position pos.  With Qwen3 attention inputs,
 * q and k are head-normalised and rotated first.  Appends this token's k and v
 * (rounded to fp16) to the cache, then attends over keys 0..pos.  Writes the
 * final hidden state (double) when x_out is not NULL, and the logits. */
ORACLE_API void oracle_decode_step(const oracle_model *mdl, const float *x_in, int pos, double *logits, double *x_out)
{
    int H = mdl->hidden, F = mdl->ffn, hd = mdl->head_dim;
    int nq = mdl->n_q_heads, nkv = mdl->n_kv_heads;
    int qdim = nq * hd, kvdim = nkv * hd;
    double *x = (double *)malloc(sizeof(double) * H);
    double *h = (double *)malloc(sizeof(double) * (F > H ? F : H));
    double *qkv = (double *)malloc(sizeof(double) * (qdim + 2 * kvdim));
    double *att = (double *)malloc(sizeof(double) * qdim);
    double *y = (double *)malloc(sizeof(double) * H);
    double *g = (double *)malloc(sizeof(double) * F);
    double *u = (double *)malloc(sizeof(double) * F);
    for (int i = 0; i < H; i++)
        x[i] = x_in[i];
    size_t plane = (size_t)nkv * mdl->max_ctx * hd;
    for (int l = 0; l < mdl->n_layers; l++) {
        rmsnorm_row(x, mdl->attn_norm[l], h, H, mdl->eps);
        gemv_any(FMT_Q4K, mdl->wqkv[l], h, qkv, qdim + 2 * kvdim, H);
        if (mdl->q_norm) { /* QK-norm, then RoPE at pos, on every q and k head */
            for (int hh = 0; hh < nq; hh++) {
                oracle_head_rmsnorm(qkv + hh * hd, mdl->q_norm[l], hd, mdl->eps);
                oracle_rope(qkv + hh * hd, hd, pos, mdl->rope_theta);
            }
            for (int kvh = 0; kvh < nkv; kvh++) {
                oracle_head_rmsnorm(qkv + qdim + kvh * hd, mdl->k_norm[l], hd, mdl->eps);
                oracle_rope(qkv + qdim + kvh * hd, hd, pos, mdl->rope_theta);
            }
        }
        uint16_t *kc = mdl->kv_cache + (size_t)l * 2 * plane;
        uint16_t *vc = kc + plane;
        for (int kvh = 0; kvh < nkv; kvh++)
            for (int dd = 0; dd < hd; dd++) {
                size_t at = ((size_t)kvh * mdl->max_ctx + pos) * hd + dd;
                kc[at] = oracle_double_to_half(qkv[qdim + kvh * hd + dd]);
                vc[at] = oracle_double_to_half(qkv[qdim + kvdim + kvh * hd + dd]);
            }
        oracle_attention(qkv, kc, vc, att, nq, nkv, hd, mdl->max_ctx, pos + 1);
        gemv_any(FMT_Q4K, mdl->wo[l], att, y, H, qdim);
        for (int i = 0; i < H; i++)
            x[i] += y[i];
        rmsnorm_row(x, mdl->ffn_norm[l], h, H, mdl->eps);
        gemv_any(FMT_Q4K, mdl->wgate[l], h, g, F, H);
        gemv_any(FMT_Q4K, mdl->wup[l], h, u, F, H);
        for (int i = 0; i < F; i++)
            g[i] = oracle_silu(g[i]) * u[i];
        gemv_any(mdl->down_fmt[l] == 2 ? FMT_Q6K : FMT_Q4K, mdl->wdown[l], g, y, H, F);
        for (int i = 0; i < H; i++)
            x[i] += y[i];
    }
    if (x_out)
        memcpy(x_out, x, sizeof(double) * H);
    rmsnorm_row(x, mdl->out_norm, h, H, mdl->eps);
    gemv_any(FMT_Q6K, mdl->wvocab, h, logits, mdl->vocab, H);
    free(x); free(h); free(qkv); free(att); free(y); free(g); free(u);
}

ORACLE_API int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
