/*
 * attn_oracle.c -- plain, slow float64 CPU oracle for the fused exact-attention
 * forward pass and for the FP8-E4M3 per-block quantiser.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table or
 * constant with the CUDA library: every formula below is written out from the
 * definitions on the pages it cites.
 *
 * Pages cited (titles as published):
 *   [WGC]  "Warp Group Cluster 优化：Flash Attention V3 在 H100 上的 FP8 融合计算实践"
 *   [JJ]   "大模型加速-核心网络算子-Flash Attention V3"
 *   [YT]   "FlashAttention V3：优化框架吞吐量的关键技术实践"
 *
 * What is computed (per head, query row i, allowed key set A_i):
 *   s_ij  = scale * sum_k q_ik k_jk                       for j in A_i
 *   m_i   = max_j s_ij,  l_i = sum_j exp(s_ij - m_i)
 *   P_ij  = exp(s_ij - m_i) / l_i,  O_i = sum_j P_ij v_j,  LSE_i = m_i + ln l_i
 * This is standard attention, which the method reaches exactly up to rounding
 * ([WGC] §背景：注意力计算的硬件瓶颈 -- tiling and recomputation keep the result
 * and drop the N x N memory; [YT] §1.2 -- softmax, mask and matmul fused in one
 * kernel).  The oracle therefore is that definition, two passes per row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Allowed key set A_i.                                                       */
/*   causal == 0, window <= 0 : all keys 0 <= j < N                          */
/*   causal == 1, window <= 0 : j <= i                                        */
/*   causal == 0, window  > 0 : i - window <= j <= i + window                 */
/*       ([YT] §2.1.2 稀疏性感知的Mask优化: row i keeps columns                */
/*        max(0, i - window) .. i + window inclusive)                         */
/*   causal == 1, window  > 0 : i - window <= j <= i  (the same left edge)    */
/* ------------------------------------------------------------------------- */
int oracle_key_allowed(long i, long j, long N, int causal, long window)
{
    if (j < 0 || j >= N) return 0;
    if (causal && j > i) return 0;
    if (window > 0) {
        if (j < i - window) return 0;
        if (!causal && j > i + window) return 0;
    }
    return 1;
}

static double dot_f64(const double* a, const double* b, long d)
{
    double acc = 0.0;
    for (long t = 0; t < d; ++t) acc += a[t] * b[t];
    return acc;
}

/* One query row, two passes: scores and their max, then the normalised sum. */
static void attn_row(const double* qi, const double* k, const double* v, long N, long d,
                     double scale, int causal, long window, long i, double* s,
                     double* oi, double* lse_i)
{
    double m = -INFINITY;
    long count = 0;
    for (long j = 0; j < N; ++j) {
        if (!oracle_key_allowed(i, j, N, causal, window)) continue;
        s[j] = scale * dot_f64(qi, k + j * d, d);
        if (s[j] > m) m = s[j];
        ++count;
    }
    for (long t = 0; t < d; ++t) oi[t] = 0.0;
    if (count == 0) { /* empty A_i: O = 0, LSE = -inf */
        *lse_i = -INFINITY;
        return;
    }
    double l = 0.0;
    for (long j = 0; j < N; ++j) {
        if (!oracle_key_allowed(i, j, N, causal, window)) continue;
        l += exp(s[j] - m);
    }
    for (long j = 0; j < N; ++j) {
        if (!oracle_key_allowed(i, j, N, causal, window)) continue;
        const double p = exp(s[j] - m) / l;
        const double* vj = v + j * d;
        for (long t = 0; t < d; ++t) oi[t] += p * vj[t];
    }
    *lse_i = m + log(l);
}

static int pick_threads(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * Selected rows of one head.
 *   q, k, v : [N, d] row-major float64 (the bf16 inputs widened exactly)
 *   rows    : R query indices in [0, N)
 *   o       : [R, d] output, lse : [R] output (natural log)
 * Returns the number of threads used.
 */
int oracle_attn_rows_f64(const double* q, const double* k, const double* v, long N, long d,
                         double scale, int causal, long window, const long* rows, long R,
                         double* o, double* lse, int nthreads)
{
    const int nt = pick_threads(nthreads);
#pragma omp parallel num_threads(nt)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < R; ++r) {
            const long i = rows[r];
            attn_row(q + i * d, k, v, N, d, scale, causal, window, i, s, o + r * d, lse + r);
        }
        free(s);
    }
    return nt;
}

/*
 * All rows of BH independent heads.
 *   q, k, v, o : [BH, N, d] row-major float64,  lse : [BH, N]
 * Returns the number of threads used.
 */
int oracle_attn_f64(const double* q, const double* k, const double* v, long BH, long N, long d,
                    double scale, int causal, long window, double* o, double* lse, int nthreads)
{
    const int nt = pick_threads(nthreads);
#pragma omp parallel num_threads(nt)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 8)
        for (long u = 0; u < BH * N; ++u) {
            const long h = u / N, i = u % N;
            const long base = h * N * d;
            attn_row(q + base + i * d, k + base, v + base, N, d, scale, causal, window, i, s,
                     o + base + i * d, lse + h * N + i);
        }
        free(s);
    }
    return nt;
}

/*
 * Tile-by-tile replay of the online softmax, one head, all rows.
 *
 * [WGC] §2 GEMM-Softmax 融合流水线: each block contributes its local max and
 * sum, the running statistics are updated, and the partial output is rescaled
 * before the next block's contribution is added; [JJ] §2.4 names the same
 * step-wise accumulation as the guard against overflow.
 *
 * Query rows are taken in blocks of BM and keys in tiles of BN.  For each
 * query block the key tiles visited are only those that can hold an allowed
 * key of some row of the block (the tile-skipping bounds below); inside a
 * visited tile, keys outside A_i are dropped.  Per row:
 *     m_new = max(m_used, tile max)
 *     if m_new - m_used > tau:  acc *= exp(m_used - m_new), l *= same, m_used = m_new
 *     acc += sum_j exp(s_j - m_used) v_j,   l += sum_j exp(s_j - m_used)
 * tau = 0 is the eager update; tau > 0 keeps a stale maximum while the new
 * one exceeds it by at most tau (natural-log units), which is exact after the
 * final O = acc / l, LSE = m_used + ln l.
 */
void oracle_online_replay_f64(const double* q, const double* k, const double* v, long N, long d,
                              double scale, int causal, long window, long BM, long BN,
                              double tau, double* o, double* lse)
{
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    for (long r0 = 0; r0 < N; r0 += BM) {
        const long r1 = (r0 + BM < N) ? r0 + BM : N; /* rows [r0, r1) */
        /* key bounds [lo, hi) covering every allowed key of rows r0..r1-1 */
        long lo = 0, hi = N;
        if (window > 0) lo = r0 - window;
        if (lo < 0) lo = 0;
        if (causal) hi = r1;
        else if (window > 0) hi = r1 - 1 + window + 1;
        if (hi > N) hi = N;
        const long t_begin = lo / BN;
        const long t_end = (hi + BN - 1) / BN;
        for (long i = r0; i < r1; ++i) {
            const double* qi = q + i * d;
            double m_used = -INFINITY, l = 0.0;
            for (long t = 0; t < d; ++t) acc[t] = 0.0;
            for (long tile = t_begin; tile < t_end; ++tile) {
                const long j0 = tile * BN;
                const long j1 = (j0 + BN < N) ? j0 + BN : N;
                double tmax = -INFINITY;
                for (long j = j0; j < j1; ++j) {
                    if (!oracle_key_allowed(i, j, N, causal, window)) continue;
                    const double s = scale * dot_f64(qi, k + j * d, d);
                    if (s > tmax) tmax = s;
                }
                if (tmax == -INFINITY) continue; /* nothing allowed in this tile */
                const double m_new = tmax > m_used ? tmax : m_used;
                if (m_used == -INFINITY || m_new - m_used > tau) {
                    const double alpha = (m_used == -INFINITY) ? 0.0 : exp(m_used - m_new);
                    for (long t = 0; t < d; ++t) acc[t] *= alpha;
                    l *= alpha;
                    m_used = m_new;
                }
                for (long j = j0; j < j1; ++j) {
                    if (!oracle_key_allowed(i, j, N, causal, window)) continue;
                    const double s = scale * dot_f64(qi, k + j * d, d);
                    const double p = exp(s - m_used);
                    l += p;
                    const double* vj = v + j * d;
                    for (long t = 0; t < d; ++t) acc[t] += p * vj[t];
                }
            }
            if (l > 0.0) {
                for (long t = 0; t < d; ++t) o[i * d + t] = acc[t] / l;
                lse[i] = m_used + log(l);
            } else {
                for (long t = 0; t < d; ++t) o[i * d + t] = 0.0;
                lse[i] = -INFINITY;
            }
        }
    }
    free(acc);
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 codec, written from the OCP 8-bit floating point definition:      */
/*   1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;                */
/*   exponent field 0 holds subnormals m * 2^-9;                              */
/*   the pattern S.1111.111 is NaN, there is no infinity, largest finite 448. */
/* [JJ] §1.5 低精度FP8 names E4M3 as the 4-exponent / 3-mantissa format.       */
/* Encoding rounds to nearest, ties to even, and saturates out-of-range       */
/* magnitudes (and infinities) to +-448 ("satfinite").                        */
/* ------------------------------------------------------------------------- */
uint8_t oracle_e4m3_encode(float x)
{
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    if (isinf(x)) return (uint8_t)(sign | 0x7E);
    const double a = fabs((double)x);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: units of 2^-9; the integer 8 is the smallest normal (code 0x08) */
        const double units = rint(a * 512.0); /* exact scaling, ties to even */
        return (uint8_t)(sign | (uint8_t)units);
    }
    int e2;
    (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;      /* a in [2^e, 2^(e+1)) */
    double r = rint(ldexp(a, 3 - e)); /* mantissa with 3 fraction bits, in [8, 16] */
    if (r == 16.0) { r = 8.0; e += 1; }
    if (e > 8) return (uint8_t)(sign | 0x7E);
    const int code = ((e + 7) << 3) | ((int)r - 8);
    if (code > 0x7E) return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | code);
}

float oracle_e4m3_decode(uint8_t c)
{
    const double sgn = (c & 0x80) ? -1.0 : 1.0;
    const int e = (c >> 3) & 0xF, m = c & 0x7;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) return (float)(sgn * ldexp((double)m, -9));
    return (float)(sgn * ldexp(1.0 + m / 8.0, e - 7));
}

void oracle_e4m3_encode_array(const float* x, uint8_t* out, long n)
{
#pragma omp parallel for schedule(static)
    for (long t = 0; t < n; ++t) out[t] = oracle_e4m3_encode(x[t]);
}

/*
 * Per-block FP8 quantisation ([WGC] §3 FP8 量化与精度保持: per-block dynamic
 * scale mapping the block's range onto the FP8 range; [JJ] §1 item 3 块量化).
 * For each head and each block of `block` consecutive rows (all d columns):
 *   amax  = max |x|           (fp32, exact)
 *   scale = amax / 448        (fp32 IEEE division);  scale = 1 when amax == 0
 *   x8    = e4m3(x / scale)   (fp32 IEEE division, then one RNE satfinite rounding)
 * x: [BH, N, d] float32 (bf16 values widened), x8: same shape, scales: [BH, ceil(N/block)].
 */
void oracle_quantize_fp8_blockwise(const float* x, uint8_t* x8, float* scales, long BH, long N,
                                   long d, long block)
{
    const long nblk = (N + block - 1) / block;
#pragma omp parallel for schedule(static)
    for (long u = 0; u < BH * nblk; ++u) {
        const long h = u / nblk, b = u % nblk;
        const long r0 = b * block, r1 = (r0 + block < N) ? r0 + block : N;
        const float* xb = x + (h * N + r0) * d;
        uint8_t* yb = x8 + (h * N + r0) * d;
        const long cnt = (r1 - r0) * d;
        float amax = 0.0f;
        for (long t = 0; t < cnt; ++t) {
            const float a = fabsf(xb[t]);
            if (a > amax) amax = a;
        }
        const float scale = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        for (long t = 0; t < cnt; ++t) {
            const float qv = xb[t] / scale;
            yb[t] = oracle_e4m3_encode(qv);
        }
        scales[u] = scale;
    }
}

/* ------------------------------------------------------------------------- */
/* FP8 E5M2 codec, written from the OCP 8-bit floating point definition:      */
/*   1 sign bit, 5 exponent bits with bias 15, 2 mantissa bits;               */
/*   exponent field 0 holds subnormals m * 2^-16; exponent field 31 holds     */
/*   infinity (mantissa 0) and NaN (mantissa != 0); largest finite 57344.     */
/* [JJ] §1.5 低精度FP8 names E5M2 as the 5-exponent / 2-mantissa format with   */
/* the wider range; [WGC] §3 lists both formats.  Encoding rounds to nearest, */
/* ties to even, and saturates out-of-range magnitudes (and infinities) to    */
/* +-57344 ("satfinite"), as the E4M3 encoder does to +-448.                  */
/* ------------------------------------------------------------------------- */
uint8_t oracle_e5m2_encode(float x)
{
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    if (isinf(x)) return (uint8_t)(sign | 0x7B);
    const double a = fabs((double)x);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: units of 2^-16; the integer 4 is the smallest normal (code 0x04) */
        const double units = rint(a * 65536.0); /* exact scaling, ties to even */
        return (uint8_t)(sign | (uint8_t)units);
    }
    int e2;
    (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;      /* a in [2^e, 2^(e+1)) */
    double r = rint(ldexp(a, 2 - e)); /* mantissa with 2 fraction bits, in [4, 8] */
    if (r == 8.0) { r = 4.0; e += 1; }
    if (e > 15) return (uint8_t)(sign | 0x7B);
    const int code = ((e + 15) << 2) | ((int)r - 4);
    if (code > 0x7B) return (uint8_t)(sign | 0x7B);
    return (uint8_t)(sign | code);
}

float oracle_e5m2_decode(uint8_t c)
{
    const double sgn = (c & 0x80) ? -1.0 : 1.0;
    const int e = (c >> 2) & 0x1F, m = c & 0x3;
    if (e == 0x1F) return (m == 0) ? (float)(sgn * INFINITY) : NAN;
    if (e == 0) return (float)(sgn * ldexp((double)m, -16));
    return (float)(sgn * ldexp(1.0 + m / 4.0, e - 15));
}

void oracle_e5m2_encode_array(const float* x, uint8_t* out, long n)
{
#pragma omp parallel for schedule(static)
    for (long t = 0; t < n; ++t) out[t] = oracle_e5m2_encode(x[t]);
}

/*
 * Per-block FP8 quantisation into either format: as oracle_quantize_fp8_blockwise,
 * with the format's largest finite value in place of 448:
 *   fmt 0 (E4M3): scale = amax / 448,   x8 = e4m3(x / scale)
 *   fmt 1 (E5M2): scale = amax / 57344, x8 = e5m2(x / scale)
 *   fmt 2 (E4M3 with power-of-two scales): s0 = amax / 448 (fp32), scale = the smallest
 *          power of two >= s0 (a shared exponent per block, as in the OCP microscaling
 *          formats; [WGC] §3 asks only for a per-block scale), x8 = e4m3(x / scale),
 *          the quotient exact.
 */
static float pow2_at_least(float s0)
{
    int e;
    const float f = frexpf(s0, &e); /* s0 = f * 2^e, f in [0.5, 1) */
    return (f == 0.5f) ? s0 : ldexpf(1.0f, e);
}

void oracle_quantize_fp8_blockwise_fmt(const float* x, uint8_t* x8, float* scales, long BH, long N,
                                       long d, long block, int fmt)
{
    const long nblk = (N + block - 1) / block;
    const float fmax = (fmt == 1) ? 57344.0f : 448.0f;
#pragma omp parallel for schedule(static)
    for (long u = 0; u < BH * nblk; ++u) {
        const long h = u / nblk, b = u % nblk;
        const long r0 = b * block, r1 = (r0 + block < N) ? r0 + block : N;
        const float* xb = x + (h * N + r0) * d;
        uint8_t* yb = x8 + (h * N + r0) * d;
        const long cnt = (r1 - r0) * d;
        float amax = 0.0f;
        for (long t = 0; t < cnt; ++t) {
            const float a = fabsf(xb[t]);
            if (a > amax) amax = a;
        }
        float scale = (amax > 0.0f) ? amax / fmax : 1.0f;
        if (fmt == 2 && amax > 0.0f) scale = pow2_at_least(scale);
        for (long t = 0; t < cnt; ++t) {
            const float qv = xb[t] / scale;
            yb[t] = (fmt == 1) ? oracle_e5m2_encode(qv) : oracle_e4m3_encode(qv);
        }
        scales[u] = scale;
    }
}

/*
 * Incoherent processing before FP8 quantisation ("大模型加速-核心网络算子-Flash
 * Attention V3", §1 item 3 and the closing summary: block quantisation together
 * with incoherent processing, credited with a 2.6x lower FP8 error).  The pages do
 * not spell out the transform; the reading taken here is the orthonormal
 * Walsh-Hadamard rotation R = H_d / sqrt(d) applied to each row of Q and of K
 * (H_d the Sylvester Hadamard matrix, entries (-1)^popcount(j & k)).  R is
 * orthogonal, so (Q R)(K R)^T = Q K^T and the attention result is unchanged,
 * while a large entry of a row is spread evenly over all d coordinates.
 *
 * The rotated values decide FP8 codes, so they are computed in fp32 in one fixed
 * order that the GPU kernel repeats exactly: the radix-2 butterfly sweep
 * h = 1, 2, 4, ..., d/2, each pair (i, i + h) with (i & h) == 0 becoming
 * (a + b, a - b), then every output multiplied by c = fp32(1 / sqrt(d)).
 * x, y: [rows, d] float32; d a power of two; y may alias x.
 */
void oracle_hadamard_rotate_f32(const float* x, float* y, long rows, long d, float c)
{
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        float* v = y + r * d;
        const float* u = x + r * d;
        for (long j = 0; j < d; ++j) v[j] = u[j];
        for (long h = 1; h < d; h <<= 1) {
            for (long i = 0; i < d; ++i) {
                if (i & h) continue;
                const float a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
        }
        for (long j = 0; j < d; ++j) v[j] = v[j] * c;
    }
}
