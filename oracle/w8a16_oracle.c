/*
 * CPU oracle for the W8A16 block-scaled GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only
 * tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg
 * may load or run it. It shares no code, header, table or constant with the
 * CUDA library under fp8_weight_only_gemm_gb300/, and includes none of it.
 *
 * What it computes (source: "metrale_model_layers/layers/ops/
 * w8a16_gemm_pipelined_m32.rs", doc comments of `w8a16_gemm_pipelined_m32_strided`
 * (tensor layouts, strides in elements, first k of each A row read, first n of
 * each C row written) and of `W8A16_M32_K_BLOCK` (one FP8 scale block per
 * 128-K step)):
 *
 *   C[m][n] = bf16_rne( sum_{k<K} A[m][k] * ( e4m3(W[n][k]) * scale[n/128][k/128] ) )
 *
 * The sum runs in FP64 in plain k order and is rounded once to BF16 with
 * round-to-nearest-even. Every term is exact in FP64: e4m3 x fp32 needs at most
 * 4 + 24 significant bits and bf16 x that at most 8 + 28 = 36 < 53, so only the
 * additions round; the result is the exact sum to within K ulps of FP64, far
 * below one BF16 ulp. Columns n >= N and A columns k >= K are never touched.
 *
 * Readings where the page is silent (each one is also listed in the design
 * notes): E4M3 is the OCP "FN" flavour (bias 7, no infinities, 0x7F/0xFF NaN,
 * max +-448, subnormals m * 2^-9); the scale grid has ceil(N/128) rows, row n
 * using scale row floor(n/128); NaN inputs propagate as in IEEE arithmetic.
 *
 * It also holds the oracle of the weight block quantiser, the step that makes
 * W and block_scale (same page: the block layout of `block_scale`, one FP32 scale
 * per 128x128 block, with E4M3 codes for W). Our reading of the encoding, the
 * plainest one consistent with it and with the 448 range of E4M3: per block,
 * amax = max |w|, scale = amax / 448 in FP32, code = e4m3_rne(w / scale) with the
 * quotient in FP32 and saturation to +-448; a block with amax = 0 gets scale 0
 * and codes 0. The FP32 divisions are the ones the GPU takes too (a quantised
 * code is decided in the precision that produces it).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -pthread (no fast-math).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- E4M3 (FN) decode, from the format definition ------------------------
 * 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits. Exponent field 0 is
 * subnormal: (m/8) * 2^(1-7). Exponent 15 with mantissa 7 is NaN; there is no
 * infinity, so exponent 15 with mantissa 0..6 is an ordinary normal number. */
double oracle_e4m3_to_double(uint8_t code)
{
    const int sign = (code >> 7) & 1;
    const int e = (code >> 3) & 0xF;
    const int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9); /* m/8 * 2^-6 */
    else
        mag = ldexp(8.0 + m, e - 7 - 3); /* (1 + m/8) * 2^(e-7) */
    return sign ? -mag : mag;
}

/* ---- BF16 <-> FP64 -------------------------------------------------------
 * BF16 is the upper half of an IEEE binary32: the value is that of the float
 * whose upper 16 bits are the code and lower 16 bits are zero. */
double oracle_bf16_to_double(uint16_t code)
{
    uint32_t u = (uint32_t)code << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to BF16 with round-to-nearest, ties to even, in one step
 * (no intermediate binary32 rounding). BF16 keeps 8 significant bits, has
 * binary32's exponent range (normal down to 2^-126) and subnormal quantum
 * 2^-133. Results past the largest finite value become infinities. */
uint16_t oracle_double_to_bf16_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    const int neg = signbit(x) ? 1 : 0;
    const double a = fabs(x);
    uint16_t mag;
    if (a == 0.0) {
        mag = 0;
    } else if (isinf(a)) {
        mag = 0x7F80;
    } else {
        int e;
        (void)frexp(a, &e); /* a = f * 2^e with f in [0.5, 1): leading bit 2^(e-1) */
        int q = (e - 1) - 7; /* weight of the last of 8 significant bits */
        if (q < -133)
            q = -133; /* subnormal range: fixed quantum */
        const double r = nearbyint(ldexp(a, -q)); /* default mode: ties to even */
        const double v = ldexp(r, q);
        if (v >= 0x1p128) {
            mag = 0x7F80;
        } else {
            const float f = (float)v; /* exact: v has <= 8 significant bits */
            uint32_t u;
            memcpy(&u, &f, sizeof u);
            mag = (uint16_t)(u >> 16);
        }
    }
    return (uint16_t)(mag | (neg ? 0x8000u : 0u));
}

/* ---- the GEMM -------------------------------------------------------------- */

typedef struct oracle_job oracle_job;

/* The sum of one output element: *sum_out = sum_k of its terms (FP64, k order),
 * *abs_out = sum_k of their magnitudes (an input of the tests' error bound). */
typedef void (*oracle_output_fn)(const oracle_job *j, uint32_t m, uint32_t n, double *sum_out,
                                 double *abs_out);

struct oracle_job {
    const uint16_t *A;    /* W8A16: BF16 activation codes [M][a_row_stride] */
    const uint8_t *Aq;    /* W8A8: E4M3 activation codes [M][a_row_stride] */
    const float *a_scale; /* W8A8: activation group scales [K/128][M] */
    uint32_t a_row_stride;
    const uint8_t *W;
    const float *scale;
    uint16_t *C;
    uint32_t c_row_stride;
    uint32_t M, N, K;
    double *exact;        /* optional [M*N] pre-rounding sums */
    double *absum;        /* optional [M*N] sums of |terms| */
    uint64_t begin, end;  /* this thread's share of the M*N outputs */
    const double *dec;    /* 256-entry E4M3 table */
    oracle_output_fn output;
};

/* One W8A16 output element, exactly as the definition reads:
 * sum_k A[m][k] * (e4m3(W[n][k]) * scale[n/128][k/128]). */
static void w8a16_output(const oracle_job *j, uint32_t m, uint32_t n, double *sum_out,
                         double *abs_out)
{
    const uint16_t *arow = j->A + (uint64_t)m * j->a_row_stride;
    const uint8_t *wrow = j->W + (uint64_t)n * j->K;
    const float *srow = j->scale + (uint64_t)(n / 128) * (j->K / 128);
    double sum = 0.0, asum = 0.0;
    for (uint32_t k = 0; k < j->K; ++k) {
        const double a = oracle_bf16_to_double(arow[k]);
        const double w = j->dec[wrow[k]];
        const double s = (double)srow[k / 128];
        const double t = a * (w * s);
        sum += t;
        asum += fabs(t);
    }
    *sum_out = sum;
    *abs_out = asum;
}

/* One W8A8 output element: sum_k (e4m3(Aq[m][k]) * a_scale[k/128][m]) *
 * (e4m3(W[n][k]) * scale[n/128][k/128]). */
static void w8a8_output(const oracle_job *j, uint32_t m, uint32_t n, double *sum_out,
                        double *abs_out)
{
    const uint8_t *arow = j->Aq + (uint64_t)m * j->a_row_stride;
    const uint8_t *wrow = j->W + (uint64_t)n * j->K;
    const float *srow = j->scale + (uint64_t)(n / 128) * (j->K / 128);
    double sum = 0.0, asum = 0.0;
    for (uint32_t k = 0; k < j->K; ++k) {
        const double a = j->dec[arow[k]] * (double)j->a_scale[(uint64_t)(k / 128) * j->M + m];
        const double w = j->dec[wrow[k]];
        const double s = (double)srow[k / 128];
        const double t = a * (w * s);
        sum += t;
        asum += fabs(t);
    }
    *sum_out = sum;
    *abs_out = asum;
}

static void *run_share(void *arg)
{
    const oracle_job *j = (const oracle_job *)arg;
    for (uint64_t idx = j->begin; idx < j->end; ++idx) {
        /* Outputs are handed out n-major so a thread reuses one W row across m. */
        const uint32_t n = (uint32_t)(idx / j->M);
        const uint32_t m = (uint32_t)(idx % j->M);
        double sum, asum;
        j->output(j, m, n, &sum, &asum);
        j->C[(uint64_t)m * j->c_row_stride + n] = oracle_double_to_bf16_rne(sum);
        if (j->exact)
            j->exact[(uint64_t)m * j->N + n] = sum;
        if (j->absum)
            j->absum[(uint64_t)m * j->N + n] = asum;
    }
    return NULL;
}

/* All M*N outputs, split evenly over nthreads POSIX threads (each output is
 * computed by one thread, so the thread count never changes a result). */
static int run_threads(oracle_job *base, int nthreads)
{
    const uint64_t total = (uint64_t)base->M * base->N;
    double dec[256];
    for (int c = 0; c < 256; ++c)
        dec[c] = oracle_e4m3_to_double((uint8_t)c);
    base->dec = dec;
    if (nthreads < 1)
        nthreads = 1;
    if ((uint64_t)nthreads > total)
        nthreads = total ? (int)total : 1;
    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *joined = (char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tids || !joined) {
        free(jobs);
        free(tids);
        free(joined);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *base;
        jobs[t].begin = total * (uint64_t)t / (uint64_t)nthreads;
        jobs[t].end = total * (uint64_t)(t + 1) / (uint64_t)nthreads;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, run_share, &jobs[t]) == 0)
            joined[t] = 1;
        else
            run_share(&jobs[t]); /* no thread available: run the share inline */
    }
    run_share(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (joined[t])
            pthread_join(tids[t], NULL);
    free(joined);
    free(jobs);
    free(tids);
    return 0;
}

/* Full product. A: [M][a_row_stride] BF16 codes, W: [N][K] E4M3 codes,
 * scale: [ceil(N/128)][K/128] FP32, C: [M][c_row_stride] BF16 codes (only the
 * first N columns of each row are written). exact/absum may be NULL.
 * Returns 0, or -1 on bad sizes / allocation failure. */
int oracle_w8a16_gemm(const uint16_t *A, uint32_t a_row_stride, const uint8_t *W,
                      const float *scale, uint16_t *C, uint32_t c_row_stride, uint32_t M,
                      uint32_t N, uint32_t K, double *exact, double *absum, int nthreads)
{
    if (M == 0 || N == 0 || K == 0 || K % 128 != 0 || a_row_stride < K || c_row_stride < N)
        return -1;
    oracle_job j;
    memset(&j, 0, sizeof j);
    j.A = A;
    j.a_row_stride = a_row_stride;
    j.W = W;
    j.scale = scale;
    j.C = C;
    j.c_row_stride = c_row_stride;
    j.M = M;
    j.N = N;
    j.K = K;
    j.exact = exact;
    j.absum = absum;
    j.output = w8a16_output;
    return run_threads(&j, nthreads);
}

/* ---- E4M3 (FN) encode, round to nearest, ties to even, saturating ----------
 * The 127 non-negative finite codes 0x00..0x7E decode to increasing values, so
 * the nearest code of |x| is found by bisection over that ordered list; on an
 * exact midpoint the code with an even mantissa (code bit 0 clear) wins. Values
 * beyond 448 saturate to 448; the sign bit is the sign of x (so -0 and negative
 * values that round to zero give 0x80); NaN gives 0x7F. */
uint8_t oracle_e4m3_encode_rne(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    int lo = 0, hi = 0x7E; /* value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (oracle_e4m3_to_double((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    const double dlo = a - oracle_e4m3_to_double((uint8_t)lo);
    const double dhi = oracle_e4m3_to_double((uint8_t)hi) - a;
    int code;
    if (dlo < dhi)
        code = lo;
    else if (dhi < dlo)
        code = hi;
    else
        code = (lo & 1) ? hi : lo; /* tie: even mantissa */
    return sign | (uint8_t)code;
}

/* Block quantiser. W: FP32 [N][w_row_stride] (first K of each row used),
 * codes: [N][K] E4M3, scales: [ceil(N/128)][K/128] FP32. A block's rows stop at N.
 * Returns 0, or -1 on bad sizes. */
int oracle_quantize_weights(const float *W, uint32_t w_row_stride, uint32_t N, uint32_t K,
                            uint8_t *codes, float *scales)
{
    if (N == 0 || K == 0 || K % 128 != 0 || w_row_stride < K)
        return -1;
    const uint32_t nb_rows = (N + 127) / 128, kb_cols = K / 128;
    for (uint32_t nb = 0; nb < nb_rows; ++nb) {
        const uint32_t r1 = (nb + 1) * 128 < N ? (nb + 1) * 128 : N;
        for (uint32_t kb = 0; kb < kb_cols; ++kb) {
            float amax = 0.0f;
            for (uint32_t r = nb * 128; r < r1; ++r)
                for (uint32_t k = kb * 128; k < kb * 128 + 128; ++k) {
                    const float v = fabsf(W[(size_t)r * w_row_stride + k]);
                    if (v > amax)
                        amax = v;
                }
            const float scale = amax / 448.0f;
            scales[(size_t)nb * kb_cols + kb] = scale;
            for (uint32_t r = nb * 128; r < r1; ++r)
                for (uint32_t k = kb * 128; k < kb * 128 + 128; ++k) {
                    uint8_t c = 0;
                    if (scale != 0.0f) {
                        const float q = W[(size_t)r * w_row_stride + k] / scale;
                        c = oracle_e4m3_encode_rne(q);
                    }
                    codes[(size_t)r * K + k] = c;
                }
        }
    }
    return 0;
}

/* ---- W8A8: FP8 activations with per-token 128-K group scales -----------------
 * The adjacent precision variant (page "metrale_model_layers/layers/ops/
 * fp8_act_quant.rs", module doc: per-token quantisation in 128-element K groups;
 * the page gives the launch shape, not the arithmetic). Our reading, the same rule
 * as the weight quantiser on 1x128 groups: per (token m, group g), amax = max |a|,
 * scale = amax / 448 in FP32, code = E4M3 RNE of a / scale (FP32 quotient),
 * saturating; amax = 0 gives scale 0 and codes 0; NaN values do not enter amax.
 * Scales are stored group-major, a_scale[g][m], so one K step's scales of
 * consecutive tokens are contiguous.
 *
 * Quantiser. A: BF16 [M][a_row_stride] (first K of a row), codes: [M][K],
 * scales: [K/128][M]. Returns 0, or -1 on bad sizes. */
int oracle_quantize_activations(const uint16_t *A, uint32_t a_row_stride, uint32_t M, uint32_t K,
                                uint8_t *codes, float *scales)
{
    if (M == 0 || K == 0 || K % 128 != 0 || a_row_stride < K)
        return -1;
    for (uint32_t m = 0; m < M; ++m)
        for (uint32_t g = 0; g < K / 128; ++g) {
            float amax = 0.0f;
            for (uint32_t k = g * 128; k < g * 128 + 128; ++k) {
                const float v = fabsf((float)oracle_bf16_to_double(A[(size_t)m * a_row_stride + k]));
                if (v > amax)
                    amax = v;
            }
            const float scale = amax / 448.0f;
            scales[(size_t)g * M + m] = scale;
            for (uint32_t k = g * 128; k < g * 128 + 128; ++k) {
                uint8_t c = 0;
                if (scale != 0.0f)
                    c = oracle_e4m3_encode_rne((float)oracle_bf16_to_double(A[(size_t)m * a_row_stride + k]) /
                                               scale);
                codes[(size_t)m * K + k] = c;
            }
        }
    return 0;
}

/* W8A8 product: C[m][n] = bf16_rne( sum_k (e4m3(Aq[m][k]) * a_scale[k/128][m]) *
 *                                          (e4m3(W[n][k]) * scale[n/128][k/128]) ),
 * the sum in FP64 in k order (each term rounds once: 28 x 28 significant bits).
 * Same layouts as oracle_w8a16_gemm otherwise. */
int oracle_w8a8_gemm(const uint8_t *Aq, uint32_t a_row_stride, const float *a_scale, const uint8_t *W,
                     const float *scale, uint16_t *C, uint32_t c_row_stride, uint32_t M, uint32_t N,
                     uint32_t K, double *exact, double *absum, int nthreads)
{
    if (M == 0 || N == 0 || K == 0 || K % 128 != 0 || a_row_stride < K || c_row_stride < N)
        return -1;
    oracle_job j;
    memset(&j, 0, sizeof j);
    j.Aq = Aq;
    j.a_scale = a_scale;
    j.a_row_stride = a_row_stride;
    j.W = W;
    j.scale = scale;
    j.C = C;
    j.c_row_stride = c_row_stride;
    j.M = M;
    j.N = N;
    j.K = K;
    j.exact = exact;
    j.absum = absum;
    j.output = w8a8_output;
    return run_threads(&j, nthreads);
}
