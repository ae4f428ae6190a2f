/*
 * CPU oracle for the W4A16 group-quantized GEMM -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this file's library.  The product path never calls it; it shares no
 * code, header, table or helper with the CUDA library.
 *
 * What it computes (plain definition, fp64, no blocking or reordering):
 *
 *     y[m][n] = sum_{k=0}^{K-1} x[m][k] * (q[k][n] - z[k/g][n]) * s[k/g][n]
 *
 * Sources: "Quantize the Target, Quantize the Drafter: Efficient Inference
 * with Qwen3.5-4B" -- pith.science review, referee report summary (AWQ INT4
 * target whose per-group scales are kept; re-packing onto the same grid) and
 * "Assumptions & free parameters" (GPTQ INT4 drafter, group size 128; packing
 * rounds weights back onto the frozen per-group scales).  The pages give no
 * formula, layout or zero-point convention; the readings taken here are:
 *   - asymmetric grid: weight = (code - zero) * scale, zero stored as is
 *     (no "+1" offset), codes and zeros unsigned 4-bit;
 *   - groups are contiguous along K: group index of row k is k / g;
 *   - canonical packing: bits 4i..4i+3 of qweight[j][n] hold the code of
 *     row k = 8j+i (low nibble first); zeros pack 8 per uint32 along N:
 *     bits 4i..4i+3 of qzeros[gi][c] hold the zero of column n = 8c+i;
 *   - x is bfloat16, scales are IEEE binary16, both decoded exactly here
 *     from their bit fields; the sum is carried in fp64.
 *
 * Every product x*(q-z)*s is exact in fp64 (8 + 11 + 5 significant bits), so
 * the only rounding is in the fp64 accumulation, done in increasing k.
 *
 * Parity pins for every function live in tests/test_oracle.py (hand-worked
 * values, closed forms, exact rational brute force, library cross-checks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- number formats (IEEE 754 field definitions) ----------------------- */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double w4o_bf16_to_f64(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int f = b & 0x7F;
    double v;
    if (e == 0xFF)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -126 - 7);          /* subnormal: 0.f * 2^-126 */
    else
        v = ldexp(128.0 + f, e - 127 - 7);       /* 1.f * 2^(e-127) */
    return sign ? -v : v;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double w4o_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0x1F)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -14 - 10);
    else
        v = ldexp(1024.0 + f, e - 15 - 10);
    return sign ? -v : v;
}

/* Round an fp64 value to bfloat16, nearest with ties to even. */
uint16_t w4o_f64_to_bf16_rne(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7FC0;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);             /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1 + 127;            /* biased exponent of a normal result */
    if (E <= 0) {
        /* subnormal range: value = f * 2^-133, f an integer < 128 */
        double f = nearbyint(ldexp(a, 133));
        return (uint16_t)(sign | (uint16_t)f);  /* f == 128 encodes 2^-126 */
    }
    /* significand with 7 fraction bits: r in [128, 256] after rounding */
    double r = nearbyint(ldexp(a, 7 - (e - 1)));
    if (r == 256.0) {
        r = 128.0;
        E += 1;
    }
    if (E >= 0xFF)
        return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | (uint16_t)(E << 7) | (uint16_t)(r - 128.0));
}

/* ---- canonical packing ------------------------------------------------- */

/* codes[k*N + n] (0..15) -> qweight[(k/8)*N + n], nibble i = row 8j+i. */
void w4o_pack_codes(const uint8_t *codes, int K, int N, uint32_t *qweight)
{
    for (int j = 0; j < K / 8; ++j)
        for (int n = 0; n < N; ++n) {
            uint32_t w = 0;
            for (int i = 0; i < 8; ++i)
                w |= (uint32_t)(codes[(size_t)(8 * j + i) * N + n] & 0xF) << (4 * i);
            qweight[(size_t)j * N + n] = w;
        }
}

void w4o_unpack_codes(const uint32_t *qweight, int K, int N, uint8_t *codes)
{
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n)
            codes[(size_t)k * N + n] =
                (uint8_t)((qweight[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 0xF);
}

/* qzeros[gi*(N/8) + c], nibble i = column 8c+i  ->  zeros[gi*N + n]. */
void w4o_unpack_zeros(const uint32_t *qzeros, int G, int N, uint8_t *zeros)
{
    for (int gi = 0; gi < G; ++gi)
        for (int n = 0; n < N; ++n)
            zeros[(size_t)gi * N + n] =
                (uint8_t)((qzeros[(size_t)gi * (N / 8) + n / 8] >> (4 * (n % 8))) & 0xF);
}

void w4o_pack_zeros(const uint8_t *zeros, int G, int N, uint32_t *qzeros)
{
    for (int gi = 0; gi < G; ++gi)
        for (int c = 0; c < N / 8; ++c) {
            uint32_t w = 0;
            for (int i = 0; i < 8; ++i)
                w |= (uint32_t)(zeros[(size_t)gi * N + 8 * c + i] & 0xF) << (4 * i);
            qzeros[(size_t)gi * (N / 8) + c] = w;
        }
}

/* ---- dequantization ---------------------------------------------------- */

/* W[k*N + n] = (q[k][n] - z[k/g][n]) * s[k/g][n], exact in fp64. */
void w4o_dequant(const uint32_t *qweight, const uint16_t *scales, const uint32_t *qzeros,
                 int K, int N, int group, double *W)
{
    for (int k = 0; k < K; ++k) {
        int gi = k / group;
        for (int n = 0; n < N; ++n) {
            int q = (int)((qweight[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 0xF);
            int z = (int)((qzeros[(size_t)gi * (N / 8) + n / 8] >> (4 * (n % 8))) & 0xF);
            double s = w4o_f16_to_f64(scales[(size_t)gi * N + n]);
            W[(size_t)k * N + n] = (double)(q - z) * s;
        }
    }
}

/* ---- the GEMM: naive triple loop, m / k / n, fp64 accumulation --------- */

/*
 * y[m*N + n] for all m < M, n < N.  Work is split over (m, column chunk)
 * pairs; each output is still summed by one thread in increasing k, so the
 * result does not depend on the thread count.  nthreads <= 0: OpenMP default.
 */
void w4o_gemm(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
              const uint32_t *qzeros, int M, int N, int K, int group, double *y,
              int nthreads)
{
    const int G = K / group;
    /* unpack once: codes[K][N], zeros[G][N], scales as fp64 [G][N] */
    uint8_t *codes = (uint8_t *)malloc((size_t)K * N);
    uint8_t *zeros = (uint8_t *)malloc((size_t)G * N);
    double *sd = (double *)malloc(sizeof(double) * (size_t)G * N);
    w4o_unpack_codes(qweight, K, N, codes);
    w4o_unpack_zeros(qzeros, G, N, zeros);
    for (size_t i = 0; i < (size_t)G * N; ++i)
        sd[i] = w4o_f16_to_f64(scales[i]);

    const int CHUNK = 512;
    const int nchunks = (N + CHUNK - 1) / CHUNK;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic) collapse(2)
#endif
    for (int m = 0; m < M; ++m)
        for (int c = 0; c < nchunks; ++c) {
            int n0 = c * CHUNK, n1 = n0 + CHUNK < N ? n0 + CHUNK : N;
            double *yr = y + (size_t)m * N;
            for (int n = n0; n < n1; ++n)
                yr[n] = 0.0;
            for (int k = 0; k < K; ++k) {
                double xv = w4o_bf16_to_f64(x[(size_t)m * K + k]);
                int gi = k / group;
                const uint8_t *qr = codes + (size_t)k * N;
                const uint8_t *zr = zeros + (size_t)gi * N;
                const double *sr = sd + (size_t)gi * N;
                for (int n = n0; n < n1; ++n)
                    yr[n] += xv * ((double)((int)qr[n] - (int)zr[n]) * sr[n]);
            }
        }
    free(codes);
    free(zeros);
    free(sd);
}

/*
 * Sampled outputs: y_out[i] = y[ms[i]][ns[i]], each summed in increasing k
 * straight from the packed words (no full unpack), for problems too large
 * for the full triple loop.
 */
void w4o_gemm_elems(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                    const uint32_t *qzeros, int M, int N, int K, int group,
                    const int64_t *ms, const int64_t *ns, int64_t count, double *y_out,
                    int nthreads)
{
    (void)M;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < count; ++i) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int k = 0; k < K; ++k) {
            int gi = k / group;
            int q = (int)((qweight[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 0xF);
            int z = (int)((qzeros[(size_t)gi * (N / 8) + n / 8] >> (4 * (n % 8))) & 0xF);
            double s = w4o_f16_to_f64(scales[(size_t)gi * N + n]);
            acc += w4o_bf16_to_f64(x[(size_t)m * K + k]) * ((double)(q - z) * s);
        }
        y_out[i] = acc;
    }
}

/* ---- documented device layout of the packed weights -------------------- */

/*
 * The GPU library's pack call re-orders the canonical words into a tiled
 * device layout whose definition is part of the library's public header.
 * This is an independent rendering of that written definition, used only to
 * check the pack output bit for bit:
 *   column tiles of 128 (the last one W = N - 128*nb wide), K blocks of 128;
 *   tile nb starts at word 128*16*KB*nb, block kb of it at + kb*W*16;
 *   inside a block, word (c*W + t)*4 + j holds column n = 128*nb + t and
 *   rows k = 128*kb + 8*(4c + j) + r, r = 0..7;
 *   inside a word, nibble position p holds row offset r = 2p for p < 4 and
 *   r = 2(p-4)+1 for p >= 4.
 * K must be a multiple of 128 and N of 8.
 */
void w4o_device_layout(const uint32_t *qweight, int K, int N, uint32_t *out)
{
    const int KB = K / 128;
    const int NB = (N + 127) / 128;
    for (int nb = 0; nb < NB; ++nb) {
        int W = N - 128 * nb < 128 ? N - 128 * nb : 128;
        size_t tile = (size_t)128 * 16 * KB * nb;
        for (int kb = 0; kb < KB; ++kb) {
            size_t blk = tile + (size_t)kb * W * 16;
            for (int c = 0; c < 4; ++c)
                for (int t = 0; t < W; ++t)
                    for (int j = 0; j < 4; ++j) {
                        int n = 128 * nb + t;
                        int kw = 16 * kb + 4 * c + j;          /* canonical word row */
                        uint32_t w = qweight[(size_t)kw * N + n];
                        uint32_t d = 0;
                        for (int p = 0; p < 8; ++p) {
                            int r = p < 4 ? 2 * p : 2 * (p - 4) + 1;
                            d |= ((w >> (4 * r)) & 0xF) << (4 * p);
                        }
                        out[blk + (size_t)(c * W + t) * 4 + j] = d;
                    }
        }
    }
}

int w4o_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
