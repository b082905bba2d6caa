/*
 * qlinear_oracle.c -- fp64 reference for the GGUF weight-only quantized linear layer.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load this file's library. The CUDA product path never links, includes or calls
 * it, and this file shares no code, header, table or helper with that path.
 *
 * What it computes (the plain definition, no blocking or reordering):
 *     y[m, n] = sum_{k < K} double(x[m, k]) * w[n, k]
 * where w[n, k] is the exact real value of the dequantised weight: element k % 256 of
 * superblock k / 256 of row n of the packed matrix. Every w is exact in fp64 (an fp16
 * value times small integers), so the only rounding is that of the fp64 sum.
 *
 * Sources (page titles as printed):
 *  - block sizes 144/176/210/136 bytes per 256 weights: tinygrad/llm/gguf.py, the
 *    _GGML_QUANT table (compare master..kimi_slop / more_kernelcount...llm_262k_minimal diff).
 *  - Q4_K = Q5_K without the high-bit array, same d/dmin/scale layout, qs at word 4:
 *    commit log of explicit-dev, commit "custom kernels: Q4_K support (ggml type 12)".
 *  - d at bytes 0..1 (Q4_K/Q5_K/IQ4_XS), dmin at bytes 2..3 (Q4_K/Q5_K), d in the last two
 *    bytes (Q6_K): test/unit/test_llm_quant_cpu.py, random_packed().
 *  - IQ4_XS codebook and nibble order (low nibbles of a 16-byte group first, then high
 *    nibbles): test/unit/test_llm_quant_cpu.py, test_unpack_lut_dot_uop.
 *  - Closed forms w = d*sc*q - dmin*m (K-quants), w = d*sc*(q-32) (Q6_K),
 *    w = d*(ls-32)*codebook[q] (IQ4_XS): the hot-path statement of this project.
 *  - Bit placement inside a block beyond the facts above is not printed on the pages; it
 *    follows the GGUF on-disk layout (the pages load real GGUF files), written out below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

enum { OR_Q4_K = 12, OR_Q5_K = 13, OR_Q6_K = 14, OR_IQ4_XS = 23 };

int oracle_block_bytes(int type) {
    switch (type) {
    case OR_Q4_K: return 144;
    case OR_Q5_K: return 176;
    case OR_Q6_K: return 210;
    case OR_IQ4_XS: return 136;
    default: return -1;
    }
}

/* IEEE 754 binary16 -> double, from the format's definition:
 * sign bit 15, exponent bits 10..14 (bias 15), fraction bits 0..9. */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)f, -24);             /* zero / subnormal: f * 2^-24 */
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp((double)(1024 + f), e - 25);         /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double le_half(const uint8_t *p) { return oracle_half_to_double((uint16_t)(p[0] | (p[1] << 8))); }

/* 6-bit (scale, min) of sub-block j (0..7) from the 12-byte packed field S of Q4_K/Q5_K.
 * Sub-blocks 0..3: low 6 bits of S[j] and S[j+4]. Sub-blocks 4..7: low 4 bits from the
 * nibbles of S[j+4], high 2 bits from the top bits of S[j-4] (scale) and S[j] (min). */
static void kq_scale_min(const uint8_t *S, int j, int *sc, int *m) {
    if (j < 4) {
        *sc = S[j] & 63;
        *m = S[j + 4] & 63;
    } else {
        *sc = (S[j + 4] & 15) | ((S[j - 4] >> 6) << 4);
        *m = (S[j + 4] >> 4) | ((S[j] >> 6) << 4);
    }
}

static const int iq4_codebook[16] = {-127, -104, -83, -65, -49, -35, -22, -10,
                                     1,    13,   25,  38,  53,  69,  89,  113};

/* Exact value of weight i (0..255) of one superblock. */
static double weight_of(int type, const uint8_t *b, int i) {
    if (type == OR_Q4_K || type == OR_Q5_K) {
        const double d = le_half(b), dmin = le_half(b + 2);
        const uint8_t *S = b + 4;
        const uint8_t *qh = b + 16;                                   /* Q5_K only */
        const uint8_t *qs = b + (type == OR_Q4_K ? 16 : 48);
        int sc, m;
        kq_scale_min(S, i / 32, &sc, &m);
        const uint8_t byte = qs[32 * (i / 64) + i % 32];
        int q = (i % 64 < 32) ? (byte & 15) : (byte >> 4);
        if (type == OR_Q5_K) q += 16 * ((qh[i % 32] >> (i / 32)) & 1);
        return d * sc * q - dmin * m;
    }
    if (type == OR_Q6_K) {
        const uint8_t *ql = b, *qh = b + 128;
        const int8_t *sc = (const int8_t *)(b + 192);
        const double d = le_half(b + 208);
        const int h = i / 128, r = i % 128, t = r / 32, l = r % 32;
        const uint8_t lbyte = ql[64 * h + 32 * (t % 2) + l];
        const int lo = (t < 2) ? (lbyte & 15) : (lbyte >> 4);
        const int hi = (qh[32 * h + l] >> (2 * t)) & 3;
        const int q = lo | (hi << 4);
        return d * sc[i / 16] * (q - 32);
    }
    if (type == OR_IQ4_XS) {
        const double d = le_half(b);
        const int scales_h = b[2] | (b[3] << 8);
        const uint8_t *scales_l = b + 4, *qs = b + 8;
        const int j = i / 32, r = i % 32;
        const int ls = ((scales_l[j / 2] >> (4 * (j % 2))) & 15) | (((scales_h >> (2 * j)) & 3) << 4);
        const uint8_t byte = qs[16 * j + r % 16];
        const int nib = (r < 16) ? (byte & 15) : (byte >> 4);
        return d * (ls - 32) * iq4_codebook[nib];
    }
    return NAN;
}

/* Dequantise rows [0, N) of a packed matrix into w[N][K] (fp64). Returns 0, or -1 on a bad
 * type, -2 on a bad shape. */
int oracle_dequant_f64(int type, const uint8_t *W, int64_t N, int64_t K, double *w) {
    const int bb = oracle_block_bytes(type);
    if (bb < 0) return -1;
    if (N < 0 || K < 0 || K % 256) return -2;
    const int64_t nsb = K / 256;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = W + (n * nsb + sb) * bb;
            for (int i = 0; i < 256; ++i) w[n * K + sb * 256 + i] = weight_of(type, blk, i);
        }
    return 0;
}

typedef struct {
    int type;
    const uint8_t *W;
    int64_t n0, n1, K, M;
    const uint16_t *x;
    double *y;
    int64_t N;
} job_t;

static void *run_rows(void *arg) {
    const job_t *j = (const job_t *)arg;
    const int bb = oracle_block_bytes(j->type);
    const int64_t nsb = j->K / 256;
    double *wrow = (double *)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
    if (!wrow) return (void *)1;
    for (int64_t n = j->n0; n < j->n1; ++n) {
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = j->W + (n * nsb + sb) * bb;
            for (int i = 0; i < 256; ++i) wrow[sb * 256 + i] = weight_of(j->type, blk, i);
        }
        for (int64_t m = 0; m < j->M; ++m) {
            const uint16_t *xr = j->x + m * j->K;
            double acc = 0.0;
            for (int64_t k = 0; k < j->K; ++k) acc += oracle_half_to_double(xr[k]) * wrow[k];
            j->y[m * j->N + n] = acc;
        }
    }
    free(wrow);
    return NULL;
}

/* y[M][N] = x[M][K] . dequant(W)[N][K]^T in fp64, summed in increasing k.
 * x holds IEEE binary16 bit patterns, row-major. Rows of W are split over n_threads
 * POSIX threads (each row's sum is computed by one thread, so the result does not depend
 * on the thread count). Returns 0, -1 bad type, -2 bad shape, -3 out of memory. */
int oracle_qlinear_f64(int type, const uint8_t *W, int64_t N, int64_t K, const uint16_t *x,
                       int64_t M, double *y, int n_threads) {
    if (oracle_block_bytes(type) < 0) return -1;
    if (N < 0 || M < 0 || K < 0 || K % 256) return -2;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > N) n_threads = (int)(N > 0 ? N : 1);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)n_threads);
    if (!tid || !jobs) { free(tid); free(jobs); return -3; }
    int rc = 0;
    char *joined = (char *)calloc((size_t)n_threads, 1);   /* 1 = ran inline, nothing to join */
    if (!joined) { free(tid); free(jobs); return -3; }
    for (int t = 0; t < n_threads; ++t) {
        jobs[t] = (job_t){type, W, N * t / n_threads, N * (t + 1) / n_threads, K, M, x, y, N};
        /* the last chunk, and any chunk whose thread cannot be started, runs on this thread */
        if (t == n_threads - 1 || pthread_create(&tid[t], NULL, run_rows, &jobs[t]) != 0) {
            joined[t] = 1;
            if (run_rows(&jobs[t]) != NULL) rc = -3;
        }
    }
    for (int t = 0; t < n_threads; ++t) {
        if (joined[t]) continue;
        void *ret = NULL;
        pthread_join(tid[t], &ret);
        if (ret != NULL) rc = -3;
    }
    free(joined);
    free(tid);
    free(jobs);
    return rc;
}
