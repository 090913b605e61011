/*
 * Seeded synthetic inputs for the BFP MoE decode path.
 *
 * This module only draws numbers. It holds none of the block-floating-point
 * arithmetic: no exponent, rounding or packing logic lives here. Both the
 * oracle side and the CUDA side of the tests (and the benchmark) take their
 * inputs from it, so that the two sides see the same fp32 values.
 *
 * Generator: Philox4x32-10, the counter-based generator published by Salmon,
 * Moraes, Dror and Shaw ("Parallel random numbers: as easy as 1, 2, 3",
 * SC'11). Key = the 64-bit seed, counter = (block index, 64-bit stream id).
 * Every value is a pure function of (seed, stream, index), so any slice of
 * any matrix can be regenerated alone and threads can split a range freely.
 *
 * Normal deviates use the Box-Muller transform (in fp32) on the four 32-bit
 * words of one Philox block: (w0, w1) -> two deviates, (w2, w3) -> two deviates.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static void philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static void philox_block(uint64_t seed, uint64_t stream, uint64_t block, uint32_t out[4]) {
    uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), (uint32_t)stream, (uint32_t)(stream >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    philox4x32_10(ctr, key, out);
}

/* (0, 1): never 0, so log() is finite. 24 significant bits, as an fp32 deviate needs. */
static float u01_open(uint32_t w) { return ((float)(w >> 8) + 0.5f) * (1.0f / 16777216.0f); }

static void normal_block(uint64_t seed, uint64_t stream, uint64_t block, double z[4]) {
    uint32_t w[4];
    philox_block(seed, stream, block, w);
    const float two_pi = 6.28318530717958647692f;
    for (int p = 0; p < 2; ++p) {
        float u1 = u01_open(w[2 * p]), u2 = u01_open(w[2 * p + 1]);
        float r = sqrtf(-2.0f * logf(u1));
        float a = two_pi * u2;
        z[2 * p] = (double)(r * cosf(a));
        z[2 * p + 1] = (double)(r * sinf(a));
    }
}

typedef struct {
    uint64_t seed, stream, offset;
    int64_t begin, end; /* range of output indices handled by this thread */
    double mean, std;
    float *out_f;
    uint32_t *out_u;
} job_t;

static void normal_range(const job_t *j) {
    int64_t i = j->begin;
    while (i < j->end) {
        uint64_t g = j->offset + (uint64_t)i; /* global value index */
        uint64_t blk = g >> 2;
        int lane = (int)(g & 3);
        double z[4];
        normal_block(j->seed, j->stream, blk, z);
        for (; lane < 4 && i < j->end; ++lane, ++i) j->out_f[i] = (float)(j->mean + j->std * z[lane]);
    }
}

static void bits_range(const job_t *j) {
    int64_t i = j->begin;
    while (i < j->end) {
        uint64_t g = j->offset + (uint64_t)i;
        uint64_t blk = g >> 2;
        int lane = (int)(g & 3);
        uint32_t w[4];
        philox_block(j->seed, j->stream, blk, w);
        for (; lane < 4 && i < j->end; ++lane, ++i) j->out_u[i] = w[lane];
    }
}

static void *normal_thread(void *p) { normal_range((const job_t *)p); return NULL; }
static void *bits_thread(void *p) { bits_range((const job_t *)p); return NULL; }

static int run_jobs(job_t base, int64_t n, int nthreads, void *(*fn)(void *)) {
    if (n <= 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n / 4096 + 1) nthreads = (int)(n / 4096 + 1);
    job_t jobs[256];
    pthread_t tids[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].begin = n * t / nthreads;
        jobs[t].end = n * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, fn, &jobs[t]) != 0) break;
        started = t;
    }
    /* Any job whose thread did not start runs here, in order. */
    fn(&jobs[0]);
    for (int t = started + 1; t < nthreads; ++t) fn(&jobs[t]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    return 0;
}

/* out[i] = mean + std * N(0,1) deviate number (offset + i) of stream (seed, stream). */
int synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double mean, double std,
                     float *out, int nthreads) {
    if (n < 0 || (n > 0 && out == NULL)) return -1;
    job_t b = {seed, stream, offset, 0, 0, mean, std, out, NULL};
    return run_jobs(b, n, nthreads, normal_thread);
}

/* out[i] = raw 32-bit Philox word number (offset + i) of stream (seed, stream). */
int synth_bits_u32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint32_t *out, int nthreads) {
    if (n < 0 || (n > 0 && out == NULL)) return -1;
    job_t b = {seed, stream, offset, 0, 0, 0.0, 0.0, NULL, out};
    return run_jobs(b, n, nthreads, bits_thread);
}

/* Single Philox4x32-10 block, exposed so tests can check it against the published known-answer vectors. */
void synth_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) { philox4x32_10(ctr, key, out); }
