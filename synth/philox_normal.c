/*
 * Seeded synthetic inputs for the multi-LoRA linear layer.
 *
 * This file holds no arithmetic of the layer itself: it only turns
 * (seed, tensor id, element index) into random bits and normal deviates.
 * Both the fp64 oracle and the CUDA path receive the values it writes.
 *
 * Generator: Philox4x64-10, the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11):
 * ten rounds of two 64x64->128 multiplies, with a Weyl key schedule.
 * Element e of a tensor uses counter (e / 4, 0, 0, 0), key (seed, tensor id),
 * and output word e % 4, so any sub-range of a tensor is reproducible alone.
 *
 * Normals: the Box-Muller transform on the word pair (2m, 2m+1) of a block:
 *   u1 = ((w[2m] >> 11) + 1) * 2^-53 in (0, 1], u2 = (w[2m+1] >> 11) * 2^-53,
 *   rad = sqrt(-2 ln u1), z(2m) = rad cos(2 pi u2), z(2m+1) = rad sin(2 pi u2).
 * bf16 values are std * z rounded to fp32 and then to bf16, both with
 * round-to-nearest-even.
 *
 * Compiled with -ffp-contract=off so that no FMA contraction changes the
 * values between hosts.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2E7470EE14C6C93ULL
#define PHILOX_M1 0xCA5A826395121157ULL
#define PHILOX_W0 0x9E3779B97F4A7C15ULL
#define PHILOX_W1 0xBB67AE8584CAA73BULL

static inline void mul_hi_lo(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
    unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(p >> 64);
    *lo = (uint64_t)p;
}

void synth_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
    uint64_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t hi0, lo0, hi1, lo1;
        mul_hi_lo(PHILOX_M0, c0, &hi0, &lo0);
        mul_hi_lo(PHILOX_M1, c2, &hi1, &lo1);
        uint64_t n0 = hi1 ^ c1 ^ k0;
        uint64_t n1 = lo1;
        uint64_t n2 = hi0 ^ c3 ^ k1;
        uint64_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u) {          /* inf or nan: truncate, keep nan quiet */
        uint16_t h = (uint16_t)(u >> 16);
        if (u & 0x007FFFFFu) h |= 0x0040u;
        return h;
    }
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static double normal_at(uint64_t seed, uint64_t tensor_id, uint64_t e) {
    const uint64_t ctr[4] = {e >> 2, 0, 0, 0};
    const uint64_t key[2] = {seed, tensor_id};
    uint64_t w[4];
    synth_philox4x64_10(ctr, key, w);
    unsigned pair = (unsigned)((e & 3u) >> 1);
    double u1 = (double)((w[2 * pair] >> 11) + 1) * 0x1p-53;
    double u2 = (double)(w[2 * pair + 1] >> 11) * 0x1p-53;
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586476925286766559 * u2;
    return (e & 1u) ? rad * sin(ang) : rad * cos(ang);
}

typedef struct {
    uint64_t seed, tensor_id, first, begin, end;
    double stddev;
    uint16_t* out_bf16;
    double* out_f64;
    uint64_t* out_u64;
} job_t;

static void* run_job(void* arg) {
    job_t* j = (job_t*)arg;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        uint64_t e = j->first + i;
        if (j->out_u64) {
            const uint64_t ctr[4] = {e >> 2, 0, 0, 0};
            const uint64_t key[2] = {j->seed, j->tensor_id};
            uint64_t w[4];
            synth_philox4x64_10(ctr, key, w);
            j->out_u64[i] = w[e & 3u];
        } else {
            double v = j->stddev * normal_at(j->seed, j->tensor_id, e);
            if (j->out_f64) j->out_f64[i] = v;
            if (j->out_bf16) j->out_bf16[i] = f32_to_bf16_rne((float)v);
        }
    }
    return 0;
}

static void run_parallel(job_t base, uint64_t n, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > n / 4096 + 1) nthreads = (int)(n / 4096 + 1);
    pthread_t tid[256];
    int joined[256];
    job_t jobs[256];
    uint64_t chunk = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].begin = (uint64_t)t * chunk < n ? (uint64_t)t * chunk : n;
        jobs[t].end = jobs[t].begin + chunk < n ? jobs[t].begin + chunk : n;
        joined[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], 0, run_job, &jobs[t]) == 0)
            joined[t] = 1;
        else
            run_job(&jobs[t]);
    }
    run_job(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (joined[t]) pthread_join(tid[t], 0);
}

/* n normal deviates * stddev, elements [first, first + n), rounded to bf16 bits. */
void synth_normal_bf16(uint64_t seed, uint64_t tensor_id, uint64_t first, uint64_t n,
                       double stddev, uint16_t* out, int nthreads) {
    job_t b = {seed, tensor_id, first, 0, 0, stddev, out, 0, 0};
    run_parallel(b, n, nthreads);
}

/* Same deviates, unrounded (fp64); used to test the transform itself. */
void synth_normal_f64(uint64_t seed, uint64_t tensor_id, uint64_t first, uint64_t n,
                      double stddev, double* out, int nthreads) {
    job_t b = {seed, tensor_id, first, 0, 0, stddev, 0, out, 0};
    run_parallel(b, n, nthreads);
}

/* Raw 64-bit words, for discrete draws made by the Python recipes. */
void synth_u64(uint64_t seed, uint64_t tensor_id, uint64_t first, uint64_t n,
               uint64_t* out, int nthreads) {
    job_t b = {seed, tensor_id, first, 0, 0, 0.0, 0, 0, out};
    run_parallel(b, n, nthreads);
}
