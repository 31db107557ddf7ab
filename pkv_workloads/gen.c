/*
 * Seeded synthetic inputs for the paged decode-attention workloads.
 *
 * This file holds random-number generation only: no allocator, append or
 * attention arithmetic.  Both the CUDA path and the CPU oracle are fed the
 * bytes it produces.
 *
 * Generator: splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; the public-domain reference by Vigna).
 * The state advances by the golden-ratio increment 0x9E3779B97F4A7C15 and each
 * state is passed through the variant-13 finaliser.  Because the state after
 * i+1 steps is seed + (i+1)*increment, the i-th output can be computed
 * directly, so the draws are counter-based and can be generated in parallel.
 *
 * Normals: Box-Muller (cosine branch) on two consecutive 53-bit uniforms,
 * rounded to fp32 (round-to-nearest) and then to bf16 (round-to-nearest-even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static const uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* i-th output (0-based) of the splitmix64 stream whose initial state is `seed`. */
uint64_t wl_splitmix64_at(uint64_t seed, uint64_t i) { return mix64(seed + (i + 1) * kGamma); }

/* uniform in (0, 1]: 53 random bits, shifted away from zero so log() is finite */
static inline double unit_open0(uint64_t u) { return ((double)(u >> 11) + 1.0) * (1.0 / 9007199254740992.0); }

static inline double normal_at(uint64_t seed, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = unit_open0(wl_splitmix64_at(seed, 2 * i));
    double u2 = unit_open0(wl_splitmix64_at(seed, 2 * i + 1));
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7f800000u) == 0x7f800000u) return (uint16_t)((x >> 16) | ((x & 0xffff) ? 0x40 : 0));
    uint32_t lsb = (x >> 16) & 1u;
    x += 0x7fffu + lsb;
    return (uint16_t)(x >> 16);
}

double wl_normal_at(uint64_t seed, uint64_t i) { return normal_at(seed, i); }

typedef struct {
    uint64_t seed, offset, begin, end;
    double mean, std;
    uint16_t* out;
} job_t;

static void* normal_job(void* arg) {
    job_t* j = (job_t*)arg;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        double z = j->mean + j->std * normal_at(j->seed, j->offset + i);
        j->out[i] = f32_to_bf16_rne((float)z);
    }
    return 0;
}

/* out[i] = bf16(mean + std * N_{offset+i}) for i in [0, n), on `threads` threads. */
void wl_normal_bf16(uint64_t seed, uint64_t offset, uint64_t n, double mean, double std, uint16_t* out,
                    int threads) {
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n < (uint64_t)threads * 65536u) threads = 1;
    pthread_t tid[256];
    job_t jobs[256];
    for (int t = 0; t < threads; ++t) {
        jobs[t].seed = seed;
        jobs[t].offset = offset;
        jobs[t].begin = n * (uint64_t)t / (uint64_t)threads;
        jobs[t].end = n * (uint64_t)(t + 1) / (uint64_t)threads;
        jobs[t].mean = mean;
        jobs[t].std = std;
        jobs[t].out = out;
    }
    if (threads == 1) {
        normal_job(&jobs[0]);
        return;
    }
    for (int t = 0; t < threads; ++t) pthread_create(&tid[t], 0, normal_job, &jobs[t]);
    for (int t = 0; t < threads; ++t) pthread_join(tid[t], 0);
}
