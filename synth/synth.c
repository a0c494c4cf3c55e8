/*
 * Seeded normal samples as 16-bit storage patterns (bf16 / fp16).
 *
 * Counter based: element i of stream `seed` is a function of (seed, i) only,
 * so slices can be drawn independently and in parallel.
 *
 *   u(n)  = ((mix64(seed + (n + 1) * 0x9E3779B97F4A7C15) >> 11) + 1) * 2^-53
 *           (SplitMix64, Steele, Lea & Flood, OOPSLA 2014; u in (0, 1])
 *   z(i)  = sqrt(-2 ln u(2i)) * cos(2 pi u(2i+1))   (Box-Muller, cosine branch)
 *   v(i)  = mean + std * z(i)
 *
 * Storage: bf16 keeps the top 16 bits of (float)v (round toward zero); fp16 is
 * the compiler's float -> _Float16 conversion.  These are sampling choices,
 * nothing more.  libm's log/cos may differ in the last bit between machines,
 * so values are reproducible on one machine; nothing stored depends on them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline double uniform01(uint64_t seed, uint64_t n) {
    uint64_t o = mix64(seed + (n + 1) * 0x9E3779B97F4A7C15ull);
    return (double)((o >> 11) + 1) * 0x1.0p-53;
}

static inline uint16_t store16(double v, int dtype) {
    float f = (float)v;
    if (dtype == 0) {
        uint32_t u;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16);
    }
    _Float16 h = (_Float16)f;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

typedef struct {
    uint16_t *out;
    uint64_t seed, begin, end;
    double mean, std;
    int dtype;
} job_t;

static void *run(void *arg) {
    const job_t *j = (const job_t *)arg;
    const double two_pi = 6.283185307179586476925286766559;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        double u1 = uniform01(j->seed, 2 * i);
        double u2 = uniform01(j->seed, 2 * i + 1);
        double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        j->out[i - j->begin] = store16(j->mean + j->std * z, j->dtype);
    }
    return 0;
}

/* Fill out[0..n) with elements [first, first + n) of stream `seed`.
 * dtype: 0 = bf16, 1 = fp16.  threads is clamped to [1, 64].  Returns 0. */
int synth_normal16(uint16_t *out, uint64_t n, uint64_t first, uint64_t seed,
                   double mean, double std, int dtype, int threads) {
    if (threads < 1) threads = 1;
    if (threads > 64) threads = 64;
    if (n < (1u << 16)) threads = 1;
    pthread_t tid[64];
    int created[64] = {0};
    job_t jobs[64];
    uint64_t per = (n + (uint64_t)threads - 1) / (uint64_t)threads;
    for (int t = 0; t < threads; ++t) {
        uint64_t b = (uint64_t)t * per, e = b + per;
        if (b >= n) break;
        if (e > n) e = n;
        jobs[t] = (job_t){out + b, seed, first + b, first + e, mean, std, dtype};
        if (e == n || pthread_create(&tid[t], 0, run, &jobs[t]) != 0)
            run(&jobs[t]);
        else
            created[t] = 1;
    }
    for (int t = 0; t < threads; ++t)
        if (created[t]) pthread_join(tid[t], 0);
    return 0;
}
