/* Seeded synthetic input generator shared by the tests, the benchmark and
 * the smoke check.  It holds none of the codec's arithmetic: it only draws
 * normal samples and outlier / zero-block choices and returns them as
 * binary32.  Conversion to bf16 happens outside (torch's own cast).
 *
 * Counter-based: every sample is a pure function of (seed, stream, index),
 * so any chunk of a huge vector can be generated alone and in parallel, and
 * the bytes do not depend on the thread count.
 *
 *  - SplitMix64 finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom
 *    number generators", OOPSLA 2014) applied to key + (counter+1) * golden
 *    gamma gives 64 uniform bits per counter.
 *  - Box-Muller (1958) in double turns two uniforms into two normals:
 *    element 2p takes r cos(t), element 2p+1 takes r sin(t).
 *  - An element (or a group of `outlier_group` consecutive elements, e.g. a
 *    matrix row) is an outlier with probability outlier_p, decided by its own
 *    uniform draw; outliers are multiplied by outlier_mult.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

static const uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GAMMA) ^ (stream * 0xD1B54A32D192ED03ull + 0x8CB92BA72F3D8DD7ull));
}

static inline uint64_t draw(uint64_t key, uint64_t counter) { return mix64(key + (counter + 1) * GAMMA); }

/* (0, 1] and [0, 1) uniforms with 53 random bits */
static inline double u_open0(uint64_t r) { return ((double)(r >> 11) + 1.0) * 0x1p-53; }
static inline double u_closed0(uint64_t r) { return (double)(r >> 11) * 0x1p-53; }

typedef struct {
    uint64_t key_z, key_o, offset, lo, hi, outlier_group, threshold;
    double sigma, mult;
    int use_outliers;
    float* out;
} job_t;

static void* run_job(void* arg) {
    job_t* J = (job_t*)arg;
    const double two_pi = 6.283185307179586476925286766559;
    for (uint64_t i = J->lo; i < J->hi;) {
        uint64_t g = J->offset + i;
        uint64_t p = g >> 1;
        double r = sqrt(-2.0 * log(u_open0(draw(J->key_z, 2 * p))));
        double t = two_pi * u_closed0(draw(J->key_z, 2 * p + 1));
        double z[2] = {r * cos(t), r * sin(t)};
        for (int h = (int)(g & 1); h < 2 && i < J->hi; ++h, ++i) {
            uint64_t gi = J->offset + i;
            double v = J->sigma * z[h];
            if (J->use_outliers && draw(J->key_o, gi / J->outlier_group) < J->threshold) v *= J->mult;
            J->out[i] = (float)v;
        }
    }
    return NULL;
}

/* out[i] = sample number (offset + i) of stream (seed, stream), i < n. */
void gen_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, double sigma,
                    double outlier_p, double outlier_mult, uint64_t outlier_group, float* out,
                    int nthreads) {
    if (n == 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
    job_t jobs[256];
    pthread_t th[256];
    uint64_t per = (n + (uint64_t)nthreads - 1) / (uint64_t)nthreads;
    per += per & 1; /* keep Box-Muller pairs inside one thread */
    uint64_t threshold = 0;
    int use_outliers = outlier_p > 0.0 && outlier_mult != 1.0;
    if (use_outliers) threshold = outlier_p >= 1.0 ? UINT64_MAX : (uint64_t)(outlier_p * 0x1p64);
    int created[256] = {0};
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        uint64_t lo = (uint64_t)t * per, hi = lo + per < n ? lo + per : n;
        if (lo >= n) break;
        job_t j = {stream_key(seed, 2 * stream), stream_key(seed, 2 * stream + 1), offset, lo, hi,
                   outlier_group ? outlier_group : 1, threshold, sigma, outlier_mult, use_outliers, out};
        jobs[t] = j;
        used = t + 1;
    }
    for (int t = 1; t < used; ++t) created[t] = pthread_create(&th[t], NULL, run_job, &jobs[t]) == 0;
    run_job(&jobs[0]);
    for (int t = 1; t < used; ++t) {
        if (created[t]) pthread_join(th[t], NULL);
        else run_job(&jobs[t]);
    }
}

/* `count` distinct indices in [0, range), in draw order. */
void gen_distinct_indices(uint64_t seed, uint64_t stream, uint64_t count, uint64_t range, uint64_t* out) {
    uint64_t key = stream_key(seed, 0x5EEDull + stream);
    uint64_t got = 0;
    for (uint64_t c = 0; got < count && got < range; ++c) {
        uint64_t v = draw(key, c) % range;
        int dup = 0;
        for (uint64_t j = 0; j < got; ++j) dup |= out[j] == v;
        if (!dup) out[got++] = v;
    }
}
