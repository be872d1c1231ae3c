/* Exhaustive proof, at unit scale, of the quotient sequence the blockwise
 * quantizer uses instead of a per-element IEEE division.
 *
 * For a block scale s and an element x the codec needs q = RN(x / s).
 * The kernel computes, with y = RN(1/s) once per block:
 *     q0 = RN(x * y)
 *     r  = RN(q0 * s - x)          (one fused multiply-add)
 *     q1 = RN(q0 - r * y)          (one fused multiply-add)
 * which is Markstein's correction step (P. Markstein, "Computation of
 * elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
 * Dev. 34(1), 1990; also "IA-64 and Elementary Functions", 2000).
 *
 * The bf16 element has an 8-bit significand, so at unit scale
 * (x in [1, 2) with 128 significands, s in [1, 2) with 2^23 significands)
 * there are 2^30 pairs; this program checks q1 == RN(x / s) for all of
 * them.  Every operation of the sequence and the reference division commute
 * with scaling x and s by powers of two while all intermediates stay
 * normal, which extends the result to every exponent the kernel admits to
 * this path (the conditions are stated next to the kernel).
 *
 * A second mode samples binary32 dividends (24-bit significands, where
 * exhaustion over every divisor is out of reach) for the two-step form the
 * ring hop uses for its elements: Markstein's theorem already proves it
 * exact; the sample is a cross-check.
 *
 * A third mode covers the block scale RN(amax / Fmax).  There the divisor is
 * one of two constants, Fmax = 448 (e4m3) or 57344 (e5m2), with the constant
 * reciprocal y = RN(1 / Fmax), and the dividend amax is a bf16 value in the
 * quantizer but the binary32 amax of the fp32 sum y in the ring hop.  With
 * the divisor fixed, every binary32 dividend of a binade is enumerable: the
 * mode checks the one-step sequence against the IEEE quotient for all 2^23
 * significands in each of several binades (from 2^-78, the smallest amax the
 * kernel sends down this path, up to 2^127) and for both constants.
 *
 * Build: cc -O2 -ffp-contract=off -pthread check.c -lm
 *   check bf16 [threads]      exhaustive one-step check (2^30 pairs)
 *   check f32 [count] [seed]  random two-step check
 *   check scale               exhaustive one-step check of RN(a / Fmax) for
 *                             binary32 a, Fmax in {448, 57344}
 * Prints the number of mismatching pairs and exits 0 only if it is 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

typedef struct { uint32_t s_lo, s_hi; uint64_t bad; uint64_t checked; } job_t;

static void* run(void* arg) {
    job_t* J = (job_t*)arg;
    for (uint32_t sm = J->s_lo; sm < J->s_hi; ++sm) {
        const float s = f_of(0x3F800000u | sm);            /* s in [1, 2) */
        const float y = 1.0f / s;                            /* RN(1/s) */
        for (uint32_t xm = 0; xm < 128; ++xm) {
            const float x = f_of(0x3F800000u | (xm << 16));  /* bf16 significand, x in [1, 2) */
            const float q0 = x * y;
            const float r = fmaf(q0, s, -x);
            const float q1 = fmaf(-r, y, q0);
            const float ref = x / s;
            J->bad += u_of(q1) != u_of(ref);
        }
        J->checked += 128;
    }
    return NULL;
}

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static int random_f32(uint64_t count, uint64_t seed) {
    uint64_t bad = 0;
    for (uint64_t i = 0; i < count; ++i) {
        const uint64_t r = mix64(seed + (i + 1) * 0x9E3779B97F4A7C15ull);
        const float x = f_of(0x3F800000u | (uint32_t)(r & 0x7FFFFF));
        const float s = f_of(0x3F800000u | (uint32_t)((r >> 23) & 0x7FFFFF));
        const float y = 1.0f / s;
        float q = x * y;
        for (int c = 0; c < 2; ++c) {
            const float e = fmaf(q, s, -x);
            q = fmaf(-e, y, q);
        }
        bad += u_of(q) != u_of(x / s);
    }
    printf("checked %llu pairs, mismatches %llu\n", (unsigned long long)count, (unsigned long long)bad);
    return bad != 0;
}

/* One step from the constant reciprocal, every binary32 significand of the
 * binades 2^e, e in the list, for both format maxima. */
static int scale_constants(void) {
    static const float dmax[2] = {448.0f, 57344.0f};
    static const int binades[] = {-78, -77, -40, -1, 0, 1, 17, 60, 126, 127};
    const int nbin = (int)(sizeof binades / sizeof binades[0]);
    uint64_t bad = 0, checked = 0;
    for (int f = 0; f < 2; ++f) {
        const float d = dmax[f];
        const float y = 1.0f / d;
        for (int b = 0; b < nbin; ++b) {
            const uint32_t ebits = (uint32_t)(binades[b] + 127) << 23;
            for (uint32_t m = 0; m < (1u << 23); ++m) {
                const float a = f_of(ebits | m);
                const float q0 = a * y;
                const float r = fmaf(q0, d, -a);
                const float q1 = fmaf(-r, y, q0);
                bad += u_of(q1) != u_of(a / d);
            }
            checked += 1u << 23;
        }
    }
    printf("checked %llu dividends, mismatches %llu\n", (unsigned long long)checked, (unsigned long long)bad);
    return bad != 0;
}

int main(int argc, char** argv) {
    if (argc > 1 && strcmp(argv[1], "scale") == 0) return scale_constants();
    if (argc > 1 && strcmp(argv[1], "f32") == 0)
        return random_f32(argc > 2 ? strtoull(argv[2], 0, 0) : 100000000ull, argc > 3 ? strtoull(argv[3], 0, 0) : 1);
    int nt = argc > 2 ? atoi(argv[2]) : 8;
    uint32_t lo = 0;
    uint32_t cnt = 1u << 23;
    if (nt < 1) nt = 1;
    if (nt > 256) nt = 256;
    pthread_t th[256];
    job_t jobs[256];
    uint32_t per = (cnt + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
        uint32_t a = lo + (uint32_t)t * per, b = a + per;
        if (b > lo + cnt) b = lo + cnt;
        if (a > b) a = b;
        jobs[t].s_lo = a; jobs[t].s_hi = b; jobs[t].bad = 0; jobs[t].checked = 0;
        pthread_create(&th[t], NULL, run, &jobs[t]);
    }
    uint64_t bad = 0, checked = 0;
    for (int t = 0; t < nt; ++t) { pthread_join(th[t], NULL); bad += jobs[t].bad; checked += jobs[t].checked; }
    printf("checked %llu pairs, mismatches %llu\n", (unsigned long long)checked, (unsigned long long)bad);
    return bad != 0;
}
