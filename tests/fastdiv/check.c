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
 * exhaustion is out of reach) for the two-step form the ring hop uses:
 * Markstein's theorem already proves it exact; the sample is a cross-check.
 *
 * Build: cc -O2 -ffp-contract=off -pthread check.c -lm
 *   check bf16 [threads]      exhaustive one-step check (2^30 pairs)
 *   check f32 [count] [seed]  random two-step check
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

int main(int argc, char** argv) {
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
