/*
 * Every binary32 bit pattern (2^32 of them) through the oracle's E4M3 encoder
 * (oracle/jetq_oracle.c: binary search over the ordered codes and comparison
 * with the exact midpoint of two neighbours) and through an independent
 * encoder written here on the bit pattern itself:
 *   NaN -> 0x7F; |v| >= 448 (and infinities) -> 448 with the sign;
 *   |v| < 2^-6: the subnormal grid of step 2^-9, code = nearest integer of
 *   |v| * 2^9 (ties to even; the product is exact), 8 meaning 2^-6 = 0x08;
 *   otherwise exponent E of v and its 23-bit mantissa rounded to 3 bits,
 *   ties to even, a carry bumping E; code = (E + 7) << 3 | mantissa.
 * The sign bit is kept (also for zero).  Exit status 0 and "mismatches=0"
 * when the two agree everywhere.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

uint8_t jo_e4m3_encode(double v);

static uint8_t enc_bits(uint32_t u)
{
    const uint8_t sign = (u >> 31) ? 0x80 : 0x00;
    const uint32_t a = u & 0x7FFFFFFFu;
    float f;
    if (a > 0x7F800000u)
        return 0x7F;
    memcpy(&f, &a, 4);
    if (f >= 448.0f)
        return (uint8_t)(sign | 0x7E);
    if (f < 0x1p-6f) {
        const float n = nearbyintf(f * 512.0f); /* default rounding: nearest, ties to even */
        return (uint8_t)(sign | (uint8_t)n);
    }
    {
        int e = (int)(a >> 23) - 127;
        uint32_t m = a & 0x7FFFFFu, q = m >> 20, rem = m & 0xFFFFFu;
        if (rem > 0x80000u || (rem == 0x80000u && (q & 1u)))
            ++q;
        if (q == 8u) {
            q = 0;
            ++e;
        }
        return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | (int)q));
    }
}

typedef struct {
    uint64_t lo, hi;
    long long bad;
    uint32_t first;
} job_t;

static void *run(void *arg)
{
    job_t *j = (job_t *)arg;
    for (uint64_t w = j->lo; w < j->hi; ++w) {
        const uint32_t u = (uint32_t)w;
        float f;
        memcpy(&f, &u, 4);
        if (jo_e4m3_encode((double)f) != enc_bits(u)) {
            if (j->bad == 0)
                j->first = u;
            j->bad++;
        }
    }
    return NULL;
}

int main(void)
{
    enum { T = 16 };
    pthread_t th[T];
    job_t jobs[T];
    long long bad = 0;
    const uint64_t total = 1ull << 32, per = total / T;
    for (int i = 0; i < T; ++i) {
        jobs[i].lo = per * (uint64_t)i;
        jobs[i].hi = i == T - 1 ? total : per * (uint64_t)(i + 1);
        jobs[i].bad = 0;
        pthread_create(&th[i], NULL, run, &jobs[i]);
    }
    for (int i = 0; i < T; ++i) {
        pthread_join(th[i], NULL);
        if (jobs[i].bad && !bad)
            printf("first mismatch 0x%08x\n", jobs[i].first);
        bad += jobs[i].bad;
    }
    printf("patterns=%llu mismatches=%lld\n", (unsigned long long)total, bad);
    return bad != 0;
}
