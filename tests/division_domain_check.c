/*
 * Exhaustive check of the quantizer's division scheme over its whole input
 * domain: every finite BF16 value x and every finite positive BF16 group
 * maximum a >= |x|, with S = fl32(a / 448).
 *
 * The CUDA quantizers replace the per-element IEEE division x / S by
 *   r = RN(1/S), q0 = RN(x*r), e = RN(x - S*q0) (exact, one FMA),
 *   q1 = RN(q0 + e*r), sign of a zero result taken from x
 * (Markstein's one-step residual correction), and use x / S itself when
 * S < 2^-96.  This program counts the pairs where that differs from IEEE
 * x / S in a way that can change the E4M3 code: a different binary32 value
 * when |x/S| >= 2^-12, or a different sign below that (every E4M3 code of a
 * value under 2^-11 is a signed zero).  Exit status 0 means no pair differs.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static float scheme(float x, float s, float r)
{
    float q0, e, q1;
    if (s < 0x1p-96f)
        return x / s;
    q0 = x * r;
    e = fmaf(-q0, s, x);
    q1 = fmaf(e, r, q0);
    return copysignf(q1, x);
}

typedef struct {
    int lo, hi;
    long long bad, pairs;
} job_t;

static void *run(void *arg)
{
    job_t *j = (job_t *)arg;
    for (int ah = j->lo; ah < j->hi; ++ah) {
        float a = bf16((uint16_t)ah);
        if (!(a > 0.0f) || isinf(a))
            continue;
        float s = a / 448.0f, r = 1.0f / s;
        for (int xh = 0; xh < 0x10000; ++xh) {
            float x = bf16((uint16_t)xh);
            if (isnan(x) || isinf(x) || fabsf(x) > a)
                continue;
            float ref = x / s, q = scheme(x, s, r);
            j->pairs++;
            if (fabsf(ref) >= 0x1p-12f) {
                if (memcmp(&q, &ref, 4) != 0)
                    j->bad++;
            } else if (signbit(q) != signbit(ref) || fabsf(q) >= 0x1p-11f) {
                j->bad++;
            }
        }
    }
    return NULL;
}

int main(void)
{
    enum { T = 16 };
    pthread_t th[T];
    job_t jobs[T];
    const int top = 0x7F80, step = top / T + 1;
    long long bad = 0, pairs = 0;
    for (int i = 0; i < T; ++i) {
        jobs[i].lo = i * step;
        jobs[i].hi = (i + 1) * step < top ? (i + 1) * step : top;
        jobs[i].bad = jobs[i].pairs = 0;
        pthread_create(&th[i], NULL, run, &jobs[i]);
    }
    for (int i = 0; i < T; ++i) {
        pthread_join(th[i], NULL);
        bad += jobs[i].bad;
        pairs += jobs[i].pairs;
    }
    printf("pairs=%lld mismatches=%lld\n", pairs, bad);
    return bad == 0 ? 0 : 1;
}
