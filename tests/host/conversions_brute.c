/* Brute force of the oracle's number conversions over every binary32 bit
 * pattern (test program, built by tests/test_oracle_brute_force.py together
 * with oracle/h3q_oracle.c).  Each conversion is compared with a formulation
 * of its own, written here from the format definitions:
 *   bf16   nearest of the two bf16 values around v by exact distance in binary64,
 *          ties to the even pattern (every non-NaN v);
 *   E2M1   the threshold count (a>0.25)+(a>=0.75)+(a>1.25)+(a>=1.75)+(a>2.5)
 *          +(a>=3.5)+(a>5) of a = |v|, sign bit from v (every non-NaN v);
 *   E4M3   for 0 <= s < 448 the grid step 2^(e-3) of s's binade (2^-9 below
 *          2^-6), the two grid points around s by exact distance, ties to the
 *          even code; s >= 448 and +inf saturate to 0x7E.
 * bf16 and E2M1 are checked on every non-NaN pattern.  E4M3 (whose oracle is a
 * linear search over the codes, about nine minutes for all of them on eight
 * threads) is checked on every s >= 0 with the argument "full", and otherwise on
 * every s >= 0 whose low eight bits are zero plus every s within 256 ulps of one
 * of its decision points (the 127 values and the midpoints between neighbours,
 * where both formulations can change their result; between two decision points
 * both are constant).  Also exp_c, the SiLU exponential: within 2 ulp of
 * binary64 exp for every binary32 z in [-104, 88.7] (the ulp of the exact
 * result's binary32 magnitude, the subnormal spacing below 2^-126), +inf above
 * 89 and +0 below -104.  Prints the mismatch counts and exits non-zero if any. */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

uint16_t orc_bf16_bits(float v);
uint8_t orc_e4m3_encode(float s);
uint8_t orc_e2m1_encode(float v);
float orc_exp(float z);

/* spacing of binary32 values at the magnitude of x (x finite) */
static double ulp_at(double x)
{
    float r = (float)fabs(x);
    if (r < 0x1p-126f) return 0x1p-149;
    return ldexp(1.0, ilogbf(r) - 23);
}

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

static uint16_t bf16_ref(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    uint32_t t = u >> 16;                                /* toward zero */
    double lo = (double)f_of(t << 16), hi = (double)f_of((t + 1) << 16), x = (double)v;
    if (isinf(v) || lo == x) return (uint16_t)t;
    if (isinf(f_of((t + 1) << 16))) {                    /* next step away is infinity */
        /* the rounding boundary is the bf16 maximum plus half its ulp: 2^128 - 2^119 */
        double limit = ldexp(1.0, 128) - ldexp(1.0, 119);
        double ax = fabs(x);
        if (ax < limit) return (uint16_t)t;
        if (ax > limit) return (uint16_t)(t + 1);
        return (uint16_t)((t & 1) ? t + 1 : t);
    }
    double dl = fabs(x - lo), dh = fabs(hi - x);
    if (dl < dh) return (uint16_t)t;
    if (dh < dl) return (uint16_t)(t + 1);
    return (uint16_t)((t & 1) ? t + 1 : t);
}

static uint8_t e2m1_ref(float v)
{
    double a = fabs((double)v);
    int idx = (a > 0.25) + (a >= 0.75) + (a > 1.25) + (a >= 1.75) + (a > 2.5) + (a >= 3.5) + (a > 5.0);
    return (uint8_t)((signbit(v) ? 8 : 0) | idx);
}

static uint8_t e4m3_ref(float s)
{
    if (!(s < 448.0f)) return 0x7E;
    double x = (double)s;
    int e = (x >= ldexp(1.0, -6)) ? ilogb(x) : -6;       /* binade; subnormal grid below 2^-6 */
    double step = ldexp(1.0, e - 3);
    double k = floor(x / step);                          /* grid index of the point below (exact) */
    double lo = k * step, hi = lo + step;
    double dl = x - lo, dh = hi - x;
    double pick = (dl < dh) ? k : (dh < dl) ? k + 1 : (fmod(k, 2.0) == 0.0 ? k : k + 1);
    /* grid index -> code: in binade e >= -6 the index counts 8 + mantissa (normal)
     * or the mantissa (subnormal); a carry to index 16 is the next binade's 1.0 */
    double val = pick * step;
    if (val == 0.0) return 0;
    int ve = ilogb(val);
    if (ve < -6) return (uint8_t)(val / ldexp(1.0, -9));  /* subnormal: m * 2^-9 */
    int m = (int)(val / ldexp(1.0, ve - 3)) - 8;
    return (uint8_t)(((ve + 7) << 3) | m);
}

static int full_e4m3;

struct job { uint64_t first, last; unsigned long long bad[4]; double worst_exp_ulp; };

static void *work(void *p)
{
    struct job *j = (struct job *)p;
    for (uint64_t i = j->first; i < j->last; ++i) {
        uint32_t u = (uint32_t)i;
        float v = f_of(u);
        if (isnan(v)) continue;
        if (orc_bf16_bits(v) != bf16_ref(v)) ++j->bad[0];
        if (orc_e2m1_encode(v) != e2m1_ref(v)) ++j->bad[1];
        if (!signbit(v) && (full_e4m3 || (u & 0xffu) == 0) && orc_e4m3_encode(v) != e4m3_ref(v)) ++j->bad[2];
        if (v >= -104.0f && v <= 88.7f) {
            double want = exp((double)v);
            double err = fabs((double)orc_exp(v) - want) / ulp_at(want);
            if (err > j->worst_exp_ulp) j->worst_exp_ulp = err;
            if (err > 2.0) ++j->bad[3];
        } else if ((v > 89.0f && !isinf(orc_exp(v))) || (v < -104.0f && orc_exp(v) != 0.0f)) {
            ++j->bad[3];
        }
    }
    return NULL;
}

static float e4m3_val(int c)
{
    int e = (c >> 3) & 15, m = c & 7;
    return e == 0 ? ldexpf((float)m, -9) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
}

/* E4M3 within 256 ulps of each value and each midpoint (a midpoint of two
 * neighbouring values is exact in binary32); the ulps above 448 too. */
static unsigned long long e4m3_near_decisions(void)
{
    unsigned long long bad = 0;
    for (int c = 0; c <= 0x7E; ++c) {
        float pts[2] = {e4m3_val(c), c < 0x7E ? 0.5f * (e4m3_val(c) + e4m3_val(c + 1)) : 464.0f};
        for (int k = 0; k < 2; ++k) {
            uint32_t b;
            memcpy(&b, &pts[k], 4);
            for (int d = -256; d <= 256; ++d) {
                int64_t u = (int64_t)b + d;
                if (u < 0 || u > 0x7F800000) continue;
                float v = f_of((uint32_t)u);
                if (orc_e4m3_encode(v) != e4m3_ref(v)) ++bad;
            }
        }
    }
    return bad;
}

int main(int argc, char **argv)
{
    full_e4m3 = argc > 1 && strcmp(argv[1], "full") == 0;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    if (n < 1) n = 1;
    if (n > 64) n = 64;
    pthread_t th[64];
    struct job jobs[64];
    const uint64_t total = 1ull << 32;
    for (long t = 0; t < n; ++t) {
        jobs[t].first = total * (uint64_t)t / (uint64_t)n;
        jobs[t].last = total * (uint64_t)(t + 1) / (uint64_t)n;
        memset(jobs[t].bad, 0, sizeof jobs[t].bad);
        jobs[t].worst_exp_ulp = 0.0;
        pthread_create(&th[t], NULL, work, &jobs[t]);
    }
    unsigned long long bad[4] = {0, 0, full_e4m3 ? 0 : e4m3_near_decisions(), 0};
    double worst = 0.0;
    for (long t = 0; t < n; ++t) {
        pthread_join(th[t], NULL);
        for (int k = 0; k < 4; ++k) bad[k] += jobs[t].bad[k];
        if (jobs[t].worst_exp_ulp > worst) worst = jobs[t].worst_exp_ulp;
    }
    printf("threads %ld bf16 mismatches %llu e2m1 mismatches %llu e4m3 (%s) mismatches %llu\n", n, bad[0],
           bad[1], full_e4m3 ? "every s >= 0" : "sampled and near every decision point", bad[2]);
    printf("exp_c outside 2 ulp %llu worst %.4f ulp\n", bad[3], worst);
    return (bad[0] || bad[1] || bad[2] || bad[3]) ? 1 : 0;
}
