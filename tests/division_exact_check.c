/* Host check of the quotient the saved-FP8 re-quantization uses in place of
 * IEEE division (neg_quotient2_exact in the CUDA sources): two Markstein
 * corrections of x * RN(1/s), run on the negated quotient with nr = -RN(1/s):
 *   n = RN(x nr); e = fma(n, s, x); n = fma(e, nr, n); e = fma(n, s, x); n = fma(e, nr, n)
 * Claim, for 2^-90 <= s <= 2^126: -n equals the IEEE quotient RN(x / s) bit
 * for bit wherever |x / s| >= 2^-11 (below that both codes are +-0), and
 * the E4M3 code of -n (sign included: -0 for x = -0) equals the code of the
 * IEEE quotient everywhere.  Sweeps:
 *   1. every significand of x in one binade, both signs of a few, against 64
 *      divisors (edge significands and random ones), quotients in [2^-2, 2^9];
 *   2. 2^27 random pairs over the whole range of s, |x / s| log-uniform in
 *      [2^-16, 448] with random signs;
 *   3. x = +0 and -0.
 * It also counts how often one correction alone misses the IEEE quotient, to
 * show that the sweeps reach the cases the second correction is there for.
 * The E4M3 encoder is a brute-force nearest search (ties to the even code,
 * saturating at 448).  Prints the counts; exit status 1 on any mismatch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static uint32_t bits_of(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

static double e4m3_value(int c) {
    const int e = (c >> 3) & 15, m = c & 7;
    return e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m / 8.0, -6);
}

static int e4m3_code(float q) {
    const int sign = signbit(q) ? 0x80 : 0;
    const double a = fabs((double)q);
    int lo = 0, hi = 0x7e;
    if (a >= e4m3_value(0x7e)) return sign | 0x7e;
    while (hi - lo > 1) {
        const int mid = (lo + hi) / 2;
        if (e4m3_value(mid) <= a) lo = mid; else hi = mid;
    }
    const double dl = a - e4m3_value(lo), dh = e4m3_value(hi) - a;
    if (dl < dh) return sign | lo;
    if (dh < dl) return sign | hi;
    return sign | ((lo & 1) ? hi : lo);
}

/* -n, the method's quotient */
static float method(float x, float s, float nr) {
    float n = x * nr;
    float e = fmaf(n, s, x);
    n = fmaf(e, nr, n);
    e = fmaf(n, s, x);
    n = fmaf(e, nr, n);
    return -n;
}

static float one_correction(float x, float s, float r) {
    const float q0 = x * r;
    return fmaf(fmaf(-s, q0, x), r, q0);
}

static uint64_t splitmix(uint64_t* st) {
    uint64_t z = (*st += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static double unit(uint64_t* st) { return (double)(splitmix(st) >> 11) * 0x1p-53; }

int main(void) {
    long long checked = 0, quotient_diffs = 0, code_diffs = 0, single_misses = 0;

    /* 1: 64 divisors x every significand of x in [1, 2) */
    float divs[64];
    {
        uint64_t st = 1;
        const float edge[8] = {1.0f, 0x1.000002p0f, 0x1.fffffep0f, 1.5f, 0x1.555556p0f, 0x1.c71c72p0f, 7.77f / 4, 1.1f};
        for (int i = 0; i < 64; ++i) {
            const float m = i < 8 ? edge[i] : (float)(1.0 + unit(&st));
            const int ex = -90 + (int)(unit(&st) * 216.0); /* [-90, 125] */
            divs[i] = ldexpf(m, ex);
        }
    }
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : checked, quotient_diffs, code_diffs, single_misses)
    for (int i = 0; i < 64; ++i) {
        const float s = divs[i];
        const float r = 1.0f / s, nr = -r;
        int es;
        frexpf(s, &es);
        const int k = (i % 12) - 2; /* quotients in [2^(k-1), 2^(k+1)) */
        for (uint32_t m = 0; m < (1u << 23); ++m) {
            float x;
            const uint32_t xb = ((uint32_t)(127 + es - 1 + k) << 23) | m;
            memcpy(&x, &xb, 4);
            if ((m & 1023u) == 5u) x = -x;
            const float q = x / s, p = method(x, s, nr);
            checked++;
            if (bits_of(p) != bits_of(q)) quotient_diffs++;
            if (e4m3_code(p) != e4m3_code(q)) code_diffs++;
            if (bits_of(one_correction(x, s, r)) != bits_of(q)) single_misses++;
        }
    }

    /* 2: random pairs over the whole range of s */
    const long long n2 = 1ll << 27;
#pragma omp parallel for schedule(static) reduction(+ : checked, quotient_diffs, code_diffs, single_misses)
    for (long long j = 0; j < n2; ++j) {
        uint64_t st = 0x5EEDull + (uint64_t)j * 0x100000001B3ull;
        const int ex = -90 + (int)(unit(&st) * 216.0);
        const float s = ldexpf((float)(1.0 + unit(&st)), ex);
        if (!(s >= 0x1p-90f && s <= 0x1p126f)) continue;
        const double u = exp2(-16.0 + unit(&st) * (16.0 + log2(448.0)));
        float x = (float)((double)s * u);
        if (!isfinite(x)) continue; /* s near 2^126 with a large quotient */
        if (splitmix(&st) & 1) x = -x;
        const float r = 1.0f / s;
        const float q = x / s, p = method(x, s, -r);
        checked++;
        if (fabsf(q) >= 0x1p-11f && bits_of(p) != bits_of(q)) quotient_diffs++;
        if (e4m3_code(p) != e4m3_code(q)) code_diffs++;
        if (fabsf(q) >= 0x1p-11f && bits_of(one_correction(x, s, r)) != bits_of(q)) single_misses++;
    }

    /* 3: signed zeros */
    for (int i = 0; i < 64; ++i) {
        const float s = divs[i], nr = -(1.0f / s);
        if (e4m3_code(method(0.0f, s, nr)) != 0x00) code_diffs++;
        if (e4m3_code(method(-0.0f, s, nr)) != 0x80) code_diffs++;
        checked += 2;
    }

    printf("checked %lld quotient_diffs %lld code_diffs %lld single_correction_misses %lld\n", checked,
           quotient_diffs, code_diffs, single_misses);
    return quotient_diffs != 0 || code_diffs != 0;
}
