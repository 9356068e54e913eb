/* Exhaustive host check of the quotients the blockwise quantizers use in
 * place of IEEE divisions (Markstein's FMA correction, see group_scale_bf16
 * and make_divider in the CUDA sources).  First, s = RN(a / 448) for every
 * positive finite bf16 a, from a * RN(1/448) and one correction.  For every bf16 x and every positive finite bf16 group
 * maximum a >= |x|, with s = RN(a / 448) >= 2^-100:
 *   nr = -RN(1 / s), n = RN(x nr), e = fma(n, s, x), n1 = fma(e, nr, n)
 * (one correction, run on the negated quotient as the kernels do) must give,
 * with the sign bit flipped, the same E4M3 code as the IEEE quotient
 * RN(x / s), signed zeros included.  The E4M3
 * encoder here is a brute-force nearest search (ties to even mantissa,
 * saturating), independent of both.  Prints the counts; exit status 1 on
 * any code mismatch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t bits_of(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

static double e4m3_value(int c) {
    const int e = (c >> 3) & 15, m = c & 7;
    return e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m / 8.0, -6);
}

/* codes 0..0x7e, nearest with ties to the even code, saturating at 448 */
static int e4m3_code(float q) {
    const int sign = signbit(q) ? 0x80 : 0;
    const double a = fabs((double)q);
    int lo = 0, hi = 0x7e;
    if (a >= e4m3_value(0x7e)) return sign | 0x7e;
    while (hi - lo > 1) { /* largest code with value <= a */
        const int mid = (lo + hi) / 2;
        if (e4m3_value(mid) <= a) lo = mid; else hi = mid;
    }
    const double dl = a - e4m3_value(lo), dh = e4m3_value(hi) - a;
    if (dl < dh) return sign | lo;
    if (dh < dl) return sign | hi;
    return sign | ((lo & 1) ? hi : lo);
}

int main(void) {
    /* the scale itself: RN(a / 448) by the same correction of a * RN(1/448) */
    long long scale_diffs = 0;
    const float inv448 = 1.0f / 448.0f;
    for (int ah = 1; ah < 0x7f80; ++ah) {
        const float a = from_bf16((uint16_t)ah);
        const float q0 = a * inv448;
        const float e = fmaf(-448.0f, q0, a);
        const float sm = fmaf(e, inv448, q0);
        if (bits_of(sm) != bits_of(a / 448.0f)) scale_diffs++;
    }
    long long pairs = 0, quotient_diffs = 0, code_diffs = 0, slow_groups = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : pairs, quotient_diffs, code_diffs, slow_groups)
    for (int ah = 1; ah < 0x7f80; ++ah) {
        const float a = from_bf16((uint16_t)ah);
        const float s = a / 448.0f;
        if (!(s >= 0x1p-100f)) {
            slow_groups++;
            continue;
        }
        const float nr = -(1.0f / s);
        for (int xh = 0; xh < 0x10000; ++xh) {
            const float x = from_bf16((uint16_t)xh);
            if (!(fabsf(x) <= a)) continue;
            const float q = x / s;
            const float n0 = x * nr;
            const float e = fmaf(n0, s, x);
            const float n1 = fmaf(e, nr, n0);
            pairs++;
            if (bits_of(n1) != (bits_of(q) ^ 0x80000000u)) {
                quotient_diffs++;
                if ((e4m3_code(n1) ^ 0x80) != e4m3_code(q)) code_diffs++;
            }
        }
    }
    printf("scale_diffs %lld pairs %lld quotient_diffs %lld code_diffs %lld slow_groups %lld\n", scale_diffs, pairs,
           quotient_diffs, code_diffs, slow_groups);
    return code_diffs != 0 || scale_diffs != 0;
}
