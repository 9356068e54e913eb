/*
 * fp8_oracle.c -- plain, slow, obviously-correct CPU model of block-scaled
 * FP8 (E4M3) quantization, the block-scaled GEMM and the on-policy weight
 * sync payload.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark load it.  It shares no header, table or
 * helper with the CUDA path.
 *
 * Sources (web pages; cited by title and section):
 *  [P1] "Anyscale、SkyRL で FP8 学習・ロールアウトをサポートし一貫性を維持"
 *       (news.ainew.jp) -- sections "独立した量子化がポリシーの一貫性を崩す場合",
 *       "On-Policy FP8 weight sync" (Fig. 3), "Deep dive: FP8 quantization
 *       with FP32 and power-of-two block scales", "実践的な知見".
 *  [P2] "AIS: Adaptive Importance Sampling for Quantized RL" explainer
 *       (kasblo.com) -- table "FP8とBF16" (E4M3 = 1/4/3 bits), equation Q(X)
 *       (symmetric linear quantization, s = max|X| / qmax), table of error
 *       sources, softmax worked example.
 *  [P3] "Jet-RL: Enabling On-Policy FP8 Reinforcement Learning with Unified
 *       Training and Rollout Precision Flow" (gist.science) -- section
 *       "Kwantisatieschema" (1x128 activations, 128x128 weights, 1x128 and
 *       128x1 operands for WGrad).
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes as well):
 *  - E4M3 is the "FN" variant: bias 7, largest finite 448, no infinities,
 *    S.1111.111 is NaN.  [P2] gives only the 1/4/3 split.
 *  - Encoding rounds to nearest, ties to even, and saturates finite
 *    magnitudes above 448 to 448; the sign is always kept (so negative
 *    values that round to zero give 0x80).  +-Inf saturates, NaN -> 0x7F|sign.
 *  - Blockwise scale s = amax / 448 as one IEEE fp32 division (Q(X) of [P2]
 *    with qmax = 448); an all-zero group uses s = 1.  Elements are encoded
 *    from the fp32 quotient x / s (IEEE division, round to nearest even).
 *  - MX scale exponent e = clamp(floor(log2 amax) - 8, -127, 127), stored as
 *    the E8M0 byte e + 127; an all-zero block uses e = -127.  Elements are
 *    encoded from the exact product x * 2^-e.
 *
 * Parity pins: every function below is checked by tests against something
 * other than itself (brute-force nearest search, a library cast, closed
 * forms, invariants, the softmax worked example of [P2]).  The naive
 * off-policy re-quantization and the checksum carry no external pin beyond
 * their invariants; see the "parity unpinned" notes at those functions.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fopenmp
 *        (no fast-math: the fp32 divisions must be IEEE).
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>
#include <omp.h>

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                            */
/* ------------------------------------------------------------------------ */

/* Widen a bf16 bit pattern to fp32 (exact: bf16 is the top half of fp32). */
static float bf16_bits_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

static uint64_t f64_bits(double d)
{
    uint64_t u;
    memcpy(&u, &d, 8);
    return u;
}

/* E4M3 decode ([P2] table "FP8とBF16": 1 sign, 4 exponent, 3 mantissa bits;
 * bias 7 and the NaN pattern are the OCP "E4M3FN" reading).
 * E == 0 is the subnormal range m * 2^-9 (covers +-0). */
double oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int E = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (E == 15 && m == 7)
        return NAN;
    if (E == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, E - 7);
    return s ? -v : v;
}

/* E4M3 encode of an exact real value (given as a double), round to nearest,
 * ties to even, saturating.  Works on the integer significand of the double
 * so no floating-point rounding helper is involved.
 *
 * Grid: for |v| >= 2^-6 the spacing is 2^(floor(log2|v|) - 3); below that it
 * is the subnormal step 2^-9. */
uint8_t oracle_e4m3_encode_f64(double v)
{
    uint64_t u = f64_bits(v);
    uint8_t sign = (uint8_t)((u >> 63) << 7);
    int bexp = (int)((u >> 52) & 0x7FF);
    uint64_t frac = u & ((1ULL << 52) - 1);

    if (bexp == 0x7FF) {
        if (frac != 0)
            return sign | 0x7F;          /* NaN */
        return sign | 0x7E;              /* +-Inf saturates to +-448 */
    }
    if (bexp == 0)                       /* zero or double subnormal (< 2^-1022) */
        return sign;

    int ex = bexp - 1023;                /* floor(log2 |v|) */
    uint64_t sig = frac | (1ULL << 52);  /* |v| = sig * 2^(ex - 52) */
    int qe = (ex >= -6 ? ex : -6) - 3;   /* exponent of the grid spacing */
    int shift = 52 + qe - ex;            /* |v| / 2^qe = sig / 2^shift */
    uint64_t q;
    if (shift >= 54) {
        q = 0;                           /* |v| < half a step: rounds to 0 */
    } else {
        uint64_t rem = sig & ((1ULL << shift) - 1);
        uint64_t half = 1ULL << (shift - 1);
        q = sig >> shift;
        if (rem > half || (rem == half && (q & 1)))
            q += 1;
    }

    if (ex < -6) {
        /* subnormal grid: q steps of 2^-9; q == 8 is exactly 2^-6, the code
         * 0x08 (exponent field 1, mantissa 0). */
        return sign | (uint8_t)q;
    }
    /* normal grid: q in [8, 16] */
    if (q == 16) {
        q = 8;
        ex += 1;
    }
    int E = ex + 7;
    int m = (int)q - 8;
    if (E > 15 || (E == 15 && m == 7))
        return sign | 0x7E;              /* saturate to 448 */
    return sign | (uint8_t)((E << 3) | m);
}

uint8_t oracle_e4m3_encode_f32(float v)
{
    return oracle_e4m3_encode_f64((double)v);
}

/* Round a double to the nearest bf16 (ties to even); returns the bit pattern.
 * Used only by the naive off-policy path. */
static uint16_t f32_to_bf16_bits(float f)
{
    uint32_t u = f32_bits(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu))
        return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void oracle_e4m3_encode_array(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode_f32(v[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------ */
/* Blockwise (fp32-scale) quantization: 1x128, 128x1 and 128x128 groups.     */
/* ------------------------------------------------------------------------ */

/* Scale of one group: s = amax / 448 in fp32 ([P2] eq. Q(X) with the E4M3
 * maximum in place of 2^(b-1)-1); s = 1 for an all-zero group, and likewise
 * when the quotient underflows to 0 (amax below 448 * 2^-150, reachable only
 * with fp32 inputs), so that no block divides by zero. */
static float group_scale(float amax)
{
    float s = amax / 448.0f;
    if (s == 0.0f)
        return 1.0f;
    return s;
}

static uint8_t encode_div(float x, float s)
{
    float q = x / s;                     /* one IEEE fp32 division */
    return oracle_e4m3_encode_f32(q);
}

/* 1x128 activation groups ([P3] "Kwantisatieschema": activations per-group
 * 1x128).  x: bf16 bits [M][ld] row-major; K % 128 == 0.
 * codes: [M][K]; scales: [K/128][M] (group-major). */
void oracle_quant_group_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ld,
                              uint8_t* codes, float* scales)
{
    int64_t G = K / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t g = 0; g < G; ++g) {
            float amax = 0.0f;
            for (int64_t j = 0; j < 128; ++j) {
                float a = fabsf(bf16_bits_to_f32(x[r * ld + g * 128 + j]));
                if (a > amax) amax = a;
            }
            float s = group_scale(amax);
            scales[g * M + r] = s;
            for (int64_t j = 0; j < 128; ++j)
                codes[r * K + g * 128 + j] =
                    encode_div(bf16_bits_to_f32(x[r * ld + g * 128 + j]), s);
        }
    }
}

/* 128x1 groups for the WGrad operand ([P3] "Kwantisatieschema", backward:
 * 1x128 and 128x1 for WGrad): one scale per column per 128 rows, codes
 * written transposed so the contraction index (rows of x) is contiguous.
 * x: bf16 [M][ld]; M % 128 == 0.  codesT: [K][M]; scales: [M/128][K]. */
void oracle_quant_group_128x1_T(const uint16_t* x, int64_t M, int64_t K, int64_t ld,
                                uint8_t* codesT, float* scales)
{
    int64_t B = M / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < K; ++c) {
        for (int64_t b = 0; b < B; ++b) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i) {
                float a = fabsf(bf16_bits_to_f32(x[(b * 128 + i) * ld + c]));
                if (a > amax) amax = a;
            }
            float s = group_scale(amax);
            scales[b * K + c] = s;
            for (int64_t i = 0; i < 128; ++i)
                codesT[c * M + b * 128 + i] =
                    encode_div(bf16_bits_to_f32(x[(b * 128 + i) * ld + c]), s);
        }
    }
}

/* 128x128 weight blocks ([P1] "なぜ強化学習に FP8 が重要なのか": 128x128 scaling
 * blocks for weights; [P3] "Kwantisatieschema").  w: bf16 [N][ld];
 * N % 128 == 0, K % 128 == 0.  codes [N][K]; scales [N/128][K/128].
 * Optional transposed copy (the same codes, transposed, for DGrad):
 * codesT [K][N] and scalesT [K/128][N/128]. */
void oracle_quant_block_128x128(const uint16_t* w, int64_t N, int64_t K, int64_t ld,
                                uint8_t* codes, float* scales,
                                uint8_t* codesT, float* scalesT)
{
    int64_t NB = N / 128, KB = K / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    float a = fabsf(bf16_bits_to_f32(w[(nb * 128 + i) * ld + kb * 128 + j]));
                    if (a > amax) amax = a;
                }
            float s = group_scale(amax);
            scales[nb * KB + kb] = s;
            if (scalesT) scalesT[kb * NB + nb] = s;
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    int64_t n = nb * 128 + i, k = kb * 128 + j;
                    uint8_t q = encode_div(bf16_bits_to_f32(w[n * ld + k]), s);
                    codes[n * K + k] = q;
                    if (codesT) codesT[k * N + n] = q;
                }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* MXFP8: 1x32 blocks with E8M0 (power-of-two) scales                        */
/* ([P1] "独立した量子化..." : one scale per 1x32 block in the MXFP8 recipe;       */
/*  "Deep dive...": Blackwell tensor cores accept only power-of-two scales). */
/* ------------------------------------------------------------------------ */

/* floor(log2 a) for a finite a > 0, read from the fp32 bit fields. */
static int floor_log2_f32(float a)
{
    uint32_t u = f32_bits(a);
    int bexp = (int)((u >> 23) & 0xFF);
    uint32_t m = u & 0x7FFFFF;
    if (bexp != 0)
        return bexp - 127;
    int p = 22;                          /* subnormal: leading bit position */
    while (p >= 0 && !((m >> p) & 1)) --p;
    return p - 149;
}

/* Shared exponent of one 1x32 block. */
static int mx_exponent(float amax)
{
    if (amax == 0.0f)
        return -127;
    int e = floor_log2_f32(amax) - 8;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Byte offset of the E8M0 scale of (row r, 32-block kb) in the scale-factor
 * layout the tensor core reads: atoms of 128 rows x 4 blocks (512 bytes),
 * atoms ordered row-tile major with the block-group index fastest; inside an
 * atom row r sits at (r%32)*16 + ((r%128)/32)*4 and block kb at kb%4.
 * K is the number of columns (a multiple of 32); atoms per row tile =
 * ceil(K/128). */
int64_t oracle_mx_scale_offset(int64_t r, int64_t kb, int64_t K)
{
    int64_t atoms_k = (K + 127) / 128;
    int64_t atom = (r / 128) * atoms_k + kb / 4;
    return atom * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (kb % 4);
}

int64_t oracle_mx_scale_bytes(int64_t R, int64_t K)
{
    return ((R + 127) / 128) * ((K + 127) / 128) * 512;
}

/* x: bf16 [R][ld], K % 32 == 0.  codes [R][K]; scales: the atom layout above
 * (oracle_mx_scale_bytes(R, K) bytes; entries for padding rows/blocks are
 * written as 0). */
void oracle_quant_mx_1x32(const uint16_t* x, int64_t R, int64_t K, int64_t ld,
                          uint8_t* codes, uint8_t* scales)
{
    memset(scales, 0, (size_t)oracle_mx_scale_bytes(R, K));
    int64_t KB = K / 32;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t j = 0; j < 32; ++j) {
                float a = fabsf(bf16_bits_to_f32(x[r * ld + kb * 32 + j]));
                if (a > amax) amax = a;
            }
            int e = mx_exponent(amax);
            scales[oracle_mx_scale_offset(r, kb, K)] = (uint8_t)(e + 127);
            for (int64_t j = 0; j < 32; ++j) {
                double v = ldexp((double)bf16_bits_to_f32(x[r * ld + kb * 32 + j]), -e);
                codes[r * K + kb * 32 + j] = oracle_e4m3_encode_f64(v);
            }
        }
    }
}

/* 32x1 blocks along the rows, codes written transposed: the MXFP8 backward
 * operands (WGrad contracts over the token dimension M, DGrad's B operand is
 * W^T) -- exactly oracle_quant_mx_1x32 of x^T.  x: bf16 [R][ld];
 * codesT [K][R]; scalesT: MX atoms of the [K][R] tensor. */
void oracle_quant_mx_32x1_T(const uint16_t* x, int64_t R, int64_t K, int64_t ld,
                            uint8_t* codesT, uint8_t* scalesT)
{
    memset(scalesT, 0, (size_t)oracle_mx_scale_bytes(K, R));
    int64_t RB = R / 32;
    #pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < K; ++c) {
        for (int64_t rb = 0; rb < RB; ++rb) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 32; ++i) {
                float a = fabsf(bf16_bits_to_f32(x[(rb * 32 + i) * ld + c]));
                if (a > amax) amax = a;
            }
            int e = mx_exponent(amax);
            scalesT[oracle_mx_scale_offset(c, rb, R)] = (uint8_t)(e + 127);
            for (int64_t i = 0; i < 32; ++i) {
                double v = ldexp((double)bf16_bits_to_f32(x[(rb * 32 + i) * ld + c]), -e);
                codesT[c * R + rb * 32 + i] = oracle_e4m3_encode_f64(v);
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Blockwise recipe with power-of-two scales ([P1] "Deep dive: FP8            */
/* quantization with FP32 and power-of-two block scales": Blackwell's tensor  */
/* cores take only power-of-two block scales, at the cost of a grid up to 2x  */
/* coarser).  Same groups as the fp32 recipe (1x128, 128x1, 128x128); the     */
/* scale is s = 2^e, e = ceil(log2(amax/448)) with amax/448 the fp32 scale of */
/* the fp32 recipe, i.e. the smallest power of two not below it, so that      */
/* max|x|/s <= 448; e clamped to the E8M0 range [-127, 127]; e = 0 (s = 1)    */
/* for an all-zero group, as in the fp32 recipe.  Codes from the exact        */
/* product x * 2^-e.  The scales are stored as E8M0 bytes (e + 127) in the    */
/* MX scale-factor layout, each group's byte repeated in every 1x32 block it  */
/* covers, so the tensor is also a valid MXFP8 tensor.                        */
/* ------------------------------------------------------------------------ */

int oracle_pow2_exponent(float amax)
{
    if (amax == 0.0f)
        return 0;
    float t = amax / 448.0f;                /* the fp32 recipe's scale */
    int e = floor_log2_f32(t);
    if ((double)t != ldexp(1.0, e))         /* not a power of two: round up */
        e += 1;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

static uint8_t encode_pow2(float x, int e)
{
    return oracle_e4m3_encode_f64(ldexp((double)x, -e));
}

/* x: bf16 [M][ld], K % 128 == 0.  codes [M][K]; scales: MX atoms of [M][K]. */
void oracle_quant_group_1x128_pow2(const uint16_t* x, int64_t M, int64_t K, int64_t ld,
                                   uint8_t* codes, uint8_t* scales)
{
    memset(scales, 0, (size_t)oracle_mx_scale_bytes(M, K));
    int64_t G = K / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t g = 0; g < G; ++g) {
            float amax = 0.0f;
            for (int64_t j = 0; j < 128; ++j) {
                float a = fabsf(bf16_bits_to_f32(x[r * ld + g * 128 + j]));
                if (a > amax) amax = a;
            }
            int e = oracle_pow2_exponent(amax);
            for (int64_t b = 0; b < 4; ++b)
                scales[oracle_mx_scale_offset(r, 4 * g + b, K)] = (uint8_t)(e + 127);
            for (int64_t j = 0; j < 128; ++j)
                codes[r * K + g * 128 + j] = encode_pow2(bf16_bits_to_f32(x[r * ld + g * 128 + j]), e);
        }
    }
}

/* 128x1 groups, codes transposed: codesT [K][M] (the WGrad operand, M
 * contiguous); scales: MX atoms of the transposed [K][M] tensor, i.e. the
 * 1x32 blocks run along M.  M % 128 == 0. */
void oracle_quant_group_128x1_T_pow2(const uint16_t* x, int64_t M, int64_t K, int64_t ld,
                                     uint8_t* codesT, uint8_t* scalesT)
{
    memset(scalesT, 0, (size_t)oracle_mx_scale_bytes(K, M));
    int64_t B = M / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < K; ++c) {
        for (int64_t b = 0; b < B; ++b) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i) {
                float a = fabsf(bf16_bits_to_f32(x[(b * 128 + i) * ld + c]));
                if (a > amax) amax = a;
            }
            int e = oracle_pow2_exponent(amax);
            for (int64_t q = 0; q < 4; ++q)
                scalesT[oracle_mx_scale_offset(c, 4 * b + q, M)] = (uint8_t)(e + 127);
            for (int64_t i = 0; i < 128; ++i)
                codesT[c * M + b * 128 + i] = encode_pow2(bf16_bits_to_f32(x[(b * 128 + i) * ld + c]), e);
        }
    }
}

/* 128x128 blocks: codes [N][K], scales MX atoms of [N][K]; optionally the
 * transposed copy codesT [K][N] with MX atoms of [K][N] (same exponents). */
void oracle_quant_block_128x128_pow2(const uint16_t* w, int64_t N, int64_t K, int64_t ld,
                                     uint8_t* codes, uint8_t* scales,
                                     uint8_t* codesT, uint8_t* scalesT)
{
    memset(scales, 0, (size_t)oracle_mx_scale_bytes(N, K));
    if (scalesT) memset(scalesT, 0, (size_t)oracle_mx_scale_bytes(K, N));
    int64_t NB = N / 128, KB = K / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    float a = fabsf(bf16_bits_to_f32(w[(nb * 128 + i) * ld + kb * 128 + j]));
                    if (a > amax) amax = a;
                }
            int e = oracle_pow2_exponent(amax);
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t q = 0; q < 4; ++q) {
                    scales[oracle_mx_scale_offset(nb * 128 + i, 4 * kb + q, K)] = (uint8_t)(e + 127);
                    if (scalesT) scalesT[oracle_mx_scale_offset(kb * 128 + i, 4 * nb + q, N)] = (uint8_t)(e + 127);
                }
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    int64_t n = nb * 128 + i, k = kb * 128 + j;
                    uint8_t q = encode_pow2(bf16_bits_to_f32(w[n * ld + k]), e);
                    codes[n * K + k] = q;
                    if (codesT) codesT[k * N + n] = q;
                }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* fp8_param ([P1] overview: FP8 parameters plus an FP32 master, no BF16     */
/* copy; "Deep dive: FP8 quantization with FP32 and power-of-two block       */
/* scales": the optimizer updates the FP32 master and, after every step, the */
/* FP8 storage is recomputed from it as Q(W_t)).  The update is the add that */
/* ends an optimizer step, W_t = W_{t-1} + dW in fp32; Q is the 128x128      */
/* block quantizer of either recipe applied to the fp32 values themselves    */
/* (no bf16 rounding in between).                                            */
/* ------------------------------------------------------------------------ */

/* master[n][k] += delta[n][k] (one IEEE fp32 addition each); both [N][ld]. */
void oracle_param_update(float* master, const float* delta, int64_t N, int64_t K, int64_t ld)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            master[n * ld + k] = master[n * ld + k] + delta[n * ld + k];
}

/* fp32 scales: as oracle_quant_block_128x128 with fp32 inputs: s =
 * RN(amax / 448) (1 for an all-zero block), codes = E4M3(RN(w / s)).
 * w: fp32 [N][ld]; codes [N][K], scales [N/128][K/128]; optional transposed
 * copy codesT [K][N], scalesT [K/128][N/128]. */
void oracle_quant_block_128x128_f32(const float* w, int64_t N, int64_t K, int64_t ld,
                                    uint8_t* codes, float* scales,
                                    uint8_t* codesT, float* scalesT)
{
    int64_t NB = N / 128, KB = K / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    float a = fabsf(w[(nb * 128 + i) * ld + kb * 128 + j]);
                    if (a > amax) amax = a;
                }
            float s = group_scale(amax);
            scales[nb * KB + kb] = s;
            if (scalesT) scalesT[kb * NB + nb] = s;
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    int64_t n = nb * 128 + i, k = kb * 128 + j;
                    uint8_t q = encode_div(w[n * ld + k], s);
                    codes[n * K + k] = q;
                    if (codesT) codesT[k * N + n] = q;
                }
        }
    }
}

/* Power-of-two scales: as oracle_quant_block_128x128_pow2 with fp32 inputs
 * (e from the fp32 recipe's scale of the block maximum, codes from the exact
 * w * 2^-e, E8M0 bytes in the MX atom layout). */
void oracle_quant_block_128x128_f32_pow2(const float* w, int64_t N, int64_t K, int64_t ld,
                                         uint8_t* codes, uint8_t* scales,
                                         uint8_t* codesT, uint8_t* scalesT)
{
    memset(scales, 0, (size_t)oracle_mx_scale_bytes(N, K));
    if (scalesT) memset(scalesT, 0, (size_t)oracle_mx_scale_bytes(K, N));
    int64_t NB = N / 128, KB = K / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    float a = fabsf(w[(nb * 128 + i) * ld + kb * 128 + j]);
                    if (a > amax) amax = a;
                }
            int e = oracle_pow2_exponent(amax);
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t q = 0; q < 4; ++q) {
                    scales[oracle_mx_scale_offset(nb * 128 + i, 4 * kb + q, K)] = (uint8_t)(e + 127);
                    if (scalesT) scalesT[oracle_mx_scale_offset(kb * 128 + i, 4 * nb + q, N)] = (uint8_t)(e + 127);
                }
            for (int64_t i = 0; i < 128; ++i)
                for (int64_t j = 0; j < 128; ++j) {
                    int64_t n = nb * 128 + i, k = kb * 128 + j;
                    uint8_t q = encode_pow2(w[n * ld + k], e);
                    codes[n * K + k] = q;
                    if (codesT) codesT[k * N + n] = q;
                }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* WGrad operand from the saved FP8 activation ([Jet-RL] "Kwantisatieschema": */
/* the activations kept for the backward pass are stored in FP8, quantized    */
/* 1x128; WGrad needs its operands in 128x1 groups along M).  Each element is */
/* dequantized once in fp32, x' = RN(dec(q) * s), and x' is quantized in      */
/* 128x1 groups with the codes transposed, exactly as bf16 inputs are.        */
/* codes [M][K] with 1x128 scales [K/128][M] -> codesT [K][M], scalesT        */
/* [M/128][K].  M % 128 == 0, K % 128 == 0.                                   */
/* ------------------------------------------------------------------------ */
void oracle_requant_1x128_to_128x1_T(const uint8_t* codes, const float* scales, int64_t M, int64_t K,
                                     uint8_t* codesT, float* scalesT)
{
    int64_t B = M / 128;
    #pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < K; ++c) {
        float col[128];
        for (int64_t b = 0; b < B; ++b) {
            float amax = 0.0f;
            for (int64_t i = 0; i < 128; ++i) {
                int64_t m = b * 128 + i;
                /* dec(q) has at most 4 significant bits: the fp64 product is
                 * exact, so the cast rounds it once to fp32 */
                col[i] = (float)(oracle_e4m3_decode(codes[m * K + c]) * (double)scales[(c / 128) * M + m]);
                float a = fabsf(col[i]);
                if (a > amax) amax = a;
            }
            float s = group_scale(amax);
            scalesT[b * K + c] = s;
            for (int64_t i = 0; i < 128; ++i)
                codesT[c * M + b * 128 + i] = encode_div(col[i], s);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Producers fused with the quantization ([P3] "Kwantisatieschema": the      */
/* activations saved for the backward pass are stored in FP8, fused with the */
/* previous operator; "Implementatie": fused activation / RMSNorm kernels).  */
/* The oracle computes each producer in fp64 and rounds its output once to   */
/* bf16; the quantizers above then take that bf16 tensor, so the fused      */
/* operation equals the producer followed by the quantizer.                  */
/* ------------------------------------------------------------------------ */

/* bf16 nearest to an exact real value (round to nearest, ties to even;
 * overflow to +-inf; bf16 subnormals down to 2^-133; NaN -> 0x7FC0|sign).
 * Works on the double's binary exponent like oracle_e4m3_encode_f64. */
uint16_t oracle_bf16_round_f64(double v)
{
    uint16_t sign = (uint16_t)((f64_bits(v) >> 63) << 15);
    if (isnan(v))
        return sign | 0x7FC0;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0 || a < ldexp(1.0, -140))   /* far below half the smallest step */
        return sign;
    int ex = ilogb(a);                       /* floor(log2 a) */
    int qe = (ex >= -126 ? ex : -126) - 7;   /* exponent of the grid spacing */
    double t = ldexp(a, -qe);                /* exact: a / 2^qe */
    double fl = floor(t);
    double rem = t - fl;                     /* exact */
    uint64_t q = (uint64_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (q & 1)))
        q += 1;
    if (ex < -126)                           /* subnormal grid: q steps of 2^-133 */
        return sign | (uint16_t)q;           /* q = 128 is 2^-126, bits 0x0080 */
    if (q == 256) {
        q = 128;
        ex += 1;
    }
    int E = ex + 127;
    if (E >= 255)
        return sign | 0x7F80;
    return sign | (uint16_t)((E << 7) | (int)(q - 128));
}

/* RMSNorm: y[r][k] = x[r][k] * rstd[r] * gamma[k] with rstd = 1 / sqrt(mean_k
 * x[r][k]^2 + eps), all in fp64, y rounded once to bf16; rstd returned as
 * fp32 (saved for the backward pass).  x bf16 [M][ld], gamma bf16 [K],
 * y bf16 [M][K]. */
void oracle_rmsnorm(const uint16_t* x, const uint16_t* gamma, int64_t M, int64_t K, int64_t ld, float eps,
                    uint16_t* y, float* rstd)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = (double)bf16_bits_to_f32(x[r * ld + k]);
            ss += v * v;
        }
        double rs = 1.0 / sqrt(ss / (double)K + (double)eps);
        if (rstd) rstd[r] = (float)rs;
        for (int64_t k = 0; k < K; ++k)
            y[r * K + k] = oracle_bf16_round_f64((double)bf16_bits_to_f32(x[r * ld + k]) * rs *
                                                 (double)bf16_bits_to_f32(gamma[k]));
    }
}

/* SwiGLU: h[r][f] = silu(g) * u with g = gu[r][f], u = gu[r][F + f] (the
 * gate and up projections side by side in one [M][2F] row), silu(g) =
 * g / (1 + exp(-g)), in fp64, h rounded once to bf16.  gu bf16 [M][ld],
 * ld >= 2F; h bf16 [M][F]. */
void oracle_swiglu(const uint16_t* gu, int64_t M, int64_t F, int64_t ld, uint16_t* h)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < M; ++r)
        for (int64_t f = 0; f < F; ++f) {
            double g = (double)bf16_bits_to_f32(gu[r * ld + f]);
            double u = (double)bf16_bits_to_f32(gu[r * ld + F + f]);
            h[r * F + f] = oracle_bf16_round_f64(g / (1.0 + exp(-g)) * u);
        }
}

/* ------------------------------------------------------------------------ */
/* Dequantization (exact in fp64: a 4-bit significand times a 24-bit scale).  */
/* ------------------------------------------------------------------------ */

/* layout 1: 1x128 groups, scales [K/128][R] */
void oracle_dequant_group(const uint8_t* codes, const float* scales, int64_t R, int64_t K,
                          double* out)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            out[r * K + k] = oracle_e4m3_decode(codes[r * K + k]) * (double)scales[(k / 128) * R + r];
}

/* layout 2: 128x128 blocks, scales [R/128][K/128] */
void oracle_dequant_block(const uint8_t* codes, const float* scales, int64_t R, int64_t K,
                          double* out)
{
    int64_t KB = K / 128;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k)
            out[r * K + k] = oracle_e4m3_decode(codes[r * K + k]) *
                             (double)scales[(r / 128) * KB + k / 128];
}

/* layout 3: MX 1x32, E8M0 scales in the atom layout */
void oracle_dequant_mx(const uint8_t* codes, const uint8_t* scales, int64_t R, int64_t K,
                       double* out)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; ++k) {
            int e = (int)scales[oracle_mx_scale_offset(r, k / 32, K)] - 127;
            out[r * K + k] = ldexp(oracle_e4m3_decode(codes[r * K + k]), e);
        }
}

/* ------------------------------------------------------------------------ */
/* GEMM reference: ref[m][n] = sum_k A[m][k] * B[n][k] in fp64, and the       */
/* magnitude sum mag[m][n] = sum_k |A[m][k] * B[n][k]| used by the tolerance  */
/* |gpu - ref| <= 2e-3 * mag + 2^-8 * |ref|.                                  */
/* A, B: dequantized operands, both with the contraction index contiguous.    */
/* ------------------------------------------------------------------------ */
void oracle_gemm_ref(const double* A, const double* B, int64_t M, int64_t N, int64_t K,
                     double* ref, double* mag)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, am = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = A[m * K + k] * B[n * K + k];
                acc += p;
                am += fabs(p);
            }
            ref[m * N + n] = acc;
            mag[m * N + n] = am;
        }
}

/* The same at a list of sampled output positions (ms[i], ns[i]); A and B are
 * given as full dequantized rows. */
void oracle_gemm_ref_sampled(const double* A, const double* B, int64_t K,
                             const int64_t* ms, const int64_t* ns, int64_t count,
                             double* ref, double* mag)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) {
        const double* a = A + ms[i] * K;
        const double* b = B + ns[i] * K;
        double acc = 0.0, am = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = a[k] * b[k];
            acc += p;
            am += fabs(p);
        }
        ref[i] = acc;
        mag[i] = am;
    }
}

/* ------------------------------------------------------------------------ */
/* Naive off-policy weight sync ([P1] "独立した量子化がポリシーの一貫性を崩す場合",  */
/* Fig. 2): the bridge dequantizes the trainer's blocks to BF16, the rollout  */
/* engine re-derives its own per-tensor scale and re-quantizes.  Test-only    */
/* counter-example.  Dequant is an fp32 product rounded to bf16 (reading).    */
/* parity unpinned: the pages give only the qualitative outcome.             */
/* ------------------------------------------------------------------------ */
float oracle_naive_requant_per_tensor(const uint8_t* codes, const float* block_scales,
                                      int64_t N, int64_t K, uint8_t* out_codes)
{
    int64_t KB = K / 128;
    int64_t n_el = N * K;
    uint16_t* tmp = (uint16_t*)malloc((size_t)n_el * sizeof(uint16_t));
    float amax = 0.0f;
    for (int64_t r = 0; r < N; ++r)
        for (int64_t k = 0; k < K; ++k) {
            float d = (float)oracle_e4m3_decode(codes[r * K + k]) * block_scales[(r / 128) * KB + k / 128];
            uint16_t b = f32_to_bf16_bits(d);
            tmp[r * K + k] = b;
            float a = fabsf(bf16_bits_to_f32(b));
            if (a > amax) amax = a;
        }
    float s = group_scale(amax);
    for (int64_t i = 0; i < n_el; ++i)
        out_codes[i] = encode_div(bf16_bits_to_f32(tmp[i]), s);
    free(tmp);
    return s;
}

/* ------------------------------------------------------------------------ */
/* On-policy weight sync payload ([P1] "On-Policy FP8 weight sync", Fig. 3:   */
/* quantized parameters travel as FP8 values plus their block scales,         */
/* precision-sensitive tensors stay BF16, the receiver installs them without  */
/* a quantizer and the result is bit-identical; "実践的な知見": values,        */
/* scales, exclusions and layouts come from one shared description).          */
/*                                                                            */
/* The byte format is this library's own definition (the pages give none):    */
/*   header, 64 bytes, little-endian:                                         */
/*     0 u64 magic "FP8SYNC1"   8 u32 version (2)   12 u32 n_entries          */
/*    16 u64 total_bytes       24 u64 data_offset   32 u64 checksum           */
/*    40..63 zero                                                             */
/*   entry table at 64, 128 bytes per entry:                                  */
/*     0 u64 tag   8 u32 kind (1 fp8, 2 bf16)   12 u32 recipe (0, 1, 2)       */
/*    16 i64 rows  24 i64 cols   32 u32 scale_layout   36 u32 zero            */
/*    40 u64 data_offset  48 u64 data_bytes  56 u64 scales_offset             */
/*    64 u64 scales_bytes  72..127 zero                                       */
/*   segments: data (codes or bf16 values) then scales, each starting at a    */
/*   256-byte boundary, zero padded; total_bytes is a multiple of 256;        */
/*   data_offset = roundup(64 + 128 n, 256).                                  */
/*   checksum: for each 8-byte word w_i at byte offset 8i >= 64, with lo_i   */
/*   and hi_i its low and high 32-bit halves,                                 */
/*     t_i = ((lo_i + i K1) mod 2^32) * ((hi_i + i K2) mod 2^32),             */
/*   K1 = 0x9E3779B9, K2 = 0x85EBCA6B, and checksum = sum of t_i mod 2^64:    */
/*   the NH inner product of UMAC (Black, Halevi, Krawczyk, Krovetz and       */
/*   Rogaway, "UMAC: Fast and Secure Message Authentication", CRYPTO 1999)    */
/*   with keys taken from the word index.  A change to one half of one word   */
/*   changes t_i by delta * (the other factor), |delta|, factor < 2^32, so it */
/*   is always detected unless that word's other factor is 0 mod 2^32; the    */
/*   keys repeat every 2^32 words (32 GiB).  (Version 1 of the format summed  */
/*   the splitmix64 finaliser of w_i XOR i instead: about eight times the     */
/*   integer work per word.)                                                  */
/* parity unpinned (format): pinned only by round-trip and corruption tests.  */
/* ------------------------------------------------------------------------ */

typedef struct {
    uint64_t tag;
    uint32_t kind;         /* 1 = fp8 codes + scales, 2 = bf16 passthrough */
    uint32_t recipe;       /* 0 for bf16, 1 blockwise fp32, 2 MXFP8 */
    int64_t rows, cols;
    uint32_t scale_layout; /* 1 group 1x128, 2 block 128x128, 3 MX 1x32 */
    const uint8_t* data;   /* host pointers (source for pack, target for install) */
    const uint8_t* scales;
} oracle_sync_entry;

/* t_i of the checksum for word w at word index i */
static uint64_t nh_term(uint64_t w, uint64_t i)
{
    const uint32_t a = (uint32_t)(w & 0xFFFFFFFFu) + (uint32_t)(i & 0xFFFFFFFFu) * 0x9E3779B9u;
    const uint32_t b = (uint32_t)(w >> 32) + (uint32_t)(i & 0xFFFFFFFFu) * 0x85EBCA6Bu;
    return (uint64_t)a * (uint64_t)b;
}

uint64_t oracle_sync_word_term(uint64_t w, uint64_t i) { return nh_term(w, i); }

static uint64_t rd64(const uint8_t* p)
{
    uint64_t v = 0;
    for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
    return v;
}

static uint32_t rd32(const uint8_t* p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static void wr64(uint8_t* p, uint64_t v)
{
    for (int i = 0; i < 8; ++i) { p[i] = (uint8_t)(v & 0xFF); v >>= 8; }
}

static void wr32(uint8_t* p, uint32_t v)
{
    for (int i = 0; i < 4; ++i) { p[i] = (uint8_t)(v & 0xFF); v >>= 8; }
}

static uint64_t round_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

static const uint64_t SYNC_MAGIC = 0x31434E5953385046ULL;  /* bytes "FP8SYNC1" */

/* bytes of the data segment and the scale segment of one entry */
static void entry_sizes(const oracle_sync_entry* e, uint64_t* data_b, uint64_t* scale_b)
{
    if (e->kind == 2) {
        *data_b = (uint64_t)(e->rows * e->cols * 2);
        *scale_b = 0;
        return;
    }
    *data_b = (uint64_t)(e->rows * e->cols);
    if (e->scale_layout == 1)
        *scale_b = (uint64_t)((e->cols / 128) * e->rows * 4);
    else if (e->scale_layout == 2)
        *scale_b = (uint64_t)((e->rows / 128) * (e->cols / 128) * 4);
    else
        *scale_b = (uint64_t)oracle_mx_scale_bytes(e->rows, e->cols);
}

uint64_t oracle_sync_checksum(const uint8_t* payload, uint64_t total_bytes)
{
    uint64_t sum = 0;
    for (uint64_t i = 8; i < total_bytes / 8; ++i)
        sum += nh_term(rd64(payload + 8 * i), i);
    return sum;
}

/* Lays out the payload for n entries; writes per-entry offsets and returns
 * total_bytes. */
static uint64_t sync_layout(const oracle_sync_entry* e, int32_t n,
                            uint64_t* data_off, uint64_t* scale_off)
{
    uint64_t off = round_up(64 + 128 * (uint64_t)n, 256);
    for (int32_t i = 0; i < n; ++i) {
        uint64_t db, sb;
        entry_sizes(&e[i], &db, &sb);
        data_off[i] = off;
        off = round_up(off + db, 256);
        scale_off[i] = sb ? off : 0;
        off = round_up(off + sb, 256);
    }
    return off;
}

uint64_t oracle_sync_payload_size(const oracle_sync_entry* e, int32_t n)
{
    uint64_t* d = (uint64_t*)calloc((size_t)n + 1, 8);
    uint64_t* s = (uint64_t*)calloc((size_t)n + 1, 8);
    uint64_t t = sync_layout(e, n, d, s);
    free(d);
    free(s);
    return t;
}

/* Packs n entries into payload (capacity bytes).  Returns total bytes, or 0
 * if the capacity is too small. */
uint64_t oracle_sync_pack(const oracle_sync_entry* e, int32_t n, uint8_t* payload,
                          uint64_t capacity)
{
    uint64_t* doff = (uint64_t*)calloc((size_t)n + 1, 8);
    uint64_t* soff = (uint64_t*)calloc((size_t)n + 1, 8);
    uint64_t total = sync_layout(e, n, doff, soff);
    if (total > capacity) {
        free(doff);
        free(soff);
        return 0;
    }
    memset(payload, 0, (size_t)total);
    wr64(payload + 0, SYNC_MAGIC);
    wr32(payload + 8, 2);
    wr32(payload + 12, (uint32_t)n);
    wr64(payload + 16, total);
    wr64(payload + 24, round_up(64 + 128 * (uint64_t)n, 256));
    for (int32_t i = 0; i < n; ++i) {
        uint8_t* t = payload + 64 + 128 * (uint64_t)i;
        uint64_t db, sb;
        entry_sizes(&e[i], &db, &sb);
        wr64(t + 0, e[i].tag);
        wr32(t + 8, e[i].kind);
        wr32(t + 12, e[i].recipe);
        wr64(t + 16, (uint64_t)e[i].rows);
        wr64(t + 24, (uint64_t)e[i].cols);
        wr32(t + 32, e[i].scale_layout);
        wr64(t + 40, doff[i]);
        wr64(t + 48, db);
        wr64(t + 56, soff[i]);
        wr64(t + 64, sb);
        memcpy(payload + doff[i], e[i].data, (size_t)db);
        if (sb)
            memcpy(payload + soff[i], e[i].scales, (size_t)sb);
    }
    wr64(payload + 32, oracle_sync_checksum(payload, total));
    free(doff);
    free(soff);
    return total;
}

/* Installs a payload into n destination entries (host buffers, written
 * through the entries' data/scales pointers).  Return codes: 0 ok,
 * 1 bad header or entry mismatch, 2 checksum mismatch.  Nothing is written
 * unless every check passes.  No quantizer is involved. */
int32_t oracle_sync_install(const uint8_t* payload, uint64_t bytes,
                            const oracle_sync_entry* dst, int32_t n)
{
    if (bytes < 64) return 1;
    if (rd64(payload) != SYNC_MAGIC || rd32(payload + 8) != 2 ||
        rd32(payload + 12) != (uint32_t)n)
        return 1;
    uint64_t total = rd64(payload + 16);
    if (total > bytes || (total % 256) != 0) return 1;
    if (rd64(payload + 24) != round_up(64 + 128 * (uint64_t)n, 256)) return 1;

    uint64_t* doff = (uint64_t*)calloc((size_t)n + 1, 8);
    uint64_t* soff = (uint64_t*)calloc((size_t)n + 1, 8);
    uint64_t expect_total = sync_layout(dst, n, doff, soff);
    int32_t rc = 0;
    if (expect_total != total) rc = 1;
    for (int32_t i = 0; i < n && rc == 0; ++i) {
        const uint8_t* t = payload + 64 + 128 * (uint64_t)i;
        uint64_t db, sb;
        entry_sizes(&dst[i], &db, &sb);
        if (rd64(t) != dst[i].tag || rd32(t + 8) != dst[i].kind ||
            rd32(t + 12) != dst[i].recipe || rd64(t + 16) != (uint64_t)dst[i].rows ||
            rd64(t + 24) != (uint64_t)dst[i].cols || rd32(t + 32) != dst[i].scale_layout ||
            rd64(t + 40) != doff[i] || rd64(t + 48) != db || rd64(t + 56) != soff[i] ||
            rd64(t + 64) != sb)
            rc = 1;
    }
    if (rc == 0 && oracle_sync_checksum(payload, total) != rd64(payload + 32))
        rc = 2;
    if (rc == 0) {
        for (int32_t i = 0; i < n; ++i) {
            uint64_t db, sb;
            entry_sizes(&dst[i], &db, &sb);
            memcpy((void*)dst[i].data, payload + doff[i], (size_t)db);
            if (sb)
                memcpy((void*)dst[i].scales, payload + soff[i], (size_t)sb);
        }
    }
    free(doff);
    free(soff);
    return rc;
}

/* Thread count of the OpenMP loops above (timing of the oracle on one
 * thread and on all cores; no effect on any result). */
void oracle_set_threads(int32_t n)
{
    omp_set_num_threads(n > 0 ? n : 1);
}

int32_t oracle_max_threads(void)
{
    return omp_get_max_threads();
}
