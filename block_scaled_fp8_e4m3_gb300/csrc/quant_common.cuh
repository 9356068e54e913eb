// Register-level pieces shared by the quantizer kernels: streaming 16-byte
// loads, bf16 unpacking, group maxima and the two E4M3 encoders (IEEE
// quotient by a block scale; exact product by a power of two).
#pragma once
#include "common.cuh"

namespace fp8bs {

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ float amax8(const float (&f)[8]) {
    float a = fabsf(f[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) a = fmaxf(a, fabsf(f[i]));
    return a;
}

// 8 values divided by s (the IEEE fp32 quotient) and encoded: 8 codes in two words.
__device__ __forceinline__ uint2 encode8_div(const float (&f)[8], const Divider& d) {
    uint2 r;
    if (d.fast) {
        r.x = codes4_div_fast(d, f[0], f[1], f[2], f[3]);
        r.y = codes4_div_fast(d, f[4], f[5], f[6], f[7]);
    } else {
        float q[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = __fdiv_rn(f[k], d.s);
        r.x = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
        r.y = e4m3x2(q[4], q[5]) | (e4m3x2(q[6], q[7]) << 16);
    }
    return r;
}

// x / s correctly rounded for any fp32 x (a full 24-bit significand), two
// values at a time: two Markstein corrections of the product with the
// correctly rounded reciprocal (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990).  q0 = RN(x r) can lie up to 1.5 ulp from x/s; the first correction
// q1 = RN(q0 + (x - s q0) r) lies within one ulp, which is the hypothesis of
// Markstein's theorem, so the second, RN(q1 + (x - s q1) r), is RN(x/s).  The
// residuals x - s q are exact by FMA.  The steps run on the negated quotient
// with nr = -r, so that a zero x ends as a zero of the opposite sign: the
// returned pair is (-q(x0), -q(x1)) with the sign of -x even for x = -0, and
// the caller flips the sign bits of the codes.  Needs 2^-90 <= s <= 2^126:
// no intermediate under- or overflows wherever the E4M3 code can be nonzero.
__device__ __forceinline__ void neg_quotient2_exact(float x0, float x1, float s, float nr, float& n0, float& n1) {
    uint64_t xs, n;
    asm("mov.b64 %0, {%1, %2};" : "=l"(xs) : "f"(x0), "f"(x1));
    asm("{\n\t.reg .b64 s2, r2, e;\n\t"
        "mov.b64 s2, {%2, %2};\n\tmov.b64 r2, {%3, %3};\n\t"
        "mul.rn.f32x2 %0, %1, r2;\n\t"
        "fma.rn.f32x2 e, %0, s2, %1;\n\t"
        "fma.rn.f32x2 %0, e, r2, %0;\n\t"
        "fma.rn.f32x2 e, %0, s2, %1;\n\t"
        "fma.rn.f32x2 %0, e, r2, %0;\n\t}\n"
        : "=&l"(n)
        : "l"(xs), "f"(s), "f"(nr));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(n0), "=f"(n1) : "l"(n));
}

__device__ __forceinline__ uint2 encode8_mul(const float (&f)[8], float m) {
    uint2 r;
    r.x = e4m3x2(__fmul_rn(f[0], m), __fmul_rn(f[1], m)) | (e4m3x2(__fmul_rn(f[2], m), __fmul_rn(f[3], m)) << 16);
    r.y = e4m3x2(__fmul_rn(f[4], m), __fmul_rn(f[5], m)) | (e4m3x2(__fmul_rn(f[6], m), __fmul_rn(f[7], m)) << 16);
    return r;
}

}  // namespace fp8bs
