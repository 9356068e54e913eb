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
    float q[8];
    if (d.fast) {
#pragma unroll
        for (int k = 0; k < 4; ++k) quotient2_fast(d, f[2 * k], f[2 * k + 1], q[2 * k], q[2 * k + 1]);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = __fdiv_rn(f[k], d.s);
    }
    uint2 r;
    r.x = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
    r.y = e4m3x2(q[4], q[5]) | (e4m3x2(q[6], q[7]) << 16);
    return r;
}

__device__ __forceinline__ uint2 encode8_mul(const float (&f)[8], float m) {
    uint2 r;
    r.x = e4m3x2(__fmul_rn(f[0], m), __fmul_rn(f[1], m)) | (e4m3x2(__fmul_rn(f[2], m), __fmul_rn(f[3], m)) << 16);
    r.y = e4m3x2(__fmul_rn(f[4], m), __fmul_rn(f[5], m)) | (e4m3x2(__fmul_rn(f[6], m), __fmul_rn(f[7], m)) << 16);
    return r;
}

}  // namespace fp8bs
