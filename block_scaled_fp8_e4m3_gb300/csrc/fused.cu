// Producers fused with the activation quantization ("Jet-RL: Enabling
// On-Policy FP8 Reinforcement Learning with Unified Training and Rollout
// Precision Flow", section "Kwantisatieschema": the activations kept for the
// backward pass are stored in FP8, fused with the operator that produces
// them; section "Implementatie": fused activation and RMSNorm kernels).
//
// Each kernel computes its producer in fp32, rounds the result to bf16 (the
// tensor an unfused pipeline would hand to the quantizer), optionally writes
// it, and quantizes those bf16 values in registers: 1x128 groups with fp32
// scales, 1x128 groups with power-of-two scales, or MXFP8 1x32 blocks.  A
// 128-element group is held by 16 lanes (8 values each), so its maximum is a
// 4-step shuffle inside a half warp; a 1x32 block is 4 lanes.
#include "common.cuh"
#include "kernels.h"
#include "quant_common.cuh"

namespace fp8bs {

namespace {

enum : int { kRecFp32 = 0, kRecPow2 = 1, kRecMx = 2 };

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// Rounds 8 fp32 results to bf16: returns the packed words and, in f, the
// rounded values as fp32 (what the quantizer sees).
__device__ __forceinline__ uint4 round8_bf16(float (&f)[8]) {
    uint4 w;
    w.x = pack_bf16x2(f[0], f[1]);
    w.y = pack_bf16x2(f[2], f[3]);
    w.z = pack_bf16x2(f[4], f[5]);
    w.w = pack_bf16x2(f[6], f[7]);
    unpack8(w, f);
    return w;
}

// Quantizes the 8 values of this lane, part of the 128-element group g of
// row r held by the 16 lanes of a half warp (sub = lane % 16 holds elements
// 8 sub .. 8 sub + 7 of the group).  All 32 lanes of the warp must call it
// (the reductions are warp shuffles); a half warp with ok = false holds no
// group and writes nothing.  Otherwise writes the lane's 8 codes at `codes`
// and the group's scale(s).
template <int kRec>
__device__ __forceinline__ void quant_group16(const float (&y)[8], bool ok, int sub, int64_t r, int64_t g, int64_t M,
                                              int64_t atoms_k, uint8_t* codes, void* scales) {
    uint2 c;
    if (kRec == kRecMx) {
        float a = amax8(y);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const int e = mx_exponent(a);
        c = encode8_mul(y, exp2_int(-e));
        // the four block exponents of the group (lanes sub = 0, 4, 8, 12)
        const int base = threadIdx.x & 16;
        const uint32_t b = (uint32_t)(e + 127);
        const uint32_t b1 = __shfl_sync(0xffffffffu, b, base + 4, 32);
        const uint32_t b2 = __shfl_sync(0xffffffffu, b, base + 8, 32);
        const uint32_t b3 = __shfl_sync(0xffffffffu, b, base + 12, 32);
        if (ok && sub == 0)
            *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scales) + mx_scale_offset(r, 4 * g, atoms_k)) =
                b | (b1 << 8) | (b2 << 16) | (b3 << 24);
    } else {
        float a = amax8(y);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (kRec == kRecPow2) {
            const int e = pow2_exponent(a);
            c = encode8_mul(y, exp2_int(-e));
            if (ok && sub == 0)
                *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scales) + mx_scale_offset(r, 4 * g, atoms_k)) =
                    (uint32_t)(e + 127) * 0x01010101u;
        } else {
            const float s = group_scale_bf16(a);
            c = encode8_div(y, make_divider(s));
            if (ok && sub == 0) static_cast<float*>(scales)[g * M + r] = s;
        }
    }
    if (ok) *reinterpret_cast<uint2*>(codes) = c;
}

// ---------------------------------------------------------------------------
// RMSNorm + quantization.  One warp per row, 8 rows per 256-thread block.
// Lane l holds chunks j < kChunks: elements 256 j + 8 l .. + 7 (each chunk is
// one 512-byte warp access); K % 128 == 0, so the last chunk is whole or its
// upper half warp idles.  Sum of squares in fp32 (per lane, then a warp
// reduction), rstd = RN(1/sqrt(RN(ss/K) + eps)), y = RN_bf16(RN(x rstd) gamma).
// ---------------------------------------------------------------------------
template <int kRec, int kChunks>
__global__ void __launch_bounds__(256, kChunks <= 8 ? 2 : 1) k_rmsnorm_quant(const uint16_t* __restrict__ x,
                                                       const uint16_t* __restrict__ gamma, int64_t M, int64_t K,
                                                       int64_t ld, float eps, uint16_t* __restrict__ y,
                                                       int64_t ldy, float* __restrict__ rstd_out,
                                                       uint8_t* __restrict__ codes, void* __restrict__ scales) {
    __shared__ __align__(16) uint16_t sgamma[256 * kChunks];
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    for (int64_t k = 8 * threadIdx.x; k < K; k += 8 * 256)
        *reinterpret_cast<uint4*>(sgamma + k) = *reinterpret_cast<const uint4*>(gamma + k);
    __syncthreads();
    if (r >= M) return;
    const uint16_t* xr = x + r * ld;
    uint4 v[kChunks];
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
        const int64_t k = 256 * j + 8 * lane;
        v[j] = k < K ? ld_stream_v4(xr + k) : make_uint4(0, 0, 0, 0);
    }
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
        float f[8];
        unpack8(v[j], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = __fmaf_rn(f[i], f[i], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float rs = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)K), eps));
    if (rstd_out != nullptr && lane == 0) rstd_out[r] = rs;
    const int64_t atoms_k = (K + 127) / 128;
    const int sub = lane & 15;
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
        const int64_t k = 256 * j + 8 * lane;
        if (256 * j >= K) break;                         // warp-uniform
        const bool ok = k < K;                           // false only for the upper half of a last half chunk
        float f[8], gm[8];
        unpack8(v[j], f);
        unpack8(ok ? *reinterpret_cast<const uint4*>(sgamma + k) : make_uint4(0, 0, 0, 0), gm);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __fmul_rn(__fmul_rn(f[i], rs), gm[i]);
        const uint4 w = round8_bf16(f);
        if (y != nullptr && ok) *reinterpret_cast<uint4*>(y + r * ldy + k) = w;
        quant_group16<kRec>(f, ok, sub, r, k / 128, M, atoms_k, codes + r * K + k, scales);
    }
}

// ---------------------------------------------------------------------------
// SwiGLU + quantization.  gu [M][ld] holds the gate projection in columns
// [0, F) and the up projection in [F, 2F); h = RN_bf16(silu(g) u) with
// silu(g) = g sigmoid(g), sigmoid from e = exp(-|g|) as 1/(1+e) for g >= 0
// and e/(1+e) for g < 0 (no overflow for large |g|).  Work unit = one
// 128-element group of one row (16 lanes); a 256-thread block takes 16 units
// per round, 4 rounds with all loads issued first.
// ---------------------------------------------------------------------------
constexpr int kSwRounds = 4;

__device__ __forceinline__ float silu_times(float g, float u) {
    const float e = expf(-fabsf(g));
    const float d = __fadd_rn(1.0f, e);
    const float sg = __fdiv_rn(g >= 0.0f ? 1.0f : e, d);
    return __fmul_rn(__fmul_rn(g, sg), u);
}

template <int kRec>
__global__ void __launch_bounds__(256) k_swiglu_quant(const uint16_t* __restrict__ gu, int64_t M, int64_t F,
                                                      int64_t ld, uint16_t* __restrict__ h, int64_t ldh,
                                                      uint8_t* __restrict__ codes, void* __restrict__ scales) {
    const int64_t G = F / 128, units = M * G;
    const int sub = threadIdx.x & 15;
    const int64_t atoms_k = (F + 127) / 128;
    uint4 vg[kSwRounds], vu[kSwRounds];
#pragma unroll
    for (int i = 0; i < kSwRounds; ++i) {
        const int64_t u = ((int64_t)blockIdx.x * kSwRounds + i) * 16 + (threadIdx.x >> 4);
        if (u < units) {
            const int64_t r = u / G, k = (u % G) * 128 + 8 * sub;
            vg[i] = ld_stream_v4(gu + r * ld + k);
            vu[i] = ld_stream_v4(gu + r * ld + F + k);
        } else {
            vg[i] = vu[i] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int i = 0; i < kSwRounds; ++i) {
        const int64_t u = ((int64_t)blockIdx.x * kSwRounds + i) * 16 + (threadIdx.x >> 4);
        if (((int64_t)blockIdx.x * kSwRounds + i) * 16 >= units) break;   // block-uniform
        const bool ok = u < units;
        const int64_t r = ok ? u / G : 0, g = ok ? u % G : 0, k = g * 128 + 8 * sub;
        float fg[8], fu[8];
        unpack8(vg[i], fg);
        unpack8(vu[i], fu);
#pragma unroll
        for (int q = 0; q < 8; ++q) fg[q] = silu_times(fg[q], fu[q]);
        const uint4 w = round8_bf16(fg);
        if (h != nullptr && ok) *reinterpret_cast<uint4*>(h + r * ldh + k) = w;
        quant_group16<kRec>(fg, ok, sub, r, g, M, atoms_k, codes + r * F + k, scales);
    }
}

template <int kRec>
cudaError_t launch_rmsnorm_rec(const uint16_t* x, const uint16_t* gamma, int64_t M, int64_t K, int64_t ld, float eps,
                               uint16_t* y, int64_t ldy, float* rstd, uint8_t* codes, void* scales,
                               cudaStream_t st) {
    const unsigned blocks = (unsigned)((M + 7) / 8);
    const int chunks = (int)((K + 255) / 256);
#define FP8BS_RMS(C) k_rmsnorm_quant<kRec, C><<<blocks, 256, 0, st>>>(x, gamma, M, K, ld, eps, y, ldy, rstd, codes, scales)
    if (chunks <= 1) FP8BS_RMS(1);
    else if (chunks <= 2) FP8BS_RMS(2);
    else if (chunks <= 4) FP8BS_RMS(4);
    else if (chunks <= 8) FP8BS_RMS(8);
    else if (chunks <= 16) FP8BS_RMS(16);
    else FP8BS_RMS(32);
#undef FP8BS_RMS
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, int64_t M, int64_t K, int64_t ld,
                                 float eps, uint16_t* y, int64_t ldy, float* rstd, uint8_t* codes, void* scales,
                                 int recipe, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    if (recipe != kRecFp32) {
        cudaError_t e = zero_mx_tail(scales, M, K, st);
        if (e != cudaSuccess) return e;
    }
    if (recipe == kRecPow2) return launch_rmsnorm_rec<kRecPow2>(x, gamma, M, K, ld, eps, y, ldy, rstd, codes, scales, st);
    if (recipe == kRecMx) return launch_rmsnorm_rec<kRecMx>(x, gamma, M, K, ld, eps, y, ldy, rstd, codes, scales, st);
    return launch_rmsnorm_rec<kRecFp32>(x, gamma, M, K, ld, eps, y, ldy, rstd, codes, scales, st);
}

cudaError_t launch_swiglu_quant(const uint16_t* gu, int64_t M, int64_t F, int64_t ld, uint16_t* h, int64_t ldh,
                                uint8_t* codes, void* scales, int recipe, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    if (recipe != kRecFp32) {
        cudaError_t e = zero_mx_tail(scales, M, F, st);
        if (e != cudaSuccess) return e;
    }
    const int64_t units = M * (F / 128);
    const unsigned blocks = (unsigned)((units + 16 * kSwRounds - 1) / (16 * kSwRounds));
    if (recipe == kRecPow2)
        k_swiglu_quant<kRecPow2><<<blocks, 256, 0, st>>>(gu, M, F, ld, h, ldh, codes, scales);
    else if (recipe == kRecMx)
        k_swiglu_quant<kRecMx><<<blocks, 256, 0, st>>>(gu, M, F, ld, h, ldh, codes, scales);
    else
        k_swiglu_quant<kRecFp32><<<blocks, 256, 0, st>>>(gu, M, F, ld, h, ldh, codes, scales);
    return cudaGetLastError();
}

}  // namespace fp8bs
