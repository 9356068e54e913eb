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
// 128-element group is held by 8 lanes (16 values each), so its maximum is a
// 3-step shuffle; a 1x32 block is the same half of 4 lanes.
#include "common.cuh"
#include "kernels.h"
#include "quant_common.cuh"

namespace fp8bs {

namespace {

enum : int { kRecFp32 = 0, kRecPow2 = 1, kRecMx = 2 };

// Two fp32 values rounded to bf16 (nearest, ties to even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t w;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
    return w;
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

// Packed fp32 pair arithmetic (one instruction for two lanes of a float2).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    uint64_t x, y, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
    return r;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t x, y, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(b.x), "f"(b.y));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(y));
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
    return r;
}

// A bf16 pair (low element in the low half) as an fp32 pair in one 64-bit
// register, ready for the packed fp32x2 instructions.
__device__ __forceinline__ uint64_t bf16x2_f32x2(uint32_t w) {
    uint64_t r;
    asm("{\n\t.reg .b32 lo, hi;\n\tshl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xFFFF0000;\n\tmov.b64 %0, {lo, hi};\n\t}"
        : "=l"(r)
        : "r"(w));
    return r;
}

// An fp32 pair rounded to a bf16 pair (nearest, ties to even).
__device__ __forceinline__ uint32_t f32x2_bf16x2(uint64_t p) {
    uint32_t w;
    asm("{\n\t.reg .f32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\tcvt.rn.bf16x2.f32 %0, hi, lo;\n\t}" : "=r"(w) : "l"(p));
    return w;
}

__device__ __forceinline__ uint64_t fma2_rn(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t mul2_rn(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// RMSNorm + quantization.  A row is split into segments of 1024 elements,
// one warp each (kW warps per row, a power of two >= K/1024; 8/kW rows per
// 256-thread block).  A segment is two rounds of four 128-element groups,
// eight lanes per group: lane (gq = l/8, sub = l%8) holds elements
// 8 sub .. 8 sub + 7 and 64 + 8 sub .. 64 + 8 sub + 7 of group gq of each
// round (so each 16-byte load instruction of the warp covers four whole
// 128-byte lines), 16 values of one group per lane and round.  The sum of
// squares is accumulated in fp32 per lane, reduced over the warp, and the kW
// warp partials of a row are added in segment order through shared memory
// (every warp of the row gets the same sum); rstd = RN(1/sqrt(RN(ss/K) +
// eps)), y = RN_bf16(RN(x rstd) gamma).  The group's maximum is a 3-step
// shuffle inside the eight lanes; a 1x32 block is the same half of four
// lanes.
// ---------------------------------------------------------------------------
template <int kRec>
__device__ __forceinline__ void quant_group8x16(float (&f)[2][8], bool ok, int sub, int64_t r, int64_t g,
                                                int64_t M, int64_t atoms_k, uint8_t* codes, void* scales) {
    uint2 c[2];
    if (kRec == kRecMx) {
        // halves h = 0, 1 lie in 1x32 blocks (sub / 4) and 2 + (sub / 4)
        int e[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float a = amax8(f[h]);
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            e[h] = mx_exponent(a);
            c[h] = encode8_mul(f[h], exp2_int(-e[h]));
        }
        const uint32_t b0 = (uint32_t)(e[0] + 127), b2 = (uint32_t)(e[1] + 127);
        const int src = (threadIdx.x & 31) + 4;  // lane sub + 4: blocks 1 and 3 (used by sub = 0 only)
        const uint32_t b1 = __shfl_sync(0xffffffffu, b0, src & 31);
        const uint32_t b3 = __shfl_sync(0xffffffffu, b2, src & 31);
        if (ok && sub == 0)
            *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scales) + mx_scale_offset(r, 4 * g, atoms_k)) =
                b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    } else {
        float a = fmaxf(amax8(f[0]), amax8(f[1]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        if (kRec == kRecPow2) {
            const int e = pow2_exponent(a);
#pragma unroll
            for (int h = 0; h < 2; ++h) c[h] = encode8_mul(f[h], exp2_int(-e));
            if (ok && sub == 0)
                *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scales) + mx_scale_offset(r, 4 * g, atoms_k)) =
                    (uint32_t)(e + 127) * 0x01010101u;
        } else {
            const float s = group_scale_bf16(a);
            const Divider dv = make_divider(s);
#pragma unroll
            for (int h = 0; h < 2; ++h) c[h] = encode8_div(f[h], dv);
            if (ok && sub == 0) static_cast<float*>(scales)[g * M + r] = s;
        }
    }
    if (ok) {
        *reinterpret_cast<uint2*>(codes) = c[0];
        *reinterpret_cast<uint2*>(codes + 64) = c[1];
    }
}

template <int kRec, int kW>
__global__ void __launch_bounds__(256, 4) k_rmsnorm_quant(const uint16_t* __restrict__ x,
                                                          const uint16_t* __restrict__ gamma, int64_t M, int64_t K,
                                                          int64_t ld, float eps, uint16_t* __restrict__ y,
                                                          int64_t ldy, float* __restrict__ rstd_out,
                                                          uint8_t* __restrict__ codes, void* __restrict__ scales) {
    __shared__ float part[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = warp % kW;
    const int64_t r = (int64_t)blockIdx.x * (8 / kW) + warp / kW;
    const bool row_ok = r < M;
    const int gq = lane >> 3, sub = lane & 7;
    const uint16_t* xr = x + r * ld;
    // element of round j, half h: seg*1024 + j*512 + gq*128 + 64h + 8sub
    const int64_t e0 = (int64_t)seg * 1024 + gq * 128 + 8 * sub;
    uint4 v[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t k = e0 + 512 * j + 64 * h;
            v[j][h] = (row_ok && k < K) ? ld_stream_v4(xr + k) : make_uint4(0, 0, 0, 0);
        }
    // sum of squares: even and odd elements in the two halves of a packed pair
    uint64_t ss2 = 0ull;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t wd[4] = {v[j][h].x, v[j][h].y, v[j][h].z, v[j][h].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint64_t p = bf16x2_f32x2(wd[q]);
                ss2 = fma2_rn(p, p, ss2);
            }
        }
    float ss;
    {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(ss2));
        ss = __fadd_rn(lo, hi);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    if (kW > 1) {
        if (lane == 0) part[warp] = ss;
        __syncthreads();
        const int w0 = warp - seg;
        ss = part[w0];
#pragma unroll
        for (int i = 1; i < kW; ++i) ss = __fadd_rn(ss, part[w0 + i]);
    }
    if (!row_ok) return;
    const float rs = __frsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)K), eps));
    if (rstd_out != nullptr && seg == 0 && lane == 0) rstd_out[r] = rs;
    const int64_t atoms_k = (K + 127) / 128;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int64_t g0 = (int64_t)seg * 1024 + 512 * j;  // first element of the round
        if (g0 >= K) break;                                // warp-uniform: the round is empty
        const int64_t k = e0 + 512 * j;                     // this lane's first element
        const bool ok = k < K;                              // K % 128 == 0: the lane's group is whole or absent
        float f[2][8];
        uint64_t rs2;
        asm("mov.b64 %0, {%1, %1};" : "=l"(rs2) : "f"(rs));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 gv = ok ? __ldg(reinterpret_cast<const uint4*>(gamma + k + 64 * h)) : make_uint4(0, 0, 0, 0);
            const uint32_t xw[4] = {v[j][h].x, v[j][h].y, v[j][h].z, v[j][h].w};
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            uint32_t yw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // y = RN_bf16(RN(x rstd) gamma), two elements per instruction
                yw[q] = f32x2_bf16x2(mul2_rn(mul2_rn(bf16x2_f32x2(xw[q]), rs2), bf16x2_f32x2(gw[q])));
                f[h][2 * q] = bf16_lo(yw[q]);
                f[h][2 * q + 1] = bf16_hi(yw[q]);
            }
            if (y != nullptr && ok) *reinterpret_cast<uint4*>(y + r * ldy + k + 64 * h) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
        }
        quant_group8x16<kRec>(f, ok, sub, r, k / 128, M, atoms_k, codes + r * K + k, scales);
    }
}

// ---------------------------------------------------------------------------
// SwiGLU + quantization.  gu [M][ld] holds the gate projection in columns
// [0, F) and the up projection in [F, 2F); h = RN_bf16(silu(g) u) with
// silu(g) = g sigmoid(g), sigmoid from e = exp(-|g|) as 1/(1+e) for g >= 0
// and e/(1+e) for g < 0 (no overflow for large |g|); h is within one bf16
// step of the exact value.  Work unit = one
// 128-element group of one row, eight lanes with 16 values each (elements
// 8 sub .. and 64 + 8 sub .., as in the RMSNorm kernel); a 256-thread block
// takes 32 units per round, 2 rounds with all loads issued first.
// ---------------------------------------------------------------------------
constexpr int kSwRounds = 2;

// silu(g) u for 8 pairs in fp32: sigmoid(g) = 1 / (1 + 2^(-g log2 e)) with
// the hardware base-2 exponential and reciprocal approximations (relative
// error below 2^-17 for |g| < 90, against the 2^-9 that would move the
// bf16 result by more than one step), two lanes per packed instruction.
// Below g = -80 the reciprocal of 1 + e would leave the normal range, so
// that (rare) tail is recomputed as e/(1+e) with e = expf(g), in a branch
// taken only by threads that hold such a value.
__device__ __forceinline__ void silu_times8(float (&g)[8], const float (&u)[8]) {
    constexpr float kNegLog2e = -1.4426950408889634f;
#pragma unroll
    for (int q = 0; q < 8; q += 2) {
        const float2 t = mul2(make_float2(g[q], g[q + 1]), make_float2(kNegLog2e, kNegLog2e));
        const float2 d = add2(make_float2(ex2_approx(t.x), ex2_approx(t.y)), make_float2(1.0f, 1.0f));
        const float2 sg = make_float2(rcp_approx(d.x), rcp_approx(d.y));
        const float2 h = mul2(mul2(make_float2(g[q], g[q + 1]), sg), make_float2(u[q], u[q + 1]));
        g[q] = h.x;
        g[q + 1] = h.y;
    }
}

template <int kRec>
__global__ void __launch_bounds__(256, 4) k_swiglu_quant(const uint16_t* __restrict__ gu, int64_t M, int64_t F,
                                                      int64_t ld, uint16_t* __restrict__ h, int64_t ldh,
                                                      uint8_t* __restrict__ codes, void* __restrict__ scales) {
    const int64_t G = F / 128, units = M * G;
    const int sub = threadIdx.x & 7;
    const int64_t atoms_k = (F + 127) / 128;
    const int64_t unit0 = (int64_t)blockIdx.x * kSwRounds * 32 + (threadIdx.x >> 3);
    // (row, group) of each round's unit: one division, then steps of 32 units
    int64_t rr[kSwRounds], gg[kSwRounds];
    rr[0] = unit0 / G;
    gg[0] = unit0 - rr[0] * G;
#pragma unroll
    for (int i = 1; i < kSwRounds; ++i) {
        rr[i] = rr[i - 1];
        gg[i] = gg[i - 1] + 32;
        while (gg[i] >= G) {
            gg[i] -= G;
            ++rr[i];
        }
    }
    uint4 vg[kSwRounds][2], vu[kSwRounds][2];
#pragma unroll
    for (int i = 0; i < kSwRounds; ++i)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            if (unit0 + 32 * i < units) {
                const uint16_t* p = gu + rr[i] * ld + gg[i] * 128 + 64 * hh + 8 * sub;
                vg[i][hh] = ld_stream_v4(p);
                vu[i][hh] = ld_stream_v4(p + F);
            } else {
                vg[i][hh] = vu[i][hh] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
    for (int i = 0; i < kSwRounds; ++i) {
        if (unit0 - (threadIdx.x >> 3) + 32 * i >= units) break;   // block-uniform
        const bool ok = unit0 + 32 * i < units;
        const int64_t r = ok ? rr[i] : 0, g = ok ? gg[i] : 0, k = g * 128 + 8 * sub;
        float fg[2][8];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float fu[8];
            unpack8(vg[i][hh], fg[hh]);
            unpack8(vu[i][hh], fu);
            const float gmin = fminf(fminf(fminf(fg[hh][0], fg[hh][1]), fminf(fg[hh][2], fg[hh][3])),
                                     fminf(fminf(fg[hh][4], fg[hh][5]), fminf(fg[hh][6], fg[hh][7])));
            float gsave[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) gsave[q] = fg[hh][q];
            silu_times8(fg[hh], fu);
            if (gmin < -80.0f) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (gsave[q] < -80.0f) {
                        const float e = expf(gsave[q]);
                        fg[hh][q] = __fmul_rn(__fmul_rn(gsave[q], __fdiv_rn(e, __fadd_rn(1.0f, e))), fu[q]);
                    }
            }
            const uint4 w = round8_bf16(fg[hh]);
            if (h != nullptr && ok) *reinterpret_cast<uint4*>(h + r * ldh + k + 64 * hh) = w;
        }
        quant_group8x16<kRec>(fg, ok, sub, r, g, M, atoms_k, codes + r * F + k, scales);
    }
}

template <int kRec>
cudaError_t launch_rmsnorm_rec(const uint16_t* x, const uint16_t* gamma, int64_t M, int64_t K, int64_t ld, float eps,
                               uint16_t* y, int64_t ldy, float* rstd, uint8_t* codes, void* scales,
                               cudaStream_t st) {
    const int64_t segs = (K + 1023) / 1024;
    const int w = segs <= 1 ? 1 : segs <= 2 ? 2 : segs <= 4 ? 4 : 8;
    const unsigned blocks = (unsigned)((M + (8 / w) - 1) / (8 / w));
#define FP8BS_RMS(W) k_rmsnorm_quant<kRec, W><<<blocks, 256, 0, st>>>(x, gamma, M, K, ld, eps, y, ldy, rstd, codes, scales)
    if (w == 1) FP8BS_RMS(1);
    else if (w == 2) FP8BS_RMS(2);
    else if (w == 4) FP8BS_RMS(4);
    else FP8BS_RMS(8);
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
    const unsigned blocks = (unsigned)((units + 32 * kSwRounds - 1) / (32 * kSwRounds));
    if (recipe == kRecPow2)
        k_swiglu_quant<kRecPow2><<<blocks, 256, 0, st>>>(gu, M, F, ld, h, ldh, codes, scales);
    else if (recipe == kRecMx)
        k_swiglu_quant<kRecMx><<<blocks, 256, 0, st>>>(gu, M, F, ld, h, ldh, codes, scales);
    else
        k_swiglu_quant<kRecFp32><<<blocks, 256, 0, st>>>(gu, M, F, ld, h, ldh, codes, scales);
    return cudaGetLastError();
}

}  // namespace fp8bs
