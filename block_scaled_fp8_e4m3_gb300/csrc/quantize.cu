// quantize.cu -- HBM-streaming quantizers (bf16 -> E4M3 codes + scales).
//
// Every kernel reads each bf16 element once with 16-byte coalesced loads,
// reduces the group maximum on chip (warp shuffles, or shared memory for
// groups that span warps), encodes with the hardware round-to-nearest-even
// saturating E4M3 conversion, and writes codes and scales once.  Algorithmic
// traffic: 2 B read + 1 B code per element + the scales.
//
// Scale conventions (see fp8bs.h): blockwise s = amax/448 by IEEE fp32
// division and codes from the IEEE fp32 quotient x/s ("AIS: Adaptive
// Importance Sampling for Quantized RL" explainer, equation Q(X)); MX
// e = floor(log2 amax) - 8 read from the exponent bits and codes from the
// exact product x * 2^-e.
#include "common.cuh"
#include "kernels.h"
#include "quant_common.cuh"

namespace fp8bs {

namespace {

// ---------------------------------------------------------------------------
// 1x128 groups along K.  Block = 256 threads = 32 rows x 4 consecutive
// groups; eight lanes share a row's group, each holding 16 of its bf16 values
// (elements 8*sub.. and 64 + 8*sub.., so that every 16-byte load instruction
// covers whole 128-byte lines).  All eight loads of a thread are issued before
// any arithmetic; the per-group work (maximum over 8 lanes, scale, reciprocal)
// is spread over 16 values per lane.
// ---------------------------------------------------------------------------
constexpr int kGK_Groups = 4;
constexpr int kGK_Rows = 32;

// 16 values of one group of one lane: two 8-value halves, encoded into two
// 8-byte code words.
__device__ __forceinline__ void encode16(const uint4 (&v)[2], const Divider& d, uint2 (&c)[2]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float f[8];
        unpack8(v[h], f);
        c[h] = encode8_div(f, d);
    }
}

// kPow2: power-of-two scales, E8M0 bytes in the MX layout, each group's
// byte in its four 1x32 slots (one 32-bit store per row and group).
template <bool kPow2>
__global__ void __launch_bounds__(256, 4) k_quant_group_k(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                          int64_t ld, uint8_t* __restrict__ codes,
                                                          void* __restrict__ scales) {
    const int G = (int)(K / 128);
    const int gchunks = (G + kGK_Groups - 1) / kGK_Groups;
    const int strip = (int)(blockIdx.x / (unsigned)gchunks);
    const int g0 = (int)(blockIdx.x - (unsigned)strip * gchunks) * kGK_Groups;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 7;
    const int64_t row = (int64_t)strip * kGK_Rows + warp * 4 + (lane >> 3);
    const bool row_ok = row < M;
    const uint16_t* xr = x + row * ld + sub * 8;

    uint4 v[kGK_Groups][2];
#pragma unroll
    for (int u = 0; u < kGK_Groups; ++u) {
        const bool ok = row_ok && g0 + u < G;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            v[u][h] = ok ? ld_stream_v4(xr + (g0 + u) * 128 + h * 64) : make_uint4(0, 0, 0, 0);
    }
    uint8_t* cr = codes + row * K + sub * 8;
#pragma unroll
    for (int u = 0; u < kGK_Groups; ++u) {
        const int g = g0 + u;
        float a = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float f[8];
            unpack8(v[u][h], f);
            a = fmaxf(a, amax8(f));
        }
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        uint2 c[2];
        if (kPow2) {
            const int e = pow2_exponent(a);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float f[8];
                unpack8(v[u][h], f);
                c[h] = encode8_mul(f, exp2_int(-e));
            }
            if (row_ok && g < G) {
                *reinterpret_cast<uint2*>(cr + g * 128) = c[0];
                *reinterpret_cast<uint2*>(cr + g * 128 + 64) = c[1];
                if (sub == 0)
                    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scales) + mx_scale_offset(row, 4 * g, G)) =
                        (uint32_t)(e + 127) * 0x01010101u;
            }
        } else {
            const float sc = group_scale_bf16(a);
            encode16(v[u], make_divider(sc), c);
            if (row_ok && g < G) {
                *reinterpret_cast<uint2*>(cr + g * 128) = c[0];
                *reinterpret_cast<uint2*>(cr + g * 128 + 64) = c[1];
                if (sub == 0) static_cast<float*>(scales)[(int64_t)g * M + row] = sc;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 128x1 groups along M, codes transposed.  Block = one 128-row x 64-column
// tile; thread (chunk = t%8, quad = t/8) holds rows 4*quad..4*quad+3 of
// columns 8*chunk..8*chunk+7.  Column maxima: in-thread over 4 rows, shuffle
// over the 4 quads of a warp, shared memory over the 8 warps.  The codes of
// a column's 4 rows form one 32-bit word of the transposed tile in shared
// memory (column stride 33 words), which is written out 16 bytes per thread.
// ---------------------------------------------------------------------------
template <bool kPow2>
__global__ void __launch_bounds__(256, 5) k_quant_group_m(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                       int64_t ld, uint8_t* __restrict__ codes_t,
                                                       void* __restrict__ scales) {
    __shared__ float red[8][64];
    __shared__ float col_scale[64], col_nrcp[64];
    __shared__ uint32_t tile[64 * 33];

    const int64_t ctiles = (K + 63) / 64;
    const int64_t mb = (int64_t)blockIdx.x / ctiles;
    const int64_t c0 = ((int64_t)blockIdx.x % ctiles) * 64;
    const int64_t m0 = mb * 128;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int chunk = t & 7, quad = t >> 3;
    const bool col_ok = c0 + chunk * 8 < K;  // K % 8 == 0: a chunk is all valid or all invalid

    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = col_ok ? ld_stream_v4(x + (m0 + quad * 4 + i) * ld + c0 + chunk * 8) : make_uint4(0, 0, 0, 0);

    float f[4][8];
    float pa[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack8(v[i], f[i]);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a = fmaxf(fmaxf(fabsf(f[0][j]), fabsf(f[1][j])), fmaxf(fabsf(f[2][j]), fabsf(f[3][j])));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
        pa[j] = a;
    }
    if (lane < 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) red[warp][chunk * 8 + j] = pa[j];
    }
    __syncthreads();
    if (t < 64) {
        float a = red[0][t];
#pragma unroll
        for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w][t]);
        if (kPow2) {
            // transposed row c0+t of the [K][M] output, 1x32 blocks 4mb..4mb+3
            const int e = pow2_exponent(a);
            col_scale[t] = exp2_int(-e);
            if (c0 + t < K)
                *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(scales) + mx_scale_offset(c0 + t, 4 * mb, M / 128)) =
                    (uint32_t)(e + 127) * 0x01010101u;
        } else {
            const float s = group_scale_bf16(a);
            col_scale[t] = s;
            col_nrcp[t] = -__frcp_rn(s);
            if (c0 + t < K) static_cast<float*>(scales)[mb * K + c0 + t] = s;
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float q[4];
        if (kPow2) {
            const float mul = col_scale[chunk * 8 + j];  // exact power of two
#pragma unroll
            for (int i = 0; i < 4; ++i) q[i] = __fmul_rn(f[i][j], mul);
            tile[(chunk * 8 + j) * 33 + quad] = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
            continue;
        }
        Divider dv;
        dv.s = col_scale[chunk * 8 + j];
        dv.nr = col_nrcp[chunk * 8 + j];
        dv.fast = dv.s >= 0x1p-100f && dv.s <= 3.402823466e38f;
        if (dv.fast) {
            tile[(chunk * 8 + j) * 33 + quad] = codes4_div_fast(dv, f[0][j], f[1][j], f[2][j], f[3][j]);
            continue;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = __fdiv_rn(f[i][j], dv.s);
        tile[(chunk * 8 + j) * 33 + quad] = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = t + 256 * i;
        const int col = idx >> 3, part = idx & 7;
        if (c0 + col < K) {
            uint4 o;
            o.x = tile[col * 33 + part * 4 + 0];
            o.y = tile[col * 33 + part * 4 + 1];
            o.z = tile[col * 33 + part * 4 + 2];
            o.w = tile[col * 33 + part * 4 + 3];
            *reinterpret_cast<uint4*>(codes_t + (c0 + col) * M + m0 + part * 16) = o;
        }
    }
}

// ---------------------------------------------------------------------------
// WGrad operand from a saved 1x128 FP8 activation ("Jet-RL", section
// "Kwantisatieschema": activations are kept in FP8 for the backward pass;
// WGrad takes 128x1 groups along M): each element is dequantized once in
// fp32, x' = RN(dec(q) s_row) (the E4M3 -> f16 conversion is exact), and x'
// is quantized in 128x1 groups with the codes transposed.  The tiling is that
// of k_quant_group_m (128 rows x 64 columns, one 1x128 scale per row); x' has
// a full fp32 significand: the scales are IEEE divisions and the quotients
// come from neg_quotient2_exact (the IEEE quotient bit for bit).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 5) k_requant_group_m(const uint8_t* __restrict__ codes, const float* __restrict__ rs,
                                                         int64_t M, int64_t K, uint8_t* __restrict__ codes_t,
                                                         float* __restrict__ scales_t) {
    __shared__ float red[8][64];
    __shared__ float col_scale[64], col_nrcp[64];
    __shared__ uint32_t tile[64 * 33];

    const int64_t ctiles = K / 64;
    const int64_t mb = (int64_t)blockIdx.x / ctiles;
    const int64_t c0 = ((int64_t)blockIdx.x % ctiles) * 64;
    const int64_t m0 = mb * 128;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int chunk = t & 7, quad = t >> 3;

    uint2 v[4];
    float srow[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + quad * 4 + i;
        v[i] = __ldcs(reinterpret_cast<const uint2*>(codes + m * K + c0 + chunk * 8));
        srow[i] = __ldg(rs + (c0 / 128) * M + m);
    }
    float f[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[2] = {v[i].x, v[i].y};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[h >> 1] >> (16 * (h & 1))), __NV_E4M3);
            const float2 d = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            f[i][2 * h] = __fmul_rn(d.x, srow[i]);
            f[i][2 * h + 1] = __fmul_rn(d.y, srow[i]);
        }
    }
    float pa[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a = fmaxf(fmaxf(fmaxf(0.0f, fabsf(f[0][j])), fabsf(f[1][j])), fmaxf(fabsf(f[2][j]), fabsf(f[3][j])));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
        pa[j] = a;
    }
    if (lane < 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) red[warp][chunk * 8 + j] = pa[j];
    }
    __syncthreads();
    if (t < 64) {
        float a = red[0][t];
#pragma unroll
        for (int w = 1; w < 8; ++w) a = fmaxf(a, red[w][t]);
        const float sc = group_scale(a);
        col_scale[t] = sc;
        col_nrcp[t] = -__frcp_rn(sc);
        scales_t[mb * K + c0 + t] = sc;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float sc = col_scale[chunk * 8 + j];
        uint32_t word;
        if (sc >= 0x1p-90f && sc <= 0x1p126f) {
            float n[4];
            neg_quotient2_exact(f[0][j], f[1][j], sc, col_nrcp[chunk * 8 + j], n[0], n[1]);
            neg_quotient2_exact(f[2][j], f[3][j], sc, col_nrcp[chunk * 8 + j], n[2], n[3]);
            word = (e4m3x2(n[0], n[1]) | (e4m3x2(n[2], n[3]) << 16)) ^ 0x80808080u;  // codes of -n: sign back
        } else {
            word = e4m3x2(__fdiv_rn(f[0][j], sc), __fdiv_rn(f[1][j], sc)) |
                   (e4m3x2(__fdiv_rn(f[2][j], sc), __fdiv_rn(f[3][j], sc)) << 16);
        }
        tile[(chunk * 8 + j) * 33 + quad] = word;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = t + 256 * i;
        const int col = idx >> 3, part = idx & 7;
        uint4 o;
        o.x = tile[col * 33 + part * 4 + 0];
        o.y = tile[col * 33 + part * 4 + 1];
        o.z = tile[col * 33 + part * 4 + 2];
        o.w = tile[col * 33 + part * 4 + 3];
        *reinterpret_cast<uint4*>(codes_t + (c0 + col) * M + m0 + part * 16) = o;
    }
}

// Writes a 128x128 code tile held in shared memory (row stride kStride)
// transposed: thread t (of 256) takes column t%128 and 64 of its rows, and
// writes them as 64 contiguous bytes of row t%128 of dst (leading dim ld).
template <int kStride>
__device__ __forceinline__ void store_tile_transposed(const uint8_t* tile, int t, uint8_t* dst, int64_t ld) {
    const int col = t & 127, half = t >> 7;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        const int r0 = half * 64 + part * 32;
        uint32_t wds[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t wd = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) wd |= (uint32_t)tile[(r0 + q * 4 + b) * kStride + col] << (8 * b);
            wds[q] = wd;
        }
        uint4* d = reinterpret_cast<uint4*>(dst + col * ld + r0);
        d[0] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
        d[1] = make_uint4(wds[4], wds[5], wds[6], wds[7]);
    }
}

// ---------------------------------------------------------------------------
// 128x128 blocks.  Block = one weight block; thread (chunk = t%16, rg = t/16)
// holds rows 8rg..8rg+7 of columns 8chunk..8chunk+7 (eight 16-byte loads in
// flight).  The block maximum is a warp shuffle reduction followed by a
// shared-memory reduction over the 8 warps.  The optional transposed copy:
// each thread transposes its four 4x4 byte blocks of codes in registers
// (byte permutes), which gives for each of its 8 columns the words of rows
// 8rg..8rg+3 and 8rg+4..8rg+7, and stores them into a shared tile of 128
// transposed rows x 32 words whose 16-byte units are permuted by
// (row / 8) % 8; each thread then writes 64 contiguous bytes of one
// transposed row.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int blk_t_word(int c, int wi) {
    return c * 32 + ((((wi >> 2) ^ (c >> 3)) & 7) << 2) + (wi & 3);
}
template <bool kPow2>
__global__ void __launch_bounds__(256) k_quant_block(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                     int64_t ld, uint8_t* __restrict__ codes,
                                                     void* __restrict__ scales, uint8_t* __restrict__ codes_t,
                                                     void* __restrict__ scales_t) {
    __shared__ float red[8];
    __shared__ __align__(16) uint32_t tile_t[128 * 32];

    const int64_t KB = K / 128, NB = N / 128;
    const int64_t nb = (int64_t)blockIdx.x / KB, kb = (int64_t)blockIdx.x % KB;
    const int64_t n0 = nb * 128, k0 = kb * 128;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int chunk = t & 15, rg = t >> 4;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ld_stream_v4(w + (n0 + rg * 8 + i) * ld + k0 + chunk * 8);
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float f[8];
        unpack8(v[i], f);
        a = fmaxf(a, amax8(f));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) red[warp] = a;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
    Divider dv;
    float mul = 1.0f;
    if (kPow2) {
        // the block's exponent fills its whole 512-byte MX atom (and the
        // transposed copy's atom): 16 bytes per thread of the first warps
        const int e = pow2_exponent(a);
        mul = exp2_int(-e);
        const uint32_t b4 = (uint32_t)(e + 127) * 0x01010101u;
        const uint4 fill = make_uint4(b4, b4, b4, b4);
        if (t < 32) reinterpret_cast<uint4*>(static_cast<uint8_t*>(scales) + (nb * KB + kb) * 512)[t] = fill;
        else if (t < 64 && scales_t)
            reinterpret_cast<uint4*>(static_cast<uint8_t*>(scales_t) + (kb * NB + nb) * 512)[t - 32] = fill;
    } else {
        const float s = group_scale_bf16(a);
        if (t == 0) {
            static_cast<float*>(scales)[nb * KB + kb] = s;
            if (scales_t) static_cast<float*>(scales_t)[kb * NB + nb] = s;
        }
        dv = make_divider(s);
    }
    uint2 c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float f[8];
        unpack8(v[i], f);
        c[i] = kPow2 ? encode8_mul(f, mul) : encode8_div(f, dv);
        *reinterpret_cast<uint2*>(codes + (n0 + rg * 8 + i) * K + k0 + chunk * 8) = c[i];
    }
    if (codes_t == nullptr) return;
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            // rows 8rg + 4k .. +3 x columns 8chunk + 4hh .. +3: word i = row i, byte j = column j
            const uint32_t w0 = hh ? c[4 * k].y : c[4 * k].x, w1 = hh ? c[4 * k + 1].y : c[4 * k + 1].x;
            const uint32_t w2 = hh ? c[4 * k + 2].y : c[4 * k + 2].x, w3 = hh ? c[4 * k + 3].y : c[4 * k + 3].x;
            const uint32_t t0 = __byte_perm(w0, w1, 0x5140), t1 = __byte_perm(w2, w3, 0x5140);
            const uint32_t t2 = __byte_perm(w0, w1, 0x7362), t3 = __byte_perm(w2, w3, 0x7362);
            const uint32_t col[4] = {__byte_perm(t0, t1, 0x5410), __byte_perm(t0, t1, 0x7632),
                                     __byte_perm(t2, t3, 0x5410), __byte_perm(t2, t3, 0x7632)};
#pragma unroll
            for (int j = 0; j < 4; ++j) tile_t[blk_t_word(chunk * 8 + hh * 4 + j, 2 * rg + k)] = col[j];
        }
    __syncthreads();
    // transposed row cr (column cr of the block), 16-byte units 4q .. 4q + 3
    const int cr = t >> 1, q = t & 1;
    const uint4* row = reinterpret_cast<const uint4*>(tile_t) + cr * 8;
    uint4* dst = reinterpret_cast<uint4*>(codes_t + (k0 + cr) * N + n0 + 64 * q);
#pragma unroll
    for (int u = 0; u < 4; ++u) dst[u] = row[((4 * q + u) ^ (cr >> 3)) & 7];
}

// ---------------------------------------------------------------------------
// fp8_param: the FP8 storage of a weight recomputed from its fp32 master
// ("Deep dive: FP8 quantization with FP32 and power-of-two block scales": the
// optimizer updates the FP32 master, and after every step it is quantized
// again into the FP8 parameters).  Block = one 128x128 block of the master;
// thread (lane, warp) holds rows 16warp..16warp+15 of columns
// 4lane..4lane+3 (sixteen 16-byte loads; each row is one 512-byte warp
// access).  With kDelta the step's final add W += dW (fp32, round to
// nearest) is applied first and written back.  fp32 recipe: s = RN(amax/448),
// 1 when that is 0; codes from the IEEE quotient w/s (fp32 inputs have full
// 24-bit significands: neg_quotient2_exact, the IEEE quotient bit for bit,
// or the IEEE division itself for scales outside its range).  Power-of-two
// recipe: e from RN(amax/448), codes from the exact product w * 2^-e.
// ---------------------------------------------------------------------------
template <bool kPow2, bool kDelta>
__global__ void __launch_bounds__(256, 3) k_param_requant(float* __restrict__ master, const float* __restrict__ delta,
                                                       int64_t N, int64_t K, int64_t ld, uint8_t* __restrict__ codes,
                                                       void* __restrict__ scales, uint8_t* __restrict__ codes_t,
                                                       void* __restrict__ scales_t) {
    constexpr int kStride = 144;
    __shared__ float red[8];
    __shared__ __align__(16) uint8_t tile[128 * kStride];

    const int64_t KB = K / 128, NB = N / 128;
    const int64_t nb = (int64_t)blockIdx.x / KB, kb = (int64_t)blockIdx.x % KB;
    const int64_t n0 = nb * 128, k0 = kb * 128;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    float* base = master + (n0 + warp * 16) * ld + k0 + lane * 4;

    float4 v[16];
    if (kDelta) {
        const float* dbase = delta + (n0 + warp * 16) * ld + k0 + lane * 4;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float4 d[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[8 * h + i] = __ldcs(reinterpret_cast<const float4*>(base + (8 * h + i) * ld));
                d[i] = __ldcs(reinterpret_cast<const float4*>(dbase + (8 * h + i) * ld));
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float4& w = v[8 * h + i];
                w.x = __fadd_rn(w.x, d[i].x);
                w.y = __fadd_rn(w.y, d[i].y);
                w.z = __fadd_rn(w.z, d[i].z);
                w.w = __fadd_rn(w.w, d[i].w);
                __stcs(reinterpret_cast<float4*>(base + (8 * h + i) * ld), w);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __ldcs(reinterpret_cast<const float4*>(base + i * ld));
    }
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(fmaxf(a, fmaxf(fabsf(v[i].x), fabsf(v[i].y))),
                                           fmaxf(fabsf(v[i].z), fabsf(v[i].w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) red[warp] = a;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
    float s = 1.0f, mul = 1.0f;
    if (kPow2) {
        const int e = a == 0.0f ? 0 : pow2_exponent_of_scale(__fdiv_rn(a, 448.0f));
        mul = exp2_int(-e);
        const uint32_t b4 = (uint32_t)(e + 127) * 0x01010101u;
        const uint4 fill = make_uint4(b4, b4, b4, b4);
        if (t < 32) reinterpret_cast<uint4*>(static_cast<uint8_t*>(scales) + (nb * KB + kb) * 512)[t] = fill;
        else if (t < 64 && scales_t)
            reinterpret_cast<uint4*>(static_cast<uint8_t*>(scales_t) + (kb * NB + nb) * 512)[t - 32] = fill;
    } else {
        s = group_scale(a);
        if (t == 0) {
            static_cast<float*>(scales)[nb * KB + kb] = s;
            if (scales_t) static_cast<float*>(scales_t)[kb * NB + nb] = s;
        }
    }
    uint8_t* crow = codes + (n0 + warp * 16) * K + k0 + lane * 4;
    const bool exact = !kPow2 && s >= 0x1p-90f && s <= 0x1p126f;
    const float nr = exact ? -__frcp_rn(s) : 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t c;
        if (kPow2) {
            c = e4m3x2(v[i].x * mul, v[i].y * mul) | (e4m3x2(v[i].z * mul, v[i].w * mul) << 16);
        } else if (exact) {
            float n0, n1, n2, n3;
            neg_quotient2_exact(v[i].x, v[i].y, s, nr, n0, n1);
            neg_quotient2_exact(v[i].z, v[i].w, s, nr, n2, n3);
            c = (e4m3x2(n0, n1) | (e4m3x2(n2, n3) << 16)) ^ 0x80808080u;  // codes of -n: sign back
        } else {
            c = e4m3x2(__fdiv_rn(v[i].x, s), __fdiv_rn(v[i].y, s)) |
                (e4m3x2(__fdiv_rn(v[i].z, s), __fdiv_rn(v[i].w, s)) << 16);
        }
        *reinterpret_cast<uint32_t*>(crow + i * K) = c;
        if (codes_t) *reinterpret_cast<uint32_t*>(tile + (warp * 16 + i) * kStride + lane * 4) = c;
    }
    if (codes_t == nullptr) return;
    __syncthreads();
    store_tile_transposed<kStride>(tile, t, codes_t + k0 * N + n0, N);
}

// ---------------------------------------------------------------------------
// MX 1x32 blocks.  Block = one 128-row x 128-column tile, i.e. exactly one
// 512-byte scale atom; thread (chunk = t%16, slot = t/16) holds rows
// slot + 16i (i < 8) of columns 8chunk..8chunk+7.  A 32-block spans 4 lanes
// (shuffle over xor 1, 2).  The atom is assembled in shared memory and
// written with 16-byte stores.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 5) k_quant_mx(const uint16_t* __restrict__ x, int64_t R, int64_t K, int64_t ld,
                                                  uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    __shared__ __align__(16) uint8_t atom[512];
    const int64_t atoms_k = (K + 127) / 128;
    const int64_t rt = (int64_t)blockIdx.x / atoms_k, ct = (int64_t)blockIdx.x % atoms_k;
    const int64_t r0 = rt * 128, k0 = ct * 128;
    const int t = threadIdx.x, chunk = t & 15, slot = t >> 4;
    const int j = chunk >> 2;                     // 32-block inside the atom
    const bool col_ok = k0 + chunk * 8 < K;      // K % 32 == 0: whole 32-blocks valid or not

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + slot + 16 * i;
        v[i] = (col_ok && r < R) ? ld_stream_v4(x + r * ld + k0 + chunk * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rl = slot + 16 * i;
        const int64_t r = r0 + rl;
        float f[8];
        unpack8(v[i], f);
        float a = amax8(f);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        const int e = mx_exponent(a);
        if ((chunk & 3) == 0) atom[(rl & 31) * 16 + (rl >> 5) * 4 + j] = (uint8_t)(e + 127);
        if (col_ok && r < R) {
            const uint2 c = encode8_mul(f, exp2_int(-e));
            *reinterpret_cast<uint2*>(codes + r * K + k0 + chunk * 8) = c;
        }
    }
    __syncthreads();
    if (t < 32)
        reinterpret_cast<uint4*>(scales + (rt * atoms_k + ct) * 512)[t] = reinterpret_cast<const uint4*>(atom)[t];
}

// ---------------------------------------------------------------------------
// MX 32x1 blocks along the rows, codes transposed (the MXFP8 backward
// operands: W^T for DGrad, dY^T and X^T for WGrad) -- the 1x32 quantization
// of x^T.  Block = one 128-row x 64-column tile; thread (chunk = t%8,
// quad = t/8) holds rows 4*quad..4*quad+3 of columns 8*chunk..8*chunk+7, so a
// warp covers 16 rows and a 32-row block is two warps.  Block maxima: in
// thread over 4 rows, shuffles over the warp's 4 quads, shared memory over
// the warp pair; one 32-bit store per column carries the 4 exponents of its
// 128 rows.  Codes are the exact products x * 2^-e, transposed through a
// 33-word-stride shared tile and written 16 bytes per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 6) k_quant_mx_t(const uint16_t* __restrict__ x, int64_t R, int64_t K,
                                                    int64_t ld, uint8_t* __restrict__ codes_t,
                                                    uint8_t* __restrict__ scales_t) {
    __shared__ float red[8][64];
    __shared__ float col_mul[4][64];
    __shared__ uint32_t tile[64 * 33];

    const int64_t ctiles = (K + 63) / 64;
    const int64_t mb = (int64_t)blockIdx.x / ctiles;
    const int64_t c0 = ((int64_t)blockIdx.x % ctiles) * 64;
    const int64_t m0 = mb * 128;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int chunk = t & 7, quad = t >> 3;
    const bool col_ok = c0 + chunk * 8 < K;  // K % 8 == 0: a chunk is all valid or all invalid

    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = col_ok ? ld_stream_v4(x + (m0 + quad * 4 + i) * ld + c0 + chunk * 8) : make_uint4(0, 0, 0, 0);
    float f[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack8(v[i], f[i]);
    float pa[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float a = fmaxf(fmaxf(fabsf(f[0][j]), fabsf(f[1][j])), fmaxf(fabsf(f[2][j]), fabsf(f[3][j])));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
        pa[j] = a;
    }
    if (lane < 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) red[warp][chunk * 8 + j] = pa[j];
    }
    __syncthreads();
    if (t < 64) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int e = mx_exponent(fmaxf(red[2 * b][t], red[2 * b + 1][t]));
            col_mul[b][t] = exp2_int(-e);
            word |= (uint32_t)(e + 127) << (8 * b);
        }
        // transposed row c0+t, 1x32 blocks 4mb..4mb+3 of the [K][R] output
        if (c0 + t < K) *reinterpret_cast<uint32_t*>(scales_t + mx_scale_offset(c0 + t, 4 * mb, R / 128)) = word;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float mul = col_mul[warp >> 1][chunk * 8 + j];
        tile[(chunk * 8 + j) * 33 + quad] = e4m3x2(__fmul_rn(f[0][j], mul), __fmul_rn(f[1][j], mul)) |
                                            (e4m3x2(__fmul_rn(f[2][j], mul), __fmul_rn(f[3][j], mul)) << 16);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = t + 256 * i;
        const int col = idx >> 3, part = idx & 7;
        if (c0 + col < K) {
            uint4 o;
            o.x = tile[col * 33 + part * 4 + 0];
            o.y = tile[col * 33 + part * 4 + 1];
            o.z = tile[col * 33 + part * 4 + 2];
            o.w = tile[col * 33 + part * 4 + 3];
            *reinterpret_cast<uint4*>(codes_t + (c0 + col) * R + m0 + part * 16) = o;
        }
    }
}

// ---------------------------------------------------------------------------
// MoE row gather of MX codes and scales into expert-contiguous groups.  One
// warp per destination row: 16-byte code copies, then one 32-bit word per
// 128-column atom (the 4 scale bytes of a row inside an atom are adjacent).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_permute_rows_mx(const uint8_t* __restrict__ src_codes,
                                                         const uint8_t* __restrict__ src_scales, int64_t src_rows,
                                                         int64_t K, const int32_t* __restrict__ gather,
                                                         const int32_t* __restrict__ offsets, int32_t G,
                                                         int64_t total, uint8_t* __restrict__ dst_codes,
                                                         uint8_t* __restrict__ dst_scales, StatusBlock* status) {
    const int lane = threadIdx.x & 31;
    const int64_t i = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (i >= total) return;
    const int64_t src = gather[i];
    if (src < 0 || src >= src_rows) {
        if (lane == 0) atomicOr(&status->error_bits, kErrDeviceArg);
        return;
    }
    // group of row i: last g with offsets[g] <= i
    int lo = 0, hi = G;  // invariant offsets[lo] <= i < offsets[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offsets[mid] <= i) lo = mid; else hi = mid;
    }
    const int g = lo;
    // the codes row lies inside dst whatever the offsets say
    const uint4* s4 = reinterpret_cast<const uint4*>(src_codes + src * K);
    uint4* d4 = reinterpret_cast<uint4*>(dst_codes + i * K);
    for (int64_t c = lane; c < K / 16; c += 32) d4[c] = s4[c];

    // atom-row base of group g: sum over h < g of ceil(M_h / 128).  The
    // offsets are checked on the way (offsets[0] = 0, non-decreasing up to
    // g, offsets[g] <= i < offsets[g + 1]): otherwise the row's scale words
    // are not written and the call is reported, so none lands outside the
    // grouped layout.
    int64_t pg = 0;
    bool ok = true;
    for (int h = lane; h < g; h += 32) {
        const int32_t a = offsets[h], b = offsets[h + 1];
        ok &= b >= a;
        pg += (b - a + 127) / 128;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pg += __shfl_xor_sync(0xffffffffu, pg, o);
    ok = __all_sync(0xffffffffu, ok) && offsets[0] == 0 && offsets[g] <= i && i < offsets[g + 1];
    if (!ok) {
        if (lane == 0) atomicOr(&status->error_bits, kErrDeviceArg);
        return;
    }
    const int64_t l = i - offsets[g];

    const int64_t atoms_k = K / 128;
    const int64_t s_in = (src & 31) * 16 + ((src & 127) >> 5) * 4;
    const int64_t d_in = (l & 31) * 16 + ((l & 127) >> 5) * 4;
    const int64_t d_row = pg + (l >> 7);
    for (int64_t a = lane; a < atoms_k; a += 32) {
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(src_scales + ((src >> 7) * atoms_k + a) * 512 + s_in);
        *reinterpret_cast<uint32_t*>(dst_scales + (d_row * atoms_k + a) * 512 + d_in) = wd;
    }
}

// ---------------------------------------------------------------------------
// MoE dispatch fused with the MX quantization, token-major: every source row
// (token) is read and quantized once, and its codes and scale words are
// written to each of its top_k destination rows in the expert-grouped layout
// (dst row dst_index[t][j]; negative entries are dropped tokens).  One warp
// per token, 8 tokens per block; a block first stages the group offsets and
// the groups' atom-row bases (prefix sums of ceil(M_g / 128)) in shared
// memory.  The row is processed 2048 columns at a time: 8 rounds of 256
// columns (lane: 8 columns, a 32-block is 4 lanes, a 128-column atom a half
// warp), all loads of a pass issued first.
// ---------------------------------------------------------------------------
constexpr int kDqMaxGroups = 1024;

__global__ void __launch_bounds__(256, 5) k_dispatch_quant_mx(const uint16_t* __restrict__ x, int64_t T, int64_t K,
                                                           int64_t ld, const int32_t* __restrict__ dst_index,
                                                           int top_k, const int32_t* __restrict__ offsets, int32_t G,
                                                           int64_t total, uint8_t* __restrict__ dst_codes,
                                                           uint8_t* __restrict__ dst_scales, StatusBlock* status) {
    __shared__ int32_t s_off[kDqMaxGroups + 1];
    __shared__ int64_t s_pg[kDqMaxGroups + 1];
    __shared__ int s_bad;
    for (int g = threadIdx.x; g <= G; g += blockDim.x) s_off[g] = offsets[g];
    __syncthreads();
    if (threadIdx.x == 0) {
        // offsets must run from 0 to total without decreasing; otherwise the
        // call is reported and nothing is written
        int bad = s_off[0] != 0 || s_off[G] != total;
        int64_t acc = 0;
        for (int g = 0; g < G; ++g) {
            s_pg[g] = acc;
            bad |= s_off[g + 1] < s_off[g];
            acc += (s_off[g + 1] - s_off[g] + 127) / 128;
        }
        s_pg[G] = acc;
        s_bad = bad;
        if (bad) atomicOr(&status->error_bits, kErrDeviceArg);
    }
    __syncthreads();
    if (s_bad) return;
    const int lane = threadIdx.x & 31, sub = lane & 15, half = lane >> 4;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const int64_t atoms_k = K / 128;
    const uint16_t* xr = x + t * ld;
    const int64_t rounds = K / 256 + ((K & 255) ? 1 : 0);   // K % 128 == 0: a last round may be half
    for (int64_t r0 = 0; r0 < rounds; r0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int64_t k = (r0 + u) * 256 + 8 * lane;
            v[u] = (r0 + u < rounds && k < K) ? ld_stream_v4(xr + k) : make_uint4(0, 0, 0, 0);
        }
        uint2 c[8];
        uint32_t sw[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float f[8];
            unpack8(v[u], f);
            float a = amax8(f);
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            const int e = mx_exponent(a);
            c[u] = encode8_mul(f, exp2_int(-e));
            const uint32_t b = (uint32_t)(e + 127);
            const uint32_t b1 = __shfl_sync(0xffffffffu, b, 16 * half + 4);
            const uint32_t b2 = __shfl_sync(0xffffffffu, b, 16 * half + 8);
            const uint32_t b3 = __shfl_sync(0xffffffffu, b, 16 * half + 12);
            sw[u] = b | (b1 << 8) | (b2 << 16) | (b3 << 24);
        }
        for (int j = 0; j < top_k; ++j) {
            const int64_t d = dst_index[t * top_k + j];
            if (d < 0) continue;                                  // dropped token (warp-uniform)
            if (d >= total) {
                if (lane == 0) atomicOr(&status->error_bits, kErrDeviceArg);
                continue;
            }
            int lo = 0, hi = G;  // group of row d: last g with offsets[g] <= d
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= d) lo = mid; else hi = mid;
            }
            const int64_t l = d - s_off[lo];
            uint8_t* srow = dst_scales + (s_pg[lo] + (l >> 7)) * atoms_k * 512 + (l & 31) * 16 + ((l & 127) >> 5) * 4;
            uint8_t* crow = dst_codes + d * K;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t k = (r0 + u) * 256 + 8 * lane;
                if (r0 + u < rounds && k < K) {
                    *reinterpret_cast<uint2*>(crow + k) = c[u];
                    if (sub == 0) *reinterpret_cast<uint32_t*>(srow + (k / 128) * 512) = sw[u];
                }
            }
        }
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Launchers (argument checks are done by the API layer).
// ---------------------------------------------------------------------------
// Padding rows of the last MX atom row (rows >= `rows`) must read as zero.
cudaError_t zero_mx_tail(void* scales, int64_t rows, int64_t cols, cudaStream_t st) {
    if (rows % 128 == 0) return cudaSuccess;
    const int64_t atoms_k = (cols + 127) / 128;
    return cudaMemsetAsync(static_cast<uint8_t*>(scales) + (rows / 128) * atoms_k * 512, 0, (size_t)atoms_k * 512, st);
}

cudaError_t launch_quant_group_k(const uint16_t* x, int64_t M, int64_t K, int64_t ld, uint8_t* codes,
                                 void* scales, bool pow2, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    const int64_t G = K / 128;
    const int64_t blocks = ((M + kGK_Rows - 1) / kGK_Rows) * ((G + kGK_Groups - 1) / kGK_Groups);
    if (pow2) {
        cudaError_t e = zero_mx_tail(scales, M, K, st);
        if (e != cudaSuccess) return e;
        k_quant_group_k<true><<<(unsigned)blocks, 256, 0, st>>>(x, M, K, ld, codes, scales);
    } else {
        k_quant_group_k<false><<<(unsigned)blocks, 256, 0, st>>>(x, M, K, ld, codes, scales);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_group_m(const uint16_t* x, int64_t M, int64_t K, int64_t ld, uint8_t* codes_t,
                                 void* scales, bool pow2, cudaStream_t st) {
    if (M == 0 || K == 0) return cudaSuccess;
    const int64_t blocks = (M / 128) * ((K + 63) / 64);
    if (pow2) {
        cudaError_t e = zero_mx_tail(scales, K, M, st);  // the output is the [K][M] transpose
        if (e != cudaSuccess) return e;
        k_quant_group_m<true><<<(unsigned)blocks, 256, 0, st>>>(x, M, K, ld, codes_t, scales);
    } else {
        k_quant_group_m<false><<<(unsigned)blocks, 256, 0, st>>>(x, M, K, ld, codes_t, scales);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_block(const uint16_t* w, int64_t N, int64_t K, int64_t ld, uint8_t* codes,
                               void* scales, uint8_t* codes_t, void* scales_t, bool pow2, cudaStream_t st) {
    if (N == 0 || K == 0) return cudaSuccess;
    const int64_t blocks = (N / 128) * (K / 128);
    if (pow2)
        k_quant_block<true><<<(unsigned)blocks, 256, 0, st>>>(w, N, K, ld, codes, scales, codes_t, scales_t);
    else
        k_quant_block<false><<<(unsigned)blocks, 256, 0, st>>>(w, N, K, ld, codes, scales, codes_t, scales_t);
    return cudaGetLastError();
}

cudaError_t launch_param_requant(float* master, const float* delta, int64_t N, int64_t K, int64_t ld,
                                 uint8_t* codes, void* scales, uint8_t* codes_t, void* scales_t, bool pow2,
                                 cudaStream_t st) {
    if (N == 0 || K == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((N / 128) * (K / 128));
    if (pow2) {
        if (delta)
            k_param_requant<true, true><<<blocks, 256, 0, st>>>(master, delta, N, K, ld, codes, scales, codes_t, scales_t);
        else
            k_param_requant<true, false><<<blocks, 256, 0, st>>>(master, delta, N, K, ld, codes, scales, codes_t, scales_t);
    } else {
        if (delta)
            k_param_requant<false, true><<<blocks, 256, 0, st>>>(master, delta, N, K, ld, codes, scales, codes_t, scales_t);
        else
            k_param_requant<false, false><<<blocks, 256, 0, st>>>(master, delta, N, K, ld, codes, scales, codes_t, scales_t);
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_mx(const uint16_t* x, int64_t R, int64_t K, int64_t ld, uint8_t* codes, uint8_t* scales,
                            cudaStream_t st) {
    if (R == 0 || K == 0) return cudaSuccess;
    const int64_t blocks = ((R + 127) / 128) * ((K + 127) / 128);
    k_quant_mx<<<(unsigned)blocks, 256, 0, st>>>(x, R, K, ld, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_quant_mx_t(const uint16_t* x, int64_t R, int64_t K, int64_t ld, uint8_t* codes_t,
                              uint8_t* scales_t, cudaStream_t st) {
    if (R == 0 || K == 0) return cudaSuccess;
    cudaError_t e = zero_mx_tail(scales_t, K, R, st);  // the output is the [K][R] transpose
    if (e != cudaSuccess) return e;
    const int64_t blocks = (R / 128) * ((K + 63) / 64);
    k_quant_mx_t<<<(unsigned)blocks, 256, 0, st>>>(x, R, K, ld, codes_t, scales_t);
    return cudaGetLastError();
}

cudaError_t launch_permute_rows_mx(const uint8_t* src_codes, const uint8_t* src_scales, int64_t src_rows,
                                   int64_t K, const int32_t* gather, const int32_t* offsets, int32_t G,
                                   int64_t total, uint8_t* dst_codes, uint8_t* dst_scales, int64_t dst_scale_bytes,
                                   StatusBlock* status, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(dst_scales, 0, (size_t)dst_scale_bytes, st);
    if (e != cudaSuccess || total == 0) return e;
    const int64_t blocks = (total + 7) / 8;
    k_permute_rows_mx<<<(unsigned)blocks, 256, 0, st>>>(src_codes, src_scales, src_rows, K, gather, offsets, G, total,
                                                        dst_codes, dst_scales, status);
    return cudaGetLastError();
}

cudaError_t launch_requant_group_m(const uint8_t* codes, const float* scales, int64_t M, int64_t K, uint8_t* codes_t,
                                   float* scales_t, cudaStream_t st) {
    if (M == 0 || K == 0) return cudaSuccess;
    const int64_t blocks = (M / 128) * (K / 64);
    k_requant_group_m<<<(unsigned)blocks, 256, 0, st>>>(codes, scales, M, K, codes_t, scales_t);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_quant_mx(const uint16_t* x, int64_t T, int64_t K, int64_t ld, const int32_t* dst_index,
                                     int top_k, const int32_t* offsets, int32_t G, int64_t total, uint8_t* dst_codes,
                                     uint8_t* dst_scales, int64_t dst_scale_bytes, StatusBlock* status,
                                     cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(dst_scales, 0, (size_t)dst_scale_bytes, st);
    if (e != cudaSuccess || T == 0 || top_k == 0) return e;
    const int64_t blocks = (T + 7) / 8;
    k_dispatch_quant_mx<<<(unsigned)blocks, 256, 0, st>>>(x, T, K, ld, dst_index, top_k, offsets, G, total, dst_codes,
                                                          dst_scales, status);
    return cudaGetLastError();
}

}  // namespace fp8bs
