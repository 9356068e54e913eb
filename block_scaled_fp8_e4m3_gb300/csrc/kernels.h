// kernels.h -- launchers of the device kernels, called by the C-ABI layer
// (api.cu) after it has validated every argument.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fp8bs {

struct StatusBlock;

// quantize.cu
// pow2: the blockwise recipe with power-of-two scales, written as E8M0 bytes
// in the MX scale-factor layout (scales then points to bytes, not floats)
cudaError_t launch_quant_group_k(const uint16_t* x, int64_t M, int64_t K, int64_t ld, uint8_t* codes,
                                 void* scales, bool pow2, cudaStream_t st);
cudaError_t launch_quant_group_m(const uint16_t* x, int64_t M, int64_t K, int64_t ld, uint8_t* codes_t,
                                 void* scales, bool pow2, cudaStream_t st);
cudaError_t launch_quant_block(const uint16_t* w, int64_t N, int64_t K, int64_t ld, uint8_t* codes,
                               void* scales, uint8_t* codes_t, void* scales_t, bool pow2, cudaStream_t st);
cudaError_t launch_quant_mx(const uint16_t* x, int64_t R, int64_t K, int64_t ld, uint8_t* codes, uint8_t* scales,
                            cudaStream_t st);
cudaError_t launch_param_requant(float* master, const float* delta, int64_t N, int64_t K, int64_t ld,
                                 uint8_t* codes, void* scales, uint8_t* codes_t, void* scales_t, bool pow2,
                                 cudaStream_t st);
cudaError_t launch_quant_mx_t(const uint16_t* x, int64_t R, int64_t K, int64_t ld, uint8_t* codes_t,
                              uint8_t* scales_t, cudaStream_t st);
cudaError_t launch_dispatch_quant_mx(const uint16_t* x, int64_t T, int64_t K, int64_t ld, const int32_t* dst_index,
                                     int top_k, const int32_t* offsets, int32_t G, int64_t total, uint8_t* dst_codes,
                                     uint8_t* dst_scales, int64_t dst_scale_bytes, StatusBlock* status,
                                     cudaStream_t st);
cudaError_t launch_requant_group_m(const uint8_t* codes, const float* scales, int64_t M, int64_t K, uint8_t* codes_t,
                                   float* scales_t, cudaStream_t st);
// Padding rows of the last MX atom row (rows >= `rows`) set to zero.
cudaError_t zero_mx_tail(void* scales, int64_t rows, int64_t cols, cudaStream_t st);

cudaError_t launch_permute_rows_mx(const uint8_t* src_codes, const uint8_t* src_scales, int64_t src_rows,
                                   int64_t K, const int32_t* gather, const int32_t* offsets, int32_t G,
                                   int64_t total, uint8_t* dst_codes, uint8_t* dst_scales, int64_t dst_scale_bytes,
                                   StatusBlock* status, cudaStream_t st);

// fused.cu: recipe 0 = 1x128 fp32 scales, 1 = 1x128 power-of-two scales,
// 2 = MXFP8 1x32 (1 and 2 write E8M0 bytes in the MX layout)
cudaError_t launch_rmsnorm_quant(const uint16_t* x, const uint16_t* gamma, int64_t M, int64_t K, int64_t ld,
                                 float eps, uint16_t* y, int64_t ldy, float* rstd, uint8_t* codes, void* scales,
                                 int recipe, cudaStream_t st);
cudaError_t launch_swiglu_quant(const uint16_t* gu, int64_t M, int64_t F, int64_t ld, uint16_t* h, int64_t ldh,
                                uint8_t* codes, void* scales, int recipe, cudaStream_t st);

// gemm_blockwise.cu, gemm_mx.cu
struct GemmBlockwiseArgs {
    const uint8_t* a_codes;  // [M][K]
    const uint8_t* b_codes;  // [N][K]
    const float* sa;         // [K/128][M]
    const float* sb;         // per-block [N/128][K/128] or per-row [K/128][N]
    int sb_per_row;          // 1 for WGRAD (B quantized 128x1)
    int64_t M, N, K;
    void* D;
    int64_t ldd;
    int d_f32;
    uint8_t* q_codes;        // fused 1x128 quantization of D (nullable)
    float* q_scales;
};
cudaError_t launch_gemm_blockwise(const GemmBlockwiseArgs& a, StatusBlock* status, cudaStream_t st);

struct GemmMxArgs {
    const uint8_t* a_codes;    // [rows_a][K]
    const uint8_t* b_codes;    // [G*N][K]
    const uint8_t* sfa;        // MX atoms (grouped layout when m_offsets != nullptr)
    const uint8_t* sfb;        // MX atoms of the B stack
    int64_t M;                 // rows of A (total rows when grouped)
    int64_t N, K;
    const int32_t* m_offsets;  // device [G+1] or nullptr (single group of M rows)
    int32_t G;
    void* D;                   // bf16 [rows][ldd]
    int64_t ldd;
    uint8_t* q_codes;          // fused MX quantization of D (nullable; single group only)
    uint8_t* q_scales;
    bool q_pow2 = false;       // fused quantization in 1x128 groups with power-of-two scales
};
cudaError_t launch_gemm_mx(const GemmMxArgs& a, StatusBlock* status, cudaStream_t st);

// sync.cu
constexpr int kMaxCopySegs = 32;
struct CopySeg {
    const uint8_t* src;
    uint8_t* dst;
    uint64_t bytes;   // bytes copied from src
    uint64_t padded;  // bytes written at dst (zero fill after `bytes`); multiple of 16
    uint64_t dst_word0;  // payload word index of dst[0] (pack: checksum position)
};
// Header + entry table of a payload (the checksum field excepted): written
// by the pack kernel, or compared on the device with the payload's own bytes
// by the install kernels; bytes == 0: none.
constexpr int kMaxExpectBytes = 64 + 128 * 24;
struct ExpectTable {
    uint32_t bytes;
    uint8_t data[kMaxExpectBytes];
};
// Pack: segment copies with the checksum accumulated into *checksum_field;
// with hdr, the first launch also writes the header and table and adds
// table_sum (the caller zeroes the checksum field first).
cudaError_t launch_sync_pack(const CopySeg* segs, int n, unsigned long long* checksum_field, const ExpectTable* hdr,
                             unsigned long long table_sum, cudaStream_t st);
// Verify + scatter in one cooperative launch; cudaErrorNotSupported when
// the device cannot run it (or n > kMaxCopySegs): use the two kernels then.
cudaError_t launch_sync_install(const uint8_t* payload, uint64_t data_offset, uint64_t total_bytes,
                                unsigned long long table_sum, StatusBlock* status, const ExpectTable* expect,
                                const CopySeg* segs, int n, cudaStream_t st);
cudaError_t launch_wait_expiry(unsigned long long limit_ns, StatusBlock* status, cudaStream_t st);
cudaError_t launch_sync_verify(const uint8_t* payload, uint64_t data_offset, uint64_t total_bytes,
                               unsigned long long table_sum, StatusBlock* status, cudaStream_t st,
                               const ExpectTable* expect = nullptr);
cudaError_t launch_sync_scatter(const CopySeg* segs, int n, const StatusBlock* status, cudaStream_t st);

}  // namespace fp8bs
