// gemm_common.cuh -- constants, shared-memory barrier block and helpers of
// the two tcgen05 GEMM kernels (gemm_blockwise.cu, gemm_mx.cu).
//
// Both kernels compute D = A B^T with A [M][K], B [N][K] E4M3 codes (K-major),
// are persistent and warp-specialised, and run as clusters of two CTAs on
// neighbouring SMs (tcgen05.mma.cta_group::2, M=256), one CTA per SM:
//   warp 0      TMA producer: A and B tiles (+ the MX scale atoms) per
//               128-wide K block into a multi-stage shared-memory ring
//   warp 1      allocates TMEM for the pair; one thread of the leader CTA
//               issues tcgen05.mma (K=32, four per K block and N slice) and
//               tcgen05.commit
//   warps 2..   epilogue: tcgen05.ld of the fp32 partials / accumulator; warp w
//               may only touch TMEM lanes 32*(w%4).., so each lane quarter is
//               served by (number of epilogue warps) / 4 warps.
// Every wait is bounded (see mbar_wait_bounded); on expiry the kernel records
// FP8_ERR_TIMEOUT, stops issuing work, and exits through the same teardown.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace fp8bs {

namespace {

constexpr int BM = 128, BK = 128;
constexpr int kThreads = 320;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiThreads = 256;
constexpr int kMaxStages = 6;
constexpr int kMaxGroups = 1024;

struct alignas(16) Barriers {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[4];
    uint64_t acc_empty[4];
    uint64_t drain;
    uint64_t sf_ready[kMaxStages];  // MX: the stage's scale factors copied into TMEM
    uint32_t tmem_base;
    int abort;
    int num_mtiles;  // MX: total 256-row cluster tiles over all groups
};



__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
    const uint32_t a = smem_u32(raw);
    return raw + ((1024u - (a & 1023u)) & 1023u);
}

// Wait that ignores the abort flag (used to let in-flight work land).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, StatusBlock* st) {
    int dummy = 0;
    mbar_wait_bounded(bar, parity, &dummy, st, 99);
}

// Empty asm that "redefines" the registers, so that no use of a TMEM load
// result can be scheduled before the preceding tcgen05.wait::ld.
__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])::"memory");
}

__device__ __forceinline__ void ld_chunk(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld_32x32b_x32(taddr, r); }

__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15])::"memory");
}


// MX 1x32 quantization of one row's 128 bf16 values: four blocks; returns
// 32-byte global store (one full L2 sector per lane).
__device__ __forceinline__ void st_v8(void* ptr, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D u8 tensor map over a row-major [rows][cols] matrix with a
// box of box_rows x 128 bytes and 128-byte swizzle; out-of-range rows read 0.
bool make_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor map over a row-major [rows][ld] matrix of which the first
// cols columns are addressed, for stores of 64-column (128-byte) x 128-row
// boxes from a 128-byte-swizzled shared tile; rows and columns outside the
// matrix are not written.  base 16-byte aligned, ld * 2 a multiple of 16.
bool make_map_store_bf16(CUtensorMap* map, void* base, uint64_t cols, uint64_t rows, uint64_t ld) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D u8 tensor map, no swizzle, over a row-major [rows][cols] byte array.
bool make_map_plain_u8(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {(cuuint32_t)cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

}  // namespace

}  // namespace fp8bs
