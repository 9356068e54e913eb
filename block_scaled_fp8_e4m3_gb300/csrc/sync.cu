// sync.cu -- on-policy weight-sync payload kernels.
//
// "Anyscale、SkyRL で FP8 学習・ロールアウトをサポートし一貫性を維持",
// "On-Policy FP8 weight sync" (Fig. 3): the trainer's FP8 codes and block
// scales travel unchanged and are installed without a quantizer, so the
// rollout weights are bit-identical.  These kernels only move bytes:
//  - pack: batched segment copy into the payload (zero padding included)
//    with the checksum of every written 8-byte word accumulated on the fly;
//  - verify: checksum of the payload's data region, compared with the value
//    stored in its header by the last block to finish;
//  - scatter: batched copy out of the payload, skipped entirely when the
//    verification failed.
// Checksum = sum of splitmix64(w_i XOR i) over 8-byte words w_i at byte
// offsets 8i >= 64, mod 2^64 (the splitmix64 finaliser of Steele, Lea and
// Flood, 2014).  Being a sum, it can be accumulated in any order.
#include "common.cuh"
#include "kernels.h"

namespace fp8bs {

namespace {

__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

struct SegTable {
    CopySeg seg[kMaxCopySegs];
    int n;
};

// chunk c of 16 bytes -> (segment, chunk within segment) by a scan of the
// per-segment chunk counts
__device__ __forceinline__ int find_seg(const uint64_t* start, int n, uint64_t c) {
    int s = 0;
    while (s + 1 < n && start[s + 1] <= c) ++s;
    return s;
}

__device__ __forceinline__ uint4 load16_tail(const uint8_t* src, uint64_t off, uint64_t bytes) {
    if (off + 16 <= bytes) return *reinterpret_cast<const uint4*>(src + off);
    uint8_t b[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) b[i] = (off + i < bytes) ? src[off + i] : 0;
    uint4 v;
    v.x = b[0] | (b[1] << 8) | (b[2] << 16) | ((uint32_t)b[3] << 24);
    v.y = b[4] | (b[5] << 8) | (b[6] << 16) | ((uint32_t)b[7] << 24);
    v.z = b[8] | (b[9] << 8) | (b[10] << 16) | ((uint32_t)b[11] << 24);
    v.w = b[12] | (b[13] << 8) | (b[14] << 16) | ((uint32_t)b[15] << 24);
    return v;
}

__device__ __forceinline__ unsigned long long block_sum(unsigned long long v) {
    __shared__ unsigned long long part[32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) part[warp] = v;
    __syncthreads();
    unsigned long long s = 0;
    if (threadIdx.x == 0)
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += part[w];
    return s;  // valid in thread 0
}

__global__ void __launch_bounds__(256) k_sync_pack(const SegTable tab, unsigned long long* checksum_field) {
    __shared__ uint64_t start[kMaxCopySegs + 1];
    if (threadIdx.x == 0) {
        uint64_t acc = 0;
        for (int s = 0; s < tab.n; ++s) {
            start[s] = acc;
            acc += tab.seg[s].padded / 16;
        }
        start[tab.n] = acc;
    }
    __syncthreads();
    const uint64_t chunks = start[tab.n];
    unsigned long long sum = 0;
    for (uint64_t c = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; c < chunks;
         c += (uint64_t)gridDim.x * blockDim.x) {
        const int s = find_seg(start, tab.n, c);
        const CopySeg& sg = tab.seg[s];
        const uint64_t off = (c - start[s]) * 16;
        const uint4 v = load16_tail(sg.src, off, sg.bytes);
        *reinterpret_cast<uint4*>(sg.dst + off) = v;
        const unsigned long long w0 = (unsigned long long)v.x | ((unsigned long long)v.y << 32);
        const unsigned long long w1 = (unsigned long long)v.z | ((unsigned long long)v.w << 32);
        const unsigned long long i0 = sg.dst_word0 + off / 8;
        sum += mix64(w0 ^ i0) + mix64(w1 ^ (i0 + 1));
    }
    const unsigned long long bs = block_sum(sum);
    if (threadIdx.x == 0 && bs != 0) atomicAdd(checksum_field, bs);
}

__global__ void __launch_bounds__(256) k_sync_verify(const uint8_t* __restrict__ payload, uint64_t data_offset,
                                                     uint64_t total_bytes, unsigned long long table_sum,
                                                     StatusBlock* st, const __grid_constant__ ExpectTable expect) {
    if (blockIdx.x == 0 && expect.bytes != 0) {
        // header and entry table against what the destinations imply (the
        // checksum field, bytes 32..39, is what the data is checked against)
        bool bad = false;
        for (uint32_t i = threadIdx.x; i < expect.bytes; i += blockDim.x)
            if ((i < 32 || i >= 40) && payload[i] != expect.data[i]) bad = true;
        if (__syncthreads_or(bad) && threadIdx.x == 0) atomicExch(&st->header_bad, 1u);
    }
    const uint64_t c0 = data_offset / 16, c1 = total_bytes / 16;
    unsigned long long sum = 0;
    for (uint64_t c = c0 + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; c < c1;
         c += (uint64_t)gridDim.x * blockDim.x) {
        const uint4 v = *reinterpret_cast<const uint4*>(payload + c * 16);
        const unsigned long long w0 = (unsigned long long)v.x | ((unsigned long long)v.y << 32);
        const unsigned long long w1 = (unsigned long long)v.z | ((unsigned long long)v.w << 32);
        sum += mix64(w0 ^ (2 * c)) + mix64(w1 ^ (2 * c + 1));
    }
    const unsigned long long bs = block_sum(sum);
    if (threadIdx.x == 0) {
        atomicAdd(&st->sum, bs);
        __threadfence();
        const unsigned int ticket = atomicAdd(&st->blocks_done, 1u);
        if (ticket == gridDim.x - 1) {
            __threadfence();
            const unsigned long long total = atomicAdd(&st->sum, 0ull) + table_sum;
            const unsigned long long stored = *reinterpret_cast<const unsigned long long*>(payload + 32);
            const unsigned int header_bad = atomicExch(&st->header_bad, 0u);
            const unsigned int bad = (total != stored || header_bad) ? 1u : 0u;
            st->verdict = bad;
            if (header_bad) atomicOr(&st->error_bits, kErrBadPayload);
            else if (bad) atomicOr(&st->error_bits, kErrChecksum);
            st->sum = 0;
            st->blocks_done = 0;
            __threadfence();
        }
    }
}

__global__ void __launch_bounds__(256) k_sync_scatter(const SegTable tab, const StatusBlock* st) {
    if (*reinterpret_cast<const volatile unsigned int*>(&st->verdict) != 0) return;
    __shared__ uint64_t start[kMaxCopySegs + 1];
    if (threadIdx.x == 0) {
        uint64_t acc = 0;
        for (int s = 0; s < tab.n; ++s) {
            start[s] = acc;
            acc += (tab.seg[s].bytes + 15) / 16;
        }
        start[tab.n] = acc;
    }
    __syncthreads();
    const uint64_t chunks = start[tab.n];
    for (uint64_t c = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; c < chunks;
         c += (uint64_t)gridDim.x * blockDim.x) {
        const int s = find_seg(start, tab.n, c);
        const CopySeg& sg = tab.seg[s];
        const uint64_t off = (c - start[s]) * 16;
        const uint4 v = *reinterpret_cast<const uint4*>(sg.src + off);   // payload side: padded, aligned
        if (off + 16 <= sg.bytes) {
            *reinterpret_cast<uint4*>(sg.dst + off) = v;
        } else {
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            for (uint64_t i = 0; off + i < sg.bytes; ++i) sg.dst[off + i] = (uint8_t)(w[i / 4] >> (8 * (i % 4)));
        }
    }
}

int grid_for(uint64_t chunks) {
    uint64_t b = (chunks + 255) / 256;
    if (b > 152 * 8) b = 152 * 8;
    return b == 0 ? 1 : (int)b;
}

}  // namespace

cudaError_t launch_sync_pack(const CopySeg* segs, int n, unsigned long long* checksum_field, cudaStream_t st) {
    SegTable tab;
    uint64_t chunks = 0;
    tab.n = n;
    for (int i = 0; i < n; ++i) {
        tab.seg[i] = segs[i];
        chunks += segs[i].padded / 16;
    }
    if (chunks == 0) return cudaSuccess;
    k_sync_pack<<<grid_for(chunks), 256, 0, st>>>(tab, checksum_field);
    return cudaGetLastError();
}

cudaError_t launch_sync_verify(const uint8_t* payload, uint64_t data_offset, uint64_t total_bytes,
                               unsigned long long table_sum, StatusBlock* status, cudaStream_t st,
                               const ExpectTable* expect) {
    static const ExpectTable none = {};
    k_sync_verify<<<grid_for((total_bytes - data_offset) / 16), 256, 0, st>>>(
        payload, data_offset, total_bytes, table_sum, status, expect ? *expect : none);
    return cudaGetLastError();
}

cudaError_t launch_sync_scatter(const CopySeg* segs, int n, const StatusBlock* status, cudaStream_t st) {
    SegTable tab;
    uint64_t chunks = 0;
    tab.n = n;
    for (int i = 0; i < n; ++i) {
        tab.seg[i] = segs[i];
        chunks += (segs[i].bytes + 15) / 16;
    }
    if (chunks == 0) return cudaSuccess;
    k_sync_scatter<<<grid_for(chunks), 256, 0, st>>>(tab, status);
    return cudaGetLastError();
}

}  // namespace fp8bs
