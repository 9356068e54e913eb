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
// Checksum (payload format version 2): over the 8-byte words w_i at byte
// offsets 8i >= 64, with lo_i, hi_i their 32-bit halves, the sum mod 2^64 of
//   ((lo_i + i * 0x9E3779B9) mod 2^32) * ((hi_i + i * 0x85EBCA6B) mod 2^32),
// the NH inner product of UMAC (Black, Halevi, Krawczyk, Krovetz, Rogaway,
// CRYPTO 1999) keyed by the word index: one 32x32->64 multiply-add per word.
// Being a sum, it can be accumulated in any order.
#include "common.cuh"
#include "kernels.h"

namespace fp8bs {

namespace {

// The checksum terms of one 16-byte chunk: words (v.x, v.y) at word index
// i0 and (v.z, v.w) at i0 + 1 (keys need the index modulo 2^32 only).
__device__ __forceinline__ unsigned long long chunk_terms(const uint4& v, uint64_t i0) {
    constexpr uint32_t kK1 = 0x9E3779B9u, kK2 = 0x85EBCA6Bu;
    const uint32_t i = (uint32_t)i0;
    const uint32_t a0 = v.x + i * kK1, b0 = v.y + i * kK2;
    const uint32_t a1 = v.z + (i + 1u) * kK1, b1 = v.w + (i + 1u) * kK2;
    return (unsigned long long)a0 * b0 + (unsigned long long)a1 * b1;
}

struct SegTable {
    CopySeg seg[kMaxCopySegs];
    int n;
};

// chunk c of 16 bytes -> its segment: the last s with start[s] <= c, by
// binary search over the per-segment chunk offsets (up to 32 segments)
__device__ __forceinline__ int find_seg(const uint64_t* start, int n, uint64_t c) {
    int lo = 0, hi = n;  // start[lo] <= c < start[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start[mid] <= c) lo = mid; else hi = mid;
    }
    return lo;
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

constexpr int kUnroll = 4;

// hdr.bytes != 0: block 0 also writes the payload's header and entry table
// (every byte but the checksum field, which the caller zeroed) and adds the
// table's share of the checksum, so the whole pack is device work.
__global__ void __launch_bounds__(256) k_sync_pack(const SegTable tab, unsigned long long* checksum_field,
                                                   const __grid_constant__ ExpectTable hdr,
                                                   unsigned long long table_sum) {
    __shared__ uint64_t start[kMaxCopySegs + 1];
    if (blockIdx.x == 0 && hdr.bytes != 0) {
        uint8_t* head = reinterpret_cast<uint8_t*>(checksum_field) - 32;
        for (uint32_t i = threadIdx.x; i < hdr.bytes; i += blockDim.x)
            if (i < 32 || i >= 40) head[i] = hdr.data[i];
        if (threadIdx.x == 0) atomicAdd(checksum_field, table_sum);
    }
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
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    unsigned long long sum = 0;
    // kUnroll chunks per thread and round, all loads issued before any store
    for (uint64_t c = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; c < chunks; c += kUnroll * stride) {
        uint4 v[kUnroll];
        int sidx[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint64_t cc = c + u * stride;
            if (cc < chunks) {
                sidx[u] = find_seg(start, tab.n, cc);
                const CopySeg& sg = tab.seg[sidx[u]];
                v[u] = load16_tail(sg.src, (cc - start[sidx[u]]) * 16, sg.bytes);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint64_t cc = c + u * stride;
            if (cc < chunks) {
                const CopySeg& sg = tab.seg[sidx[u]];
                const uint64_t off = (cc - start[sidx[u]]) * 16;
                *reinterpret_cast<uint4*>(sg.dst + off) = v[u];
                sum += chunk_terms(v[u], sg.dst_word0 + off / 8);
            }
        }
    }
    const unsigned long long bs = block_sum(sum);
    if (threadIdx.x == 0 && bs != 0) atomicAdd(checksum_field, bs);
}

// Checksum of the data region of the payload (this block's share) and, in
// block 0, the header/table check; returns the block's partial sum (valid in
// thread 0).
__device__ __forceinline__ unsigned long long verify_part(const uint8_t* __restrict__ payload, uint64_t data_offset,
                                                          uint64_t total_bytes, StatusBlock* st,
                                                          const ExpectTable& expect) {
    if (blockIdx.x == 0 && expect.bytes != 0) {
        // header and entry table against what the destinations imply (the
        // checksum field, bytes 32..39, is what the data is checked against)
        bool bad = false;
        for (uint32_t i = threadIdx.x; i < expect.bytes; i += blockDim.x)
            if ((i < 32 || i >= 40) && payload[i] != expect.data[i]) bad = true;
        if (__syncthreads_or(bad) && threadIdx.x == 0) atomicExch(&st->header_bad, 1u);
    }
    const uint64_t c0 = data_offset / 16, c1 = total_bytes / 16;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint4* p4 = reinterpret_cast<const uint4*>(payload);
    unsigned long long sum = 0;
    auto mix_chunk = [&](const uint4& v, uint64_t cc) { sum += chunk_terms(v, 2 * cc); };
    // whole rounds of kUnroll chunks: one bounds check per round, and the
    // next round's loads issued before this round is mixed
    uint64_t c = c0 + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t span = (kUnroll - 1) * stride;
    if (c + span < c1) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = p4[c + u * stride];
        while (true) {
            const uint64_t cn = c + kUnroll * stride;
            const bool more = cn + span < c1;
            uint4 nv[kUnroll];
            if (more) {
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) nv[u] = p4[cn + u * stride];
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) mix_chunk(v[u], c + u * stride);
            c = cn;
            if (!more) break;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) v[u] = nv[u];
        }
    }
    // this thread's last chunks (fewer than kUnroll)
    for (; c < c1; c += stride) mix_chunk(p4[c], c);
    return block_sum(sum);
}

// ---- arrival at the end of the checksum pass (thread 0 of each block)
__device__ __forceinline__ unsigned int atom_add_acq_rel_gpu(unsigned int* p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned int ld_relaxed_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned int* p, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Adds the block's partial sum (a reduction that does not wait for its
// result) and counts the block in with one acq_rel increment, which orders
// the sum before it; true in the block that arrives last, which then sees
// every block's sum and the header/table flag of block 0.
__device__ __forceinline__ bool arrive_last(StatusBlock* st, unsigned long long bs) {
    if (bs != 0) atomicAdd(&st->sum, bs);
    return atom_add_acq_rel_gpu(&st->blocks_done, 1u) == gridDim.x - 1;
}

// In the last block: the verdict (1 when the sum or the header/table check
// fails), written to the status block.  `stored` is the payload's checksum
// field, read when the block started.
__device__ __forceinline__ unsigned int decide_verdict(StatusBlock* st, unsigned long long table_sum,
                                                       unsigned long long stored, unsigned int& header_bad) {
    const unsigned long long total = ld_relaxed_gpu(&st->sum) + table_sum;
    header_bad = ld_relaxed_gpu(&st->header_bad);
    const unsigned int bad = (total != stored || header_bad) ? 1u : 0u;
    st->verdict = bad;
    return bad;
}

// After the verdict is out: error bits, and the accumulators reset for the
// next call (which runs after this kernel in stream order).
__device__ __forceinline__ void close_verdict(StatusBlock* st, unsigned int bad, unsigned int header_bad) {
    if (header_bad) atomicOr(&st->error_bits, kErrBadPayload);
    else if (bad) atomicOr(&st->error_bits, kErrChecksum);
    st->sum = 0;
    st->header_bad = 0;
    st->blocks_done = 0;
}

// This block's share of the segment copies payload -> destinations.
__device__ __forceinline__ void scatter_part(const SegTable& tab) {
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
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t c = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; c < chunks; c += kUnroll * stride) {
        uint4 v[kUnroll];
        int sidx[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint64_t cc = c + u * stride;
            if (cc < chunks) {
                sidx[u] = find_seg(start, tab.n, cc);
                // payload side: padded to 16 bytes and aligned
                v[u] = *reinterpret_cast<const uint4*>(tab.seg[sidx[u]].src + (cc - start[sidx[u]]) * 16);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint64_t cc = c + u * stride;
            if (cc >= chunks) continue;
            const CopySeg& sg = tab.seg[sidx[u]];
            const uint64_t off = (cc - start[sidx[u]]) * 16;
            if (off + 16 <= sg.bytes) {
                *reinterpret_cast<uint4*>(sg.dst + off) = v[u];
            } else {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                for (uint64_t i = 0; off + i < sg.bytes; ++i) sg.dst[off + i] = (uint8_t)(w[i / 4] >> (8 * (i % 4)));
            }
        }
    }
}

__global__ void __launch_bounds__(256) k_sync_verify(const uint8_t* __restrict__ payload, uint64_t data_offset,
                                                     uint64_t total_bytes, unsigned long long table_sum,
                                                     StatusBlock* st, const __grid_constant__ ExpectTable expect) {
    unsigned long long stored = 0;
    if (threadIdx.x == 0) stored = *reinterpret_cast<const unsigned long long*>(payload + 32);
    const unsigned long long bs = verify_part(payload, data_offset, total_bytes, st, expect);
    if (threadIdx.x == 0 && arrive_last(st, bs)) {
        unsigned int header_bad;
        const unsigned int bad = decide_verdict(st, table_sum, stored, header_bad);
        close_verdict(st, bad, header_bad);
    }
}

__global__ void __launch_bounds__(256) k_sync_scatter(const SegTable tab, const StatusBlock* st) {
    if (*reinterpret_cast<const volatile unsigned int*>(&st->verdict) != 0) return;
    scatter_part(tab);
}

// Verify and scatter in one cooperative launch (every block resident): the
// blocks checksum the payload, meet at a grid barrier kept in the status
// block, and copy only if the verdict is clean -- no destination byte is
// written before the whole payload has been verified.  The second read of
// the payload mostly hits L2.  The block that arrives last decides and
// releases the others with one store of the barrier generation, which
// carries the verdict (+2 clean, +3 mismatch), so the barrier costs the
// arrival increment, one load of the sum and that store.  The wait is
// bounded: on expiry the block records a timeout (site 40) and copies
// nothing.
__global__ void __launch_bounds__(256) k_sync_install(const uint8_t* __restrict__ payload, uint64_t data_offset,
                                                      uint64_t total_bytes, unsigned long long table_sum,
                                                      StatusBlock* st, const __grid_constant__ ExpectTable expect,
                                                      const __grid_constant__ SegTable tab) {
    __shared__ unsigned int proceed;
    unsigned int gen0 = 0;
    unsigned long long stored = 0;
    if (threadIdx.x == 0) {
        gen0 = ld_relaxed_gpu(&st->barrier_gen);
        stored = *reinterpret_cast<const unsigned long long*>(payload + 32);
    }
    const unsigned long long bs = verify_part(payload, data_offset, total_bytes, st, expect);
    if (threadIdx.x == 0) {
        unsigned int go;
        if (arrive_last(st, bs)) {
            unsigned int header_bad;
            const unsigned int bad = decide_verdict(st, table_sum, stored, header_bad);
            st_release_gpu(&st->barrier_gen, gen0 + 2u + bad);
            close_verdict(st, bad, header_bad);
            go = bad ? 0u : 1u;
        } else {
            const unsigned long long t0 = global_timer_ns();
            unsigned int g;
            while ((g = ld_acquire_gpu(&st->barrier_gen)) == gen0) {
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    report_timeout(st, 40);
                    break;
                }
                __nanosleep(64);
            }
            go = g == gen0 + 2u ? 1u : 0u;
        }
        proceed = go;
    }
    __syncthreads();
    if (proceed) scatter_part(tab);
}

// Blocks for a grid-stride copy of `chunks` 16-byte chunks: no more than fit
// on the device at once (SM count x resident blocks of `kernel`, looked up
// once per device and kernel), so that no block waits for a second wave.
template <typename Kernel>
int grid_for(Kernel kernel, uint64_t chunks) {
    static int resident[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    int& r = resident[dev & 63];
    if (r == 0) {
        int sms = 0, per_sm = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0);
        r = sms * (per_sm > 0 ? per_sm : 1);
    }
    uint64_t b = (chunks + 256 * kUnroll - 1) / (256 * kUnroll);
    if (b > (uint64_t)r) b = (uint64_t)r;
    return b == 0 ? 1 : (int)b;
}

// Diagnostic: one warp waits on a shared-memory mbarrier that nothing will
// complete, giving up after limit_ns exactly as every bounded wait of the
// library does (timeout recorded in the status block, site 90), then
// returns -- the path taken when a peer of a real wait never signals.
__global__ void k_wait_expiry(unsigned long long limit_ns, StatusBlock* st) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x != 0) return;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(&bar, 0)) {
        if (global_timer_ns() - t0 > limit_ns) {
            report_timeout(st, 90);
            return;
        }
        __nanosleep(1000);
    }
}

}  // namespace

cudaError_t launch_wait_expiry(unsigned long long limit_ns, StatusBlock* status, cudaStream_t st) {
    k_wait_expiry<<<1, 32, 0, st>>>(limit_ns, status);
    return cudaGetLastError();
}

cudaError_t launch_sync_pack(const CopySeg* segs, int n, unsigned long long* checksum_field, const ExpectTable* hdr,
                             unsigned long long table_sum, cudaStream_t st) {
    static const ExpectTable none = {};
    SegTable tab;
    uint64_t chunks = 0;
    tab.n = n;
    for (int i = 0; i < n; ++i) {
        tab.seg[i] = segs[i];
        chunks += segs[i].padded / 16;
    }
    if (chunks == 0 && hdr == nullptr) return cudaSuccess;
    const unsigned grid = chunks == 0 ? 1u : grid_for(k_sync_pack, chunks);
    k_sync_pack<<<grid, 256, 0, st>>>(tab, checksum_field, hdr ? *hdr : none, table_sum);
    return cudaGetLastError();
}

cudaError_t launch_sync_verify(const uint8_t* payload, uint64_t data_offset, uint64_t total_bytes,
                               unsigned long long table_sum, StatusBlock* status, cudaStream_t st,
                               const ExpectTable* expect) {
    static const ExpectTable none = {};
    k_sync_verify<<<grid_for(k_sync_verify, (total_bytes - data_offset) / 16), 256, 0, st>>>(
        payload, data_offset, total_bytes, table_sum, status, expect ? *expect : none);
    return cudaGetLastError();
}

cudaError_t launch_sync_install(const uint8_t* payload, uint64_t data_offset, uint64_t total_bytes,
                                unsigned long long table_sum, StatusBlock* status, const ExpectTable* expect,
                                const CopySeg* segs, int n, cudaStream_t st) {
    static const ExpectTable none = {};
    static int coop[64] = {}, resident[64] = {};   // per device: 1 supported / 2 not; blocks that fit at once
    int dev = 0;
    cudaGetDevice(&dev);
    dev &= 63;
    if (coop[dev] == 0) {
        int attr = 0, sms = 0, per_sm = 0;
        cudaDeviceGetAttribute(&attr, cudaDevAttrCooperativeLaunch, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_sync_install, 256, 0);
        resident[dev] = sms * per_sm;
        coop[dev] = (attr && resident[dev] > 0) ? 1 : 2;
    }
    if (n > kMaxCopySegs || coop[dev] != 1) return cudaErrorNotSupported;
    SegTable tab;
    tab.n = n;
    for (int i = 0; i < n; ++i) tab.seg[i] = segs[i];
    const ExpectTable* et = expect ? expect : &none;
    const int grid = grid_for(k_sync_install, (total_bytes - data_offset) / 16);
    void* args[] = {(void*)&payload, (void*)&data_offset, (void*)&total_bytes, (void*)&table_sum, (void*)&status,
                    (void*)et, (void*)&tab};
    return cudaLaunchCooperativeKernel((const void*)k_sync_install, dim3(grid), dim3(256), args, 0, st);
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
    k_sync_scatter<<<grid_for(k_sync_scatter, chunks), 256, 0, st>>>(tab, status);
    return cudaGetLastError();
}

}  // namespace fp8bs
