// gemm_blockwise.cu -- blockwise (fp32-scale) FP8 GEMM on CTA pairs.
//
// Blockwise recipe (fp32 scales; "Jet-RL: Enabling On-Policy FP8 ...",
// "Kwantisatieschema"): the fp32 scales cannot be applied inside the MMA, so
// each K block is accumulated into a fresh TMEM buffer P (kind::f8f6f4) and
// the epilogue warps promote it into register accumulators:
//   acc[m][n] += P[m][n] * sa[kb][m] * sb(n, kb)
// with sb per 128x128 weight block (forward, DGrad) or per row of B (WGrad,
// whose operands come from 128x1 groups).
//
// Layout of the work (each choice measured on GB300 against its alternatives):
//  * a cluster of two CTAs on neighbouring SMs computes a 256x256 tile with
//    tcgen05.mma.cta_group::2, M=256, N=256: one MMA per 32-wide K step, so
//    a 128-wide K block is four MMAs (one thread issues a tcgen05 instruction
//    every ~60 cycles; N=128 halves would double that and starve the pipe);
//  * each CTA stages its 128 rows of A and its half (128 rows) of the tile's
//    B rows: 32 KB per SM per K block, four-stage TMA ring (measured faster
//    than six, five or three stages);
//  * two 256-column TMEM sets hold the partials of consecutive K blocks;
//    two threads issue the MMAs (even and odd K blocks), so the thread that
//    may reuse a set is never the one blocked issuing the other set;
//  * 16 epilogue warps per CTA hold the 128x256 fp32 result (64 accumulators
//    per thread, 32 columns of each N half) and read each partial in four
//    16-column chunks through a two-buffer software pipeline, handing the set
//    back to the leader CTA as soon as the last chunk is in registers;
//  * setmaxnreg gives the four epilogue warpgroups 112 registers and the
//    control warpgroup (TMA, two MMA issuers, scale loader) 32;
//  * a bf16 D tile leaves through shared memory: the epilogue warps write it
//    into a 128-byte-swizzled 64 KB tile and one thread stores it with four
//    asynchronous TMA stores, so the tile end no longer waits on 32 rows of
//    scattered 32-byte stores per warp instruction (1.65 us per tile).
#include "gemm_common.cuh"
#include "quant_common.cuh"

namespace fp8bs {

namespace {

constexpr int kBwBN = 256;                                 // tile columns (both CTAs)
constexpr int kBwStages = 4;                               // one 128-wide K block per stage
constexpr uint32_t kBwABytes = 128 * BK;                   // 16 KB: this CTA's 128 rows of A
constexpr uint32_t kBwBBytes = 128 * BK;                   // 16 KB: this CTA's 128 rows of B
constexpr uint32_t kBwStageBytes = kBwABytes + kBwBBytes;  // 32 KB
constexpr int kBwSets = 2;                                 // TMEM partial sets of 256 columns
constexpr uint32_t kBwTmemCols = 512;
constexpr int kBwEpi0 = 4;                                 // first epilogue warp (warpgroup 1)
constexpr int kBwEpiWarps = 16;                            // 4 per TMEM lane quarter
constexpr int kBwThreads = (kBwEpi0 + kBwEpiWarps) * 32;   // 640: five warpgroups
constexpr int kBwCols = kBwBN / (kBwEpiWarps / 4);         // 64 columns per epilogue thread
constexpr int kBwHalfCols = kBwCols / 2;                   // 32 of them in each 128-column N half
constexpr uint32_t kIdescBlockwise = idesc_f8f6f4(2 * BM, kBwBN);
// register split: 640 threads launch with 96 registers each (61440); the
// control warpgroup drops to 32 so that the epilogue can rise to 112
constexpr int kCtlRegs = 32, kEpiRegs = 112;
static_assert(4 * 32 * kCtlRegs + kBwEpiWarps * 32 * kEpiRegs <= kBwThreads * 96, "register split over budget");

struct alignas(16) BwBarriers {
    uint64_t full[kBwStages];       // leader: both CTAs' operand bytes of a stage landed
    uint64_t empty[kBwStages];      // stage consumed by the MMAs (both CTAs)
    uint64_t set_full[kBwSets];     // partial set written (both CTAs)
    uint64_t set_empty[kBwSets];    // leader: all 32 epilogue warps of the pair read the set
    uint64_t xch[4];                // per lane quarter: row maxima exchanged (fused quantization)
    uint64_t drain;                 // both issuers' MMAs completed (teardown)
    uint64_t d_staged;              // the 16 epilogue warps wrote their part of a D tile
    uint64_t d_free;                // the staged D tile has been read by its TMA stores
    uint32_t tmem_base;
    int abort;
};

constexpr int kBwScaleSlots = 8;
struct alignas(16) BwShared {
    uint64_t sc_full[kBwScaleSlots];   // scale slot filled (32 cp.async arrivals of the loader warp)
    uint64_t sc_empty[kBwScaleSlots];  // scale slot read by all epilogue warps
    float amax_xch[2][4][128];         // fused quantization: per-warp row maxima, double-buffered
    float sa[kBwScaleSlots][128];      // per K block: row scales of this CTA's 128 rows
    float sb[kBwScaleSlots][kBwBN];    // per K block: column scales (WGrad) or the two block scales at [.][0..1]
};

constexpr uint32_t kBwDStageBytes = 128 * kBwBN * 2;      // 64 KB: this CTA's bf16 D tile, 4 boxes of 128 x 64
constexpr size_t kSmemBlockwise =
    1024 + (size_t)kBwStages * kBwStageBytes + kBwDStageBytes + sizeof(BwBarriers) + sizeof(BwShared);
static_assert(sizeof(BwBarriers) % 16 == 0, "BwShared must start 16-byte aligned");
static_assert(kSmemBlockwise <= 232448, "blockwise shared memory over the 227 KB limit");

struct BwParams {
    const float* sa;
    const float* sb;
    int sb_per_row;
    int M, N, K;
    void* D;
    long long ldd;
    int d_f32;
    uint8_t* q_codes;
    float* q_scales;
    StatusBlock* st;
    int tiles_m, tiles_n;  // 256x256 cluster tiles
    int d_v8, q_v8;        // D rows / code rows allow 32-byte stores
    int d_tma;             // bf16 D stored through shared memory by TMA (tmD valid)
};

// {c, c} as one 64-bit register pair (the fp32x2 multiplier)
__device__ __forceinline__ uint64_t pair2(float c) {
    uint64_t x;
    asm("mov.b64 %0, {%1, %1};" : "=l"(x) : "f"(c));
    return x;
}

// acc2[i] += {P[2i], P[2i+1]} * c2, 16 columns (accumulator pairs held as
// 64-bit registers, packed fp32x2 FMAs)
__device__ __forceinline__ void promote16(uint64_t* acc2, const uint32_t* r, uint64_t c2) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint64_t x;
        asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "r"(r[2 * i]), "r"(r[2 * i + 1]));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[i]) : "l"(x), "l"(c2));
    }
}

// acc2[i] += ({P[2i], P[2i+1]} * {sb[2i], sb[2i+1]}) * {sa, sa}: per-column
// scales (WGrad), 16 columns, sb from shared memory
__device__ __forceinline__ void promote16_cols(uint64_t* acc2, const uint32_t* r, const float* sb, uint64_t sa2) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 v = *reinterpret_cast<const float4*>(sb + 4 * i);
        uint64_t s0, s1, x0, x1;
        asm("mov.b64 %0, {%1, %2};" : "=l"(s0) : "f"(v.x), "f"(v.y));
        asm("mov.b64 %0, {%1, %2};" : "=l"(s1) : "f"(v.z), "f"(v.w));
        asm("mov.b64 %0, {%1, %2};" : "=l"(x0) : "r"(r[4 * i]), "r"(r[4 * i + 1]));
        asm("mov.b64 %0, {%1, %2};" : "=l"(x1) : "r"(r[4 * i + 2]), "r"(r[4 * i + 3]));
        asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x0) : "l"(s0));
        asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x1) : "l"(s1));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[2 * i]) : "l"(x0), "l"(sa2));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[2 * i + 1]) : "l"(x1), "l"(sa2));
    }
}

// Cluster c of C visits the 256x256 tiles c, c + C, ...  Tile t is numbered
// down bands of 16 tile rows (the last band may be shorter): within a band the
// index walks down the rows first, then across the columns.  The clusters
// running at one time then share the A rows of one band and a few B column
// tiles, which stay in L2, instead of each column tile of B being fetched
// again for every row of tiles.
__device__ __forceinline__ void bw_tile(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
    constexpr int kBand = 16;
    const int band = t / (kBand * tiles_n);
    const int first = band * kBand;
    const int rows = tiles_m - first < kBand ? tiles_m - first : kBand;
    const int idx = t - band * kBand * tiles_n;
    tm = first + idx % rows;
    tn = idx / rows;
}

template <uint32_t R>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* smem_src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(smem_src)), "r"(x), "r"(y)
                 : "memory");
}

template <bool kColScales>
__global__ void __launch_bounds__(kBwThreads, 1)
    k_gemm_blockwise(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmD, const BwParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    uint8_t* dstage = smem + kBwStages * kBwStageBytes;  // 1024-byte aligned (the swizzle's period)
    BwBarriers* bar = reinterpret_cast<BwBarriers*>(dstage + kBwDStageBytes);
    BwShared* bws = reinterpret_cast<BwShared*>(bar + 1);
    volatile int* abort = &bar->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = p.K / BK;
    const int num_tiles = p.tiles_m * p.tiles_n;
    const int cid = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);
    const int my_tiles = cid < num_tiles ? (num_tiles - 1 - cid) / ncl + 1 : 0;
    const int total = my_tiles * KB;          // K blocks this CTA pair computes
    const uint32_t rank = cluster_ctarank();  // 0: leader CTA (issues the MMAs)
    const int row0 = BM * (int)rank;          // this CTA's rows within the 256-row tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < kBwStages; ++s) {
            mbar_init(&bar->full[s], 1);
            mbar_init(&bar->empty[s], 1);
        }
        for (int b = 0; b < kBwSets; ++b) {
            mbar_init(&bar->set_full[b], 1);
            mbar_init(&bar->set_empty[b], 2 * kBwEpiWarps);
        }
        for (int q = 0; q < 4; ++q) mbar_init(&bar->xch[q], kBwEpiWarps / 4);
        for (int i = 0; i < kBwScaleSlots; ++i) {
            mbar_init(&bws->sc_full[i], 32);
            mbar_init(&bws->sc_empty[i], kBwEpiWarps);
        }
        mbar_init(&bar->drain, 2);
        mbar_init(&bar->d_staged, kBwEpiWarps);
        mbar_init(&bar->d_free, 1);
        bar->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.d_tma) prefetch_tensormap(&tmD);
    }
    if (warp == 1) tmem_alloc_pair(&bar->tmem_base, kBwTmemCols);
    tc_fence_before();
    cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem = bar->tmem_base;

    if (warp < kBwEpi0) {
        regs_dec<kCtlRegs>();
        if (warp == 0) {
            // TMA producer: per K block, this CTA's 128 rows of A and 128 rows
            // of B, both completing on the leader CTA's full barrier
            if (lane == 0) {
                const uint32_t full_leader = mapa_shared(&bar->full[0], 0);  // + 8 * stage
                int tm = 0, tn = 0, kb = 0, ti = 0;
                for (int g = 0; g < total; ++g) {
                    if (kb == 0) bw_tile(cid + ti * ncl, p.tiles_m, p.tiles_n, tm, tn);
                    const int s = g % kBwStages;
                    if (!mbar_wait_bounded(&bar->empty[s], ((g / kBwStages) & 1) ^ 1, abort, p.st, 1)) break;
                    uint8_t* stage = smem + s * kBwStageBytes;
                    if (rank == 0) mbar_arrive_expect_tx(&bar->full[s], 2 * kBwStageBytes);
                    const uint32_t fb = full_leader + 8u * (uint32_t)s;
                    const int k0 = kb * BK;
                    tma_load_2d_pair(stage, &tmA, fb, k0, tm * 2 * BM + row0);
                    tma_load_2d_pair(stage + kBwABytes, &tmB, fb, k0, tn * kBwBN + 128 * (int)rank);
                    if (++kb == KB) {
                        kb = 0;
                        ++ti;
                    }
                }
            }
        } else if (warp == 1 || warp == 3) {
            // MMA issue (leader CTA): warp 1 the even K blocks (set 0), warp 3
            // the odd ones (set 1)
            if (lane == 0 && rank == 0) {
                for (int g = warp == 1 ? 0 : 1; g < total; g += 2) {
                    const int s = g % kBwStages;
                    const int set = g & 1;
                    if (!mbar_wait_bounded(&bar->full[s], (g / kBwStages) & 1, abort, p.st, 3)) break;
                    if (!mbar_wait_bounded(&bar->set_empty[set], ((g >> 1) & 1) ^ 1, abort, p.st, 6)) break;
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * kBwStageBytes);
                    const uint64_t adesc = sdesc_k_sw128(a_addr);
                    const uint64_t bdesc = sdesc_k_sw128(a_addr + kBwABytes);
                    const uint32_t dcol = tmem + (uint32_t)(256 * set);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        tc_mma_f8f6f4_pair(dcol, adesc + 2 * k, bdesc + 2 * k, kIdescBlockwise, k > 0 ? 1u : 0u);
                    tc_commit_pair(&bar->empty[s], 3);      // stage free in both CTAs
                    tc_commit_pair(&bar->set_full[set], 3);  // partial set ready in both CTAs
                }
                tc_commit_pair(&bar->drain, 1);
                mbar_wait_drain(&bar->drain, 0, p.st);
            }
        } else {
            // scale loader (warp 2): per K block, the row scales of this CTA's
            // 128 rows and the tile's column (WGrad) or two block scales, by
            // cp.async into ring slot g % 8; each lane's copies complete onto
            // sc_full
            const int nblocks = p.N / 128;
            int tm = 0, tn = 0, kb = 0, ti = 0;
            for (int g = 0; g < total; ++g) {
                if (kb == 0) bw_tile(cid + ti * ncl, p.tiles_m, p.tiles_n, tm, tn);
                const int slot = g % kBwScaleSlots;
                if (!mbar_wait_bounded(&bws->sc_empty[slot], ((g / kBwScaleSlots) & 1) ^ 1, abort, p.st, 7)) break;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int m = tm * 2 * BM + row0 + 4 * lane + i;
                    const bool ok = m < p.M;
                    const float* src = ok ? p.sa + (size_t)kb * p.M + m : p.sa;
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                                     smem_u32(&bws->sa[slot][4 * lane + i])),
                                 "l"(src), "r"(ok ? 4 : 0)
                                 : "memory");
                }
                if (!p.sb_per_row) {
                    if (lane < 2) {
                        const int nb = 2 * tn + lane;
                        const bool ok = nb < nblocks;
                        const float* src = ok ? p.sb + (size_t)nb * KB + kb : p.sb;
                        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                                         smem_u32(&bws->sb[slot][lane])),
                                     "l"(src), "r"(ok ? 4 : 0)
                                     : "memory");
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int col = tn * kBwBN + 8 * lane + 4 * i;
                        const bool ok = col < p.N;
                        const float* src = ok ? p.sb + (size_t)kb * p.N + col : p.sb;
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                                         smem_u32(&bws->sb[slot][8 * lane + 4 * i])),
                                     "l"(src), "r"(ok ? 16 : 0)
                                     : "memory");
                    }
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                                 smem_u32(&bws->sc_full[slot]))
                             : "memory");
                if (++kb == KB) {
                    kb = 0;
                    ++ti;
                }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
        }
    } else {
        regs_inc<kEpiRegs>();
        // epilogue: warp (q = warp % 4, w) promotes rows 32q.. of this CTA and,
        // in each 128-column N half h, tile columns 128h + 32w .. +31
        const int q = warp & 3, w = (warp - kBwEpi0) >> 2;
        const int rl = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t set_empty_leader = mapa_shared(&bar->set_empty[0], 0);  // + 8 * set

        bool ok = true;
        for (int ti = 0; ti < my_tiles && ok; ++ti) {
            int ctm, ctn;
            bw_tile(cid + ti * ncl, p.tiles_m, p.tiles_n, ctm, ctn);
            uint64_t acc2[kBwCols / 2];
#pragma unroll
            for (int i = 0; i < kBwCols / 2; ++i) acc2[i] = 0ull;
            // Software pipeline over the four 16-column chunks this warp reads
            // of each K block's partial (chunks 0, 1: N half 0; chunks 2, 3:
            // N half 1): the next chunk's TMEM load is in flight while the
            // current one is promoted, and the first chunk of the next K
            // block is loaded before the last chunk of this one is promoted.
            uint32_t ra[16], rb[16];
            {
                const int g0 = ti * KB;
                if (!mbar_wait_bounded(&bar->set_full[g0 & 1], (g0 >> 1) & 1, abort, p.st, 4)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_ld_32x32b_x16(tmem + lane_base + (uint32_t)(256 * (g0 & 1) + kBwHalfCols * w), ra);
                tmem_ld_wait();
                reg_fence16(ra);
            }
            for (int kb = 0; kb < KB; ++kb) {
                const int g = ti * KB + kb;
                const int slot = g % kBwScaleSlots;
                const int set = g & 1;
                if (!mbar_wait_bounded(&bws->sc_full[slot], (g / kBwScaleSlots) & 1, abort, p.st, 5)) {
                    ok = false;
                    break;
                }
                const float sa = bws->sa[slot][rl];
                // forward / DGrad: one multiplier per N half; WGrad: sa, with
                // the column scales read from shared memory per chunk
                const uint64_t cs0 = pair2(kColScales ? sa : sa * bws->sb[slot][0]);
                const uint64_t cs1 = kColScales ? cs0 : pair2(sa * bws->sb[slot][1]);
                const float* sb0 = &bws->sb[slot][kBwHalfCols * w];
                const float* sb1 = sb0 + 128;
                const uint32_t base = tmem + lane_base + (uint32_t)(256 * set + kBwHalfCols * w);
                // chunk 1 in flight, promote chunk 0
                tmem_ld_32x32b_x16(base + 16, rb);
                if (!kColScales) promote16(acc2, ra, cs0); else promote16_cols(acc2, ra, sb0, cs0);
                tmem_ld_wait();
                reg_fence16(rb);
                // chunk 2 in flight, promote chunk 1
                tmem_ld_32x32b_x16(base + 128, ra);
                if (!kColScales) promote16(acc2 + 8, rb, cs0); else promote16_cols(acc2 + 8, rb, sb0 + 16, cs0);
                tmem_ld_wait();
                reg_fence16(ra);
                // chunk 3 in flight, promote chunk 2
                tmem_ld_32x32b_x16(base + 144, rb);
                if (!kColScales) promote16(acc2 + 16, ra, cs1); else promote16_cols(acc2 + 16, ra, sb1, cs0);
                tmem_ld_wait();
                reg_fence16(rb);
                // this warp's share of the set is in registers: hand it back
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(set_empty_leader + 8u * (uint32_t)set);
                // first chunk of the next K block in flight, promote chunk 3
                const bool more = kb + 1 < KB;
                if (more) {
                    if (!mbar_wait_bounded(&bar->set_full[set ^ 1], ((g + 1) >> 1) & 1, abort, p.st, 4)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    tmem_ld_32x32b_x16(tmem + lane_base + (uint32_t)(256 * (set ^ 1) + kBwHalfCols * w), ra);
                }
                if (!kColScales) promote16(acc2 + 24, rb, cs1); else promote16_cols(acc2 + 24, rb, sb1 + 16, cs0);
                // the scale slot is no longer read by this warp
                __syncwarp();
                if (lane == 0) mbar_arrive(&bws->sc_empty[slot]);
                if (more) {
                    tmem_ld_wait();
                    reg_fence16(ra);
                }
            }
            if (!ok) {
                tmem_ld_wait();  // no TMEM load of this thread outlives the loop
                break;
            }

            // tile done: store D (and the fused 1x128 quantization)
            float acc[kBwCols];
#pragma unroll
            for (int i = 0; i < kBwCols / 2; ++i)
                asm("mov.b64 {%0, %1}, %2;" : "=f"(acc[2 * i]), "=f"(acc[2 * i + 1]) : "l"(acc2[i]));
            const int m = ctm * 2 * BM + row0 + rl;
            const bool row_ok = m < p.M;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int ncol0 = ctn * kBwBN + 128 * h + kBwHalfCols * w;
                const bool valid = row_ok && ncol0 < p.N;  // N % 128 == 0: a half is all in or all out
                const float* ah = acc + kBwHalfCols * h;
                if (p.d_f32) {
                    if (valid) {
                        float* drow = reinterpret_cast<float*>(p.D) + (size_t)m * p.ldd + ncol0;
                        if (p.d_v8) {
#pragma unroll
                            for (int i = 0; i < kBwHalfCols / 8; ++i) {
                                uint32_t wv[8];
#pragma unroll
                                for (int k = 0; k < 8; ++k) wv[k] = __float_as_uint(ah[8 * i + k]);
                                st_v8(drow + 8 * i, wv);
                            }
                        } else {
                            float4* d = reinterpret_cast<float4*>(drow);
#pragma unroll
                            for (int i = 0; i < kBwHalfCols / 4; ++i)
                                d[i] = make_float4(ah[4 * i], ah[4 * i + 1], ah[4 * i + 2], ah[4 * i + 3]);
                        }
                    }
                } else {
                    uint32_t packed[kBwHalfCols / 2];
#pragma unroll
                    for (int i = 0; i < kBwHalfCols / 2; ++i) packed[i] = pack_bf16x2(ah[2 * i], ah[2 * i + 1]);
                    if (p.d_tma) {
                        if (h == 0 && ti > 0) {
                            // the previous tile's TMA stores must have read the staged tile
                            if (warp == kBwEpi0 && lane == 0) {
                                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                                mbar_arrive(&bar->d_free);
                            }
                            if (!mbar_wait_bounded(&bar->d_free, (ti - 1) & 1, abort, p.st, 12)) {
                                ok = false;
                                break;
                            }
                        }
                        // box c = 2h + w/2 holds tile columns 64c .. 64c + 63: this
                        // thread's 32 columns are 16-byte units 4 (w % 2) .. + 3 of its
                        // 128-byte row there, each unit index xor-ed with row % 8
                        uint8_t* rowp = dstage + (2 * h + (w >> 1)) * 16384 + rl * 128;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<uint4*>(rowp + ((((w & 1) * 4 + j) ^ (rl & 7)) << 4)) =
                                make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                    } else if (valid) {
                        uint16_t* drow = reinterpret_cast<uint16_t*>(p.D) + (size_t)m * p.ldd + ncol0;
                        if (p.d_v8) {
                            st_v8(drow, packed);
                            st_v8(drow + 16, packed + 8);
                        } else {
                            uint4* d = reinterpret_cast<uint4*>(drow);
#pragma unroll
                            for (int i = 0; i < kBwHalfCols / 8; ++i)
                                d[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                        }
                    }
                    if (p.q_codes != nullptr) {
                        // a 1x128 group of a row is one N half: the four warps of
                        // this lane quarter hold 32 columns each and exchange
                        // their maxima through shared memory (double-buffered by
                        // exchange parity, bounded wait)
                        float a = 0.0f;
#pragma unroll
                        for (int i = 0; i < kBwHalfCols / 2; ++i)
                            a = fmaxf(a, fmaxf(fabsf(bf16_lo(packed[i])), fabsf(bf16_hi(packed[i]))));
                        const int e = 2 * ti + h;  // exchange number
                        float (*xs)[128] = bws->amax_xch[e & 1];
                        xs[w][rl] = a;
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar->xch[q]);
                        if (!mbar_wait_bounded(&bar->xch[q], e & 1, abort, p.st, 8)) {
                            ok = false;
                            break;
                        }
                        a = fmaxf(fmaxf(xs[0][rl], xs[1][rl]), fmaxf(xs[2][rl], xs[3][rl]));
                        const float sc = group_scale_bf16(a);  // D was rounded to bf16
                        const Divider dv = make_divider(sc);
                        if (valid) {
                            uint8_t* codes = p.q_codes + (size_t)m * p.N + ncol0;
                            uint32_t cw[kBwHalfCols / 4];
#pragma unroll
                            for (int i = 0; i < kBwHalfCols / 8; ++i) {
                                float f[8];
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    f[2 * k] = bf16_lo(packed[4 * i + k]);
                                    f[2 * k + 1] = bf16_hi(packed[4 * i + k]);
                                }
                                const uint2 c = encode8_div(f, dv);
                                cw[2 * i] = c.x;
                                cw[2 * i + 1] = c.y;
                            }
                            if (p.q_v8) {
                                st_v8(codes, cw);
                            } else {
                                reinterpret_cast<uint4*>(codes)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                                reinterpret_cast<uint4*>(codes)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
                            }
                            if (w == 0) p.q_scales[(size_t)(ncol0 / 128) * p.M + m] = sc;
                        }
                    }
                }
            }
            if (p.d_tma && ok) {
                // the tile is staged once all 16 warps arrived; one thread
                // stores its four boxes (rows and columns outside D are clipped)
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->d_staged);
                if (warp == kBwEpi0) {
                    bool issued = true;
                    if (lane == 0) {
                        issued = mbar_wait_bounded(&bar->d_staged, ti & 1, abort, p.st, 13);
                        if (issued) {
                            const int y = ctm * 2 * BM + row0;
#pragma unroll
                            for (int c = 0; c < 4; ++c) tma_store_2d(&tmD, dstage + c * 16384, ctn * kBwBN + 64 * c, y);
                            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, issued ? 1 : 0, 0) != 0;
                }
            }
        }
    }

    // the last D tile's TMA stores complete before the CTA's shared memory goes
    if (p.d_tma && warp == kBwEpi0 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    // neither CTA leaves while the other may still signal its barriers or
    // the leader's MMAs may still write its TMEM
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, kBwTmemCols);
    }
}

}  // namespace

cudaError_t launch_gemm_blockwise(const GemmBlockwiseArgs& a, StatusBlock* status, cudaStream_t st) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    CUtensorMap tmA, tmB, tmD;
    if (!make_map(&tmA, a.a_codes, (uint64_t)a.K, (uint64_t)a.M, BM) ||
        !make_map(&tmB, a.b_codes, (uint64_t)a.K, (uint64_t)a.N, 128))
        return cudaErrorInvalidValue;
    // bf16 D leaves through shared memory and TMA stores when its base and
    // row pitch are 16-byte aligned; otherwise, and for WGrad (whose
    // per-column promotion keeps shared memory busier; measured 0.8 % slower
    // with the staged store), each thread stores its rows
    memset(&tmD, 0, sizeof(tmD));
    const bool d_tma = !a.d_f32 && !a.sb_per_row && reinterpret_cast<uintptr_t>(a.D) % 16 == 0 &&
                       (a.ldd * 2) % 16 == 0 &&
                       make_map_store_bf16(&tmD, a.D, (uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.ldd);
    BwParams p;
    p.sa = a.sa;
    p.sb = a.sb;
    p.sb_per_row = a.sb_per_row;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.D = a.D;
    p.ldd = a.ldd;
    p.d_f32 = a.d_f32;
    p.q_codes = a.q_codes;
    p.q_scales = a.q_scales;
    p.st = status;
    p.tiles_m = (int)((a.M + 2 * BM - 1) / (2 * BM));
    p.tiles_n = (int)((a.N + kBwBN - 1) / kBwBN);
    const int64_t row_bytes = a.ldd * (a.d_f32 ? 4 : 2);
    p.d_v8 = (reinterpret_cast<uintptr_t>(a.D) % 32 == 0) && (row_bytes % 32 == 0);
    p.q_v8 = reinterpret_cast<uintptr_t>(a.q_codes) % 32 == 0;
    p.d_tma = d_tma ? 1 : 0;
    const int tiles = p.tiles_m * p.tiles_n;
    auto kfn = a.sb_per_row ? k_gemm_blockwise<true> : k_gemm_blockwise<false>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBlockwise);
    if (e != cudaSuccess) return e;
    // persistent grid of CTA pairs (clusters of 2): as many as can be resident
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)tiles);
    cfg.blockDim = dim3(kBwThreads);
    cfg.dynamicSmemBytes = kSmemBlockwise;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int max_pairs[64] = {0};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int& mp = max_pairs[dev & 63];
    if (mp <= 0) {
        e = cudaOccupancyMaxActiveClusters(&mp, kfn, &cfg);
        if (e != cudaSuccess) return e;
        if (mp <= 0) return cudaErrorInvalidConfiguration;
    }
    const int pairs = tiles < mp ? tiles : mp;
    cfg.gridDim = dim3(2 * (unsigned)pairs);
    return cudaLaunchKernelEx(&cfg, kfn, tmA, tmB, tmD, p);
}

}  // namespace fp8bs
