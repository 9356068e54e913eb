// gemm_blockwise.cu -- blockwise (fp32-scale) FP8 GEMM on CTA pairs.
//
// Blockwise recipe (fp32 scales; "Jet-RL: Enabling On-Policy FP8 ...",
// "Kwantisatieschema"): the fp32 scales cannot be applied inside the MMA, so
// each K block is accumulated into a fresh TMEM buffer P (kind::f8f6f4) and
// the epilogue warps promote it into register accumulators:
//   acc[m][n] += P[m][n] * sa[kb][m] * sb(n, kb)
// with sb per 128x128 weight block (forward, DGrad) or per row of B (WGrad,
// whose operands come from 128x1 groups).  CTA pairs compute 256x256 tiles;
// 16 epilogue warps per CTA hold a 128x256 fp32 result (64 accumulators per
// thread); a scale-loader warp stages sa/sb through shared memory.
#include "gemm_common.cuh"

namespace fp8bs {

namespace {

// blockwise kernel: a cluster of two CTAs on neighbouring SMs computes a
// 256x256 tile with tcgen05.mma.cta_group::2 (M=256, N=128, two N halves per
// K step).  Each CTA stages its own 128 rows of A and, of each 128-column N
// half, the 64 rows of B it contributes, so an SM takes in 32 KB per
// 128x256x128 of work -- half of what a 128x128 tile needs.  Each CTA keeps
// a 128x256 fp32 result in its 16 epilogue warps (64 columns each); the
// per-K-block partials P live in two TMEM sets of 256 columns, so the
// tensor cores fill one set while the epilogue promotes the other.
constexpr int kBwBN = 256;                               // tile columns (both CTAs)
constexpr int kBwStages = 6;                             // one 128-wide K block per stage
constexpr uint32_t kBwABytes = 128 * BK;                 // 16 KB: this CTA's 128 rows of A
constexpr uint32_t kBwBQuarter = 64 * BK;                // 8 KB: 64 rows of B (one N half's share)
constexpr uint32_t kBwStageBytes = kBwABytes + 2 * kBwBQuarter;  // 32 KB
constexpr uint32_t kBwTmemCols = 512;
constexpr int kBwEpiWarps = 16;                          // 4 per TMEM lane quarter
constexpr int kBwLoaderWarp = kEpiWarp0 + kBwEpiWarps;   // fills the scale ring
constexpr int kBwThreads = (kBwLoaderWarp + 1) * 32;     // 608
constexpr int kBwCols = kBwBN / (kBwEpiWarps / 4);       // 64 columns per epilogue thread
constexpr uint32_t kIdescBlockwise = idesc_f8f6f4(2 * BM, 128);

// blockwise kernel only (16-byte aligned: float4 reads and 16-byte cp.async)
constexpr int kBwScaleSlots = 8;
struct alignas(16) BwShared {
    uint64_t sc_full[kBwScaleSlots];   // scale slot filled (32 cp.async arrivals of the loader warp)
    uint64_t sc_empty[kBwScaleSlots];  // scale slot read by all epilogue warps
    float amax_xch[kBwEpiWarps / 4][128];  // fused quantization: per-warp row maxima
    float sa[kBwScaleSlots][128];      // per K block: row scales of this CTA's 128 rows
    float sb[kBwScaleSlots][kBwBN];    // per K block: column scales (WGrad) or the two block scales at [.][0..1]
};


constexpr size_t kSmemBlockwise = 1024 + (size_t)kBwStages * kBwStageBytes + sizeof(Barriers) + sizeof(BwShared);
static_assert(sizeof(Barriers) % 16 == 0, "BwShared must start 16-byte aligned");
static_assert(kSmemBlockwise <= 232448, "blockwise shared memory over the 227 KB limit");

// ===========================================================================
// Blockwise (fp32-scale) GEMM with promotion
// ===========================================================================
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
};

// acc[2i..2i+1] += (P * c) with packed fp32x2 FMAs, 16 columns
__device__ __forceinline__ void promote16x2(float* acc, const uint32_t (&r)[16], float c) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        asm("{\n\t.reg .b64 a, x, y;\n\t"
            "mov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\t"
            "fma.rn.f32x2 a, x, y, a;\n\tmov.b64 {%0, %1}, a;\n\t}\n"
            : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
            : "f"(__uint_as_float(r[2 * i])), "f"(__uint_as_float(r[2 * i + 1])), "f"(c));
}

// acc += (P * sb) * sa with per-column sb (16 columns, sb from shared memory)
__device__ __forceinline__ void promote16x2_cols(float* acc, const uint32_t (&r)[16], const float* sb, float sa) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 v = *reinterpret_cast<const float4*>(sb + 4 * i);
        const float sv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 2; ++k)
            asm("{\n\t.reg .b64 a, x, s, t;\n\t"
                "mov.b64 a, {%0, %1};\n\tmov.b64 x, {%2, %3};\n\tmov.b64 s, {%4, %5};\n\tmov.b64 t, {%6, %6};\n\t"
                "mul.rn.f32x2 x, x, s;\n\tfma.rn.f32x2 a, x, t, a;\n\tmov.b64 {%0, %1}, a;\n\t}\n"
                : "+f"(acc[4 * i + 2 * k]), "+f"(acc[4 * i + 2 * k + 1])
                : "f"(__uint_as_float(r[4 * i + 2 * k])), "f"(__uint_as_float(r[4 * i + 2 * k + 1])),
                  "f"(sv[2 * k]), "f"(sv[2 * k + 1]), "f"(sa));
    }
}

// Cluster c of C visits the 256x256 tiles c, c + C, ...; its g-th K block
// (over all its tiles) is K block g % KB of tile c + (g / KB) * C.
__device__ __forceinline__ void bw_tile(int t, int tiles_n, int& tm, int& tn) {
    tm = t / tiles_n;
    tn = t - tm * tiles_n;
}

__global__ void __launch_bounds__(kBwThreads, 1)
    k_gemm_blockwise(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const BwParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    Barriers* bar = reinterpret_cast<Barriers*>(smem + kBwStages * kBwStageBytes);
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
        // full[s] (used in the leader only): the leader producer's expect_tx
        // arrival for both CTAs' bytes plus one arrival from each epilogue
        // warp of both CTAs granting its share of the TMEM set to the stage
        for (int s = 0; s < kBwStages; ++s) {
            mbar_init(&bar->full[s], 1 + 2 * kBwEpiWarps);
            mbar_init(&bar->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) mbar_init(&bar->acc_full[b], 1);
        for (int i = 0; i < kBwScaleSlots; ++i) {
            mbar_init(&bws->sc_full[i], 32);
            mbar_init(&bws->sc_empty[i], kBwEpiWarps);
        }
        mbar_init(&bar->drain, 1);
        bar->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) tmem_alloc_pair(&bar->tmem_base, kBwTmemCols);
    tc_fence_before();
    cluster_sync();  // barriers initialised and TMEM allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem = bar->tmem_base;
    const uint32_t full_leader = mapa_shared(&bar->full[0], 0);  // + 8 * stage

    if (warp == 0) {
        if (lane == 0) {
            int tm = 0, tn = 0, kb = 0, ti = 0;
            for (int g = 0; g < total; ++g) {
                if (kb == 0) bw_tile(cid + ti * ncl, p.tiles_n, tm, tn);
                const int s = g % kBwStages;
                if (!mbar_wait_bounded(&bar->empty[s], ((g / kBwStages) & 1) ^ 1, abort, p.st, 1)) break;
                uint8_t* stage = smem + s * kBwStageBytes;
                if (rank == 0) mbar_arrive_expect_tx(&bar->full[s], 2 * kBwStageBytes);
                const uint32_t fb = full_leader + 8u * (uint32_t)s;
                const int k0 = kb * BK, by = tn * kBwBN + 64 * (int)rank;
                tma_load_2d_pair(stage, &tmA, fb, k0, tm * 2 * BM + row0);
                tma_load_2d_pair(stage + kBwABytes, &tmB, fb, k0, by);
                tma_load_2d_pair(stage + kBwABytes + kBwBQuarter, &tmB, fb, k0, by + 128);
                if (++kb == KB) {
                    kb = 0;
                    ++ti;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            for (int g = 0; g < total; ++g) {
                const int s = g % kBwStages;
                if (!mbar_wait_bounded(&bar->full[s], (g / kBwStages) & 1, abort, p.st, 3)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + s * kBwStageBytes);
                const uint64_t adesc = sdesc_k_sw128(a_addr);
                const uint32_t pset = tmem + (uint32_t)((g & 1) * kBwBN);
#pragma unroll
                for (int nh = 0; nh < 2; ++nh) {
                    const uint64_t bdesc = sdesc_k_sw128(a_addr + kBwABytes + nh * kBwBQuarter);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        tc_mma_f8f6f4_pair(pset + (uint32_t)(128 * nh), adesc + 2 * k, bdesc + 2 * k, kIdescBlockwise,
                                           k > 0 ? 1u : 0u);
                }
                tc_commit_pair(&bar->empty[s], 3);        // stage free in both CTAs
                tc_commit_pair(&bar->acc_full[g & 1], 3);  // P set ready in both CTAs
            }
            tc_commit_pair(&bar->drain, 1);
            mbar_wait_drain(&bar->drain, 0, p.st);
        }
    } else if (warp == kBwLoaderWarp) {
        // scale loader: per K block, the row scales of this CTA's 128 rows and
        // the tile's column (WGrad) or two block scales, by cp.async into ring
        // slot g % 8; each lane's copies complete onto sc_full.
        const int nblocks = p.N / 128;
        int tm = 0, tn = 0, kb = 0, ti = 0;
        for (int g = 0; g < total; ++g) {
            if (kb == 0) bw_tile(cid + ti * ncl, p.tiles_n, tm, tn);
            const int slot = g % kBwScaleSlots;
            if (!mbar_wait_bounded(&bws->sc_empty[slot], ((g / kBwScaleSlots) & 1) ^ 1, abort, p.st, 7)) break;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = tm * 2 * BM + row0 + 4 * lane + i;
                const bool ok = m < p.M;
                const float* src = ok ? p.sa + (size_t)kb * p.M + m : p.sa;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(&bws->sa[slot][4 * lane + i])),
                             "l"(src), "r"(ok ? 4 : 0)
                             : "memory");
            }
            if (!p.sb_per_row) {
                if (lane < 2) {
                    const int nb = 2 * tn + lane;
                    const bool ok = nb < nblocks;
                    const float* src = ok ? p.sb + (size_t)nb * KB + kb : p.sb;
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(&bws->sb[slot][lane])),
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
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&bws->sc_full[slot]))
                         : "memory");
            if (++kb == KB) {
                kb = 0;
                ++ti;
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // epilogue: warp (q = warp % 4, h) promotes rows 32q.. of this CTA,
        // tile columns 64h .. 64h+63 (N half h / 2)
        const int q = warp & 3, h = (warp - kEpiWarp0) >> 2;
        const int rl = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        // grant the TMEM sets of K blocks 0 and 1
        if (lane == 0) {
            mbar_arrive_cluster(full_leader);
            mbar_arrive_cluster(full_leader + 8u);
        }

        bool ok = true;
        for (int ti = 0; ti < my_tiles && ok; ++ti) {
            int ctm, ctn;
            bw_tile(cid + ti * ncl, p.tiles_n, ctm, ctn);
            float acc[kBwCols];
#pragma unroll
            for (int i = 0; i < kBwCols; ++i) acc[i] = 0.0f;
            for (int kb = 0; kb < KB; ++kb) {
                const int g = ti * KB + kb;
                const int slot = g % kBwScaleSlots;
                if (!mbar_wait_bounded(&bws->sc_full[slot], (g / kBwScaleSlots) & 1, abort, p.st, 5) ||
                    !mbar_wait_bounded(&bar->acc_full[g & 1], (g >> 1) & 1, abort, p.st, 4)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tb = tmem + lane_base + (uint32_t)((g & 1) * kBwBN + kBwCols * h);
                const float sa = bws->sa[slot][rl];
                const float cs = sa * bws->sb[slot][h >> 1];
                const float* sbc = &bws->sb[slot][kBwCols * h];
#pragma unroll
                for (int cc = 0; cc < kBwCols / 16; ++cc) {
                    uint32_t r[16];
                    tmem_ld_32x32b_x16(tb + 16 * cc, r);
                    tmem_ld_wait();
                    reg_fence16(r);
                    if (!p.sb_per_row)
                        promote16x2(acc + 16 * cc, r, cs);
                    else
                        promote16x2_cols(acc + 16 * cc, r, sbc + 16 * cc, sa);
                }
                // this warp's share of the TMEM set is read: grant it to K
                // block g + 2, and hand the scale slot back to the loader
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (g + 2 < total) mbar_arrive_cluster(full_leader + 8u * (uint32_t)((g + 2) % kBwStages));
                    mbar_arrive(&bws->sc_empty[slot]);
                }
            }
            if (!ok) break;

            // tile done: store D (and the fused 1x128 quantization)
            const int m = ctm * 2 * BM + row0 + rl;
            const int ncol0 = ctn * kBwBN + kBwCols * h;
            const bool valid = m < p.M && ncol0 < p.N;  // N % 128 == 0: a warp's columns are all in or all out
            if (p.d_f32) {
                if (valid) {
                    float* drow = reinterpret_cast<float*>(p.D) + (size_t)m * p.ldd + ncol0;
                    if (p.d_v8) {
#pragma unroll
                        for (int i = 0; i < kBwCols / 8; ++i) {
                            uint32_t w[8];
#pragma unroll
                            for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(acc[8 * i + k]);
                            st_v8(drow + 8 * i, w);
                        }
                    } else {
                        float4* d = reinterpret_cast<float4*>(drow);
#pragma unroll
                        for (int i = 0; i < kBwCols / 4; ++i)
                            d[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
                    }
                }
            } else {
                uint32_t packed[kBwCols / 2];
#pragma unroll
                for (int i = 0; i < kBwCols / 2; ++i) packed[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
                if (valid) {
                    uint16_t* drow = reinterpret_cast<uint16_t*>(p.D) + (size_t)m * p.ldd + ncol0;
                    if (p.d_v8) {
#pragma unroll
                        for (int i = 0; i < kBwCols / 16; ++i) st_v8(drow + 16 * i, packed + 8 * i);
                    } else {
                        uint4* d = reinterpret_cast<uint4*>(drow);
#pragma unroll
                        for (int i = 0; i < kBwCols / 8; ++i)
                            d[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                    }
                }
                if (p.q_codes != nullptr) {
                    // a 1x128 group of a row spans warps h and h ^ 1 of this
                    // lane quarter: exchange their maxima through shared memory
                    float a = 0.0f;
#pragma unroll
                    for (int i = 0; i < kBwCols / 2; ++i)
                        a = fmaxf(a, fmaxf(fabsf(bf16_lo(packed[i])), fabsf(bf16_hi(packed[i]))));
                    bws->amax_xch[h][rl] = a;
                    const int bar_id = 1 + 2 * q + (h >> 1);
                    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(64) : "memory");
                    a = fmaxf(a, bws->amax_xch[h ^ 1][rl]);
                    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(64) : "memory");
                    const float sc = group_scale_bf16(a);  // D was rounded to bf16
                    const Divider dv = make_divider(sc);
                    if (valid) {
                        uint8_t* codes = p.q_codes + (size_t)m * p.N + ncol0;
                        uint32_t cw[kBwCols / 4];
#pragma unroll
                        for (int i = 0; i < kBwCols / 8; ++i) {
                            float f[8], qv[8];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                f[2 * k] = bf16_lo(packed[4 * i + k]);
                                f[2 * k + 1] = bf16_hi(packed[4 * i + k]);
                            }
                            if (dv.fast) {
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    quotient2_fast(dv, f[2 * k], f[2 * k + 1], qv[2 * k], qv[2 * k + 1]);
                            } else {
#pragma unroll
                                for (int k = 0; k < 8; ++k) qv[k] = __fdiv_rn(f[k], dv.s);
                            }
                            cw[2 * i] = e4m3x2(qv[0], qv[1]) | (e4m3x2(qv[2], qv[3]) << 16);
                            cw[2 * i + 1] = e4m3x2(qv[4], qv[5]) | (e4m3x2(qv[6], qv[7]) << 16);
                        }
                        if (p.q_v8) {
#pragma unroll
                            for (int i = 0; i < kBwCols / 32; ++i) st_v8(codes + 32 * i, cw + 8 * i);
                        } else {
#pragma unroll
                            for (int i = 0; i < kBwCols / 16; ++i)
                                reinterpret_cast<uint4*>(codes)[i] =
                                    make_uint4(cw[4 * i], cw[4 * i + 1], cw[4 * i + 2], cw[4 * i + 3]);
                        }
                        if ((h & 1) == 0) p.q_scales[(size_t)(ncol0 / 128) * p.M + m] = sc;
                    }
                }
            }
        }
    }

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
    CUtensorMap tmA, tmB;
    if (!make_map(&tmA, a.a_codes, (uint64_t)a.K, (uint64_t)a.M, BM) ||
        !make_map(&tmB, a.b_codes, (uint64_t)a.K, (uint64_t)a.N, 64))
        return cudaErrorInvalidValue;
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
    const int tiles = p.tiles_m * p.tiles_n;
    cudaError_t e = cudaFuncSetAttribute(k_gemm_blockwise, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBlockwise);
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
        e = cudaOccupancyMaxActiveClusters(&mp, k_gemm_blockwise, &cfg);
        if (e != cudaSuccess) return e;
        if (mp <= 0) return cudaErrorInvalidConfiguration;
    }
    const int pairs = tiles < mp ? tiles : mp;
    cfg.gridDim = dim3(2 * (unsigned)pairs);
    return cudaLaunchKernelEx(&cfg, k_gemm_blockwise, tmA, tmB, p);
}

}  // namespace fp8bs
