// gemm_mx.cu -- MXFP8 GEMM (hardware block scaling), plain or grouped, on
// CTA pairs.
//
// MXFP8 recipe ("Anyscale、SkyRL で FP8 ...", "Deep dive: FP8 quantization
// with FP32 and power-of-two block scales": Blackwell tensor cores apply
// power-of-two block scales themselves): kind::mxf8f6f4.block_scale with the
// E8M0 scale atoms copied shared -> TMEM by tcgen05.cp; the accumulator stays
// in TMEM for the whole K loop.  Tile 256x256 per CTA pair, 6-stage ring, 8
// epilogue warps per CTA.  The grouped (MoE) variant walks a tile list over
// (expert, 256-row cluster tile, 256-col tile).
#include "gemm_common.cuh"

namespace fp8bs {

namespace {

// MX kernel
// CTA pairs compute 256x256 tiles (tcgen05.mma.cta_group::2, M=256, N=256):
// each CTA stages its 128 rows of A, its 128 of the tile's 256 rows of B, the
// scale atom of its A rows and both scale atoms of the tile's B rows.
constexpr int kMxBN = 256;
constexpr int kMxEpiWarps = 8;                        // warps 2..9
constexpr int kMxSfWarp = kEpiWarp0 + kMxEpiWarps;    // copies the scale factors into TMEM
constexpr int kMxThreads = (kMxSfWarp + 1) * 32;      // 352
constexpr int kMxStages = 6;
constexpr uint32_t kMxStageBytes = (BM + kMxBN / 2) * BK;  // 32 KB
constexpr uint32_t kSfStageBytes = 1536;                    // SFA atom + two SFB atoms
constexpr uint32_t kMxTmemCols = 512;                       // accumulator 256 + scale factors

constexpr size_t kSmemMx = 1024 + (size_t)kMxStages * (kMxStageBytes + kSfStageBytes) + sizeof(Barriers) +
                           3 * (kMaxGroups + 1) * sizeof(int);
static_assert(kSmemMx <= 232448, "MX shared memory over the 227 KB limit");

// the four E8M0 bytes packed little-endian.
__device__ __forceinline__ uint32_t quant_row_mx(const uint32_t (&packed)[64], uint8_t* codes) {
    uint32_t sc = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            a = fmaxf(a, fmaxf(fabsf(bf16_lo(packed[16 * b + j])), fabsf(bf16_hi(packed[16 * b + j]))));
        const int e = mx_exponent(a);
        const float mul = exp2_int(-e);
        sc |= (uint32_t)(e + 127) << (8 * b);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t p0 = packed[16 * b + 8 * i + 2 * k], p1 = packed[16 * b + 8 * i + 2 * k + 1];
                w[k] = e4m3x2(__fmul_rn(bf16_lo(p0), mul), __fmul_rn(bf16_hi(p0), mul)) |
                       (e4m3x2(__fmul_rn(bf16_lo(p1), mul), __fmul_rn(bf16_hi(p1), mul)) << 16);
            }
            reinterpret_cast<uint4*>(codes + 32 * b)[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    return sc;
}

// The same 128 values as one 1x128 group with a power-of-two scale (the
// blockwise recipe's Blackwell variant): one exponent, repeated in the four
// returned E8M0 bytes.
__device__ __forceinline__ uint32_t quant_row_pow2(const uint32_t (&packed)[64], uint8_t* codes) {
    float a = 0.0f;
#pragma unroll
    for (int j = 0; j < 64; ++j) a = fmaxf(a, fmaxf(fabsf(bf16_lo(packed[j])), fabsf(bf16_hi(packed[j]))));
    const int e = pow2_exponent(a);
    const float mul = exp2_int(-e);
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t p0 = packed[8 * b + 2 * k], p1 = packed[8 * b + 2 * k + 1];
            w[k] = e4m3x2(__fmul_rn(bf16_lo(p0), mul), __fmul_rn(bf16_hi(p0), mul)) |
                   (e4m3x2(__fmul_rn(bf16_lo(p1), mul), __fmul_rn(bf16_hi(p1), mul)) << 16);
        }
        reinterpret_cast<uint4*>(codes)[b] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return (uint32_t)(e + 127) * 0x01010101u;
}

// ===========================================================================
// MXFP8 GEMM (hardware block scaling), plain or grouped
// ===========================================================================
struct MxParams {
    const uint8_t* sfa;
    const uint8_t* sfb;
    const int32_t* m_offsets;  // nullptr: one group of M rows
    int G;
    int M, N, K;
    uint16_t* D;
    long long ldd;
    uint8_t* q_codes;
    uint8_t* q_scales;
    StatusBlock* st;
    int tiles_n;
    int d_v8;    // D rows allow 32-byte stores
    int q_pow2;  // fused quantization: 1x128 groups, power-of-two scales
};

struct TileCoord {
    int g;          // group
    int mt;         // this CTA's 128-row tile within the group
    int atom_row;   // its row of scale atoms (clamped into the group)
    int row0, rows;  // first row of the tile; valid rows of the group in it (0..128)
    int tn;
};

// Cluster tile -> (group, 256-row cluster tile, 256-column tile); then this
// CTA's half.  Cluster tiles are numbered down bands of 16 cluster-tile rows
// (the last band may be shorter), rows first within a band, so that the pairs
// running at one time share a band of A and a few column tiles of B in L2;
// the group comes from a binary search over the prefix of cluster tiles per
// group.
__device__ __forceinline__ TileCoord mx_tile(int tile, int tiles_m, int tiles_n, const int* pfx, const int* pfx2, const int* offs,
                                            int G, uint32_t rank) {
    TileCoord c;
    constexpr int kBand = 16;
    const int band = tile / (kBand * tiles_n);
    const int first = band * kBand;
    const int rows = tiles_m - first < kBand ? tiles_m - first : kBand;
    const int idx = tile - band * kBand * tiles_n;
    const int mt2_global = first + idx % rows;
    c.tn = idx / rows;
    int lo = 0, hi = G;  // largest g with pfx2[g] <= mt2_global
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pfx2[mid] <= mt2_global) lo = mid; else hi = mid;
    }
    c.g = lo;
    c.mt = 2 * (mt2_global - pfx2[lo]) + (int)rank;
    const int ntiles = pfx[lo + 1] - pfx[lo];  // 128-row tiles of the group (>= 1 here)
    c.atom_row = pfx[lo] + (c.mt < ntiles ? c.mt : ntiles - 1);
    c.row0 = offs[lo] + c.mt * BM;
    const int left = offs[lo + 1] - c.row0;
    c.rows = left < 0 ? 0 : (left < BM ? left : BM);
    return c;
}

__global__ void __launch_bounds__(kMxThreads, 1)
    k_gemm_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB, const MxParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = aligned_smem(smem_raw);
    uint8_t* sf = smem + kMxStages * kMxStageBytes;
    Barriers* bar = reinterpret_cast<Barriers*>(sf + kMxStages * kSfStageBytes);
    int* offs = reinterpret_cast<int*>(bar + 1);  // [G+1] row offsets
    int* pfx = offs + (kMaxGroups + 1);           // [G+1] prefix of 128-row tiles (= scale atom rows)
    int* pfx2 = pfx + (kMaxGroups + 1);           // [G+1] prefix of 256-row cluster tiles
    volatile int* abort = &bar->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;
    const uint32_t rank = cluster_ctarank();  // 0: leader CTA (issues the MMAs)
    const int cid = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        // full[s], acc_empty (leader only): the leader producer's expect_tx
        // arrival for both CTAs' bytes; one arrival per epilogue warp of both CTAs
        for (int s = 0; s < kMxStages; ++s) {
            mbar_init(&bar->full[s], 1);
            mbar_init(&bar->empty[s], 1);
        }
        mbar_init(&bar->acc_full[0], 1);
        mbar_init(&bar->acc_empty[0], 2 * (kEpiThreads / 32));
        for (int st = 0; st < kMxStages; ++st) mbar_init(&bar->sf_ready[st], 1);
        mbar_init(&bar->drain, 1);
        bar->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmSFA);
        prefetch_tensormap(&tmSFB);
    }
    if (warp == 1) tmem_alloc_pair(&bar->tmem_base, kMxTmemCols);
    if (warp == 2) {
        // group row offsets and the prefix sums of their 128- and 256-row tile
        // counts.  Offsets outside [0, M] or decreasing are reported
        // (FP8_ERR_INVALID_ARG at the next status poll) and clamped to [0, M],
        // so every row the kernel touches stays inside A and D.
        int carry = 0, carry2 = 0;
        bool bad = false;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int o0 = 0, o1 = 0;
            if (g < G) {
                o0 = p.m_offsets ? p.m_offsets[g] : 0;
                o1 = p.m_offsets ? p.m_offsets[g + 1] : p.M;
                bad |= o0 < 0 || o1 < o0 || o1 > p.M || (g == 0 && o0 != 0);
                o0 = o0 < 0 ? 0 : (o0 > p.M ? p.M : o0);
                o1 = o1 < o0 ? o0 : (o1 > p.M ? p.M : o1);
                offs[g] = o0;
            }
            int cnt = (g < G) ? (o1 - o0 + BM - 1) / BM : 0;
            if (cnt < 0) cnt = 0;
            const int cnt2 = (cnt + 1) / 2;
            int incl = cnt, incl2 = cnt2;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                const int v2 = __shfl_up_sync(0xffffffffu, incl2, o);
                if (lane >= o) {
                    incl += v;
                    incl2 += v2;
                }
            }
            if (g < G) {
                pfx[g] = carry + incl - cnt;
                pfx2[g] = carry2 + incl2 - cnt2;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
            carry2 += __shfl_sync(0xffffffffu, incl2, 31);
        }
        if (lane == 0) {
            pfx[G] = carry;
            pfx2[G] = carry2;
            const int oG = p.m_offsets ? p.m_offsets[G] : p.M;
            offs[G] = oG < 0 ? 0 : (oG > p.M ? p.M : oG);
            bar->num_mtiles = carry2;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0 && rank == 0) atomicOr(&p.st->error_bits, kErrDeviceArg);
    }
    tc_fence_before();
    cluster_sync();  // barriers, group tables and TMEM ready in both CTAs
    tc_fence_after();
    const uint32_t tmem = bar->tmem_base;
    const int KB = p.K / BK;
    const int num_tiles = bar->num_mtiles * p.tiles_n;
    const uint32_t sf_col0 = 256;  // TMEM columns [256, 256 + 16*kMxStages): scale factors
    const uint32_t full_leader = mapa_shared(&bar->full[0], 0);
    const uint32_t acc_empty_leader = mapa_shared(&bar->acc_empty[0], 0);

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            const int atoms_k = p.K / 128;
            const int b_atom_rows = (p.G * p.N + 127) / 128;
            for (int tile = cid; tile < num_tiles && ok; tile += ncl) {
                const TileCoord c = mx_tile(tile, bar->num_mtiles, p.tiles_n, pfx, pfx2, offs, G, rank);
                const int bcol0 = c.g * p.N + c.tn * kMxBN;        // first B row of the tile
                const int batom0 = bcol0 / 128;                      // its scale atom row
                const int batom1 = c.tn * kMxBN + 128 < p.N && batom0 + 1 < b_atom_rows ? batom0 + 1 : batom0;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait_bounded(&bar->empty[s], ph ^ 1, abort, p.st, 11)) {
                        ok = false;
                        break;
                    }
                    uint8_t* stage = smem + s * kMxStageBytes;
                    uint8_t* sfs = sf + s * kSfStageBytes;
                    if (rank == 0) mbar_arrive_expect_tx(&bar->full[s], 2 * (kMxStageBytes + kSfStageBytes));
                    const uint32_t fb = full_leader + 8u * (uint32_t)s;
                    tma_load_2d_pair(stage, &tmA, fb, kb * BK, c.row0);
                    tma_load_2d_pair(stage + BM * BK, &tmB, fb, kb * BK, bcol0 + 128 * (int)rank);
                    // scale atoms as 2 x 256-byte rows of the [atoms * 2][256] byte views
                    tma_load_2d_pair(sfs, &tmSFA, fb, 0, 2 * (c.atom_row * atoms_k + kb));
                    tma_load_2d_pair(sfs + 512, &tmSFB, fb, 0, 2 * (batom0 * atoms_k + kb));
                    tma_load_2d_pair(sfs + 1024, &tmSFB, fb, 0, 2 * (batom1 * atoms_k + kb));
                    if (++s == kMxStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            int s = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int tile = cid; tile < num_tiles && ok; tile += ncl) {
                if (!mbar_wait_bounded(&bar->acc_empty[0], aph ^ 1, abort, p.st, 12)) break;
                for (int kb = 0; kb < KB; ++kb) {
                    // the stage's operands landed and its scale factors are in
                    // TMEM (copied by the scale-factor warp)
                    if (!mbar_wait_bounded(&bar->full[s], ph, abort, p.st, 13) ||
                        !mbar_wait_bounded(&bar->sf_ready[s], ph, abort, p.st, 15)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * kMxStageBytes);
                    const uint32_t tsfa = tmem + sf_col0 + 16u * s;
                    const uint32_t tsfb = tsfa + 4;
                    const uint64_t adesc = sdesc_k_sw128(a_addr);
                    const uint64_t bdesc = sdesc_k_sw128(a_addr + BM * BK);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        tc_mma_mxf8f6f4_pair(tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8f6f4(2 * BM, kMxBN, k, k),
                                             tsfa, tsfb, (kb > 0 || k > 0) ? 1u : 0u);
                    tc_commit_pair(&bar->empty[s], 3);
                    if (++s == kMxStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit_pair(&bar->acc_full[0], 3);
                aph ^= 1;
            }
            tc_commit_pair(&bar->drain, 1);
            mbar_wait_drain(&bar->drain, 0, p.st);
        }
    } else if (warp == kMxSfWarp) {
        // scale factors: per stage, each CTA's A atom and the tile's two B
        // atoms copied shared -> TMEM (tcgen05.cp, issued by the leader for
        // both CTAs), then sf_ready[s].  A thread issues a tcgen05 instruction
        // every ~60 cycles, so these three copies on the MMA thread would
        // stretch every K block; here they run one or more stages ahead.
        // Stage s's TMEM slot was last read by the MMAs of the K block six
        // earlier, which completed before the producer refilled stage s.
        if (lane == 0 && rank == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int tile = cid; tile < num_tiles && ok; tile += ncl) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait_bounded(&bar->full[s], ph, abort, p.st, 16)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_addr = smem_u32(sf + s * kSfStageBytes);
                    const uint32_t tsfa = tmem + sf_col0 + 16u * s;
                    const uint32_t tsfb = tsfa + 4;
                    // each CTA copies its own shared-memory scales into its own TMEM
                    tc_cp_pair_32x128b_warpx4(tsfa, sdesc_sf_32x16(sf_addr));
                    tc_cp_pair_32x128b_warpx4(tsfb, sdesc_sf_32x16(sf_addr + 512));
                    tc_cp_pair_32x128b_warpx4(tsfb + 4, sdesc_sf_32x16(sf_addr + 1024));
                    tc_commit_pair(&bar->sf_ready[s], 1);
                    if (++s == kMxStages) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
        }
    } else if (warp >= kEpiWarp0) {
        const int q = warp & 3, h = (warp - kEpiWarp0) >> 2;
        const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(128 * h);
        const int64_t q_atoms_k = (p.N + 127) / 128;
        uint32_t aph = 0;
        for (int tile = cid; tile < num_tiles; tile += ncl) {
            const TileCoord c = mx_tile(tile, bar->num_mtiles, p.tiles_n, pfx, pfx2, offs, G, rank);
            const int rl = 32 * q + lane;
            const int ncol0 = c.tn * kMxBN + 128 * h;
            const bool mvalid = rl < c.rows, hvalid = ncol0 < p.N;
            if (!mbar_wait_bounded(&bar->acc_full[0], aph, abort, p.st, 14)) break;
            tc_fence_after();
            // two halves of 64 columns: load, wait, round to bf16
            uint32_t packed[64];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r0[32], r1[32];
                ld_chunk(tb + 64 * half, r0);
                ld_chunk(tb + 64 * half + 32, r1);
                tmem_ld_wait();
                reg_fence32(r0);
                reg_fence32(r1);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    packed[32 * half + j] = pack_bf16x2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
                    packed[32 * half + 16 + j] =
                        pack_bf16x2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
                }
            }
            // the accumulator is read: hand it back to the leader's MMA thread
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
            aph ^= 1;
            const int64_t m = (int64_t)c.row0 + rl;
            if (mvalid && hvalid) {
                uint16_t* d = p.D + m * p.ldd + ncol0;
                if (p.d_v8) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (ncol0 + 16 * i < p.N) st_v8(d + 16 * i, packed + 8 * i);  // N % 16 == 0
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (ncol0 + 8 * i < p.N)
                            reinterpret_cast<uint4*>(d)[i] =
                                make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
                }
                if (p.q_codes != nullptr) {
                    const uint32_t sc = p.q_pow2 ? quant_row_pow2(packed, p.q_codes + m * p.N + ncol0)
                                                 : quant_row_mx(packed, p.q_codes + m * p.N + ncol0);
                    *reinterpret_cast<uint32_t*>(p.q_scales + mx_scale_offset(m, ncol0 / 32, q_atoms_k)) = sc;
                }
            } else if (p.q_codes != nullptr && hvalid && m < ((int64_t)p.M + 127) / 128 * 128) {
                // padding rows of the last scale atom row: zero, as the standalone quantizer writes
                *reinterpret_cast<uint32_t*>(p.q_scales + mx_scale_offset(m, ncol0 / 32, q_atoms_k)) = 0u;
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
        tmem_dealloc_pair(tmem, kMxTmemCols);
    }
}

}  // namespace

cudaError_t launch_gemm_mx(const GemmMxArgs& a, StatusBlock* status, cudaStream_t st) {
    if (a.M == 0 || a.N == 0) return cudaSuccess;
    // scale buffers: per-group padded atom rows (grouped) or ceil(M/128) atom rows
    const int64_t atoms_k = a.K / 128;
    const int64_t a_atom_rows = a.m_offsets ? (a.M + BM - 1) / BM + a.G : (a.M + BM - 1) / BM;
    const int64_t b_atom_rows = (a.N * a.G + 127) / 128;
    CUtensorMap tmA, tmB, tmSFA, tmSFB;
    if (!make_map(&tmA, a.a_codes, (uint64_t)a.K, (uint64_t)a.M, BM) ||
        !make_map(&tmB, a.b_codes, (uint64_t)a.K, (uint64_t)a.N * (uint64_t)a.G, kMxBN / 2) ||
        !make_map_plain_u8(&tmSFA, a.sfa, 256, (uint64_t)(2 * a_atom_rows * atoms_k), 2) ||
        !make_map_plain_u8(&tmSFB, a.sfb, 256, (uint64_t)(2 * b_atom_rows * atoms_k), 2))
        return cudaErrorInvalidValue;
    MxParams p;
    p.sfa = a.sfa;
    p.sfb = a.sfb;
    p.m_offsets = a.m_offsets;
    p.G = a.G;
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.D = reinterpret_cast<uint16_t*>(a.D);
    p.ldd = a.ldd;
    p.q_codes = a.q_codes;
    p.q_scales = a.q_scales;
    p.q_pow2 = a.q_pow2 ? 1 : 0;
    p.st = status;
    p.tiles_n = (int)((a.N + kMxBN - 1) / kMxBN);
    p.d_v8 = (reinterpret_cast<uintptr_t>(a.D) % 32 == 0) && ((a.ldd * 2) % 32 == 0);
    // upper bound of the cluster-tile count (the exact count depends on device-side offsets)
    const int64_t mtiles = a.m_offsets ? (a.M + 2 * BM - 1) / (2 * BM) + a.G : (a.M + 2 * BM - 1) / (2 * BM);
    const int64_t tiles = mtiles * p.tiles_n;
    cudaError_t e = cudaFuncSetAttribute(k_gemm_mx, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMx);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)tiles);
    cfg.blockDim = dim3(kMxThreads);
    cfg.dynamicSmemBytes = kSmemMx;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static int max_pairs[64] = {0};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int& mp = max_pairs[dev & 63];
    if (mp <= 0) {
        e = cudaOccupancyMaxActiveClusters(&mp, k_gemm_mx, &cfg);
        if (e != cudaSuccess) return e;
        if (mp <= 0) return cudaErrorInvalidConfiguration;
    }
    const int64_t pairs = tiles < mp ? tiles : mp;
    cfg.gridDim = dim3(2 * (unsigned)pairs);
    return cudaLaunchKernelEx(&cfg, k_gemm_mx, tmA, tmB, tmSFA, tmSFB, p);
}

}  // namespace fp8bs
