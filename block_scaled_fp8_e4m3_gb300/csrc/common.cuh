// common.cuh -- shared device helpers of the fp8bs library (sm_103a only).
//
// Holds: the per-device status block that device code reports into, the
// bounded waits every spin loop goes through, bf16/E4M3 conversions, and
// thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk[.tensor]) and
// the tcgen05 tensor-core instructions (TMEM alloc, mma, commit, cp, ld).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8bs.h"

namespace fp8bs {

// ---------------------------------------------------------------- status
enum : unsigned int {
    kErrTimeout = 1u,
    kErrChecksum = 2u,
    kErrDeviceArg = 4u,
    kErrBadPayload = 8u,
};

// One per device, allocated on first use; cleared by fp8_status_poll().
struct StatusBlock {
    unsigned int error_bits;     // kErr* bits
    unsigned int timeout_site;   // which bounded wait gave up (diagnostics)
    unsigned long long sum;      // checksum accumulator of fp8_sync_install
    unsigned int blocks_done;    // blocks of the verify kernel that finished
    unsigned int verdict;        // 0: payload verified, 1: mismatch
    unsigned int header_bad;     // set by fp8_sync_install's device-side header/table check
    unsigned int barrier_gen;    // generation of the install kernel's grid barrier
    unsigned long long reserved[3];
};

// A bounded wait gives up after this long.  Legitimate waits inside one
// kernel last microseconds; a second means the peer is gone.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void report_timeout(StatusBlock* st, int site) {
    atomicOr(&st->error_bits, kErrTimeout);
    atomicExch(&st->timeout_site, (unsigned int)site);
}

// ---------------------------------------------------------------- scalars
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> two E4M3 codes (round to nearest even, saturating to +-448);
// low byte from a, high byte from b.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Blockwise scale s = amax / 448 (IEEE fp32 quotient); 1 for an all-zero
// group and whenever the quotient underflows to 0 (amax below 448 * 2^-150,
// possible only for fp32 inputs), so no block divides by zero.
__device__ __forceinline__ float group_scale(float amax) {
    const float s = __fdiv_rn(amax, 448.0f);
    return s == 0.0f ? 1.0f : s;
}

// The same scale for a group maximum that is a bf16 value: Markstein's FMA
// correction of amax * RN(1/448) (see quotient() below); a host check over
// every positive finite bf16 value gives the IEEE quotient bit for bit.  The
// maximum (a fmaxf reduction from 0) is never NaN; an infinite one gives
// inf / 448 = inf.
__device__ __forceinline__ float group_scale_bf16(float amax) {
    constexpr float kInv448 = 1.0f / 448.0f;
    const float q0 = __fmul_rn(amax, kInv448);
    const float e = __fmaf_rn(-448.0f, q0, amax);
    const float s = __fmaf_rn(e, kInv448, q0);
    return amax == 0.0f ? 1.0f : (amax <= 3.402823466e38f ? s : amax);
}

// x / s for the quotients of the blockwise quantizers: x a bf16 value and
// s = RN(amax / 448) of the group maximum amax >= |x|.  For s >= 2^-100 it
// takes Markstein's FMA correction of the product with the correctly rounded
// reciprocal (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(x r),
// e = x - s q0 (exact by FMA), q = RN(q0 + e r).  An exhaustive host check
// over every bf16 x and every bf16 group maximum gives the E4M3 code of the
// IEEE quotient in every case (the quotient bits differ only below 2^-11,
// where the code is zero either way); smaller or non-finite s take the IEEE
// division.
struct Divider {
    float s, nr;  // nr = -RN(1/s)
    bool fast;
};

__device__ __forceinline__ Divider make_divider(float s) {
    Divider d;
    d.s = s;
    d.nr = -__frcp_rn(s);
    d.fast = s >= 0x1p-100f && s <= 3.402823466e38f;
    return d;
}

// The codes of x0..x3 / s as above (four E4M3 bytes, x0 in the lowest);
// d.fast must hold.  The correction runs on the negated quotient, two values
// per packed instruction: n = RN(x nr), e = x + n s (exact), -q = RN(n + e nr).
// A zero x then ends as a zero of the opposite sign (RN(+0 + -0) = +0 and
// RN(-0 + -0) = -0), so flipping the sign bits of the four codes gives the
// codes of q with the sign of x, -0 included, and no copysign per value.
__device__ __forceinline__ uint32_t codes4_div_fast(const Divider& d, float x0, float x1, float x2, float x3) {
    uint64_t a, b, na, nb;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(x0), "f"(x1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(x2), "f"(x3));
    asm("{\n\t.reg .b64 r2, s2, e;\n\t"
        "mov.b64 r2, {%4, %4};\n\tmov.b64 s2, {%5, %5};\n\t"
        "mul.rn.f32x2 %0, %2, r2;\n\t"
        "mul.rn.f32x2 %1, %3, r2;\n\t"
        "fma.rn.f32x2 e, %0, s2, %2;\n\t"
        "fma.rn.f32x2 %0, e, r2, %0;\n\t"
        "fma.rn.f32x2 e, %1, s2, %3;\n\t"
        "fma.rn.f32x2 %1, e, r2, %1;\n\t}\n"
        : "=&l"(na), "=&l"(nb)
        : "l"(a), "l"(b), "f"(d.nr), "f"(d.s));
    float n0, n1, n2, n3;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(n0), "=f"(n1) : "l"(na));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(n2), "=f"(n3) : "l"(nb));
    return (e4m3x2(n0, n1) | (e4m3x2(n2, n3) << 16)) ^ 0x80808080u;
}

// MX shared exponent e = clamp(floor(log2 amax) - 8, -127, 127) from the fp32
// bit fields (no log2 evaluation); -127 for an all-zero block.
__device__ __forceinline__ int mx_exponent(float amax) {
    if (amax == 0.0f) return -127;
    uint32_t u = __float_as_uint(amax);
    int bexp = (int)(u >> 23);
    int E = bexp != 0 ? bexp - 127 : (31 - __clz(u & 0x7FFFFFu)) - 149;
    int e = E - 8;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^k as fp32 for k in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2_int(int k) {
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

// Exponent of the blockwise recipe's power-of-two scale: e = ceil(log2(t)),
// t = RN(amax/448) the fp32 recipe's scale, i.e. the smallest power of two
// not below t; clamped to the E8M0 range [-127, 127].  pow2_exponent takes
// the group maximum amax (a bf16 value or +inf) and gives 0 (s = 1) for an
// all-zero group.
__device__ __forceinline__ int pow2_exponent_of_scale(float t) {
    const uint32_t u = __float_as_uint(t);
    const int bexp = (int)(u >> 23);
    const uint32_t m = u & 0x7FFFFFu;
    int e;
    if (bexp == 0xFF)
        e = 127;
    else if (bexp != 0)
        e = bexp - 127 + (m != 0u ? 1 : 0);
    else
        e = (31 - __clz(m)) - 149 + ((m & (m - 1u)) != 0u ? 1 : 0);  // t = 0 gives -150
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

__device__ __forceinline__ int pow2_exponent(float amax) {
    return amax == 0.0f ? 0 : pow2_exponent_of_scale(group_scale_bf16(amax));
}

// Byte offset of the E8M0 scale of (row r, 32-column block j) in the
// 128x4 atom layout (atoms_k = ceil(cols/128) atoms per 128-row tile).
__device__ __forceinline__ int64_t mx_scale_offset(int64_t r, int64_t j, int64_t atoms_k) {
    return ((r >> 7) * atoms_k + (j >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (j & 3);
}

// ---------------------------------------------------------------- smem / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// (returns false) when *abort is raised by another warp, or after
// kWaitLimitNs, in which case it records the timeout and raises *abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  StatusBlock* st, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    unsigned long long t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                report_timeout(st, site);
                *abort = 1;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor: K-major operand tile whose rows are 128
// bytes, written by TMA with 128-byte swizzle (8-row atoms of 1024 bytes).
//   [0,14) start>>4  [16,30) LBO>>4 (unused for swizzled K-major)
//   [32,46) SBO>>4 = 1024>>4  [46,49) = 0b001  [61,64) swizzle: 2 = 128B
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Descriptor of a 32-row x 16-byte, unswizzled source for tcgen05.cp
// (core matrices of 8 rows x 16 bytes, stacked every 128 bytes).
__device__ __forceinline__ uint64_t sdesc_sf_32x16(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) |
           ((uint64_t)(128 >> 4) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor, kind::f8f6f4, E4M3 x E4M3 -> F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f8f6f4(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled, E4M3 x E4M3, UE8M0
// scale factors; sfa/sfb select the scale byte for this MMA's 32-wide K step.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(int M, int N, uint32_t sfa_id, uint32_t sfb_id) {
    return (sfb_id << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) |
           (sfa_id << 29);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- CTA pairs (cluster of two CTAs on neighbouring SMs) -----------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory object in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// arrive on an mbarrier given by its shared::cluster address (any CTA of the
// cluster).  Default (CTA-scope release) semantics: a cluster-scope release
// waits for this thread's outstanding memory traffic and costs over a
// thousand cycles; the arrivals here only hand back TMEM that the thread has
// finished reading (tcgen05.wait::ld + tcgen05.fence::before_thread_sync).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}

// all threads of both CTAs
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA 2-D load into this CTA's shared memory whose completion is counted on
// an mbarrier of the pair's leader CTA (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar_cluster_addr,
                                                 int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr)
        : "memory");
}

// TMEM allocation shared by the pair: one warp of each CTA executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (TMEM, both CTAs) (+)= A (each CTA's 128 rows) x B^T (N/2 rows per CTA);
// issued by one thread of the leader CTA.
__device__ __forceinline__ void tc_mma_f8f6f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                   uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// block-scaled MX MMA on a CTA pair; each CTA's tensor core applies the
// scale factors in its own TMEM (its A rows' scales, all N columns' B scales)
__device__ __forceinline__ void tc_mma_mxf8f6f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                     uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::
            "r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// shared -> TMEM copy on a CTA pair: each CTA copies from its own shared
// memory (same address) into its own TMEM
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// arrive on the barrier at the same offset in every CTA of cta_mask once the
// pair MMAs issued so far by this thread have completed
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::
            "r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Arrives once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Copies a 32-row x 128-bit block from shared memory into TMEM, replicated
// into all four 32-lane quarters (the scale-factor staging copy).
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (quarter_base + t), columns [col, col+32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace fp8bs
