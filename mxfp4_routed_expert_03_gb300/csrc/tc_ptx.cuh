// Inline-PTX wrappers for the Blackwell tensor-core path (sm_103a):
// mbarriers with bounded waits, TMA tile / gather4 loads, cp.async,
// tcgen05 TMEM allocation, block-scaled MMA, smem->TMEM copies and TMEM loads.
// Written from the public PTX ISA description of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that may suspend the thread for up to `ns` nanoseconds while the
// phase is incomplete (it resumes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for waits expected to be long: the waiting warp sleeps inside
// try_wait instead of spinning, so it takes no issue slots from warps that
// have work.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, long long limit_cycles,
                                                volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (true) {
        if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit_cycles) return false;
    }
}

// Bounded wait on phase `parity`: gives up after `limit_cycles` SM clocks
// (or as soon as *abort becomes non-zero) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit_cycles,
                                          volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit_cycles) return false;
    }
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier `id` over `nthreads` threads that also ANDs a predicate:
// returns true only if every participating thread passed ok = true. Used so
// that a group of warps takes one decision after its bounded waits (none is
// left waiting at a later barrier for a warp that gave up).
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// Four rows (r0..r3) of one 2D tensor, columns [c0, c0 + box), into
// consecutive rows of dst. The tensor map's box is one row high.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int r0, int r1, int r2, int r3,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Contiguous bulk copy global -> shared (16-byte aligned, size multiple of 16),
// completion counted on bar's transaction count.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}

// Arrive on bar once all prior cp.async of this thread have landed
// (does not add to the barrier's expected arrival count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T with per-32-K E8M0 scales from TMEM.
// kind::mxf8f6f4: A and B each E4M3 / E5M2 / E2M3 / E3M2 / E2M1 (set in idesc).
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], "
        "[%6], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, both operands E2M1 packed two per byte
// (kind::mxf4), 64 K per instruction, one E8M0 scale per 32 K from TMEM
// (scale_vec::2X: the two scale bytes of a row are the byte pair the sf ids
// in idesc select, 0 or 2).
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], "
        "[%6], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, bf16 operands (kind::f16), 16 K per
// instruction, fp32 accumulation.
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on bar when all prior tcgen05 async ops of this thread finish.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 rows x 128 bits from smem (descriptor) into TMEM at taddr, replicated to
// all four 32-lane quadrants.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// 128 rows x 256 bits from smem (descriptor) into TMEM: row i -> lane i,
// 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- wind-down
// After a timeout: wait until every MMA this thread issued has completed
// (one commit to `bar`, a barrier used for nothing else, then a bounded wait
// on its first phase), so that tensor memory can be released.
__device__ __forceinline__ void drain_mmas(uint64_t *bar, long long limit) {
    int never = 0;
    mma_commit(bar);
    mbar_wait(bar, 0, limit / 100 + 100000, &never);
}

// After a timeout: wait (bounded) until every fill a single producer issued
// into a ring of n_slots stages has landed. Fill i went to stage i % n_slots
// in round i / n_slots; with one arrival per phase the last round of each
// stage completes once its bytes are in.
__device__ __forceinline__ void wait_issued_fills(uint64_t *full, int n_slots, int issued,
                                                  long long limit) {
    int never = 0;
    for (int s = 0; s < n_slots; ++s) {
        const int rounds = issued > s ? (issued - s + n_slots - 1) / n_slots : 0;
        if (rounds > 0) mbar_wait(&full[s], (uint32_t)((rounds - 1) & 1), limit / 100 + 100000, &never);
    }
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128
// bytes, 8-row (1024-byte) swizzle atoms stacked along M/N.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);       // start address
    d |= (uint64_t)(16u >> 4) << 16;                 // leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                          // descriptor version (tcgen05)
    d |= (uint64_t)2 << 61;                          // 128-byte swizzle
    return d;
}

// Descriptor of a plain (unswizzled) 32-row x 16-byte block for tcgen05.cp:
// core matrices of 8 rows x 16 bytes, 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_plain_32x16(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Descriptor of 32 rows x 16 bytes for tcgen05.cp.32x128b whose 8-row core
// matrices lie 256 bytes apart (the first 16 bytes of each row of a 1 KB
// 128x256b-layout block). Both offset fields carry the 256-byte stride; the
// block has a single 16-byte core matrix along K.
__device__ __forceinline__ uint64_t sdesc_plain_32x16_groups256(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(256u >> 4) << 16;
    d |= (uint64_t)(256u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Descriptor of a plain (unswizzled) 128-row x 32-byte block for
// tcgen05.cp.128x256b: K-major core matrices of 8 rows x 16 bytes, the two
// 16-byte halves of a row 128 bytes apart, 8-row groups 256 bytes apart.
__device__ __forceinline__ uint64_t sdesc_plain_128x32(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;  // leading (K) byte offset
    d |= (uint64_t)(256u >> 4) << 32;  // stride (row-group) byte offset
    d |= (uint64_t)1 << 46;
    return d;
}

// MMA element formats of kind::mxf8f6f4.
enum { FMT_E4M3 = 0, FMT_E5M2 = 1, FMT_E2M3 = 3, FMT_E3M2 = 4, FMT_E2M1 = 5 };

// Instruction descriptor of kind::mxf8f6f4 block-scaled MMA, both operands
// K-major, E8M0 scales; sf ids pick the scale byte (the 32-wide K block within
// a 4-block scale group) for A and B.
__host__ __device__ __forceinline__ uint32_t idesc_mxf8f6f4(int a_fmt, int b_fmt, int M, int N,
                                                           int a_sf_id, int b_sf_id) {
    uint32_t d = 0;
    d |= (uint32_t)(b_sf_id & 3) << 4;
    d |= (uint32_t)(a_fmt & 7) << 7;
    d |= (uint32_t)(b_fmt & 7) << 10;
    d |= (uint32_t)((N >> 3) & 0x3F) << 17;
    d |= 1u << 23;                                   // scale type: UE8M0
    d |= (uint32_t)((M >> 4) & 0x1F) << 24;
    d |= (uint32_t)(a_sf_id & 3) << 29;
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulator (bit 4), bf16 A and B
// (bits 7-9 and 10-12 = 1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of kind::mxf4 block-scaled MMA: the same fields as
// idesc_mxf8f6f4, with E2M1 coded 1 for both operands in this kind.
__host__ __device__ __forceinline__ uint32_t idesc_mxf4(int M, int N, int a_sf_id, int b_sf_id) {
    constexpr int MXF4_E2M1 = 1;
    return idesc_mxf8f6f4(MXF4_E2M1, MXF4_E2M1, M, N, a_sf_id, b_sf_id);
}

}  // namespace tc
