// q4moe_sm100.cuh -- thin inline-PTX wrappers for the Blackwell features the
// kernels use: mbarriers, cp.async, proxy fences and the tcgen05 tensor core
// (TMEM allocation, MMA, commit, loads).  Written from the PTX ISA; sm_100a
// family only.
#pragma once

#include <cstdint>

#include "q4moe.h"

namespace q4moe {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Ask L2 to fetch [p, p + bytes) (16-byte aligned, a multiple of 16 bytes).
// A prefetch only warms L2, the point of coherence, so it never makes data
// stale: it may be issued before a dependency wait.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p),
                 "r"(bytes)
                 : "memory");
}

// Ask L2 for the 128-byte line holding p (an ordinary per-thread prefetch,
// through the load path rather than the TMA unit).
__device__ __forceinline__ void prefetch_l2_line(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Arrive and add `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::
            "r"(smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

// Limit of every on-chip wait of the library's kernels.
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // 4 s

// Bounded wait on an mbarrier phase.  Returns false (and, the first time,
// raises Q4MOE_DEV_WAIT_TIMEOUT) once the CTA has aborted or the wait ran
// out (limit_ns).
static __device__ __noinline__ bool wait_phase(uint64_t *bar, uint32_t parity,
                                               volatile int *abort,
                                               unsigned int *status,
                                               uint64_t limit_ns =
                                                   kWaitLimitNs) {
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (*abort)
                return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                if (atomicExch((int *)abort, 1) == 0)
                    atomicOr(status, Q4MOE_DEV_WAIT_TIMEOUT);
                return false;
            }
        }
    }
}

// Non-blocking test of an mbarrier phase (no suspend: cheaper than
// try_wait when the phase is usually complete already).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait by spinning on test_wait, for the one thread whose issue
// rate sets the pace (the MMA issuer): returns false (and, the first time,
// raises Q4MOE_DEV_WAIT_TIMEOUT) once the CTA has aborted or the wait ran
// out (limit_ns).
__device__ __forceinline__ bool wait_spin(uint64_t *bar, uint32_t parity,
                                          volatile int *abort,
                                          unsigned int *status,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_test_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test_wait(bar, parity))
            return true;
        if ((it & 255u) == 0) {
            if (*abort)
                return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                if (atomicExch((int *)abort, 1) == 0)
                    atomicOr(status, Q4MOE_DEV_WAIT_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag, used while draining copies
// before exit (they land within microseconds; 0.2 s is ample).
__device__ __forceinline__ void drain_phase(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity) &&
           globaltimer_ns() - t0 < 200000000ull) {
    }
}

// ---------------------------------------------------------------- cp.async --
// 16-byte global -> shared copy; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src,
                                            uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// The same copy with an L2 cache policy (l2_policy_evict_last).
__device__ __forceinline__ void cp_async_16_hint(uint32_t dst, const void *src,
                                                 uint32_t src_bytes,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(
            dst),
        "l"(src), "r"(src_bytes), "l"(policy)
        : "memory");
}

// L2 policy for data that many CTAs re-read (the activations): keep it
// resident while the weights stream through.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;"
                 : "=l"(p));
    return p;
}

// Arrive on *bar (counted as one of its expected arrivals) once every
// cp.async this thread issued so far has landed in shared memory.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor core reads its operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------------------- TMA --
// Tiled 2-D tensor load of one box into shared memory; completion is
// reported to *bar as transaction bytes.  c0 is the inner (contiguous)
// coordinate in elements, c1 the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap,
                                            int32_t c0, int32_t c1,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
        "complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1),
        "r"(smem_u32(bar))
        : "memory");
}

// Tiled 3-D tensor load (c0 inner, c1 row, c2 outer).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap,
                                            int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::"
        "complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2),
        "r"(smem_u32(bar))
        : "memory");
}

// Fetch a tensor map (a __grid_constant__ kernel parameter) into the
// descriptor cache ahead of its first use.
__device__ __forceinline__ void tma_desc_prefetch(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap))
                 : "memory");
}

// Prefetch one box of a tiled 2-D tensor into L2 (no shared memory write,
// no completion to track).
__device__ __forceinline__ void tma_prefetch_2d(const void *tmap, int32_t c0,
                                                int32_t c1) {
    asm volatile(
        "cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(c0), "r"(c1)
        : "memory");
}

// ----------------------------------------------------------------- tcgen05 --
// TMEM allocation (whole warp): the base address is written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::
            "r"(smem_u32(dst)),
        "r"(ncols)
        : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                     taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] x B[smem desc]^T, bf16 in, f32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc,
                                          uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on *bar when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
        "[%0];" ::"r"(smem_u32(bar))
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit TMEM columns: thread t of the warp gets
// lane (taddr.lane + t), columns taddr.col .. +15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
          "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
          "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// The same for 8 consecutive columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
          "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr)
        : "memory");
}

// Wait for this thread's TMEM loads, naming the two 8-column destination
// arrays as operands so that no read of them is moved above the wait.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&a)[8],
                                                  uint32_t (&b)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]),
                   "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(b[0]), "+r"(b[1]),
                   "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
                   "+r"(b[7])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes (64 bf16 along K), 8-row groups of
// 1024 bytes (stride-dimension offset), 1024-byte aligned groups.  Fields:
// start address >> 4 in bits 0-13, leading-dimension offset >> 4 in 16-29
// (unused for this swizzled K-major form), stride offset >> 4 in 32-45,
// descriptor version 1 in bits 46-47, swizzle mode 2 (128 B) in bits 61-63.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major), f32
// accumulator, M = 128 and the given N (multiple of 16, 16..256): D format in
// bits 4-5, A/B formats in 7-9 / 10-12, N >> 3 in 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_m128(uint32_t n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) |
           ((128u >> 4) << 24);
}

}  // namespace sm100
}  // namespace q4moe
