// tcgen05 / TMEM building blocks shared by the tensor-core prefix kernels
// (sm_103a): shared-memory matrix descriptors, instruction descriptors, MMA
// issue and completion, tensor-memory loads and stores, and a few mbarrier
// and math helpers. All inline PTX.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "va_common.cuh"

namespace va {
namespace tc {

// Shared-memory matrix descriptor (sm_100 format: version 1 at bit 46, layout
// type at bits 61..63: 0 = no swizzle, 2 = 128-byte swizzle). Addresses,
// leading and stride byte offsets in units of 16 bytes; a later offset (>> 4)
// adds straight into the 14-bit address field.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)layout << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulate, A and B both bf16
// (bf16 = 1) or both fp16 (bf16 = 0), M x N, operand majors (0 = K, 1 = MN).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn, int bf16) {
    return (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) | ((uint32_t)a_mn << 15) |
           ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] x B[smem]
__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
// the same with the A operand in TMEM (rows = lanes, 16-bit pairs per 32-bit column)
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, int acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
// arrive on this CTA's barrier once the MMAs issued so far have completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(slot)),
                 "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(base), "r"(cols));
}

// 32 lanes x 32 consecutive 32-bit columns (warp-collective; lane quadrant = warp % 4)
#define VA_TC_LD32(taddr, r)                                                                         \
    asm volatile(                                                                                    \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14," \
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"             \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),       \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),   \
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),             \
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),             \
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])              \
        : "r"(taddr))
#define VA_TC_ST32(taddr, r)                                                                         \
    asm volatile(                                                                                    \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"  \
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr), \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),     \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),           \
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),         \
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),         \
        "r"(r[29]), "r"(r[30]), "r"(r[31])                                                           \
        : "memory")

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// 3-d tiled TMA load of a box at {c0, c1, c2} into this CTA's shared memory
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                       uint32_t bar) {
    // the KV stream is read once: its lines go first when L2 needs room (the
    // partials, page table and queries stay)
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;\n" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
        : "memory");
}

// non-blocking: has the phase with this parity completed?
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// an event-driven MMA issuer's no-progress limit in SM cycles (about 2 s at
// 2 GHz, longer at lower clocks)
constexpr long long kSpinCycles = 1LL << 32;

// Bounded wait shared by every waiter of a kernel, one copy of the spin loop
// for all call sites (the loop sits on the instruction stream of every
// waiting warp). After a timeout it flags VA_ERR_TIMEOUT with the wait site
// and raises the CTA's abort flag; once the flag is up nobody waits again.
static __device__ __noinline__ void wait_or_abort(uint32_t bar, uint32_t parity, int site, int* abort_flag,
                                                  int* header) {
    if (*(volatile int*)abort_flag) return;
    if (!mbar_wait(bar, parity)) {
        atomicOr(header + kHdrError, VA_ERR_TIMEOUT);
        atomicOr(header + kHdrWaitSites, 1 << site);
        *(volatile int*)abort_flag = 1;
    }
}
// The common case -- the phase has already completed -- stays inline.
__device__ __forceinline__ void wait_fast(uint32_t bar, uint32_t parity, int site, int* abort_flag, int* header) {
    if (!mbar_try_wait(bar, parity)) wait_or_abort(bar, parity, site, abort_flag, header);
}

}  // namespace tc
}  // namespace va
