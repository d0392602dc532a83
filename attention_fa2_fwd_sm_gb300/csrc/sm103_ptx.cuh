// sm103_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family,
// built for sm_103a) features the kernels use: mbarriers with time-bounded
// waits, TMA tensor loads, tcgen05 MMA / TMEM access, and shared-memory
// matrix descriptors.  Encodings follow the public PTX ISA description of
// tcgen05 (instruction descriptor, shared-memory descriptor, canonical
// 128-byte-swizzled layouts).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace attn {

// ----------------------------------------------------------------- status
// Bits OR-ed into a kernel's device status word.
enum : int {
    kStatusTimeout = 1,   // a bounded wait ran out
    kStatusDrainTimeout = 2,  // the teardown drain of in-flight copies ran out
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// --------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of the same condition.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with parity `parity` of barrier `bar` has completed.
// Gives up after `limit_ns` nanoseconds or as soon as *abort is set by
// another role of the CTA; on giving up it sets *abort (so the other roles
// leave too) and ORs kStatusTimeout into *status.  Returns true on success.
// A limit of 0 fails any wait whose phase is not complete at the first,
// non-blocking probe.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  volatile int *abort, int *status) {
    if (limit_ns == 0) {
        if (mbar_test_wait(bar, parity)) return true;
        *abort = 1;
        atomicOr(status, kStatusTimeout);
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                *abort = 1;
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
}

// Warp-collective form of mbar_wait_bounded: all 32 lanes call it together
// and leave together (success or give-up), so warp-synchronous instructions
// that follow never see a partial warp.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                               volatile int *abort, int *status) {
    if (limit_ns == 0) {
        if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
        if ((threadIdx.x & 31) == 0) {
            *abort = 1;
            atomicOr(status, kStatusTimeout);
        }
        __syncwarp();
        return false;
    }
    bool done = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, done)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (!done) done = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, done)) return true;
        if ((it & 15u) == 0) {
            int give_up = 0;
            if ((threadIdx.x & 31) == 0) {
                if (*abort) {
                    give_up = 1;
                } else if (global_timer_ns() - t0 > limit_ns) {
                    *abort = 1;
                    atomicOr(status, kStatusTimeout);
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
        }
    }
}

// ------------------------------------------- programmatic dependent launch
// A grid launched with programmatic stream serialization may start before
// the grid ahead of it on the stream has finished.  griddep_wait() blocks
// until that grid has completed and its memory writes are visible (it
// returns at once when the launch has no such dependency);
// griddep_launch_dependents() lets the grid behind this one be scheduled
// before this one completes.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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
// MMA issue, warp-collective: all 32 lanes execute these together and the
// lane that elect.sync picks (the lowest, the same one every time) issues
// the instruction, so the issuing loop runs warp-uniform; a commit then
// covers every MMA issued before it.  Each call issues a group of four MMAs
// (kind::f16, one CTA) from one asm block, so the issuer spends no
// instructions between them; `acc0` enables accumulation for the first MMA
// and the later ones always accumulate.  SS: a[i], b[i] are the
// shared-memory descriptors of MMA i; TS: a[i] are the TMEM addresses of A,
// b[i] the shared-memory descriptors of B.
__device__ __forceinline__ void tc_mma_ss_x4_elect(uint32_t d, const uint64_t (&a)[4], const uint64_t (&b)[4],
                                                   uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p0, p1, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %9, 0;\n\t"
        "setp.eq.b32 p1, %9, %9;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %10, p0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %10, p1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %10, p1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %10, p1;\n\t}" ::"r"(d),
        "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc0),
        "r"(idesc)
        : "memory");
}
__device__ __forceinline__ void tc_mma_ts_x4_elect(uint32_t d, const uint32_t (&a)[4], const uint64_t (&b)[4],
                                                   uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p0, p1, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %9, 0;\n\t"
        "setp.eq.b32 p1, %9, %9;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %10, p0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %10, p1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %10, p1;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %10, p1;\n\t}" ::"r"(d),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(acc0),
        "r"(idesc)
        : "memory");
}
__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B,
// A K-major, B K-major (b_mn_major = 0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn_major) {
    return (1u << 4)                      // D format: f32
           | (1u << 7)                    // A format: bf16
           | (1u << 10)                   // B format: bf16
           | (uint32_t(b_mn_major) << 16) // B major-ness
           | (uint32_t(N >> 3) << 17)     // N / 8
           | (uint32_t(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor for a 128-byte-swizzled canonical layout.
// lbo / sbo in bytes (multiples of 16).  K-major: rows of 128 B, 8-row groups
// sbo apart (lbo unused).  MN-major: 64-element MN chunks lbo apart, 8-row K
// groups sbo apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t((lbo >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;  // descriptor version for tcgen05
    d |= uint64_t(2) << 61;  // layout: 128-byte swizzle
    return d;
}

// TMEM loads / stores: warp w (w % 4 = quarter) touches lanes [32*quarter, +32);
// thread `lane` gets lane 32*quarter+lane, consecutive 32-bit columns.
#define ATTN_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                   "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define ATTN_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                   "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24)
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        ATTN_W8(0), ATTN_W8(8), ATTN_W8(16), ATTN_W8(24)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        ATTN_W8(0), ATTN_W8(8)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef ATTN_R8
#undef ATTN_W8

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1) as one paired fp32 FMA.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %5};\n\t"
        "mov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// (d0, d1) += (a0, a1) as one paired fp32 add.
__device__ __forceinline__ void fadd2(float &d0, float &d1, float a0, float a1) {
    asm("{\n\t.reg .b64 a, d;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 d, {%0, %1};\n\t"
        "add.rn.f32x2 d, d, a;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace attn
