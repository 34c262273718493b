// ptx.cuh -- hand-written inline-PTX wrappers for sm_103a: mbarrier, TMA
// (cp.async.bulk.tensor), tcgen05 (TMEM alloc / MMA / commit / ld / st) and
// the shared-memory and instruction descriptors the MMAs take.
//
// Every wait on an mbarrier is bounded: after `kWaitLimitNs` of global time it
// records a timeout in the library's device status word and returns false so
// the caller can unwind (no trap, no endless spin).
#pragma once

#include <cstdint>
#include <cuda.h>

namespace tme {

// Device status word (one per library, passed to every kernel):
// bit 0 = an mbarrier wait timed out.
constexpr unsigned kStatusTimeout = 1u;

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
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

// As above, but a thread whose phase is not complete yet is suspended by the
// hardware until it completes (or about `hint_ns` pass), so waiting warps do
// not take issue slots from the warps that share their SM sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

constexpr uint32_t kSuspendHintNs = 200000;  // 0.2 ms per suspension at most

// Wait until the phase with the given parity has completed.  Bounded: gives up
// after kWaitLimitNs (or at once when *abort is already set), sets *abort and
// the device status word, and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(a, parity, kSuspendHintNs)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Same bound, no shared abort flag (teardown waits).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned int* status) {
    const uint32_t a = smem_u32(bar);
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(a, parity, kSuspendHintNs)) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// Warp-uniform wait: every lane polls, and the warp proceeds only if all
// lanes saw the phase complete (so a timeout never splits the warp before a
// .sync.aligned tcgen05 instruction).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status) {
    const bool ok = mbar_wait(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completes `bytes` on `bar`.
__device__ __forceinline__ void tma_load_3d(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16);
// completes `bytes` on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 16-byte asynchronous copy global -> shared, cached in L2 only (both
// addresses 16-byte aligned).  Completion: cp_async_wait_all in the issuing
// thread, which then sees the data; other threads of the warp see it after a
// __syncwarp that follows that wait.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05

// Whole warp: allocate `ncols` TMEM columns, base address written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
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

// Groups of MMAs along K from one asm block with a single elect: the K-major
// operands of a 128-byte-swizzled tile advance by 32 bytes (descriptor +2) per
// K=16 step and by a 16 KiB block (+1024) every four steps.  `acc` selects
// accumulate for the first MMA; the others always accumulate.
__device__ __forceinline__ void mma_ss_k64(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n\t.reg .b32 lid;\n\t.reg .pred e, p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
        "elect.sync lid|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
        "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// O (+)= P V for 128 keys: 8 MMAs, A = P from TMEM (+8 columns per step), B =
// V MN-major in shared memory (+16 rows = 2048 bytes = +128 per step).
__device__ __forceinline__ void mma_ts_k128(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile(
        "{\n\t.reg .b32 lid, a1, a2, a3, a4, a5, a6, a7;\n\t.reg .pred e, p, t;\n\t"
        ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
        "elect.sync lid|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "add.s32 a1, %1, 8;\n\tadd.s32 a2, %1, 16;\n\tadd.s32 a3, %1, 24;\n\t"
        "add.s32 a4, %1, 32;\n\tadd.s32 a5, %1, 40;\n\tadd.s32 a6, %1, 48;\n\t"
        "add.s32 a7, %1, 56;\n\t"
        "add.s64 b1, %2, 128;\n\tadd.s64 b2, %2, 256;\n\tadd.s64 b3, %2, 384;\n\t"
        "add.s64 b4, %2, 512;\n\tadd.s64 b5, %2, 640;\n\tadd.s64 b6, %2, 768;\n\t"
        "add.s64 b7, %2, 896;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, t;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Four MMAs along K (64 values): A from TMEM columns a, a+8, a+16, a+24
// (packed 16-bit pairs), B descriptor advanced by 128 (2048 bytes: 16 rows of
// an MN-major 128-byte-swizzled tile) per step.
__device__ __forceinline__ void mma_ts_k64(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n\t.reg .b32 lid, a1, a2, a3;\n\t.reg .pred e, p, t;\n\t"
        ".reg .b64 b1, b2, b3;\n\t"
        "elect.sync lid|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "add.s32 a1, %1, 8;\n\tadd.s32 a2, %1, 16;\n\tadd.s32 a3, %1, 24;\n\t"
        "add.s64 b1, %2, 128;\n\tadd.s64 b2, %2, 256;\n\tadd.s64 b3, %2, 384;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// As mma_ts_k64, but the 64 K values of A come from two TMEM column ranges:
// steps 0-1 from a_lo, a_lo+8, steps 2-3 from a_hi, a_hi+8.
__device__ __forceinline__ void mma_ts_k64_split(uint32_t d, uint32_t a_lo, uint32_t a_hi,
                                                 uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .b32 lid, a1, a3;\n\t.reg .pred e, p, t;\n\t"
        ".reg .b64 b1, b2, b3;\n\t"
        "elect.sync lid|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "add.s32 a1, %1, 8;\n\tadd.s32 a3, %2, 8;\n\t"
        "add.s64 b1, %3, 128;\n\tadd.s64 b2, %3, 256;\n\tadd.s64 b3, %3, 384;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %3, %4, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %4, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], b2, %4, t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %4, t;\n\t}" ::"r"(d),
        "r"(a_lo), "r"(a_hi), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b32 lid;\n\t.reg .pred e;\n\t"
        "elect.sync lid|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Orders later uses of registers written by tcgen05.ld after the preceding
// tcgen05.wait::ld (a volatile asm with the registers as in/out operands).
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Warp-collective: lane i reads 32 consecutive 32-bit columns of TMEM lane
// (lane base of taddr) + i.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// 64 consecutive columns in one instruction: lane i reads columns 0-31 of
// TMEM lane (lane base) + i into r0 and columns 32-63 into r1.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r0)[32], uint32_t (&r1)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]),
          "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]),
          "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]), "=r"(r0[16]), "=r"(r0[17]),
          "=r"(r0[18]), "=r"(r0[19]), "=r"(r0[20]), "=r"(r0[21]), "=r"(r0[22]), "=r"(r0[23]),
          "=r"(r0[24]), "=r"(r0[25]), "=r"(r0[26]), "=r"(r0[27]), "=r"(r0[28]), "=r"(r0[29]),
          "=r"(r0[30]), "=r"(r0[31]), "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]),
          "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]), "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]),
          "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]), "=r"(r1[14]), "=r"(r1[15]),
          "=r"(r1[16]), "=r"(r1[17]), "=r"(r1[18]), "=r"(r1[19]), "=r"(r1[20]), "=r"(r1[21]),
          "=r"(r1[22]), "=r"(r1[23]), "=r"(r1[24]), "=r"(r1[25]), "=r"(r1[26]), "=r"(r1[27]),
          "=r"(r1[28]), "=r"(r1[29]), "=r"(r1[30]), "=r"(r1[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// ------------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor (tcgen05 form), 128-byte swizzle.
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-48 fixed 0b001
//   bits 49-51 base offset (0: every tile is 1024-byte aligned)
//   bit  52    LBO mode (0: relative)
//   bits 61-63 swizzle mode (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes & 0x3FFFFu) >> 4) << 16;
    d |= static_cast<uint64_t>((sbo_bytes & 0x3FFFFu) >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
//   bits 4-5 D format (1 = f32); bits 7-9 / 10-12 A / B format (0 = f16, 1 = bf16);
//   bit 15 / 16 A / B major (0 = K-major, 1 = MN-major); bits 17-22 N >> 3;
//   bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------ numerics

__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Pack two fp32 into one 32-bit word of two 16-bit values (round to nearest
// even); the first argument goes to the low half.
// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (one 64-bit register holds two floats, low = first).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    return static_cast<uint64_t>(__float_as_uint(lo)) |
           (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ float f2lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2hi(uint64_t v) {
    return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// 32-byte global store (one whole 32-byte sector when the address is
// 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// 32-bit shared-memory store / load at a shared-window address (smem_u32).
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}
// Named barrier `id` (1..15) over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (BF16) {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    } else {
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    }
    return r;
}

// Two softmax terms in one step: x = s * scale2 + negm2 (packed pair),
// p = 2^x per lane (flush-to-zero), acc += p (packed pair), and p rounded to a
// 16-bit pair (low half = first term): bf16 when OUT_BF16, else fp16.  Written
// as one asm block so the 64-bit pairs stay register pairs.
template <bool OUT_BF16, bool ADD = true>
__device__ __forceinline__ uint32_t softmax_pair(uint32_t s0, uint32_t s1, uint64_t scale2,
                                                 uint64_t negm2, uint64_t& acc) {
    if constexpr (!ADD) {
        // the accumulator's first pair: acc = p
        float a, b;
        asm("{\n\t.reg .b64 x;\n\t"
            "mov.b64 x, {%2, %3};\n\t"
            "fma.rn.f32x2 x, x, %4, %5;\n\t"
            "mov.b64 {%0, %1}, x;\n\t"
            "ex2.approx.ftz.f32 %0, %0;\n\t"
            "ex2.approx.ftz.f32 %1, %1;\n\t}"
            : "=f"(a), "=f"(b)
            : "r"(s0), "r"(s1), "l"(scale2), "l"(negm2));
        acc = f2(a, b);
        return pack2<OUT_BF16>(a, b);
    } else if constexpr (OUT_BF16) {
        uint32_t w;
        asm("{\n\t.reg .b64 x, p;\n\t.reg .f32 a, b;\n\t"
            "mov.b64 x, {%2, %3};\n\t"
            "fma.rn.f32x2 x, x, %4, %5;\n\t"
            "mov.b64 {a, b}, x;\n\t"
            "ex2.approx.ftz.f32 a, a;\n\t"
            "ex2.approx.ftz.f32 b, b;\n\t"
            "mov.b64 p, {a, b};\n\t"
            "add.rn.f32x2 %1, %1, p;\n\t"
            "cvt.rn.bf16x2.f32 %0, b, a;\n\t}"
            : "=r"(w), "+l"(acc)
            : "r"(s0), "r"(s1), "l"(scale2), "l"(negm2));
        return w;
    } else {
        uint32_t w;
        asm("{\n\t.reg .b64 x, p;\n\t.reg .f32 a, b;\n\t"
            "mov.b64 x, {%2, %3};\n\t"
            "fma.rn.f32x2 x, x, %4, %5;\n\t"
            "mov.b64 {a, b}, x;\n\t"
            "ex2.approx.ftz.f32 a, a;\n\t"
            "ex2.approx.ftz.f32 b, b;\n\t"
            "mov.b64 p, {a, b};\n\t"
            "add.rn.f32x2 %1, %1, p;\n\t"
            "cvt.rn.f16x2.f32 %0, b, a;\n\t}"
            : "=r"(w), "+l"(acc)
            : "r"(s0), "r"(s1), "l"(scale2), "l"(negm2));
        return w;
    }
}

// The softmax term of a score s: p = 2^(s * scale - m) computed exactly as
// softmax_pair computes it (the same fused multiply-add and ex2), and the
// rounding error of the 16-bit value the PV product uses for it: returns
// round16(p) - p (exact in fp32: the two are within one 16-bit ulp).
template <bool OUT_BF16>
__device__ __forceinline__ float round16_residual(float s, float scale, float neg_m) {
    float p, r;
    asm("{\n\t.reg .f32 x;\n\t"
        "fma.rn.f32 x, %1, %2, %3;\n\t"
        "ex2.approx.ftz.f32 %0, x;\n\t}"
        : "=f"(p)
        : "f"(s), "f"(scale), "f"(neg_m));
    if constexpr (OUT_BF16) {
        asm("{\n\t.reg .b16 h;\n\t"
            "cvt.rn.bf16.f32 h, %1;\n\t"
            "cvt.f32.bf16 %0, h;\n\t}"
            : "=f"(r)
            : "f"(p));
    } else {
        asm("{\n\t.reg .b16 h;\n\t"
            "cvt.rn.f16.f32 h, %1;\n\t"
            "cvt.f32.f16 %0, h;\n\t}"
            : "=f"(r)
            : "f"(p));
    }
    return r - p;
}

// Two bf16 values (one 32-bit word) as two fp16 values, rounded to nearest
// (exact for magnitudes in [2^-14, 2^16); smaller ones become fp16
// subnormals, off by at most 2^-25).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;"
        : "=r"(r)
        : "f"(__uint_as_float(w & 0xffff0000u)), "f"(__uint_as_float(w << 16)));
    return r;
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.mma operands) that another thread's barrier
// arrival releases.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}


}  // namespace tme
