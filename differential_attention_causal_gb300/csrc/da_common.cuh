// da_common.cuh -- device helpers shared by the CUDA kernels of libdiffattn:
// bounded mbarrier waits, TMA tensor loads, tcgen05 (TMEM + tensor-core MMA)
// wrappers, warp-level mma.sync / ldmatrix / movmatrix wrappers.
//
// All inline PTX here is hand-written against the public PTX ISA for sm_100a /
// sm_103a.  Every wait is bounded: after kWaitTimeoutNs of global time, or as
// soon as another CTA has recorded an error, the wait records an error bit in
// the caller's device error word and returns false so the kernel can unwind
// instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "da_internal.h"

namespace da {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s of global time

// Bounds checks of the debug build (compiled with -DDA_DEBUG_CHECKS): at the
// places where a kernel writes memory through a computed index, DA_CHECK(cond,
// err) tests the index against the extent of its tensor or tile; a failed
// test records kErrBounds in the error word and yields false, and the caller
// skips the access.  Nothing traps.  In the release build DA_CHECK is the
// constant true and the test is not compiled.
#ifdef DA_DEBUG_CHECKS
__device__ __forceinline__ bool da_check(bool c, uint32_t *err) {
    if (!c && err) atomicOr(err, kErrBounds);
    return c;
}
#define DA_CHECK(cond, err) ::da::da_check((cond), (err))
#else
#define DA_CHECK(cond, err) true
#endif


__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Arrive once per warp, from the lane elect.sync chooses, with no branch.
__device__ __forceinline__ void mbar_arrive_elect(uint32_t bar) {
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t@e mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar)
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
// Wait for the phase with the given parity to complete.  Returns false after
// recording kErrWaitTimeout if it does not within kWaitTimeoutNs, or false at
// once if the error word already holds a fatal bit (another CTA gave up).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0) {
            if ((ld_volatile_u32(err) & kErrFatal) != 0) return false;
            if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                atomicOr(err, kErrWaitTimeout);
                return false;
            }
        }
    }
}

// Named barrier over `nthreads` threads (multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warp-uniform bounded wait: every lane waits, the result is the AND over the
// warp (so warp-collective tcgen05 instructions that follow stay uniform).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t *err, bool ok) {
    if (ok) ok = mbar_wait(bar, parity, err);
    return __all_sync(0xffffffffu, ok);
}
// The same wait as a loop whose every decision (done, another CTA's fatal
// error, the time limit) is a warp vote, so it has no divergent branch and
// the warp never leaves the converged path.  Returns false at once if any
// lane comes in with ok == false.  Measured on GB300: the V1 d = 64 prefill
// 7 % faster with it, the V1 backward 4 % slower, so the prefill uses it.
__device__ __forceinline__ bool warp_wait_vote(uint32_t bar, uint32_t parity, uint32_t *err, bool ok) {
    if (!__all_sync(0xffffffffu, ok)) return false;
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if ((i & 63u) == 0) {
            const bool fatal = (ld_volatile_u32(err) & kErrFatal) != 0;
            const bool late = global_timer_ns() - t0 > kWaitTimeoutNs;
            if (__any_sync(0xffffffffu, fatal)) return false;
            if (__any_sync(0xffffffffu, late)) {
                if ((threadIdx.x & 31) == 0) atomicOr(err, kErrWaitTimeout);
                return false;
            }
        }
    }
}

// Waits for copies or MMAs that this CTA issued itself, before it exits or
// frees TMEM: bounded by the time limit only, and not cut short when another
// CTA has recorded an error, because shared memory and TMEM must not be
// released under an asynchronous write.  Such phases always complete (the
// copy or MMA was issued), so these return at once in practice.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint32_t *err) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && global_timer_ns() - t0 > kWaitTimeoutNs) {
            atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
}
__device__ __forceinline__ bool warp_wait_drain(uint32_t bar, uint32_t parity, uint32_t *err) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if ((i & 63u) == 63u && __any_sync(0xffffffffu, global_timer_ns() - t0 > kWaitTimeoutNs)) {
            if ((threadIdx.x & 31) == 0) atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 4-D tiled load, coordinates innermost first.  c0 * element size must be a
// multiple of 16 bytes (callers pass multiples of 64 elements).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// L2 eviction priorities for TMA copies (createpolicy, the whole access
// range): evict_first for data read or written once, evict_last for tiles
// that other CTAs read again.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// tma_load_4d with an L2 cache policy.
__device__ __forceinline__ void tma_load_4d_hint(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(pol)
        : "memory");
}
// Warp-converged forms of the above: every lane executes them, one lane
// chosen by elect.sync issues.
__device__ __forceinline__ void tma_load_4d_hint_elect(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                       int c0, int c1, int c2, int c3, uint64_t pol) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_load_4d_elect(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                                  int c0, int c1, int c2, int c3) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}
// tma_store_4d with an L2 cache policy.
__device__ __forceinline__ void tma_store_4d_hint(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2, int c3,
                                                  uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4, %5}], [%1], %6;" ::"l"(
            reinterpret_cast<uint64_t>(m)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(pol)
        : "memory");
}

// 4-D tiled store from shared memory (bulk group); the box comes from the map.
// 5-D tiled load (coordinates innermost first); the same alignment rule on c0.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(m)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until the shared-memory sources of all committed bulk stores have been read
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// wait until all committed bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------------------- tcgen05
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
// D(tmem) (+)= A(smem desc) * B(smem desc)^T, kind::f16 (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D(tmem) (+)= A(tmem) * B(smem desc)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Warp-converged issue: every lane of the warp executes these, one lane
// chosen by elect.sync issues the MMA or the commit.
__device__ __forceinline__ void mma_ss_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_elect(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
                 : "memory");
}
// Arrive (once) on an mbarrier when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bit, 16 consecutive columns -> r[0..15] (thread t <-> lane base+t)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
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

// Shared-memory matrix descriptor (tcgen05 format): 128-byte swizzle, rows of
// 128 bytes.  lbo / sbo in bytes; the address must lie in a tile whose base is
// 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;     // descriptor version for this architecture
    d |= static_cast<uint64_t>(2u) << 61;     // layout: 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16: bf16 A and B, fp32 D, dense.
// b_mn_major: B given with its N dimension contiguous.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4)                                   // D format: f32
           | (1u << 7)                                 // A format: bf16
           | (1u << 10)                                // B format: bf16
           | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// --------------------------------------------------------- warp-level MMA
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}
// C[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_16816(float *c, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Per-warpgroup register budget changes (all four warps of a warpgroup must
// execute the same one).  An increase waits until decreases elsewhere in the
// CTA have returned enough registers, so the host must check that the
// launch-time budget covers the sum before launching.
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------- math
__device__ __forceinline__ float ex2(float x) {   // 2^x, hardware approximation
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
// Row max of 128 raw scores with eight independent chains of 3-input max.
__device__ __forceinline__ float row_max128(const uint32_t *s) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = fmaxf(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
#pragma unroll
    for (int k = 16; k < 128; k += 16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = fmax3(a[i], __uint_as_float(s[k + 2 * i]), __uint_as_float(s[k + 2 * i + 1]));
    }
    return fmaxf(fmax3(a[0], a[1], a[2]), fmax3(fmax3(a[3], a[4], a[5]), a[6], a[7]));
}

// Rotary embedding: f_i = base^(-2i/D) for pair i < D/2, in double, kept as
// the float pair fhi + flo.
__device__ __forceinline__ void rope_freq(double base, int i, int D, float &fhi, float &flo) {
    const double f = exp(-2.0 * static_cast<double>(i) / static_cast<double>(D) * log(base));
    fhi = static_cast<float>(f);
    flo = static_cast<float>(f - static_cast<double>(fhi));
}
// cos and sin of the angle pos * (fhi + flo).  The product is carried as a
// float pair (its rounding error recovered with an fma) and reduced modulo
// 2 pi against 2 pi split into three floats, each step an fma (Cody and
// Waite's additive reduction): the reduced angle, in [-pi, pi], is within a
// few 1e-7 rad of the exact one for any position below 2^24.  Its cosine and
// sine come from the hardware approximations __cosf / __sinf, whose absolute
// error on [-pi, pi] is below 2^-21.4.  Every kernel that rotates calls this
// one function, so the prologue and the prefill's in-place Q rotation apply
// the same bits.
__device__ __forceinline__ float2 rope_cs(float pos, float fhi, float flo) {
    constexpr double TWO_PI = 6.283185307179586476925286766559;
    constexpr float P1 = static_cast<float>(TWO_PI);
    constexpr float P2 = static_cast<float>(TWO_PI - static_cast<double>(P1));
    constexpr float P3 = static_cast<float>(TWO_PI - static_cast<double>(P1) - static_cast<double>(P2));
    constexpr float INV_2PI = static_cast<float>(1.0 / TWO_PI);
    const float hi = pos * fhi;
    const float lo = fmaf(pos, flo, fmaf(pos, fhi, -hi));
    const float k = rintf(hi * INV_2PI);
    float r = fmaf(-k, P1, hi);
    r = fmaf(-k, P2, r);
    r = fmaf(-k, P3, r) + lo;
    return make_float2(__cosf(r), __sinf(r));
}

// Rotary embedding of one pair (a = x_i, b = x_{i + D/2}) by the angle whose
// cosine and sine are c, s: (a c - b s, b c + a s), each an fma over a
// rounded product, so that every kernel that rotates gets the same bits.
__device__ __forceinline__ void rope_rotate(float a, float b, float c, float s, float &ra, float &rb) {
    ra = fmaf(a, c, -(b * s));
    rb = fmaf(b, c, a * s);
}
// The same for two pairs at once on the paired fp32 units (same bits per lane).
__device__ __forceinline__ void rope_rotate2(float2 a, float2 b, float2 c, float2 s, float2 &ra, float2 &rb) {
    const float2 bs = __fmul2_rn(b, s);
    ra = __ffma2_rn(a, c, make_float2(-bs.x, -bs.y));
    rb = __ffma2_rn(b, c, __fmul2_rn(a, s));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace da
