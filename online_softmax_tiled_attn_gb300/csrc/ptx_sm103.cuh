// ptx_sm103.cuh -- thin inline-PTX wrappers for the sm_103a features the kernels use:
// mbarriers (with bounded waits), TMA tensor loads, tcgen05 MMA / TMEM and fences.
//
// Every wait here is bounded: it polls with mbarrier.try_wait and gives up after a
// %globaltimer deadline, reporting failure to the caller so the kernel can record an error
// code and leave cleanly instead of hanging the GPU.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace osm {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
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

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// As mbar_try_wait, but the thread may be suspended until the phase completes or about
// `suspend_ns` nanoseconds have passed, instead of returning at once: waiting threads then
// take no issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity,
                                                      uint32_t suspend_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if `timeout_ns`
// elapsed first (the caller then records an error and stops).  Waits on the critical path
// poll; the others (`suspend`) let the thread sleep between polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                          bool suspend = false) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (suspend ? mbar_try_wait_suspend(bar, parity, 100000u) : mbar_try_wait(bar, parity))
            return true;
        if ((suspend || (it & 63u) == 63u) && globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// ------------------------------------------------------------------------------------------
// fences
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Register reallocation between warpgroups (all four warps of a warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// Named barrier over a subset of warps (id 1..15; count a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate over the participating threads: every thread gets
// true only if all of them passed true.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------------------------------
// TMA
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// 4-D tiled load of one box into shared memory, completing bytes on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3)
        : "memory");
}

// 3-D tiled store of one box from shared memory (the tensor map's layout and swizzle) to
// global memory, in the issuing thread's bulk group; elements outside the tensor are not
// written.  The shared-memory writes it reads must be fenced for the async proxy first.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int32_t c0,
                                             int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until at most N of this thread's bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Until at most N of this thread's bulk groups are still incomplete (writes done).
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Untiled bulk copy of `bytes` contiguous bytes from global memory into this CTA's shared
// memory, completing the bytes on `bar`.  Both addresses must be 16-byte aligned and `bytes`
// a multiple of 16 (the caller checks).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05: TMEM allocation
// ------------------------------------------------------------------------------------------
// Whole warp: allocates `ncols` TMEM columns and writes the base address to *dst (smem).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
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

// ------------------------------------------------------------------------------------------
// tcgen05: MMA (kind::f16: bf16 in, fp32 accumulate) and commit
// ------------------------------------------------------------------------------------------
// Eight back-to-back TS MMAs D += A_k B_k (k = 0..7) in one statement, so that the issuing
// thread spends as few instructions as possible between them: A_k at TMEM column a_tmem + 8k
// (16 bf16 values per row), B_k described by b_desc with its start address advanced by
// b_step16 x 16 bytes per k.  The first MMA overwrites D when `accumulate` is 0.
__device__ __forceinline__ void umma_ts_x8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t b_step16, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t.reg .b64 st;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.eq.b32 q, %5, %5;\n\t"
        "cvt.u64.u32 st, %3;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t"
        "add.u32 a, %1, 8;\n\tadd.s64 b, %2, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(b_step16), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four back-to-back SS MMAs D (+)= A_k B_k over one 64-column half of K-major, 128-byte
// swizzled A and B tiles: the K16 steps advance both start addresses by 32 bytes.  The first
// MMA overwrites D when `accumulate` is 0.
__device__ __forceinline__ void umma_ss_x4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 a, b;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "add.s64 a, %1, 2;\n\tadd.s64 b, %2, 2;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
        "add.s64 a, a, 2;\n\tadd.s64 b, b, 2;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
        "add.s64 a, a, 2;\n\tadd.s64 b, b, 2;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four back-to-back TS MMAs D (+)= A_k B_k with A (bf16 pairs) in TMEM at a_tmem + 16 k (8
// columns each: the operand of every K16 step starts a 16-column group); B_k described by
// b_desc advanced by 2048 bytes (16 rows of a 128-byte swizzled MN-major tile) per step.
__device__ __forceinline__ void umma_ts_x4_stride16(uint32_t d_tmem, uint32_t a_tmem,
                                                    uint64_t b_desc, uint32_t idesc,
                                                    uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 a, %1, 16;\n\tadd.s64 b, %2, 128;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
        "add.u32 a, %1, 32;\n\tadd.s64 b, b, 128;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
        "add.u32 a, %1, 48;\n\tadd.s64 b, b, 128;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four back-to-back TS MMAs, as umma_ts_x8.
__device__ __forceinline__ void umma_ts_x4(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t b_step16, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t.reg .b64 st;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.eq.b32 q, %5, %5;\n\t"
        "cvt.u64.u32 st, %3;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t"
        "add.u32 a, %1, 8;\n\tadd.s64 b, %2, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(b_step16), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ------------------------------------------------------------------------------------------
// The same issue paths for a whole, converged warp: every lane runs the issuing loop (so the
// operands are warp-uniform values) and the lane that elect.sync picks issues each
// instruction.  One warp issues M128 N64 K16 products this way at the tensor core's full rate
// (32 clocks each); a loop run by lane 0 alone reaches one per ~49 clocks.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void umma_ss_x4_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t.reg .b64 a, b;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "add.s64 a, %1, 2;\n\tadd.s64 b, %2, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
        "add.s64 a, a, 2;\n\tadd.s64 b, b, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t"
        "add.s64 a, a, 2;\n\tadd.s64 b, b, 2;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, q;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_ts_x4_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t b_step16, uint32_t idesc,
                                                uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t.reg .b64 st;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.eq.b32 q, %5, %5;\n\t"
        "cvt.u64.u32 st, %3;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t"
        "add.u32 a, %1, 8;\n\tadd.s64 b, %2, st;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t"
        "add.u32 a, a, 8;\n\tadd.s64 b, b, st;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %4, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(b_step16), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_ts_x8_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t b_step16, uint32_t idesc,
                                                uint32_t accumulate) {
    umma_ts_x4_warp(d_tmem, a_tmem, b_desc, b_step16, idesc, accumulate);
    umma_ts_x4_warp(d_tmem, a_tmem + 32, b_desc + 4ull * b_step16, b_step16, idesc, 1u);
}

__device__ __forceinline__ void umma_ts_x4_stride16_warp(uint32_t d_tmem, uint32_t a_tmem,
                                                         uint64_t b_desc, uint32_t idesc,
                                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t.reg .b64 b;\n\t.reg .b32 a;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "add.u32 a, %1, 16;\n\tadd.s64 b, %2, 128;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
        "add.u32 a, %1, 32;\n\tadd.s64 b, b, 128;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t"
        "add.u32 a, %1, 48;\n\tadd.s64 b, b, 128;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_cp_128x256b_warp(uint32_t taddr, uint64_t s_desc) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.128x256b [%0], %1;\n\t}" ::"r"(taddr), "l"(s_desc)
        : "memory");
}

// Arrives once on `bar` when all tcgen05 operations issued so far by the elected lane end.
// Every MMA of a warp that uses these helpers is issued by the same elected lane (elect.sync
// picks the lowest active lane, and the loops run fully converged).
__device__ __forceinline__ void umma_commit_warp(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

// An MMA issuer's primitives, for a converged warp (W = true; the helpers above) or for a loop
// run by lane 0 alone (W = false): waits (made warp-uniform in the first case), products,
// copies and commits.
template <bool W>
__device__ __forceinline__ bool issuer_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                            bool sleep = false);
template <bool W>
__device__ __forceinline__ void issue_commit(uint64_t* bar);
template <bool W>
__device__ __forceinline__ void issue_ss_x4(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                            uint32_t acc);
template <bool W>
__device__ __forceinline__ void issue_ts_x4(uint32_t d, uint32_t a, uint64_t b, uint32_t step,
                                            uint32_t id, uint32_t acc);
template <bool W>
__device__ __forceinline__ void issue_ts_x8(uint32_t d, uint32_t a, uint64_t b, uint32_t step,
                                            uint32_t id, uint32_t acc);
template <bool W>
__device__ __forceinline__ void issue_ts_x4_stride16(uint32_t d, uint32_t a, uint64_t b,
                                                     uint32_t id, uint32_t acc);
template <bool W>
__device__ __forceinline__ void issue_tmem_cp(uint32_t taddr, uint64_t desc);

// Asynchronous copy of a 128-row x 256-bit matrix from shared memory (described by a matrix
// descriptor, like an MMA operand) into TMEM lanes 0-127, 8 columns from `taddr`.  Ordered
// before the tcgen05.mma instructions that the same thread issues after it.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t s_desc) {
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(s_desc)
                 : "memory");
}

// Arrives once on `bar` when all tcgen05 async operations issued so far by this thread end.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor (sm_100 family format): start address, leading and stride
// byte offsets (all in 16-byte units), descriptor version 1, and the 128-byte swizzle mode.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;  // version
    d |= (uint64_t)2u << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn) {
    return (1u << 4)            // D format: f32
           | (1u << 7)          // A format: bf16
           | (1u << 10)         // B format: bf16
           | (0u << 15)         // A K-major
           | (b_mn << 16)       // B major-ness
           | ((N >> 3) << 17)   // N / 8
           | ((M >> 4) << 24);  // M / 16
}

// As idesc_bf16_f32 with the major-ness of A chosen too (a_mn = 1: M contiguous in memory).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_ab(uint32_t M, uint32_t N, uint32_t a_mn,
                                                         uint32_t b_mn) {
    return idesc_bf16_f32(M, N, b_mn) | (a_mn << 15);
}

// ------------------------------------------------------------------------------------------
// tcgen05: TMEM <-> registers, 32 lanes x 32 bits shape (thread t of the warp <-> lane t)
// ------------------------------------------------------------------------------------------
// Each load is issued together with its tcgen05.wait::ld in ONE asm statement, so the
// compiler cannot schedule a use of the destination registers before the data has arrived.
// Each store is likewise followed by its tcgen05.wait::st in the same statement.

// 32 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 16 consecutive columns at each of two TMEM addresses of this thread's lane (two loads,
// one wait).
__device__ __forceinline__ void tmem_ld16x2_sync(uint32_t ta, uint32_t tb, uint32_t (&a)[16],
                                                 uint32_t (&b)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
        : "r"(ta), "r"(tb)
        : "memory");
}

// 8 consecutive columns at each of two TMEM addresses of this thread's lane (two loads, one
// wait).
__device__ __forceinline__ void tmem_ld8x2_sync(uint32_t ta, uint32_t tb, uint32_t (&a)[8],
                                                uint32_t (&b)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
          "=r"(a[7]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]),
          "=r"(b[6]), "=r"(b[7])
        : "r"(ta), "r"(tb)
        : "memory");
}

// 16 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16_sync(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// 128 consecutive columns of this thread's lane (four 32-column loads, one wait).
__device__ __forceinline__ void tmem_ld128_sync(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "{\n\t.reg .b32 ta;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
        "add.u32 ta, %128, 32;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [ta];\n\t"
        "add.u32 ta, %128, 64;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [ta];\n\t"
        "add.u32 ta, %128, 96;\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [ta];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n\t}"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st32_sync(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 8 consecutive columns at each of two TMEM addresses of this thread's lane (two stores,
// one wait).
__device__ __forceinline__ void tmem_st8x2_sync(uint32_t ta, const uint32_t (&a)[8], uint32_t tb,
                                                const uint32_t (&b)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%2,%3,%4,%5,%6,%7,%8,%9};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%1], {%10,%11,%12,%13,%14,%15,%16,%17};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(ta), "r"(tb),
        "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "r"(b[0]), "r"(b[1]), "r"(b[2]), "r"(b[3]), "r"(b[4]), "r"(b[5]), "r"(b[6]), "r"(b[7])
        : "memory");
}

// 8 consecutive columns of this thread's lane.
__device__ __forceinline__ void tmem_st8_sync(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// 64 consecutive columns of this thread's lane (two 32-column stores, one wait).
__device__ __forceinline__ void tmem_st64_sync(uint32_t taddr, const uint32_t (&r)[64]) {
    asm volatile(
        "{\n\t.reg .b32 ta;\n\t"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "add.u32 ta, %0, 32;\n\t"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [ta], {%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n\t"
        "tcgen05.wait::st.sync.aligned;\n\t}" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

// ------------------------------------------------------------------------------------------
// arithmetic
// ------------------------------------------------------------------------------------------
// Hardware base-2 exponential (MUFU), flush-to-zero; ex2(-inf) = +0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed pairs of fp32 (one instruction for two lanes of arithmetic on sm_100 and later).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <bool W>
__device__ __forceinline__ bool issuer_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                            bool sleep) {
    const bool ok = mbar_wait(bar, parity, timeout_ns, sleep);
    if constexpr (W) return __all_sync(0xffffffffu, ok);
    else return ok;
}
template <bool W>
__device__ __forceinline__ void issue_commit(uint64_t* bar) {
    if constexpr (W) umma_commit_warp(bar);
    else umma_commit(bar);
}
template <bool W>
__device__ __forceinline__ void issue_ss_x4(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                            uint32_t acc) {
    if constexpr (W) umma_ss_x4_warp(d, a, b, id, acc);
    else umma_ss_x4(d, a, b, id, acc);
}
template <bool W>
__device__ __forceinline__ void issue_ts_x4(uint32_t d, uint32_t a, uint64_t b, uint32_t step,
                                            uint32_t id, uint32_t acc) {
    if constexpr (W) umma_ts_x4_warp(d, a, b, step, id, acc);
    else umma_ts_x4(d, a, b, step, id, acc);
}
template <bool W>
__device__ __forceinline__ void issue_ts_x8(uint32_t d, uint32_t a, uint64_t b, uint32_t step,
                                            uint32_t id, uint32_t acc) {
    if constexpr (W) umma_ts_x8_warp(d, a, b, step, id, acc);
    else umma_ts_x8(d, a, b, step, id, acc);
}
template <bool W>
__device__ __forceinline__ void issue_ts_x4_stride16(uint32_t d, uint32_t a, uint64_t b,
                                                     uint32_t id, uint32_t acc) {
    if constexpr (W) umma_ts_x4_stride16_warp(d, a, b, id, acc);
    else umma_ts_x4_stride16(d, a, b, id, acc);
}
template <bool W>
__device__ __forceinline__ void issue_tmem_cp(uint32_t taddr, uint64_t desc) {
    if constexpr (W) tmem_cp_128x256b_warp(taddr, desc);
    else tmem_cp_128x256b(taddr, desc);
}

}  // namespace osm
