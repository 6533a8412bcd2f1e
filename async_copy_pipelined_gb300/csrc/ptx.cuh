// Inline-PTX wrappers for sm_103a: cp.async with group completion, mbarrier
// with bounded waits, TMA bulk-tensor loads, and tcgen05 (TMEM alloc, MMA,
// commit, load).  Written from the public PTX ISA; nothing here falls back to
// another instruction: each wrapper emits exactly the instruction it names
// ("cp.async", section "Completion and errors": lowering never substitutes a
// synchronous copy or a narrower instruction).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pg {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- cp.async
// 16-byte copy, L2 only (.cg).  `src_bytes` in 0..16: that many bytes are
// read from `src`, the rest of the 16 are zero-filled.  `src` must be a valid
// 16-byte-aligned global address even when src_bytes == 0.
__device__ __forceinline__ void cp_async_cg16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

// 16-byte copy of an in-range chunk (no source-size operand).
__device__ __forceinline__ void cp_async_cg16_full(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}

// Optional cache qualifiers of a cp.async copy ("cp.async" tile-op
// reference, "Call parameters": a cache_policy operand; "Operand contract":
// the .L2::64B / 128B / 256B prefetch size).  CopyForm bit 0: .L2::128B
// prefetch; bit 1: .L2::cache_hint with a 64-bit policy from createpolicy.
// Form 0 is the plain instruction.
template <int Form>
__device__ __forceinline__ void cp_async_cg16_full_f(uint32_t dst, const void *src, uint64_t pol)
{
    if constexpr (Form == 0)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
    else if constexpr (Form == 1)
        asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
    else if constexpr (Form == 2)
        asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "l"(pol)
                     : "memory");
    else
        asm volatile("cp.async.cg.shared.global.L2::cache_hint.L2::128B [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                     "l"(pol)
                     : "memory");
}

template <int Form>
__device__ __forceinline__ void cp_async_cg16_f(uint32_t dst, const void *src, uint32_t src_bytes, uint64_t pol)
{
    if constexpr (Form == 0)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
    else if constexpr (Form == 1)
        asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                     "r"(src_bytes)
                     : "memory");
    else if constexpr (Form == 2)
        asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst), "l"(src),
                     "r"(src_bytes), "l"(pol)
                     : "memory");
    else
        asm volatile("cp.async.cg.shared.global.L2::cache_hint.L2::128B [%0], [%1], 16, %2, %3;\n" ::"r"(dst),
                     "l"(src), "r"(src_bytes), "l"(pol)
                     : "memory");
}

// The 4-byte .ca copy takes the prefetch qualifier only (Form bit 0): the
// library never attaches a cache policy to it (see gemm_f32's option check).
template <int Form>
__device__ __forceinline__ void cp_async_ca4_f(uint32_t dst, const void *src, uint32_t src_bytes)
{
    static_assert(Form == 0 || Form == 1, "no cache policy on 4-byte copies");
    if constexpr (Form == 0)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                     : "memory");
    else
        asm volatile("cp.async.ca.shared.global.L2::128B [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
                     "r"(src_bytes)
                     : "memory");
}

// L2 eviction policy for the .L2::cache_hint forms: kind 1 evict_first,
// 2 evict_last, anything else evict_normal (the default behaviour), each for
// the whole access (fraction 1.0).
__device__ __forceinline__ uint64_t l2_policy(int kind)
{
    uint64_t p;
    if (kind == 1)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    else if (kind == 2)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}

// 4-byte copy (.ca: the only cache qualifier allowed below 16 bytes).
__device__ __forceinline__ void cp_async_ca4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

// Make `bar` track this thread's prior cp.async copies: one arrive-on is
// triggered on the barrier when they have all completed.  .noinc: the
// barrier's expected count already includes that arrival.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// Wait until at most N of this thread's committed groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Hard cap on polls, whatever the timer says: every wait ends.
constexpr uint32_t kMaxPolls = 1u << 30;

// Wait for the phase of `bar` with the given parity to complete.  Gives up
// after `limit_ns` nanoseconds (checked every 64 polls) or kMaxPolls polls and
// returns false; returns true once the phase has completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t poll = 1; poll < kMaxPolls; ++poll) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((poll & 63u) == 0 && global_timer_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}

// Flags between CTAs of one grid, in global memory: a release store after
// this thread's (and, through a preceding CTA barrier, its CTA's) writes, and
// an acquire load that orders the reads after it.
__device__ __forceinline__ void st_release_gpu_u64(unsigned long long *addr, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;\n" ::"l"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu_u64(const unsigned long long *addr)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(addr) : "memory");
    return v;
}

// Wait until *flag == value, bounded like mbar_wait_bounded.
__device__ __forceinline__ bool flag_wait_bounded(const unsigned long long *flag, unsigned long long value,
                                                  uint64_t limit_ns)
{
    if (ld_acquire_gpu_u64(flag) == value)
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t poll = 1; poll < kMaxPolls; ++poll) {
        if (ld_acquire_gpu_u64(flag) == value)
            return true;
        if ((poll & 63u) == 0 && global_timer_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}

// Record the first error of this launch sequence in the device status word.
__device__ __forceinline__ void record_error(unsigned int *status, unsigned int code)
{
    if (status)
        atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at coordinates (x = innermost, y) into shared
// memory at `dst`, completing `bytes` of transaction count on `bar`.  No
// multicast: the copy goes only to this CTA's own shared memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];\n" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// The same load carrying an L2 cache policy (.L2::cache_hint).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y,
                                                 uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
        "%4}], [%2], %5;\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(pol)
        : "memory");
}

// Either form: `hint` selects the cache-policy form (one elected thread
// issues these, so a run-time choice costs nothing measurable).
__device__ __forceinline__ void tma_load_2d_opt(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y,
                                                bool hint, uint64_t pol)
{
    if (hint)
        tma_load_2d_hint(dst, map, bar, x, y, pol);
    else
        tma_load_2d(dst, map, bar, x, y);
}

// 2-D tiled store of the box at coordinates (x = innermost, y) from shared
// memory at `src` to global memory; parts of the box outside the tensor are
// not written.  The store joins this thread's current bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}

// Wait until at most N of this thread's bulk async-groups are still reading
// their shared-memory source (the source may then be overwritten).
template <int N>
__device__ __forceinline__ void bulk_wait_group_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk async-groups are incomplete
// (their global writes done).
template <int N>
__device__ __forceinline__ void bulk_wait_group()
{
    asm volatile("cp.async.bulk.wait_group %0;\n" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 x bf16 -> f32).
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all tcgen05 operations issued so far by this
// thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (base lane + t), columns col .. col+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Warp-wide store of 32 lanes x 32 consecutive 32-bit columns into tensor
// memory (the inverse of tmem_ld_32x32b_x32: lane i's r[j] goes to lane
// i, column taddr + j).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
          "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
          "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait()
{
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

} // namespace pg
