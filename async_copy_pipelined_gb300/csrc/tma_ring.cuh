// A ring of S shared-memory stages guarded by full/empty mbarriers: the
// block-scoped pipeline of "A study on CUDA async memcpy" (section
// "block-scoped pipeline": per stage a produced and a consumed barrier,
// consumers pre-release every stage so producers can start, acquire = wait
// consumed, commit = arrive produced, consumer_wait = wait produced,
// release = arrive consumed), driven here by TMA transaction counts.
//
// Position f (0, 1, 2, ...) uses stage f % S; the barrier phase it waits for
// has parity (f / S) & 1.  Instead of a pre-release, the producer's first
// pass waits on parity 1 of the empty barriers, a phase a freshly initialised
// mbarrier reports as already complete.
//
// Shared by the FP32 TMA fill and the BF16 tensor-core kernel: the FP32
// consumers release a stage with an mbarrier arrive per warp, the tensor-core
// path with tcgen05.commit once its MMAs have read the stage.
#pragma once

#include "ptx.cuh"

namespace pg {

template <int S>
struct TmaRing {
    uint32_t full0;  // shared address of full[0]; full[s] at full0 + 8 s
    uint32_t empty0; // shared address of empty[0]

    __device__ __forceinline__ uint32_t full_bar(int f) const { return full0 + 8u * static_cast<uint32_t>(f % S); }
    __device__ __forceinline__ uint32_t empty_bar(int f) const { return empty0 + 8u * static_cast<uint32_t>(f % S); }
    __device__ __forceinline__ static uint32_t parity(int f) { return static_cast<uint32_t>((f / S) & 1); }
    // The same for unsigned positions: a position whose start is not known
    // to the compiler (a persistent kernel's) then costs no sign fix-ups.
    __device__ __forceinline__ uint32_t full_bar(unsigned f) const { return full0 + 8u * (f % S); }
    __device__ __forceinline__ uint32_t empty_bar(unsigned f) const { return empty0 + 8u * (f % S); }
    __device__ __forceinline__ static uint32_t parity(unsigned f) { return (f / S) & 1u; }

    // One thread, before the CTA barrier that publishes the ring.
    // full: `fills` arrivals per filling (1: the TMA producer's
    // arrive.expect_tx, completed by the copy bytes; or one per copying
    // thread).  empty: `releases` arrivals per consumption.
    __device__ __forceinline__ void init(uint32_t releases, uint32_t fills = 1) const
    {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, fills);
            mbar_init(empty0 + 8u * s, releases);
        }
        fence_barrier_init();
    }

    // Producer: wait until stage f % S has been released by its last user.
    template <class F>
    __device__ __forceinline__ bool producer_acquire(F f, uint64_t limit_ns) const
    {
        return mbar_wait_bounded(empty_bar(f), parity(f) ^ 1u, limit_ns);
    }

    // Producer: announce the bytes the copies of position f will deliver.
    template <class F>
    __device__ __forceinline__ void producer_commit(F f, uint32_t bytes) const
    {
        mbar_arrive_expect_tx(full_bar(f), bytes);
    }

    // Consumer: wait until every byte of position f has landed.
    template <class F>
    __device__ __forceinline__ bool consumer_wait(F f, uint64_t limit_ns) const
    {
        return mbar_wait_bounded(full_bar(f), parity(f), limit_ns);
    }

    // Consumer: one arrival on the stage's empty barrier.
    template <class F>
    __device__ __forceinline__ void consumer_release(F f) const { mbar_arrive(empty_bar(f)); }
};

// Round a shared-memory address up to `align` bytes (a power of two).
__device__ __forceinline__ uint32_t align_smem(uint32_t addr, uint32_t align)
{
    return (addr + align - 1u) & ~(align - 1u);
}

} // namespace pg
