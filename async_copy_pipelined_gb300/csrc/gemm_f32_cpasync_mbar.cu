// FP32 GEMM, fill (d): cp.async whose completion is tracked by mbarriers.
//
// The block-scoped pipeline of "A study on CUDA async memcpy" (sections
// "mbarrier based approach" and "block-scoped pipeline") as it comes out of
// the lesson's cuda::pipeline ("Day 74: Async copies and pipelines",
// "Results": the piped kernel lowers to cp.async plus
// cp.async.mbarrier.arrive).  Every thread is both producer and consumer, as
// in the lesson, but completion is no longer a per-thread group count plus a
// CTA barrier:
//
//   producer_acquire  wait empty[s]: every thread has released the stage
//   memcpy_async      this thread's cp.async copies of the slice
//   producer_commit   cp.async.mbarrier.arrive.noinc full[s]: the barrier's
//                     phase completes once all 256 threads' copies landed
//   consumer_wait     wait full[s]
//   consumer_release  one arrive per thread on empty[s]
//
// No CTA-wide barrier sits in the main loop; a warp only waits for the
// slowest warp of the slice whose stage it is about to refill.  From three
// stages on, that refill is issued halfway through a slice into the stage
// released two slices earlier, so the wait is normally already satisfied.
// Zero fill, chunk mapping and the inner product are those of the cp.async
// fill, so results are bit-identical to the other fills.  Waits are
// bounded; on expiry the warp records GEMM_ERR_TIMEOUT and stops, and every
// thread drains its own copies (cp.async.wait_all) before exit.
#include "f32_tile.cuh"
#include "tma_ring.cuh"

namespace pg {

template <class T, int S, int OPT>
__global__ void __launch_bounds__(T::kThreads, T::kMinBlocks) gemm_f32_cpasync_mbar_kernel(const F32Args p)
{
    // OPT: the copy form (cache qualifiers, 0..3), or 4 for plain copies
    // with the accumulators starting from C (GEMM_OPT_ACCUMULATE).
    constexpr int CF = OPT & 3;
    constexpr bool ACC = (OPT & 4) != 0;
    static_assert(S >= 2 && S <= 6, "stages");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = align_smem(smem_u32(smem_raw), 1024);
    float *stage0 = reinterpret_cast<float *>(smem_raw + (base - smem_u32(smem_raw)));
    const uint32_t bars = base + S * T::kStageBytes;
    const uint32_t full0 = bars;
    const uint32_t empty0 = bars + 8u * S;

    const int tid = threadIdx.x;
    const int lane = tid % 32;
    int m0, n0;
    tile_origin(T::BM, T::BN, m0, n0);
    const int tr = tid / T::kThreadCols;
    const int tc = tid % T::kThreadCols;
    const int k_slices = (p.K + T::BK - 1) / T::BK;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, T::kThreads); // one asynchronous arrival per thread
            mbar_init(empty0 + 8u * s, T::kThreads); // one release per thread
        }
        fence_barrier_init();
    }
    __syncthreads();

    auto full_bar = [&](int f) { return full0 + 8u * static_cast<uint32_t>(f % S); };
    auto empty_bar = [&](int f) { return empty0 + 8u * static_cast<uint32_t>(f % S); };
    auto parity = [](int f) { return static_cast<uint32_t>((f / S) & 1); };
    const CopyPolicies<CF> pol(p);
    auto issue = [&](int f) {
        if (f == p.withhold)
            return; // test hook: no copies and no arrival for this position
        issue_slice_cpasync_f<T, CF>(stage0 + (f % S) * T::kStageFloats, p, tid, m0, n0, f, pol.a, pol.b);
        cp_async_mbar_arrive_noinc(full_bar(f));
    };

    Accum<T> acc;
    init_tile<T, ACC>(p, m0, n0, tr, tc, acc);
    bool ok = true;

    // Lookahead: S-1 slices issued at the top of each slice for two stages;
    // from three stages on, S-2 slices ahead plus the refill issued halfway
    // through the slice, into the stage released two slices earlier, so the
    // empty-barrier wait is already satisfied and the copies take issue
    // slots among the FMAs (measured on GB300 at 4096^3: S = 6 52.7 -> 54.4
    // TFLOP/s, 64 tile S = 4 44.3 -> 45.9; refilling the stage released one
    // slice earlier, which waits for the slowest warp, gained nothing).
    constexpr int kAhead = S >= 3 ? S - 2 : S - 1;
    for (int f = 0; f < kAhead && f < k_slices; ++f)
        issue(f);

    auto wait_full = [&](int kt) {
        const bool landed = mbar_wait_bounded(full_bar(kt), parity(kt), p.wait_limit_ns);
        if (__all_sync(0xffffffffu, landed))
            return true;
        if (lane == 0)
            record_error(p.status, kErrFamilyF32CpAsyncMbar | kErrRoleConsumer);
        return false;
    };
    FragPipe<T, T::kBDistCpAsync> frag;
    auto refill = [&](int fetch) {
        if (fetch >= k_slices)
            return true;
        const bool free = mbar_wait_bounded(empty_bar(fetch), parity(fetch) ^ 1u, p.wait_limit_ns);
        if (!__all_sync(0xffffffffu, free)) {
            if (lane == 0)
                record_error(p.status, kErrFamilyF32CpAsyncMbar | kErrRoleProducer);
            return false;
        }
        issue(fetch);
        return true;
    };
    for (int kt = 0; kt < k_slices && ok; ++kt) {
        const int fetch = kt + kAhead;
        if constexpr (S < 3) {
            if (!refill(fetch)) {
                ok = false;
                break;
            }
        }
        if (!wait_full(kt)) {
            ok = false;
            break;
        }
        const float *sA = stage0 + (kt % S) * T::kStageFloats;
        frag.prime(sA, sA + T::kAFloats, tr, tc);
        // Every thread releases the stage once its own reads of it are
        // issued (its arrival orders them before the refill), rather than a
        // warp gathering at __syncwarp for one lane to arrive.  Measured on
        // GB300 at 4096^3: S4 53.4 -> 54.7 TFLOP/s, S3 52.4 -> 52.8, 64 tile
        // S4 43.5 -> 44.4.  (The same change cost the TMA and producer-warp
        // fills 0.5-4 %; they keep one arrival per warp.)
        frag.run_mid(sA, sA + T::kAFloats, tr, tc, acc, [&]() {
            mbar_arrive(empty_bar(kt));
        }, []() -> const float * { return nullptr; }, [&]() {
            if constexpr (S >= 3) {
                if (!refill(fetch))
                    ok = false;
            }
        });
    }
    cp_async_wait_all(); // none of this thread's copies may land after it exits

    if (ok)
        store_tile<T>(p, m0, n0, tr, tc, acc);
}

template <class T, int S, int CF>
static int launch_cpasync_mbar_t(const F32Args &a, cudaStream_t s)
{
    const int smem = f32_smem_bytes(T::BM, GEMM_FILL_CPASYNC_MBAR, S);
    static std::atomic<unsigned long long> limit_set[kMaxDevices];
    if (ensure_smem_limit(gemm_f32_cpasync_mbar_kernel<T, S, CF>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    const dim3 grid((a.N + T::BN - 1) / T::BN, (a.M + T::BM - 1) / T::BM);
    gemm_f32_cpasync_mbar_kernel<T, S, CF><<<grid, T::kThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

template <class T, int CF>
static int launch_cpasync_mbar_tile(const F32Args &a, cudaStream_t s)
{
    switch (a.stages) {
    case 2: return launch_cpasync_mbar_t<T, 2, CF>(a, s);
    case 3: return launch_cpasync_mbar_t<T, 3, CF>(a, s);
    case 4: return launch_cpasync_mbar_t<T, 4, CF>(a, s);
    case 5: return launch_cpasync_mbar_t<T, 5, CF>(a, s);
    case 6: return launch_cpasync_mbar_t<T, 6, CF>(a, s);
    default: return GEMM_ERR_INVALID_ARG;
    }
}

// The copy form is a template parameter, as for the group-completed fill.
template <int CF>
static int launch_cpasync_mbar_form(const F32Args &a, cudaStream_t s)
{
    if (a.tile == 32)
        return launch_cpasync_mbar_tile<TileXS, CF>(a, s);
    return a.tile == 128 ? launch_cpasync_mbar_tile<TileL, CF>(a, s) : launch_cpasync_mbar_tile<TileS, CF>(a, s);
}

int launch_f32_cpasync_mbar(const F32Args &a, cudaStream_t s)
{
    if (a.accumulate) // plain copies only: the planner refuses accumulate with cache qualifiers
        return launch_cpasync_mbar_form<4>(a, s);
    switch (a.copy_form) {
    case 0: return launch_cpasync_mbar_form<0>(a, s);
    case 1: return launch_cpasync_mbar_form<1>(a, s);
    case 2: return launch_cpasync_mbar_form<2>(a, s);
    default: return launch_cpasync_mbar_form<3>(a, s);
    }
}

} // namespace pg
