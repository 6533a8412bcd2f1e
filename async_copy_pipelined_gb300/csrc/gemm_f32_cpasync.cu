// FP32 GEMM, fill (b): cp.async with commit_group / wait_group completion.
//
// Each thread copies its chunks of the slice straight from global to shared
// memory with cp.async (no register on the way, "Day 74: Async copies and
// pipelines", section "A copy that skips the registers"), closes them into
// one commit group per slice, and keeps S-1 slices in flight ahead of the
// one being computed.  wait_group S-2 returns once at most S-2 of this
// thread's groups are pending, i.e. once its copies of the slice about to be
// consumed have landed ("A study on CUDA async memcpy", section
// "async-group based approach": wait until only the N most recent groups are
// in flight).  Completion is per thread, so one CTA barrier per slice makes
// every thread's copies visible to every other thread; the same barrier
// proves the stage about to be refilled has been consumed by all threads
// ("Day 74", "Pitfalls": a barrier alone does not wait for copies).
//
// The lookahead is the lesson's top-up loop ("pipelined_gemm.cu",
// matmulTilePiped) with the per-slice acquire/release of its pipeline object
// replaced by the group count and the barrier.  An empty group is committed
// past the last slice so the wait count stays uniform.
#include "f32_tile.cuh"

namespace pg {

template <class T, int S, int OPT>
__global__ void __launch_bounds__(T::kThreads, T::kMinBlocks) gemm_f32_cpasync_kernel(const F32Args p)
{
    // OPT: the copy form (cache qualifiers, 0..3), or 4 for plain copies
    // with the accumulators starting from C (GEMM_OPT_ACCUMULATE).
    constexpr int CF = OPT & 3;
    constexpr bool ACC = (OPT & 4) != 0;
    static_assert(S >= 2 && S <= 6, "stages");
    extern __shared__ __align__(1024) float smem[];

    const int tid = threadIdx.x;
    int m0, n0;
    tile_origin(T::BM, T::BN, m0, n0);
    const int tr = tid / T::kThreadCols;
    const int tc = tid % T::kThreadCols;
    const int k_slices = (p.K + T::BK - 1) / T::BK;

    const CopyPolicies<CF> pol(p);
    auto issue = [&](int stage, int kt) {
        issue_slice_cpasync_f<T, CF>(smem + stage * T::kStageFloats, p, tid, m0, n0, kt, pol.a, pol.b);
    };

    Accum<T> acc;
    init_tile<T, ACC>(p, m0, n0, tr, tc, acc);

    // Prologue: slices 0 .. S-2 in flight, one group each.
#pragma unroll
    for (int st = 0; st < S - 1; ++st) {
        if (st < k_slices)
            issue(st, st);
        cp_async_commit();
    }

    for (int kt = 0; kt < k_slices; ++kt) {
        cp_async_wait<S - 2>(); // this thread's copies of slice kt have landed
        __syncthreads();        // ... and everyone's; slice kt-1 fully consumed
        const int fetch = kt + S - 1;
        const float *sA = smem + (kt % S) * T::kStageFloats;
        FragPipe<T, T::kBDistCpAsync> frag;
        frag.prime(sA, sA + T::kAFloats, tr, tc);
        // The refill of the stage slice kt-1 used is issued halfway through
        // slice kt's FMAs, where it takes otherwise idle issue slots, rather
        // than ahead of them (measured on GB300 at 4096^3, S = 4: 52.8 ->
        // 55.8 TFLOP/s).  The barrier above already covers the stage.
        frag.run_mid(sA, sA + T::kAFloats, tr, tc, acc, []() {}, []() -> const float * { return nullptr; }, [&]() {
            if (fetch < k_slices)
                issue(fetch % S, fetch);
            cp_async_commit();
        });
    }
    cp_async_wait<0>();

    store_tile<T>(p, m0, n0, tr, tc, acc);
}

template <class T, int S, int CF>
static int launch_cpasync_t(const F32Args &a, cudaStream_t s)
{
    const int smem = S * T::kStageBytes;
    static std::atomic<unsigned long long> limit_set[kMaxDevices];
    if (ensure_smem_limit(gemm_f32_cpasync_kernel<T, S, CF>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    const dim3 grid((a.N + T::BN - 1) / T::BN, (a.M + T::BM - 1) / T::BM);
    gemm_f32_cpasync_kernel<T, S, CF><<<grid, T::kThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

template <class T, int CF>
static int launch_cpasync_tile(const F32Args &a, cudaStream_t s)
{
    switch (a.stages) {
    case 2: return launch_cpasync_t<T, 2, CF>(a, s);
    case 3: return launch_cpasync_t<T, 3, CF>(a, s);
    case 4: return launch_cpasync_t<T, 4, CF>(a, s);
    case 5: return launch_cpasync_t<T, 5, CF>(a, s);
    case 6: return launch_cpasync_t<T, 6, CF>(a, s);
    default: return GEMM_ERR_INVALID_ARG;
    }
}

// The copy form (cache qualifiers) is a template parameter: the plain form's
// kernels carry no trace of the optional ones (a run-time choice inside the
// slice loop cost 2-3.5 % on GB300 at 4096^3).
template <int CF>
static int launch_cpasync_form(const F32Args &a, cudaStream_t s)
{
    if (a.tile == 32)
        return launch_cpasync_tile<TileXS, CF>(a, s);
    return a.tile == 128 ? launch_cpasync_tile<TileL, CF>(a, s) : launch_cpasync_tile<TileS, CF>(a, s);
}

int launch_f32_cpasync(const F32Args &a, cudaStream_t s)
{
    if (a.accumulate) // plain copies only: the planner refuses accumulate with cache qualifiers
        return launch_cpasync_form<4>(a, s);
    switch (a.copy_form) {
    case 0: return launch_cpasync_form<0>(a, s);
    case 1: return launch_cpasync_form<1>(a, s);
    case 2: return launch_cpasync_form<2>(a, s);
    default: return launch_cpasync_form<3>(a, s);
    }
}

} // namespace pg
