// FP32 GEMM, fill (e): cp.async from dedicated producer warps on an mbarrier
// ring, the consumers those of the TMA fill.
//
// "A study on CUDA async memcpy" closes its block-scoped pipeline with the
// remark that producers and consumers need not be the same threads: a few
// warps can fill the stages while the rest only compute.  Here one or four
// producer warps (one for the 64x64 and 32x32 tiles, four for 128x128) issue
// every 16-byte cp.async of a slice, each thread then arranging with
// cp.async.mbarrier.arrive.noinc that the stage's full barrier (count: the
// producer threads) completes once its copies have landed.  The consumers
// wait on the full barrier, run the shared inner product and release the
// stage with one arrival per warp, exactly as with TMA.  The consumers thus
// spend no issue slots on copies or their addresses, which in the
// every-thread cp.async fills contend with the fragment loads and FMAs.
//
// Zero fill, chunk layout and the inner product are the cp.async fill's, so
// results are bit-identical to every other fill.  Every wait is bounded; a
// producer thread that gives up still waits for its own copies before it
// exits (cp.async.wait_all).
#include "f32_tile.cuh"
#include "tma_ring.cuh"

namespace pg {

// Producer threads: four warps on the 128x128 tile (GB300, 4096^3, TFLOP/s
// for 2 / 3 / 4 stages with one, two and four producer warps: 57.2 / 57.0 /
// 56.8, 57.9 / 56.5 / 55.5, 58.1 / 57.3 / 57.3; 3000 x 5000 x 1000 at two
// stages 42.3, 48.5, 49.4); one on the smaller tiles, whose three CTAs per
// SM leave no registers for more.
template <class T>
constexpr int ws_producer_threads() { return T::kThreads >= 256 && T::BM == 128 ? 128 : 32; }

template <class T>
constexpr int ws_threads() { return T::kThreads + ws_producer_threads<T>(); }

template <class T, int S, int OPT>
__global__ void __launch_bounds__(ws_threads<T>(), T::kMinBlocksTma) gemm_f32_cpasync_ws_kernel(const F32Args p)
{
    // OPT: the copy form (cache qualifiers, 0..3), or 4 for plain copies
    // with the accumulators starting from C (GEMM_OPT_ACCUMULATE).
    constexpr int CF = OPT & 3;
    constexpr bool ACC = (OPT & 4) != 0;
    static_assert(S >= 2 && S <= 6, "stages");
    constexpr int NP = ws_producer_threads<T>();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = align_smem(smem_u32(smem_raw), 1024);
    float *stage0 = reinterpret_cast<float *>(smem_raw + (base - smem_u32(smem_raw)));
    const uint32_t bars = base + S * T::kStageBytes;
    const TmaRing<S> ring{bars, bars + 8u * S};

    constexpr int kConsumerWarps = T::kThreads / 32;
    const int tid = threadIdx.x;
    const int lane = tid % 32;
    int m0, n0;
    tile_origin(T::BM, T::BN, m0, n0);
    const int k_slices = (p.K + T::BK - 1) / T::BK;

    if (tid == 0)
        ring.init(kConsumerWarps, NP);
    __syncthreads();

    if (tid >= T::kThreads) {
        // --------------------------------------------------------- producers
        const int ptid = tid - T::kThreads;
        const CopyPolicies<CF> pol(p);
        CpAsyncShare<T, NP> share;
        share.init(p, ptid, m0, n0);
        for (int f = 0; f < k_slices; ++f) {
            if (f == p.withhold)
                continue; // test hook: no copies and no arrival for this position
            const bool free = ring.producer_acquire(f, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, free)) {
                if (lane == 0)
                    record_error(p.status, kErrFamilyF32CpAsyncWs | kErrRoleProducer);
                break;
            }
            share.template issue<CF>(stage0 + (f % S) * T::kStageFloats, p, ptid, m0, n0, f, pol.a, pol.b);
            cp_async_mbar_arrive_noinc(ring.full_bar(f));
        }
        cp_async_wait_all(); // none of this thread's copies may land after it exits
        return;
    }

    // -------------------------------------------------------------- consumers
    const int tr = tid / T::kThreadCols;
    const int tc = tid % T::kThreadCols;
    Accum<T> acc;
    init_tile<T, ACC>(p, m0, n0, tr, tc, acc);

    auto stage_of = [&](int kt) { return stage0 + (kt % S) * T::kStageFloats; };
    auto wait_full = [&](int kt) {
        const bool ok = ring.consumer_wait(kt, p.wait_limit_ns);
        if (__all_sync(0xffffffffu, ok))
            return true;
        if (lane == 0)
            record_error(p.status, kErrFamilyF32CpAsyncWs | kErrRoleConsumer);
        return false;
    };
    FragPipe<T> frag;
    bool chained = false; // slice kt's full barrier already waited and its k = 0 fragments loaded
    bool failed = false;
    for (int kt = 0; kt < k_slices; ++kt) {
        const float *sA = stage_of(kt);
        if (!chained) {
            if (!wait_full(kt))
                return;
            frag.prime(sA, sA + T::kAFloats, tr, tc);
        }
        chained = frag.run(sA, sA + T::kAFloats, tr, tc, acc, [&]() {
            __syncwarp(); // every lane's reads of the stage precede the release
            if (lane == 0)
                ring.consumer_release(kt);
        }, [&]() -> const float * {
            if (!T::kChainSlices || kt + 1 >= k_slices)
                return nullptr;
            if (!wait_full(kt + 1)) {
                failed = true;
                return nullptr;
            }
            return stage_of(kt + 1);
        }) != nullptr;
        if (failed)
            return;
    }

    store_tile<T>(p, m0, n0, tr, tc, acc);
}

template <class T, int S, int CF>
static int launch_cpasync_ws_t(const F32Args &a, cudaStream_t s)
{
    const int smem = f32_smem_bytes(T::BM, GEMM_FILL_CPASYNC_WS, S);
    static std::atomic<unsigned long long> limit_set[kMaxDevices];
    if (ensure_smem_limit(gemm_f32_cpasync_ws_kernel<T, S, CF>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    const dim3 grid((a.N + T::BN - 1) / T::BN, (a.M + T::BM - 1) / T::BM);
    gemm_f32_cpasync_ws_kernel<T, S, CF><<<grid, ws_threads<T>(), smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

template <class T, int CF>
static int launch_cpasync_ws_tile(const F32Args &a, cudaStream_t s)
{
    switch (a.stages) {
    case 2: return launch_cpasync_ws_t<T, 2, CF>(a, s);
    case 3: return launch_cpasync_ws_t<T, 3, CF>(a, s);
    case 4: return launch_cpasync_ws_t<T, 4, CF>(a, s);
    case 5: return launch_cpasync_ws_t<T, 5, CF>(a, s);
    case 6: return launch_cpasync_ws_t<T, 6, CF>(a, s);
    default: return GEMM_ERR_INVALID_ARG;
    }
}

template <int CF>
static int launch_cpasync_ws_form(const F32Args &a, cudaStream_t s)
{
    if (a.tile == 32)
        return launch_cpasync_ws_tile<TileXS, CF>(a, s);
    return a.tile == 128 ? launch_cpasync_ws_tile<TileL, CF>(a, s) : launch_cpasync_ws_tile<TileS, CF>(a, s);
}

int launch_f32_cpasync_ws(const F32Args &a, cudaStream_t s)
{
    if (a.accumulate) // plain copies only: the planner refuses accumulate with cache qualifiers
        return launch_cpasync_ws_form<4>(a, s);
    switch (a.copy_form) {
    case 0: return launch_cpasync_ws_form<0>(a, s);
    case 1: return launch_cpasync_ws_form<1>(a, s);
    case 2: return launch_cpasync_ws_form<2>(a, s);
    default: return launch_cpasync_ws_form<3>(a, s);
    }
}

int f32_cpasync_ws_threads(int tile)
{
    return tile == 32 ? ws_threads<TileXS>() : tile == 128 ? ws_threads<TileL>() : ws_threads<TileS>();
}

} // namespace pg
