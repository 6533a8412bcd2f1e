// FP32 GEMM, fill (c): TMA bulk-tensor copies on an mbarrier ring with a
// dedicated producer warp.
//
// One elected thread of the producer warp walks the K slices: acquire the
// stage, announce the slice's bytes on its full barrier, and issue two 2-D
// tensor copies (the BM x 16 A box and the 16 x BN B box).  The 256 consumer
// threads wait on the full barrier, run the same inner product as the other
// fills, and release the stage with one arrival per warp.  No CTA-wide
// barrier sits in the main loop.  Out-of-range rows, columns and K elements
// of a box are filled with zeros by the copy engine itself, and the
// transaction count still covers the whole box.
//
// Sources: "A study on CUDA async memcpy", sections "mbarrier based
// approach" (phase, pending count, tx-count) and "block-scoped pipeline"
// (produced/consumed barriers per stage), and its remark on warp
// specialisation (dedicated producer warps); "Day 74: Async copies and
// pipelines" (TMA is the same pattern with one descriptor moving the tile).
//
// Every wait is bounded; on expiry the thread records GEMM_ERR_TIMEOUT in the
// status word and its warp returns.  The producer then waits (bounded) for
// its own copies still in flight before returning, so no copy lands in shared
// memory the CTA no longer owns.
#include "f32_tile.cuh"
#include "tma_ring.cuh"

namespace pg {

template <class T>
constexpr int tma_threads() { return T::kThreads + 32; }

template <class T, int S>
__global__ void __launch_bounds__(T::kThreads + 32, T::kMinBlocksTma)
    gemm_f32_tma_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const F32Args p)
{
    static_assert(S >= 2 && S <= 6, "stages");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = align_smem(smem_u32(smem_raw), 1024);
    float *stage0 = reinterpret_cast<float *>(smem_raw + (base - smem_u32(smem_raw)));
    const uint32_t bars = base + S * T::kStageBytes;
    const TmaRing<S> ring{bars, bars + 8u * S};

    constexpr int kConsumerWarps = T::kThreads / 32;
    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int lane = tid % 32;
    int m0, n0;
    tile_origin(T::BM, T::BN, m0, n0);
    const int k_slices = (p.K + T::BK - 1) / T::BK;

    if (tid == 0)
        ring.init(kConsumerWarps);
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_map(&map_a);
            tma_prefetch_map(&map_b);
            int f = 0;
            for (; f < k_slices; ++f) {
                if (f == p.withhold)
                    continue; // test hook: this position is never filled
                if (!ring.producer_acquire(f, p.wait_limit_ns)) {
                    record_error(p.status, kErrFamilyF32Tma | kErrRoleProducer);
                    break;
                }
                const uint32_t dst = base + static_cast<uint32_t>(f % S) * T::kStageBytes;
                ring.producer_commit(f, T::kStageBytes);
                tma_load_2d(dst, &map_a, ring.full_bar(f), f * T::BK, m0);
                tma_load_2d(dst + T::kAFloats * 4, &map_b, ring.full_bar(f), n0, f * T::BK);
            }
            // Copies still in flight must land before the CTA exits: only
            // the last S positions issued can still be in flight (issuing
            // position g + S waited for g's release, which followed its
            // landing).  Each is waited for, with its own bound, even after
            // another has expired.
            bool drained = true;
            for (int g = f > S ? f - S : 0; g < f; ++g)
                if (g != p.withhold && !ring.consumer_wait(g, p.wait_limit_ns))
                    drained = false;
            if (!drained)
                record_error(p.status, kErrFamilyF32Tma | kErrRoleDrain);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int tr = tid / T::kThreadCols;
    const int tc = tid % T::kThreadCols;
    Accum<T> acc;
    acc.zero();

    auto stage_of = [&](int kt) { return stage0 + (kt % S) * T::kStageFloats; };
    auto wait_full = [&](int kt) {
        const bool ok = ring.consumer_wait(kt, p.wait_limit_ns);
        if (__all_sync(0xffffffffu, ok))
            return true;
        if (lane == 0)
            record_error(p.status, kErrFamilyF32Tma | kErrRoleConsumer);
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

template <class T, int S>
static int launch_tma_t(const F32Args &a, cudaStream_t s)
{
    alignas(64) CUtensorMap map_a;
    alignas(64) CUtensorMap map_b;
    // A: K columns (innermost) x M rows, box 16 x BM.  B: N columns x K rows, box BN x 16.
    int st = encode_tensor_map_2d(&map_a, 0, a.A, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M),
                                  static_cast<uint64_t>(a.lda) * 4u, T::BK, T::BM, 0);
    if (st != GEMM_OK)
        return st;
    st = encode_tensor_map_2d(&map_b, 0, a.B, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                              static_cast<uint64_t>(a.ldb) * 4u, T::BN, T::BK, 0);
    if (st != GEMM_OK)
        return st;
    const int smem = f32_smem_bytes(T::BM, GEMM_FILL_TMA, S);
    static std::atomic<unsigned long long> limit_set[kMaxDevices];
    if (ensure_smem_limit(gemm_f32_tma_kernel<T, S>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    const dim3 grid((a.N + T::BN - 1) / T::BN, (a.M + T::BM - 1) / T::BM);
    gemm_f32_tma_kernel<T, S><<<grid, tma_threads<T>(), smem, s>>>(map_a, map_b, a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

template <class T>
static int launch_tma_tile(const F32Args &a, cudaStream_t s)
{
    switch (a.stages) {
    case 2: return launch_tma_t<T, 2>(a, s);
    case 3: return launch_tma_t<T, 3>(a, s);
    case 4: return launch_tma_t<T, 4>(a, s);
    case 5: return launch_tma_t<T, 5>(a, s);
    case 6: return launch_tma_t<T, 6>(a, s);
    default: return GEMM_ERR_INVALID_ARG;
    }
}

int launch_f32_tma(const F32Args &a, cudaStream_t s)
{
    if (a.tile == 32)
        return launch_tma_tile<TileXS>(a, s);
    return a.tile == 128 ? launch_tma_tile<TileL>(a, s) : launch_tma_tile<TileS>(a, s);
}

} // namespace pg
