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
#include "f32_schedule.cuh"
#include "f32_tile.cuh"
#include "tma_ring.cuh"

namespace pg {

template <class T>
constexpr int tma_threads() { return T::kThreads + 32; }

template <class T, int S, bool ACC>
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
    // With a split of the last round (gemm_f32_ws), this launch covers the
    // whole-tile rounds only and the split-region kernel does the rest.
    if (static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x) >= p.tile_limit)
        return;
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
            // Optional L2 policies (.L2::cache_hint) on the loads.
            const bool hint = (p.copy_form & 2) != 0;
            const uint64_t pol_a = hint ? l2_policy(p.pol_a) : 0, pol_b = hint ? l2_policy(p.pol_b) : 0;
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
                tma_load_2d_opt(dst, &map_a, ring.full_bar(f), f * T::BK, m0, hint, pol_a);
                tma_load_2d_opt(dst + T::kAFloats * 4, &map_b, ring.full_bar(f), n0, f * T::BK, hint, pol_b);
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
    init_tile<T, ACC>(p, m0, n0, tr, tc, acc);

    auto stage_of = [&](int kt) { return stage0 + (kt % S) * T::kStageFloats; };
    auto wait_full = [&](int kt) {
        const bool ok = ring.consumer_wait(kt, p.wait_limit_ns);
        if (__all_sync(0xffffffffu, ok))
            return true;
        if (lane == 0)
            record_error(p.status, kErrFamilyF32Tma | kErrRoleConsumer);
        return false;
    };
    auto release = [&](int kt) {
        __syncwarp(); // every lane's reads of the stage precede the release
        if (lane == 0)
            ring.consumer_release(kt);
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
        chained = frag.run(sA, sA + T::kAFloats, tr, tc, acc, [&]() { release(kt); }, [&]() -> const float * {
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

// ---------------------------------------------------------------------------
// The split region of gemm_f32_ws (f32_schedule.cuh), 128 x 128 tile.  When
// the tile count is not a multiple of the CTA count, the one-tile kernel
// above runs the whole rounds but the last (tile_limit), and this kernel's
// a.ctas CTAs (one per SM) share the remaining ctas + (tiles mod ctas) tiles
// as equal runs of K slices: first the head of the tile the next CTA
// finishes, then whole tiles, then the tail of the tile the previous CTA
// started.  A tail continues from the FP32 accumulators its head handed over,
// so every element is the same FMA chain as in an unsplit tile.  The
// producer's ring runs on across pieces.
//
// Why two kernels: the K loop's speed turned out to hang on how the compiler
// schedules it, and inside a kernel that also carries the schedule and the
// hand-over it came out 4-8 % slower than in the one-tile kernel (GB300, one
// wave of 128 x 128 tiles; several code shapes measured).  This kernel only
// runs the last round or so.

// Consumers: wait until the previous CTA has raised its hand-over flag.  One
// thread polls the flag (bounded) and arrives on `received`; the others wait
// on `received` (bounded), so a warp that has already given up strands no
// one.  True when the accumulators may be read.  The polling thread, the
// flag's only reader, lowers it again once it has seen it: every flag a call
// raises is back at 0 when the call ends, so a call replayed with the same
// flag value (a captured CUDA graph) cannot mistake an old flag for a new
// one.
__device__ __noinline__ bool f32_handover_wait(unsigned long long *flag, unsigned long long epoch,
                                               uint64_t limit_ns, unsigned int *status, uint32_t received,
                                               volatile int *failed)
{
    const int lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        *failed = flag_wait_bounded(flag, epoch, limit_ns) ? 0 : 1;
        if (*failed)
            record_error(status, kErrFamilyF32Tma | kErrRoleHandover);
        else
            st_release_gpu_u64(flag, 0ull);
        mbar_arrive(received); // releases *failed to the other warps
    }
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(received, 0, limit_ns))) {
        if (lane == 0)
            record_error(status, kErrFamilyF32Tma | kErrRoleHandover);
        return false;
    }
    return *failed == 0;
}

// Consumers, after storing their accumulators to the hand-over slot: once
// every consumer warp's part is written, one thread raises the flag.
__device__ __noinline__ void f32_handover_publish(unsigned long long *flag, unsigned long long epoch,
                                                  uint64_t limit_ns, unsigned int *status, uint32_t written,
                                                  int withhold)
{
    __threadfence();
    __syncwarp();
    if (threadIdx.x % 32 == 0)
        mbar_arrive(written);
    if (threadIdx.x == 0) {
        if (mbar_wait_bounded(written, 0, limit_ns)) {
            __threadfence();
            if (!withhold) // test hook: the successor must give up
                st_release_gpu_u64(flag, epoch);
        } else {
            record_error(status, kErrFamilyF32Tma | kErrRoleHandover);
        }
    }
}

template <int S, bool ACC>
__global__ void __launch_bounds__(TileL::kThreads + 32, 1)
    gemm_f32_tma_persistent_kernel(const __grid_constant__ CUtensorMap map_a,
                                   const __grid_constant__ CUtensorMap map_b, const F32Args p)
{
    using T = TileL;
    static_assert(S >= 2 && S <= 6, "stages");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = align_smem(smem_u32(smem_raw), 1024);
    float *stage0 = reinterpret_cast<float *>(smem_raw + (base - smem_u32(smem_raw)));
    const uint32_t bars = base + S * T::kStageBytes;
    const TmaRing<S> ring{bars, bars + 8u * S};
    // Hand-over barriers (each used at most once per CTA): `written` counts
    // the consumer warps whose accumulators are in the hand-over slot;
    // `received` is arrived on once the previous CTA's flag has been seen
    // (or given up on).
    const uint32_t written = bars + 16u * S;
    const uint32_t received = written + 8u;
    volatile int *handover_failed = reinterpret_cast<volatile int *>(smem_raw + (received + 8u - smem_u32(smem_raw)));

    constexpr int kConsumerWarps = T::kThreads / 32;
    const int tid = threadIdx.x;
    const int warp = tid / 32;
    const int lane = tid % 32;
    const int tiles_n = (p.N + T::BN - 1) / T::BN;
    const int tiles_m = (p.M + T::BM - 1) / T::BM;
    const F32CtaPieces work = F32CtaPieces::make(
        F32Schedule::make(tiles_m * tiles_n, static_cast<int>(gridDim.x), (p.K + T::BK - 1) / T::BK, true),
        static_cast<int>(blockIdx.x));
    // This kernel's pieces, in order: head (if any), the region's whole
    // tiles, tail (if any).  The whole rounds before the region are the
    // one-tile kernel's.
    const int first = work.whole;
    const int pieces = work.count();
    if (tid == 0) {
        ring.init(kConsumerWarps);
        mbar_init(written, kConsumerWarps);
        mbar_init(received, 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            tma_prefetch_map(&map_a);
            tma_prefetch_map(&map_b);
            const bool hint = (p.copy_form & 2) != 0;
            const uint64_t pol_a = hint ? l2_policy(p.pol_a) : 0, pol_b = hint ? l2_policy(p.pol_b) : 0;
            unsigned f = 0;
            bool ok = true;
            for (int idx = first; ok && idx < pieces; ++idx) {
                const F32Piece pc = work.piece(idx);
                int m0, n0;
                tile_origin_linear(pc.tile, tiles_m, tiles_n, T::BM, T::BN, m0, n0);
                for (int ks = pc.s_begin; ks < pc.s_end; ++ks, ++f) {
                    if (static_cast<int>(f) == p.withhold)
                        continue; // test hook: this position is never filled
                    if (!ring.producer_acquire(f, p.wait_limit_ns)) {
                        record_error(p.status, kErrFamilyF32Tma | kErrRoleProducer);
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + (f % S) * T::kStageBytes;
                    ring.producer_commit(f, T::kStageBytes);
                    tma_load_2d_opt(dst, &map_a, ring.full_bar(f), ks * T::BK, m0, hint, pol_a);
                    tma_load_2d_opt(dst + T::kAFloats * 4, &map_b, ring.full_bar(f), n0, ks * T::BK, hint, pol_b);
                }
            }
            // As in the one-tile kernel: only the last S positions issued can
            // still be in flight, and each is waited for.
            bool drained = true;
            for (unsigned g = f > S ? f - S : 0; g < f; ++g)
                if (static_cast<int>(g) != p.withhold && !ring.consumer_wait(g, p.wait_limit_ns))
                    drained = false;
            if (!drained)
                record_error(p.status, kErrFamilyF32Tma | kErrRoleDrain);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int tr = tid / T::kThreadCols;
    const int tc = tid % T::kThreadCols;
    auto stage_of = [&](unsigned kt) { return stage0 + (kt % S) * T::kStageFloats; };
    auto wait_full = [&](unsigned kt) {
        const bool ok = ring.consumer_wait(kt, p.wait_limit_ns);
        if (__all_sync(0xffffffffu, ok))
            return true;
        if (lane == 0)
            record_error(p.status, kErrFamilyF32Tma | kErrRoleConsumer);
        return false;
    };
    auto release = [&](unsigned kt) {
        __syncwarp(); // every lane's reads of the stage precede the release
        if (lane == 0)
            ring.consumer_release(kt);
    };
    // Hand-over space: CTA c's accumulators at slot c, laid out so that each
    // of a warp's 16-byte accesses is 512 contiguous bytes; the ready flags
    // follow the slots.
    const int cta = static_cast<int>(blockIdx.x);
    ulonglong2 *slots = static_cast<ulonglong2 *>(p.handover);
    unsigned long long *flags =
        reinterpret_cast<unsigned long long *>(static_cast<uint8_t *>(p.handover) + gridDim.x * kF32HandoverTileBytes);

    unsigned f0 = 0; // ring position of the piece's first slice
    for (int idx = first; idx < pieces; ++idx) {
        const F32Piece pc = work.piece(idx);
        int m0, n0;
        tile_origin_linear(pc.tile, tiles_m, tiles_n, T::BM, T::BN, m0, n0);
        Accum<T> acc;
        if (pc.from_partial) {
            // The previous CTA computed this tile's first slices: continue
            // from its accumulators once its flag is up.
            if (!f32_handover_wait(flags + (cta - 1), p.epoch, p.wait_limit_ns, p.status, received, handover_failed))
                return;
            const ulonglong2 *src = slots + static_cast<long long>(cta - 1) * (T::kThreads * 16);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const ulonglong2 v = __ldcg(src + j * T::kThreads + tid);
                acc.pair[j / 2][2 * (j % 2)] = v.x;
                acc.pair[j / 2][2 * (j % 2) + 1] = v.y;
            }
        } else {
            init_tile<T, ACC>(p, m0, n0, tr, tc, acc);
        }
        const unsigned f_end = f0 + static_cast<unsigned>(pc.s_end - pc.s_begin);
        FragPipe<T> frag;
        bool chained = false; // slice kt's full barrier already waited and its k = 0 fragments loaded
        bool failed = false;
#pragma unroll 2
        for (unsigned kt = f0; kt < f_end; ++kt) {
            const float *sA = stage_of(kt);
            if (!chained) {
                if (!wait_full(kt))
                    return;
                frag.prime(sA, sA + T::kAFloats, tr, tc);
            }
            chained = frag.run(sA, sA + T::kAFloats, tr, tc, acc, [&]() { release(kt); }, [&]() -> const float * {
                if (kt + 1 >= f_end)
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
        f0 = f_end;
        if (pc.to_partial) {
            ulonglong2 *dst = slots + static_cast<long long>(cta) * (T::kThreads * 16);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                __stcg(dst + j * T::kThreads + tid,
                       make_ulonglong2(acc.pair[j / 2][2 * (j % 2)], acc.pair[j / 2][2 * (j % 2) + 1]));
            f32_handover_publish(flags + cta, p.epoch, p.wait_limit_ns, p.status, written, p.withhold_handover);
        } else {
            store_tile<T>(p, m0, n0, tr, tc, acc);
        }
    }
}

template <int S, bool ACC>
static int launch_tma_persistent_t(const F32Args &a, const CUtensorMap &map_a, const CUtensorMap &map_b,
                                   cudaStream_t s)
{
    const int smem = f32_smem_bytes(128, GEMM_FILL_TMA, S);
    static std::atomic<unsigned long long> limit_set[kMaxDevices];
    if (ensure_smem_limit(gemm_f32_tma_persistent_kernel<S, ACC>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    gemm_f32_tma_persistent_kernel<S, ACC><<<a.ctas, tma_threads<TileL>(), smem, s>>>(map_a, map_b, a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

template <class T, int S, bool ACC>
static int launch_tma_acc(const F32Args &a, cudaStream_t s)
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
    if (ensure_smem_limit(gemm_f32_tma_kernel<T, S, ACC>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    const dim3 grid((a.N + T::BN - 1) / T::BN, (a.M + T::BM - 1) / T::BM);
    if (a.tile_limit > 0) {
        gemm_f32_tma_kernel<T, S, ACC><<<grid, tma_threads<T>(), smem, s>>>(map_a, map_b, a);
        if (cudaGetLastError() != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    if constexpr (T::BM == 128) {
        if (a.ctas > 0) // the split region, after the whole rounds on the same stream
            return launch_tma_persistent_t<S, ACC>(a, map_a, map_b, s);
    }
    return GEMM_OK;
}

template <class T, int S>
static int launch_tma_t(const F32Args &a, cudaStream_t s)
{
    return a.accumulate ? launch_tma_acc<T, S, true>(a, s) : launch_tma_acc<T, S, false>(a, s);
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
