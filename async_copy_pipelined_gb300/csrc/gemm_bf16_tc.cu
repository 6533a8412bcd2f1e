// BF16 -> FP32 GEMM on the 5th-generation tensor cores, fed by the same ring
// of full/empty mbarriers as the FP32 TMA fill, with three ways to fill it.
//
// The pages' tensor-core loop ("异步拷贝与现代 Pipeline", section 6.1
// "BF16 GEMM 的异步拷贝": prefetch the next K tile, commit, compute the current
// tile on the tensor cores, wait, barrier) re-designed for sm_103a.  A CTA
// tile is MH x 128 rows by 256 columns (MH = 1 or 2):
//
//   warp 0      TMA producer: per 64-deep K block, one (MH x 128) x 64 box of
//               A and four 64 x 64 boxes of B (128-byte swizzle) into ring
//               stage f % S, announced on full[f % S].
//   next warp   allocates all 512 columns of tensor memory and, from one
//               thread, issues tcgen05.mma.cta_group::1.kind::f16 (M 128,
//               N 256, K 16; four per K block for each 128-row half, the
//               halves sharing each B slice); tcgen05.commit releases each
//               ring stage once its MMAs have read it, and marks the
//               accumulator full after a tile's last K block.
//   4 x MH warps  epilogue: tcgen05.ld of the finished accumulator (each warp
//               a 32-lane quarter of tensor memory for one half), then TMA
//               stores of 32 x 32 FP32 boxes through a swizzled per-warp
//               staging buffer, then hand the accumulator back.
//
// Tensor memory holds two 128 x 256 FP32 accumulators.  The 128-row tile uses
// them as a double buffer, so the epilogue of tile i overlaps the MMAs of
// tile i+1.  The 256-row tile uses both for one tile: each B slice then feeds
// two MMAs, so the fill writes a third fewer shared-memory bytes per
// multiply-add (the tensor core still reads B once per MMA, so its reads per
// multiply-add stay the same).  Shared-memory bandwidth, which the fill's
// writes and the tensor core's reads share, is what bounds the 128-row tile
// (measured on GB300 at 8192^3: the MMAs alone, with no loads after the
// first ring, run at 2140 TFLOP/s, the full kernel at 1667); the price is an
// epilogue that no longer overlaps the next tile's MMAs.
//
// The fills, as in the FP32 family ("Day 74: Async copies and pipelines", day
// 80's goal of this pipeline feeding tensor cores):
//   TMA       as above: one thread, one descriptor per box.
//   cp.async  eight producer warps copy 16-byte chunks straight into the
//             swizzled stage with cp.async, keep S-1 stages in flight per
//             thread (wait_group S-2), and mark a stage full once their own
//             copies of it have landed.  In an interior tile each thread's
//             chunks sit at the same stage offsets for every K block and
//             their sources advance by a fixed step, so the addresses are
//             computed once per tile and each copy is one unguarded
//             instruction.
//   sync      sixteen producer warps load chunks into registers (an interior
//             tile's chunks of a thread all at once) and store them into the
//             one and only stage; loads and MMAs strictly alternate.
// The cp.async and sync producers write the 128-byte-swizzled layout the TMA
// would write (16-byte chunk index XOR row mod 8 within each 1024-byte atom)
// through the generic proxy; each writer issues fence.proxy.async before its
// mbarrier arrive so the tensor core (async proxy) sees the data.  Every
// fill and both tiles issue the same MMAs in the same K order for every
// output element, so all of them give the same bits.
//
// Persistent: one CTA per SM walks tiles blockIdx.x, +gridDim.x, ... in
// groups of 4096 rows of tiles so the tiles in flight share A and B rows in
// L2.  Ragged M, N, K: TMA zero-fills out-of-range box elements (zeros add
// nothing to the products), the TMA stores clip at the matrix edge, and the
// plain-store epilogue (C not 16-byte aligned) guards each element.
//
// Layouts (PTX ISA shared-memory matrix descriptors, 128-byte swizzle):
//   A stage  MH x 128 rows (m) x 128 bytes (64 k), K-major; 8-row groups
//            1024 B apart (SBO); the K step of 16 elements advances 32 bytes;
//            half h starts 16 KiB in.
//   B stage  four 64(n) x 64(k) boxes, each 64 rows (k) of 128 bytes (64 n):
//            N-major ("MN-major"); 64-column atoms 8192 B apart (LBO), 8-row K
//            groups 1024 B apart (SBO); the K step advances 16 rows = 2048 B.
//   staging  per epilogue warp 32 rows x 128 bytes (32 FP32 columns), 16-byte
//            chunk index XOR row mod 8, as the C tensor map's 128-byte
//            swizzle expects.
#include <cstring>
#include <type_traits>

#include "f32_schedule.cuh"
#include "gemm_internal.h"
#include "ptx.cuh"
#include "tma_ring.cuh"

namespace pg {

namespace bf16 {
constexpr int BN = kBf16BlockN;
constexpr int BK = kBf16BlockK;
constexpr int kUmmaM = 128;
constexpr int kUmmaK = 16;
constexpr uint32_t kAHalfBytes = kUmmaM * BK * 2;          // 16 KiB: one 128-row half of A
constexpr uint32_t kBBoxCols = 64;                          // n per B box (128 bytes)
constexpr uint32_t kBBoxBytes = kBBoxCols * BK * 2;         // 8 KiB
constexpr uint32_t kBTileBytes = BN * BK * 2;               // 32 KiB
constexpr uint32_t kTmemCols = 512;                         // two 128 x 256 FP32 accumulators
// Rows of tiles per raster group.  Measured on GB300 at 8192^3 (256-row
// tile, ncu DRAM bytes per launch): 2048 rows 1112 MB, 4096 rows 1055 MB, at
// equal time; L2 eviction policies on A and B moved neither by more than 5 %.
constexpr int kGroupRows = 4096;
constexpr int kEpiBoxCols = 32;                             // FP32 columns per staged store
constexpr uint32_t kStagingBytes = 32 * kEpiBoxCols * 4;    // 4 KiB per epilogue warp

// Tile of MH 128-row halves.
template <int MH>
struct Tile {
    static_assert(MH == 1 || MH == 2, "one or two 128-row halves");
    static constexpr int BM = kUmmaM * MH;
    static constexpr uint32_t kATileBytes = kAHalfBytes * MH;
    static constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes; // 48 or 64 KiB
    static constexpr int kStageChunks = kStageBytes / 16;
    static constexpr int kAccBufs = 2 / MH;   // accumulators in flight
    static constexpr int kEpiWarps = 4 * MH;  // one per 32-lane quarter and half
    static constexpr int kGroupTiles = kGroupRows / BM;
};

// Producer warps per fill: the TMA fill needs one elected thread; the
// thread-issued fills spread a stage's chunks over many threads (GB300,
// 8192^3, 128-row tile, four stages: cp.async 833 TFLOP/s with sixteen warps
// recomputing every address, 1390 with sixteen and 1420 with eight
// precomputing them; the register path 236 with sixteen warps in batches of
// two loads, 438 with all six of a thread's loads in flight at once).
constexpr int kCpAsyncCopyWarps = 8;
constexpr int kSyncCopyWarps = 16;

template <int Fill>
constexpr int copy_warps()
{
    return Fill == GEMM_FILL_TMA ? 1 : Fill == GEMM_FILL_CPASYNC ? kCpAsyncCopyWarps : kSyncCopyWarps;
}

template <int Fill, int MH>
struct Roles {
    static constexpr int kProducerWarps = copy_warps<Fill>();
    static constexpr int kCopyThreads = kProducerWarps * 32;
    static constexpr int kMmaWarp = kProducerWarps;
    static constexpr int kEpiWarp0 = kMmaWarp + 1;
    static constexpr int kThreads = (kEpiWarp0 + Tile<MH>::kEpiWarps) * 32;
    static constexpr uint32_t kFullArrivals = Fill == GEMM_FILL_TMA ? 1u : static_cast<uint32_t>(kCopyThreads);
};

// Instruction descriptor, kind::f16: D = F32 (bits 4-5 = 1), A = BF16
// (bits 7-9 = 1), B = BF16 (bits 10-12 = 1), A K-major (bit 15 = 0), B
// MN-major (bit 16 = 1), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | (static_cast<uint32_t>(BN >> 3) << 17) |
                            (static_cast<uint32_t>(kUmmaM >> 4) << 24);

// Shared-memory matrix descriptor: start address >> 4 (bits 0-13), leading
// byte offset >> 4 (16-29), stride byte offset >> 4 (32-45), descriptor
// version 1 (46-47), base offset 0 (atoms are 1024-byte aligned), swizzle
// mode 2 = 128-byte (61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

template <int MH>
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int &mb, int &nb)
{
    constexpr int kGroup = Tile<MH>::kGroupTiles;
    const int per_group = kGroup * tiles_n;
    const int group = t / per_group;
    const int first_m = group * kGroup;
    const int gm = min(kGroup, tiles_m - first_m);
    const int r = t - group * per_group;
    mb = first_m + r % gm;
    nb = r / gm;
}

// 16-byte chunk q of the stage for tile (mb, nb), K block kb: chunks
// 0 .. 8 BM - 1 are the A box (row r = q/8 of BM, chunk c = q%8 of the
// 128-byte K row), the rest the four B boxes (box j, K row r of 64, chunk c
// of the 128-byte N row).  Gives the global element (row, col) of the
// chunk's first value, whether it is an A chunk, and its byte offset in the
// 128-byte-swizzled stage.
template <int MH>
__device__ __forceinline__ void stage_chunk(int q, int mb, int nb, int kb, int &grow, int &gcol, bool &is_a,
                                            uint32_t &dst)
{
    constexpr int BM = Tile<MH>::BM;
    if (q < BM * 8) {
        const int r = q >> 3, c = q & 7;
        is_a = true;
        grow = mb * BM + r;
        gcol = kb * BK + c * 8;
        dst = static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
    } else {
        q -= BM * 8;
        const int j = q >> 9, r = (q >> 3) & 63, c = q & 7;
        is_a = false;
        grow = kb * BK + r;
        gcol = nb * BN + j * static_cast<int>(kBBoxCols) + c * 8;
        dst = Tile<MH>::kATileBytes + static_cast<uint32_t>(j) * kBBoxBytes +
              static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
    }
}

// Eight consecutive bfloat16 (row, col..col+7) of an R x C row-major matrix,
// zero outside it; a full in-range chunk is one 16-byte load.
__device__ __forceinline__ uint4 load_chunk_bf16(const uint16_t *__restrict__ base, long long ld, int row, int col,
                                                 int R, int C)
{
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < R && col < C) {
        const uint16_t *src = base + static_cast<long long>(row) * ld + col;
        if (col + 8 <= C) {
            v = *reinterpret_cast<const uint4 *>(src);
        } else {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            for (int e = 0; e < 8 && col + e < C; ++e)
                w[e >> 1] |= static_cast<uint32_t>(src[e]) << (16 * (e & 1));
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    return v;
}
} // namespace bf16

template <int Fill, int S, int MH>
__global__ void __launch_bounds__(bf16::Roles<Fill, MH>::kThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                        const __grid_constant__ CUtensorMap map_c, const Bf16Args p)
{
    using namespace bf16;
    using R = Roles<Fill, MH>;
    using T = Tile<MH>;
    constexpr int BM = T::BM;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align_smem(raw, 1024);
    const uint32_t staging0 = base + S * T::kStageBytes; // kEpiWarps x 4 KiB, 1024-byte aligned
    const uint32_t bars = staging0 + T::kEpiWarps * kStagingBytes;
    const TmaRing<S> ring{bars, bars + 8u * S};
    const uint32_t tmem_full0 = bars + 16u * S;    // [kAccBufs]
    const uint32_t tmem_empty0 = tmem_full0 + 16u; // [kAccBufs]
    const uint32_t epi_done = tmem_empty0 + 16u;
    const uint32_t mma_done = epi_done + 8u;
    // K split (each used at most once per CTA): the epilogue warps have put
    // the previous CTA's accumulators into tensor memory / have written this
    // CTA's accumulators to the hand-over space.
    const uint32_t acc_loaded = mma_done + 8u;
    const uint32_t handover_written = acc_loaded + 8u;
    const uint32_t tmem_slot = handover_written + 8u;
    volatile uint32_t *tmem_slot_ptr = reinterpret_cast<volatile uint32_t *>(smem_raw + (tmem_slot - raw));

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int tiles_m = (p.M + BM - 1) / BM;
    const int tiles_n = (p.N + BN - 1) / BN;
    const int num_tiles = tiles_m * tiles_n;
    const int k_blocks = (p.K + BK - 1) / BK;
    // The pieces this CTA computes (f32_schedule.cuh): without a split, the
    // tiles blockIdx.x, + gridDim.x, ... whole; with one (TMA fill and
    // hand-over space), the whole rounds but the last, then its share of the
    // rest as head, whole tiles and tail.
    const bool split = Fill == GEMM_FILL_TMA && p.handover != nullptr;
    const F32CtaPieces work = F32CtaPieces::make(
        F32Schedule::make(num_tiles, static_cast<int>(gridDim.x), k_blocks, split), static_cast<int>(blockIdx.x));
    const int pieces = work.count();
    const int cta = static_cast<int>(blockIdx.x);
    constexpr int kHandoverQuads = BM * BN / 4; // 16-byte units of one CTA's hand-over slot
    uint4 *handover_slots = static_cast<uint4 *>(p.handover);
    unsigned long long *handover_flags = reinterpret_cast<unsigned long long *>(
        static_cast<uint8_t *>(p.handover) + static_cast<size_t>(gridDim.x) * kHandoverQuads * 16u);

    if (threadIdx.x == 0) {
        ring.init(1, R::kFullArrivals);
        for (int b = 0; b < T::kAccBufs; ++b) {
            mbar_init(tmem_full0 + 8u * b, 1);
            mbar_init(tmem_empty0 + 8u * b, T::kEpiWarps);
        }
        mbar_init(epi_done, T::kEpiWarps);
        mbar_init(mma_done, 1);
        mbar_init(acc_loaded, T::kEpiWarps);
        mbar_init(handover_written, T::kEpiWarps);
        fence_barrier_init();
    }
    if (warp == R::kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot_ptr;

    if (Fill == GEMM_FILL_TMA && warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_map(&map_a);
            tma_prefetch_map(&map_b);
            // Optional L2 policies (.L2::cache_hint) on the loads.
            const bool hint = (p.copy_form & 2) != 0;
            const uint64_t pol_a = hint ? l2_policy(p.pol_a) : 0, pol_b = hint ? l2_policy(p.pol_b) : 0;
            int f = 0;
            bool ok = true;
            for (int idx = 0; idx < pieces && ok; ++idx) {
                const F32Piece pc = work.piece(idx);
                int mb, nb;
                tile_coords<MH>(pc.tile, tiles_m, tiles_n, mb, nb);
                for (int kb = pc.s_begin; kb < pc.s_end; ++kb, ++f) {
                    if (f == p.withhold)
                        continue; // test hook: this position is never filled
                    if (!ring.producer_acquire(f, p.wait_limit_ns)) {
                        record_error(p.status, kErrFamilyBf16 | kErrRoleProducer);
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + static_cast<uint32_t>(f % S) * T::kStageBytes;
                    const uint32_t full = ring.full_bar(f);
                    ring.producer_commit(f, T::kStageBytes);
                    tma_load_2d_opt(dst, &map_a, full, kb * BK, mb * BM, hint, pol_a);
#pragma unroll
                    for (int j = 0; j < BN / static_cast<int>(kBBoxCols); ++j)
                        tma_load_2d_opt(dst + T::kATileBytes + j * kBBoxBytes, &map_b, full,
                                        nb * BN + j * static_cast<int>(kBBoxCols), kb * BK, hint, pol_b);
                }
            }
            // Only the last S positions issued can still be in flight; each
            // is waited for, with its own bound, even after another expired.
            bool drained = true;
            for (int g = f > S ? f - S : 0; g < f; ++g)
                if (g != p.withhold && !ring.consumer_wait(g, p.wait_limit_ns))
                    drained = false;
            if (!drained)
                record_error(p.status, kErrFamilyBf16 | kErrRoleDrain);
        }
    } else if (Fill != GEMM_FILL_TMA && warp < R::kProducerWarps) {
        // ------------------------------------------- cp.async / sync producers
        const int ptid = threadIdx.x;
        // Stages of copies each thread keeps in flight beyond the one it has
        // just issued: the full barrier of stage f is arrived on kLag stages
        // later, once this thread's copies of it have landed.  The producer
        // acquiring stage f needs stage f - S released, whose arrival came
        // at stage f - S + kLag, so kLag <= S - 1 cannot deadlock.
        constexpr int kLag = S >= 3 ? S - 2 : 1;
        int f = 0;
        bool ok = true;
        constexpr int kCopyThreads = R::kCopyThreads;
        constexpr int kStageChunks = T::kStageChunks;
        constexpr int kChunksPerThread = kStageChunks / kCopyThreads;
        static_assert(kStageChunks % kCopyThreads == 0, "whole chunks per thread");
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int mb, nb;
            tile_coords<MH>(t, tiles_m, tiles_n, mb, nb);
            // An interior tile's chunks: the same shared-memory offsets in
            // every stage, sources that advance by a fixed step per K block.
            const bool tile_interior = (mb + 1) * BM <= p.M && (nb + 1) * BN <= p.N;
            uint32_t c_off[kChunksPerThread];
            const uint16_t *c_src[kChunksPerThread];
            long long c_step[kChunksPerThread];
            if (tile_interior) {
#pragma unroll
                for (int i = 0; i < kChunksPerThread; ++i) {
                    int grow, gcol;
                    bool is_a;
                    stage_chunk<MH>(ptid + i * kCopyThreads, mb, nb, 0, grow, gcol, is_a, c_off[i]);
                    c_src[i] = is_a ? p.A + static_cast<long long>(grow) * p.lda + gcol
                                    : p.B + static_cast<long long>(grow) * p.ldb + gcol;
                    c_step[i] = is_a ? static_cast<long long>(BK) : static_cast<long long>(BK) * p.ldb;
                }
            }
            for (int kb = 0; kb < k_blocks; ++kb, ++f) {
                const bool free = ring.producer_acquire(f, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, free)) {
                    if (lane == 0)
                        record_error(p.status, kErrFamilyBf16 | kErrRoleProducer);
                    ok = false;
                    break;
                }
                const uint32_t dst = base + static_cast<uint32_t>(f % S) * T::kStageBytes;
                // Test hook: position p.withhold gets no copies and no
                // arrival, so whoever waits for it must give up.
                const bool fill_it = f != p.withhold;
                if constexpr (Fill == GEMM_FILL_CPASYNC) {
                    // One stage of copies in cache-qualifier form F (CopyForm
                    // in ptx.cuh; 0 is the plain copy).
                    auto copy_stage = [&](auto form) {
                        constexpr int F = decltype(form)::value;
                        const uint64_t pol_a = F & 2 ? l2_policy(p.pol_a) : 0;
                        const uint64_t pol_b = F & 2 ? l2_policy(p.pol_b) : 0;
                        if (tile_interior && (kb + 1) * BK <= p.K) {
                            // Every chunk is a whole in-range 16-byte copy (the
                            // planner requires 16-byte row pitches); chunks
                            // below BM * 8 belong to A.
                            if (fill_it) {
#pragma unroll
                                for (int i = 0; i < kChunksPerThread; ++i)
                                    cp_async_cg16_full_f<F>(dst + c_off[i], c_src[i],
                                                            i * kCopyThreads < BM * 8 ? pol_a : pol_b);
                            }
#pragma unroll
                            for (int i = 0; i < kChunksPerThread; ++i)
                                c_src[i] += c_step[i];
                        } else if (fill_it) {
                            for (int q = ptid; q < kStageChunks; q += kCopyThreads) {
                                int grow, gcol;
                                bool is_a;
                                uint32_t off;
                                stage_chunk<MH>(q, mb, nb, kb, grow, gcol, is_a, off);
                                const uint16_t *gbase = is_a ? p.A : p.B;
                                const long long ld = is_a ? p.lda : p.ldb;
                                const int rows = is_a ? p.M : p.K, cols = is_a ? p.K : p.N;
                                uint32_t nbytes = 0;
                                const uint16_t *src = gbase;
                                if (grow < rows && gcol < cols) {
                                    nbytes = static_cast<uint32_t>(min(cols - gcol, 8)) * 2u;
                                    src = gbase + static_cast<long long>(grow) * ld + gcol;
                                }
                                cp_async_cg16_f<F>(dst + off, src, nbytes, is_a ? pol_a : pol_b);
                            }
                        }
                    };
                    switch (p.copy_form) {
                    case 0: copy_stage(std::integral_constant<int, 0>{}); break;
                    case 1: copy_stage(std::integral_constant<int, 1>{}); break;
                    case 2: copy_stage(std::integral_constant<int, 2>{}); break;
                    default: copy_stage(std::integral_constant<int, 3>{}); break;
                    }
                    cp_async_commit();
                    if (f >= kLag) {
                        cp_async_wait<kLag>(); // this thread's copies of stage f - kLag have landed
                        fence_proxy_async_smem();
                        if (f - kLag != p.withhold)
                            mbar_arrive(ring.full_bar(f - kLag));
                    }
                } else if (tile_interior && (kb + 1) * BK <= p.K) {
                    // Interior: every chunk of this thread loaded at once, then stored.
                    if (fill_it) {
                        uint4 v[kChunksPerThread];
#pragma unroll
                        for (int i = 0; i < kChunksPerThread; ++i)
                            v[i] = *reinterpret_cast<const uint4 *>(c_src[i]);
#pragma unroll
                        for (int i = 0; i < kChunksPerThread; ++i)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst + c_off[i]),
                                         "r"(v[i].x), "r"(v[i].y), "r"(v[i].z), "r"(v[i].w)
                                         : "memory");
                        fence_proxy_async_smem();
                        mbar_arrive(ring.full_bar(f));
                    }
#pragma unroll
                    for (int i = 0; i < kChunksPerThread; ++i)
                        c_src[i] += c_step[i];
                } else if (fill_it) {
                    // Each batch keeps kBatch chunk loads per thread in flight;
                    // the batches tile the stage exactly (no chunk index past it).
                    constexpr int kBatch = 32 / R::kProducerWarps;
                    static_assert(kBatch >= 1 && kStageChunks % (kBatch * kCopyThreads) == 0,
                                  "batches tile the stage exactly");
                    for (int q0 = ptid; q0 < kStageChunks; q0 += kBatch * kCopyThreads) {
                        uint4 v[kBatch];
                        uint32_t off[kBatch];
#pragma unroll
                        for (int b = 0; b < kBatch; ++b) {
                            int grow, gcol;
                            bool is_a;
                            stage_chunk<MH>(q0 + b * kCopyThreads, mb, nb, kb, grow, gcol, is_a, off[b]);
                            v[b] = is_a ? load_chunk_bf16(p.A, p.lda, grow, gcol, p.M, p.K)
                                        : load_chunk_bf16(p.B, p.ldb, grow, gcol, p.K, p.N);
                        }
#pragma unroll
                        for (int b = 0; b < kBatch; ++b)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst + off[b]), "r"(v[b].x),
                                         "r"(v[b].y), "r"(v[b].z), "r"(v[b].w)
                                         : "memory");
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(ring.full_bar(f));
                }
            }
        }
        if constexpr (Fill == GEMM_FILL_CPASYNC) {
            cp_async_wait<0>();
            if (ok) {
                fence_proxy_async_smem();
                for (int g = f - kLag > 0 ? f - kLag : 0; g < f; ++g)
                    if (g != p.withhold)
                        mbar_arrive(ring.full_bar(g));
            }
        }
    } else if (warp == R::kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int f = 0;
            bool ok = true;
            for (int local = 0; local < pieces && ok; ++local) {
                const F32Piece pc = work.piece(local);
                const int slot = local % T::kAccBufs;
                const uint32_t use_parity = static_cast<uint32_t>((local / T::kAccBufs) & 1);
                if (!mbar_wait_bounded(tmem_empty0 + 8u * slot, use_parity ^ 1u, p.wait_limit_ns)) {
                    record_error(p.status, kErrFamilyBf16 | kErrRoleMma);
                    break;
                }
                // A tail continues from the accumulators the epilogue warps
                // have put into this slot.  Every epilogue warp has then seen
                // the previous CTA's flag, so it goes back to 0 (as in the
                // FP32 split: a replayed call cannot mistake it for new).
                if (pc.from_partial) {
                    if (!mbar_wait_bounded(acc_loaded, 0, p.wait_limit_ns)) {
                        record_error(p.status, kErrFamilyBf16 | kErrRoleHandover);
                        break;
                    }
                    st_release_gpu_u64(handover_flags + (cta - 1), 0ull);
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(slot * MH * BN);
                for (int kb = pc.s_begin; kb < pc.s_end; ++kb, ++f) {
                    if (!ring.consumer_wait(f, p.wait_limit_ns)) {
                        record_error(p.status, kErrFamilyBf16 | kErrRoleMma);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_addr = base + static_cast<uint32_t>(f % S) * T::kStageBytes;
                    const uint32_t b_addr = a_addr + T::kATileBytes;
#pragma unroll
                    for (int ks = 0; ks < BK / kUmmaK; ++ks) {
                        const uint64_t bdesc = smem_desc_sw128(b_addr + ks * kUmmaK * 128, kBBoxBytes, 1024);
#pragma unroll
                        for (int h = 0; h < MH; ++h) {
                            const uint64_t adesc = smem_desc_sw128(a_addr + h * kAHalfBytes + ks * kUmmaK * 2, 16, 1024);
                            mma_f16_ss(d_tmem + static_cast<uint32_t>(h * BN), adesc, bdesc, kIdesc,
                                       (pc.from_partial || kb != pc.s_begin || ks != 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(ring.empty_bar(f)); // stage free once these MMAs have read it
                }
                if (!ok)
                    break;
                mma_commit(tmem_full0 + 8u * slot); // accumulator complete
            }
            // Every MMA this thread issued must finish before tensor memory is freed.
            mma_commit(mma_done);
            if (!mbar_wait_bounded(mma_done, 0, p.wait_limit_ns))
                record_error(p.status, kErrFamilyBf16 | kErrRoleDrain);
        }
        __syncwarp();
        if (!mbar_wait_bounded(epi_done, 0, p.wait_limit_ns) && lane == 0)
            record_error(p.status, kErrFamilyBf16 | kErrRoleDrain);
        tc_fence_after_sync();
        __syncwarp();
        tmem_dealloc(tmem_base, kTmemCols);
    } else if (warp >= R::kEpiWarp0) {
        // ------------------------------------------------------- epilogue
        // Warp w reads tensor-memory lanes 32 (w % 4) .. +31 (the quarter
        // its warp index allows) of half h.
        const int quarter = warp & 3;
        const int half = (warp - R::kEpiWarp0) / 4;
        const int epi = warp - R::kEpiWarp0;
        const uint32_t staging = staging0 + static_cast<uint32_t>(epi) * kStagingBytes;
        // This warp's 32 rows x 256 columns of a hand-over slot, laid out so
        // that each warp-wide 16-byte access is 512 contiguous bytes.
        constexpr int kWarpQuads = 32 * BN / 4;
        for (int local = 0; local < pieces; ++local) {
            const F32Piece pc = work.piece(local);
            const int slot = local % T::kAccBufs;
            const uint32_t use_parity = static_cast<uint32_t>((local / T::kAccBufs) & 1);
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>((slot * MH + half) * BN);
            if (pc.from_partial) {
                // The slot is free (this warp drained its previous use); put
                // the previous CTA's accumulators there once its flag is up.
                const bool got = flag_wait_bounded(handover_flags + (cta - 1), p.epoch, p.wait_limit_ns);
                if (!__all_sync(0xffffffffu, got)) {
                    if (lane == 0)
                        record_error(p.status, kErrFamilyBf16 | kErrRoleHandover);
                    break;
                }
                const uint4 *src = handover_slots + static_cast<size_t>(cta - 1) * kHandoverQuads +
                                   static_cast<size_t>(epi) * kWarpQuads;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 v = __ldcg(src + (c * 8 + j) * 32 + lane);
                        r[4 * j] = v.x;
                        r[4 * j + 1] = v.y;
                        r[4 * j + 2] = v.z;
                        r[4 * j + 3] = v.w;
                    }
                    tmem_st_32x32b_x32(taddr + static_cast<uint32_t>(c * 32), r);
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(acc_loaded);
            }
            const bool ok = mbar_wait_bounded(tmem_full0 + 8u * slot, use_parity, p.wait_limit_ns);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0)
                    record_error(p.status, kErrFamilyBf16 | kErrRoleEpilogue);
                break;
            }
            tc_fence_after_sync();
            if (pc.to_partial) {
                // A head: the next CTA finishes this tile from these
                // accumulators.  All 256 columns and rows move, in or out of
                // the matrix.
                uint4 *dst = handover_slots + static_cast<size_t>(cta) * kHandoverQuads +
                             static_cast<size_t>(epi) * kWarpQuads;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c * 32), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        __stcg(dst + (c * 8 + j) * 32 + lane,
                               make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]));
                }
                __threadfence();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(handover_written);
                    mbar_arrive(tmem_empty0 + 8u * slot);
                }
                if (epi == 0 && lane == 0) {
                    // Every epilogue warp's part is written: raise the flag.
                    if (mbar_wait_bounded(handover_written, 0, p.wait_limit_ns)) {
                        __threadfence();
                        if (!p.withhold_handover) // test hook: the successor must give up
                            st_release_gpu_u64(handover_flags + cta, p.epoch);
                    } else {
                        record_error(p.status, kErrFamilyBf16 | kErrRoleHandover);
                    }
                }
                continue;
            }
            int mb, nb;
            tile_coords<MH>(pc.tile, tiles_m, tiles_n, mb, nb);
            const int row0 = mb * BM + half * kUmmaM + quarter * 32; // first row of this warp's box
            const int row = row0 + lane;
            float *crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll 1
            for (int c = 0; c < BN / kEpiBoxCols; ++c) {
                const int col0 = nb * BN + c * kEpiBoxCols;
                if (col0 >= p.N)
                    break; // warp-uniform
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c * kEpiBoxCols), r);
                tmem_ld_wait();
                if (row0 >= p.M)
                    continue; // warp-uniform: the whole box lies below the matrix
                if (p.c_tma) {
                    // The previous box's store must have read the staging
                    // buffer before it is overwritten.
                    if (lane == 0)
                        bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                                         staging + static_cast<uint32_t>(lane * 128 + ((j ^ (lane & 7)) << 4))),
                                     "r"(r[4 * j]), "r"(r[4 * j + 1]), "r"(r[4 * j + 2]), "r"(r[4 * j + 3])
                                     : "memory");
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&map_c, staging, col0, row0);
                        bulk_commit_group();
                    }
                } else if (row < p.M) {
                    // C is not 16-byte aligned or ldc not a multiple of 4
                    // (otherwise TMA stores write it): one guarded float each.
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + j < p.N)
                            crow[col0 + j] = __uint_as_float(r[j]);
                }
            }
            // The accumulator has been read (tcgen05.wait::ld above); the
            // stores still in flight read only the staging buffer.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(tmem_empty0 + 8u * slot);
        }
        if (lane == 0)
            bulk_wait_group<0>(); // every store of this warp has written C
        __syncwarp();
        if (lane == 0)
            mbar_arrive(epi_done);
    }
}

__global__ void gemm_bf16_zero_kernel(float *C, int M, int N, long long ldc)
{
    const long long total = static_cast<long long>(M) * N;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x)
        C[(idx / N) * ldc + idx % N] = 0.0f;
}

template <int Fill, int S, int MH>
static int launch_bf16_t(const Bf16Args &a, cudaStream_t s)
{
    using namespace bf16;
    using T = Tile<MH>;
    alignas(64) CUtensorMap map_a;
    alignas(64) CUtensorMap map_b;
    alignas(64) CUtensorMap map_c;
    if constexpr (Fill == GEMM_FILL_TMA) {
        int st = encode_tensor_map_2d(&map_a, 1, a.A, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M),
                                      static_cast<uint64_t>(a.lda) * 2u, BK, T::BM, 1);
        if (st != GEMM_OK)
            return st;
        st = encode_tensor_map_2d(&map_b, 1, a.B, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                                  static_cast<uint64_t>(a.ldb) * 2u, kBBoxCols, BK, 1);
        if (st != GEMM_OK)
            return st;
    } else {
        // The register and cp.async fills read A and B through plain pointers.
        std::memset(&map_a, 0, sizeof map_a);
        std::memset(&map_b, 0, sizeof map_b);
    }
    if (a.c_tma) {
        // C as FP32 rows, 32 x 32 boxes, 128-byte swizzle (the staging layout).
        const int st = encode_tensor_map_2d(&map_c, 0, a.C, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.M),
                                            static_cast<uint64_t>(a.ldc) * 4u, kEpiBoxCols, 32, 1);
        if (st != GEMM_OK)
            return st;
    } else {
        std::memset(&map_c, 0, sizeof map_c);
    }
    const int smem = bf16_smem_bytes(S, T::BM);
    static std::atomic<unsigned long long> limit_set[kMaxDevices];
    if (ensure_smem_limit(gemm_bf16_tc_kernel<Fill, S, MH>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    const long long tiles = static_cast<long long>((a.M + T::BM - 1) / T::BM) * ((a.N + BN - 1) / BN);
    const int grid = static_cast<int>(tiles < a.num_sms ? tiles : a.num_sms);
    gemm_bf16_tc_kernel<Fill, S, MH><<<grid, Roles<Fill, MH>::kThreads, smem, s>>>(map_a, map_b, map_c, a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

int bf16_threads(int fill, int block_m)
{
    using namespace bf16;
    if (block_m == 256) {
        if (fill == GEMM_FILL_TMA)
            return Roles<GEMM_FILL_TMA, 2>::kThreads;
        return fill == GEMM_FILL_CPASYNC ? Roles<GEMM_FILL_CPASYNC, 2>::kThreads : Roles<GEMM_FILL_SYNC, 2>::kThreads;
    }
    if (fill == GEMM_FILL_TMA)
        return Roles<GEMM_FILL_TMA, 1>::kThreads;
    return fill == GEMM_FILL_CPASYNC ? Roles<GEMM_FILL_CPASYNC, 1>::kThreads : Roles<GEMM_FILL_SYNC, 1>::kThreads;
}

template <int Fill, int MH>
static int launch_bf16_ring(const Bf16Args &a, cudaStream_t s)
{
    switch (a.stages) {
    case 2: return launch_bf16_t<Fill, 2, MH>(a, s);
    case 3: return launch_bf16_t<Fill, 3, MH>(a, s);
    case 4:
        if constexpr (MH == 1)
            return launch_bf16_t<Fill, 4, MH>(a, s);
        else
            return GEMM_ERR_INVALID_ARG; // four 64 KiB stages do not fit
    default: return GEMM_ERR_INVALID_ARG;
    }
}

int launch_bf16(const Bf16Args &a, int fill, cudaStream_t s)
{
    const bool tall = a.block_m == 256;
    if (fill == GEMM_FILL_SYNC) {
        if (a.stages != 1)
            return GEMM_ERR_INVALID_ARG;
        return tall ? launch_bf16_t<GEMM_FILL_SYNC, 1, 2>(a, s) : launch_bf16_t<GEMM_FILL_SYNC, 1, 1>(a, s);
    }
    if (fill == GEMM_FILL_CPASYNC)
        return tall ? launch_bf16_ring<GEMM_FILL_CPASYNC, 2>(a, s) : launch_bf16_ring<GEMM_FILL_CPASYNC, 1>(a, s);
    return tall ? launch_bf16_ring<GEMM_FILL_TMA, 2>(a, s) : launch_bf16_ring<GEMM_FILL_TMA, 1>(a, s);
}

int launch_bf16_zero(const Bf16Args &a, cudaStream_t s)
{
    const long long total = static_cast<long long>(a.M) * a.N;
    long long blocks = (total + 255) / 256;
    blocks = blocks > 4096 ? 4096 : (blocks < 1 ? 1 : blocks);
    gemm_bf16_zero_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a.C, a.M, a.N, a.ldc);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

} // namespace pg
