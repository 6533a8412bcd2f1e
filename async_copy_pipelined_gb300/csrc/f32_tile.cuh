// FP32 register-tiled GEMM: tile shapes, the shared-memory layout every fill
// writes, the per-thread micro-kernel every fill runs, the guarded chunk
// loaders and the epilogue.
//
// Design source: "pipelined_gemm.cu" (tile shapes, computeTile, the two
// fills) and "Day 74: Async copies and pipelines", section "Two kernels, one
// arithmetic": a block tile filled one 16-deep K slice at a time, a micro-tile
// of C per thread, and one shared inner product so that the fills execute
// identical floating-point operations in an identical order.
#pragma once

#include "gemm_internal.h"
#include "ptx.cuh"

namespace pg {

// Block tile BM x BN, K slice BK = 16, micro-tile TM x TN per thread.
//
// Shared-memory layout of one stage (identical for all fills):
//   A slice: BM rows x 16 floats, row-major [m][k] (64 bytes per row);
//   B slice: 16 rows x BN floats, row-major [k][n].
// Global chunk c (16 bytes) of either slice lands at float offset 4*c, so a
// warp's 32 chunks are 512 contiguous bytes: conflict-free 16-byte stores,
// and exactly the dense box a TMA copy writes.
//
// Thread (tr, tc) = (tid / (BN/TN), tid % (BN/TN)) owns rows tr + i*(BM/TM)
// and columns g*(BN/(TN/4)) + 4*tc + e.  With these strides a warp's A reads
// hit two adjacent rows (distinct banks, broadcast within each) and its B
// reads cover 256 contiguous bytes per 16-byte load: no bank conflicts.
template <int BM_, int BN_, int TM_, int TN_, int MIN_BLOCKS_, int MIN_BLOCKS_TMA_, bool CHAIN_>
struct F32Tile {
    static constexpr int BM = BM_, BN = BN_, BK = 16, TM = TM_, TN = TN_;
    // Resident CTAs per SM the register budget is sized for.  The 8x8
    // micro-tile with double-buffered fragments needs about 140 registers, so
    // the 128-tile kernels run one CTA (8 consumer warps) per SM; a second
    // CTA, or the TMA fill's producer warp in two CTAs, would not fit an SM
    // sub-partition's 16K registers.
    static constexpr int kMinBlocks = MIN_BLOCKS_;
    static constexpr int kMinBlocksTma = MIN_BLOCKS_TMA_;
    // Whether the TMA consumers chain slices (FragPipe).  Measured on GB300:
    // +1 to 4 % for the 128 tile at 4096^3; slower for the register-tight 64
    // tile and for the one-warp 32 tile of the latency-bound tall-K shape
    // (there a warp that waits early for slice kt+1 has nothing to hide it
    // behind), which therefore run slice by slice.
    static constexpr bool kChainSlices = CHAIN_;
    static constexpr int kThreadCols = BN / TN;
    static constexpr int kThreadRows = BM / TM;
    static constexpr int kThreads = kThreadCols * kThreadRows;
    // How many k ahead of its use the cp.async fills load a B fragment.  A
    // one-warp CTA has no other warp to cover a shared load's latency, its
    // warp also issues the copies, and the 8x4 tile's 16 paired FMAs per k
    // are too few to hide it: there B is loaded two k ahead (measured on
    // GB300, 32x32x65536, four stages: cp.async 1926 -> 1819 us, cp.async +
    // mbarrier 2477 -> 2420 us).  The TMA and register-path fills gain
    // nothing from it (TMA S2 / S4 unchanged, six stages slower), and a third
    // k ahead costs more registers than it hides.
    static constexpr int kBDistCpAsync = kThreads == 32 ? 2 : 1;
    static constexpr int kColGroups = TN / 4;
    static constexpr int kColGroupStride = BN / kColGroups;
    static constexpr int kAFloats = BM * BK;
    static constexpr int kBFloats = BK * BN;
    static constexpr int kStageFloats = kAFloats + kBFloats;
    static constexpr int kStageBytes = kStageFloats * 4;
    static constexpr int kAChunksPerThread = kAFloats / 4 / kThreads;
    static constexpr int kBChunksPerThread = kBFloats / 4 / kThreads;
    static constexpr int kBChunksPerRow = BN / 4;

    static_assert(kThreads % 32 == 0, "whole warps");
    static_assert(TN % 4 == 0 && BN % 4 == 0, "float4 columns");
    static_assert(kColGroupStride == 4 * kThreadCols, "column groups tile BN exactly");
    static_assert((kAFloats / 4) % kThreads == 0 && (kBFloats / 4) % kThreads == 0,
                  "each thread moves whole chunks of both slices");
};

// One warp, 32x32 tile, 8x4 micro-tile: the latency-bound shape of "A study
// on CUDA async memcpy", section "Real world example" (M = N = 32, long K,
// one block of one warp), where the fill rather than the FMAs sets the pace.
using TileXS = F32Tile<32, 32, 8, 4, 8, 8, false>;
using TileS = F32Tile<64, 64, 4, 4, 3, 3, false>;   // the lesson's 64x64x16, 4x4, 256 threads
using TileL = F32Tile<128, 128, 8, 8, 1, 1, true>; // 128x128x16, 8x8, 256 threads

// CTA -> tile.  CTAs are dispatched in linear order (x fastest); walking
// kGroupM tile rows down before stepping one tile column right keeps the
// tiles in flight on a few A row-blocks and B column-blocks at a time, so
// they are fetched from HBM about once and re-read from L2.  Only the
// assignment of tiles to CTAs changes, never a value.
constexpr int kGroupM = 16;

__device__ __forceinline__ void tile_origin(int bm, int bn, int &m0, int &n0)
{
    const int tiles_n = static_cast<int>(gridDim.x);
    const int tiles_m = static_cast<int>(gridDim.y);
    const int id = static_cast<int>(blockIdx.y) * tiles_n + static_cast<int>(blockIdx.x);
    const int per_group = kGroupM * tiles_n;
    const int group = id / per_group;
    const int first_m = group * kGroupM;
    const int gm = min(kGroupM, tiles_m - first_m);
    const int r = id - group * per_group;
    m0 = (first_m + r % gm) * bm;
    n0 = (r / gm) * bn;
}

// The same walk for a linear tile index t of a persistent kernel (tiles_m x
// tiles_n tiles): t takes the place of the CTA's linear block index.
__device__ __forceinline__ void tile_origin_linear(int t, int tiles_m, int tiles_n, int bm, int bn, int &m0, int &n0)
{
    const int per_group = kGroupM * tiles_n;
    const int group = t / per_group;
    const int first_m = group * kGroupM;
    const int gm = min(kGroupM, tiles_m - first_m);
    const int r = t - group * per_group;
    m0 = (first_m + r % gm) * bm;
    n0 = (r / gm) * bn;
}

// One thread's micro-tile of C, held as pairs of adjacent columns: pair p of
// row i is columns (2p, 2p+1) of the thread's TN columns, packed in one
// 64-bit register pair so a single fma.rn.f32x2 updates both.
template <class T>
struct Accum {
    unsigned long long pair[T::TM][T::TN / 2];

    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int i = 0; i < T::TM; ++i)
#pragma unroll
            for (int p = 0; p < T::TN / 2; ++p)
                pair[i][p] = 0ull; // both halves +0.0f
    }
};

__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack_f32x2(unsigned long long v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// d = a * b + d on both halves.  Each half is an independent, correctly
// rounded fma.rn.f32: the paired form halves the issue slots an FMA costs and
// changes no result bit.
__device__ __forceinline__ void fma_f32x2(unsigned long long &d, unsigned long long a, unsigned long long b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// A fragment: rows tr + i*(BM/TM), four consecutive k (one 16-byte load each).
template <class T>
__device__ __forceinline__ void load_a_frag(const float *__restrict__ sA, int tr, int kq, float4 (&a)[T::TM])
{
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
        a[i] = *reinterpret_cast<const float4 *>(sA + (tr + i * T::kThreadRows) * T::BK + kq * 4);
}

// B fragment of row k: the thread's TN columns as TN/2 column pairs.
template <class T>
__device__ __forceinline__ void load_b_frag(const float *__restrict__ sB, int tc, int k,
                                            unsigned long long (&b)[T::TN / 2])
{
#pragma unroll
    for (int g = 0; g < T::kColGroups; ++g) {
        const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(sB + k * T::BN + g * T::kColGroupStride + tc * 4);
        b[2 * g + 0] = v.x;
        b[2 * g + 1] = v.y;
    }
}

// The inner product all fills share ("pipelined_gemm.cu", computeTile):
// for each k of the slice, ascending, acc[i][j] = fma(a[i][k], b[k][j],
// acc[i][j]).  Each C element sees exactly one fused multiply-add per k, in
// ascending k, whichever fill staged the slice, so every fill gives the same
// bits.
//
// The fragment registers are double buffered: the B fragment of k+BDist
// (BDist + 1 buffers) and the A fragment of the next four k are loaded
// while the FMAs of k run, so shared-memory latency hides behind the paired
// FMAs of k.  They also live
// across slices: prime() loads the first k of a slice, and run() computes
// one slice.  At the start of its last k every shared-memory read of the
// slice has been issued, so run() calls `release` (the stage may be refilled)
// and then asks `next` for the following slice's stage (nullptr if there is
// none or it is not to be chained) and loads that slice's k = 0 fragments
// into the buffers k = 16 would use.  A consumer that waits for the next slice
// inside `next` thus overlaps the wait and the first shared loads of slice
// kt+1 with the FMAs of slice kt, without holding slice kt's stage.
template <class T, int BDist = 1>
struct FragPipe {
    static constexpr int kBBufs = BDist + 1;
    static_assert(!T::kChainSlices || BDist == 1, "a chained slice loads B one k ahead");
    float4 a[2][T::TM];
    unsigned long long b[kBBufs][T::TN / 2];

    __device__ __forceinline__ void prime(const float *__restrict__ sA, const float *__restrict__ sB, int tr, int tc)
    {
        load_a_frag<T>(sA, tr, 0, a[0]);
#pragma unroll
        for (int d = 0; d < BDist; ++d)
            load_b_frag<T>(sB, tc, d, b[d]);
    }

    template <class Release, class Next>
    __device__ __forceinline__ const float *run(const float *__restrict__ sA, const float *__restrict__ sB, int tr,
                                                int tc, Accum<T> &acc, Release &&release, Next &&next)
    {
        return run_mid(sA, sB, tr, tc, acc, release, next, []() {});
    }

    // As run(), and calls `mid` once, halfway through the slice (before the
    // FMAs of k = BK/2): a fill can issue its next copies there.
    template <class Release, class Next, class Mid>
    __device__ __forceinline__ const float *run_mid(const float *__restrict__ sA, const float *__restrict__ sB,
                                                    int tr, int tc, Accum<T> &acc, Release &&release, Next &&next,
                                                    Mid &&mid)
    {
        const float *nA = nullptr;
#pragma unroll
        for (int k = 0; k < T::BK; ++k) {
            const int ab = (k / 4) & 1;
            const int bb = k % kBBufs;
            if (k == T::BK / 2)
                mid();
            if ((k & 3) == 0 && k + 4 < T::BK)
                load_a_frag<T>(sA, tr, k / 4 + 1, a[ab ^ 1]);
            if (k + BDist < T::BK)
                load_b_frag<T>(sB, tc, k + BDist, b[(k + BDist) % kBBufs]);
            if (k + 1 == T::BK) {
                release();
                nA = next();
                if (nA) {
                    load_a_frag<T>(nA, tr, 0, a[ab ^ 1]);
                    load_b_frag<T>(nA + T::kAFloats, tc, 0, b[(k + 1) % kBBufs]);
                }
            }
#pragma unroll
            for (int i = 0; i < T::TM; ++i) {
                const int kk = k & 3;
                const float av = kk == 0 ? a[ab][i].x : kk == 1 ? a[ab][i].y : kk == 2 ? a[ab][i].z : a[ab][i].w;
                const unsigned long long aa = pack_f32x2(av, av);
#pragma unroll
                for (int q = 0; q < T::TN / 2; ++q)
                    fma_f32x2(acc.pair[i][q], aa, b[bb][q]);
            }
        }
        return nA;
    }
};

// One slice on its own (the sync and cp.async fills, whose CTA barrier sits
// between slices).
template <class T>
__device__ __forceinline__ void compute_tile(const float *__restrict__ sA, const float *__restrict__ sB, int tr,
                                             int tc, Accum<T> &acc)
{
    FragPipe<T> frag;
    frag.prime(sA, sB, tr, tc);
    frag.run(sA, sB, tr, tc, acc, []() {}, []() -> const float * { return nullptr; });
}

// Four consecutive elements (r, c..c+3) of an R x C row-major matrix with
// leading dimension ld, zero outside the matrix.  `vec` means the row pitch
// and base allow one 16-byte load.
__device__ __forceinline__ float4 load_chunk_guarded(const float *__restrict__ base, long long ld, int r, int c, int R,
                                                     int C, bool vec)
{
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < R && c < C) {
        const float *p = base + static_cast<long long>(r) * ld + c;
        if (vec && c + 4 <= C) {
            v = *reinterpret_cast<const float4 *>(p);
        } else {
            v.x = p[0];
            if (c + 1 < C)
                v.y = p[1];
            if (c + 2 < C)
                v.z = p[2];
            if (c + 3 < C)
                v.w = p[3];
        }
    }
    return v;
}

// The same four elements into shared memory at `dst` through cp.async.
// Aligned rows: one 16-byte cp.async.cg whose source size (0, 4, 8, 12 or 16
// bytes) zero-fills whatever lies outside the matrix.  Unaligned rows: four
// 4-byte cp.async.ca with source size 4 or 0.  A zero-size copy still names a
// valid address (the matrix base), never a skipped issue: a predicated-off
// cp.async would leave stale data instead of zeros ("cp.async", section
// "Predication is different from zero fill").
template <int Form>
__device__ __forceinline__ void cp_chunk_guarded(uint32_t dst, const float *__restrict__ base, long long ld, int r,
                                                 int c, int R, int C, bool vec, uint64_t pol)
{
    const bool row_ok = r < R;
    if (vec) {
        uint32_t nbytes = 0;
        const float *src = base;
        if (row_ok && c < C) {
            nbytes = static_cast<uint32_t>(min(C - c, 4)) * 4u;
            src = base + static_cast<long long>(r) * ld + c;
        }
        cp_async_cg16_f<Form>(dst, src, nbytes, pol);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool ok = row_ok && (c + e) < C;
            const float *src = ok ? base + static_cast<long long>(r) * ld + c + e : base;
            cp_async_ca4_f<Form & 1>(dst + 4u * e, src, ok ? 4u : 0u);
        }
    }
}

// Chunk c of the A slice: row c/4, k offset 4*(c%4).  Of the B slice: row
// c/(BN/4), n offset 4*(c%(BN/4)).  Both land at float offset 4*c.
template <class T>
__device__ __forceinline__ void a_chunk_coords(int c, int m0, int k0, int &r, int &k)
{
    r = m0 + c / 4;
    k = k0 + (c % 4) * 4;
}

template <class T>
__device__ __forceinline__ void b_chunk_coords(int c, int k0, int n0, int &k, int &n)
{
    k = k0 + c / T::kBChunksPerRow;
    n = n0 + (c % T::kBChunksPerRow) * 4;
}

// Issue this thread's cp.async copies of slice kt into the stage at `stage`
// (A slice then B slice).  Completion is tracked by the caller: a commit
// group (cp.async fill) or an mbarrier arrive (mbarrier-completed fill).
// `Form` selects the optional cache qualifiers (ptx.cuh, CopyForm) with the
// L2 policies `pol_a`, `pol_b`; Form 0 is the plain copy.
template <class T, int Form>
__device__ __forceinline__ void issue_slice_cpasync_f(float *stage, const F32Args &p, int tid, int m0, int n0, int kt,
                                                      uint64_t pol_a, uint64_t pol_b)
{
    float *sA = stage;
    float *sB = stage + T::kAFloats;
    const int k0 = kt * T::BK;
    if (p.a_vec && p.b_vec && m0 + T::BM <= p.M && n0 + T::BN <= p.N && k0 + T::BK <= p.K) {
        // Interior slice with 16-byte rows: every chunk is a whole in-range
        // 16-byte copy, so no guard and no source size are needed.
#pragma unroll
        for (int q = 0; q < T::kAChunksPerThread; ++q) {
            const int c = tid + q * T::kThreads;
            int r, k;
            a_chunk_coords<T>(c, m0, k0, r, k);
            cp_async_cg16_full_f<Form>(smem_u32(sA + 4 * c), p.A + static_cast<long long>(r) * p.lda + k, pol_a);
        }
#pragma unroll
        for (int q = 0; q < T::kBChunksPerThread; ++q) {
            const int c = tid + q * T::kThreads;
            int k, n;
            b_chunk_coords<T>(c, k0, n0, k, n);
            cp_async_cg16_full_f<Form>(smem_u32(sB + 4 * c), p.B + static_cast<long long>(k) * p.ldb + n, pol_b);
        }
        return;
    }
#pragma unroll
    for (int q = 0; q < T::kAChunksPerThread; ++q) {
        const int c = tid + q * T::kThreads;
        int r, k;
        a_chunk_coords<T>(c, m0, k0, r, k);
        cp_chunk_guarded<Form>(smem_u32(sA + 4 * c), p.A, p.lda, r, k, p.M, p.K, p.a_vec, pol_a);
    }
#pragma unroll
    for (int q = 0; q < T::kBChunksPerThread; ++q) {
        const int c = tid + q * T::kThreads;
        int k, n;
        b_chunk_coords<T>(c, k0, n0, k, n);
        cp_chunk_guarded<Form>(smem_u32(sB + 4 * c), p.B, p.ldb, k, n, p.K, p.N, p.b_vec, pol_b);
    }
}

// A group of NP producer threads (thread ptid of them) copying their share
// of a slice: the copies of issue_slice_cpasync_f, dealt over NP threads
// instead of all of the tile's threads.  For an interior tile with 16-byte
// rows, each thread's chunk addresses are worked out once per tile
// (CpAsyncShare::init) and stepped per slice; other tiles and the K tail take
// the guarded copies.
template <class T, int NP>
struct CpAsyncShare {
    static constexpr int kA = T::kAFloats / 4 / NP; // A chunks per producer thread
    static constexpr int kB = T::kBFloats / 4 / NP; // B chunks per producer thread
    static_assert(kA * NP * 4 == T::kAFloats && kB * NP * 4 == T::kBFloats, "whole chunks per producer thread");
    const float *src_a[kA];
    const float *src_b[kB];
    bool interior;

    __device__ __forceinline__ void init(const F32Args &p, int ptid, int m0, int n0)
    {
        interior = p.a_vec && p.b_vec && m0 + T::BM <= p.M && n0 + T::BN <= p.N;
#pragma unroll
        for (int q = 0; q < kA; ++q) {
            int r, k;
            a_chunk_coords<T>(ptid + q * NP, m0, 0, r, k);
            src_a[q] = p.A + static_cast<long long>(r) * p.lda + k;
        }
#pragma unroll
        for (int q = 0; q < kB; ++q) {
            int k, n;
            b_chunk_coords<T>(ptid + q * NP, 0, n0, k, n);
            src_b[q] = p.B + static_cast<long long>(k) * p.ldb + n;
        }
    }

    // Copies of slice kt into `stage`; the sources then step one slice on.
    template <int Form>
    __device__ __forceinline__ void issue(float *stage, const F32Args &p, int ptid, int m0, int n0, int kt,
                                          uint64_t pol_a, uint64_t pol_b)
    {
        float *sA = stage;
        float *sB = stage + T::kAFloats;
        const int k0 = kt * T::BK;
        if (interior && k0 + T::BK <= p.K) {
#pragma unroll
            for (int q = 0; q < kA; ++q)
                cp_async_cg16_full_f<Form>(smem_u32(sA + 4 * (ptid + q * NP)), src_a[q] + k0, pol_a);
#pragma unroll
            for (int q = 0; q < kB; ++q)
                cp_async_cg16_full_f<Form>(smem_u32(sB + 4 * (ptid + q * NP)),
                                           src_b[q] + static_cast<long long>(k0) * p.ldb, pol_b);
            return;
        }
#pragma unroll
        for (int q = 0; q < kA; ++q) {
            const int c = ptid + q * NP;
            int r, k;
            a_chunk_coords<T>(c, m0, k0, r, k);
            cp_chunk_guarded<Form>(smem_u32(sA + 4 * c), p.A, p.lda, r, k, p.M, p.K, p.a_vec, pol_a);
        }
#pragma unroll
        for (int q = 0; q < kB; ++q) {
            const int c = ptid + q * NP;
            int k, n;
            b_chunk_coords<T>(c, k0, n0, k, n);
            cp_chunk_guarded<Form>(smem_u32(sB + 4 * c), p.B, p.ldb, k, n, p.K, p.N, p.b_vec, pol_b);
        }
    }
};

// The L2 policies a kernel of copy form CF hands to its copies: built once
// per thread, and only by the forms that carry a cache hint.
template <int CF>
struct CopyPolicies {
    uint64_t a = 0, b = 0;
    __device__ __forceinline__ explicit CopyPolicies(const F32Args &p)
    {
        if constexpr ((CF & 2) != 0) {
            a = l2_policy(p.pol_a);
            b = l2_policy(p.pol_b);
        }
    }
};

// Write the micro-tile; rows >= M and columns >= N are skipped.
// The accumulators a tile starts from: +0, or with ACC (GEMM_OPT_ACCUMULATE)
// the values C holds, so that each element's FMA chain continues from C.
// Loads follow store_tile's layout and guards; elements outside C stay +0
// and are never stored.  ACC is a template parameter so that the kernels
// without it compile exactly as before (a run-time flag here moved the K
// loop's scheduling and cost 2 % at 4096^3).
template <class T, bool ACC>
__device__ __forceinline__ void init_tile(const F32Args &p, int m0, int n0, int tr, int tc, Accum<T> &acc)
{
    acc.zero();
    if constexpr (!ACC)
        return;
#pragma unroll
    for (int i = 0; i < T::TM; ++i) {
        const int row = m0 + tr + i * T::kThreadRows;
        if (row >= p.M)
            continue;
        const float *crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll
        for (int g = 0; g < T::kColGroups; ++g) {
            const int col = n0 + g * T::kColGroupStride + tc * 4;
            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (p.c_vec && col + 4 <= p.N) {
                const float4 c4 = *reinterpret_cast<const float4 *>(crow + col);
                v[0] = c4.x;
                v[1] = c4.y;
                v[2] = c4.z;
                v[3] = c4.w;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < p.N)
                        v[e] = crow[col + e];
            }
            acc.pair[i][2 * g] = pack_f32x2(v[0], v[1]);
            acc.pair[i][2 * g + 1] = pack_f32x2(v[2], v[3]);
        }
    }
}

template <class T>
__device__ __forceinline__ void store_tile(const F32Args &p, int m0, int n0, int tr, int tc, const Accum<T> &acc)
{
#pragma unroll
    for (int i = 0; i < T::TM; ++i) {
        const int row = m0 + tr + i * T::kThreadRows;
        if (row >= p.M)
            continue;
        float *crow = p.C + static_cast<long long>(row) * p.ldc;
#pragma unroll
        for (int g = 0; g < T::kColGroups; ++g) {
            const int col = n0 + g * T::kColGroupStride + tc * 4;
            float v[4];
            unpack_f32x2(acc.pair[i][2 * g], v[0], v[1]);
            unpack_f32x2(acc.pair[i][2 * g + 1], v[2], v[3]);
            if (p.c_vec && col + 4 <= p.N) {
                *reinterpret_cast<float4 *>(crow + col) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (col + e < p.N)
                        crow[col + e] = v[e];
            }
        }
    }
}

} // namespace pg
