// FP32 GEMM, TMA fill, wide rows: 128 x 256 tiles, an 8 x 16 micro-tile per
// thread, and no producer warp.
//
// The arithmetic is the shared inner product of every fill ("pipelined_gemm.cu",
// computeTile): each C element is one fma.rn chain over k ascending from +0 (or
// from C with GEMM_OPT_ACCUMULATE), so the results are bit-identical to the
// 128 x 128 kernels and to the oracle's FMA chain.  Only the block shape and
// who issues the copies change:
//
//  * Eight consumer warps, each thread owning 8 rows x 16 columns of C
//    (columns in four groups of four, 64 apart, so a warp's 16-byte B loads
//    cover 256 contiguous bytes).  Per k a thread issues 64 paired FMAs
//    against 8 scalar A values (loaded as pairs, one LDS.64 per row per two
//    k) and four 16-byte B loads: half the shared-memory loads per FMA of the
//    8 x 8 micro-tile.
//  * That needs about 210 registers a thread.  A ninth (producer) warp would
//    put three warps on one SM sub-partition and cap every thread at 168
//    registers, so the copies are issued by consumer thread 0 instead: the
//    first S slices up front, then, halfway through slice kt, slice kt-1+S
//    into the stage slice kt-1 used (released by every warp at the start of
//    its last k, so the wait for it is normally already over).
//  * The ring, the chained wait for slice kt+1 during slice kt's last k's,
//    the per-warp stage release and the bounded waits are those of the
//    128 x 128 TMA kernel.
//
// Measured on GB300 (probe of this kernel, TFLOP/s, bits equal): one round
// of 152 tiles, 2432 x 2048 x 4096, 64.9 against 61.8 for the 128 x 128 TMA
// kernel's two rounds; x 16384 K 65.5 against 62.9; two / three / four /
// five / six stages 62.7 / 64.5 / 64.9 / 64.5 / 64.3; A as one LDS.32 per
// row per k instead of pairs 63.3.  At 4096^3 the call (wide rows 0-2431,
// then the 128 x 128 path) ran 62.1 against 61.2.
//
// A tile twice as wide makes half as many tiles, so whole rounds are rarer:
// f32_wide_rows() gives the kernel the top rows of a call only where that
// shortens the call, and the 128 x 128 path (with its K split of the last
// round) computes the rest.
#include <numeric>

#include "f32_schedule.cuh"
#include "f32_tile.cuh"
#include "tma_ring.cuh"

namespace pg {

using TileW = F32Tile<128, 256, 8, 16, 1, 1, true>;

template <bool ACC>
__global__ void __launch_bounds__(TileW::kThreads, 1)
    gemm_f32_tma_wide_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                             const F32Args p)
{
    using T = TileW;
    constexpr int S = kF32WideStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = align_smem(smem_u32(smem_raw), 1024);
    float *stage0 = reinterpret_cast<float *>(smem_raw + (base - smem_u32(smem_raw)));
    const uint32_t bars = base + S * T::kStageBytes;
    const TmaRing<S> ring{bars, bars + 8u * S};

    const int tid = threadIdx.x;
    const int lane = tid % 32;
    int m0, n0;
    tile_origin(T::BM, T::BN, m0, n0);
    const int k_slices = (p.K + T::BK - 1) / T::BK;

    if (tid == 0) {
        ring.init(T::kThreads / 32);
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
    }
    __syncthreads();

    // Copies (thread 0 only): ring position f holds K slice f.
    int issued = 0;       // positions issued so far
    bool issuing = true;  // false once a wait for a free stage gave up
    auto issue = [&](int f) {
        if (f == p.withhold)
            return; // test hook: this position is never filled
        const uint32_t dst = base + static_cast<uint32_t>(f % S) * T::kStageBytes;
        ring.producer_commit(f, T::kStageBytes);
        tma_load_2d(dst, &map_a, ring.full_bar(f), f * T::BK, m0);
        tma_load_2d(dst + T::kAFloats * 4, &map_b, ring.full_bar(f), n0, f * T::BK);
    };
    if (tid == 0)
        for (; issued < S && issued < k_slices; ++issued)
            issue(issued);

    const int tr = tid / T::kThreadCols;
    const int tc = tid % T::kThreadCols;
    Accum<T> acc;
    init_tile<T, ACC>(p, m0, n0, tr, tc, acc);

    auto wait_full = [&](int kt) {
        const bool ok = ring.consumer_wait(kt, p.wait_limit_ns);
        if (__all_sync(0xffffffffu, ok))
            return true;
        if (lane == 0)
            record_error(p.status, kErrFamilyF32TmaWide | kErrRoleConsumer);
        return false;
    };
    // A as pairs of consecutive k (rows tr + 16 i), B as the thread's 16
    // columns (8 pairs) of one k; both double buffered.
    float2 a[2][T::TM];
    unsigned long long b[2][T::TN / 2];
    auto load_a2 = [&](const float *sA, int k, float2 (&dst)[T::TM]) {
#pragma unroll
        for (int i = 0; i < T::TM; ++i)
            dst[i] = *reinterpret_cast<const float2 *>(sA + (tr + i * T::kThreadRows) * T::BK + k);
    };

    bool ok = wait_full(0);
    if (ok) {
        load_a2(stage0, 0, a[0]);
        load_b_frag<T>(stage0 + T::kAFloats, tc, 0, b[0]);
    }
    for (int kt = 0; ok && kt < k_slices; ++kt) {
        const float *sA = stage0 + (kt % S) * T::kStageFloats;
        const float *sB = sA + T::kAFloats;
        const bool has_next = kt + 1 < k_slices;
        const float *nA = stage0 + ((kt + 1) % S) * T::kStageFloats;
#pragma unroll
        for (int k = 0; k < T::BK; ++k) {
            const int ab = (k / 2) & 1;
            const int bb = k & 1;
            if (k == T::BK / 2 && tid == 0 && issuing && issued < k_slices && issued == kt - 1 + S) {
                // Slice kt-1's stage, released by every warp during its last k.
                if (ring.producer_acquire(issued, p.wait_limit_ns)) {
                    issue(issued);
                    ++issued;
                } else {
                    record_error(p.status, kErrFamilyF32TmaWide | kErrRoleProducer);
                    issuing = false;
                }
            }
            if (k == T::BK - 2 && has_next && !wait_full(kt + 1))
                ok = false; // this slice's FMAs finish on registers already loaded; no further loads
            if ((k & 1) == 0) {
                if (k + 2 < T::BK)
                    load_a2(sA, k + 2, a[ab ^ 1]);
                else if (has_next && ok)
                    load_a2(nA, 0, a[ab ^ 1]);
            }
            if (k + 1 < T::BK)
                load_b_frag<T>(sB, tc, k + 1, b[bb ^ 1]);
            else if (has_next && ok)
                load_b_frag<T>(nA + T::kAFloats, tc, 0, b[bb ^ 1]);
            if (k == T::BK - 1) {
                __syncwarp(); // every lane's reads of the stage precede the release
                if (lane == 0)
                    ring.consumer_release(kt);
            }
#pragma unroll
            for (int i = 0; i < T::TM; ++i) {
                const float av = (k & 1) ? a[ab][i].y : a[ab][i].x;
                const unsigned long long aa = pack_f32x2(av, av);
#pragma unroll
                for (int q = 0; q < T::TN / 2; ++q)
                    fma_f32x2(acc.pair[i][q], aa, b[bb][q]);
            }
        }
    }

    if (tid == 0) {
        // Only the last S positions issued can still be in flight (issuing
        // position g + S waited for g's release, which followed its landing);
        // each is waited for, with its own bound, before the CTA may exit.
        bool drained = true;
        for (int g = issued > S ? issued - S : 0; g < issued; ++g)
            if (g != p.withhold && !ring.consumer_wait(g, p.wait_limit_ns))
                drained = false;
        if (!drained)
            record_error(p.status, kErrFamilyF32TmaWide | kErrRoleDrain);
    }
    if (ok)
        store_tile<T>(p, m0, n0, tr, tc, acc);
}

int f32_wide_smem_bytes()
{
    return kF32WideStages * TileW::kStageBytes + 1024 /* alignment slack */ + 16 * kF32WideStages /* barriers */;
}

template <bool ACC>
static int launch_wide_t(const F32Args &a, cudaStream_t s)
{
    using T = TileW;
    alignas(64) CUtensorMap map_a;
    alignas(64) CUtensorMap map_b;
    // A: K columns x M rows, box 16 x 128.  B: N columns x K rows, box 256 x 16.
    int st = encode_tensor_map_2d(&map_a, 0, a.A, static_cast<uint64_t>(a.K), static_cast<uint64_t>(a.M),
                                  static_cast<uint64_t>(a.lda) * 4u, T::BK, T::BM, 0);
    if (st != GEMM_OK)
        return st;
    st = encode_tensor_map_2d(&map_b, 0, a.B, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K),
                              static_cast<uint64_t>(a.ldb) * 4u, T::BN, T::BK, 0);
    if (st != GEMM_OK)
        return st;
    const int smem = f32_wide_smem_bytes();
    static std::atomic<unsigned long long> limit_set[kMaxDevices];
    if (ensure_smem_limit(gemm_f32_tma_wide_kernel<ACC>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    const dim3 grid((a.N + T::BN - 1) / T::BN, (a.M + T::BM - 1) / T::BM);
    gemm_f32_tma_wide_kernel<ACC><<<grid, T::kThreads, smem, s>>>(map_a, map_b, a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

int launch_f32_tma_wide(const F32Args &a, cudaStream_t s)
{
    return a.accumulate ? launch_wide_t<true>(a, s) : launch_wide_t<false>(a, s);
}

// Cost of a call in rounds of 152 one-tile 128 x 128 CTAs, measured on GB300
// at K = 4096 and 16384: a round of the wide kernel takes 1.91 of them (it
// does twice the work of one), and the split region's persistent kernel 1.04
// per round's worth of tiles.
namespace {
constexpr double kWideRoundCost = 1.91;
constexpr double kRegionRoundCost = 1.04;

double cost_128(long long tiles, int sms, int k_slices)
{
    if (tiles <= 0)
        return 0.0;
    const F32Schedule s = F32Schedule::make(static_cast<int>(tiles), sms, k_slices, true);
    if (!s.split())
        return static_cast<double>((tiles + sms - 1) / sms);
    return s.whole_rounds + static_cast<double>(tiles - s.region0) / sms * kRegionRoundCost;
}
} // namespace

int f32_wide_rows(int M, int N, int K, int sms, int mode)
{
    if (mode == 0 || sms < 1 || M < 128 || N < 256 || K < kF32WideMinK)
        return 0;
    const long long strips = (M + 127) / 128;  // 128-row strips of C
    const long long wn = (N + 255) / 256;      // wide tiles per strip
    const long long tn = (N + 127) / 128;      // 128 x 128 tiles per strip
    const int k_slices = (K + 15) / 16;
    // Strips the wide kernel can take in whole rounds: multiples of s0.
    const long long s0 = sms / std::gcd(static_cast<long long>(sms), wn);
    const double none = cost_128(strips * tn, sms, k_slices);
    double best = none;
    long long best_s = 0;
    for (long long sw = s0; sw <= strips; sw += s0) {
        const double c = static_cast<double>(sw * wn / sms) * kWideRoundCost + cost_128((strips - sw) * tn, sms, k_slices);
        if (c < best || (mode == 1 && best_s == 0)) {
            best = c;
            best_s = sw;
        }
    }
    // Take the wide kernel only for a gain of at least 1 % (or when forced).
    if (best_s == 0 || (mode != 1 && best > 0.99 * none))
        return 0;
    return best_s == strips ? M : static_cast<int>(best_s * 128);
}

} // namespace pg
