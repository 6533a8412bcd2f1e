// C ABI of the pipelined GEMM library: argument validation, launch planning,
// the device status word, TMA tensor-map encoding and the bounded-wait
// self-test.  Everything here runs on the host except the two tiny kernels at
// the bottom.
//
// Validation mirrors the lesson program's gates ("pipelined_gemm.cu", main:
// refuse an unsuitable device before doing anything, check every result
// before timing) but reports a status code instead of exiting.
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstring>

#include <cudaTypedefs.h>

#include "f32_schedule.cuh"
#include "gemm_internal.h"
#include "pipelined_gemm_testing.h"
#include "ptx.cuh"
#include "tma_ring.cuh"

namespace pg {

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull; // 2 s
// Four stages for every FP32 ring fill.  Measured on GB300 (TFLOP/s, 3 / 4
// stages, 128x128 tile at 4096^3): cp.async 55.8 / 56.0, cp.async +
// mbarrier 52.6 / 53.7, TMA 59.7 / 60.2.  The latency-bound one-warp
// 32x32x65536 shape needs the depth most (cp.async 3435 us at 2 stages,
// 1923 us at 4).  At one CTA per SM the fourth 32 KiB stage costs no
// occupancy; the 64x64 tile's three CTAs per SM take 96 KiB.
constexpr int kDefaultStagesF32 = 4;
// Except the TMA fill on the 128x128 tile, which runs best with two (GB300,
// TFLOP/s for 2 / 3 / 4 / 6 stages: 61.3 / 60.3 / 61.0 / 60.4 at 4096^3,
// 55.9 / - / 55.5 / - at 3000 x 5000 x 1000; with the K split of the last
// round).  Its consumers chain slices, so two stages already keep a slice
// in flight while one is computed.
constexpr int kDefaultStagesF32TmaTile128 = 2;
// The producer-warp cp.async fill runs best with two (GB300, 4096^3,
// TFLOP/s for 2 / 3 / 4 stages with four producer warps: 58.1 / 57.3 /
// 57.3).
constexpr int kDefaultStagesF32CpAsyncWs = 2;
// BF16 ring depth: four 48 KiB stages for the 128-row tile, three 64 KiB
// stages for the 256-row tile (four of those do not fit in 227 KiB).
constexpr int kDefaultStagesBf16Tile128 = 4;
constexpr int kDefaultStagesBf16Tile256 = 3;
// block_m = 0 weighs the two BF16 tiles by waves of persistent CTAs: a
// 256-row tile does twice the work of a 128-row one at this much higher
// throughput (per cent; GB300, 8192^3: 1881 against 1738 TFLOP/s).  The
// model picks the faster tile on every shape measured (1536^2 .. 8192^2,
// 512 x 16384, 1024 x 8192, 8192 x 1024); e.g. 3584^2 x 4096 keeps the
// 128-row tile (392 tiles in 3 waves against 196 in 2 double waves:
// measured 1341 against 1172 TFLOP/s) and 2304^2 x 4096 takes the 256-row
// tile (910 against 822).
constexpr long long kBf16TallTileSpeedPct = 108;
// SM count assumed when no device can be asked (a GB300 has 152).
constexpr int kPlanningSms = 152;
// block_tile = 0 picks the 128x128 tile from this many 128x128 tiles on (a
// little under one wave at one CTA per SM on a 152-SM GB300); below it the
// 64x64 tile, three CTAs per SM, fills the GPU better.  Measured on GB300
// (TMA, four stages, TFLOP/s for the 64 / 128 tile): 64 tiles (1024^3)
// 37.0 / 23.9, 100 tiles (1280^3) 40.7 / 38.1, 128 tiles (512 x 4096 x
// 4096 and two other shapes) 41.8 / 51.1, 144 tiles (1536^3) 43.8 / 55.4;
// the cp.async and register fills cross over at the same point.
constexpr long long kLargeTileMinTiles = 120;

__device__ unsigned int g_status_word;

// ------------------------------------------------------------ device state
static std::atomic<int> g_arch_ok[kMaxDevices];     // 0 unknown, 1 ok, 2 wrong arch
static std::atomic<int> g_num_sms[kMaxDevices];

// Test hooks (pipelined_gemm_testing.h): a shorter wait limit and a ring
// position the producers leave unfilled.  Read once per call.
static std::atomic<unsigned long long> g_hook_wait_limit_ns{0}; // 0: kDefaultWaitLimitNs
static std::atomic<int> g_hook_withhold{-1};
static std::atomic<int> g_hook_withhold_handover{0};
static std::atomic<int> g_hook_f32_wide{-1}; // f32_wide_rows mode: -1 model, 0 off, 1 forced

// Unique id of the calling thread's current CUDA context (cuCtxGetId), or 0
// if the driver cannot say.  Per-context state (the status word's address,
// raised shared-memory limits) is keyed on it, so a context created after
// cudaDeviceReset starts afresh.
unsigned long long current_context_id()
{
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static std::atomic<void *> get_current{nullptr};
    static std::atomic<void *> get_id{nullptr};
    void *gc = get_current.load(), *gi = get_id.load();
    if (!gc || !gi) {
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &gc, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &gi, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        get_current.store(gc);
        get_id.store(gi);
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (reinterpret_cast<GetCurrentFn>(gc)(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        reinterpret_cast<GetIdFn>(gi)(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

static int current_device(int *dev)
{
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices)
        return GEMM_ERR_CUDA;
    return GEMM_OK;
}

// The kernels are built for sm_103a only; refuse anything else up front
// rather than launching code that cannot run there.
static int check_device(int *dev_out)
{
    int dev;
    if (current_device(&dev) != GEMM_OK)
        return GEMM_ERR_CUDA;
    int state = g_arch_ok[dev].load();
    if (state == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_num_sms[dev].store(sms);
        g_arch_ok[dev].store(state);
    }
    if (state != 1)
        return GEMM_ERR_ARCH;
    *dev_out = dev;
    return GEMM_OK;
}

// Address of this library's status word in the current context of device
// `dev`.  Looked up once per context (`ctx` from current_context_id()); with
// no context id it is looked up on every call.
static unsigned int *status_word(int dev, unsigned long long ctx)
{
    struct Cached {
        std::atomic<unsigned long long> ctx{0};
        std::atomic<uintptr_t> addr{0};
    };
    static Cached cache[kMaxDevices];
    if (ctx != 0 && cache[dev].ctx.load(std::memory_order_acquire) == ctx) {
        const uintptr_t p = cache[dev].addr.load(std::memory_order_relaxed);
        if (p != 0)
            return reinterpret_cast<unsigned int *>(p);
    }
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess)
        return nullptr;
    if (ctx != 0) {
        cache[dev].addr.store(reinterpret_cast<uintptr_t>(addr), std::memory_order_relaxed);
        cache[dev].ctx.store(ctx, std::memory_order_release);
    }
    return static_cast<unsigned int *>(addr);
}

// Value the ready flags of the next persistent FP32 call carry: unique per
// call within the process, and salted so that no value left in a reused
// hand-over buffer by another process or library instance matches it.
static unsigned long long next_epoch()
{
    static std::atomic<unsigned long long> counter{0};
    unsigned long long v = counter.load();
    if (v == 0) {
        // SplitMix64's finaliser (Steele, Lea & Flood 2014) over the clock
        // and an address of this instance.
        unsigned long long z = static_cast<unsigned long long>(
                                   std::chrono::steady_clock::now().time_since_epoch().count()) ^
                               reinterpret_cast<uintptr_t>(&counter);
        z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
        z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
        z ^= z >> 31;
        unsigned long long expected = 0;
        counter.compare_exchange_strong(expected, z | 1ull);
    }
    return counter.fetch_add(1) + 1;
}

static unsigned long long hook_wait_limit_ns()
{
    const unsigned long long v = g_hook_wait_limit_ns.load();
    return v != 0 ? v : kDefaultWaitLimitNs;
}

// ------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn()
{
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load();
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

int encode_tensor_map_2d(void *map_out, int dtype_is_bf16, const void *base, uint64_t cols, uint64_t rows,
                         uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, int swizzle_128b)
{
    if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (pitch_bytes & 15u) != 0)
        return GEMM_ERR_MISALIGNED;
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_fn();
    if (!encode)
        return GEMM_ERR_CUDA;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(static_cast<CUtensorMap *>(map_out),
                              dtype_is_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle_128b ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// ------------------------------------------------------------ sizes
int f32_threads(int tile, int fill)
{
    if (fill == GEMM_FILL_CPASYNC_WS)
        return f32_cpasync_ws_threads(tile);
    return (tile == 32 ? 32 : 256) + (fill == GEMM_FILL_TMA ? 32 : 0);
}

int f32_smem_bytes(int tile, int fill, int stages)
{
    const int stage_bytes = (tile * 16 + 16 * tile) * 4;
    if (fill == GEMM_FILL_SYNC)
        return stage_bytes;
    if (fill == GEMM_FILL_CPASYNC)
        return stages * stage_bytes;
    // TMA / mbarrier ring: + its barriers, two hand-over barriers, a flag and
    // the work schedule (the persistent TMA kernel), and alignment slack.
    return stages * stage_bytes + 16 * stages + 64 + 1024;
}


// The tensor-core kernel is persistent (one CTA per SM) and allocates all of
// an SM's tensor memory, so a second CTA placed on the same SM would block in
// tcgen05.alloc until the first had finished every tile while another SM sat
// idle.  Small rings (two stages, or the one-stage register fill) would leave
// room for a second CTA; the request is raised so that two never fit in an
// SM's 228 KB.
constexpr int kBf16ExclusiveSmemBytes = 116 * 1024;

int bf16_smem_bytes(int stages, int block_m)
{
    const int stage_bytes = (block_m * kBf16BlockK + kBf16BlockK * kBf16BlockN) * 2;
    const int staging = (block_m / 128) * 4 * 4096; // one 32 x 32 FP32 box per epilogue warp
    const int need = stages * stage_bytes + staging + 1024 /* barriers, TMEM slot */ + 1024 /* alignment slack */;
    return need > kBf16ExclusiveSmemBytes ? need : kBf16ExclusiveSmemBytes;
}

// ------------------------------------------------------------ planning
// SMs of the current device for choosing a tile (cached once the device has
// been checked), or kPlanningSms where there is no device to ask.
static int planning_sms();

int device_sms() { return planning_sms(); }

int device_checked(int *dev) { return check_device(dev); }

unsigned int *device_status_word(int dev, unsigned long long ctx) { return status_word(dev, ctx); }

static int planning_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        const int cached = g_num_sms[dev].load();
        if (cached > 0)
            return cached;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
            return sms;
    }
    (void)cudaGetLastError();
    return kPlanningSms;
}

// Split fill_mode into the fill (low byte) and the options (GEMM_OPT_*), and
// check that the cache qualifiers suit the fill: the prefetch size is a
// cp.async qualifier; L2 policies go on cp.async and TMA copies, not on the
// register path's plain loads.  Fills out the copy form, the policies and
// the accumulate flag.
static int decode_options(int fill_mode, int *fill, int *copy_form, int *pol_a, int *pol_b, bool *accumulate)
{
    const int opts = fill_mode & ~0xFF;
    *fill = fill_mode & 0xFF;
    *copy_form = 0;
    *pol_a = *pol_b = 0;
    *accumulate = (opts & GEMM_OPT_ACCUMULATE) != 0;
    if (opts & ~GEMM_OPT_MASK)
        return GEMM_ERR_INVALID_ARG;
    if ((opts & GEMM_OPT_A_EVICT_FIRST) && (opts & GEMM_OPT_A_EVICT_LAST))
        return GEMM_ERR_INVALID_ARG;
    if ((opts & GEMM_OPT_B_EVICT_FIRST) && (opts & GEMM_OPT_B_EVICT_LAST))
        return GEMM_ERR_INVALID_ARG;
    const bool cpasync =
        *fill == GEMM_FILL_CPASYNC || *fill == GEMM_FILL_CPASYNC_MBAR || *fill == GEMM_FILL_CPASYNC_WS;
    const bool policy = (opts & (GEMM_OPT_A_EVICT_FIRST | GEMM_OPT_A_EVICT_LAST | GEMM_OPT_B_EVICT_FIRST |
                                 GEMM_OPT_B_EVICT_LAST)) != 0;
    if ((opts & GEMM_OPT_L2_PREFETCH_128B) && !cpasync)
        return GEMM_ERR_INVALID_ARG;
    if (policy && !cpasync && *fill != GEMM_FILL_TMA)
        return GEMM_ERR_INVALID_ARG;
    // The kernels that start from C are built with plain copies only.
    if (*accumulate && (opts & ~GEMM_OPT_ACCUMULATE) != 0)
        return GEMM_ERR_UNSUPPORTED;
    *copy_form = ((opts & GEMM_OPT_L2_PREFETCH_128B) ? 1 : 0) | (policy ? 2 : 0);
    *pol_a = (opts & GEMM_OPT_A_EVICT_FIRST) ? 1 : (opts & GEMM_OPT_A_EVICT_LAST) ? 2 : 0;
    *pol_b = (opts & GEMM_OPT_B_EVICT_FIRST) ? 1 : (opts & GEMM_OPT_B_EVICT_LAST) ? 2 : 0;
    return GEMM_OK;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

static int plan_f32(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                    int fill_mode, int stages, int tile, gemm_plan *plan, F32Args *args)
{
    if (M < 0 || N < 0 || K < 0)
        return GEMM_ERR_INVALID_ARG;
    int fill, copy_form, pol_a, pol_b;
    bool accumulate;
    const int opt_status = decode_options(fill_mode, &fill, &copy_form, &pol_a, &pol_b, &accumulate);
    if (opt_status != GEMM_OK)
        return opt_status;
    if (fill != GEMM_FILL_SYNC && fill != GEMM_FILL_CPASYNC && fill != GEMM_FILL_TMA &&
        fill != GEMM_FILL_CPASYNC_MBAR && fill != GEMM_FILL_CPASYNC_WS)
        return GEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
        return GEMM_ERR_INVALID_ARG;
    const bool work = M > 0 && N > 0;
    if (work && (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))))
        return GEMM_ERR_INVALID_ARG;
    if (!aligned4(A) || !aligned4(B) || !aligned4(C))
        return GEMM_ERR_MISALIGNED;
    if (fill == GEMM_FILL_SYNC) {
        if (stages != 0 && stages != 1)
            return GEMM_ERR_INVALID_ARG;
        stages = 1;
    } else if (stages != 0 && (stages < 2 || stages > 6)) {
        return GEMM_ERR_INVALID_ARG;
    }
    if (tile == 0) {
        const long long t128 = static_cast<long long>((M + 127) / 128) * ((N + 127) / 128);
        tile = t128 >= kLargeTileMinTiles ? 128 : 64;
    } else if (tile != 32 && tile != 64 && tile != 128) {
        return GEMM_ERR_INVALID_ARG;
    }
    if (stages == 0)
        stages = fill == GEMM_FILL_CPASYNC_WS               ? kDefaultStagesF32CpAsyncWs
                 : (fill == GEMM_FILL_TMA && tile == 128) ? kDefaultStagesF32TmaTile128
                                                          : kDefaultStagesF32;
    const bool a_vec = aligned16(A) && (lda % 4) == 0;
    const bool b_vec = aligned16(B) && (ldb % 4) == 0;
    const bool c_vec = aligned16(C) && (ldc % 4) == 0;
    if (fill == GEMM_FILL_TMA && K > 0 && work && (!a_vec || !b_vec))
        return GEMM_ERR_MISALIGNED;
    // Rows that are not 16-byte aligned are copied 4 bytes at a time
    // (cp.async.ca); those copies carry no cache policy.
    if ((copy_form & 2) != 0 &&
        (fill == GEMM_FILL_CPASYNC || fill == GEMM_FILL_CPASYNC_MBAR || fill == GEMM_FILL_CPASYNC_WS) && K > 0 &&
        work && (!a_vec || !b_vec))
        return GEMM_ERR_UNSUPPORTED;
    const long long grid_y = (M + tile - 1) / tile;
    const long long grid_x = (N + tile - 1) / tile;
    if (grid_y > 65535 || grid_x * grid_y > 0x7fffffffLL)
        return GEMM_ERR_INVALID_ARG;
    // The TMA fill's 128 x 128 tile: with hand-over space (gemm_f32_ws) and
    // a tile count that is not a multiple of the SM count, the last round
    // and one more are split in K over one CTA per SM (f32_schedule.cuh).
    //
    // Before that, the top rows may go to the wide-row kernel (128 x 256
    // tiles, gemm_f32_tma_wide.cu) where it shortens the call; the 128 x 128
    // path, split included, then covers the rows below them.  Plain copies
    // only: the wide kernel carries no cache qualifiers.
    int ctas = 0;
    long long handover = 0;
    int region0 = 0x7fffffff;
    int wide_rows = 0;
    if (fill == GEMM_FILL_TMA && tile == 128 && work && K > 0) {
        const int sms = planning_sms();
        if (copy_form == 0 && pol_a == 0 && pol_b == 0)
            wide_rows = f32_wide_rows(M, N, K, sms, g_hook_f32_wide.load());
        const long long tiles = grid_x * ((M - wide_rows + tile - 1) / tile);
        if (tiles > 0) {
            const F32Schedule sch = F32Schedule::make(static_cast<int>(tiles), sms, (K + 15) / 16, true);
            if (sch.split()) {
                ctas = sms;
                handover = f32_handover_bytes(sms);
                region0 = sch.region0;
            }
        }
    }

    if (plan) {
        std::memset(plan, 0, sizeof *plan);
        plan->fill_mode = fill;
        plan->block_m = tile;
        plan->block_n = tile;
        plan->block_k = 16;
        plan->thread_m = tile == 64 ? 4 : 8;
        plan->thread_n = tile == 128 ? 8 : 4;
        plan->threads = f32_threads(tile, fill);
        plan->stages = stages;
        if (fill == GEMM_FILL_TMA) {
            plan->a_copy_bytes = tile * 16 * 4;
            plan->b_copy_bytes = 16 * tile * 4;
        } else {
            plan->a_copy_bytes = a_vec ? 16 : 4;
            plan->b_copy_bytes = b_vec ? 16 : 4;
        }
        plan->smem_bytes = f32_smem_bytes(tile, fill, stages);
        plan->grid_x = static_cast<int>(grid_x);
        plan->grid_y = static_cast<int>(grid_y);
        plan->k_slices = (K + 15) / 16;
        plan->options = fill_mode & GEMM_OPT_MASK;
        plan->persistent_ctas = ctas;
        plan->workspace_bytes = static_cast<int>(handover);
        plan->wide_rows = wide_rows;
    }
    if (args) {
        args->M = M;
        args->N = N;
        args->K = K;
        args->A = A;
        args->lda = lda;
        args->B = B;
        args->ldb = ldb;
        args->C = C;
        args->ldc = ldc;
        args->a_vec = a_vec;
        args->b_vec = b_vec;
        args->c_vec = c_vec;
        args->accumulate = accumulate;
        args->stages = stages;
        args->tile = tile;
        args->status = nullptr;
        args->wait_limit_ns = hook_wait_limit_ns();
        args->withhold = g_hook_withhold.load();
        args->copy_form = copy_form;
        args->pol_a = pol_a;
        args->pol_b = pol_b;
        args->ctas = 0;         // set when the call brings hand-over space
        args->wide_rows = wide_rows;
        args->tile_limit = 0x7fffffff;
        args->split_ctas = ctas;
        args->split_region0 = region0;
        args->withhold_handover = g_hook_withhold_handover.load();
        args->handover = nullptr;
        args->handover_bytes = handover;
        args->epoch = 0;
        args->device = 0;
        args->ctx = 0;
    }
    return GEMM_OK;
}

static int plan_bf16(int M, int N, int K, const uint16_t *A, int lda, const uint16_t *B, int ldb, float *C, int ldc,
                     int fill_mode, int stages, int block_m, gemm_plan *plan, Bf16Args *args)
{
    if (M < 0 || N < 0 || K < 0)
        return GEMM_ERR_INVALID_ARG;
    int fill, copy_form, pol_a, pol_b;
    bool accumulate;
    const int opt_status = decode_options(fill_mode, &fill, &copy_form, &pol_a, &pol_b, &accumulate);
    if (opt_status != GEMM_OK)
        return opt_status;
    if (fill == GEMM_FILL_CPASYNC_MBAR || fill == GEMM_FILL_CPASYNC_WS || accumulate)
        return GEMM_ERR_UNSUPPORTED;
    if (block_m != 0 && block_m != 128 && block_m != 256)
        return GEMM_ERR_INVALID_ARG;
    if (fill != GEMM_FILL_TMA && fill != GEMM_FILL_CPASYNC && fill != GEMM_FILL_SYNC)
        return GEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
        return GEMM_ERR_INVALID_ARG;
    const bool work = M > 0 && N > 0;
    if (work && (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))))
        return GEMM_ERR_INVALID_ARG;
    if (fill == GEMM_FILL_SYNC && stages != 0 && stages != 1)
        return GEMM_ERR_INVALID_ARG; // the register-path fill has one stage: loads and MMAs alternate
    if (fill != GEMM_FILL_SYNC && stages != 0 && (stages < 2 || stages > kDefaultStagesBf16Tile128))
        return GEMM_ERR_INVALID_ARG;
    if (block_m == 0) {
        // Four stages only fit the 128-row tile.  Otherwise compare the time
        // of ceil(tiles / SMs) waves of each tile.
        const long long sms = planning_sms();
        const long long tiles_n_ = (N + kBf16BlockN - 1) / kBf16BlockN;
        const long long waves128 = ((static_cast<long long>(M) + 127) / 128 * tiles_n_ + sms - 1) / sms;
        const long long waves256 = ((static_cast<long long>(M) + 255) / 256 * tiles_n_ + sms - 1) / sms;
        block_m = (stages != 4 && 2 * waves256 * 100 < waves128 * kBf16TallTileSpeedPct) ? 256 : 128;
    }
    if (fill == GEMM_FILL_SYNC)
        stages = 1;
    else if (stages == 0)
        stages = block_m == 256 ? kDefaultStagesBf16Tile256 : kDefaultStagesBf16Tile128;
    if (block_m == 256 && stages > kDefaultStagesBf16Tile256)
        return GEMM_ERR_INVALID_ARG;
    if (!aligned4(C))
        return GEMM_ERR_MISALIGNED;
    if (work && K > 0 && (!aligned16(A) || !aligned16(B) || (lda % 8) != 0 || (ldb % 8) != 0))
        return GEMM_ERR_MISALIGNED;
    const long long tiles_m = (M + block_m - 1) / block_m;
    const long long tiles_n = (N + kBf16BlockN - 1) / kBf16BlockN;
    if (tiles_m * tiles_n > 0x7fffffffLL)
        return GEMM_ERR_INVALID_ARG;
    // The TMA fill, like the FP32 one, can split the last round of tiles and
    // one more in K between the persistent CTAs (gemm_bf16_ws): hand-over
    // space of one block_m x 256 FP32 accumulator tile and an 8-byte flag
    // per CTA.
    long long handover = 0;
    if (fill == GEMM_FILL_TMA && work && K > 0) {
        const int sms = planning_sms();
        const F32Schedule sch = F32Schedule::make(static_cast<int>(tiles_m * tiles_n), sms,
                                                  (K + kBf16BlockK - 1) / kBf16BlockK, true);
        if (sch.split())
            handover = static_cast<long long>(sms) * (static_cast<long long>(block_m) * kBf16BlockN * 4 + 8);
    }
    if (plan) {
        std::memset(plan, 0, sizeof *plan);
        plan->fill_mode = fill;
        plan->block_m = block_m;
        plan->block_n = kBf16BlockN;
        plan->block_k = kBf16BlockK;
        plan->threads = bf16_threads(fill, block_m);
        plan->stages = stages;
        plan->a_copy_bytes = fill == GEMM_FILL_TMA ? block_m * kBf16BlockK * 2 : 16;
        plan->b_copy_bytes = fill == GEMM_FILL_TMA ? kBf16BlockK * 64 * 2 : 16;
        plan->smem_bytes = bf16_smem_bytes(stages, block_m);
        plan->grid_x = static_cast<int>(tiles_m * tiles_n); // upper bound; capped at the SM count on launch
        plan->grid_y = 1;
        plan->k_slices = (K + kBf16BlockK - 1) / kBf16BlockK;
        plan->options = fill_mode & GEMM_OPT_MASK;
        plan->persistent_ctas = static_cast<int>(tiles_m * tiles_n < planning_sms() ? tiles_m * tiles_n
                                                                                    : planning_sms());
        plan->workspace_bytes = static_cast<int>(handover);
    }
    if (args) {
        args->M = M;
        args->N = N;
        args->K = K;
        args->A = A;
        args->lda = lda;
        args->B = B;
        args->ldb = ldb;
        args->C = C;
        args->ldc = ldc;
        args->stages = stages;
        args->block_m = block_m;
        args->c_tma = aligned16(C) && (ldc % 4) == 0 ? 1 : 0;
        args->status = nullptr;
        args->wait_limit_ns = hook_wait_limit_ns();
        args->withhold = g_hook_withhold.load();
        args->copy_form = copy_form;
        args->pol_a = pol_a;
        args->pol_b = pol_b;
        args->num_sms = 0;
        args->device = 0;
        args->ctx = 0;
        args->handover = nullptr; // set when the call brings hand-over space
        args->handover_bytes = handover;
        args->epoch = 0;
        args->withhold_handover = g_hook_withhold_handover.load();
    }
    return GEMM_OK;
}

// ------------------------------------------------------------ self-test kernel
__global__ void selftest_wait_kernel(unsigned int *status, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the wait must expire and report.
        if (!mbar_wait_bounded(b, 0, limit_ns))
            record_error(status, kErrFamilySelftest | kErrRoleConsumer);
    }
}

int launch_selftest_wait(unsigned int *status, unsigned long long limit_ns, cudaStream_t s)
{
    selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

} // namespace pg

using namespace pg;

// ================================================================ C ABI
extern "C" {

int gemm_version(void) { return 10200; }

const char *gemm_status_string(int status)
{
    switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid size, leading dimension, pointer, fill, stages or tile";
    case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED: base or row pitch not aligned as the fill requires";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: the library does not implement this request";
    case GEMM_ERR_ARCH: return "GEMM_ERR_ARCH: current device is not compute capability 10.3 (sm_103a)";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: a CUDA runtime or driver call failed";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a kernel's bounded wait expired";
    default: return "unknown gemm_status";
    }
}

int gemm_f32_plan(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                  int fill_mode, int stages, int block_tile, gemm_plan *plan)
{
    if (!plan)
        return GEMM_ERR_INVALID_ARG;
    return plan_f32(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_tile, plan, nullptr);
}

int gemm_f32(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc, int fill_mode,
             int stages, int block_tile, void *stream)
{
    return gemm_f32_ws(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_tile, nullptr, 0, stream);
}

int gemm_f32_ws(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C, int ldc,
                int fill_mode, int stages, int block_tile, void *workspace, size_t workspace_bytes, void *stream)
{
    F32Args args;
    int st = plan_f32(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_tile, nullptr, &args);
    if (st != GEMM_OK)
        return st;
    if (workspace != nullptr && args.handover_bytes > 0) {
        if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
            return GEMM_ERR_MISALIGNED;
        if (workspace_bytes < static_cast<size_t>(args.handover_bytes))
            return GEMM_ERR_INVALID_ARG;
        args.handover = workspace;
        args.epoch = next_epoch();
        args.ctas = args.split_ctas;
        args.tile_limit = args.split_region0;
    }
    int dev;
    st = check_device(&dev);
    if (st != GEMM_OK)
        return st;
    if (M == 0 || N == 0)
        return GEMM_OK;
    args.device = dev;
    args.ctx = current_context_id();
    args.status = status_word(dev, args.ctx);
    if (!args.status)
        return GEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) // C = +0, or with accumulate C as it is
        return args.accumulate ? GEMM_OK : launch_f32_zero(args, s);
    switch (fill_mode & 0xFF) {
    case GEMM_FILL_SYNC: return launch_f32_sync(args, s);
    case GEMM_FILL_CPASYNC: return launch_f32_cpasync(args, s);
    case GEMM_FILL_CPASYNC_MBAR: return launch_f32_cpasync_mbar(args, s);
    case GEMM_FILL_CPASYNC_WS: return launch_f32_cpasync_ws(args, s);
    default: break;
    }
    if (args.wide_rows > 0) {
        // Rows [0, wide_rows) on 128 x 256 tiles, then the rest on the
        // 128 x 128 path, in that order on the stream (disjoint rows of C).
        F32Args wide = args;
        wide.M = args.wide_rows;
        st = launch_f32_tma_wide(wide, s);
        if (st != GEMM_OK || args.wide_rows == M)
            return st;
        args.A += static_cast<long long>(args.wide_rows) * args.lda;
        args.C += static_cast<long long>(args.wide_rows) * args.ldc;
        args.M = M - args.wide_rows;
    }
    return launch_f32_tma(args, s);
}

int gemm_bf16_plan(int M, int N, int K, const uint16_t *A, int lda, const uint16_t *B, int ldb, float *C, int ldc,
                   int fill_mode, int stages, int block_m, gemm_plan *plan)
{
    if (!plan)
        return GEMM_ERR_INVALID_ARG;
    return plan_bf16(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_m, plan, nullptr);
}

int gemm_bf16(int M, int N, int K, const uint16_t *A, int lda, const uint16_t *B, int ldb, float *C, int ldc,
              int fill_mode, int stages, int block_m, void *stream)
{
    return gemm_bf16_ws(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_m, nullptr, 0, stream);
}

int gemm_bf16_ws(int M, int N, int K, const uint16_t *A, int lda, const uint16_t *B, int ldb, float *C, int ldc,
                 int fill_mode, int stages, int block_m, void *workspace, size_t workspace_bytes, void *stream)
{
    Bf16Args args;
    int st = plan_bf16(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_m, nullptr, &args);
    if (st != GEMM_OK)
        return st;
    if (workspace != nullptr && args.handover_bytes > 0) {
        if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
            return GEMM_ERR_MISALIGNED;
        if (workspace_bytes < static_cast<size_t>(args.handover_bytes))
            return GEMM_ERR_INVALID_ARG;
        args.handover = workspace;
        args.epoch = next_epoch();
    }
    int dev;
    st = check_device(&dev);
    if (st != GEMM_OK)
        return st;
    if (M == 0 || N == 0)
        return GEMM_OK;
    args.device = dev;
    args.ctx = current_context_id();
    args.status = status_word(dev, args.ctx);
    if (!args.status)
        return GEMM_ERR_CUDA;
    args.num_sms = g_num_sms[dev].load();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0)
        return launch_bf16_zero(args, s);
    return launch_bf16(args, fill_mode & 0xFF, s);
}

int gemm_device_status(void *stream, unsigned int *detail)
{
    int dev;
    if (current_device(&dev) != GEMM_OK)
        return GEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int *word = status_word(dev, current_context_id());
    if (!word)
        return GEMM_ERR_CUDA;
    unsigned int value = 0;
    if (cudaMemcpyAsync(&value, word, sizeof value, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(word, 0, sizeof(unsigned int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (detail)
        *detail = value;
    return value == 0 ? GEMM_OK : GEMM_ERR_TIMEOUT;
}

int gemm_selftest_bounded_wait(int timeout_us, void *stream)
{
    if (timeout_us < 1 || timeout_us > 1000000)
        return GEMM_ERR_INVALID_ARG;
    int dev;
    int st = check_device(&dev);
    if (st != GEMM_OK)
        return st;
    unsigned int *word = status_word(dev, current_context_id());
    if (!word)
        return GEMM_ERR_CUDA;
    return launch_selftest_wait(word, static_cast<unsigned long long>(timeout_us) * 1000ull,
                                static_cast<cudaStream_t>(stream));
}

int gemm_testing_withhold_handover(int on)
{
    g_hook_withhold_handover.store(on ? 1 : 0);
    return GEMM_OK;
}

int gemm_testing_f32_piece(int tiles, int ctas, int k_slices, int split, int cta, int idx, int *out)
{
    if (!out || tiles < 0 || ctas < 1 || k_slices < 1 || cta < 0 || cta >= ctas || idx < 0)
        return 0;
    const F32CtaPieces q = F32CtaPieces::make(F32Schedule::make(tiles, ctas, k_slices, split != 0), cta);
    if (idx >= q.count())
        return 0;
    const F32Piece pc = q.piece(idx);
    out[0] = pc.tile;
    out[1] = pc.s_begin;
    out[2] = pc.s_end;
    out[3] = pc.from_partial ? 1 : 0;
    out[4] = pc.to_partial ? 1 : 0;
    return 1;
}

int gemm_testing_f32_wide(int mode)
{
    if (mode < -1 || mode > 1)
        return GEMM_ERR_INVALID_ARG;
    g_hook_f32_wide.store(mode);
    return GEMM_OK;
}

int gemm_testing_f32_wide_rows(int M, int N, int K, int sms, int mode)
{
    if (M < 0 || N < 0 || K < 0 || sms < 1 || mode < -1 || mode > 1)
        return -1;
    return f32_wide_rows(M, N, K, sms, mode);
}

int gemm_testing_set_hooks(unsigned long long wait_limit_ns, int withhold_position)
{
    if (withhold_position < -1 || (wait_limit_ns != 0 && wait_limit_ns < 1000000ull))
        return GEMM_ERR_INVALID_ARG;
    g_hook_wait_limit_ns.store(wait_limit_ns);
    g_hook_withhold.store(withhold_position);
    return GEMM_OK;
}

} // extern "C"
