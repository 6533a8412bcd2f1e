// gemm_f32_noalloc: gemm_f32_ws for callers that cannot allocate device
// memory.  The hand-over space the FP32 TMA fill's split of the last round
// of tiles needs lives in a fixed array of this library's module instead of
// a caller buffer, so the call allocates nothing and frees nothing.
//
// Some callers cannot allocate: an allocator that needs a GEMM while serving
// an allocation (re-entering cudaMalloc from inside it is not possible),
// code with a fixed, pre-planned memory budget, or latency-bound code that
// must not run cudaMalloc / cudaFree, which can synchronise the whole device.
#include <atomic>
#include <cstdint>

#include "f32_schedule.cuh"
#include "gemm_internal.h"

namespace pg {

// Room for the hand-over of this many CTAs (one per SM): 152 on GB300.
constexpr int kNoAllocMaxCtas = 160;
constexpr long long kNoAllocBytes = kNoAllocMaxCtas * (kF32HandoverTileBytes + 8);

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch in the current context.  In host code
// the array's name stands for a host-side shadow, not device memory, so the
// kernel must be given this address instead.  Looked up once per context
// (a context made after cudaDeviceReset looks it up again).
static void *noalloc_scratch(int dev)
{
    struct Cached {
        std::atomic<unsigned long long> ctx{0};
        std::atomic<uintptr_t> addr{0};
    };
    static Cached cache[kMaxDevices];
    const unsigned long long ctx = current_context_id();
    if (ctx != 0 && cache[dev].ctx.load(std::memory_order_acquire) == ctx) {
        const uintptr_t a = cache[dev].addr.load(std::memory_order_relaxed);
        if (a != 0)
            return reinterpret_cast<void *>(a);
    }
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (ctx != 0) {
        cache[dev].addr.store(reinterpret_cast<uintptr_t>(ptr), std::memory_order_relaxed);
        cache[dev].ctx.store(ctx, std::memory_order_release);
    }
    return ptr;
}

} // namespace pg

using namespace pg;

extern "C" int gemm_f32_noalloc(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float *C,
                                int ldc, int fill_mode, int stages, int block_tile, void *stream)
{
    gemm_plan plan;
    const int st = gemm_f32_plan(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_tile, &plan);
    if (st != GEMM_OK)
        return st;
    if (plan.workspace_bytes == 0) // nothing to hand over: exactly gemm_f32
        return gemm_f32_ws(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_tile, nullptr, 0, stream);
    if (plan.workspace_bytes > kNoAllocBytes)
        return GEMM_ERR_UNSUPPORTED; // more SMs than the fixed array has room for
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return GEMM_ERR_CUDA;
    void *scratch = noalloc_scratch(dev);
    if (!scratch)
        return GEMM_ERR_CUDA;
    return gemm_f32_ws(M, N, K, A, lda, B, ldb, C, ldc, fill_mode, stages, block_tile, scratch,
                       static_cast<size_t>(kNoAllocBytes), stream);
}
