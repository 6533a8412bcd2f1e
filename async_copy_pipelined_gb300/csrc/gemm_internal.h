// Internal host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; not part of the public header.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "pipelined_gemm.h"

namespace pg {

// One FP32 GEMM request after validation.
struct F32Args {
    int M, N, K;
    const float *A;
    long long lda;
    const float *B;
    long long ldb;
    float *C;
    long long ldc;
    bool a_vec; // A base and row pitch allow 16-byte copies
    bool b_vec; // same for B
    bool c_vec; // C base and ldc allow float4 stores
    bool accumulate; // tiles start from C's values instead of +0
    int stages;
    int tile; // 64 or 128
    unsigned int *status; // device status word
    unsigned long long wait_limit_ns;
    int withhold;          // ring position a producer leaves unfilled (test hook; -1: none)
    int copy_form;         // cp.async qualifiers: bit 0 .L2::128B prefetch, bit 1 .L2::cache_hint
    int pol_a, pol_b;      // L2 policy per operand: 0 normal, 1 evict_first, 2 evict_last
    int wide_rows;         // TMA fill, 128 tile: rows [0, wide_rows) go to the wide-row kernel (0: none)
    int tile_limit;        // one-tile TMA kernel: CTAs of linear tile index >= this exit at once
    int ctas;              // split-region TMA kernel: CTAs launched (0: no split)
    int split_ctas;        // what a split would use (planning; 0: nothing to split)
    int split_region0;     // first tile of the split region (planning)
    int withhold_handover; // test hook: hand-over flags are never raised
    void *handover;        // persistent TMA kernel: accumulator hand-over space (nullptr: no split)
    long long handover_bytes; // bytes a split of this call needs (0: the schedule has no split)
    unsigned long long epoch; // value this call's ready flags carry
    int device;            // current device index
    unsigned long long ctx; // unique id of the current context (0: unknown)
};

struct Bf16Args {
    int M, N, K;
    const uint16_t *A;
    long long lda;
    const uint16_t *B;
    long long ldb;
    float *C;
    long long ldc;
    int stages;
    int block_m;  // 128 or 256 rows per CTA tile
    int c_tma;    // 1: C is written by TMA stores (16-byte aligned C, ldc % 4 == 0)
    unsigned int *status;
    unsigned long long wait_limit_ns;
    int withhold; // ring position the producers leave unfilled (test hook; -1: none)
    int copy_form;     // as F32Args
    int pol_a, pol_b;
    int num_sms;
    int device;
    unsigned long long ctx;
    // K split of the last round of tiles (TMA fill; gemm_bf16_ws), as for
    // the FP32 persistent kernel: hand-over space (nullptr: no split), the
    // bytes a split of this call needs, this call's flag value, test hook.
    void *handover;
    long long handover_bytes;
    unsigned long long epoch;
    int withhold_handover;
};

constexpr int kMaxDevices = 64;

// Raise a kernel's dynamic shared-memory limit once per context rather than
// on every launch: `done[dev]` holds the id of the context in which it was
// last raised, so a context created after cudaDeviceReset raises it again.
template <class Kernel>
int ensure_smem_limit(Kernel kernel, int smem, int dev, unsigned long long ctx,
                      std::atomic<unsigned long long> (&done)[kMaxDevices])
{
    if (ctx != 0 && dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire) == ctx)
        return GEMM_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (ctx != 0 && dev >= 0 && dev < kMaxDevices)
        done[dev].store(ctx, std::memory_order_release);
    return GEMM_OK;
}

// Launchers: each returns a gemm_status.  They assume validated arguments.
int launch_f32_sync(const F32Args &a, cudaStream_t s);
int launch_f32_cpasync(const F32Args &a, cudaStream_t s);
int launch_f32_tma(const F32Args &a, cudaStream_t s);
// The TMA fill's wide-row kernel (128 x 256 tiles, gemm_f32_tma_wide.cu) on
// rows [0, a.M): the caller passes a.M = the wide rows.
int launch_f32_tma_wide(const F32Args &a, cudaStream_t s);
// Rows of an M x N x K TMA call on the 128 tile that the wide-row kernel
// takes (a multiple of 128, or M), chosen by its measured round times;
// `mode` -1 decides by the model, 0 never, 1 whenever some cut is possible.
int f32_wide_rows(int M, int N, int K, int sms, int mode);
constexpr int kF32WideStages = 4;       // the wide-row kernel's ring (measured best of 2, 3, 4)
constexpr int kF32WideMinK = 1024;      // shorter K stays on the 128 x 128 tile
int f32_wide_smem_bytes();
int launch_f32_cpasync_mbar(const F32Args &a, cudaStream_t s);
int launch_f32_cpasync_ws(const F32Args &a, cudaStream_t s);
int f32_cpasync_ws_threads(int tile);
int launch_f32_zero(const F32Args &a, cudaStream_t s);
int launch_bf16(const Bf16Args &a, int fill, cudaStream_t s);
int launch_bf16_zero(const Bf16Args &a, cudaStream_t s);
int launch_selftest_wait(unsigned int *status, unsigned long long limit_ns, cudaStream_t s);

// Shared-memory bytes the FP32 kernels request for (tile, fill, stages).
int f32_smem_bytes(int tile, int fill, int stages);
int f32_threads(int tile, int fill);
int bf16_smem_bytes(int stages, int block_m);
int bf16_threads(int fill, int block_m);
constexpr int kBf16BlockM = 128;
constexpr int kBf16BlockN = 256;
constexpr int kBf16BlockK = 64;

// Unique id of the calling thread's current CUDA context (0 if unknown).
unsigned long long current_context_id();

// SM count of the current device (152 where no device can be asked).
int device_sms();

// The current device, checked to be an sm_103 part: GEMM_OK or an error.
int device_checked(int *dev);

// Device address of the library's status word in context `ctx` of `dev`.
unsigned int *device_status_word(int dev, unsigned long long ctx);

// Encode a 2-D tiled tensor map (row-major rows x cols, pitch in bytes).
// Returns GEMM_OK or GEMM_ERR_CUDA / GEMM_ERR_MISALIGNED.
int encode_tensor_map_2d(void *map_out, int dtype_is_bf16, const void *base, uint64_t cols, uint64_t rows,
                         uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, int swizzle_128b);

// Status codes recorded on device: low byte = kernel family, next byte = role.
constexpr unsigned int kErrFamilyF32Tma = 1;
constexpr unsigned int kErrFamilyBf16 = 2;
constexpr unsigned int kErrFamilySelftest = 3;
constexpr unsigned int kErrFamilyF32CpAsyncMbar = 4;
constexpr unsigned int kErrFamilyF32CpAsyncWs = 5;
constexpr unsigned int kErrFamilyF32TmaWide = 6;
constexpr unsigned int kErrRoleConsumer = 1u << 8;
constexpr unsigned int kErrRoleProducer = 2u << 8;
constexpr unsigned int kErrRoleMma = 3u << 8;
constexpr unsigned int kErrRoleEpilogue = 4u << 8;
constexpr unsigned int kErrRoleDrain = 5u << 8;
constexpr unsigned int kErrRoleHandover = 6u << 8;

} // namespace pg
