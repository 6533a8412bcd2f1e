// FP32 GEMM, fill (a): the register path.
//
// Per K slice every thread loads its float4 chunks of A and B from global
// memory into registers, stores them to shared memory, and the block meets at
// a barrier before and after the inner product ("pipelined_gemm.cu",
// matmulTileSync; "Day 74: Async copies and pipelines", section "A copy that
// skips the registers": load, wait, compute, repeat).  One stage only: the
// load of slice k+1 cannot start until slice k's compute has finished.
//
// Also: the K == 0 kernel that writes the empty-sum zeros.
#include "f32_tile.cuh"

namespace pg {

template <class T, bool ACC>
__global__ void __launch_bounds__(T::kThreads, T::kMinBlocks) gemm_f32_sync_kernel(const F32Args p)
{
    extern __shared__ __align__(1024) float smem[];
    float *sA = smem;
    float *sB = smem + T::kAFloats;

    const int tid = threadIdx.x;
    int m0, n0;
    tile_origin(T::BM, T::BN, m0, n0);
    const int tr = tid / T::kThreadCols;
    const int tc = tid % T::kThreadCols;

    Accum<T> acc;
    init_tile<T, ACC>(p, m0, n0, tr, tc, acc);

    const int k_slices = (p.K + T::BK - 1) / T::BK;
    for (int kt = 0; kt < k_slices; ++kt) {
        const int k0 = kt * T::BK;
        float4 ra[T::kAChunksPerThread];
        float4 rb[T::kBChunksPerThread];
#pragma unroll
        for (int q = 0; q < T::kAChunksPerThread; ++q) {
            int r, k;
            a_chunk_coords<T>(tid + q * T::kThreads, m0, k0, r, k);
            ra[q] = load_chunk_guarded(p.A, p.lda, r, k, p.M, p.K, p.a_vec);
        }
#pragma unroll
        for (int q = 0; q < T::kBChunksPerThread; ++q) {
            int k, n;
            b_chunk_coords<T>(tid + q * T::kThreads, k0, n0, k, n);
            rb[q] = load_chunk_guarded(p.B, p.ldb, k, n, p.K, p.N, p.b_vec);
        }
#pragma unroll
        for (int q = 0; q < T::kAChunksPerThread; ++q)
            *reinterpret_cast<float4 *>(sA + 4 * (tid + q * T::kThreads)) = ra[q];
#pragma unroll
        for (int q = 0; q < T::kBChunksPerThread; ++q)
            *reinterpret_cast<float4 *>(sB + 4 * (tid + q * T::kThreads)) = rb[q];
        __syncthreads();

        compute_tile<T>(sA, sB, tr, tc, acc);
        __syncthreads();
    }

    store_tile<T>(p, m0, n0, tr, tc, acc);
}

// C = 0 for an empty K (the sum over no terms).
__global__ void gemm_f32_zero_kernel(const F32Args p)
{
    const long long total = static_cast<long long>(p.M) * p.N;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = idx / p.N;
        const long long c = idx % p.N;
        p.C[r * p.ldc + c] = 0.0f;
    }
}

template <class T, bool ACC>
static int launch_sync_acc(const F32Args &a, cudaStream_t s)
{
    const int smem = T::kStageBytes;
    static std::atomic<unsigned long long> limit_set[kMaxDevices];
    if (ensure_smem_limit(gemm_f32_sync_kernel<T, ACC>, smem, a.device, a.ctx, limit_set) != GEMM_OK)
        return GEMM_ERR_CUDA;
    const dim3 grid((a.N + T::BN - 1) / T::BN, (a.M + T::BM - 1) / T::BM);
    gemm_f32_sync_kernel<T, ACC><<<grid, T::kThreads, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

template <class T>
static int launch_sync_t(const F32Args &a, cudaStream_t s)
{
    return a.accumulate ? launch_sync_acc<T, true>(a, s) : launch_sync_acc<T, false>(a, s);
}

int launch_f32_sync(const F32Args &a, cudaStream_t s)
{
    if (a.tile == 32)
        return launch_sync_t<TileXS>(a, s);
    return a.tile == 128 ? launch_sync_t<TileL>(a, s) : launch_sync_t<TileS>(a, s);
}

int launch_f32_zero(const F32Args &a, cudaStream_t s)
{
    const long long total = static_cast<long long>(a.M) * a.N;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096)
        blocks = 4096;
    if (blocks < 1)
        blocks = 1;
    gemm_f32_zero_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

} // namespace pg
