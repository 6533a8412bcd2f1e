/*
 * GEMM oracle: TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct CPU reference for C = A * B.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load this
 * library; the CUDA product path never calls it and shares no code with it.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no -ffast-math).
 * -ffp-contract=off keeps every `a * b + c` below a separate multiply and add;
 * the only fused operation is the explicit fmaf() of the FP32 mirror.
 *
 * Conventions: all matrices row-major, element (r, c) of X at X[r * ldx + c];
 * the caller owns every buffer; nothing is allocated here.  OpenMP threads
 * split output rows only, so each element's summation order is fixed whatever
 * the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * The definition C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j], accumulated in
 * double, k ascending for every element, i-p-j loop order.
 *
 * Follows the CPU reference of "pipelined_gemm.cu" (the day-74 lesson's
 * program, section "CPU reference": plain loops, double accumulation, caller
 * owns the buffers), generalised to M x N x K with leading dimensions.
 * A float32 x float32 product is exact in double (24 + 24 <= 53 significand
 * bits), so the only rounding is the double addition.
 */
void oracle_gemm_f64(long M, long N, long K,
                     const float *A, long lda,
                     const float *B, long ldb,
                     double *C, long ldc)
{
    long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; ++i) {
        double *c = C + i * ldc;
        long j, p;
        for (j = 0; j < N; ++j)
            c[j] = 0.0;
        for (p = 0; p < K; ++p) {
            const double a = (double)A[i * lda + p];
            const float *b = B + p * ldb;
            for (j = 0; j < N; ++j)
                c[j] += a * (double)b[j];
        }
    }
}

/*
 * FP32 mirror of the kernels' arithmetic: every C element is one float32
 * fused multiply-add chain over k ascending, starting from +0.
 *
 * Follows "pipelined_gemm.cu", section "computeTile" (the inner product both
 * kernels share: per K step p each thread's accumulator gets one product
 * added, p ascending within a slice and slices ascending), and "Day 74: Async
 * copies and pipelines", section "Two kernels, one arithmetic" (identical
 * floating-point operations in an identical order).  The fused form is the
 * one CUDA emits for `acc += a * b` at its default contraction setting.
 */
void oracle_gemm_fmaf_chain(long M, long N, long K,
                            const float *A, long lda,
                            const float *B, long ldb,
                            float *C, long ldc)
{
    long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; ++i) {
        float *c = C + i * ldc;
        long j, p;
        for (j = 0; j < N; ++j)
            c[j] = 0.0f;
        for (p = 0; p < K; ++p) {
            const float a = A[i * lda + p];
            const float *b = B + p * ldb;
            for (j = 0; j < N; ++j)
                c[j] = fmaf(a, b[j], c[j]);
        }
    }
}

/* bfloat16 bit pattern -> float32, exactly (bfloat16 is the top half of a float32). */
static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * BF16 inputs, exact products, double accumulation: the same definition as
 * oracle_gemm_f64 with each bfloat16 operand widened exactly.  The BF16 path
 * is the tensor-core form of the pipelined GEMM ("异步拷贝与现代 Pipeline",
 * section 6.1 "BF16 GEMM 的异步拷贝": BF16 operands, FP32 accumulation); the
 * reference result is the exact-product sum.
 */
void oracle_gemm_bf16_f64(long M, long N, long K,
                          const uint16_t *A, long lda,
                          const uint16_t *B, long ldb,
                          double *C, long ldc)
{
    long i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < M; ++i) {
        double *c = C + i * ldc;
        long j, p;
        for (j = 0; j < N; ++j)
            c[j] = 0.0;
        for (p = 0; p < K; ++p) {
            const double a = (double)bf16_to_float(A[i * lda + p]);
            const uint16_t *b = B + p * ldb;
            for (j = 0; j < N; ++j)
                c[j] += a * (double)bf16_to_float(b[j]);
        }
    }
}

/* Threads OpenMP will use for the loops above (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
