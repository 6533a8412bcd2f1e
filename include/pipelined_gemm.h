/*
 * pipelined_gemm.h -- C ABI of the GB300 (sm_103a) pipelined GEMM library.
 *
 * The operation is the register-tiled GEMM of "Day 74: Async copies and
 * pipelines" (section "Two kernels, one arithmetic") and its program
 * "pipelined_gemm.cu": C = A * B, where the block's shared-memory tiles are
 * filled one 16-deep K slice at a time and the fill is the only thing that
 * differs between variants.  Three fills are offered:
 *
 *   GEMM_FILL_SYNC     register path: global -> register -> shared, then a
 *                      CTA barrier ("pipelined_gemm.cu", matmulTileSync;
 *                      day 74, "A copy that skips the registers").
 *   GEMM_FILL_CPASYNC  cp.async global -> shared with commit_group /
 *                      wait_group completion ("A study on CUDA async
 *                      memcpy", section "async-group based approach";
 *                      day 74, "Two kernels, one arithmetic").
 *   GEMM_FILL_TMA      one producer warp issues TMA bulk-tensor copies into
 *                      a ring of stages guarded by full/empty mbarriers
 *                      ("A study on CUDA async memcpy", sections "mbarrier
 *                      based approach" and "block-scoped pipeline"; the
 *                      producer/consumer split of its "Real world example").
 *   GEMM_FILL_CPASYNC_MBAR
 *                      cp.async whose completion is tracked by a full/empty
 *                      mbarrier ring (cp.async.mbarrier.arrive.noinc): the
 *                      form the lesson's block-scoped cuda::pipeline lowers
 *                      to (day 74, "Results"; "A study on CUDA async
 *                      memcpy", "block-scoped pipeline").  Every thread
 *                      copies and computes; no CTA barrier in the loop.
 *   GEMM_FILL_CPASYNC_WS
 *                      the same cp.async copies and mbarrier completion,
 *                      issued by one or four dedicated producer warps while
 *                      the other warps only compute ("A study on CUDA async
 *                      memcpy", "block-scoped pipeline": producers and
 *                      consumers need not be the same threads).  FP32 only.
 *
 * Every FP32 fill runs the same per-thread FMA micro-kernel, so for every C
 * element the result is one float32 fused multiply-add chain over k
 * ascending, starting from +0: the three fills are bit-identical to each
 * other (the pages' memcmp invariant) and to that chain.
 *
 * Layout: all matrices row-major.  A is M x K with leading dimension lda
 * (element (i,k) at A[i*lda + k]), B is K x N with ldb, C is M x N with ldc.
 * Elements beyond the logical extents (ragged tiles) are read as zero
 * ("cp.async", section "Predication is different from zero fill": a partial
 * source size copies a prefix and zero-fills the rest); padding columns
 * between K and lda are never read.
 *
 * Ownership: every pointer is a device pointer owned by the caller; the
 * library keeps no reference after the call returns.  The entry points
 * allocate no memory.  The library cannot check two preconditions, and
 * breaking either is undefined behaviour: A, B and C are memory of the
 * current device (cudaSetDevice), and C shares no byte with A or B (other
 * blocks still read A and B while C tiles are written).
 *
 * Asynchrony: gemm_f32 / gemm_bf16 enqueue one kernel on `stream` (a
 * cudaStream_t; NULL means the legacy default stream) and return without
 * synchronising.  C is valid once the stream has reached that point.
 *
 * Errors: a status code is returned; nothing is enqueued unless the status
 * is GEMM_OK.  The library never exits the process and never falls back
 * silently from one fill to another.  A kernel whose internal wait exceeds
 * its time limit (2 s) records GEMM_ERR_TIMEOUT in a device status word,
 * which gemm_device_status() reads: a caller of the device path checks it
 * before trusting C.  Test hooks that make those waits expire on purpose are
 * declared in pipelined_gemm_testing.h.
 */
#ifndef PIPELINED_GEMM_H
#define PIPELINED_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum gemm_fill_mode {
    GEMM_FILL_SYNC = 0,
    GEMM_FILL_CPASYNC = 1,
    GEMM_FILL_TMA = 2,
    GEMM_FILL_CPASYNC_MBAR = 3,
    GEMM_FILL_CPASYNC_WS = 4
};

/*
 * Optional cache qualifiers, OR-ed into a call's fill_mode.  Off by default;
 * none changes a result bit.  They are the two qualifiers the "cp.async"
 * tile-op reference lists: the prefetch size of the operand contract
 * (.L2::64B / 128B / 256B; 128 B is offered) and the cache_policy call
 * parameter (an L2 eviction priority carried by .L2::cache_hint).
 *
 *   GEMM_OPT_L2_PREFETCH_128B   every 16-byte cp.async copy also prefetches
 *                               its 128-byte L2 line (cp.async fills only).
 *   GEMM_OPT_{A,B}_EVICT_FIRST  copies of A (or B) carry an evict_first /
 *   GEMM_OPT_{A,B}_EVICT_LAST   evict_last L2 policy (cp.async and TMA fills).
 *
 * Asking for both priorities of one operand, an option a fill does not
 * take (the register-path fill takes none), or an unknown bit returns
 * GEMM_ERR_INVALID_ARG.  An L2 policy on a cp.async fill whose A or B rows
 * are not 16-byte aligned (so copied 4 bytes at a time) returns
 * GEMM_ERR_UNSUPPORTED: the 4-byte copies take the prefetch size only.
 */
/*
 * GEMM_OPT_ACCUMULATE (FP32 only; gemm_bf16 returns GEMM_ERR_UNSUPPORTED):
 * C = C + A·B with each element's FMA chain starting from the value C holds
 * instead of +0: C's value, then one fused multiply-add per k, ascending.
 * If C holds the result of an earlier call over the first K0 columns of A
 * and rows of B, a call over the remaining columns and rows with this
 * option gives, bit for bit, what one call over all of them gives.  The
 * pages have no counterpart: the host-buffer path uses it to start on the
 * first rows of C while B is still arriving in row blocks.  With K = 0 the
 * call leaves C as it is.  It does not combine with the cache qualifiers
 * above (GEMM_ERR_UNSUPPORTED).  A starting value of -0 may come out as +0 where
 * a zero-filled K tail adds +0 to it; a chain started from +0 never holds -0.
 */
enum gemm_fill_option {
    GEMM_OPT_L2_PREFETCH_128B = 0x100,
    GEMM_OPT_A_EVICT_FIRST = 0x200,
    GEMM_OPT_A_EVICT_LAST = 0x400,
    GEMM_OPT_B_EVICT_FIRST = 0x800,
    GEMM_OPT_B_EVICT_LAST = 0x1000,
    GEMM_OPT_ACCUMULATE = 0x2000,
    GEMM_OPT_MASK = 0x3F00
};

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* bad size, leading dimension, pointer, fill, stages or tile   */
    GEMM_ERR_MISALIGNED = 2,  /* TMA needs 16-byte aligned bases and row pitches              */
    GEMM_ERR_UNSUPPORTED = 3, /* valid request the library does not implement                 */
    GEMM_ERR_ARCH = 4,        /* current device is not compute capability 10.3 (sm_103a)      */
    GEMM_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed (launch, attribute, ...)   */
    GEMM_ERR_TIMEOUT = 6      /* a kernel's bounded wait expired (read via gemm_device_status) */
} gemm_status;

/* What a call would launch.  Filled by gemm_f32_plan / gemm_bf16_plan. */
typedef struct gemm_plan {
    int fill_mode;       /* GEMM_FILL_*                                                */
    int block_m;         /* CTA tile rows                                              */
    int block_n;         /* CTA tile columns                                           */
    int block_k;         /* K slice depth per pipeline stage                           */
    int thread_m;        /* micro-tile rows per thread (FP32); 0 for the tensor path   */
    int thread_n;        /* micro-tile columns per thread (FP32); 0 for tensor path    */
    int threads;         /* threads per CTA, including any producer / MMA warps        */
    int stages;          /* shared-memory stages in the ring (1 for the sync fill)     */
    int a_copy_bytes;    /* bytes per copy instruction for A: 16 (float4 / cp.async.cg),
                            4 (scalar / cp.async.ca, used when A rows are not 16-byte
                            aligned), or the TMA box size in bytes                    */
    int b_copy_bytes;    /* same for B                                                 */
    int smem_bytes;      /* dynamic shared memory per CTA                              */
    int grid_x;          /* CTAs launched along x                                      */
    int grid_y;          /* CTAs launched along y                                      */
    int k_slices;        /* ceil(K / block_k)                                          */
    int options;         /* the GEMM_OPT_* bits the call carries                       */
    int persistent_ctas; /* FP32: CTAs of the split-region kernel gemm_f32_ws would add
                            (one per SM, each walking several tile pieces), or 0;
                            BF16: CTAs of the persistent kernel                      */
    int workspace_bytes; /* device workspace gemm_f32_ws / gemm_bf16_ws can use to split
                            the last round of tiles in K (0: nothing to split)         */
    int wide_rows;       /* FP32 TMA fill, 128x128 tile: rows [0, wide_rows) of C that
                            the call computes on 128x256 tiles (8x16 micro-tile, 256
                            threads, 4 stages, no producer warp) before the 128x128
                            path computes the rest; 0 when the wide kernel would not
                            shorten the call (K < 1024, cache options, or no cut in
                            whole rounds of wide tiles that gains 1 %).  grid_x and
                            grid_y still count the 128x128 tiles of the whole C;
                            persistent_ctas and workspace_bytes describe the rows
                            below wide_rows.  Same bits either way.           */
} gemm_plan;

/*
 * gemm_f32: C[M x N] = A[M x K] * B[K x N], float32 in and out.
 *
 *   M, N, K     logical sizes, >= 0.  M == 0 or N == 0 is a no-op; K == 0
 *               writes zeros to C (an empty sum), or with
 *               GEMM_OPT_ACCUMULATE leaves C as it is.
 *   A, lda      device pointer, leading dimension >= max(K, 1).
 *   B, ldb      device pointer, leading dimension >= max(N, 1).
 *   C, ldc      device pointer, leading dimension >= max(N, 1).  Only the
 *               M x N logical elements are written; columns N..ldc-1 are
 *               left untouched.
 *   fill_mode   GEMM_FILL_SYNC, GEMM_FILL_CPASYNC, GEMM_FILL_TMA,
 *               GEMM_FILL_CPASYNC_MBAR or GEMM_FILL_CPASYNC_WS, optionally
 *               OR-ed with GEMM_OPT_* cache qualifiers and
 *               GEMM_OPT_ACCUMULATE (C = C + A·B).
 *   stages      sync: 0 or 1.  Others: 2..6, or 0 for the default: 4, or 2
 *               for GEMM_FILL_CPASYNC_WS and for GEMM_FILL_TMA on the
 *               128x128 tile.
 *               Each stage is one more slice in flight
 *               and one more copy of both tiles in shared memory (day 74,
 *               "Exercise").
 *   block_tile  64 (64x64 tile, 4x4 micro-tile per thread, 256 threads: the
 *               lesson's shape), 128 (128x128 tile, 8x8 micro-tile, 256
 *               threads), 32 (32x32 tile, 8x4 micro-tile, one warp: the
 *               latency-bound shape of "A study on CUDA async memcpy",
 *               "Real world example"), or 0 to let the library choose by
 *               problem size (64 or 128).  With GEMM_FILL_TMA and 128, a
 *               large call may compute its top rows on 128x256 tiles
 *               (gemm_plan.wide_rows) before the 128x128 tiles below them;
 *               the bits are the same.
 *   stream      cudaStream_t to enqueue on.
 *
 * Alignment: the sync and both cp.async fills accept any lda/ldb; rows that are
 * not 16-byte aligned are copied with 4-byte operations (reported by
 * gemm_f32_plan).  The TMA fill requires A and B 16-byte aligned and
 * lda, ldb multiples of 4 (row pitch a multiple of 16 bytes); otherwise it
 * returns GEMM_ERR_MISALIGNED.
 *
 * Returns GEMM_OK or an error code (nothing enqueued on error).
 */
int gemm_f32(int M, int N, int K,
             const float *A, int lda,
             const float *B, int ldb,
             float *C, int ldc,
             int fill_mode, int stages, int block_tile,
             void *stream);

/*
 * gemm_f32_ws: gemm_f32 with an optional device workspace.
 *
 * With the TMA fill's 128 x 128 tile, one CTA computes one tile, in rounds
 * of one tile per SM.  When the tile count is not a multiple of the SM
 * count, the last round would leave SMs idle.  Given `workspace`, the
 * rounds but the last run as usual and the remaining
 * SMs + (tiles mod SMs) tiles go to a second, persistent kernel of one CTA
 * per SM (plan.persistent_ctas), launched right after on the same stream,
 * which shares them out in equal runs of K slices.  A tile cut between two
 * CTAs is computed in K order: the first computes its first slices and
 * hands its float32 accumulators over through the workspace, the second
 * continues from them.  Every element is still the same fused multiply-add
 * chain over k ascending, so the result is bit for bit that of gemm_f32.
 *
 *   workspace        device memory of the current device, 16-byte aligned,
 *                    at least plan.workspace_bytes long (gemm_f32_plan), or
 *                    NULL to run without the split (exactly gemm_f32).  It
 *                    needs no initialisation and holds nothing between calls,
 *                    but one workspace serves one call at a time: calls that
 *                    may overlap on the GPU (other streams) need their own.
 *                    Ignored when plan.workspace_bytes is 0.
 *   workspace_bytes  its size; smaller than needed: GEMM_ERR_INVALID_ARG.
 *
 * A CTA waits (bounded) for the CTA before it to hand a tile over; CTAs
 * start in index order, so the one it waits for is running or done.  If
 * the wait expires, GEMM_ERR_TIMEOUT is recorded (role 6) as for any wait.
 * Other arguments, errors and ownership as gemm_f32.
 *
 * CUDA graphs: a hand-over's ready flag carries a value fixed when the call
 * is made, which a captured graph replays unchanged; each flag's one reader
 * lowers it to 0 once it has seen it, so a call that completes leaves every
 * flag at 0 and a replay waits for its own hand-overs.  A call that ended
 * with GEMM_ERR_TIMEOUT may leave a flag raised: clear the workspace's flags
 * (the last ctas x 8 bytes of plan.workspace_bytes) before replaying a graph
 * that uses it.  The same holds for gemm_bf16_ws.
 */
int gemm_f32_ws(int M, int N, int K,
                const float *A, int lda,
                const float *B, int ldb,
                float *C, int ldc,
                int fill_mode, int stages, int block_tile,
                void *workspace, size_t workspace_bytes,
                void *stream);

/*
 * gemm_f32_noalloc: gemm_f32_ws for callers that cannot allocate device
 * memory -- an allocator that needs a GEMM while it is serving a request
 * (cudaMalloc cannot be re-entered from there), code that runs on a fixed,
 * pre-planned memory budget, or latency-bound code that must not call
 * cudaMalloc / cudaFree, which may synchronise the whole device.  Not part of
 * the pages' method: they have no counterpart.
 *
 * The split's hand-over space is a fixed array inside this library, sized
 * for up to 160 SMs (10,487,040 bytes); every GPU that loads the library
 * holds it until the process exits.  The call itself allocates and frees
 * nothing.  Arguments, results and errors as gemm_f32, plus:
 *   - GEMM_ERR_UNSUPPORTED when the current device has more SMs than the
 *     array has room for (a call with nothing to split still runs);
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress), so make it before any stream capture;
 *   - every call shares the one array.  It keeps the last call's contents,
 *     and none of them needs clearing (each call's ready flags carry a value
 *     no earlier call used), but calls that overlap on the GPU -- on other
 *     streams, or from other host threads -- race on it: serialise them.
 */
int gemm_f32_noalloc(int M, int N, int K,
                     const float *A, int lda,
                     const float *B, int ldb,
                     float *C, int ldc,
                     int fill_mode, int stages, int block_tile,
                     void *stream);

/*
 * gemm_f32_host: C = A·B in FP32 with A, B and C in HOST memory (page-locked
 * for the copies to overlap; pageable memory works but each copy then waits
 * for the host).  The pages measure device-resident operands; this entry
 * point is the library's own host-buffer path, not a counterpart of theirs.
 *
 *   M, N, K, fill_mode, stages, block_tile
 *               as gemm_f32 (block_tile 0 picks the whole problem's tile).
 *               GEMM_OPT_ACCUMULATE in fill_mode is refused: the executor
 *               uses it itself.
 *   A, B, C     host pointers, 4-byte aligned; only the M x N logical
 *               elements of C are written.
 *   lda, ldb, ldc  row pitches in floats, at least max(K, 1), max(N, 1),
 *               max(N, 1).  Any pitch works for every fill: the GEMMs read
 *               device copies laid out at 16-byte row pitches.
 *   scratch     device memory of at least gemm_f32_host_scratch() bytes,
 *               256-byte aligned, owned by the caller: device copies of A,
 *               B and C and the K-split hand-over spaces.  Nothing in it
 *               needs clearing, and it may be reused by the next call.
 *   status_out  host pointer or NULL.  If given, the call's last step
 *               copies the device status word there and clears it (as
 *               gemm_device_status does, without synchronising): once
 *               `stream` has reached the end of the call, *status_out is 0
 *               or the family | role word of the first bounded wait that
 *               gave up, in which case C is undefined.  Page-locked memory
 *               keeps that copy asynchronous.
 *   stream      the call starts after the work already on `stream`, and
 *               `stream` waits for its end; it returns without waiting.
 *               A, B, C, scratch and status_out must stay valid, and A and
 *               B unchanged, until `stream` has reached that point.
 *
 * Work runs on three streams the library makes per device and context
 * (copies in, GEMMs, copies out), ordered by events: B's rows and A's
 * columns cross the link in K blocks, each block's GEMM over all rows
 * starts as soon as it has landed and continues every element's FMA chain
 * from the previous block's C (GEMM_OPT_ACCUMULATE), and the last block runs
 * in row chunks, each copied out as soon as it is done (K under 2048: one
 * block, with A moved chunk by chunk).  Its blocks: 512, then up to 2048
 * each, the last 2048 or a little more; its row chunks: about two waves of
 * 128x128 tiles each, the last about one (gemm_f32_host_schedule).  The result is bit-identical to
 * gemm_f32 on the same fill.  Calls on one device are serialised: each
 * starts after the previous one has finished on the GPU.  Kernel timeouts
 * are recorded in the status word as for gemm_f32 (see status_out).
 * Returns GEMM_OK or an error (GEMM_ERR_INVALID_ARG for a missing or small
 * scratch, GEMM_ERR_MISALIGNED for a misaligned one); after an error some
 * work may already be enqueued, and `stream` still waits for it.
 */
int gemm_f32_host(int M, int N, int K,
                  const float *A, int lda,
                  const float *B, int ldb,
                  float *C, int ldc,
                  int fill_mode, int stages, int block_tile,
                  void *scratch, size_t scratch_bytes,
                  unsigned int *status_out,
                  void *stream);

/* gemm_f32_host_scratch: device bytes gemm_f32_host needs for these sizes on
 * the current device (*bytes, a host pointer).  No device memory is touched. */
int gemm_f32_host_scratch(int M, int N, int K, size_t *bytes);

/* gemm_f32_host_schedule: the cut gemm_f32_host makes for these sizes on
 * `sms` SMs, without touching the device: K-block bounds k_bounds[0..*n_k]
 * (0 = k_bounds[0] < ... < k_bounds[*n_k] = K) and the row-chunk bounds of
 * the last block, row_bounds[0..*n_rows] (0 ... M).  k_cap and row_cap are
 * the arrays' lengths; GEMM_ERR_INVALID_ARG if either is too short (17 and
 * 65 always suffice). */
int gemm_f32_host_schedule(int M, int N, int K, int sms,
                           int *k_bounds, int k_cap, int *n_k,
                           int *row_bounds, int row_cap, int *n_rows);

/* gemm_f32_plan: validate exactly as gemm_f32 does and describe the launch it
 * would make, without touching the device.  `plan` is a host pointer. */
int gemm_f32_plan(int M, int N, int K,
                  const float *A, int lda,
                  const float *B, int ldb,
                  float *C, int ldc,
                  int fill_mode, int stages, int block_tile,
                  gemm_plan *plan);

/*
 * gemm_bf16: C[M x N] (float32) = A[M x K] * B[K x N] with bfloat16 operands
 * given as raw uint16 bit patterns, products and sums on the 5th-generation
 * tensor cores (tcgen05.mma, float32 accumulation in tensor memory).  This
 * is the tensor-core form of the same pipelined GEMM ("异步拷贝与现代
 * Pipeline", section 6.1 "BF16 GEMM 的异步拷贝": prefetch the next K tile
 * while the tensor cores work on the current one).
 *
 *   fill_mode   GEMM_FILL_TMA (one thread issues 2-D tensor copies),
 *               GEMM_FILL_CPASYNC (eight producer warps copy 16-byte
 *               chunks with cp.async into the same swizzled stages), or
 *               GEMM_FILL_SYNC (the register path: sixteen producer warps
 *               load and store, one stage, loads and MMAs alternate).
 *               GEMM_FILL_CPASYNC_MBAR and GEMM_FILL_CPASYNC_WS return
 *               GEMM_ERR_UNSUPPORTED.
 *   stages      TMA / cp.async: 2..4 with the 128-row tile (4 x 48 KiB
 *               stages fill shared memory), 2..3 with the 256-row tile
 *               (64 KiB stages), or 0 for the tile's default (4 or 3).
 *               sync: 0 or 1.
 *   block_m     rows per CTA tile, every tile 256 columns wide:
 *               128 (one 128 x 256 accumulator per tile, two in tensor
 *               memory so a tile's stores overlap the next tile's MMAs),
 *               256 (two 128-row MMAs share each B slice: the fill writes
 *               a third fewer shared-memory bytes per multiply-add; one
 *               tile in tensor memory at a time), or 0 to let the library
 *               choose: 128
 *               when stages is 4, else whichever tile needs less time for
 *               its waves of persistent CTAs over the current device's SMs
 *               (152 when no device can be asked), a 256-row tile counting
 *               as 2 / 1.08 waves of the 128-row tile.  Anything else, or
 *               256 with 4 stages, is GEMM_ERR_INVALID_ARG.  Every fill and
 *               both tiles give bit-identical results.
 *   Alignment   A, B 16-byte aligned; lda, ldb multiples of 8 (16-byte row
 *               pitch), else GEMM_ERR_MISALIGNED.  C needs 4-byte alignment;
 *               a 16-byte aligned C with ldc a multiple of 4 is written by
 *               TMA stores, any other C by plain stores.
 *   Accuracy    the tensor core's internal summation order is its own, so
 *               results are not bit-identical to a sequential sum; they
 *               match the exact-product sum within float32 rounding.
 * Other arguments, sizes and ownership as gemm_f32.
 */
int gemm_bf16(int M, int N, int K,
              const uint16_t *A, int lda,
              const uint16_t *B, int ldb,
              float *C, int ldc,
              int fill_mode, int stages, int block_m,
              void *stream);

/*
 * gemm_bf16_ws: gemm_bf16 with hand-over space for the TMA fill's K split of
 * the last round of tiles, as gemm_f32_ws does for FP32.  When the tile
 * count is not a multiple of the SM count, the persistent CTAs share the
 * last round and one more as equal runs of 64-deep K blocks; a tile cut
 * between two CTAs is computed in K order, the second continuing from the
 * first one's FP32 accumulators, which cross through `workspace` (read
 * back into tensor memory), so the tensor cores issue the same MMAs on the
 * same accumulator values as without the split: every result bit is
 * unchanged.
 *
 *   workspace, workspace_bytes
 *               device memory of at least gemm_plan.workspace_bytes
 *               (gemm_bf16_plan; one block_m x 256 FP32 tile and an 8-byte
 *               flag per SM, 0 when the call has nothing to split), 16-byte
 *               aligned, owned by the caller; nothing in it needs clearing.
 *               NULL (or a call with nothing to split, or a fill other than
 *               TMA) runs without the split.
 *
 * Calls that overlap on the GPU must not share a workspace.  Returns as
 * gemm_bf16, plus GEMM_ERR_INVALID_ARG for a workspace smaller than the plan
 * asks and GEMM_ERR_MISALIGNED for a misaligned one.
 *
 * Unlike the FP32 split, this one does not pay on GB300 at 8192^3: each
 * split tile adds an accumulator drain to global memory and a load back
 * into tensor memory that the MMAs wait for, and on the 256-row tile (whose
 * epilogue does not overlap the next tile's MMAs) that costs more than the
 * idle SMs of the partial last round (603 against 584 us; 128-row tile 647
 * against 651 us; 4096 x 4096 x 8192, 128 rows: 181 against 191 us).
 * gemm_bf16 therefore runs without it.
 */
int gemm_bf16_ws(int M, int N, int K,
                 const uint16_t *A, int lda,
                 const uint16_t *B, int ldb,
                 float *C, int ldc,
                 int fill_mode, int stages, int block_m,
                 void *workspace, size_t workspace_bytes,
                 void *stream);

/* gemm_bf16_plan: validate exactly as gemm_bf16 does and describe the launch
 * it would make.  With block_m = 0 it asks the current device for its SM
 * count (152 if there is none); it launches nothing.  `plan` is a host
 * pointer. */
int gemm_bf16_plan(int M, int N, int K,
                   const uint16_t *A, int lda,
                   const uint16_t *B, int ldb,
                   float *C, int ldc,
                   int fill_mode, int stages, int block_m,
                   gemm_plan *plan);

/* Human-readable name of a status code (static storage; never NULL). */
const char *gemm_status_string(int status);

/*
 * gemm_device_status: synchronise `stream`, then read and clear the current
 * device's status word.  Returns GEMM_OK, GEMM_ERR_TIMEOUT (a kernel gave up
 * on a wait and returned early; its C output is undefined), or
 * GEMM_ERR_CUDA if the synchronisation itself failed.  If `detail` is not
 * NULL it receives the raw word (0 when clean): bits 0-7 the kernel family
 * (1 FP32 TMA, 2 BF16, 3 self-test, 4 FP32 mbarrier-completed cp.async,
 * 5 FP32 cp.async from producer warps, 6 FP32 TMA wide-row kernel),
 * bits 8-15 the waiting role (1 consumer, 2 producer, 3 MMA issuer,
 * 4 epilogue, 5 drain of copies or MMAs still in flight, 6 hand-over of
 * accumulators between CTAs in gemm_f32_ws).
 *
 * The word is ONE per device (per CUDA context), shared by every call on
 * every stream and every host thread.  A kernel records only the first
 * expiry after the last clear.  Consequences:
 *   - the synchronisation covers only work ordered before this point of
 *     `stream`; a kernel on another stream that has not finished yet may
 *     still record an expiry after the read;
 *   - the read and the clear are two separate steps, so an expiry recorded
 *     between them by a kernel on another stream is lost, and calls that
 *     overlap on the GPU race on the word: whichever caller reads first
 *     sees (and clears) the other's error.
 * Callers that need a status per call serialise their GEMMs on one stream
 * and call gemm_device_status after each.  GEMM results on the device path
 * are only known good once gemm_device_status has returned GEMM_OK for a
 * point after them.
 */
int gemm_device_status(void *stream, unsigned int *detail);

/*
 * gemm_selftest_bounded_wait: launch one CTA whose thread waits on an
 * mbarrier that nothing ever arrives on, with the same bounded-wait routine
 * the GEMM kernels use and a limit of `timeout_us` microseconds (1..1000000).
 * The kernel records GEMM_ERR_TIMEOUT in the status word and returns; read it
 * with gemm_device_status.  Exists so tests can exercise the timeout path
 * without ever hanging or faulting the GPU.
 */
int gemm_selftest_bounded_wait(int timeout_us, void *stream);

/* Library version, major * 10000 + minor * 100 + patch. */
int gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PIPELINED_GEMM_H */
