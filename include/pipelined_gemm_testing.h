/*
 * pipelined_gemm_testing.h -- test hooks of the pipelined GEMM library.
 *
 * Not for production use.  The hooks exist so that a test can make the GEMM
 * kernels' own bounded waits expire, and check that each kernel gives up,
 * reports GEMM_ERR_TIMEOUT, waits for its own copies and tensor-core work
 * still in flight, frees its tensor memory and returns, leaving the CUDA
 * context usable.  No GPU is faulted, trapped or hung to do so: a producer
 * simply never fills one ring position, the way a partial commit would
 * strand the block ("Day 74: Async copies and pipelines", section
 * "Pitfalls": a missing commit or arrival leaves the waiting threads
 * waiting forever), and every wait on that position runs into its limit.
 */
#ifndef PIPELINED_GEMM_TESTING_H
#define PIPELINED_GEMM_TESTING_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gemm_testing_set_hooks: process-wide settings that every later gemm_f32 /
 * gemm_bf16 call reads when it is made (calls already enqueued keep theirs).
 *
 *   wait_limit_ns      limit of every bounded wait in the GEMM kernels, in
 *                      nanoseconds; 0 restores the default of 2 s.  Values
 *                      below 1 ms are refused.
 *   withhold_position  ring position (0, 1, 2, ... counted per CTA over all
 *                      of its K slices, and over its tiles for the
 *                      persistent tensor-core kernel) that the producers of
 *                      the FP32 TMA fill (its wide-row kernel included),
 *                      both FP32 mbarrier-completed
 *                      cp.async fills and all three BF16 fills leave
 *                      unfilled: no copy is issued and no arrival (and, for
 *                      TMA, no expected-transaction count) is made for it.
 *                      -1 restores normal operation.  The FP32 sync and
 *                      group-completed cp.async fills have no waits and
 *                      ignore it.
 *
 * With a position withheld, the C output of a call is undefined and the call
 * ends with GEMM_ERR_TIMEOUT in the status word (gemm_device_status).
 * Returns GEMM_OK or GEMM_ERR_INVALID_ARG.  Not thread-safe against
 * concurrent GEMM calls that expect the defaults.
 */
int gemm_testing_set_hooks(unsigned long long wait_limit_ns, int withhold_position);

/*
 * gemm_testing_f32_wide: how later FP32 TMA calls on the 128x128 tile choose
 * their wide rows (gemm_plan.wide_rows): -1 by the measured cost model (the
 * default), 0 never (every row on 128x128 tiles), 1 whenever a cut in whole
 * rounds of 128x256 tiles exists, gain or not.  Results are bit-identical in
 * every mode.  Returns GEMM_OK or GEMM_ERR_INVALID_ARG.  Not thread-safe
 * against concurrent calls that expect the default.
 */
int gemm_testing_f32_wide(int mode);

/*
 * gemm_testing_f32_wide_rows: the wide rows an M x N x K call would take on
 * a device of `sms` SMs in `mode` (as above), computed on the host without a
 * device; -1 for invalid arguments.
 */
int gemm_testing_f32_wide_rows(int M, int N, int K, int sms, int mode);

/*
 * gemm_testing_withhold_handover: with `on` non-zero, every later
 * gemm_f32_ws call whose persistent kernel splits tiles between CTAs
 * computes and stores the handed-over accumulators but never raises the
 * ready flag, so each CTA waiting for one gives up after the wait limit and
 * records GEMM_ERR_TIMEOUT with role 6.  0 restores normal operation.
 * Returns GEMM_OK.
 */
int gemm_testing_withhold_handover(int on);

/*
 * gemm_testing_f32_piece: the work schedule of the persistent FP32 TMA
 * kernel, computed on the host exactly as the kernel computes it: piece
 * `idx` of CTA `cta` when `ctas` CTAs share `tiles` tiles of `k_slices` K
 * slices, with the last round split (`split` non-zero) or not.  Returns 1
 * and fills out[0..4] = {tile, first slice, end slice, starts from handed-over
 * accumulators, hands its accumulators over}, or 0 when the CTA has no such
 * piece (or an argument is out of range).  No device is touched.
 */
int gemm_testing_f32_piece(int tiles, int ctas, int k_slices, int split, int cta, int idx, int *out);

/*
 * gemm_testing_host_policy: override the constants of gemm_f32_host's
 * schedule for later calls (0 keeps a constant's default): the first and
 * last K block, the longest block between them, the shortest K cut into
 * blocks, and the rows of the last and of the other row chunks in hundredths
 * of a wave of 128 x 128 tiles.  Block lengths are rounded up to multiples
 * of 16.  Returns GEMM_OK, or GEMM_ERR_INVALID_ARG for a negative value or
 * a block under 16.  For schedule sweeps and tests only.
 */
int gemm_testing_host_policy(int k_first, int k_last, int k_mid_max, int k_steps_min,
                             int last_rows_waves100, int rows_waves100);

/*
 * gemm_testing_host_streams: how many GEMM streams gemm_f32_host uses (1 to
 * 3; with more than one, row chunk i's GEMMs of every K step run on stream
 * i mod n, so kernels of different chunks can share the GPU), whether its
 * GEMMs split their last round of tiles in K (1) or not (0), and whether
 * its first row chunk is the largest block of rows whose tiles fill whole
 * rounds of SMs (1) or not (0).  0, -1 and -1 restore the defaults.
 * Returns GEMM_OK or GEMM_ERR_INVALID_ARG.  For schedule sweeps and tests
 * only.
 */
int gemm_testing_host_streams(int comp_streams, int split, int round_chunks);

#ifdef __cplusplus
}
#endif

#endif /* PIPELINED_GEMM_TESTING_H */
