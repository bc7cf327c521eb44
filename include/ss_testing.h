/*
 * ss_testing.h - test hook of libss.so (not for production use).
 *
 * There is no counterpart on the pages: these exist so the test suite can
 * check the library's failure path without faulting or hanging a GPU, and
 * run each kernel variant on shapes the planner would give to another.
 */
#ifndef SS_TESTING_H
#define SS_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * The next launch of ss_affine_scan, ss_selective_scan_fwd or
 * ss_selective_scan_bidir lets work unit `unit` (affine: tile index; S6:
 * sequence * chunks + chunk, chunked launches only) skip publishing its
 * look-back descriptors. Units that wait on it give up after the spin
 * timeout (ss_set_spin_timeout_ns), record SS_ERR_TIMEOUT in the workspace
 * and finish; the output of that launch is undefined. The request applies
 * to one launch and is then cleared. unit < 0 clears a pending request.
 */
void ss_testing_skip_publish_once(int64_t unit);

/*
 * Forces the plan the S6 forward, state and bidirectional calls (and their
 * workspace-size queries) use from now on, so tests can run every code path
 * on any shape. kind 0 restores the planner's own choice. kind 1: the
 * chunked kernel with `a` warps per CTA along time and `b` timesteps per
 * warp (a == b == 0: the planner's values) and `c` lanes per channel (2 or
 * 4; 0 or 1: one); kind 2: the time-parallel single pass with `a` channels
 * per warp, `b` steps per lane and `c` warps per CTA (built variants: a in
 * {2, 4, 8}, b in {7, 9}); kind 3: the wavefront single pass with `a` steps
 * per warp slice and `b` slices (warps) per CTA (built: (9, 4), (11, 4),
 * (13, 4), (15, 4), (9, 2), (13, 2)). Kinds 2 and 3 apply to forward calls only (else the
 * planner's choice applies). A workspace sized under one setting is only valid under that
 * setting; calls made while another thread changes it may take either.
 */
void ss_testing_s6_plan(int kind, int a, int b, int c);

/*
 * Describes the plan an S6 call of this shape would use under the current
 * setting: returns 2 for the wavefront single pass (out = steps per slice,
 * slices per CTA, channels per CTA, blocks per sequence, CTAs, steps per
 * block), 1 for the time-parallel single pass (out = channels per
 * warp, steps per lane, warps per CTA, blocks per sequence, CTAs, steps per
 * block), 0 for the chunked kernel (out = lanes per channel, warps per CTA,
 * timesteps per warp, chunks per sequence, CTAs, states per lane), -1 for an
 * invalid shape. out: six host int64 values.
 */
int ss_testing_s6_describe_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_dtype,
                                int bidir, int64_t *out);

/*
 * Runs the layer's projection GEMM alone, so tests can compare it with the
 * oracle's projections directly: out (M x Nout bf16, row stride ld_out
 * elements) = x (M x K bf16, row-major) times W (Nout x K bf16, row-major)
 * transposed, fp32 accumulation, bias[j] (fp32, device) added to columns
 * j < n_bias (bias may be null) before the one rounding to bf16. Columns
 * from Nout up to the next multiple of 8 may be written (the output leaves
 * as 16-byte tile stores); columns from there to ld_out are left untouched.
 * workspace: a zero-filled device block of at least 256 bytes (its header
 * takes device errors, read with ss_get_device_status). Returns
 * SS_ERR_UNSUPPORTED unless K and ld_out are multiples of 8, ld_out >= Nout,
 * M, K and Nout are at most 2^31 - 256 (tile coordinates are 32-bit) and x,
 * W, out are 16-byte aligned. Asynchronous on `stream`.
 */
int ss_testing_proj_gemm(const void *x, const void *W, void *out, const float *bias,
                         int64_t n_bias, int64_t M, int64_t K, int64_t Nout, int64_t ld_out,
                         void *workspace, void *stream);

/*
 * Describes the launch plan of ss_testing_proj_gemm (and of the bf16 layer's
 * projections) for an M x K by Nout x K product, on the host, without a GPU:
 * out = eight host int64 values {N-tile width BN, N-tiles, K-columns per
 * shared-memory stage, K-blocks, stages, 1 if CTA pairs share one M = 256
 * MMA (two M-blocks or more) else 0, work units (tiles, or tile pairs),
 * dynamic shared memory bytes per CTA}. Returns 0, or -1 for a shape with a
 * size <= 0 or above 2^31 - 256, or a null out.
 */
int ss_testing_proj_gemm_describe_plan(int64_t M, int64_t K, int64_t Nout, int64_t *out);

#ifdef __cplusplus
}
#endif

#endif /* SS_TESTING_H */
