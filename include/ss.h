/*
 * ss.h - C ABI of the GB300 selective-scan library (libss.so).
 *
 * The library computes, on one NVIDIA GB300 GPU (sm_103a), the first-order
 * affine recurrence and the Mamba S6 selective-scan forward built on it:
 *
 *   affine scan   h[t] = a[t] * h[t-1] + b[t],  h[-1] = 0
 *                 ("Selective-scan CUDA kernels", persus.netlify.app, opening
 *                 paragraphs: the recurrence is a prefix scan over affine
 *                 pairs, associative but not commutative)
 *
 *   S6 forward    delta' = softplus(delta) if requested, else delta
 *                 dA  = exp(delta' * A[d, n])
 *                 dBx = delta' * Bt[b, t, n] * x[b, t, d]
 *                 h[n] = dA * h[n] + dBx,  h starts at 0
 *                 y[b, t, d] = sum_n h[n] * Ct[b, t, n] + Dskip[d] * x[b, t, d]
 *                 ("POPCORNBENCH FW-GLM-5-1 l2_p30", arjun-banerjee.github.io,
 *                 forward-pass derivation and kernel layouts)
 *
 *   S6 bidir      y = forward output + output of the reverse recurrence
 *                 h_rev[n] = dA[t] * h_rev[n] + dBx[t] run from t = L-1 down
 *                 to 0 over the same dA, dBx, each direction with its own
 *                 Dskip * x term ("ARM-Scan", krithiksama.me, Approach: the
 *                 two directions share the discretisation; What broke: the
 *                 fused result equals the two scans run independently).
 *
 * Conventions for every call:
 *  - Pointers named a, b, h, x, delta, Bt, Ct, A, Dskip, y and workspace are
 *    DEVICE pointers owned by the caller. The library allocates nothing and
 *    frees nothing.
 *  - Tensors are dense and row-major: x, delta, y are (B, L, D) with element
 *    (b, t, d) at b*L*D + t*D + d; Bt, Ct are (B, L, N) with (b, t, n) at
 *    (b*L + t)*N + n; A is (D, N); Dskip is (D,). Any 4-byte (fp32) or
 *    2-byte (bf16) aligned pointer is accepted; 16-byte aligned rows take the
 *    vectorised load path.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous on that stream and return once the work is enqueued.
 *  - The workspace is scratch device memory of at least the size the
 *    matching *_workspace_bytes() call returns, 256-byte aligned. It must be
 *    zero-filled (cudaMemset) before its first use and before it is used
 *    for a different entry point or a different S6 shape; between calls of
 *    the same entry point and shape the kernels leave it ready for the next
 *    call. Calls that may run at the same time on the GPU need distinct
 *    workspaces. Results are bitwise reproducible from call to call.
 *  - Argument errors are returned synchronously, with nothing launched.
 *    A failed launch returns SS_ERR_CUDA. Errors the GPU detects while
 *    running (a look-back wait that exceeded the spin timeout) are recorded
 *    in the workspace and returned by ss_get_device_status().
 *  - Sizes of zero (n == 0, or B, L or D == 0) are valid and launch nothing.
 */
#ifndef SS_H
#define SS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SS_ABI_VERSION 1

/* Storage type of x, delta, Bt, Ct and y. State and arithmetic are fp32. */
typedef enum { SS_F32 = 0, SS_BF16 = 1 } ss_dtype;

typedef enum {
    SS_OK = 0,
    SS_ERR_INVALID = 1,      /* null pointer, negative size, bad dtype       */
    SS_ERR_UNSUPPORTED = 2,  /* N outside [1, 16], or a size above a limit   */
    SS_ERR_WORKSPACE = 3,    /* workspace missing, too small or misaligned   */
    SS_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
    SS_ERR_TIMEOUT = 5,      /* a device-side wait exceeded the spin timeout */
    SS_ERR_BOUNDS = 6        /* a device-side index check failed             */
} ss_status;

/* Human-readable name of a status code (static storage, never NULL). */
const char *ss_status_string(int status);

/* SS_ABI_VERSION of the loaded library. */
int ss_abi_version(void);

/* ------------------------------------------------------------ affine scan */

/* Bytes of workspace ss_affine_scan needs for n elements (0 for n <= 0). */
size_t ss_affine_scan_workspace_bytes(int64_t n);

/*
 * h[t] = a[t] * h[t-1] + b[t] for t in [0, n), h[-1] = 0, all fp32.
 * ("Selective-scan CUDA kernels", persus.netlify.app: the recurrence and its
 * single-pass decoupled look-back scan.)
 * a, b: n input floats each; h: n output floats (may alias neither input).
 * One launch: tiles of 4096 elements staged into shared memory by bulk
 * copies, a register and warp-shuffle scan inside each tile, and a
 * decoupled look-back across tiles whose fold order makes the result
 * independent of scheduling.
 */
ss_status ss_affine_scan(const float *a, const float *b, float *h, int64_t n,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * Comparison kernel, not the fast path: ss_affine_scan with each tile scanned
 * by the log-step (Hillis-Steele) algorithm instead of the work-efficient
 * register scan, inside the same persistent look-back kernel. "Selective-scan
 * CUDA kernels" (persus.netlify.app), the predictions: the page's
 * Hillis-Steele measurement ran in PyTorch, which the page itself calls an
 * unfair comparison with its single-pass kernel; this one runs on the GPU
 * under identical staging, look-back and fix-up, so the two measure the
 * algorithms. Each 4096-element tile takes 12 steps; in step k every element
 * E >= 2^k is combined with element E - 2^k as it was after step k-1 (values
 * in registers, exchanged through the tile's shared-memory buffer). Same
 * arguments, workspace (ss_affine_scan_workspace_bytes), results up to
 * rounding order (deterministic) and errors as ss_affine_scan.
 */
ss_status ss_affine_scan_log_step(const float *a, const float *b, float *h, int64_t n,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * ss_affine_scan continued from a state: h[-1] = *h0 instead of 0, so a long
 * sequence can be scanned segment by segment, each segment started from the
 * previous one's last output ("Selective-scan CUDA kernels", opening
 * paragraphs: the recurrence; its h[-1] is the state the segment inherits).
 * h0: DEVICE pointer to one float, read by the kernel when it runs (so it may
 * be written by earlier work on the same stream), or NULL for 0; it must not
 * lie inside h (SS_ERR_INVALID). Workspace, results (deterministic) and
 * errors as ss_affine_scan.
 */
ss_status ss_affine_scan_state(const float *a, const float *b, float *h, int64_t n,
                               const float *h0, void *workspace, size_t workspace_bytes,
                               void *stream);

/* Bytes of DEVICE workspace ss_affine_scan_host needs for n elements (0 for
 * n <= 0): the scan's own workspace plus three device slots of a, b and h
 * for one chunk each. */
size_t ss_affine_scan_host_workspace_bytes(int64_t n);

/*
 * The affine scan of HOST arrays: a, b (inputs) and h (output) are host
 * pointers, best page-locked (cudaHostAlloc / cudaHostRegister), else the
 * copies are staged by the driver and do not overlap. The input is cut into
 * chunks of 2^23 elements; each chunk is copied into a device slot of the
 * workspace, scanned there from the previous chunk's last state (the
 * ss_affine_scan_state kernel) and copied back, with the copies towards the
 * device, the scans and the copies back on three streams so the two
 * directions of the host link and the GPU all work at once. Same h as the
 * recurrence from h[-1] = 0, up to rounding order (deterministic for a
 * given n). workspace: DEVICE memory of ss_affine_scan_host_workspace_bytes
 * (n) bytes, zero-filled before first use like every workspace. The call
 * returns once everything is enqueued; `stream` then waits for the last copy
 * back, so h is complete when `stream` is. Calls on the same device are
 * serialised while they enqueue (the library's two copy streams and their
 * events are shared); the arrays must stay valid until then.
 */
ss_status ss_affine_scan_host(const float *a, const float *b, float *h, int64_t n,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Largest n ss_affine_scan_noalloc accepts (2^24 elements). Its scratch
 * array is 256 + 32 * (SS_AFFINE_NOALLOC_MAX_N / 4096) = 131,328 bytes.
 */
#define SS_AFFINE_NOALLOC_MAX_N (1LL << 24)

/*
 * ss_affine_scan without a workspace argument, for callers that cannot
 * allocate device memory (code that runs where cudaMalloc is not allowed or
 * not safe, such as inside an allocator, a plugin that must leave the device
 * heap alone, or a path that may not allocate after start-up). The pages
 * describing the method have no counterpart to this entry point.
 * Computes the same h as ss_affine_scan (same kernel, same results) for
 * 0 <= n <= SS_AFFINE_NOALLOC_MAX_N; larger n returns SS_ERR_UNSUPPORTED
 * with nothing launched. a, b, h: caller-owned device arrays as for
 * ss_affine_scan; stream: a cudaStream_t.
 * The scratch it needs lives in one static device array inside the library
 * (131,328 bytes, reserved on every GPU that loads the library until the
 * process exits); the call allocates and frees nothing. The first call on a
 * device looks up that array's device address (cudaGetSymbolAddress), so
 * make it before any stream capture on that device. Every call uses the same
 * array: calls that can run at the same time on the GPU (different streams,
 * or threads without ordering between them) race and must not be made.
 * Each call clears the array's error word on `stream` when it starts; read a
 * call's device-detected errors with ss_affine_scan_noalloc_status().
 */
ss_status ss_affine_scan_noalloc(const float *a, const float *b, float *h, int64_t n,
                                 void *stream);

/*
 * Device-detected error of the last ss_affine_scan_noalloc call on the
 * current device (a look-back wait that exceeded the spin timeout:
 * SS_ERR_TIMEOUT, whose output is then undefined), or SS_OK. Synchronises
 * `stream` first (pass the stream of that call), then reads and clears the
 * error word of the library's static array; allocates nothing. The pages
 * describing the method have no counterpart to it. SS_ERR_CUDA if the
 * synchronisation or the read fails.
 */
ss_status ss_affine_scan_noalloc_status(void *stream);

/* ------------------------------------------------------------ S6 */

/* Bytes of workspace the S6 calls need for this shape and storage type on
 * the current device (bidir != 0 for ss_selective_scan_bidir). 0 when the
 * call needs none, in which case workspace may be NULL. */
size_t ss_selective_scan_workspace_bytes(int64_t B, int64_t L, int64_t D,
                                         int64_t N, int io_dtype, int bidir);

/*
 * S6 selective-scan forward (see the top of this file for the arithmetic).
 * x, delta: (B, L, D); Bt, Ct: (B, L, N); y: (B, L, D), all of `io_dtype`.
 * A: (D, N) fp32 (already negative, e.g. -exp(A_log)); Dskip: (D,) fp32 or
 * NULL for no skip term. delta_softplus != 0 applies softplus(v) =
 * log(1 + exp(v)) to delta in the kernel (v > 20 passes v through).
 * 1 <= N <= 16. y must not alias an input.
 * Long sequences are split into chunks over L whose carries are exchanged by
 * a decoupled look-back; short ones run one register-resident chain per
 * (b, d, n) group over all of L.
 */
ss_status ss_selective_scan_fwd(const void *x, const void *delta,
                                const void *Bt, const void *Ct,
                                const float *A, const float *Dskip, void *y,
                                int64_t B, int64_t L, int64_t D, int64_t N,
                                int io_dtype, int delta_softplus,
                                void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * Bidirectional S6: y = forward output + time-reversed output, with dA and
 * dBx computed from the same delta, x, Bt (same arguments as
 * ss_selective_scan_fwd). Runs chunked over L with a forward look-back and
 * a reverse look-forward; every chunk of one (b, d-tile) sequence must be
 * resident at once, which the call checks against the GPU's occupancy
 * (SS_ERR_UNSUPPORTED if L is too long for that).
 */
ss_status ss_selective_scan_bidir(const void *x, const void *delta,
                                  const void *Bt, const void *Ct,
                                  const float *A, const float *Dskip, void *y,
                                  int64_t B, int64_t L, int64_t D, int64_t N,
                                  int io_dtype, int delta_softplus,
                                  void *workspace, size_t workspace_bytes,
                                  void *stream);

/*
 * Forward scan that starts from a given state and returns the final one, so
 * a long sequence can be run in pieces (streaming inference, or a sequence
 * longer than one call should hold): running [0, L1) and then [L1, L) with
 * the first call's h_last as the second call's h0 computes the same
 * recurrence as running [0, L) in one call (equal up to fp32 rounding; the
 * two orders of fma differ). The pages fix the state before t = 0 at zero
 * ("POPCORNBENCH FW-GLM-5-1 l2_p30", forward-pass derivation); this entry
 * point generalises that one step, which they leave open.
 * Arguments as ss_selective_scan_fwd, plus:
 *   h0:     (B, D, N) fp32 device array, row-major, the state h[-1] of every
 *           (b, d, n) chain; NULL means zeros.
 *   h_last: (B, D, N) fp32 device array receiving h[L-1]; NULL means not
 *           written. Must not alias h0 or any other argument.
 * Both are caller-owned and 4-byte aligned (else SS_ERR_INVALID). The
 * workspace is the one ss_selective_scan_workspace_bytes(..., bidir = 0)
 * asks for. With L == 0 the call copies nothing: h_last is left unwritten.
 */
ss_status ss_selective_scan_fwd_state(const void *x, const void *delta,
                                      const void *Bt, const void *Ct,
                                      const float *A, const float *Dskip,
                                      const float *h0, void *y, float *h_last,
                                      int64_t B, int64_t L, int64_t D, int64_t N,
                                      int io_dtype, int delta_softplus,
                                      void *workspace, size_t workspace_bytes,
                                      void *stream);

/*
 * Selective-scan layer forward ("POPCORNBENCH FW-GLM-5-1 l2_p30", the
 * model's parameters and forward pass): the input projections, then the
 * scan of ss_selective_scan_fwd:
 *   delta = softplus(x W_delta^T + b_delta)   (B, L, D)
 *   B_t = x W_B^T,  C_t = x W_C^T             (B, L, N)
 *   y = S6(x, delta, B_t, C_t, A, Dskip)      (B, L, D)
 * x, y: (B, L, D) of io_dtype. W_proj: (D + 2N, D) of io_dtype, row-major in
 * the Linear weight layout (out_features x in_features): rows [0, D) are
 * proj_delta, [D, D + N) proj_B, [D + N, D + 2N) proj_C. b_delta: (D,) fp32.
 * A: (D, N) fp32 (already negative); Dskip: (D,) fp32 or NULL. proj_B and
 * proj_C carry no bias (the pages give one for proj_delta only).
 * The three projections are one dense GEMM, x times W_proj transposed with
 * fp32 accumulation, into one (B*L)-row workspace buffer of io_dtype (a row:
 * pre-activation, B_t, C_t of one step); the scan reads the three blocks at
 * that row stride and applies softplus itself. As a Linear layer with a
 * bias, the pre-activation is the product plus b_delta rounded once to
 * io_dtype: for SS_BF16 the library's tensor-core GEMM adds the bias to the
 * fp32 accumulator before the one rounding to bf16 (D must be a multiple of
 * 8, x and W_proj 16-byte aligned and B*L at most 2^31 - 256, else
 * SS_ERR_UNSUPPORTED); for SS_F32 a
 * cuBLASLt fp32 GEMM writes the product and the scan adds the bias in fp32.
 * The workspace (ss_selective_scan_layer_workspace_bytes) holds the
 * projections, any GEMM scratch and the scan's workspace (first, so
 * ss_get_device_status reads the error word from it: the scan's, and the
 * GEMM's for a wait that ran out); zero it once before first use, as for the
 * scan. Errors as for ss_selective_scan_fwd; SS_ERR_UNSUPPORTED also if no
 * GEMM algorithm fits the shape.
 */
size_t ss_selective_scan_layer_workspace_bytes(int64_t B, int64_t L, int64_t D,
                                               int64_t N, int io_dtype);

ss_status ss_selective_scan_layer_fwd(const void *x, const void *W_proj,
                                      const float *b_delta, const float *A,
                                      const float *Dskip, void *y,
                                      int64_t B, int64_t L, int64_t D, int64_t N,
                                      int io_dtype, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * Backward pass of ss_selective_scan_fwd_state: the gradients of the scalar
 * sum_{b,t,d} dy*y + sum_{b,d,n} dh_last*h_last with respect to every input,
 * i.e. the exact derivative of the forward recurrence ("POPCORNBENCH
 * FW-GLM-5-1 l2_p30", forward-pass derivation; the pages give no backward
 * pass, so this is that definition differentiated). The adjoint of h runs in
 * reverse time over the same dA: lam_t = dy_t*C_t + dA_{t+1}*lam_{t+1}.
 * Inputs as ss_selective_scan_fwd_state (h0 may be NULL), plus
 *   dy:      (B, L, D) of io_dtype, the gradient of y;
 *   dh_last: (B, D, N) fp32 gradient of h_last, or NULL (zeros).
 * Outputs, all caller-owned device arrays, fully overwritten:
 *   dx, ddelta: (B, L, D) of io_dtype (ddelta is the gradient of the delta
 *               input, through softplus when delta_softplus != 0);
 *   dA: (D, N) fp32;  dBt, dCt: (B, L, N) fp32;
 *   dDskip: (D,) fp32, or NULL to skip it;  dh0: (B, D, N) fp32, or NULL.
 * Every sum over channels or time is taken in a fixed order: results are
 * bitwise reproducible. Outputs must not alias inputs or each other. The
 * workspace (ss_selective_scan_bwd_workspace_bytes) needs no zeroing.
 * Four launches on `stream`: chunk aggregates, carries across chunks,
 * gradients, and the final fixed-order sums.
 */
size_t ss_selective_scan_bwd_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N);

ss_status ss_selective_scan_bwd(const void *x, const void *delta,
                                const void *Bt, const void *Ct,
                                const float *A, const float *Dskip,
                                const float *h0, const void *dy,
                                const float *dh_last,
                                void *dx, void *ddelta, float *dA,
                                float *dBt, float *dCt, float *dDskip,
                                float *dh0,
                                int64_t B, int64_t L, int64_t D, int64_t N,
                                int io_dtype, int delta_softplus,
                                void *workspace, size_t workspace_bytes,
                                void *stream);

/* ------------------------------------------------------------ errors */

/*
 * Synchronises `stream`, then reads and clears the error word the kernels
 * keep in `workspace` (SS_OK if nothing went wrong since the last call).
 * SS_ERR_CUDA if the synchronisation itself fails.
 */
ss_status ss_get_device_status(void *workspace, void *stream);

/*
 * Upper bound, in nanoseconds, on any single device-side wait in later
 * launches (default 1e9 = 1 s). A wait that runs out records SS_ERR_TIMEOUT
 * in the workspace and the kernel finishes without hanging.
 * SS_ERR_INVALID for 0.
 */
ss_status ss_set_spin_timeout_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* SS_H */
