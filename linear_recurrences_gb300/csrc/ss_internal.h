// Internal launch entry points shared by the C-ABI translation unit.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ss.h"

namespace ss {

// SMs and shared memory per SM of the current device (planning inputs; the
// GB300's values if the query fails, e.g. in a process without a GPU).
inline int device_sm_count() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return 152;
    }
    return v;
}
inline int device_smem_per_sm() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        v <= 0) {
        cudaGetLastError();
        return 233472;
    }
    return v;
}

// Encodes a tiled TMA tensor map (cuTensorMapEncodeTiled through the
// runtime's driver entry point) into `map` (a 128-byte CUtensorMap): `rank`
// dimensions innermost first, dims[i] elements each, strides[i] bytes
// between consecutive indices of dimension i + 1, box[i] elements per copy,
// fp32 or bf16 elements, zero fill outside the extent; swizzle: the
// shared-memory swizzle span in bytes (64 or 128; the box's inner extent
// must not exceed it), 0 for none. false if the entry point is missing or
// the driver rejects the layout.
bool encode_tiled_map(void *map, const void *base, bool bf16, int rank, const uint64_t *dims,
                      const uint64_t *strides, const uint32_t *box, int swizzle = 0);

// Projection GEMM on the tensor cores (tcgen05): out (M x Nout, row stride
// ld_out, bf16) = x (M x K, bf16, row-major) times W (Nout x K, bf16,
// row-major) transposed, fp32 accumulation, bias[j] (fp32) added to columns
// j < n_bias before the single rounding to bf16 (bias may be null).
// workspace: a 256-byte workspace header (device errors). Supported when
// proj_gemm_supported() holds: K and ld_out multiples of 8 elements, the
// three pointers 16-byte aligned.
bool proj_gemm_supported(const void *x, const void *W, const void *out, int64_t M, int64_t K,
                         int64_t Nout, int64_t ld_out);
ss_status proj_gemm_launch(const void *x, const void *W, void *out, const float *bias,
                           int64_t n_bias, int64_t M, int64_t K, int64_t Nout, int64_t ld_out,
                           void *workspace, cudaStream_t stream, unsigned long long timeout_ns);
// The launch plan of a GEMM of this shape (host only, no GPU needed): out =
// {BN, N-tiles, K-columns per stage, K-blocks, stages, pair (1 or 0), work
// units, dynamic shared memory bytes}; -1 for an invalid shape.
int proj_gemm_describe_plan(int64_t M, int64_t K, int64_t Nout, int64_t *out);

size_t affine_workspace_bytes(int64_t n);
// log_step_tiles: scan each tile with the log-step (Hillis-Steele) algorithm
// instead of the work-efficient register scan (comparison variant).
// h0: device pointer to the state before element 0 (null: 0); must not lie
// inside h.
ss_status affine_launch(const float *a, const float *b, float *h, int64_t n, void *workspace,
                        cudaStream_t stream, unsigned long long timeout_ns, long long skip_unit,
                        bool log_step_tiles = false, const float *h0 = nullptr);

// Affine scan over host (or any UVA-addressable) buffers, pipelined through
// device slots in the workspace; see ss_affine_scan_host.
size_t affine_host_workspace_bytes(int64_t n);
ss_status affine_host_launch(const float *a, const float *b, float *h, int64_t n, void *workspace,
                             size_t ws_bytes, cudaStream_t stream, unsigned long long timeout_ns);

struct S6Args {
    const void *x, *delta, *Bt, *Ct;
    const float *A, *Dskip;
    void *y;
    const float *delta_bias = nullptr;  // (D,) added to delta before softplus, or null
    const float *h0;  // (B, D, N) initial state or null (zeros); forward only
    float *h_last;    // (B, D, N) final state or null; forward only
    int64_t ld_delta = 0;  // row stride (elements) of delta; 0: D (dense)
    int64_t ld_bc = 0;     // row stride (elements) of Bt and Ct; 0: N (dense)
    int64_t B, L, D, N;
    int io_bf16;
    int softplus;
    int bidir;
};

// Raises the dynamic shared-memory limit of kernel `fn` on the current
// device to at least `bytes` (a per-device attribute). The limit only ever
// grows, under a lock, so a launch sized under an earlier call stays valid
// while another host thread launches the same kernel with another size.
ss_status raise_smem_limit(const void *fn, int bytes);

// Current bound on device-side waits (ss_set_spin_timeout_ns).
unsigned long long spin_timeout_ns();
// Consumes a pending ss_testing_skip_publish_once request (-1 if none).
long long take_skip_unit();

size_t s6_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int bidir);
// Test hooks behind ss_testing_s6_plan / ss_testing_s6_describe_plan.
void s6_set_plan_override(int kind, int a, int b, int c);
int s6_describe_plan(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16, int bidir,
                     int64_t *out);


struct S6BwdArgs {
    const void *x, *delta, *Bt, *Ct, *dy;
    const float *A, *Dskip, *h0, *dh_last;
    void *dx, *ddelta;
    float *dA, *dBt, *dCt, *dDskip, *dh0;
    int64_t B, L, D, N;
    int io_bf16;
    int softplus;
};
size_t s6_bwd_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N);
size_t layer_workspace_bytes(int64_t B, int64_t L, int64_t D, int64_t N, int io_bf16);
ss_status layer_fwd_launch(const void *x, const void *W_proj, const float *b_delta, const float *A,
                           const float *Dskip, void *y, int64_t B, int64_t L, int64_t D,
                           int64_t N, int io_bf16, void *workspace, size_t ws_bytes,
                           cudaStream_t stream, unsigned long long timeout_ns, long long skip_unit);
ss_status s6_bwd_launch(const S6BwdArgs &a, void *workspace, size_t ws_bytes, cudaStream_t stream);
ss_status s6_launch(const S6Args &a, void *workspace, size_t ws_bytes, cudaStream_t stream,
                    unsigned long long timeout_ns, long long skip_unit);

}  // namespace ss
