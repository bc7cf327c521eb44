// MUFU ex2 throughput probe (measurement only, see include/ss_probe.h).
#include "ss_common.cuh"
#include "ss_probe.h"

namespace {

__global__ void __launch_bounds__(256) mufu_ex2_probe(float *out, int iters) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = -0.001f * (float)(threadIdx.x + 32 * i + 1);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = ss::ex2_approx(v[i]) - 1.0f;  // stays in [-1, 0]
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i];
    out[blockIdx.x * 256 + threadIdx.x] = s;
}

}  // namespace

extern "C" ss_status ss_probe_mufu_ex2(float *out, int blocks, int iters, void *stream) {
    if (!out || blocks <= 0 || iters <= 0) return SS_ERR_INVALID;
    mufu_ex2_probe<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(out, iters);
    return cudaGetLastError() == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}
