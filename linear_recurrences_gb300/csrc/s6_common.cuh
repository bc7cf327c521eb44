// Elementwise helpers shared by the S6 kernels (sm_103a): storage-type
// conversions and softplus on the MUFU unit.
#pragma once

#include <cuda_bf16.h>

#include "ss_common.cuh"

namespace ss {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
// Output store to GLOBAL memory (fp32 as a streaming store).
__device__ __forceinline__ void store_io(float *p, float v) { __stcs(p, v); }
__device__ __forceinline__ void store_io(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }
// Output store to a SHARED-memory tile (plain store; bf16 rounded to nearest even).
__device__ __forceinline__ void store_smem(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_smem(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// softplus(v) = log(1 + exp(v)); v > 20 returns v. exp and log on MUFU; for
// exp(v) < 1/64 the log is replaced by its alternating series so that the
// rounding of 1 + exp(v) does not swamp small results. Both forms are
// computed and selected, so the step has no branch.
__device__ __forceinline__ float softplus_mufu(float v) {
    const float e = ex2_approx(fminf(v, 20.0f) * kLog2e);
    const float series = e * (1.0f - e * (0.5f - e * (1.0f / 3.0f - 0.25f * e)));
    const float logged = lg2_approx(1.0f + e) * kLn2;
    const float r = e < 0.015625f ? series : logged;
    return v > 20.0f ? v : r;
}

}  // namespace ss
