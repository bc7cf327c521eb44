// Packed pairs of fp32 values in one 64-bit register and the sm_100+
// f32x2 arithmetic on them (two lanes of work per instruction).
#pragma once

#include <cstdint>

namespace ss {

typedef unsigned long long u64;
__device__ __forceinline__ u64 f2(float lo, float hi) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float f2lo(u64 v) {
    float lo;
    asm("mov.b64 {%0, _}, %1;" : "=f"(lo) : "l"(v));
    return lo;
}
__device__ __forceinline__ float f2hi(u64 v) {
    float hi;
    asm("mov.b64 {_, %0}, %1;" : "=f"(hi) : "l"(v));
    return hi;
}
__device__ __forceinline__ u64 f2mul(u64 a, u64 b) {
    u64 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 f2add(u64 a, u64 b) {
    u64 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 f2fma(u64 a, u64 b, u64 c) {
    u64 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// 2^(delta * A2) for a pair of states in one PTX block, so both MUFU results
// land in the two halves of one 64-bit register.
__device__ __forceinline__ u64 f2_exp2_scaled(u64 dd, u64 a2) {
    u64 r;
    asm("{\n .reg .b64 t;\n .reg .f32 lo, hi;\n"
        " mul.rn.f32x2 t, %1, %2;\n"
        " mov.b64 {lo, hi}, t;\n"
        " ex2.approx.ftz.f32 lo, lo;\n"
        " ex2.approx.ftz.f32 hi, hi;\n"
        " mov.b64 %0, {lo, hi};\n}"
        : "=l"(r) : "l"(dd), "l"(a2));
    return r;
}

}  // namespace ss
