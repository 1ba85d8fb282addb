// Device helpers shared by the scan kernels: element loads/stores, the fast base-2
// exponential/logarithm instructions, softplus and SiLU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the special-function unit (ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(x) on the special-function unit.
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// softplus(v) = ln(1 + e^v) = max(v, 0) + ln(1 + e^{-|v|}).
// ln(1 + e) for e = e^{-|v|} in (0, 1]: for e < 2^-6 the alternating series
// e - e^2/2 + e^3/3 - e^4/4 (truncation below 1e-9 relative), else log2(1 + e) * ln 2
// (1 + e is then far enough from 1 that its rounding costs < 4e-6 relative).
__device__ __forceinline__ float softplus(float v) {
    const float e = ex2(-fabsf(v) * kLog2e);
    const float series = e * (1.0f - e * (0.5f - e * (0.33333334f - 0.25f * e)));
    const float viaLog = lg2(1.0f + e) * kLn2;
    return fmaxf(v, 0.0f) + (e < 0.015625f ? series : viaLog);
}

// SiLU(z) = z / (1 + e^{-z}).
__device__ __forceinline__ float silu(float z) {
    return __fdividef(z, 1.0f + ex2(-z * kLog2e));
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

}  // namespace ssm
