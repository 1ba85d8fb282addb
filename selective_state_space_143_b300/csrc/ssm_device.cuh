// Device helpers shared by the scan kernels: element loads/stores, the fast base-2
// exponential/logarithm instructions, softplus and SiLU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---- bounds checks (builds with SSM_BOUNDS_CHECK) ---------------------------------
// A store site checks its address against the byte range of the buffer it writes.  In a
// build with SSM_BOUNDS_CHECK an address outside the range is not written: the kernel
// records status code kStatusBounds in the per-device status word (the first code
// recorded stays) and skips the store.  Other builds compile the check away.
constexpr int kStatusBounds = 9;

struct Span {
    const char* lo = nullptr;  // first byte of the buffer
    const char* hi = nullptr;  // one past its last byte
};

inline Span span_of(const void* base, size_t bytes) {
    Span s;
    s.lo = static_cast<const char*>(base);
    s.hi = s.lo + (base ? bytes : 0);
    return s;
}

#ifdef SSM_BOUNDS_CHECK
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif

__device__ __forceinline__ bool span_ok(const Span& s, const void* p, int bytes, int* status) {
    if (!kBoundsCheck) return true;
    const char* q = static_cast<const char*>(p);
    if (q >= s.lo && q + bytes <= s.hi) return true;
    if (status) atomicCAS(status, 0, kStatusBounds);
    return false;
}

// atomicAdd(p, v) when p lies in the span (always, without SSM_BOUNDS_CHECK).
__device__ __forceinline__ void atomic_add_checked(const Span& s, float* p, float v, int* status) {
    if (span_ok(s, p, 4, status)) atomicAdd(p, v);
}

// Four consecutive fp32 atomic adds as one vector atomic (16-byte aligned p).
__device__ __forceinline__ void atomic_add4_checked(const Span& s, float* p, float4 v, int* status) {
    if (span_ok(s, p, 16, status)) atomicAdd(reinterpret_cast<float4*>(p), v);
}

// *p = v when p lies in the span (always, without SSM_BOUNDS_CHECK).
template <typename V>
__device__ __forceinline__ void store_checked(const Span& s, V* p, V v, int* status) {
    if (span_ok(s, p, (int)sizeof(V), status)) *p = v;
}

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

// Accurate variants (CUDA's log1pf / expf / IEEE division) for fp32 inputs, where the
// tolerance is tighter than the approximate instructions allow.
__device__ __forceinline__ float softplus_precise(float v) {
    return fmaxf(v, 0.0f) + log1pf(expf(-fabsf(v)));
}
__device__ __forceinline__ float silu_precise(float z) { return z / (1.0f + expf(-z)); }

// Fast path for 16-bit inputs, accurate path for fp32 inputs.
template <bool PRECISE>
__device__ __forceinline__ float softplus_t(float v) {
    return PRECISE ? softplus_precise(v) : softplus(v);
}
template <bool PRECISE>
__device__ __forceinline__ float silu_t(float z) {
    return PRECISE ? silu_precise(z) : silu(z);
}

// ln(1 + e) for e in [0, 1] as e * q(e), q a degree-6 polynomial fitted here to
// ln(1 + e) / e by least squares on Chebyshev nodes of [0, 1] (max relative error
// 1.5e-6 in fp32 Horner evaluation); runs on the FMA pipe instead of the SFU.
__device__ __forceinline__ float2 log1p01_2(float2 e) {
    float2 q = make_float2(0.014202826f, 0.014202826f);
    q = __ffma2_rn(q, e, make_float2(-0.066588052f, -0.066588052f));
    q = __ffma2_rn(q, e, make_float2(0.14943458f, 0.14943458f));
    q = __ffma2_rn(q, e, make_float2(-0.23514864f, -0.23514864f));
    q = __ffma2_rn(q, e, make_float2(0.33112052f, 0.33112052f));
    q = __ffma2_rn(q, e, make_float2(-0.49987191f, -0.49987191f));
    q = __ffma2_rn(q, e, make_float2(0.99999875f, 0.99999875f));
    return __fmul2_rn(e, q);
}

// softplus of two values: max(v, 0) + ln(1 + exp(-|v|)), the logarithm by polynomial.
__device__ __forceinline__ float2 softplus2_fma(float2 v) {
    const float2 e = make_float2(ex2(-fabsf(v.x) * kLog2e), ex2(-fabsf(v.y) * kLog2e));
    return __fadd2_rn(make_float2(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f)), log1p01_2(e));
}

// 1 / d for d >= 1 without the SFU: the integer-subtraction first approximation
// (Blinn, "Floating-point tricks", IEEE CG&A 1997; relative error < 13%) refined by
// two Newton steps r <- r (2 - d r) (relative error < 3e-4, enough for 16-bit outputs).
__device__ __forceinline__ float2 rcp2_newton(float2 d) {
    float2 r = make_float2(__int_as_float(0x7EF311C7 - __float_as_int(d.x)),
                           __int_as_float(0x7EF311C7 - __float_as_int(d.y)));
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const float2 t = __ffma2_rn(make_float2(-d.x, -d.y), r, make_float2(1.0f, 1.0f));
        r = __ffma2_rn(r, t, r);
    }
    return r;
}

// SiLU of two values with one SFU exponential each; z is clamped below at -30, where
// SiLU(z) is below 1e-11 and the clamp changes it by less than that.
__device__ __forceinline__ float2 silu2_fma(float2 z) {
    const float2 zc = make_float2(fmaxf(z.x, -30.0f), fmaxf(z.y, -30.0f));
    const float2 m = __fmul2_rn(zc, make_float2(-kLog2e, -kLog2e));
    const float2 d = __fadd2_rn(make_float2(ex2(m.x), ex2(m.y)), make_float2(1.0f, 1.0f));
    return __fmul2_rn(z, rcp2_newton(d));
}

// softplus of two values with packed fp32x2 arithmetic where it applies.
__device__ __forceinline__ float2 softplus2(float2 v) {
    const float e0 = ex2(-fabsf(v.x) * kLog2e), e1 = ex2(-fabsf(v.y) * kLog2e);
    const float2 e = make_float2(e0, e1);
    // e (1 - e (1/2 - e (1/3 - e/4)))
    float2 p = __ffma2_rn(e, make_float2(-0.25f, -0.25f), make_float2(0.33333334f, 0.33333334f));
    p = __ffma2_rn(e, make_float2(-p.x, -p.y), make_float2(0.5f, 0.5f));
    p = __ffma2_rn(e, make_float2(-p.x, -p.y), make_float2(1.0f, 1.0f));
    p = __fmul2_rn(e, p);
    const float2 one_e = __fadd2_rn(e, make_float2(1.0f, 1.0f));
    const float l0 = lg2(one_e.x) * kLn2, l1 = lg2(one_e.y) * kLn2;
    const float r0 = e0 < 0.015625f ? p.x : l0;
    const float r1 = e1 < 0.015625f ? p.y : l1;
    return __fadd2_rn(make_float2(fmaxf(v.x, 0.0f), fmaxf(v.y, 0.0f)), make_float2(r0, r1));
}

// SiLU of two values.
__device__ __forceinline__ float2 silu2(float2 z) {
    const float2 m = __fmul2_rn(z, make_float2(-kLog2e, -kLog2e));
    const float2 d = __fadd2_rn(make_float2(ex2(m.x), ex2(m.y)), make_float2(1.0f, 1.0f));
    return make_float2(__fdividef(z.x, d.x), __fdividef(z.y, d.y));
}

template <bool PRECISE>
__device__ __forceinline__ float2 softplus2_t(float2 v) {
    if (PRECISE) return make_float2(softplus_precise(v.x), softplus_precise(v.y));
    return softplus2(v);
}
template <bool PRECISE>
__device__ __forceinline__ float2 silu2_t(float2 z) {
    if (PRECISE) return make_float2(silu_precise(z.x), silu_precise(z.y));
    return silu2(z);
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
