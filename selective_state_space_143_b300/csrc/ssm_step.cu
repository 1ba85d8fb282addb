// Single-token recurrent step (streaming decode) with the state carried between calls.
//
// The recurrent form of the scan ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里",
// 背景问题: each step needs only h_{t-1}, so generation runs in constant memory; the
// "引言：Attention的天花板" article's streaming example hands the state from one call to
// the next).  For every sequence b and channel c:
//   Delta = softplus(dt + dt_bias)
//   h[n]  <- exp(Delta A[c,n]) h[n] + Delta B[n] x        (in place)
//   out   =  (sum_n C[n] h[n] + D x) * SiLU(z)
// The step reads and writes the whole state once, so it is bound by HBM (or L2 when the
// state fits there).  LPC lanes share one channel's state row, each lane taking 16-byte
// pieces of it, so a warp's accesses are contiguous; the C.h partial sums are combined
// with shuffles inside the LPC-lane group.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kStepThreads = 256;

struct StepArgs {
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* dt_bias;
    float* state;
    void* out;
    int64_t batch, H, P, N, G;
    int diag;  // A per (channel, n) when set, one scalar per head otherwise
};

// Four consecutive elements of a B or C row as fp32 (the row start is 8-byte aligned for
// bf16 and 16-byte aligned for fp32 because N is a multiple of 4).
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

template <bool PRECISE>
__device__ __forceinline__ float decay(float de_times_a) {
    return PRECISE ? expf(de_times_a) : ex2(de_times_a * kLog2e);
}

template <typename T, int LPC>
__global__ void __launch_bounds__(kStepThreads) ssm_step_kernel(const StepArgs a) {
    constexpr bool PRECISE = sizeof(T) == 4;
    constexpr int CPB = kStepThreads / LPC;  // channels per block
    const int lane = threadIdx.x % LPC;
    const int64_t ch = (int64_t)blockIdx.x * CPB + threadIdx.x / LPC;  // flat (b, h, p)
    const bool ok = ch < a.batch * a.H * a.P;
    float y = 0.0f, xv = 0.0f;
    int64_t h = 0;
    if (ok) {
        const int64_t b = ch / (a.H * a.P);
        h = (ch / a.P) % a.H;
        const int64_t g = h / (a.H / a.G);
        const T* Bs = static_cast<const T*>(a.B) + (b * a.G + g) * a.N;
        const T* Cs = static_cast<const T*>(a.C) + (b * a.G + g) * a.N;
        xv = to_f32<T>(static_cast<const T*>(a.x)[ch]);
        const float v = to_f32<T>(static_cast<const T*>(a.dt)[b * a.H + h]) + (a.dt_bias ? a.dt_bias[h] : 0.0f);
        const float de = softplus_t<PRECISE>(v);
        const float u = de * xv;
        float* st = a.state + ch * a.N;
        const float* Arow = a.A + h * a.N;
        const float ah = a.diag ? 0.0f : decay<PRECISE>(de * a.A[h]);
        for (int64_t n = 4 * lane; n < a.N; n += 4 * LPC) {
            float4 hv = *reinterpret_cast<const float4*>(st + n);
            const float4 Bv = load4(Bs + n);
            const float4 Cv = load4(Cs + n);
            float4 av = make_float4(ah, ah, ah, ah);
            if (a.diag) {
                const float4 Av = load4(Arow + n);
                av = make_float4(decay<PRECISE>(de * Av.x), decay<PRECISE>(de * Av.y),
                                 decay<PRECISE>(de * Av.z), decay<PRECISE>(de * Av.w));
            }
            hv.x = fmaf(av.x, hv.x, u * Bv.x);
            hv.y = fmaf(av.y, hv.y, u * Bv.y);
            hv.z = fmaf(av.z, hv.z, u * Bv.z);
            hv.w = fmaf(av.w, hv.w, u * Bv.w);
            *reinterpret_cast<float4*>(st + n) = hv;
            y = fmaf(Cv.x, hv.x, y);
            y = fmaf(Cv.y, hv.y, y);
            y = fmaf(Cv.z, hv.z, y);
            y = fmaf(Cv.w, hv.w, y);
        }
    }
    // every lane of the warp takes part; an LPC group never straddles the ok boundary
#pragma unroll
    for (int o = LPC / 2; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o, LPC);
    if (!ok || lane != 0) return;
    if (a.D) y = fmaf(a.D[h], xv, y);
    if (a.z) y *= silu_t<PRECISE>(to_f32<T>(static_cast<const T*>(a.z)[ch]));
    static_cast<T*>(a.out)[ch] = from_f32<T>(y);
}

template <typename T, int LPC>
void launch_lpc(const StepArgs& s, int64_t nch, cudaStream_t stream) {
    constexpr int CPB = kStepThreads / LPC;
    const unsigned blocks = (unsigned)((nch + CPB - 1) / CPB);
    ssm_step_kernel<T, LPC><<<blocks, kStepThreads, 0, stream>>>(s);
}

template <typename T>
void launch_typed(const StepArgs& s, int64_t nch, cudaStream_t stream) {
    // lanes per channel: one 16-byte piece of the state row each, at most a warp
    const int64_t pieces = s.N / 4;
    if (pieces >= 32) return launch_lpc<T, 32>(s, nch, stream);
    if (pieces >= 16) return launch_lpc<T, 16>(s, nch, stream);
    if (pieces >= 8) return launch_lpc<T, 8>(s, nch, stream);
    if (pieces >= 4) return launch_lpc<T, 4>(s, nch, stream);
    if (pieces >= 2) return launch_lpc<T, 2>(s, nch, stream);
    return launch_lpc<T, 1>(s, nch, stream);
}

}  // namespace

cudaError_t step_launch(const ScanArgs& a, bool diag_a, float* state, cudaStream_t stream) {
    StepArgs s;
    s.x = a.x;
    s.dt = a.dt;
    s.A = a.A;
    s.B = a.B;
    s.C = a.C;
    s.D = a.D;
    s.z = a.z;
    s.dt_bias = a.dt_bias;
    s.state = state;
    s.out = a.out;
    s.batch = a.batch;
    s.H = a.nheads;
    s.P = a.headdim;
    s.N = a.dstate;
    s.G = a.ngroups;
    s.diag = diag_a ? 1 : 0;
    const int64_t nch = a.batch * a.nheads * a.headdim;
    if (nch == 0) return cudaSuccess;
    if (a.dtype == 1)
        launch_typed<__nv_bfloat16>(s, nch, stream);
    else
        launch_typed<float>(s, nch, stream);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace ssm
