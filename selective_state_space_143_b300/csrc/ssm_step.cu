// Single-token recurrent step (streaming decode) with the state carried between calls.
//
// The recurrent form of the scan ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里",
// 背景问题: each step needs only h_{t-1}, so generation runs in constant memory; the
// "引言：Attention的天花板" article's streaming example hands the state from one call to
// the next).  For every sequence b and channel c:
//   Delta = softplus(dt + dt_bias)
//   h[n]  <- exp(Delta A[c,n]) h[n] + Delta B[n] x        (in place)
//   out   =  (sum_n C[n] h[n] + D x) * SiLU(z)
// With a convolution ahead of the scan ("论文解读：Mamba — 线性时间的序列建模革命", 五 Mamba块架构)
// x is first replaced by x' = SiLU(bias + sum_k w[k] x_{t-K+1+k}), the K-1 earlier
// inputs coming from the carried convolution state, which is then shifted by one token.
// The step reads and writes the whole state once, so it is bound by HBM (or L2 when the
// state fits there).  LPC lanes share one channel's state row, each lane taking PPL
// 16-byte pieces of it (pieces lane, lane + LPC, ...), so a warp's accesses are
// contiguous; a lane issues every load of its pieces before its first store, which keeps
// PPL state pieces per thread in flight; the C.h partial sums are combined with shuffles
// inside the LPC-lane group.
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
    const float* conv_w;  // (H*P, conv_k) or null
    const float* conv_b;  // (H*P,) or null
    const void* x_prev;   // (batch, conv_k-1, H*P) or null (zeros)
    void* x_last;         // (batch, conv_k-1, H*P) or null; may equal x_prev
    int64_t batch, H, P, N, G;
    int diag;  // A per (channel, n) when set, one scalar per head otherwise
    int conv_k;
    // byte ranges of the buffers written (stores checked in SSM_BOUNDS_CHECK builds)
    int* status;
    Span state_s, out_s, xlast_s;
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

template <typename T, int LPC, int PPL, bool CONV>
__global__ void __launch_bounds__(kStepThreads) ssm_step_kernel(const StepArgs a) {
    constexpr bool PRECISE = sizeof(T) == 4;
    constexpr int CPB = kStepThreads / LPC;  // channels per block
    const int lane = threadIdx.x % LPC;
    const int64_t b = blockIdx.y;                                         // sequence
    const int nc = (int)(a.H * a.P);                                      // channels per sequence
    const int cs = blockIdx.x * CPB + threadIdx.x / LPC;                  // channel (h, p)
    const int64_t ch = b * nc + cs;                                       // flat (b, h, p)
    const bool ok = cs < nc;
    float y = 0.0f, xv = 0.0f, x_raw = 0.0f;
    float prev[3] = {0.0f, 0.0f, 0.0f};  // convolution state of the channel, oldest first
    int h = 0;
    if (ok) {
        h = a.P == 1 ? cs : cs / (int)a.P;
        const int g = a.G == 1 ? 0 : h / (int)(a.H / a.G);
        const T* Bs = static_cast<const T*>(a.B) + (b * a.G + g) * a.N;
        const T* Cs = static_cast<const T*>(a.C) + (b * a.G + g) * a.N;
        xv = to_f32<T>(static_cast<const T*>(a.x)[ch]);
        if (CONV) {
            const int64_t c = cs;
            const int km1 = a.conv_k - 1;
            float acc = a.conv_b ? a.conv_b[c] : 0.0f;
            for (int j = 0; j < km1; ++j) {
                prev[j] = a.x_prev ? to_f32<T>(static_cast<const T*>(a.x_prev)[(b * km1 + j) * nc + c]) : 0.0f;
                acc = fmaf(a.conv_w[c * a.conv_k + j], prev[j], acc);
            }
            acc = fmaf(a.conv_w[c * a.conv_k + km1], xv, acc);
            x_raw = xv;
            xv = silu_t<PRECISE>(acc);
        }
        const float v = to_f32<T>(static_cast<const T*>(a.dt)[b * a.H + h]) + (a.dt_bias ? a.dt_bias[h] : 0.0f);
        const float de = softplus_t<PRECISE>(v);
        const float u = de * xv;
        float* st = a.state + ch * a.N;
        const float* Arow = a.A + h * a.N;
        const float ah = a.diag ? 0.0f : decay<PRECISE>(de * a.A[h]);
        float4 hv[PPL], Bv[PPL], Cv[PPL], Av[PPL];
#pragma unroll
        for (int q = 0; q < PPL; ++q) {  // every load first
            const int n = 4 * (lane + q * LPC);
            if (n < a.N) {
                hv[q] = *reinterpret_cast<const float4*>(st + n);
                Bv[q] = load4(Bs + n);
                Cv[q] = load4(Cs + n);
                if (a.diag) Av[q] = load4(Arow + n);
            }
        }
#pragma unroll
        for (int q = 0; q < PPL; ++q) {
            const int n = 4 * (lane + q * LPC);
            if (n >= a.N) break;
            float4 av = make_float4(ah, ah, ah, ah);
            if (a.diag)
                av = make_float4(decay<PRECISE>(de * Av[q].x), decay<PRECISE>(de * Av[q].y),
                                 decay<PRECISE>(de * Av[q].z), decay<PRECISE>(de * Av[q].w));
            float4 hn = hv[q];
            hn.x = fmaf(av.x, hn.x, u * Bv[q].x);
            hn.y = fmaf(av.y, hn.y, u * Bv[q].y);
            hn.z = fmaf(av.z, hn.z, u * Bv[q].z);
            hn.w = fmaf(av.w, hn.w, u * Bv[q].w);
            store_checked(a.state_s, reinterpret_cast<float4*>(st + n), hn, a.status);
            y = fmaf(Cv[q].x, hn.x, y);
            y = fmaf(Cv[q].y, hn.y, y);
            y = fmaf(Cv[q].z, hn.z, y);
            y = fmaf(Cv[q].w, hn.w, y);
        }
    }
    // every lane of the warp takes part; an LPC group never straddles the ok boundary
#pragma unroll
    for (int o = LPC / 2; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o, LPC);
    if (CONV) __syncwarp();  // every lane has read the old convolution state
    if (!ok || lane != 0) return;
    if (CONV && a.x_last) {
        // shift the convolution state by one token (in place when x_last == x_prev)
        const int64_t c = cs;
        const int km1 = a.conv_k - 1;
        T* xl = static_cast<T*>(a.x_last) + b * km1 * nc + c;
        for (int j = 0; j < km1; ++j)
            store_checked(a.xlast_s, &xl[j * nc], from_f32<T>(j + 1 < km1 ? prev[j + 1] : x_raw), a.status);
    }
    if (a.D) y = fmaf(a.D[h], xv, y);
    if (a.z) y *= silu_t<PRECISE>(to_f32<T>(static_cast<const T*>(a.z)[ch]));
    store_checked(a.out_s, &static_cast<T*>(a.out)[ch], from_f32<T>(y), a.status);
}

template <typename T, int LPC, int PPL>
void launch_lpc(const StepArgs& s, int64_t nch, cudaStream_t stream) {
    constexpr int CPB = kStepThreads / LPC;
    (void)nch;
    const dim3 blocks((unsigned)((s.H * s.P + CPB - 1) / CPB), (unsigned)s.batch);
    if (s.conv_k > 0)
        ssm_step_kernel<T, LPC, PPL, true><<<blocks, kStepThreads, 0, stream>>>(s);
    else
        ssm_step_kernel<T, LPC, PPL, false><<<blocks, kStepThreads, 0, stream>>>(s);
}

template <typename T>
void launch_typed(const StepArgs& s, int64_t nch, cudaStream_t stream) {
    // 16-byte pieces of a state row: two per lane (the smallest power-of-two lane count
    // that covers the row), one when the row is a single piece; N <= 256 is at most 64
    const int64_t pieces = s.N / 4;
    if (pieces > 32) return launch_lpc<T, 32, 2>(s, nch, stream);
    if (pieces > 16) return launch_lpc<T, 16, 2>(s, nch, stream);
    if (pieces > 8) return launch_lpc<T, 8, 2>(s, nch, stream);
    if (pieces > 4) return launch_lpc<T, 4, 2>(s, nch, stream);
    if (pieces > 2) return launch_lpc<T, 2, 2>(s, nch, stream);
    if (pieces == 2) return launch_lpc<T, 1, 2>(s, nch, stream);
    return launch_lpc<T, 1, 1>(s, nch, stream);
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
    s.conv_w = a.conv_w;
    s.conv_b = a.conv_b;
    s.x_prev = a.x_prev;
    s.x_last = a.x_last;
    s.conv_k = a.conv_k;
    const int64_t nch = a.batch * a.nheads * a.headdim;
    s.status = nullptr;
    if (kBoundsCheck) {
        const cudaError_t e = device_status_address(&s.status);
        if (e != cudaSuccess) return e;
    }
    const size_t E = a.dtype == 1 ? 2 : 4;
    s.state_s = span_of(state, (size_t)nch * a.dstate * sizeof(float));
    s.out_s = span_of(a.out, (size_t)nch * E);
    s.xlast_s = span_of(a.x_last, (size_t)a.batch * (a.conv_k > 1 ? a.conv_k - 1 : 0) * a.nheads * a.headdim * E);
    if (nch == 0) return cudaSuccess;
    cudaEvent_t t0 = timing_begin(stream, "ssm_step_kernel");
    if (a.dtype == 1)
        launch_typed<__nv_bfloat16>(s, nch, stream);
    else
        launch_typed<float>(s, nch, stream);
    note_launch("ssm_step_kernel", stream, t0);
    return cudaGetLastError();
}

}  // namespace ssm
