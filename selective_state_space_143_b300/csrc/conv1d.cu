// Causal depthwise convolution + SiLU over the sequence, ahead of the SSD kernels.
//
// The x branch of the Mamba block runs a short convolution and SiLU before the selective
// scan ("论文解读：Mamba — 线性时间的序列建模革命", 五 Mamba块架构; width 4 in the
// "引言：Attention的天花板" article's example):
//   x'[b,t,c] = SiLU(bias[c] + sum_{k<K} w[c,k] x[b, t-K+1+k, c]),
// inputs before t = 0 taken from the previous call (x_prev) or zero.  The diagonal scan
// fuses this into its own input staging; the SSD path runs this pass into fp32 scratch
// and reads x' from there (the tensor-core SSD kernels take x as an exact bf16 operand,
// so an fp32 x' runs on the CUDA-core SSD kernels).  One thread per (b, t, channel pair); the K rows a thread reads
// are shared with its neighbours in time through L1/L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kConvThreads = 256;

struct ConvArgs {
    const void* x;
    const float* w;
    const float* bias;
    const void* x_prev;
    void* xc;
    void* x_last;
    int64_t batch, T, ch;
    int K;
};

template <typename T>
__device__ __forceinline__ float x_at(const ConvArgs& a, int64_t b, int64_t s, int64_t c) {
    if (s >= 0) return to_f32<T>(static_cast<const T*>(a.x)[(b * a.T + s) * a.ch + c]);
    const int64_t j = a.K - 1 + s;  // row of x_prev
    if (a.x_prev && j >= 0) return to_f32<T>(static_cast<const T*>(a.x_prev)[(b * (a.K - 1) + j) * a.ch + c]);
    return 0.0f;
}

template <typename T>
__global__ void __launch_bounds__(kConvThreads) conv_silu_kernel(const ConvArgs a) {
    constexpr bool PRECISE = sizeof(T) == 4;
    const int64_t i = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;  // flat (b, t, c)
    const int64_t total = a.batch * a.T * a.ch;
    if (i >= total) return;
    const int64_t c = i % a.ch;
    const int64_t t = (i / a.ch) % a.T;
    const int64_t b = i / (a.ch * a.T);
    float acc = a.bias ? a.bias[c] : 0.0f;
    for (int k = 0; k < a.K; ++k) acc = fmaf(a.w[c * a.K + k], x_at<T>(a, b, t - a.K + 1 + k, c), acc);
    static_cast<float*>(a.xc)[i] = silu_t<PRECISE>(acc);
}

// x_last[b, j, c] = input at time T-K+1+j (raw copy).
template <typename T>
__global__ void __launch_bounds__(kConvThreads) conv_tail_kernel(const ConvArgs a) {
    const int64_t i = (int64_t)blockIdx.x * kConvThreads + threadIdx.x;  // flat (b, j, c)
    const int km1 = a.K - 1;
    if (i >= a.batch * km1 * a.ch) return;
    const int64_t c = i % a.ch;
    const int64_t j = (i / a.ch) % km1;
    const int64_t b = i / (a.ch * km1);
    const int64_t s = a.T - km1 + j;
    T v = from_f32<T>(0.0f);
    if (s >= 0)
        v = static_cast<const T*>(a.x)[(b * a.T + s) * a.ch + c];
    else if (a.x_prev)
        v = static_cast<const T*>(a.x_prev)[(b * km1 + (km1 + s)) * a.ch + c];
    static_cast<T*>(a.x_last)[i] = v;
}

ConvArgs conv_args(const ScanArgs& a, void* xc) {
    ConvArgs c;
    c.x = a.x;
    c.w = a.conv_w;
    c.bias = a.conv_b;
    c.x_prev = a.x_prev;
    c.xc = xc;
    c.x_last = a.x_last;
    c.batch = a.batch;
    c.T = a.seqlen;
    c.ch = a.nheads * a.headdim;
    c.K = a.conv_k;
    return c;
}

}  // namespace

cudaError_t conv_prepass_launch(const ScanArgs& a, void* xc, cudaStream_t stream) {
    const ConvArgs c = conv_args(a, xc);
    const int64_t total = c.batch * c.T * c.ch;
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + kConvThreads - 1) / kConvThreads);
    cudaEvent_t t0 = timing_begin(stream);
    if (a.dtype == 1)
        conv_silu_kernel<__nv_bfloat16><<<blocks, kConvThreads, 0, stream>>>(c);
    else
        conv_silu_kernel<float><<<blocks, kConvThreads, 0, stream>>>(c);
    note_launch("conv_silu_kernel", stream, t0);
    return cudaGetLastError();
}

cudaError_t conv_tail_launch(const ScanArgs& a, cudaStream_t stream) {
    const ConvArgs c = conv_args(a, nullptr);
    const int64_t total = c.batch * (c.K - 1) * c.ch;
    if (!a.x_last || total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + kConvThreads - 1) / kConvThreads);
    cudaEvent_t t0 = timing_begin(stream);
    if (a.dtype == 1)
        conv_tail_kernel<__nv_bfloat16><<<blocks, kConvThreads, 0, stream>>>(c);
    else
        conv_tail_kernel<float><<<blocks, kConvThreads, 0, stream>>>(c);
    note_launch("conv_tail_kernel", stream, t0);
    return cudaGetLastError();
}

}  // namespace ssm
