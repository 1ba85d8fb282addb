// Causal depthwise convolution + SiLU over the sequence, ahead of the SSD kernels.
//
// The x branch of the Mamba block runs a short convolution and SiLU before the selective
// scan ("论文解读：Mamba — 线性时间的序列建模革命", 五 Mamba块架构; width 4 in the
// "引言：Attention的天花板" article's example):
//   x'[b,t,c] = SiLU(bias[c] + sum_{k<K} w[c,k] x[b, t-K+1+k, c]),
// inputs before t = 0 taken from the previous call (x_prev) or zero.  The diagonal scan
// fuses this into its own input staging; the SSD path runs this pass into scratch.  x'
// is kept at fp32 precision, either as fp32 (read by the CUDA-core SSD kernels) or as two
// bf16 planes x_hi = bf16(x'), x_lo = bf16(x' - x_hi) (read by the tensor-core SSD
// kernels, which multiply both planes against exact bf16 operands).
//
// One thread per 4 channels and 16 consecutive steps: the three inputs before
// its current step slide through registers, so each input row is read once per thread
// (plus a three-row halo per 16 steps); a warp's loads and stores are contiguous rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kConvThreads = 256;
constexpr int kConvTT = 32;  // steps per thread (c3 pass: 16 -> 197 us, 32 -> 177, 64 -> 171; c4: 388, 339, 325)
constexpr int kConvVX = 32;  // channel vectors per block
constexpr int kConvTY = kConvThreads / kConvVX;  // step blocks per block

struct ConvArgs {
    const void* x;
    const float* w;
    const float* bias;
    const void* x_prev;
    void* xc;
    void* x_last;
    int64_t batch, T, ch;
    int K;
    // byte ranges of the buffers written (stores checked in SSM_BOUNDS_CHECK builds)
    int* status;
    Span xc_s, xlast_s;
};

// One vector of inputs (VW channels from c0: 8 bytes of bf16 or 16 of fp32) at step s,
// as fp32; rows before t = 0 come from x_prev, else zero.
template <typename T, int VW>
__device__ __forceinline__ void load_vec(const ConvArgs& a, int64_t b, int64_t s, int64_t c0, float (&v)[VW]) {
    const T* src = nullptr;
    if (s >= 0)
        src = static_cast<const T*>(a.x) + (b * a.T + s) * a.ch + c0;
    else if (a.x_prev && a.K - 1 + s >= 0)
        src = static_cast<const T*>(a.x_prev) + (b * (a.K - 1) + (a.K - 1 + s)) * a.ch + c0;
    if (!src) {
#pragma unroll
        for (int j = 0; j < VW; ++j) v[j] = 0.0f;
        return;
    }
    uint4 r;
    if constexpr (VW * sizeof(T) == 16) {
        r = *reinterpret_cast<const uint4*>(src);
    } else {
        const uint2 h = *reinterpret_cast<const uint2*>(src);
        r = make_uint4(h.x, h.y, 0u, 0u);
    }
    if constexpr (sizeof(T) == 2) {
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
        for (int j = 0; j < VW / 2; ++j) {
            const float2 f = __bfloat1622float2(p[j]);
            v[2 * j] = f.x;
            v[2 * j + 1] = f.y;
        }
    } else {
        const float* p = reinterpret_cast<const float*>(&r);
#pragma unroll
        for (int j = 0; j < VW; ++j) v[j] = p[j];
    }
}

// SPLIT: xc holds the bf16 planes x_hi (first batch*T*ch elements) and x_lo; else fp32.
template <typename T, bool SPLIT>
__global__ void __launch_bounds__(kConvThreads) conv_silu_kernel(const ConvArgs a) {
    constexpr int VW = 4;  // channels per thread (8-byte bf16 vectors, 16-byte fp32 vectors)
    constexpr bool PRECISE = sizeof(T) == 4;
    const int64_t c0 = ((int64_t)blockIdx.x * kConvVX + threadIdx.x) * VW;
    const int64_t b = blockIdx.z;
    if (c0 >= a.ch) return;
    // taps left-padded to width 4: tap k weights the input at t - 3 + k
    float w[4][VW], bias[VW];
#pragma unroll
    for (int j = 0; j < VW; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int kk = k - (4 - a.K);
            w[k][j] = kk >= 0 ? a.w[(c0 + j) * a.K + kk] : 0.0f;
        }
        bias[j] = a.bias ? a.bias[c0 + j] : 0.0f;
    }
    const int64_t plane = a.batch * a.T * a.ch;
    for (int64_t t0 = ((int64_t)blockIdx.y * kConvTY + threadIdx.y) * kConvTT; t0 < a.T;
         t0 += (int64_t)gridDim.y * kConvTY * kConvTT) {
        float win[3][VW];  // inputs at t-3, t-2, t-1
#pragma unroll
        for (int r = 0; r < 3; ++r) load_vec<T, VW>(a, b, t0 - 3 + r, c0, win[r]);
        const int tt = (int)min((int64_t)kConvTT, a.T - t0);
        // four rows loaded together, then their four outputs
        for (int i0 = 0; i0 < tt; i0 += 4) {
            float cur[4][VW];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i0 + u < tt) {
                    load_vec<T, VW>(a, b, t0 + i0 + u, c0, cur[u]);
                } else {
#pragma unroll
                    for (int j = 0; j < VW; ++j) cur[u][j] = 0.0f;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i0 + u >= tt) break;
                const int64_t t = t0 + i0 + u;
                float y[VW];
#pragma unroll
                for (int j = 0; j < VW; ++j) {
                    float acc = fmaf(w[0][j], win[0][j], bias[j]);
                    acc = fmaf(w[1][j], win[1][j], acc);
                    acc = fmaf(w[2][j], win[2][j], acc);
                    acc = fmaf(w[3][j], cur[u][j], acc);
                    y[j] = silu_t<PRECISE>(acc);
                    win[0][j] = win[1][j];
                    win[1][j] = win[2][j];
                    win[2][j] = cur[u][j];
                }
                const int64_t o = (b * a.T + t) * a.ch + c0;
                if constexpr (SPLIT) {
                    uint32_t hi[VW / 2], lo[VW / 2];
#pragma unroll
                    for (int j = 0; j < VW / 2; ++j) {
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(y[2 * j], y[2 * j + 1]);
                        const float2 hf = __bfloat1622float2(h2);
                        const __nv_bfloat162 l2 = __floats2bfloat162_rn(y[2 * j] - hf.x, y[2 * j + 1] - hf.y);
                        hi[j] = *reinterpret_cast<const uint32_t*>(&h2);
                        lo[j] = *reinterpret_cast<const uint32_t*>(&l2);
                    }
                    __nv_bfloat16* xh = static_cast<__nv_bfloat16*>(a.xc);
                    store_checked(a.xc_s, reinterpret_cast<uint2*>(xh + o), make_uint2(hi[0], hi[1]), a.status);
                    store_checked(a.xc_s, reinterpret_cast<uint2*>(xh + plane + o), make_uint2(lo[0], lo[1]), a.status);
                } else {
                    float* xf = static_cast<float*>(a.xc) + o;
#pragma unroll
                    for (int j = 0; j < VW; j += 4)
                        store_checked(a.xc_s, reinterpret_cast<float4*>(xf + j), make_float4(y[j], y[j + 1], y[j + 2], y[j + 3]), a.status);
                }
            }
        }
    }
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
    store_checked(a.xlast_s, &static_cast<T*>(a.x_last)[i], v, a.status);
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
    c.status = nullptr;
    const size_t E = a.dtype == 1 ? 2 : 4;
    c.xc_s = span_of(xc, (size_t)c.batch * c.T * c.ch * 4);  // fp32, or two bf16 planes
    c.xlast_s = span_of(a.x_last, (size_t)c.batch * (c.K > 1 ? c.K - 1 : 0) * c.ch * E);
    return c;
}

}  // namespace

cudaError_t conv_prepass_launch(const ScanArgs& a, void* xc, bool split, cudaStream_t stream) {
    ConvArgs c = conv_args(a, xc);
    if (kBoundsCheck) {
        const cudaError_t e = device_status_address(&c.status);
        if (e != cudaSuccess) return e;
    }
    if (c.batch * c.T * c.ch == 0) return cudaSuccess;
    if (split && a.dtype != 1) return cudaErrorInvalidValue;  // planes are for bf16 inputs
    const int vw = 4;  // channels per thread (ch is a multiple of 4 for either dtype)
    const int64_t nvec = c.ch / vw;
    const int64_t tblocks = (c.T + kConvTT * kConvTY - 1) / (kConvTT * kConvTY);
    const dim3 grid((unsigned)((nvec + kConvVX - 1) / kConvVX), (unsigned)std::min<int64_t>(tblocks, 65535),
                    (unsigned)c.batch);
    const dim3 block(kConvVX, kConvTY);
    cudaEvent_t t0 = timing_begin(stream, "conv_silu_kernel");
    if (a.dtype == 1) {
        if (split)
            conv_silu_kernel<__nv_bfloat16, true><<<grid, block, 0, stream>>>(c);
        else
            conv_silu_kernel<__nv_bfloat16, false><<<grid, block, 0, stream>>>(c);
    } else {
        conv_silu_kernel<float, false><<<grid, block, 0, stream>>>(c);
    }
    note_launch("conv_silu_kernel", stream, t0);
    return cudaGetLastError();
}

cudaError_t conv_tail_launch(const ScanArgs& a, cudaStream_t stream) {
    ConvArgs c = conv_args(a, nullptr);
    if (kBoundsCheck) {
        const cudaError_t e = device_status_address(&c.status);
        if (e != cudaSuccess) return e;
    }
    const int64_t total = c.batch * (c.K - 1) * c.ch;
    if (!a.x_last || total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((total + kConvThreads - 1) / kConvThreads);
    cudaEvent_t t0 = timing_begin(stream, "conv_tail_kernel");
    if (a.dtype == 1)
        conv_tail_kernel<__nv_bfloat16><<<blocks, kConvThreads, 0, stream>>>(c);
    else
        conv_tail_kernel<float><<<blocks, kConvThreads, 0, stream>>>(c);
    note_launch("conv_tail_kernel", stream, t0);
    return cudaGetLastError();
}

}  // namespace ssm
