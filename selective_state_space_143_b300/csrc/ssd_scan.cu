// Mamba-2 / SSD selective scan: scalar A per head, evaluated chunk by chunk.
//
// With A scalar per head the scan operator is y = (L o M) x with a semiseparable M
// ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里", 第二步 and
// 关键技术点 1-3).  Its diagonal blocks (one chunk of Q steps) are dense and are
// computed directly; its off-diagonal blocks are low rank and pass through the state
// carried between chunks.  With s_t the in-chunk inclusive cumulative sum of
// Delta_t * A_h:
//   Y_diag[t, :] = sum_{s<=t} exp(s_t - s_s) (C_t . B_s) Delta_s x_s[:]
//   S_c          = sum_s exp(s_last - s_s) Delta_s x_s[:] B_s^T           (P x N)
//   h_c          = exp(s_last) h_{c-1} + S_c                             (chunk carry)
//   Y_off[t, :]  = exp(s_t) h_{c-1} C_t
//   out          = (Y_diag + Y_off + D x) * SiLU(z)
//
// This file holds the CUDA-core implementation, three kernels:
//   ssd_chunk_state  : Delta, cumulative decay sums and the local chunk states S_c
//   ssd_state_pass   : sequential carry over chunks, h_{c-1} stored per chunk, final state
//   ssd_chunk_scan   : Y_diag + Y_off + skip + gate for each chunk
// the tensor-core path's carry (ssd_state_pass_split), and the dispatch between the two
// paths (ssd_tc.cu holds the tensor-core chunk-state and scan kernels).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "ssm_device.cuh"
#include "ssd_tc.h"
#include "tc_util.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;   // P-tile, N-tile and row tile
constexpr int kSub = 32;    // inner time sub-tile

struct SsdArgs {
    const char* x;
    const char* dt;
    const char* z;
    const char* B;
    const char* C;
    const float* A;
    const float* D;
    const float* dt_bias;
    const float* init;  // (b, H, P, N) or null
    char* out;
    float* final_state;
    float* dl;      // (b, H, nchunks, Q) Delta
    float* cum;     // (b, H, nchunks, Q) inclusive cumsum of Delta*A_h within the chunk
    float* states;  // (b, nchunks, H, P, N)
    int64_t T, H, P, N, G, Q, nchunks;
    int x_f32;      // x is stored as fp32 whatever the dtype (the convolved input)
    // byte ranges of the buffers written (stores checked in SSM_BOUNDS_CHECK builds)
    int* status;
    Span out_s, final_s, dl_s, cum_s, states_s;
};

template <typename T>
__device__ __forceinline__ float ld(const char* base, int64_t idx) {
    return to_f32<T>(reinterpret_cast<const T*>(base)[idx]);
}

// an element of x, which is fp32 when it holds the convolved input
template <typename T>
__device__ __forceinline__ float ld_x(const SsdArgs& a, int64_t idx) {
    return a.x_f32 ? reinterpret_cast<const float*>(a.x)[idx] : ld<T>(a.x, idx);
}

// e^x: CUDA's accurate expf for fp32 inputs, the fast intrinsic for 16-bit inputs.
template <typename T>
__device__ __forceinline__ float exp_t(float x) {
    return sizeof(T) == 4 ? expf(x) : __expf(x);
}

// Delta and the inclusive cumulative sum of Delta * A_h over one chunk, into smem.
template <typename T>
__device__ void chunk_delta_cumsum(const SsdArgs& a, int64_t b, int64_t h, int64_t c,
                                   float* s_dl, float* s_cum, float* s_warp) {
    const int tid = threadIdx.x;
    const int64_t t0 = c * a.Q;
    const int len = (int)min(a.Q, a.T - t0);
    float dA = 0.0f;
    if (tid < len) {
        const float v = ld<T>(a.dt, (b * a.T + t0 + tid) * a.H + h) + (a.dt_bias ? a.dt_bias[h] : 0.0f);
        const float de = softplus_t<sizeof(T) == 4>(v);
        s_dl[tid] = de;
        dA = de * a.A[h];
    } else if (tid < a.Q) {
        s_dl[tid] = 0.0f;
    }
    // block inclusive scan of dA (blockDim == 256 >= Q)
    const int lane = tid & 31, warp = tid >> 5;
    float v = dA;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float w = lane < kThreads / 32 ? s_warp[lane] : 0.0f;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        if (lane < kThreads / 32) s_warp[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += s_warp[warp - 1];
    if (tid < a.Q) s_cum[tid] = v;  // rows past the end repeat the last sum
    __syncthreads();
}

// grid: (nchunks, H * nP * nN, b)
template <typename T>
__global__ void __launch_bounds__(kThreads) ssd_chunk_state(const SsdArgs a) {
    __shared__ float s_dl[256], s_cum[256], s_warp[8], s_w[kSub];
    __shared__ float s_x[kSub][kTile + 1];
    __shared__ float s_b[kSub][kTile + 1];
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const int nP = (int)((a.P + kTile - 1) / kTile), nN = (int)((a.N + kTile - 1) / kTile);
    const int64_t h = blockIdx.y / (nP * nN);
    const int pt = (blockIdx.y / nN) % nP, nt = blockIdx.y % nN;
    const int64_t g = h / (a.H / a.G);
    chunk_delta_cumsum<T>(a, b, h, c, s_dl, s_cum, s_warp);
    const int tid = threadIdx.x;
    const int64_t t0 = c * a.Q;
    const int len = (int)min(a.Q, a.T - t0);
    if (pt == 0 && nt == 0 && tid < a.Q) {
        const int64_t o = ((b * a.H + h) * a.nchunks + c) * a.Q + tid;
        store_checked(a.dl_s, &a.dl[o], s_dl[tid], a.status);
        store_checked(a.cum_s, &a.cum[o], s_cum[tid], a.status);
    }
    const float last = s_cum[len - 1];
    const int pi = (tid / 16) * 4, nj = (tid % 16) * 4;
    float acc[4][4] = {};
    for (int s0 = 0; s0 < len; s0 += kSub) {
        __syncthreads();
        for (int i = tid; i < kSub * kTile; i += kThreads) {
            const int r = i / kTile, q = i % kTile;
            const int64_t t = t0 + s0 + r;
            const int64_t p = (int64_t)pt * kTile + q, n = (int64_t)nt * kTile + q;
            const bool rok = s0 + r < len;
            s_x[r][q] = (rok && p < a.P) ? ld_x<T>(a, ((b * a.T + t) * a.H + h) * a.P + p) : 0.0f;
            s_b[r][q] = (rok && n < a.N) ? ld<T>(a.B, ((b * a.T + t) * a.G + g) * a.N + n) : 0.0f;
        }
        if (tid < kSub) {
            const int s = s0 + tid;
            s_w[tid] = s < len ? exp_t<T>(last - s_cum[s]) * s_dl[s] : 0.0f;
        }
        __syncthreads();
        for (int r = 0; r < kSub; ++r) {
            const float w = s_w[r];
            float xv[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = s_x[r][pi + i] * w;
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = s_b[r][nj + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], bv[j], acc[i][j]);
        }
    }
    float* S = a.states + (((b * a.nchunks + c) * a.H + h) * a.P) * a.N;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t p = (int64_t)pt * kTile + pi + i, n = (int64_t)nt * kTile + nj + j;
            if (p < a.P && n < a.N) store_checked(a.states_s, &S[p * a.N + n], acc[i][j], a.status);
        }
}

// grid: (ceil(P*N / 4 / 256), H, b).  In place: states[c] <- state entering chunk c,
// h_c = exp(s_last,c) h_{c-1} + S_c.  Each thread carries 4 consecutive state entries;
// the loads of S_c do not depend on the carry, so 8 chunks are fetched ahead.
constexpr int kPassAhead = 8;

__global__ void __launch_bounds__(kThreads) ssd_state_pass(const SsdArgs a) {
    const int64_t i4 = (int64_t)blockIdx.x * kThreads + threadIdx.x;  // float4 index
    const int64_t h = blockIdx.y, b = blockIdx.z;
    const int64_t PN = a.P * a.N;
    if (i4 * 4 >= PN) return;
    float4 st = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (a.init) st = *reinterpret_cast<const float4*>(a.init + (b * a.H + h) * PN + i4 * 4);
    const int64_t cstride = a.H * PN;  // floats between consecutive chunks of one head
    float* base = a.states + (b * a.nchunks * a.H + h) * PN + i4 * 4;
    const float* cum = a.cum + (b * a.H + h) * a.nchunks * a.Q;
    for (int64_t c0 = 0; c0 < a.nchunks; c0 += kPassAhead) {
        float4 S[kPassAhead];
        float dec[kPassAhead];
#pragma unroll
        for (int j = 0; j < kPassAhead; ++j) {
            const int64_t c = c0 + j;
            if (c < a.nchunks) {
                S[j] = *reinterpret_cast<const float4*>(base + c * cstride);
                const int len = (int)min(a.Q, a.T - c * a.Q);
                dec[j] = expf(cum[c * a.Q + len - 1]);
            }
        }
#pragma unroll
        for (int j = 0; j < kPassAhead; ++j) {
            const int64_t c = c0 + j;
            if (c < a.nchunks) {
                store_checked(a.states_s, reinterpret_cast<float4*>(base + c * cstride), st, a.status);
                st.x = fmaf(dec[j], st.x, S[j].x);
                st.y = fmaf(dec[j], st.y, S[j].y);
                st.z = fmaf(dec[j], st.z, S[j].z);
                st.w = fmaf(dec[j], st.w, S[j].w);
            }
        }
    }
    if (a.final_state) store_checked(a.final_s, reinterpret_cast<float4*>(a.final_state + (b * a.H + h) * PN + i4 * 4), st, a.status);
}

// The tensor-core path's carry.  S_c arrives in the split-ready layout of the
// tensor-core chunk-state kernel: the 8 values of (p, n..n+7) as two float4 at the byte
// offsets o and o + P*N*2 that their bf16 hi and lo halves take in the scan kernel's
// K-major h tile.  Each thread owns one such unit: it reads S_c there and writes
// h_{c-1} back in place as bf16 hi = bf16(h) and lo = bf16(h - hi), so the scan kernel
// copies the tiles straight into shared memory.  Initial and final states are fp32 in
// the plain (b, H, P, N) layout.  grid: (ceil(P*N / 8 / 256), H, b).
constexpr int kPassAheadSplit = 2;

__global__ void __launch_bounds__(kThreads) ssd_state_pass_split(const SsdArgs a) {
    // units in memory order: unit u sits at byte 16 u of each half, so consecutive
    // threads touch consecutive 16-byte pieces; u = (core-matrix block) * 8 + (p & 7)
    const int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t h = blockIdx.y, b = blockIdx.z;
    const int64_t PN = a.P * a.N;
    if (u * 8 >= PN) return;
    const int64_t blk = u >> 3, kb = a.N / 8;
    const int p = (int)((blk / kb) * 8 + (u & 7)), n0 = (int)(blk % kb) * 8;
    const uint32_t o = (uint32_t)(16 * u);  // == off_kmajor(p, n0, N)
    const int64_t half = PN * 2;  // bytes of the hi (or lo) tile
    float st[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) st[k] = a.init ? a.init[(b * a.H + h) * PN + p * a.N + n0 + k] : 0.0f;
    const int64_t cstride = a.H * PN * 4;  // bytes between consecutive chunks of one head
    char* base = reinterpret_cast<char*>(a.states + (b * a.nchunks * a.H + h) * PN);
    const float* cum = a.cum + (b * a.H + h) * a.nchunks * a.Q;
    for (int64_t c0 = 0; c0 < a.nchunks; c0 += kPassAheadSplit) {
        float4 S0[kPassAheadSplit], S1[kPassAheadSplit];
        float dec[kPassAheadSplit];
#pragma unroll
        for (int j = 0; j < kPassAheadSplit; ++j) {
            const int64_t c = c0 + j;
            if (c < a.nchunks) {
                S0[j] = *reinterpret_cast<const float4*>(base + c * cstride + o);
                S1[j] = *reinterpret_cast<const float4*>(base + c * cstride + half + o);
                const int len = (int)min(a.Q, a.T - c * a.Q);
                dec[j] = expf(cum[c * a.Q + len - 1]);
            }
        }
#pragma unroll
        for (int j = 0; j < kPassAheadSplit; ++j) {
            const int64_t c = c0 + j;
            if (c < a.nchunks) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 hv = __floats2bfloat162_rn(st[2 * k], st[2 * k + 1]);
                    const float2 hf = __bfloat1622float2(hv);
                    const __nv_bfloat162 lv = __floats2bfloat162_rn(st[2 * k] - hf.x, st[2 * k + 1] - hf.y);
                    hi[k] = *reinterpret_cast<const uint32_t*>(&hv);
                    lo[k] = *reinterpret_cast<const uint32_t*>(&lv);
                }
                store_checked(a.states_s, reinterpret_cast<uint4*>(base + c * cstride + o), make_uint4(hi[0], hi[1], hi[2], hi[3]), a.status);
                store_checked(a.states_s, reinterpret_cast<uint4*>(base + c * cstride + half + o), make_uint4(lo[0], lo[1], lo[2], lo[3]), a.status);
                const float s[8] = {S0[j].x, S0[j].y, S0[j].z, S0[j].w, S1[j].x, S1[j].y, S1[j].z, S1[j].w};
#pragma unroll
                for (int k = 0; k < 8; ++k) st[k] = fmaf(dec[j], st[k], s[k]);
            }
        }
    }
    if (a.final_state) {
#pragma unroll
        for (int k = 0; k < 8; ++k) store_checked(a.final_s, &a.final_state[(b * a.H + h) * PN + p * a.N + n0 + k], st[k], a.status);
    }
}

// grid: (nchunks, H * nP, b * nTq); output tile of 64 rows x 64 head channels.
template <typename T, bool GATE>
__global__ void __launch_bounds__(kThreads) ssd_chunk_scan(const SsdArgs a) {
    extern __shared__ __align__(16) float dsm[];
    const int nP = (int)((a.P + kTile - 1) / kTile);
    const int nTq = (int)((a.Q + kTile - 1) / kTile);
    const int64_t c = blockIdx.x;
    const int64_t h = blockIdx.y / nP;
    const int pt = blockIdx.y % nP;
    const int64_t b = blockIdx.z / nTq;
    const int tq = blockIdx.z % nTq;
    const int64_t g = h / (a.H / a.G);
    const int tid = threadIdx.x;
    const int64_t t0 = c * a.Q;
    const int len = (int)min(a.Q, a.T - t0);
    const int r0 = tq * kTile;  // first row of this tile inside the chunk
    if (r0 >= len) return;
    const int Nn = (int)a.N;
    // smem: cum[Q] dl[Q] | C tile [64][N+1] | B sub [32][N+1] | x sub [32][65] | G [64][33]
    float* s_cum = dsm;
    float* s_dl = s_cum + a.Q;
    float* s_c = s_dl + a.Q;
    float* s_b = s_c + kTile * (Nn + 1);
    float* s_x = s_b + kSub * (Nn + 1);
    float* s_g = s_x + kSub * (kTile + 1);
    for (int i = tid; i < a.Q; i += kThreads) {
        const int64_t o = ((b * a.H + h) * a.nchunks + c) * a.Q + i;
        s_cum[i] = a.cum[o];
        s_dl[i] = a.dl[o];
    }
    for (int i = tid; i < kTile * Nn; i += kThreads) {
        const int r = i / Nn, n = i % Nn;
        s_c[r * (Nn + 1) + n] = (r0 + r < len) ? ld<T>(a.C, ((b * a.T + t0 + r0 + r) * a.G + g) * a.N + n) : 0.0f;
    }
    __syncthreads();
    const int ti = (tid / 16) * 4, pj = (tid % 16) * 4;
    float acc[4][4] = {};
    const int s_end = min(len, r0 + kTile);
    for (int s0 = 0; s0 < s_end; s0 += kSub) {
        __syncthreads();
        for (int i = tid; i < kSub * Nn; i += kThreads) {
            const int r = i / Nn, n = i % Nn;
            s_b[r * (Nn + 1) + n] = (s0 + r < len) ? ld<T>(a.B, ((b * a.T + t0 + s0 + r) * a.G + g) * a.N + n) : 0.0f;
        }
        for (int i = tid; i < kSub * kTile; i += kThreads) {
            const int r = i / kTile, q = i % kTile;
            const int64_t p = (int64_t)pt * kTile + q;
            s_x[r * (kTile + 1) + q] = (s0 + r < len && p < a.P) ? ld_x<T>(a, ((b * a.T + t0 + s0 + r) * a.H + h) * a.P + p) : 0.0f;
        }
        __syncthreads();
        // G'[t][s] = (s <= t) (C_t . B_s) exp(cum_t - cum_s) Delta_s for the 64 x 32 block
        for (int i = tid; i < kTile * kSub; i += kThreads) {
            const int r = i / kSub, s = i % kSub;
            const int tt = r0 + r, ss = s0 + s;
            float v = 0.0f;
            if (ss <= tt && tt < len && ss < len) {
                const float* cr = s_c + r * (Nn + 1);
                const float* br = s_b + s * (Nn + 1);
                float dot = 0.0f;
                for (int n = 0; n < Nn; ++n) dot = fmaf(cr[n], br[n], dot);
                v = dot * exp_t<T>(s_cum[tt] - s_cum[ss]) * s_dl[ss];
            }
            s_g[r * (kSub + 1) + s] = v;
        }
        __syncthreads();
        for (int s = 0; s < kSub; ++s) {
            float gv[4], xv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) gv[i] = s_g[(ti + i) * (kSub + 1) + s];
#pragma unroll
            for (int j = 0; j < 4; ++j) xv[j] = s_x[s * (kTile + 1) + pj + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(gv[i], xv[j], acc[i][j]);
        }
    }
    // Y_off = exp(cum_t) * sum_n C_t[n] hin[p][n]
    const float* hin = a.states + (((b * a.nchunks + c) * a.H + h) * a.P) * a.N;
    float off[4][4] = {};
    for (int n0 = 0; n0 < Nn; n0 += kSub) {
        __syncthreads();
        // reuse s_x as hin sub-tile [32 n][65 p]
        for (int i = tid; i < kSub * kTile; i += kThreads) {
            const int nn = i / kTile, q = i % kTile;
            const int64_t p = (int64_t)pt * kTile + q;
            s_x[nn * (kTile + 1) + q] = (n0 + nn < Nn && p < a.P) ? hin[p * a.N + n0 + nn] : 0.0f;
        }
        __syncthreads();
        const int nlim = min(kSub, Nn - n0);
        for (int nn = 0; nn < nlim; ++nn) {
            float cv[4], hv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) cv[i] = s_c[(ti + i) * (Nn + 1) + n0 + nn];
#pragma unroll
            for (int j = 0; j < 4; ++j) hv[j] = s_x[nn * (kTile + 1) + pj + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) off[i][j] = fmaf(cv[i], hv[j], off[i][j]);
        }
    }
    const float Dh = a.D ? a.D[h] : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int tt = r0 + ti + i;
        if (tt >= len) continue;
        const float e = exp_t<T>(s_cum[tt]);
        const int64_t row = ((b * a.T + t0 + tt) * a.H + h) * a.P;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t p = (int64_t)pt * kTile + pj + j;
            if (p >= a.P) continue;
            const float xv = ld_x<T>(a, row + p);
            float y = acc[i][j] + e * off[i][j] + Dh * xv;
            if (GATE) y *= silu_t<sizeof(T) == 4>(ld<T>(a.z, row + p));
            store_checked(a.out_s, &reinterpret_cast<T*>(a.out)[row + p], from_f32<T>(y), a.status);
        }
    }
}

// The SSM_TUNE_SSD_CUDA_CORES override (1) keeps every shape on the CUDA-core kernels (a
// cross-check of the tensor-core kernels; both compute the same chunk algebra).
bool force_cuda_cores() { return tuning(1) == 1; }

struct SsdPlan {
    int64_t Q, nchunks;
    size_t dl_off, cum_off, st_off, total;
};

SsdPlan ssd_plan(const ScanArgs& a) {
    SsdPlan p;
    p.Q = a.chunk > 0 ? a.chunk : 256;
    p.nchunks = (a.seqlen + p.Q - 1) / p.Q;
    const size_t vec = (size_t)a.batch * a.nheads * p.nchunks * p.Q * sizeof(float);
    const size_t st = (size_t)a.batch * p.nchunks * a.nheads * a.headdim * a.dstate * sizeof(float);
    p.dl_off = 0;
    p.cum_off = align_up(vec, 256);
    p.st_off = p.cum_off + align_up(vec, 256);
    p.total = p.st_off + align_up(st, 256);
    return p;
}

template <typename T>
cudaError_t ssd_launch_typed(const ScanArgs& a, void* ws, cudaStream_t stream) {
    const SsdPlan pl = ssd_plan(a);
    SsdArgs s;
    s.x = (const char*)a.x;
    s.dt = (const char*)a.dt;
    s.z = (const char*)a.z;
    s.B = (const char*)a.B;
    s.C = (const char*)a.C;
    s.A = a.A;
    s.D = a.D;
    s.dt_bias = a.dt_bias;
    s.init = a.initial_state;
    s.out = (char*)a.out;
    s.final_state = a.final_state;
    s.dl = (float*)((char*)ws + pl.dl_off);
    s.cum = (float*)((char*)ws + pl.cum_off);
    s.states = (float*)((char*)ws + pl.st_off);
    s.T = a.seqlen;
    s.H = a.nheads;
    s.P = a.headdim;
    s.N = a.dstate;
    s.G = a.ngroups;
    s.Q = pl.Q;
    s.nchunks = pl.nchunks;
    s.x_f32 = a.x_f32;
    s.status = nullptr;
    if (kBoundsCheck) {
        cudaError_t e = device_status_address(&s.status);
        if (e != cudaSuccess) return e;
    }
    {
        const size_t vec = (size_t)a.batch * a.nheads * pl.nchunks * pl.Q * sizeof(float);
        s.out_s = span_of(a.out, (size_t)a.batch * a.seqlen * a.nheads * a.headdim * sizeof(T));
        s.final_s = span_of(a.final_state, (size_t)a.batch * a.nheads * a.headdim * a.dstate * sizeof(float));
        s.dl_s = span_of(s.dl, vec);
        s.cum_s = span_of(s.cum, vec);
        s.states_s = span_of(s.states, (size_t)a.batch * pl.nchunks * a.nheads * a.headdim * a.dstate * sizeof(float));
    }
    const unsigned nP = (unsigned)((a.headdim + kTile - 1) / kTile);
    const unsigned nN = (unsigned)((a.dstate + kTile - 1) / kTile);
    const unsigned nTq = (unsigned)((pl.Q + kTile - 1) / kTile);
    // The tensor-core kernels take x as an exact bf16 MMA operand, or as bf16 hi/lo
    // planes (the convolved input where ssd_conv_split holds); an fp32 x runs on the
    // CUDA-core kernels.
    const bool tc = pl.nchunks > 0 && !a.x_f32 && ssd_tc_supported(a, pl.Q) && !force_cuda_cores();
    if (a.x_lo && !tc) return cudaErrorInvalidValue;  // split planes exist only for the tc kernels
    if (tc) {
        SsdTcArgs t;
        t.x = (const __nv_bfloat16*)a.x;
        t.x_lo = (const __nv_bfloat16*)a.x_lo;
        t.dt = (const __nv_bfloat16*)a.dt;
        t.z = (const __nv_bfloat16*)a.z;
        t.B = (const __nv_bfloat16*)a.B;
        t.C = (const __nv_bfloat16*)a.C;
        t.A = a.A;
        t.D = a.D;
        t.dt_bias = a.dt_bias;
        t.out = (__nv_bfloat16*)a.out;
        t.dl = s.dl;
        t.cum = s.cum;
        t.states = s.states;
        t.T = a.seqlen;
        t.H = a.nheads;
        t.N = a.dstate;
        t.G = a.ngroups;
        t.Q = pl.Q;
        t.nchunks = pl.nchunks;
        t.out_s = s.out_s;
        t.dl_s = s.dl_s;
        t.cum_s = s.cum_s;
        t.states_s = s.states_s;
        cudaError_t e = ssd_tc_chunk_state(t, a.batch, stream);
        if (e != cudaSuccess) return e;
        cudaEvent_t t0 = timing_begin(stream, "ssd_state_pass_split");
        ssd_state_pass_split<<<dim3((unsigned)((a.headdim * a.dstate / 8 + kThreads - 1) / kThreads), (unsigned)a.nheads, (unsigned)a.batch), kThreads, 0, stream>>>(s);
        note_launch("ssd_state_pass_split", stream, t0);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return ssd_tc_chunk_scan(t, a.batch, a.z != nullptr, stream);
    }
    if (pl.nchunks > 0) {
        cudaEvent_t t0 = timing_begin(stream, "ssd_chunk_state");
        ssd_chunk_state<T><<<dim3((unsigned)pl.nchunks, (unsigned)a.nheads * nP * nN, (unsigned)a.batch), kThreads, 0, stream>>>(s);
        note_launch("ssd_chunk_state", stream, t0);
    }
    {
        cudaEvent_t t0 = timing_begin(stream, "ssd_state_pass");
        ssd_state_pass<<<dim3((unsigned)((a.headdim * a.dstate / 4 + kThreads - 1) / kThreads), (unsigned)a.nheads, (unsigned)a.batch), kThreads, 0, stream>>>(s);
        note_launch("ssd_state_pass", stream, t0);
    }
    if (pl.nchunks > 0) {
        const size_t smem = sizeof(float) * (2 * pl.Q + kTile * (a.dstate + 1) + kSub * (a.dstate + 1) +
                                             kSub * (kTile + 1) + kTile * (kSub + 1));
        const dim3 grid((unsigned)pl.nchunks, (unsigned)a.nheads * nP, (unsigned)a.batch * nTq);
        cudaEvent_t t0 = timing_begin(stream, "ssd_chunk_scan");
        if (a.z) {
            cudaFuncSetAttribute(ssd_chunk_scan<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            ssd_chunk_scan<T, true><<<grid, kThreads, smem, stream>>>(s);
        } else {
            cudaFuncSetAttribute(ssd_chunk_scan<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            ssd_chunk_scan<T, false><<<grid, kThreads, smem, stream>>>(s);
        }
        note_launch("ssd_chunk_scan", stream, t0);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t ssd_tc_forward_carry(const ScanArgs& a, int64_t Q, int64_t nchunks, const float* cum, float* states,
                                 float* final_state, cudaStream_t stream) {
    SsdArgs s = {};
    s.init = a.initial_state;
    s.final_state = final_state;
    s.cum = const_cast<float*>(cum);
    s.states = states;
    s.T = a.seqlen;
    s.H = a.nheads;
    s.P = a.headdim;
    s.N = a.dstate;
    s.G = a.ngroups;
    s.Q = Q;
    s.nchunks = nchunks;
    s.status = nullptr;
    if (kBoundsCheck) {
        const cudaError_t e = device_status_address(&s.status);
        if (e != cudaSuccess) return e;
    }
    s.final_s = span_of(final_state, (size_t)a.batch * a.nheads * a.headdim * a.dstate * sizeof(float));
    s.states_s = span_of(states, (size_t)a.batch * nchunks * a.nheads * a.headdim * a.dstate * sizeof(float));
    cudaEvent_t t0 = timing_begin(stream, "ssd_state_pass_split");
    ssd_state_pass_split<<<dim3((unsigned)((a.headdim * a.dstate / 8 + kThreads - 1) / kThreads), (unsigned)a.nheads,
                                (unsigned)a.batch),
                           kThreads, 0, stream>>>(s);
    note_launch("ssd_state_pass_split", stream, t0);
    return cudaGetLastError();
}

bool ssd_conv_split(const ScanArgs& a) {
    const SsdPlan pl = ssd_plan(a);
    return pl.nchunks > 0 && ssd_tc_supported(a, pl.Q) && !force_cuda_cores();
}

size_t ssd_workspace_bytes(const ScanArgs& a) {
    if (a.batch == 0) return 0;
    return ssd_plan(a).total;
}

cudaError_t ssd_launch(const ScanArgs& a, void* ws, cudaStream_t stream) {
    if (a.batch == 0) return cudaSuccess;
    if (a.dtype == 1) return ssd_launch_typed<__nv_bfloat16>(a, ws, stream);
    return ssd_launch_typed<float>(a, ws, stream);
}

}  // namespace ssm
