// Mamba-1 selective scan with a diagonal A (one decay per channel and state index).
//
// Operation ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里", 背景问题 and
// 第一步; skip term from the "引言：Attention的天花板" article, 基本原理; gate from
// "论文解读：Mamba — 线性时间的序列建模革命", 五 Mamba块架构), per batch b and channel c:
//   Delta_t = softplus(dt_t + dt_bias)
//   h_t[n]  = exp(Delta_t A[c,n]) h_{t-1}[n] + Delta_t B_t[n] x_t
//   y_t     = (sum_n C_t[n] h_t[n] + D x_t) * SiLU(z_t)
//
// Design (B300):
//  * The expanded state (b, T, d_inner, N) never leaves registers: each thread owns
//    NPT = NK / LPC state entries of one channel, LPC lanes cover one channel.
//  * Inputs are token-major (channels innermost).  A block owns CPB channels of one
//    group and walks time in tiles of 32 steps.  Each tile of x, dt, z, B, C is staged
//    into shared memory by 16-byte cp.async copies in a 3-deep pipeline, so HBM reads
//    are coalesced rows and overlap the arithmetic of the previous tiles.
//  * Per tile: (A) every thread computes softplus and Delta*x for a few (t, c) pairs and
//    converts B, C to fp32 (per-(t,c) work done once, not once per state entry);
//    (B) the scan: exp via ex2.approx, packed fp32x2 multiply/FMA for the decay, the
//    input term, the state update and the C.h partial sum; (C) the partial sums over the
//    LPC lanes are combined, D*x and the SiLU gate applied, and bf16/fp32 pairs stored.
//  * Time parallelism when there are few channels: the sequence is cut into segments.
//    A state-only pass computes each segment's local end state (from zero) and its
//    sum of Delta; the output pass folds those summaries into the segment's initial
//    state, h <- exp(A sum Delta_j) h + H_j, which is the affine combine
//    (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2) of the parallel-scan formulation
//    ("引言：Attention的天花板" article, 硬件感知算法).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kThreads = 128;
constexpr int kTT = 32;      // time steps per tile
constexpr int kStages = 3;   // cp.async pipeline depth

template <typename T, int NK, int LPC>
struct DiagCfg {
    static constexpr int NPT = NK / LPC;      // state entries per thread
    static constexpr int CPB = kThreads / LPC;  // channels per block
    static constexpr int kElem = (int)sizeof(T);
    static constexpr int kRowBytes = CPB * kElem;         // one time row of the x/dt/z tile
    static constexpr int kRowChunks = kRowBytes / 16;
    static constexpr int kXBytes = kTT * kRowBytes;
    static constexpr int kBCRowBytes = NK * kElem;
    static constexpr int kBCRowChunks = kBCRowBytes / 16;
    static constexpr int kBCBytes = kTT * kBCRowBytes;
    static constexpr int kStageBytes = 3 * kXBytes + 2 * kBCBytes;
    // working buffers
    static constexpr int kDuBytes = kTT * CPB * 8;        // float2 (Delta, Delta*x)
    static constexpr int kBfBytes = kTT * NK * 4;         // fp32 B (and C)
    static constexpr int kYpBytes = kTT * CPB * LPC * 4;  // partial C.h per lane
    static constexpr int kSmemBytes = kStages * kStageBytes + kDuBytes + 2 * kBfBytes + kYpBytes;
    static_assert(NK % LPC == 0 && NPT % 4 == 0, "NPT must be a multiple of 4");
    static_assert(kRowBytes % 16 == 0 && kBCRowBytes % 16 == 0, "16-byte rows");
    static_assert((CPB / 2) * kTT % kThreads == 0, "pair mapping");
};

struct DiagKernelArgs {
    const char* x;
    const char* dt;
    const char* z;
    const char* B;
    const char* C;
    const float* A;
    const float* D;
    const float* dt_bias;
    const float* init;   // initial state (b, dim, N) or null
    char* out;
    float* final_state;  // (b, dim, N) or null
    float* seg_h;        // (nseg-1, b, dim, N): local end state of each segment but the last
    float* seg_dsum;     // (nseg-1, b, dim): sum of Delta over the segment
    int64_t T, dim, N, G, cpg;
    int64_t seg_len;
    int nseg, tiles_per_group;
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

template <typename T>
__device__ __forceinline__ float2 load_pair(const char* p);
template <>
__device__ __forceinline__ float2 load_pair<float>(const char* p) {
    return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 load_pair<__nv_bfloat16>(const char* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

template <typename T>
__device__ __forceinline__ void store_pair(char* p, float2 v);
template <>
__device__ __forceinline__ void store_pair<float>(char* p, float2 v) {
    *reinterpret_cast<float2*>(p) = v;
}
template <>
__device__ __forceinline__ void store_pair<__nv_bfloat16>(char* p, float2 v) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
}

// STATE_ONLY: compute each segment's local end state from zero (segments 0..nseg-2).
// Otherwise: full output pass over every segment with the folded initial state.
template <typename T, int NK, int LPC, bool STATE_ONLY, bool GATE>
__global__ void __launch_bounds__(kThreads) diag_scan_kernel(const DiagKernelArgs a) {
    using Cfg = DiagCfg<T, NK, LPC>;
    constexpr int NPT = Cfg::NPT, CPB = Cfg::CPB, E = Cfg::kElem;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* stage0 = smem;
    float2* du = reinterpret_cast<float2*>(smem + kStages * Cfg::kStageBytes);
    float* Bf = reinterpret_cast<float*>(smem + kStages * Cfg::kStageBytes + Cfg::kDuBytes);
    float* Cf = Bf + kTT * NK;
    float* yp = Cf + kTT * NK;

    const int tid = threadIdx.x;
    const int group = blockIdx.x / a.tiles_per_group;
    const int64_t c_begin = (int64_t)group * a.cpg + (int64_t)(blockIdx.x % a.tiles_per_group) * CPB;
    const int64_t c_end = (int64_t)(group + 1) * a.cpg;  // exclusive, within this group
    const int seg = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t t_begin = (int64_t)seg * a.seg_len;
    const int64_t t_end = min(a.T, t_begin + a.seg_len);
    const int ntiles = (int)((t_end - t_begin + kTT - 1) / kTT);

    // scan-phase role: channel cc within the block, lane group g over the state index
    const int cc = tid / LPC;
    const int g = tid % LPC;
    const int64_t c = c_begin + cc;
    const bool c_ok = c < c_end;

    float A2[NPT];
    float h[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
        const int n = g * NPT + j;
        A2[j] = (c_ok && n < a.N) ? a.A[c * a.N + n] * kLog2e : 0.0f;
        h[j] = 0.0f;
    }
    if (!STATE_ONLY) {
        // state entering this segment: the initial state decayed through the earlier
        // segments plus their local end states
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const int n = g * NPT + j;
            if (c_ok && n < a.N && a.init) h[j] = a.init[(b * a.dim + c) * a.N + n];
        }
        for (int s = 0; s < seg; ++s) {
            if (!c_ok) break;
            const float dsum = a.seg_dsum[((int64_t)s * gridDim.z + b) * a.dim + c];
            const float* Hs = a.seg_h + (((int64_t)s * gridDim.z + b) * a.dim + c) * a.N;
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const int n = g * NPT + j;
                if (n < a.N) h[j] = ex2(A2[j] * dsum) * h[j] + Hs[n];
            }
        }
    }

    // pair role for phases A and C: channels (2*cp, 2*cp+1) of the tile, rows r0 + k*RS
    constexpr int PAIRS = CPB / 2;
    constexpr int RS = kThreads / PAIRS;  // rows handled per sweep
    const int cp = tid % PAIRS;
    const int r0 = tid / PAIRS;
    const int64_t cA = c_begin + 2 * cp;
    const bool pair_ok = cA < c_end;  // cpg is even (16-byte rows), so both or neither
    const float bias0 = (pair_ok && a.dt_bias) ? a.dt_bias[cA] : 0.0f;
    const float bias1 = (pair_ok && a.dt_bias) ? a.dt_bias[cA + 1] : 0.0f;
    const float d0 = (pair_ok && a.D) ? a.D[cA] : 0.0f;
    const float d1 = (pair_ok && a.D) ? a.D[cA + 1] : 0.0f;
    float dsum0 = 0.0f, dsum1 = 0.0f;  // running sum of Delta (state-only pass)

    const int64_t row_stride = a.dim * E;     // bytes between consecutive time rows
    const int64_t bc_stride = a.G * a.N * E;  // bytes between consecutive B/C rows
    const char* bc_off_B = a.B + (int64_t)group * a.N * E;
    const char* bc_off_C = a.C + (int64_t)group * a.N * E;

    auto issue_tile = [&](int k) {
        if (k < ntiles) {
            unsigned char* st = stage0 + (k % kStages) * Cfg::kStageBytes;
            const int64_t t0 = t_begin + (int64_t)k * kTT;
            const int rows = (int)min((int64_t)kTT, t_end - t0);
            for (int i = tid; i < kTT * Cfg::kRowChunks; i += kThreads) {
                const int r = i / Cfg::kRowChunks, q = i % Cfg::kRowChunks;
                const int64_t ch = c_begin + q * (16 / E);
                const bool ok = r < rows && ch < c_end;
                const int64_t off = ok ? ((b * a.T + t0 + r) * row_stride + ch * E) : 0;
                cp_async16(st + r * Cfg::kRowBytes + q * 16, a.x + off, ok);
                cp_async16(st + Cfg::kXBytes + r * Cfg::kRowBytes + q * 16, a.dt + off, ok);
                if (GATE && !STATE_ONLY)
                    cp_async16(st + 2 * Cfg::kXBytes + r * Cfg::kRowBytes + q * 16, a.z + off, ok);
            }
            for (int i = tid; i < kTT * Cfg::kBCRowChunks; i += kThreads) {
                const int r = i / Cfg::kBCRowChunks, q = i % Cfg::kBCRowChunks;
                const bool ok = r < rows && q * (16 / E) < a.N;
                const int64_t off = ok ? ((b * a.T + t0 + r) * bc_stride + q * 16) : 0;
                unsigned char* dB = st + 3 * Cfg::kXBytes + r * Cfg::kBCRowBytes + q * 16;
                cp_async16(dB, bc_off_B + off, ok);
                if (!STATE_ONLY) cp_async16(dB + Cfg::kBCBytes, bc_off_C + off, ok);
            }
        }
        cp_async_commit();
    };

#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) issue_tile(k);

    for (int k = 0; k < ntiles; ++k) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        issue_tile(k + kStages - 1);
        const unsigned char* st = stage0 + (k % kStages) * Cfg::kStageBytes;
        const int64_t t0 = t_begin + (int64_t)k * kTT;
        const int rows = (int)min((int64_t)kTT, t_end - t0);

        // ---- phase A: Delta and Delta*x per (t, c); B, C to fp32
#pragma unroll
        for (int kk = 0; kk < kTT / RS; ++kk) {
            const int r = r0 + kk * RS;
            const float2 dtv = load_pair<T>((const char*)st + Cfg::kXBytes + r * Cfg::kRowBytes + 2 * cp * E);
            const float2 xv = load_pair<T>((const char*)st + r * Cfg::kRowBytes + 2 * cp * E);
            const float de0 = softplus(dtv.x + bias0);
            const float de1 = softplus(dtv.y + bias1);
            float4 v;
            v.x = de0;
            v.y = de0 * xv.x;
            v.z = de1;
            v.w = de1 * xv.y;
            *reinterpret_cast<float4*>(&du[r * CPB + 2 * cp]) = v;
            if (STATE_ONLY && r < rows) {
                dsum0 += de0;
                dsum1 += de1;
            }
        }
        for (int i = tid; i < kTT * NK / 2; i += kThreads) {
            const float2 bv = load_pair<T>((const char*)st + 3 * Cfg::kXBytes + i * 2 * E);
            *reinterpret_cast<float2*>(&Bf[2 * i]) = bv;
            if (!STATE_ONLY) {
                const float2 cv = load_pair<T>((const char*)st + 3 * Cfg::kXBytes + Cfg::kBCBytes + i * 2 * E);
                *reinterpret_cast<float2*>(&Cf[2 * i]) = cv;
            }
        }
        __syncthreads();

        // ---- phase B: the recurrence over this tile's rows
        for (int r = 0; r < rows; ++r) {
            const float2 dv = du[r * CPB + cc];
            const float2 dd = make_float2(dv.x, dv.x);
            const float2 uu = make_float2(dv.y, dv.y);
            float2 y2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < NPT; j += 4) {
                const float4 bq = *reinterpret_cast<const float4*>(&Bf[r * NK + g * NPT + j]);
                const float2 dA0 = __fmul2_rn(dd, make_float2(A2[j], A2[j + 1]));
                const float2 dA1 = __fmul2_rn(dd, make_float2(A2[j + 2], A2[j + 3]));
                const float2 a0 = make_float2(ex2(dA0.x), ex2(dA0.y));
                const float2 a1 = make_float2(ex2(dA1.x), ex2(dA1.y));
                const float2 ub0 = __fmul2_rn(uu, make_float2(bq.x, bq.y));
                const float2 ub1 = __fmul2_rn(uu, make_float2(bq.z, bq.w));
                const float2 h0 = __ffma2_rn(a0, make_float2(h[j], h[j + 1]), ub0);
                const float2 h1 = __ffma2_rn(a1, make_float2(h[j + 2], h[j + 3]), ub1);
                h[j] = h0.x;
                h[j + 1] = h0.y;
                h[j + 2] = h1.x;
                h[j + 3] = h1.y;
                if (!STATE_ONLY) {
                    const float4 cq = *reinterpret_cast<const float4*>(&Cf[r * NK + g * NPT + j]);
                    y2 = __ffma2_rn(make_float2(cq.x, cq.y), h0, y2);
                    y2 = __ffma2_rn(make_float2(cq.z, cq.w), h1, y2);
                }
            }
            if (!STATE_ONLY) yp[(r * CPB + cc) * LPC + g] = y2.x + y2.y;
        }

        if (!STATE_ONLY) {
            __syncthreads();
            // ---- phase C: combine the LPC partial sums, skip term, gate, store
#pragma unroll
            for (int kk = 0; kk < kTT / RS; ++kk) {
                const int r = r0 + kk * RS;
                if (r >= rows || !pair_ok) continue;
                float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
                for (int q = 0; q < LPC; ++q) {
                    y0 += yp[(r * CPB + 2 * cp) * LPC + q];
                    y1 += yp[(r * CPB + 2 * cp + 1) * LPC + q];
                }
                const float2 xv = load_pair<T>((const char*)st + r * Cfg::kRowBytes + 2 * cp * E);
                y0 = fmaf(d0, xv.x, y0);
                y1 = fmaf(d1, xv.y, y1);
                if (GATE) {
                    const float2 zv = load_pair<T>((const char*)st + 2 * Cfg::kXBytes + r * Cfg::kRowBytes + 2 * cp * E);
                    y0 *= silu(zv.x);
                    y1 *= silu(zv.y);
                }
                store_pair<T>(a.out + (b * a.T + t0 + r) * row_stride + cA * E, make_float2(y0, y1));
            }
        }
    }
    cp_async_wait<0>();

    if (STATE_ONLY) {
        // local end state and Delta sum of this segment
        if (c_ok) {
            float* Hs = a.seg_h + (((int64_t)seg * gridDim.z + b) * a.dim + c) * a.N;
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const int n = g * NPT + j;
                if (n < a.N) Hs[n] = h[j];
            }
        }
        // Delta sums: the pair role accumulated rows r0, r0+RS, ...; reduce over the RS
        // threads that share a pair (they are tid = cp + PAIRS * k)
        __syncthreads();
        float* red = yp;  // reuse: RS x CPB floats
        red[r0 * CPB + 2 * cp] = dsum0;
        red[r0 * CPB + 2 * cp + 1] = dsum1;
        __syncthreads();
        if (tid < CPB) {
            float s = 0.0f;
            for (int k = 0; k < RS; ++k) s += red[k * CPB + tid];
            const int64_t cc2 = c_begin + tid;
            if (cc2 < c_end) a.seg_dsum[((int64_t)seg * gridDim.z + b) * a.dim + cc2] = s;
        }
    } else if (a.final_state && seg == a.nseg - 1 && c_ok) {
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const int n = g * NPT + j;
            if (n < a.N) a.final_state[(b * a.dim + c) * a.N + n] = h[j];
        }
    }
}

// ---- host side ---------------------------------------------------------------

struct Plan {
    int NK;
    int LPC;
    int64_t seg_len;
    int nseg;
    int tiles_per_group;
    int blocks_x;
};

int pick_nk(int64_t N) {
    if (N <= 8) return 8;
    if (N <= 16) return 16;
    if (N <= 32) return 32;
    return 64;
}

Plan make_plan(const ScanArgs& a) {
    Plan p;
    p.NK = pick_nk(a.dstate);
    p.LPC = p.NK == 8 ? 2 : 4;  // 4 state entries per lane (2 lanes/ch for N <= 8)
    const int cpb = kThreads / p.LPC;
    const int64_t cpg = a.nheads / a.ngroups;
    p.tiles_per_group = (int)((cpg + cpb - 1) / cpb);
    p.blocks_x = (int)(a.ngroups * p.tiles_per_group);
    const int64_t units = (int64_t)p.blocks_x * a.batch;
    // Aim for >= 4 resident blocks on each of the B300's 148 SMs; split time only when
    // channels are scarce.  (A fixed count keeps the plan, and so the workspace size, a
    // function of the shape alone.)
    const int sms = 148;
    const int64_t target = (int64_t)sms * 4;
    int64_t seg_len;
    if (a.chunk > 0) {
        seg_len = a.chunk;
    } else {
        int64_t nseg = units > 0 ? (target + units - 1) / units : 1;
        nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, a.seqlen / 128));
        seg_len = (a.seqlen + nseg - 1) / nseg;
    }
    seg_len = std::max<int64_t>(kTT, (seg_len + kTT - 1) / kTT * kTT);
    p.seg_len = seg_len;
    p.nseg = (int)std::max<int64_t>(1, (a.seqlen + seg_len - 1) / seg_len);
    return p;
}

template <typename T, int NK, int LPC, bool STATE_ONLY, bool GATE>
cudaError_t launch_one(const DiagKernelArgs& ka, dim3 grid, cudaStream_t stream) {
    using Cfg = DiagCfg<T, NK, LPC>;
    auto kern = diag_scan_kernel<T, NK, LPC, STATE_ONLY, GATE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, Cfg::kSmemBytes, stream>>>(ka);
    note_launches(1);
    return cudaGetLastError();
}

template <typename T, int NK, int LPC>
cudaError_t launch_typed(const ScanArgs& a, const Plan& p, void* ws, cudaStream_t stream) {
    DiagKernelArgs ka;
    ka.x = (const char*)a.x;
    ka.dt = (const char*)a.dt;
    ka.z = (const char*)a.z;
    ka.B = (const char*)a.B;
    ka.C = (const char*)a.C;
    ka.A = a.A;
    ka.D = a.D;
    ka.dt_bias = a.dt_bias;
    ka.init = a.initial_state;
    ka.out = (char*)a.out;
    ka.final_state = a.final_state;
    ka.T = a.seqlen;
    ka.dim = a.nheads;
    ka.N = a.dstate;
    ka.G = a.ngroups;
    ka.cpg = a.nheads / a.ngroups;
    ka.seg_len = p.seg_len;
    ka.nseg = p.nseg;
    ka.tiles_per_group = p.tiles_per_group;
    ka.seg_h = nullptr;
    ka.seg_dsum = nullptr;
    if (p.nseg > 1) {
        const size_t hbytes = (size_t)(p.nseg - 1) * a.batch * a.nheads * a.dstate * sizeof(float);
        ka.seg_h = (float*)ws;
        ka.seg_dsum = (float*)((char*)ws + align_up(hbytes, 256));
        const dim3 g1(p.blocks_x, p.nseg - 1, (unsigned)a.batch);
        cudaError_t e = launch_one<T, NK, LPC, true, false>(ka, g1, stream);
        if (e != cudaSuccess) return e;
    }
    const dim3 g2(p.blocks_x, p.nseg, (unsigned)a.batch);
    if (a.z) return launch_one<T, NK, LPC, false, true>(ka, g2, stream);
    return launch_one<T, NK, LPC, false, false>(ka, g2, stream);
}

template <typename T>
cudaError_t launch_dtype(const ScanArgs& a, const Plan& p, void* ws, cudaStream_t stream) {
    switch (p.NK) {
        case 8: return launch_typed<T, 8, 2>(a, p, ws, stream);
        case 16: return launch_typed<T, 16, 4>(a, p, ws, stream);
        case 32: return launch_typed<T, 32, 4>(a, p, ws, stream);
        default: return launch_typed<T, 64, 4>(a, p, ws, stream);
    }
}

}  // namespace

size_t diag_workspace_bytes(const ScanArgs& a) {
    if (a.batch == 0 || a.seqlen == 0) return 0;
    const Plan p = make_plan(a);
    if (p.nseg <= 1) return 0;
    const size_t hbytes = (size_t)(p.nseg - 1) * a.batch * a.nheads * a.dstate * sizeof(float);
    const size_t dbytes = (size_t)(p.nseg - 1) * a.batch * a.nheads * sizeof(float);
    return align_up(hbytes, 256) + align_up(dbytes, 256);
}

cudaError_t diag_launch(const ScanArgs& a, void* ws, cudaStream_t stream) {
    if (a.batch == 0) return cudaSuccess;
    const Plan p = make_plan(a);
    if (a.dtype == 1) return launch_dtype<__nv_bfloat16>(a, p, ws, stream);
    return launch_dtype<float>(a, p, ws, stream);
}

}  // namespace ssm
