// Complex diagonal selective scan: the rotating, complex-valued state update read for
// Mamba-3 ("状态空间模型与 Mamba：不用注意力读取长序列的方法", the Mamba-3 paragraph: an
// input-dependent rotation in the state update, read as underdamped oscillation;
// "基础知识：Mamba 与混合 SSM 架构", section 6: complex-valued state update).  Per batch b,
// channel c and complex state entry n:
//   Delta_t = softplus(dt_t + dt_bias)
//   h_t[n]  = exp(Delta_t A[c,n]) h_{t-1}[n] + Delta_t B_t[n] x_t          (complex)
//   y_t     = (Re(sum_n C_t[n] h_t[n]) + D x_t) * SiLU(z_t)
// exp(Delta A) = e^{Delta Re A} (cos(Delta Im A) + i sin(Delta Im A)): a decay and a
// rotation whose angle follows the input through Delta.
//
// Design (B300): the same layout of work as the real diagonal scan, with simpler phases.
//  * LPC lanes own one channel, four complex entries each (fp32 re/im pairs in
//    registers); a block of 128 threads owns CPB channels of one group.
//  * Time is walked in tiles of 16 steps.  Each tile's x, dt, z, B, C rows are staged in
//    shared memory by 16-byte cp.async copies two tiles ahead (a 3-deep ring).
//  * Per tile three phases separated by block barriers: (1) Delta and Delta*x per (t, c),
//    once per channel and step; (2) the recurrence, each lane over its entries for the
//    16 steps, writing its partial Re(C.h) per (t, c); (3) the partials summed, D*x,
//    the SiLU gate, the store.
//  * The per-entry work is one ex2 (decay), one sin and one cos (rotation; the angle is
//    first reduced to [-pi, pi]) on the SFU for 16-bit inputs, or CUDA's expf/sincosf for
//    fp32 inputs, and ten FP32 operations.
//  * Few channels: the sequence is cut into segments; a state-only pass writes each
//    segment's local end state from zero and its sum of Delta, and the output pass folds
//    them into its entering state, h <- exp(A sum Delta) h + H_j (the affine combine of
//    the parallel-scan formulation, "引言：Attention的天花板" article, 硬件感知算法).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kCTT = 16;       // time steps per tile
constexpr int kCStages = 3;    // cp.async ring
constexpr int kCThreads = 128;
constexpr int kEPL = 4;        // complex entries per lane (the B/C tile reads below take
                               // exactly four: two float4 of (re, im) pairs)
static_assert(kEPL == 4, "the recurrence loads a lane's B and C entries as two float4");
constexpr float kTwoPi = 6.283185307179586f;
constexpr float kInvTwoPi = 0.15915494309189535f;

template <typename T, int NK>
struct CCfg {
    static constexpr int LPC = NK / kEPL;               // lanes per channel
    static constexpr int CPB = kCThreads / LPC;          // channels per block
    static constexpr int E = (int)sizeof(T);
    static constexpr int kRowBytes = CPB * E;            // one time row of x / dt / z
    static constexpr int kRowChunks = kRowBytes / 16;
    static constexpr int kXBytes = kCTT * kRowBytes;
    static constexpr int kBCRowBytes = NK * 2 * E;       // one time row of B (re, im pairs)
    static constexpr int kBCRowChunks = kBCRowBytes / 16;
    static constexpr int kBCBytes = kCTT * kBCRowBytes;
    static constexpr int kStageBytes = 3 * kXBytes + 2 * kBCBytes;
    static constexpr int kDuBytes = kCTT * CPB * 8;      // (Delta, Delta x) per (t, c)
    static constexpr int kYsBytes = kCTT * CPB * LPC * 4;
    static constexpr int kBfBytes = kCTT * NK * 8;        // B (or C) of a tile as fp32 (re, im)
    static constexpr int kSmem = kCStages * kStageBytes + kDuBytes + kYsBytes + 2 * kBfBytes;
    static_assert(kRowBytes % 16 == 0 && kBCRowBytes % 16 == 0, "16-byte rows");
};

struct CDiagArgs {
    const char* x;
    const char* dt;
    const char* z;
    const char* B;        // (b, T, G, N, 2)
    const char* C;
    const float* A;       // (dim, N, 2)
    const float* D;
    const float* dt_bias;
    const float* init;    // (b, dim, N, 2) or null
    char* out;
    float* final_state;   // (b, dim, N, 2) or null
    float* seg_h;         // (nseg-1, b, dim, N, 2)
    float* seg_dsum;      // (nseg-1, b, dim)
    int64_t T, dim, N, G, cpg, seg_len;
    int nseg, tiles_per_group;
    // byte ranges of the buffers written (stores checked in SSM_BOUNDS_CHECK builds)
    int* status;
    Span out_s, final_s, segh_s, segd_s;
};

__device__ __forceinline__ void ccp_async16(void* smem, const void* gmem, bool valid) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(valid ? 16 : 0));
}

template <typename T>
__device__ __forceinline__ float2 cld2(const unsigned char* p);
template <>
__device__ __forceinline__ float2 cld2<float>(const unsigned char* p) {
    return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 cld2<__nv_bfloat16>(const unsigned char* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// exp(d * A) for A = (re, im): (e^{d re} cos(d im), e^{d re} sin(d im)).  16-bit inputs
// (a.x holding re * log2 e): ex2 on the SFU and sin/cos of the angle reduced to
// [-pi, pi] (where the SFU's approximations are accurate), the two products as one
// packed multiply; fp32 inputs: CUDA's expf and sincosf.
template <bool PRECISE>
__device__ __forceinline__ float2 cexp_da(float d, float2 a) {
    float s, c;
    if (PRECISE) {
        const float r = expf(d * a.x);
        sincosf(d * a.y, &s, &c);
        return make_float2(r * c, r * s);
    }
    const float r = ex2(d * a.x);
    float th = d * a.y;
    th = fmaf(-kTwoPi, rintf(th * kInvTwoPi), th);
    asm("sin.approx.ftz.f32 %0, %1;" : "=f"(s) : "f"(th));
    asm("cos.approx.ftz.f32 %0, %1;" : "=f"(c) : "f"(th));
    return __fmul2_rn(make_float2(r, r), make_float2(c, s));
}

// STATE_ONLY: each segment's local end state (from zero) and its sum of Delta, for the
// segments 0..nseg-2.  Otherwise the output pass over every segment.
// grid (blocks over the groups' channels, segments, batch); 128 threads.
template <typename T, int NK, bool STATE_ONLY, bool GATE>
__global__ void __launch_bounds__(kCThreads) cdiag_scan_kernel(const CDiagArgs a) {
    using Cfg = CCfg<T, NK>;
    constexpr int LPC = Cfg::LPC, CPB = Cfg::CPB, E = Cfg::E;
    constexpr bool PRECISE = sizeof(T) == 4;
    extern __shared__ __align__(128) unsigned char smem[];
    float2* du = reinterpret_cast<float2*>(smem + kCStages * Cfg::kStageBytes);  // [kCTT][CPB]
    float* ys = reinterpret_cast<float*>(smem + kCStages * Cfg::kStageBytes + Cfg::kDuBytes);  // [kCTT][CPB][LPC]
    float2* Bf = reinterpret_cast<float2*>(smem + kCStages * Cfg::kStageBytes + Cfg::kDuBytes + Cfg::kYsBytes);  // [kCTT][NK]
    float2* Cf = Bf + kCTT * NK;                                                                                // [kCTT][NK]

    const int tid = threadIdx.x;
    const int group = blockIdx.x / a.tiles_per_group;
    const int64_t c_begin = (int64_t)group * a.cpg + (int64_t)(blockIdx.x % a.tiles_per_group) * CPB;
    const int64_t c_end = (int64_t)(group + 1) * a.cpg;
    const int chans = (int)min((int64_t)CPB, c_end - c_begin);
    const int seg = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t t_begin = (int64_t)seg * a.seg_len;
    const int64_t t_end = min(a.T, t_begin + a.seg_len);
    const int rows_total = (int)(t_end - t_begin);
    const int ntiles = (rows_total + kCTT - 1) / kCTT;

    // recurrence role: channel cc, lane g, complex entries g*kEPL + j
    const int cc = tid / LPC, g = tid % LPC;
    const int64_t c = c_begin + cc;
    const bool c_ok = cc < chans;
    float2 Ac[kEPL], h[kEPL];
#pragma unroll
    for (int j = 0; j < kEPL; ++j) {
        const int n = g * kEPL + j;
        const bool ok = c_ok && n < a.N;
        // the decay rate pre-scaled by log2 e for the ex2 of 16-bit inputs
        Ac[j] = ok ? make_float2(a.A[(c * a.N + n) * 2] * (PRECISE ? 1.0f : kLog2e), a.A[(c * a.N + n) * 2 + 1])
                   : make_float2(0.0f, 0.0f);
        h[j] = make_float2(0.0f, 0.0f);
    }
    if (!STATE_ONLY && c_ok) {
        // state entering the segment: the initial state carried through the earlier
        // segments' summaries
#pragma unroll
        for (int j = 0; j < kEPL; ++j) {
            const int n = g * kEPL + j;
            if (a.init && n < a.N) {
                const float* p = a.init + ((b * a.dim + c) * a.N + n) * 2;
                h[j] = make_float2(p[0], p[1]);
            }
        }
        for (int s = 0; s < seg; ++s) {
            const float ds = a.seg_dsum[((int64_t)s * gridDim.z + b) * a.dim + c];
            const float* Hs = a.seg_h + (((int64_t)s * gridDim.z + b) * a.dim + c) * a.N * 2;
#pragma unroll
            for (int j = 0; j < kEPL; ++j) {
                const int n = g * kEPL + j;
                if (n >= a.N) continue;
                const float2 e = cexp_da<PRECISE>(ds, Ac[j]);
                h[j] = make_float2(e.x * h[j].x - e.y * h[j].y + Hs[2 * n], e.x * h[j].y + e.y * h[j].x + Hs[2 * n + 1]);
            }
        }
    }

    const int64_t row_stride = a.dim * E;
    const int64_t bc_stride = a.G * a.N * 2 * E;
    const int64_t row_base = (b * a.T + t_begin) * row_stride;
    const int64_t bc_base = (b * a.T + t_begin) * bc_stride + (int64_t)group * a.N * 2 * E;
    auto stage = [&](int k) { return smem + (k % kCStages) * Cfg::kStageBytes; };
    auto issue = [&](int k) {
        if (k < ntiles) {
            unsigned char* st = stage(k);
            const int rows = min(kCTT, rows_total - k * kCTT);
            for (int i = tid; i < kCTT * Cfg::kRowChunks; i += kCThreads) {
                const int r = i / Cfg::kRowChunks, q = i % Cfg::kRowChunks;
                const bool ok = r < rows && q * (16 / E) < chans;
                const int64_t off = ok ? row_base + (int64_t)(k * kCTT + r) * row_stride + c_begin * E + q * 16 : 0;
                ccp_async16(st + r * Cfg::kRowBytes + q * 16, a.x + off, ok);
                ccp_async16(st + Cfg::kXBytes + r * Cfg::kRowBytes + q * 16, a.dt + off, ok);
                if (GATE && !STATE_ONLY) ccp_async16(st + 2 * Cfg::kXBytes + r * Cfg::kRowBytes + q * 16, a.z + off, ok);
            }
            for (int i = tid; i < kCTT * Cfg::kBCRowChunks; i += kCThreads) {
                const int r = i / Cfg::kBCRowChunks, q = i % Cfg::kBCRowChunks;
                const bool ok = r < rows && q * 16 < a.N * 2 * E;
                const int64_t off = ok ? bc_base + (int64_t)(k * kCTT + r) * bc_stride + q * 16 : 0;
                unsigned char* dst = st + 3 * Cfg::kXBytes + r * Cfg::kBCRowBytes + q * 16;
                ccp_async16(dst, a.B + off, ok);
                if (!STATE_ONLY) ccp_async16(dst + Cfg::kBCBytes, a.C + off, ok);
            }
        }
        asm volatile("cp.async.commit_group;\n" ::);
    };

    float dsum = 0.0f;  // sum of Delta of this thread's prep items (state-only pass)
    issue(0);
    issue(1);
    for (int k = 0; k < ntiles; ++k) {
        asm volatile("cp.async.wait_group 1;\n" ::);
        __syncthreads();  // tile k landed; the previous tile's readers are done
        issue(k + 2);
        const unsigned char* st = stage(k);
        const int rows = min(kCTT, rows_total - k * kCTT);
        // (1) Delta and Delta x per (t, c); rows past the tile's end get Delta 0.  B and C
        // of the tile to fp32 (re, im) pairs, once for all the block's channels.
        for (int i = tid; i < kCTT * CPB; i += kCThreads) {
            const int r = i / CPB, ch = i % CPB;
            float dl = 0.0f, u = 0.0f;
            if (r < rows && ch < chans) {
                const float dtv = to_f32<T>(*reinterpret_cast<const T*>(st + Cfg::kXBytes + r * Cfg::kRowBytes + ch * E));
                const float xv = to_f32<T>(*reinterpret_cast<const T*>(st + r * Cfg::kRowBytes + ch * E));
                dl = softplus_t<PRECISE>(dtv + (a.dt_bias ? a.dt_bias[c_begin + ch] : 0.0f));
                u = dl * xv;
            }
            du[r * CPB + ch] = make_float2(dl, u);
            if (STATE_ONLY) dsum += dl;
        }
        for (int i = tid; i < kCTT * NK; i += kCThreads) {
            const unsigned char* src = st + 3 * Cfg::kXBytes + i * 2 * E;  // row i / NK, entry i % NK
            Bf[i] = cld2<T>(src);
            if (!STATE_ONLY) Cf[i] = cld2<T>(src + Cfg::kBCBytes);
        }
        __syncthreads();
        // (2) the recurrence over the tile's rows
        for (int r = 0; r < kCTT; ++r) {
            const float2 dv = du[r * CPB + cc];
            float2 bv[kEPL], cv[kEPL];
            const float4* bq = reinterpret_cast<const float4*>(Bf + r * NK + g * kEPL);
            const float4 b0 = bq[0], b1 = bq[1];
            bv[0] = make_float2(b0.x, b0.y);
            bv[1] = make_float2(b0.z, b0.w);
            bv[2] = make_float2(b1.x, b1.y);
            bv[3] = make_float2(b1.z, b1.w);
            if (!STATE_ONLY) {
                const float4* cq = reinterpret_cast<const float4*>(Cf + r * NK + g * kEPL);
                const float4 c0 = cq[0], c1 = cq[1];
                cv[0] = make_float2(c0.x, -c0.y);
                cv[1] = make_float2(c0.z, -c0.w);
                cv[2] = make_float2(c1.x, -c1.y);
                cv[3] = make_float2(c1.z, -c1.w);
            }
            float2 y2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < kEPL; ++j) {
                const float2 e = cexp_da<PRECISE>(dv.x, Ac[j]);
                // h <- e h + u B in fp32 pairs: (e.re h.re - e.im h.im, e.re h.im + e.im h.re) + u B
                float2 hn = __ffma2_rn(make_float2(dv.y, dv.y), bv[j], __fmul2_rn(make_float2(e.x, e.x), h[j]));
                hn = __ffma2_rn(make_float2(-e.y, e.y), make_float2(h[j].y, h[j].x), hn);
                h[j] = hn;
                if (!STATE_ONLY) y2 = __ffma2_rn(cv[j], hn, y2);  // Re(C h) = C.re h.re - C.im h.im
            }
            if (!STATE_ONLY) ys[(r * CPB + cc) * LPC + g] = y2.x + y2.y;
        }
        if (!STATE_ONLY) {
            __syncthreads();
            // (3) partial sums, skip term, gate, store
            for (int i = tid; i < rows * CPB; i += kCThreads) {
                const int r = i / CPB, ch = i % CPB;
                if (ch >= chans) continue;
                float y = 0.0f;
#pragma unroll
                for (int q = 0; q < LPC; ++q) y += ys[(r * CPB + ch) * LPC + q];
                const float xv = to_f32<T>(*reinterpret_cast<const T*>(st + r * Cfg::kRowBytes + ch * E));
                if (a.D) y = fmaf(a.D[c_begin + ch], xv, y);
                if (GATE) y *= silu_t<PRECISE>(to_f32<T>(*reinterpret_cast<const T*>(st + 2 * Cfg::kXBytes + r * Cfg::kRowBytes + ch * E)));
                store_checked(a.out_s, reinterpret_cast<T*>(a.out + row_base + (int64_t)(k * kCTT + r) * row_stride + (c_begin + ch) * E),
                              from_f32<T>(y), a.status);
            }
        }
    }
    asm volatile("cp.async.wait_group 0;\n" ::);

    if (STATE_ONLY) {
        if (c_ok) {
            float* Hs = a.seg_h + (((int64_t)seg * gridDim.z + b) * a.dim + c) * a.N * 2;
#pragma unroll
            for (int j = 0; j < kEPL; ++j) {
                const int n = g * kEPL + j;
                if (n < a.N) {
                    store_checked(a.segh_s, &Hs[2 * n], h[j].x, a.status);
                    store_checked(a.segh_s, &Hs[2 * n + 1], h[j].y, a.status);
                }
            }
        }
        // Delta sums: thread i summed the items i, i + 128, ... of each tile, i.e. the
        // channel i % CPB; combine the threads of one channel
        __syncthreads();
        float* red = ys;
        red[tid] = dsum;
        __syncthreads();
        if (tid < chans) {
            float s = 0.0f;
            for (int q = tid; q < kCThreads; q += CPB) s += red[q];
            store_checked(a.segd_s, &a.seg_dsum[((int64_t)seg * gridDim.z + b) * a.dim + c_begin + tid], s, a.status);
        }
    } else if (a.final_state && seg == a.nseg - 1 && c_ok) {
        float* fs = a.final_state + (b * a.dim + c) * a.N * 2;
#pragma unroll
        for (int j = 0; j < kEPL; ++j) {
            const int n = g * kEPL + j;
            if (n < a.N) {
                store_checked(a.final_s, &fs[2 * n], h[j].x, a.status);
                store_checked(a.final_s, &fs[2 * n + 1], h[j].y, a.status);
            }
        }
    }
}

// ---- host side ---------------------------------------------------------------

struct CPlan {
    int NK, cpb, tiles_per_group, blocks_x, nseg;
    int64_t seg_len;
};

int cpick_nk(int64_t N) { return N <= 4 ? 4 : N <= 8 ? 8 : N <= 16 ? 16 : 32; }

// Segments: when the channels give fewer than two warps per SM sub-partition, cut the
// sequence so that both passes have about three (at least 128 steps per segment).
CPlan make_cplan(const ScanArgs& a) {
    CPlan p;
    p.NK = cpick_nk(a.dstate);
    p.cpb = kCThreads / (p.NK / kEPL);
    const int64_t cpg = a.nheads / a.ngroups;
    p.tiles_per_group = (int)((cpg + p.cpb - 1) / p.cpb);
    p.blocks_x = (int)(a.ngroups * p.tiles_per_group);
    const int64_t warps = (int64_t)p.blocks_x * a.batch * (kCThreads / 32);
    const int64_t smsp = (int64_t)sm_count() * 4;
    int64_t seg_len = a.seqlen;
    if (a.chunk > 0) {
        seg_len = a.chunk;
    } else if (warps > 0 && warps < 2 * smsp) {
        int64_t nseg = (3 * smsp + warps - 1) / warps;
        nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, a.seqlen / 128));
        seg_len = (a.seqlen + nseg - 1) / nseg;
    }
    seg_len = std::max<int64_t>(kCTT, (seg_len + kCTT - 1) / kCTT * kCTT);
    p.seg_len = seg_len;
    p.nseg = (int)std::max<int64_t>(1, (a.seqlen + seg_len - 1) / seg_len);
    return p;
}

template <typename T, int NK, bool STATE_ONLY, bool GATE>
cudaError_t claunch_one(const CDiagArgs& ka, dim3 grid, cudaStream_t stream) {
    using Cfg = CCfg<T, NK>;
    auto kern = cdiag_scan_kernel<T, NK, STATE_ONLY, GATE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    cudaEvent_t t0 = timing_begin(stream, STATE_ONLY ? "cdiag_scan_kernel (segment state pass)" : "cdiag_scan_kernel (output pass)");
    kern<<<grid, kCThreads, Cfg::kSmem, stream>>>(ka);
    note_launch(STATE_ONLY ? "cdiag_scan_kernel (segment state pass)" : "cdiag_scan_kernel (output pass)", stream, t0);
    return cudaGetLastError();
}

template <typename T, int NK>
cudaError_t claunch_typed(const ScanArgs& a, const CPlan& p, void* ws, cudaStream_t stream) {
    CDiagArgs ka;
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
    ka.status = nullptr;
    if (kBoundsCheck) {
        cudaError_t e = device_status_address(&ka.status);
        if (e != cudaSuccess) return e;
    }
    ka.out_s = span_of(a.out, (size_t)a.batch * a.seqlen * a.nheads * (a.dtype == 1 ? 2 : 4));
    ka.final_s = span_of(a.final_state, (size_t)a.batch * a.nheads * a.dstate * 2 * sizeof(float));
    if (p.nseg > 1) {
        const size_t hbytes = (size_t)(p.nseg - 1) * a.batch * a.nheads * a.dstate * 2 * sizeof(float);
        ka.seg_h = (float*)ws;
        ka.seg_dsum = (float*)((char*)ws + align_up(hbytes, 256));
        ka.segh_s = span_of(ka.seg_h, hbytes);
        ka.segd_s = span_of(ka.seg_dsum, (size_t)(p.nseg - 1) * a.batch * a.nheads * sizeof(float));
        cudaError_t e = claunch_one<T, NK, true, false>(ka, dim3(p.blocks_x, p.nseg - 1, (unsigned)a.batch), stream);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid(p.blocks_x, p.nseg, (unsigned)a.batch);
    return a.z ? claunch_one<T, NK, false, true>(ka, grid, stream) : claunch_one<T, NK, false, false>(ka, grid, stream);
}

template <typename T>
cudaError_t claunch_dtype(const ScanArgs& a, const CPlan& p, void* ws, cudaStream_t stream) {
    switch (p.NK) {
        case 4: return claunch_typed<T, 4>(a, p, ws, stream);
        case 8: return claunch_typed<T, 8>(a, p, ws, stream);
        case 16: return claunch_typed<T, 16>(a, p, ws, stream);
        default: return claunch_typed<T, 32>(a, p, ws, stream);
    }
}

}  // namespace

size_t cdiag_workspace_bytes(const ScanArgs& a) {
    if (a.batch == 0 || a.seqlen == 0) return 0;
    const CPlan p = make_cplan(a);
    if (p.nseg <= 1) return 0;
    const size_t hbytes = (size_t)(p.nseg - 1) * a.batch * a.nheads * a.dstate * 2 * sizeof(float);
    const size_t dbytes = (size_t)(p.nseg - 1) * a.batch * a.nheads * sizeof(float);
    return align_up(hbytes, 256) + align_up(dbytes, 256);
}

cudaError_t cdiag_launch(const ScanArgs& a, void* ws, cudaStream_t stream) {
    if (a.batch == 0) return cudaSuccess;
    const CPlan p = make_cplan(a);
    if (a.dtype == 1) return claunch_dtype<__nv_bfloat16>(a, p, ws, stream);
    return claunch_dtype<float>(a, p, ws, stream);
}

}  // namespace ssm
