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
//  * The expanded state (b, T, d_inner, N) never leaves registers: LPC lanes own one
//    channel, each lane NPT = NK/LPC state entries held as fp32 pairs (NPT 4 or 8,
//    chosen by the host plan from the channel count).
//  * Inputs are token-major (channels innermost).  A block owns 16 (or 32) channels of
//    one group and walks time in tiles of 16 steps; each tile of x, dt, z, B, C is
//    staged into shared memory by 16-byte cp.async copies in a 4-deep ring, so HBM
//    reads are coalesced rows that overlap the arithmetic of earlier tiles.
//  * One software-pipelined loop body per tile k: the recurrence of tile k's rows
//    (decays of 4 rows formed before their dependent updates: ex2.approx of the decay
//    argument, packed fp32x2 multiply/FMA for the argument, the input term, the update
//    and the C.h partial sum), interleaved with the per-(t, c) prep of tile k+1
//    (softplus(dt + dt_bias) and Delta*x per channel pair, B and C to fp32) and the
//    epilogue of tile k-1 (the LPC partial sums, D*x, the SiLU gate, the store).  Every
//    per-(t, c) operation runs once, by one thread of a channel pair.
//  * B300's SFU runs ex2 at 32/clk/SM (lg2, rcp at 16) and packed fp32x2 FMA gives no
//    extra lane throughput over scalar FMA (128 lane-ops/clk/SM), so the scan is bound
//    by the SFU and FMA pipes (one exp and four FP32 operations per state entry and
//    step), above the HBM time of its 8 bytes per token-channel.
//  * Time parallelism when there are few channels: the sequence is cut into segments.
//    A state-only pass computes each segment's local end state (from zero) and its
//    sum of Delta; the output pass folds those summaries into the segment's initial
//    state, h <- exp(A sum Delta_j) h + H_j, which is the affine combine
//    (a1, b1) o (a2, b2) = (a1 a2, a2 b1 + b2) of the parallel-scan formulation
//    ("引言：Attention的天花板" article, 硬件感知算法).  The output pass is launched as a
//    programmatic dependent of the state-only pass, so its blocks stage their first tiles
//    while that pass finishes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kTT = 16;      // time steps per tile
constexpr int kStages = 4;   // cp.async ring: tiles k-1 (epilogue), k+1 (prep), k+2, k+3 (loads)
constexpr int kRB = 4;       // rows whose decays are formed together
constexpr int kConvHalo = 3; // inputs before a tile that the width-4 convolution reads

// LPC lanes per channel, WARPS warps per block; CONV adds the convolved-input ring and
// the halo of inputs before the segment.
template <typename T, int NK, int LPC, int WARPS, bool CONV = false>
struct DiagCfg {
    static constexpr int NT = 32 * WARPS;       // threads per block
    static constexpr int CPB = NT / LPC;        // channels per block
    static constexpr int NPT = NK / LPC;        // state entries per thread
    static constexpr int P2 = CPB / 2;          // channel pairs per block
    static constexpr int kElem = (int)sizeof(T);
    static constexpr int kRowBytes = CPB * kElem;  // one time row of the x/dt/z tile
    static constexpr int kRowChunks = kRowBytes / 16;
    static constexpr int kXBytes = kTT * kRowBytes;
    static constexpr int kBCRowBytes = NK * kElem;
    static constexpr int kBCRowChunks = kBCRowBytes / 16;
    static constexpr int kBCBytes = kTT * kBCRowBytes;
    static constexpr int kStageBytes = 3 * kXBytes + 2 * kBCBytes;
    static constexpr int kBfFloats = kTT * NK;         // fp32 B (and C) of one tile
    static constexpr int kDuFloat2 = kTT * CPB;        // (Delta, Delta*x) of one tile
    static constexpr int kYsFloats = kTT * CPB * LPC;  // partial C.h of one tile
    static constexpr int kXsFloats = kTT * CPB;        // convolved x of one tile
    static constexpr int kHaloFloats = kConvHalo * CPB;  // inputs before the segment
    // two buffers (tile parity) of each derived array; three for the convolved x, which
    // is written two tiles ahead of the epilogue that reads it
    static constexpr int kSmemBytes = kStages * kStageBytes + 2 * (2 * kBfFloats * 4 + kDuFloat2 * 8 + kYsFloats * 4) +
                                      (CONV ? (3 * kXsFloats + kHaloFloats) * 4 : 0);
    static constexpr int RS = NT / P2;                 // rows per sweep of the pair roles
    static constexpr int kPairItems = kTT / RS;        // pair items per thread per tile
    static constexpr int kBCItems = kTT * NK / 2 / NT; // B/C pair conversions per thread per tile
    static constexpr int kBatches = kTT / kRB;
    static_assert(NPT % 4 == 0, "state entries are processed in groups of 4");
    static_assert(kRowBytes % 16 == 0 && kBCRowBytes % 16 == 0, "16-byte rows");
    static_assert(NT % P2 == 0 && kTT % RS == 0, "pair mapping");
    static_assert(kTT * NK / 2 % NT == 0, "B/C conversion mapping");
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
    const float* conv_w; // (dim, conv_k) depthwise convolution ahead of the scan, or null
    const float* conv_b; // (dim,) or null
    const char* x_prev;  // (b, conv_k-1, dim) inputs before t = 0, or null (zeros)
    char* x_last;        // (b, conv_k-1, dim) receives the last conv_k-1 inputs, or null
    int conv_k;          // convolution width 1..4 (CONV kernels only)
    char* out;
    float* final_state;  // (b, dim, N) or null
    float* seg_h;        // (nseg-1, b, dim, N): local end state of each segment but the last
    float* seg_dsum;     // (nseg-1, b, dim): sum of Delta over the segment
    int64_t T, dim, N, G, cpg;
    int64_t seg_len;
    int nseg, tiles_per_group;
    int nsub_launched;   // host side: a state-only pass was launched ahead of this pass
    // byte ranges of the buffers written (stores checked in SSM_BOUNDS_CHECK builds)
    int* status;
    Span out_s, final_s, segh_s, segd_s, xlast_s;
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
__device__ __forceinline__ float2 load_pair(const unsigned char* p);
template <>
__device__ __forceinline__ float2 load_pair<float>(const unsigned char* p) {
    return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 load_pair<__nv_bfloat16>(const unsigned char* p) {
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

// softplus / SiLU of a channel pair: accurate library functions for fp32 inputs; for
// 16-bit inputs one SFU exponential each, the rest on the FMA pipe.
template <bool PRECISE>
__device__ __forceinline__ float2 softplus_pair(float2 v) {
    if (PRECISE) return make_float2(softplus_precise(v.x), softplus_precise(v.y));
    return softplus2_fma(v);
}
template <bool PRECISE>
__device__ __forceinline__ float2 silu_pair(float2 z) {
    if (PRECISE) return make_float2(silu_precise(z.x), silu_precise(z.y));
    return silu2_fma(z);
}

// 2^x for x <= 0 on the FMA pipe, two values at a time (the alternative to the SFU's
// ex2 that the SSM_TUNE_DIAG_EXP_POLY plan override selects): x is clamped at -126 (below
// it the decay is zero to fp32 precision), n = rint(x) by adding 1.5 * 2^23 (the integer
// lands in the low mantissa bits), f = x - n in [-1/2, 1/2], 2^f by a degree-5
// polynomial and 2^n written directly as the exponent field.  The coefficients are the
// relative-error minimax fit of fit_exp2.py (Lawson's iteration on Chebyshev nodes); the
// fp32 evaluation stays within 2.5e-7 of 2^f.
__device__ __forceinline__ float2 exp2_fma2(float2 x) {
    constexpr float kC0 = 1.000000119e+00f, kC1 = 6.931469440e-01f, kC2 = 2.402212024e-01f;
    constexpr float kC3 = 5.550713092e-02f, kC4 = 9.675540961e-03f, kC5 = 1.327647129e-03f;
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    x = make_float2(fmaxf(x.x, -126.0f), fmaxf(x.y, -126.0f));
    const float2 t = __fadd2_rn(x, make_float2(kRound, kRound));
    const float2 r = __fadd2_rn(t, make_float2(-kRound, -kRound));  // rint(x), exact
    const float2 f = __ffma2_rn(r, make_float2(-1.0f, -1.0f), x);   // x - rint(x), exact
    float2 p = __ffma2_rn(make_float2(kC5, kC5), f, make_float2(kC4, kC4));
    p = __ffma2_rn(p, f, make_float2(kC3, kC3));
    p = __ffma2_rn(p, f, make_float2(kC2, kC2));
    p = __ffma2_rn(p, f, make_float2(kC1, kC1));
    p = __ffma2_rn(p, f, make_float2(kC0, kC0));
    // the bits of t are those of 1.5 * 2^23 plus n: shifted left by 23 only n survives,
    // and adding 127 << 23 gives the exponent field of 2^n (n >= -126: a normal number)
    const float2 s2 = make_float2(__int_as_float(__float_as_int(t.x) * 8388608 + 0x3F800000),
                                  __int_as_float(__float_as_int(t.y) * 8388608 + 0x3F800000));
    return __fmul2_rn(p, s2);
}

// STATE_ONLY: compute each segment's local end state from zero (segments 0..nseg-2).
// Otherwise: full output pass over every segment with the folded initial state.
//
// Software pipeline over tiles of 16 steps.  Iteration k of the tile loop, in one
// fused loop body over groups of 4 rows:
//   scan(k):      the recurrence of tile k's rows (state entries of one channel per lane,
//                 decays of 4 rows formed before the dependent updates), partial C.h
//                 sums to shared memory;
//   prep(k+1):    softplus(dt + dt_bias) and Delta*x of tile k+1 per channel pair, B and C
//                 of tile k+1 to fp32;
//   finish(k-1):  the LPC partial sums of tile k-1 per channel pair, D*x, SiLU gate, store.
// Interleaving the per-(t, c) work (SFU-latency chains) with the scan keeps the SFU and
// FMA pipes busy at the low occupancy these channel counts give.
//
// CONV: x is first replaced by x' = SiLU(conv_b + sum_k conv_w[k] x_{t-K+1+k}) (causal
// depthwise convolution, "论文解读：Mamba — 线性时间的序列建模革命", 五 Mamba块架构),
// formed in prep from the staged rows of this tile and the three rows before it (the
// previous tile's stage, or a halo loaded once per segment); the epilogue reads x' for
// the skip term from a ring of three tile buffers.
//
// PX: of each group of 4 state entries per step, the decays of PX pairs come from
// exp2_fma2 (FMA pipe) and the rest from the SFU's ex2 (0: all SFU, the default).
template <typename T, int NK, int LPC, int WARPS, bool STATE_ONLY, bool GATE, bool CONV, int PX = 0>
__global__ void __launch_bounds__(32 * WARPS) diag_scan_kernel(const DiagKernelArgs a) {
    using Cfg = DiagCfg<T, NK, LPC, WARPS, CONV>;
    constexpr int NT = Cfg::NT, CPB = Cfg::CPB, NPT = Cfg::NPT, P2 = Cfg::P2, E = Cfg::kElem;
    constexpr int RS = Cfg::RS;
    constexpr bool PRECISE = sizeof(T) == 4;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* stage0 = smem;
    float* Bf0 = reinterpret_cast<float*>(smem + kStages * Cfg::kStageBytes);  // [2][kBfFloats]
    float* Cf0 = Bf0 + 2 * Cfg::kBfFloats;                                   // [2][kBfFloats]
    float2* du0 = reinterpret_cast<float2*>(Cf0 + 2 * Cfg::kBfFloats);        // [2][kDuFloat2]
    float* ys0 = reinterpret_cast<float*>(du0 + 2 * Cfg::kDuFloat2);          // [2][kYsFloats]
    float* xs0 = ys0 + 2 * Cfg::kYsFloats;                                    // [3][kXsFloats] (CONV)
    float* halo = xs0 + 3 * Cfg::kXsFloats;                                   // [3][CPB] (CONV)

    const int tid = threadIdx.x;
    const int group = blockIdx.x / a.tiles_per_group;
    const int64_t c_begin = (int64_t)group * a.cpg + (int64_t)(blockIdx.x % a.tiles_per_group) * CPB;
    const int64_t c_end = (int64_t)(group + 1) * a.cpg;  // exclusive, within this group
    const int seg = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int64_t t_begin = (int64_t)seg * a.seg_len;
    const int64_t t_end = min(a.T, t_begin + a.seg_len);
    const int ntiles = (int)((t_end - t_begin + kTT - 1) / kTT);

    // scan role: channel cc, lane g of LPC
    const int cc = tid / LPC;
    const int g = tid % LPC;
    const int64_t c = c_begin + cc;
    const bool c_ok = c < c_end;

    // pair role (prep and finish): channels 2*pp, 2*pp+1; rows r0, r0 + RS, ...
    const int pp = tid % P2;
    const int r0 = tid / P2;
    const int64_t cA = c_begin + 2 * pp;
    const bool pair_ok = cA < c_end;  // group runs are whole 16-byte chunks: even
    const float2 bias2 = (pair_ok && a.dt_bias) ? make_float2(a.dt_bias[cA], a.dt_bias[cA + 1])
                                                : make_float2(0.0f, 0.0f);
    const float2 d2 = (pair_ok && a.D) ? make_float2(a.D[cA], a.D[cA + 1]) : make_float2(0.0f, 0.0f);
    float2 dsum2 = make_float2(0.0f, 0.0f);  // sum of Delta (state-only pass)
    // convolution taps of the pair, left-padded to width 4 (tap 3 weights the current row)
    float2 cw[4];
    float2 cb2 = make_float2(0.0f, 0.0f);
    if (CONV) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int kk = k - (4 - a.conv_k);
            cw[k] = (pair_ok && kk >= 0) ? make_float2(a.conv_w[cA * a.conv_k + kk], a.conv_w[(cA + 1) * a.conv_k + kk])
                                         : make_float2(0.0f, 0.0f);
        }
        if (pair_ok && a.conv_b) cb2 = make_float2(a.conv_b[cA], a.conv_b[cA + 1]);
    }

    // state entries and decay rates (times log2 e) in fp32 pairs, as the packed
    // fp32x2 instructions take them
    float2 A2[NPT / 2];
    float2 h[NPT / 2];
#pragma unroll
    for (int k = 0; k < NPT / 2; ++k) {
        const int n = g * NPT + 2 * k;
        A2[k].x = (c_ok && n < a.N) ? a.A[c * a.N + n] * kLog2e : 0.0f;
        A2[k].y = (c_ok && n + 1 < a.N) ? a.A[c * a.N + n + 1] * kLog2e : 0.0f;
        h[k] = make_float2(0.0f, 0.0f);
    }
    // state entering this segment: the initial state decayed through the earlier segments
    // plus their local end states (the state-only pass's results)
    auto fold_initial_state = [&]() {
        if (c_ok && a.init) {
            const float* hi = a.init + (b * a.dim + c) * a.N;
#pragma unroll
            for (int k = 0; k < NPT / 2; ++k) {
                const int n = g * NPT + 2 * k;
                if (n < a.N) h[k].x = hi[n];
                if (n + 1 < a.N) h[k].y = hi[n + 1];
            }
        }
        for (int s = 0; s < seg && c_ok; ++s) {
            const float dsum = a.seg_dsum[((int64_t)s * gridDim.z + b) * a.dim + c];
            const float* Hs = a.seg_h + (((int64_t)s * gridDim.z + b) * a.dim + c) * a.N;
#pragma unroll
            for (int k = 0; k < NPT / 2; ++k) {
                const int n = g * NPT + 2 * k;
                if (n < a.N) h[k].x = ex2(A2[k].x * dsum) * h[k].x + Hs[n];
                if (n + 1 < a.N) h[k].y = ex2(A2[k].y * dsum) * h[k].y + Hs[n + 1];
            }
        }
    };

    const int64_t row_stride = a.dim * E;     // bytes between consecutive time rows
    const int64_t bc_stride = a.G * a.N * E;  // bytes between consecutive B/C rows
    const char* bc_off_B = a.B + (int64_t)group * a.N * E;
    const char* bc_off_C = a.C + (int64_t)group * a.N * E;

    // 32-bit tile arithmetic and 64-bit bases computed once (a segment holds < 2^31
    // steps): byte offsets of the segment's first x and B/C rows, this pair's output column
    const int seg_rows = (int)(t_end - t_begin);
    const int chans = (int)(c_end - c_begin);  // channels of the group from c_begin
    const int64_t row_base = (b * a.T + t_begin) * row_stride;
    const int64_t bc_base = (b * a.T + t_begin) * bc_stride;
    char* const out_base = a.out + row_base + cA * E;
    auto tile_rows = [&](int k) { return min(kTT, seg_rows - k * kTT); };
    auto stage = [&](int k) { return stage0 + (k % kStages) * Cfg::kStageBytes; };

    auto issue_tile = [&](int k) {
        if (k < ntiles) {
            unsigned char* st = stage(k);
            const int rows = tile_rows(k);
            for (int i = tid; i < kTT * Cfg::kRowChunks; i += NT) {
                const int r = i / Cfg::kRowChunks, q = i % Cfg::kRowChunks;
                const bool ok = r < rows && q * (16 / E) < chans;
                const int64_t off = ok ? (row_base + (int64_t)(k * kTT + r) * row_stride + (c_begin * E + q * 16)) : 0;
                cp_async16(st + r * Cfg::kRowBytes + q * 16, a.x + off, ok);
                cp_async16(st + Cfg::kXBytes + r * Cfg::kRowBytes + q * 16, a.dt + off, ok);
                if (GATE && !STATE_ONLY)
                    cp_async16(st + 2 * Cfg::kXBytes + r * Cfg::kRowBytes + q * 16, a.z + off, ok);
            }
            for (int i = tid; i < kTT * Cfg::kBCRowChunks; i += NT) {
                const int r = i / Cfg::kBCRowChunks, q = i % Cfg::kBCRowChunks;
                const bool ok = r < rows && q * (16 / E) < a.N;
                const int64_t off = ok ? (bc_base + (int64_t)(k * kTT + r) * bc_stride + q * 16) : 0;
                unsigned char* dB = st + 3 * Cfg::kXBytes + r * Cfg::kBCRowBytes + q * 16;
                cp_async16(dB, bc_off_B + off, ok);
                if (!STATE_ONLY) cp_async16(dB + Cfg::kBCBytes, bc_off_C + off, ok);
            }
        }
        cp_async_commit();
    };

    // input pair of row rr of tile k, rr in [-3, kTT): rows before the tile come from the
    // previous tile's stage or, for the segment's first tile, from the halo
    auto x_row = [&](int k, int rr) -> float2 {
        if (rr >= 0) return load_pair<T>(stage(k) + rr * Cfg::kRowBytes + 2 * pp * E);
        if (k > 0) return load_pair<T>(stage(k - 1) + (kTT + rr) * Cfg::kRowBytes + 2 * pp * E);
        return *reinterpret_cast<const float2*>(&halo[(kConvHalo + rr) * CPB + 2 * pp]);
    };

    // prep item it (0..kPairItems-1) of tile k: one (row, channel pair)
    auto prep_item = [&](int k, int it) {
        const unsigned char* st = stage(k);
        float2* du = du0 + (k & 1) * Cfg::kDuFloat2;
        const int r = r0 + it * RS;
        const float2 dtv = load_pair<T>(st + Cfg::kXBytes + r * Cfg::kRowBytes + 2 * pp * E);
        float2 xv = load_pair<T>(st + r * Cfg::kRowBytes + 2 * pp * E);
        if (CONV) {
            float2 acc = __ffma2_rn(cw[3], xv, cb2);
#pragma unroll
            for (int j = 1; j <= kConvHalo; ++j) acc = __ffma2_rn(cw[3 - j], x_row(k, r - j), acc);
            xv = silu_pair<PRECISE>(acc);
            if (!STATE_ONLY) *reinterpret_cast<float2*>(&xs0[(k % 3) * Cfg::kXsFloats + r * CPB + 2 * pp]) = xv;
        }
        float2 de = softplus_pair<PRECISE>(__fadd2_rn(dtv, bias2));
        if (r >= tile_rows(k)) de = make_float2(0.0f, 0.0f);  // no-op rows: Delta = 0 keeps h
        const float2 u = __fmul2_rn(de, xv);
        *reinterpret_cast<float4*>(&du[r * CPB + 2 * pp]) = make_float4(de.x, u.x, de.y, u.y);
        if (STATE_ONLY) dsum2 = __fadd2_rn(dsum2, de);
    };
    // B/C conversion item it of tile k
    auto conv_item = [&](int k, int it) {
        const unsigned char* st = stage(k);
        const int i = tid + it * NT;
        float* Bf = Bf0 + (k & 1) * Cfg::kBfFloats;
        *reinterpret_cast<float2*>(&Bf[2 * i]) = load_pair<T>(st + 3 * Cfg::kXBytes + i * 2 * E);
        if (!STATE_ONLY) {
            float* Cf = Cf0 + (k & 1) * Cfg::kBfFloats;
            *reinterpret_cast<float2*>(&Cf[2 * i]) = load_pair<T>(st + 3 * Cfg::kXBytes + Cfg::kBCBytes + i * 2 * E);
        }
    };
    // finish item it of tile k: combine partial sums, skip term, gate, store
    auto finish_item = [&](int k, int it) {
        const int r = r0 + it * RS;
        if (r >= tile_rows(k) || !pair_ok) return;
        const unsigned char* st = stage(k);
        const float* ys = ys0 + (k & 1) * Cfg::kYsFloats;
        float2 y = make_float2(0.0f, 0.0f);
        if (LPC == 1) {
            y = *reinterpret_cast<const float2*>(&ys[r * CPB + 2 * pp]);
        } else {
#pragma unroll
            for (int q = 0; q < LPC; q += 2) {
                const float2 p0 = *reinterpret_cast<const float2*>(&ys[(r * CPB + 2 * pp) * LPC + q]);
                const float2 p1 = *reinterpret_cast<const float2*>(&ys[(r * CPB + 2 * pp + 1) * LPC + q]);
                y = __fadd2_rn(y, make_float2(p0.x + p0.y, p1.x + p1.y));
            }
        }
        const float2 xv = CONV ? *reinterpret_cast<const float2*>(&xs0[(k % 3) * Cfg::kXsFloats + r * CPB + 2 * pp])
                               : load_pair<T>(st + r * Cfg::kRowBytes + 2 * pp * E);
        y = __ffma2_rn(d2, xv, y);
        if (GATE) y = __fmul2_rn(y, silu_pair<PRECISE>(load_pair<T>(st + 2 * Cfg::kXBytes + r * Cfg::kRowBytes + 2 * pp * E)));
        char* dst = out_base + (int64_t)(k * kTT + r) * row_stride;
        if (span_ok(a.out_s, dst, 2 * E, a.status)) store_pair<T>(dst, y);
    };

    // The output pass may start while the state-only pass is finishing (programmatic
    // dependent launch): inputs only until griddepcontrol.wait, which returns once that
    // grid has completed and its writes are visible; before it, nothing is written.
    if (STATE_ONLY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // prologue: tiles 0..2 in flight, tile 0 prepared
    issue_tile(0);
    issue_tile(1);
    issue_tile(2);
    if (!STATE_ONLY) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        fold_initial_state();
    }
    if (CONV) {
        // the three inputs before the segment: earlier rows of x, else the previous
        // call's last inputs, else zero
        const T* xg = reinterpret_cast<const T*>(a.x);
        const T* xp = reinterpret_cast<const T*>(a.x_prev);
        for (int i = tid; i < kConvHalo * CPB; i += NT) {
            const int j = i / CPB, cch = i % CPB;
            const int64_t ch = c_begin + cch;
            const int64_t s = t_begin - kConvHalo + j;
            float v = 0.0f;
            if (ch < c_end) {
                if (s >= 0)
                    v = to_f32<T>(xg[(b * a.T + s) * a.dim + ch]);
                else if (xp && a.conv_k - 1 + s >= 0)
                    v = to_f32<T>(xp[(b * (a.conv_k - 1) + (a.conv_k - 1 + s)) * a.dim + ch]);
            }
            halo[j * CPB + cch] = v;
        }
    }
    if (ntiles > 0) {
        cp_async_wait<2>();
        __syncthreads();
#pragma unroll
        for (int it = 0; it < Cfg::kPairItems; ++it) prep_item(0, it);
#pragma unroll
        for (int it = 0; it < Cfg::kBCItems; ++it) conv_item(0, it);
    }

    for (int k = 0; k < ntiles; ++k) {
        cp_async_wait<1>();  // tile k+1 landed (tile k+2 may still be in flight)
        __syncthreads();     // ... and visible; tile k's derived data visible
        const bool next = k + 1 < ntiles;
        const bool prev = !STATE_ONLY && k > 0;
        const float2* du = du0 + (k & 1) * Cfg::kDuFloat2;
        const float* Bf = Bf0 + (k & 1) * Cfg::kBfFloats;
        const float* Cf = Cf0 + (k & 1) * Cfg::kBfFloats;
        float* ys = ys0 + (k & 1) * Cfg::kYsFloats;
        const int rows = tile_rows(k);
#pragma unroll
        for (int bt = 0; bt < Cfg::kBatches; ++bt) {
            const int rb = bt * kRB;
            // per-(t, c) work of the neighbouring tiles, interleaved with this batch
            if (next) {
                for (int it = bt; it < Cfg::kPairItems; it += Cfg::kBatches) prep_item(k + 1, it);
                for (int it = bt; it < Cfg::kBCItems; it += Cfg::kBatches) conv_item(k + 1, it);
            }
            if (prev)
                for (int it = bt; it < Cfg::kPairItems; it += Cfg::kBatches) finish_item(k - 1, it);
            if (rb >= rows) continue;
            // decays and input terms of kRB rows first, then the dependent updates;
            // rows past the tile's end have Delta = 0 and x*Delta = 0 and leave h as is
            float2 av[kRB][NPT / 2], ub[kRB][NPT / 2];
#pragma unroll
            for (int i = 0; i < kRB; ++i) {
                const float2 dv = du[(rb + i) * CPB + cc];
                const float2 dd = make_float2(dv.x, dv.x);
                const float2 uu = make_float2(dv.y, dv.y);
#pragma unroll
                for (int kk = 0; kk < NPT / 2; kk += 2) {
                    const float4 bq = *reinterpret_cast<const float4*>(&Bf[(rb + i) * NK + g * NPT + 2 * kk]);
                    const float2 dA0 = __fmul2_rn(dd, A2[kk]);
                    const float2 dA1 = __fmul2_rn(dd, A2[kk + 1]);
                    av[i][kk] = PX >= 2 ? exp2_fma2(dA0) : make_float2(ex2(dA0.x), ex2(dA0.y));
                    av[i][kk + 1] = PX >= 1 ? exp2_fma2(dA1) : make_float2(ex2(dA1.x), ex2(dA1.y));
                    ub[i][kk] = __fmul2_rn(uu, make_float2(bq.x, bq.y));
                    ub[i][kk + 1] = __fmul2_rn(uu, make_float2(bq.z, bq.w));
                }
            }
#pragma unroll
            for (int i = 0; i < kRB; ++i) {
                float2 ya = make_float2(0.0f, 0.0f), yb = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int kk = 0; kk < NPT / 2; kk += 2) {
                    h[kk] = __ffma2_rn(av[i][kk], h[kk], ub[i][kk]);
                    h[kk + 1] = __ffma2_rn(av[i][kk + 1], h[kk + 1], ub[i][kk + 1]);
                    if (!STATE_ONLY) {
                        const float4 cq = *reinterpret_cast<const float4*>(&Cf[(rb + i) * NK + g * NPT + 2 * kk]);
                        ya = __ffma2_rn(make_float2(cq.x, cq.y), h[kk], ya);
                        yb = __ffma2_rn(make_float2(cq.z, cq.w), h[kk + 1], yb);
                    }
                }
                if (!STATE_ONLY) {
                    const float2 ys2 = __fadd2_rn(ya, yb);
                    ys[((rb + i) * CPB + cc) * LPC + g] = ys2.x + ys2.y;
                }
            }
        }
        __syncthreads();      // every thread is done with stage k-1 before it is reloaded
        issue_tile(k + 3);    // into the stage of tile k-1
    }
    if (!STATE_ONLY && ntiles > 0) {
        __syncthreads();
#pragma unroll
        for (int it = 0; it < Cfg::kPairItems; ++it) finish_item(ntiles - 1, it);
    }
    cp_async_wait<0>();

    if (STATE_ONLY) {
        // local end state and Delta sum of this segment
        if (c_ok) {
            float* Hs = a.seg_h + (((int64_t)seg * gridDim.z + b) * a.dim + c) * a.N;
#pragma unroll
            for (int k = 0; k < NPT / 2; ++k) {
                const int n = g * NPT + 2 * k;
                if (n < a.N) store_checked(a.segh_s, &Hs[n], h[k].x, a.status);
                if (n + 1 < a.N) store_checked(a.segh_s, &Hs[n + 1], h[k].y, a.status);
            }
        }
        // the RS threads of a pair each summed a subset of rows
        __syncthreads();
        float2* red = du0;  // reuse: RS x P2 partial sums
        red[r0 * P2 + pp] = dsum2;
        __syncthreads();
        if (tid < P2) {
            float2 s = make_float2(0.0f, 0.0f);
            for (int k = 0; k < RS; ++k) s = __fadd2_rn(s, red[k * P2 + tid]);
            const int64_t c0 = c_begin + 2 * tid;
            if (c0 < c_end) {
                float* dst = a.seg_dsum + ((int64_t)seg * gridDim.z + b) * a.dim + c0;
                store_checked(a.segd_s, dst, s.x, a.status);
                store_checked(a.segd_s, dst + 1, s.y, a.status);
            }
        }
    }
    if (CONV && !STATE_ONLY && a.x_last && seg == a.nseg - 1) {
        // the last conv_k-1 inputs (raw) for a following call
        const T* xg = reinterpret_cast<const T*>(a.x);
        const T* xp = reinterpret_cast<const T*>(a.x_prev);
        T* xl = reinterpret_cast<T*>(a.x_last);
        const int km1 = a.conv_k - 1;
        for (int i = tid; i < km1 * CPB; i += NT) {
            const int j = i / CPB, cch = i % CPB;
            const int64_t ch = c_begin + cch;
            if (ch >= c_end) continue;
            const int64_t s = a.T - km1 + j;
            T v = from_f32<T>(0.0f);
            if (s >= 0)
                v = xg[(b * a.T + s) * a.dim + ch];
            else if (xp)
                v = xp[(b * km1 + (km1 + s)) * a.dim + ch];
            store_checked(a.xlast_s, &xl[(b * km1 + j) * a.dim + ch], v, a.status);
        }
    }
    if (!STATE_ONLY && a.final_state && seg == a.nseg - 1 && c_ok) {
        float* fs = a.final_state + (b * a.dim + c) * a.N;
#pragma unroll
        for (int k = 0; k < NPT / 2; ++k) {
            const int n = g * NPT + 2 * k;
            if (n < a.N) store_checked(a.final_s, &fs[n], h[k].x, a.status);
            if (n + 1 < a.N) store_checked(a.final_s, &fs[n + 1], h[k].y, a.status);
        }
    }
}

// ---- host side ---------------------------------------------------------------

struct Plan {
    int NK;
    int LPC;
    int px;  // SSM_TUNE_DIAG_EXP_POLY (bf16, dstate <= 16, no convolution): 0, 1 or 2
    int warps;
    int cpb;
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

// State entries per lane: the SSM_TUNE_DIAG_NPT override (4 or 8) when set, else 8 when
// the channels alone fill the GPU and 4 when the sequence has to be split.
int npt_override() {
    const int64_t v = tuning(0);
    return v == 4 || v == 8 ? (int)v : 0;
}

Plan make_plan(const ScanArgs& a) {
    Plan p;
    p.NK = pick_nk(a.dstate);
    const int64_t px = tuning(4);
    p.px = px == 1 || px == 2 ? (int)px : 0;
    const int64_t smsp = (int64_t)sm_count() * 4;  // SM sub-partitions
    auto fill = [&](int npt) {
        p.LPC = std::max(1, std::min(8, p.NK / npt));
        p.cpb = p.LPC == 1 ? 32 : 16;
        p.warps = p.cpb * p.LPC / 32;
        const int64_t cpg = a.nheads / a.ngroups;
        p.tiles_per_group = (int)((cpg + p.cpb - 1) / p.cpb);
        p.blocks_x = (int)(a.ngroups * p.tiles_per_group);
        return (int64_t)p.blocks_x * a.batch * p.warps;
    };
    // Measured on B300: 8 state entries per lane is fastest when the channels give at
    // least 2 warps per sub-partition; below that, 4 per lane plus time segments of
    // about 3 warps per sub-partition (segment folding costs a state-only pass).
    int64_t warps = fill(npt_override() ? npt_override() : 8);
    const bool split = a.chunk == 0 && warps > 0 && warps < 2 * smsp;
    if (split && !npt_override()) warps = fill(4);
    int64_t seg_len;
    if (a.chunk > 0) {
        seg_len = a.chunk;
    } else if (!split) {
        seg_len = a.seqlen;
    } else {
        int64_t nseg = (3 * smsp + warps - 1) / warps;
        nseg = std::max<int64_t>(1, std::min<int64_t>(nseg, a.seqlen / 128));
        seg_len = (a.seqlen + nseg - 1) / nseg;
    }
    seg_len = std::max<int64_t>(kTT, (seg_len + kTT - 1) / kTT * kTT);
    p.seg_len = seg_len;
    p.nseg = (int)std::max<int64_t>(1, (a.seqlen + seg_len - 1) / seg_len);
    return p;
}

template <typename T, int NK, int LPC, bool STATE_ONLY, bool GATE, bool CONV, int PX>
cudaError_t launch_one(const DiagKernelArgs& ka, dim3 grid, cudaStream_t stream) {
    constexpr int WARPS = (LPC == 1 ? 32 : 16) * LPC / 32;
    using Cfg = DiagCfg<T, NK, LPC, WARPS, CONV>;
    auto kern = diag_scan_kernel<T, NK, LPC, WARPS, STATE_ONLY, GATE, CONV, PX>;
    // the shared-memory attribute is set once per instantiation and device
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_relaxed) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(bit, std::memory_order_relaxed);
    }
    cudaEvent_t t0 = timing_begin(stream, STATE_ONLY ? "diag_scan_kernel (segment state pass)" : "diag_scan_kernel (output pass)");
    if (!STATE_ONLY && ka.nsub_launched) {
        // after a state-only pass: programmatic dependent launch (see the kernel)
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(Cfg::NT);
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;
        cfg.stream = stream;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, ka);
        if (e != cudaSuccess) {
            launch_failed(t0);
            return e;
        }
    } else {
        kern<<<grid, Cfg::NT, Cfg::kSmemBytes, stream>>>(ka);
    }
    note_launch(STATE_ONLY ? "diag_scan_kernel (segment state pass)" : "diag_scan_kernel (output pass)", stream, t0);
    return cudaGetLastError();
}

template <typename T, int NK, int LPC, bool CONV, int PX = 0>
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
    ka.conv_w = a.conv_w;
    ka.conv_b = a.conv_b;
    ka.x_prev = (const char*)a.x_prev;
    ka.x_last = (char*)a.x_last;
    ka.conv_k = a.conv_k;
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
    ka.nsub_launched = 0;
    ka.status = nullptr;
    if (kBoundsCheck) {
        cudaError_t e = device_status_address(&ka.status);
        if (e != cudaSuccess) return e;
    }
    const size_t E = a.dtype == 1 ? 2 : 4;
    ka.out_s = span_of(a.out, (size_t)a.batch * a.seqlen * a.nheads * E);
    ka.final_s = span_of(a.final_state, (size_t)a.batch * a.nheads * a.dstate * sizeof(float));
    ka.xlast_s = span_of(a.x_last, (size_t)a.batch * (a.conv_k > 1 ? a.conv_k - 1 : 0) * a.nheads * E);
    if (p.nseg > 1) {
        const size_t hbytes = (size_t)(p.nseg - 1) * a.batch * a.nheads * a.dstate * sizeof(float);
        const size_t dbytes = (size_t)(p.nseg - 1) * a.batch * a.nheads * sizeof(float);
        ka.seg_h = (float*)ws;
        ka.seg_dsum = (float*)((char*)ws + align_up(hbytes, 256));
        ka.segh_s = span_of(ka.seg_h, hbytes);
        ka.segd_s = span_of(ka.seg_dsum, dbytes);
        const dim3 g1(p.blocks_x, p.nseg - 1, (unsigned)a.batch);
        cudaError_t e = CONV ? launch_one<T, NK, LPC, true, false, true, PX>(ka, g1, stream)
                             : launch_one<T, NK, LPC, true, false, false, PX>(ka, g1, stream);
        if (e != cudaSuccess) return e;
        ka.nsub_launched = 1;
    }
    const dim3 g2(p.blocks_x, p.nseg, (unsigned)a.batch);
    if (a.z) return launch_one<T, NK, LPC, false, true, CONV, PX>(ka, g2, stream);
    return launch_one<T, NK, LPC, false, false, CONV, PX>(ka, g2, stream);
}

template <typename T, bool CONV>
cudaError_t launch_conv(const ScanArgs& a, const Plan& p, void* ws, cudaStream_t stream) {
    switch (p.NK) {
        case 8: return p.LPC == 1 ? launch_typed<T, 8, 1, CONV>(a, p, ws, stream) : launch_typed<T, 8, 2, CONV>(a, p, ws, stream);
        case 16:
            // the FMA-pipe exponential variants exist for bf16 without the convolution
            if constexpr (std::is_same<T, __nv_bfloat16>::value && !CONV) {
                if (p.px == 1)
                    return p.LPC == 2 ? launch_typed<T, 16, 2, CONV, 1>(a, p, ws, stream)
                                      : launch_typed<T, 16, 4, CONV, 1>(a, p, ws, stream);
                if (p.px == 2)
                    return p.LPC == 2 ? launch_typed<T, 16, 2, CONV, 2>(a, p, ws, stream)
                                      : launch_typed<T, 16, 4, CONV, 2>(a, p, ws, stream);
            }
            return p.LPC == 2 ? launch_typed<T, 16, 2, CONV>(a, p, ws, stream) : launch_typed<T, 16, 4, CONV>(a, p, ws, stream);
        case 32: return p.LPC == 4 ? launch_typed<T, 32, 4, CONV>(a, p, ws, stream) : launch_typed<T, 32, 8, CONV>(a, p, ws, stream);
        default: return launch_typed<T, 64, 8, CONV>(a, p, ws, stream);
    }
}

template <typename T>
cudaError_t launch_dtype(const ScanArgs& a, const Plan& p, void* ws, cudaStream_t stream) {
    return a.conv_k > 0 ? launch_conv<T, true>(a, p, ws, stream) : launch_conv<T, false>(a, p, ws, stream);
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
