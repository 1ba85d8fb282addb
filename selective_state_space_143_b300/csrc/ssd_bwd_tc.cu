// Backward pass of the SSD (Mamba-2) scan in chunk form on the B300 tensor cores.
//
// The pages give the forward only and say that training evaluates the recurrence in
// parallel ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里", 背景问题 "训练时并行化";
// the chunk algebra of 第二步 and 关键技术点 1-3).  The gradients below are those of the
// chunk form, transposed.  Per batch, head h (scalar A_h), chunk of Q = 128 steps with
// in-chunk cumulative sums cum_t of a_t = Delta_t A_h, state h_in entering the chunk,
// R = dL/dh_out the gradient of the state leaving it, and dy_t = dout_t SiLU(z_t):
//   G_ts  = C_t . B_s,   M_ts = G_ts exp(cum_t - cum_s),   Z_ts = (dy_t . x_s) exp(cum_t - cum_s) Delta_s
//           (s <= t; zero above the diagonal)
//   dX_pre = M^T dY + diag(exp(cum_last - cum)) B R^T         dx = diag(Delta) dX_pre + D dy
//   dC     = Z B + diag(exp(cum)) dY h_in                      (per head; summed over the group)
//   dB     = Z^T C + diag(w) X R,   w_s = Delta_s exp(cum_last - cum_s)
//   dcum_t = C_t . dC_t - B_t . dB_t  (+ <R, h_out> at the chunk's last step)
//   da_t   = sum_{t' >= t in the chunk} dcum_t'       dDelta_t = A_h da_t + x_t . dX_pre_t
//   <R, h_out> = exp(cum_last) <R, h_in> + sum_s w_s x_s . (B R^T)_s
//   ddt_t  = dDelta_t sigmoid(dt_t + dt_bias_h),  ddt_bias_h = sum ddt,  dA_h = sum Delta_t da_t
// dcum needs no Q x Q reduction: the row sums of (G o Z) are C_t . (Z B)_t and its column
// sums B_s . (Z^T C)_s.  R itself follows the adjoint recurrence over chunks,
//   R_{c-1} = exp(cum_last(c)) R_c + sum_t exp(cum_t) dy_t C_t^T,   R_last = dfinal,
// whose chunk terms are the forward chunk-state kernel run on (dy, C) with weights
// exp(cum_t) (ssd_state_tc, adjoint variant).  dD = sum dy x comes from the chunk
// kernel's epilogue, dz (per element) from the dy pass.  Without a gate dy = dout is exact
// in bf16: the dy pass is skipped and the kernels read dout as dy's only plane.
//
// Kernels, in launch order:
//   forward recompute: ssd_state_tc, ssd_state_pass_split (h_in of every chunk as bf16
//     hi/lo tiles, final state), and with a gate ssd_scan_tc without it (y before the gate);
//   ssd_bwd_dy        : with a gate, dy as bf16 hi/lo planes and dz;
//   ssd_state_tc (adjoint), ssd_bwd_reverse_carry: R_c of every chunk as hi/lo tiles,
//     dinitial_state;
//   ssd_bwd_chunk_tc  : one CTA per (chunk, batch, heads of one group): every product above
//     on tcgen05 (bf16 operands, scaled ones split into hi + lo, fp32 accumulators in
//     TMEM), then the per-row epilogues; dB and dC summed over the CTA's heads in TMEM and
//     added to global memory once per CTA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssd_tc.h"
#include "tc_util.cuh"

namespace ssm {
namespace {

constexpr int kP = 64;              // headdim of this path
constexpr int kQ = 128;             // chunk length of this path
constexpr int kStatusTimeout = 8;

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 t = __bfloat1622float2(p[j]);
        f[2 * j] = t.x;
        f[2 * j + 1] = t.y;
    }
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// v = hi + lo with hi = bf16(v), lo = bf16(v - hi), two values at a time
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack2(a - hf.x, b - hf.y);
}
__device__ __forceinline__ float sigmoid_fast(float v) { return __fdividef(1.0f, 1.0f + ex2(-v * kLog2e)); }

// ---- dy pass ------------------------------------------------------------------------
// With a gate: dy = dout SiLU(z) as bf16 hi/lo planes and dz = dout y SiLU'(z), y the
// output before the gate.  grid (ceil(HP / 8 / 256), ceil(T / kDyRows), batch); a thread
// owns one 8-column vector (16 bytes of bf16) over kDyRows rows.
constexpr int kDyRows = 32;

struct DyArgs {
    const __nv_bfloat16* dout;
    const __nv_bfloat16* z;
    const __nv_bfloat16* y;  // output before the gate
    __nv_bfloat16* dy_hi;
    __nv_bfloat16* dy_lo;
    float* dz;
    int64_t T, HP;
    int* status;
    Span dyh_s, dyl_s, dz_s;
};

__global__ void __launch_bounds__(256) ssd_bwd_dy(const DyArgs a) {
    const int64_t v = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (v >= a.HP / 8) return;
    const int64_t b = blockIdx.z;
    const int64_t t0 = (int64_t)blockIdx.y * kDyRows;
    for (int r = 0; r < kDyRows; ++r) {
        const int64_t t = t0 + r;
        if (t >= a.T) break;
        const int64_t o = (b * a.T + t) * a.HP + v * 8;
        float d[8], zz[8], yy[8], dyv[8], dzv[8];
        unpack8(*reinterpret_cast<const uint4*>(a.dout + o), d);
        unpack8(*reinterpret_cast<const uint4*>(a.z + o), zz);
        unpack8(*reinterpret_cast<const uint4*>(a.y + o), yy);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float sg = sigmoid_fast(zz[k]);
            dyv[k] = d[k] * zz[k] * sg;
            dzv[k] = d[k] * yy[k] * sg * (1.0f + zz[k] * (1.0f - sg));
        }
        float4* dzp = reinterpret_cast<float4*>(a.dz + o);
        store_checked(a.dz_s, dzp, make_float4(dzv[0], dzv[1], dzv[2], dzv[3]), a.status);
        store_checked(a.dz_s, dzp + 1, make_float4(dzv[4], dzv[5], dzv[6], dzv[7]), a.status);
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) split2(dyv[2 * j], dyv[2 * j + 1], hi[j], lo[j]);
        store_checked(a.dyh_s, reinterpret_cast<uint4*>(a.dy_hi + o), make_uint4(hi[0], hi[1], hi[2], hi[3]), a.status);
        store_checked(a.dyl_s, reinterpret_cast<uint4*>(a.dy_lo + o), make_uint4(lo[0], lo[1], lo[2], lo[3]), a.status);
    }
}

// ---- reverse carry ---------------------------------------------------------------------
// R over chunks in reverse, in place over the adjoint chunk states (split-ready layout of
// the chunk-state kernel): reads S^g_c, writes R_c = dL/dh_out(c) as bf16 hi/lo tiles,
// R_{c-1} = exp(cum_last(c)) R_c + S^g_c, and dinitial_state = R_{-1}.  grid (ceil(P*N / 8 / 256), H, b); a thread owns the 8 values
// (p, n..n+7) of one 16-byte unit, as the forward carry does.
constexpr int kRevAhead = 2;

struct RevArgs {
    float* ast;
    const float* cum;
    const float* dfinal;
    float* dinit;
    int64_t T, H, P, N, Q, nchunks;
    int* status;
    Span ast_s, dinit_s;
};

__global__ void __launch_bounds__(256) ssd_bwd_reverse_carry(const RevArgs a) {
    const int64_t u = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const int64_t h = blockIdx.y, b = blockIdx.z;
    const int64_t PN = a.P * a.N;
    if (u * 8 >= PN) return;
    const int64_t blk = u >> 3, kb = a.N / 8;
    const int p = (int)((blk / kb) * 8 + (u & 7)), n0 = (int)(blk % kb) * 8;
    const uint32_t o = (uint32_t)(16 * u);
    const int64_t half = PN * 2;
    float R[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) R[k] = a.dfinal ? a.dfinal[(b * a.H + h) * PN + p * a.N + n0 + k] : 0.0f;
    const int64_t cstride = a.H * PN * 4;
    char* base = reinterpret_cast<char*>(a.ast + (b * a.nchunks * a.H + h) * PN);
    const float* cum = a.cum + (b * a.H + h) * a.nchunks * a.Q;
    for (int64_t c0 = a.nchunks - 1; c0 >= 0; c0 -= kRevAhead) {
        float4 S0[kRevAhead], S1[kRevAhead];
        float dec[kRevAhead];
#pragma unroll
        for (int j = 0; j < kRevAhead; ++j) {
            const int64_t c = c0 - j;
            if (c >= 0) {
                S0[j] = *reinterpret_cast<const float4*>(base + c * cstride + o);
                S1[j] = *reinterpret_cast<const float4*>(base + c * cstride + half + o);
                const int len = (int)min(a.Q, a.T - c * a.Q);
                dec[j] = expf(cum[c * a.Q + len - 1]);
            }
        }
#pragma unroll
        for (int j = 0; j < kRevAhead; ++j) {
            const int64_t c = c0 - j;
            if (c < 0) break;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) split2(R[2 * k], R[2 * k + 1], hi[k], lo[k]);
            store_checked(a.ast_s, reinterpret_cast<uint4*>(base + c * cstride + o), make_uint4(hi[0], hi[1], hi[2], hi[3]), a.status);
            store_checked(a.ast_s, reinterpret_cast<uint4*>(base + c * cstride + half + o), make_uint4(lo[0], lo[1], lo[2], lo[3]), a.status);
            const float s[8] = {S0[j].x, S0[j].y, S0[j].z, S0[j].w, S1[j].x, S1[j].y, S1[j].z, S1[j].w};
#pragma unroll
            for (int k = 0; k < 8; ++k) R[k] = fmaf(dec[j], R[k], s[k]);
        }
    }
    if (a.dinit) {
#pragma unroll
        for (int k = 0; k < 8; ++k) store_checked(a.dinit_s, &a.dinit[(b * a.H + h) * PN + p * a.N + n0 + k], R[k], a.status);
    }
}

// ---- chunk gradients on the tensor cores ------------------------------------------------
// Shared memory (N = dstate 64 or 128):
//   sC, sB   : the chunk's C and B rows, [n/64][t 128][64] in the 128-byte swizzle layout
//              (TMA).  K-major operands along n (G = C B^T, B R^T), MN-major along t (Z B,
//              Z^T C).
//   sDy      : dy hi and lo planes of the head, [t][64] swizzled (TMA): K-major along p
//              (dY X^T) and MN-major along t (M^T dY); the epilogue reads D dy from it.
//   region A : the head's x rows [s][64] swizzled (TMA) for dY X^T; then M hi/lo (no
//              swizzle, K-major along s: (t, s) at (t/8)*2048 + (s/8)*128 + (t%8)*16 +
//              (s%8)*2, the same bytes as M^T MN-major); once M^T dY is done, the h_in and
//              R hi/lo tiles (bulk copies of the split-ready layout: K-major along n,
//              MN-major along p).
//   region Z : Z hi/lo (same layout as M); then w o X hi/lo and exp(cum) dY hi/lo
//              (swizzled, written by threads).
// TMEM (512 columns): G [0,128), Z' = dY X^T [128,256) while M and Z are built; then dX
// [0,64), B R^T [64,128); dC [256, 256+N) and dB [256+N, 256+2N) accumulate over the
// CTA's heads (per-head dot products by differences of running sums).
template <int N>
struct BwdCfg {
    static constexpr uint32_t kCB = 128u * N * 2;           // C (or B) rows of the chunk
    static constexpr uint32_t kDy = 128u * kP * 2;          // one dy (or x) plane
    static constexpr uint32_t kMat = 128u * 128 * 2;        // one 128 x 128 operand plane
    static constexpr uint32_t kHt = (uint32_t)kP * N * 2;   // one h or R plane
    static constexpr uint32_t oC = 0, oB = kCB, oDy = 2 * kCB, oA = oDy + 2 * kDy, oZ = oA + 2 * kMat;
    static constexpr uint32_t kSmem = oZ + 2 * kMat;
    static_assert(4 * kHt <= 2 * kMat, "h and R tiles fit region A");
    static_assert(4 * kDy <= 2 * kMat, "w o X and exp(cum) dY fit region Z");
};

struct __align__(16) BwdShared {
    uint64_t mb_cb, mb_x, mb_dy, mb_hr, mb_mfree, mb_mma;
    float dl[kQ], cum[kQ];
    float part[2][kQ];  // per row: x . dX_pre, dcum
    float wsum[4];
    float rsum[8];      // warp partials of <R, h_out>
    float red[4][3];
    uint32_t tmem;
    volatile int abort;
};

struct BwdTcArgs {
    const __nv_bfloat16* x;
    const __nv_bfloat16* dt;
    const float* A;
    const float* D;
    const float* dt_bias;
    const float* dl;     // (b, H, nchunks, Q)
    const float* cum;
    const float* fst;    // forward h_in tiles (hi/lo) of every (b, chunk, head)
    const float* ast;    // R tiles (hi/lo)
    float *dx, *ddt, *dA, *dB, *dC, *dD, *ddt_bias;
    int64_t T, H, G, nchunks;
    Span dx_s, ddt_s, dA_s, dB_s, dC_s, dD_s, ddtb_s;
};

__device__ __forceinline__ void bwd_wait(BwdShared& sh, uint64_t* mb, uint32_t phase) {
    if (sh.abort) return;
    if (!tc::mbar_wait(mb, phase)) sh.abort = 1;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
// 8 bf16 of a 16-byte word, scaled, split into hi / lo words
__device__ __forceinline__ void scale_split8(const float (&f)[8], float w, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) split2(f[2 * k] * w, f[2 * k + 1] * w, h[k], l[k]);
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// grid (nchunks, H / hpc, batch), 256 threads (8 warps; warp w reads TMEM lanes
// 32*(w%4).. and takes column half w/4 of the M and Z builds).  Warps 0-3 own the rows of
// the dx epilogue, w o X and the suffix sums (their thread index is the row); warps 4-7
// those of the dcum epilogue and exp(cum) dY.  DYLO: dy has a lo plane (with a gate);
// without it dy = dout is exact in bf16 and its lo products are skipped.
template <int N, bool DYLO>
__global__ void __launch_bounds__(256, 1)
    ssd_bwd_chunk_tc(const BwdTcArgs a, const int hpc, int* status, const __grid_constant__ CUtensorMap tm_c,
                     const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_dyh, const __grid_constant__ CUtensorMap tm_dyl) {
    using Cfg = BwdCfg<N>;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* sC = smem + Cfg::oC;
    unsigned char* sB = smem + Cfg::oB;
    unsigned char* sDy = smem + Cfg::oDy;
    unsigned char* sA = smem + Cfg::oA;
    unsigned char* sZ = smem + Cfg::oZ;
    BwdShared& sh = *reinterpret_cast<BwdShared*>(smem + Cfg::kSmem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, half = warp >> 2;
    const int r = q * 32 + lane;  // TMEM lane: row t (or s) of the chunk
    const int64_t c = blockIdx.x;
    const int hbeg = blockIdx.y * hpc;
    const int b = blockIdx.z;
    const int row0 = (int)(c * kQ);
    const int len = (int)min((int64_t)kQ, a.T - c * kQ);
    const int g = hbeg / (int)(a.H / a.G);
    const int64_t HP = a.H * kP;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;

    if (tid == 0) {
        tc::mbar_init(&sh.mb_cb, 1);
        tc::mbar_init(&sh.mb_x, 1);
        tc::mbar_init(&sh.mb_dy, 1);
        tc::mbar_init(&sh.mb_hr, 1);
        tc::mbar_init(&sh.mb_mfree, 1);
        tc::mbar_init(&sh.mb_mma, 1);
        sh.abort = 0;
        tc::mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(&sh.tmem, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh.tmem;
    const uint32_t tG = tmem, tZ = tmem + 128, tX = tmem, tXi = tmem + 64;
    const uint32_t tC = tmem + 256, tB = tmem + 256 + N;

    auto issue_x = [&](int hi) {
        tc::mbar_arrive_expect_tx(&sh.mb_x, Cfg::kDy);
        tc::tma_load_3d(sA, &tm_x, (hbeg + hi) * kP, row0, b, &sh.mb_x);
    };
    auto issue_dy = [&](int hi) {
        tc::mbar_arrive_expect_tx(&sh.mb_dy, (DYLO ? 2 : 1) * Cfg::kDy);
        tc::tma_load_3d(sDy, &tm_dyh, (hbeg + hi) * kP, row0, b, &sh.mb_dy);
        if (DYLO) tc::tma_load_3d(sDy + Cfg::kDy, &tm_dyl, (hbeg + hi) * kP, row0, b, &sh.mb_dy);
    };
    if (tid == 0) {
        tc::mbar_arrive_expect_tx(&sh.mb_cb, 2 * Cfg::kCB);
        for (int j = 0; j < N / 64; ++j) {
            tc::tma_load_3d(sC + j * 128 * 128, &tm_c, g * N + 64 * j, row0, b, &sh.mb_cb);
            tc::tma_load_3d(sB + j * 128 * 128, &tm_b, g * N + 64 * j, row0, b, &sh.mb_cb);
        }
        issue_x(0);
        issue_dy(0);
    }

    // per-head values of row tid (tid < 128), fetched one head ahead: Delta, cum, dt
    float pdl = 0.0f, pcum = 0.0f, pdt = 0.0f;
    auto fetch = [&](int hi) {
        const int h = hbeg + hi;
        const int64_t o = (((int64_t)b * a.H + h) * a.nchunks + c) * kQ + tid;
        pdl = a.dl[o];
        pcum = a.cum[o];
        pdt = tid < len ? __bfloat162float(a.dt[((int64_t)b * a.T + row0 + tid) * a.H + h]) : 0.0f;
    };
    if (tid < kQ) fetch(0);

    float prev_c = 0.0f, prev_b = 0.0f;  // running C.dC and B.dB of this thread's row (warps 4-7)
    uint32_t mma_uses = 0;
    auto mma_done = [&]() {
        bwd_wait(sh, &sh.mb_mma, mma_uses & 1);
        ++mma_uses;
        tc::fence_after_sync();
    };

    for (int hi = 0; hi < hpc; ++hi) {
        const int h = hbeg + hi;
        float cdt = 0.0f;
        uint4 cx[8] = {};  // x row tid of this head (warps 0-3), for w o X and x . dX_pre
        if (tid < kQ) {
            sh.dl[tid] = pdl;
            sh.cum[tid] = pcum;
            cdt = pdt;
            const uint4* xr = reinterpret_cast<const uint4*>(a.x + ((int64_t)b * a.T + row0 + tid) * HP + (int64_t)h * kP);
#pragma unroll
            for (int k = 0; k < 8; ++k) cx[k] = tid < len ? xr[k] : make_uint4(0, 0, 0, 0);
            if (hi + 1 < hpc) fetch(hi + 1);
        }
        __syncthreads();
        if (sh.abort) break;
        const float cum_last = sh.cum[kQ - 1];  // rows past len keep the last sum (Delta 0)

        // ---- phase 1: G = C B^T, Z' = dY X^T
        if (tid == 0) {
            if (hi == 0) bwd_wait(sh, &sh.mb_cb, 0);
            bwd_wait(sh, &sh.mb_x, hi & 1);
            bwd_wait(sh, &sh.mb_dy, hi & 1);
            tc::fence_after_sync();
            if (!sh.abort) {
                constexpr uint32_t id = tc::idesc_bf16(128, 128, 0, 0);
#pragma unroll
                for (int ks = 0; ks < N / 16; ++ks) {
                    const uint32_t o = (uint32_t)(ks >> 2) * 128 * 128 + (uint32_t)(ks & 3) * 32;
                    tc::mma_bf16(tG, tc::desc_sw128(tc::smem_u32(sC) + o, 16, 1024),
                                 tc::desc_sw128(tc::smem_u32(sB) + o, 16, 1024), id, ks > 0);
                }
#pragma unroll
                for (int pl = 0; pl < (DYLO ? 2 : 1); ++pl)
#pragma unroll
                    for (int ks = 0; ks < kP / 16; ++ks)
                        tc::mma_bf16(tZ, tc::desc_sw128(tc::smem_u32(sDy + pl * Cfg::kDy) + ks * 32, 16, 1024),
                                     tc::desc_sw128(tc::smem_u32(sA) + ks * 32, 16, 1024), id, (pl | ks) != 0);
            }
            tc::mma_commit(&sh.mb_mma);
        }
        mma_done();

        // ---- phase 2: M (region A) and Z (region Z), hi/lo, from TMEM row t = r, columns
        // s of this warp's half
        {
            const int t = r;
            const float at = sh.cum[t] * kLog2e;
            const uint32_t aM = tc::smem_u32(sA), aZ = tc::smem_u32(sZ);
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                const int s0 = half * 64 + j * 16;
                uint32_t gv[16], zv[16];
                tc::tmem_ld16_async(tG + lane_base + (uint32_t)s0, gv);
                tc::tmem_ld16_async(tZ + lane_base + (uint32_t)s0, zv);
                tc::tmem_wait_ld();
                uint32_t mh[8], ml[8], zh[8], zl[8];
#pragma unroll
                for (int k = 0; k < 16; k += 2) {
                    float m2[2], z2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int s = s0 + k + e;
                        const float dec = s <= t ? ex2(at - sh.cum[s] * kLog2e) : 0.0f;
                        m2[e] = __uint_as_float(gv[k + e]) * dec;
                        z2[e] = __uint_as_float(zv[k + e]) * dec * sh.dl[s];
                    }
                    split2(m2[0], m2[1], mh[k / 2], ml[k / 2]);
                    split2(z2[0], z2[1], zh[k / 2], zl[k / 2]);
                }
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    const uint32_t off = (uint32_t)((t >> 3) * 2048 + ((s0 >> 3) + c8) * 128 + (t & 7) * 16);
                    const int w0 = c8 * 4;
                    sts128(aM + off, mh[w0], mh[w0 + 1], mh[w0 + 2], mh[w0 + 3]);
                    sts128(aM + Cfg::kMat + off, ml[w0], ml[w0 + 1], ml[w0 + 2], ml[w0 + 3]);
                    sts128(aZ + off, zh[w0], zh[w0 + 1], zh[w0 + 2], zh[w0 + 3]);
                    sts128(aZ + Cfg::kMat + off, zl[w0], zl[w0 + 1], zl[w0 + 2], zl[w0 + 3]);
                }
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();

        // ---- phase 3a: dX = M^T dY (then region A is free: h_in and R tiles are copied in
        // while the rest runs); dC += Z B; dB += Z^T C
        if (tid == 0) {
            tc::fence_after_sync();
            if (!sh.abort) {
                const uint32_t aM = tc::smem_u32(sA), aZ = tc::smem_u32(sZ), aDy = tc::smem_u32(sDy);
                constexpr uint32_t idX = tc::idesc_bf16(128, kP, 1, 1);
                const int combo_m[3] = {0, 1, 0}, combo_d[3] = {0, 0, 1};
#pragma unroll
                for (int cb = 0; cb < (DYLO ? 3 : 2); ++cb)
#pragma unroll
                    for (int ks = 0; ks < kQ / 16; ++ks)
                        tc::mma_bf16(tX, tc::desc_mnmajor(aM + combo_m[cb] * Cfg::kMat, 128, ks),
                                     tc::desc_sw128(aDy + combo_d[cb] * Cfg::kDy + ks * 2048, 1024, 1024), idX,
                                     (cb | ks) != 0);
                tc::mma_commit(&sh.mb_mfree);
                constexpr uint32_t idC = tc::idesc_bf16(128, N, 0, 1);
                constexpr uint32_t idB = tc::idesc_bf16(128, N, 1, 1);
#pragma unroll
                for (int pl = 0; pl < 2; ++pl)
#pragma unroll
                    for (int ks = 0; ks < kQ / 16; ++ks) {
                        const uint32_t acc = (hi > 0 || pl > 0 || ks > 0) ? 1u : 0u;
                        tc::mma_bf16(tC, tc::desc_strided(aZ + pl * Cfg::kMat + ks * 256, 128, 2048),
                                     tc::desc_sw128(tc::smem_u32(sB) + ks * 2048, 128 * 128, 1024), idC, acc);
                        tc::mma_bf16(tB, tc::desc_mnmajor(aZ + pl * Cfg::kMat, 128, ks),
                                     tc::desc_sw128(tc::smem_u32(sC) + ks * 2048, 128 * 128, 1024), idB, acc);
                    }
            } else {
                tc::mma_commit(&sh.mb_mfree);
            }
            tc::mma_commit(&sh.mb_mma);
            bwd_wait(sh, &sh.mb_mfree, hi & 1);
            if (!sh.abort) {
                const int64_t tile = (((int64_t)b * a.nchunks + c) * a.H + h) * (int64_t)kP * N;
                tc::mbar_arrive_expect_tx(&sh.mb_hr, 4 * Cfg::kHt);
                tc::bulk_load(sA, a.fst + tile, 2 * Cfg::kHt, &sh.mb_hr);
                tc::bulk_load(sA + 2 * Cfg::kHt, a.ast + tile, 2 * Cfg::kHt, &sh.mb_hr);
            }
        }
        mma_done();

        // ---- phase 3b prep (region Z is free): w o X from the x row in registers
        // (warps 0-3), exp(cum_t) dY from sDy (warps 4-7), both swizzled like TMA tiles
        if (half == 0) {
            const int s = r;  // == tid
            const float w = s < len ? sh.dl[s] * __expf(cum_last - sh.cum[s]) : 0.0f;
#pragma unroll
            for (int pc = 0; pc < 8; ++pc) {
                float fx[8];
                unpack8(cx[pc], fx);
                uint4 vh, vl;
                scale_split8(fx, w, vh, vl);
                const uint32_t off = (uint32_t)(s * 128 + ((pc ^ (s & 7)) * 16));
                *reinterpret_cast<uint4*>(sZ + off) = vh;
                *reinterpret_cast<uint4*>(sZ + Cfg::kDy + off) = vl;
            }
        } else {
            const int t = r;
            const float e = __expf(sh.cum[t]);
#pragma unroll
            for (int pc = 0; pc < 8; ++pc) {
                const uint32_t off = (uint32_t)(t * 128 + ((pc ^ (t & 7)) * 16));
                float fh[8];
                unpack8(*reinterpret_cast<const uint4*>(sDy + off), fh);
                if (DYLO) {
                    float fl[8];
                    unpack8(*reinterpret_cast<const uint4*>(sDy + Cfg::kDy + off), fl);
#pragma unroll
                    for (int k = 0; k < 8; ++k) fh[k] += fl[k];
                }
                uint4 vh, vl;
                scale_split8(fh, e, vh, vl);
                *reinterpret_cast<uint4*>(sZ + 2 * Cfg::kDy + off) = vh;
                *reinterpret_cast<uint4*>(sZ + 3 * Cfg::kDy + off) = vl;
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();

        // ---- phase 3b: dXi = B R^T; dC += (e dY) h_in; dB += (w o X) R
        if (tid == 0) {
            bwd_wait(sh, &sh.mb_hr, hi & 1);
            tc::fence_after_sync();
            if (!sh.abort) {
                const uint32_t aH = tc::smem_u32(sA), aR = aH + 2 * Cfg::kHt, aW = tc::smem_u32(sZ),
                               aE = aW + 2 * Cfg::kDy;
                constexpr uint32_t idXi = tc::idesc_bf16(128, kP, 0, 0);
#pragma unroll
                for (int pl = 0; pl < 2; ++pl)
#pragma unroll
                    for (int ks = 0; ks < N / 16; ++ks)
                        tc::mma_bf16(tXi,
                                     tc::desc_sw128(tc::smem_u32(sB) + (uint32_t)(ks >> 2) * 128 * 128 + (uint32_t)(ks & 3) * 32,
                                                    16, 1024),
                                     tc::desc_strided(aR + pl * Cfg::kHt + ks * 256, 128, (N / 8) * 128), idXi,
                                     (pl | ks) != 0);
                constexpr uint32_t idCB = tc::idesc_bf16(128, N, 0, 1);
                const int combo_a[3] = {0, 1, 0}, combo_b[3] = {0, 0, 1};
#pragma unroll
                for (int cb = 0; cb < 3; ++cb)
#pragma unroll
                    for (int ks = 0; ks < kP / 16; ++ks) {
                        tc::mma_bf16(tC, tc::desc_sw128(aE + combo_a[cb] * Cfg::kDy + ks * 32, 16, 1024),
                                     tc::desc_mnmajor(aH + combo_b[cb] * Cfg::kHt, N, ks), idCB, 1u);
                        tc::mma_bf16(tB, tc::desc_sw128(aW + combo_a[cb] * Cfg::kDy + ks * 32, 16, 1024),
                                     tc::desc_mnmajor(aR + combo_b[cb] * Cfg::kHt, N, ks), idCB, 1u);
                    }
            }
            tc::mma_commit(&sh.mb_mma);
        }
        // meanwhile <R, h_in> over the two tiles in region A (hi + lo of each)
        float phr = 0.0f;
        if (tid != 0) bwd_wait(sh, &sh.mb_hr, hi & 1);
        if (!sh.abort) {
            constexpr int kWords = (int)(Cfg::kHt / 16);  // 16-byte words per plane
#pragma unroll
            for (int i = tid; i < kWords; i += 256) {
                float hh[8], hl[8], rh[8], rl[8];
                unpack8(*reinterpret_cast<const uint4*>(sA + i * 16), hh);
                unpack8(*reinterpret_cast<const uint4*>(sA + Cfg::kHt + i * 16), hl);
                unpack8(*reinterpret_cast<const uint4*>(sA + 2 * Cfg::kHt + i * 16), rh);
                unpack8(*reinterpret_cast<const uint4*>(sA + 3 * Cfg::kHt + i * 16), rl);
#pragma unroll
                for (int k = 0; k < 8; ++k) phr = fmaf(hh[k] + hl[k], rh[k] + rl[k], phr);
            }
        }
        mma_done();
        __syncthreads();
        if (sh.abort) break;
        if (tid == 0 && hi + 1 < hpc) issue_x(hi + 1);  // region A is free again
        float prd = __expf(cum_last) * phr;  // this thread's part of <R, h_out>
        float pdd = 0.0f;                      // this thread's part of dD (row s, warps 0-3)

        // ---- phase 4: epilogues
        if (half == 0) {
            // dx and x . dX_pre of row s = r
            const int s = r;
            float ddir = 0.0f;
            const float dec = __expf(cum_last - sh.cum[s]);
            const float Dh = a.D ? a.D[h] : 0.0f;
            const float dls = sh.dl[s];
            float xri = 0.0f;  // x_s . (B R^T)_s
            float xdy = 0.0f;  // x_s . dy_s (dD)
            float* dxr = a.dx + ((int64_t)b * a.T + row0 + s) * HP + (int64_t)h * kP;
#pragma unroll
            for (int p0 = 0; p0 < kP; p0 += 16) {
                uint32_t xv[16], xi[16];
                tc::tmem_ld16_async(tX + lane_base + (uint32_t)p0, xv);
                tc::tmem_ld16_async(tXi + lane_base + (uint32_t)p0, xi);
                tc::tmem_wait_ld();
                if (s < len) {
                    float out[16];
#pragma unroll
                    for (int c8 = 0; c8 < 2; ++c8) {
                        const int pc = (p0 >> 3) + c8;
                        const uint32_t off = (uint32_t)(s * 128 + ((pc ^ (s & 7)) * 16));
                        float fx[8], fh[8], fl[8] = {};
                        unpack8(cx[pc], fx);
                        unpack8(*reinterpret_cast<const uint4*>(sDy + off), fh);
                        if (DYLO) unpack8(*reinterpret_cast<const uint4*>(sDy + Cfg::kDy + off), fl);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int j = c8 * 8 + k;
                            const float pre = fmaf(dec, __uint_as_float(xi[j]), __uint_as_float(xv[j]));
                            const float dy = fh[k] + fl[k];
                            ddir = fmaf(fx[k], pre, ddir);
                            xri = fmaf(fx[k], __uint_as_float(xi[j]), xri);
                            xdy = fmaf(fx[k], dy, xdy);
                            out[j] = fmaf(dls, pre, Dh * dy);
                        }
                    }
                    float4* dst = reinterpret_cast<float4*>(dxr + p0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        store_checked(a.dx_s, dst + k, make_float4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]), status);
                }
            }
            sh.part[0][s] = ddir;
            prd = fmaf(dls * dec, xri, prd);  // w_s x_s . (B R^T)_s: <R, S_c> of row s
            pdd = xdy;
        } else {
            // dcum of row t = r: C_t . dC_t - B_t . dB_t for this head (running sums over
            // the CTA's heads, differenced)
            const int t = r;
            float sc = 0.0f, sb = 0.0f;
#pragma unroll 1
            for (int n0 = 0; n0 < N; n0 += 16) {
                uint32_t cv[16], bv[16];
                tc::tmem_ld16_async(tC + lane_base + (uint32_t)n0, cv);
                tc::tmem_ld16_async(tB + lane_base + (uint32_t)n0, bv);
                tc::tmem_wait_ld();
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    const int n = n0 + c8 * 8;
                    const uint32_t off = (uint32_t)((n >> 6) * 128 * 128 + t * 128 + ((((n & 63) >> 3) ^ (t & 7)) * 16));
                    float fc[8], fb[8];
                    unpack8(*reinterpret_cast<const uint4*>(sC + off), fc);
                    unpack8(*reinterpret_cast<const uint4*>(sB + off), fb);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        sc = fmaf(fc[k], __uint_as_float(cv[c8 * 8 + k]), sc);
                        sb = fmaf(fb[k], __uint_as_float(bv[c8 * 8 + k]), sb);
                    }
                }
            }
            sh.part[1][t] = (sc - prev_c) - (sb - prev_b);
            prev_c = sc;
            prev_b = sb;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) prd += __shfl_xor_sync(0xffffffffu, prd, o);
        if (lane == 0) sh.rsum[warp] = prd;
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0 && hi + 1 < hpc) issue_dy(hi + 1);  // the epilogue has read sDy
        if (half == 0) {
            // da_t = sum of dcum over t' >= t (suffix sum over the chunk's 128 rows; the
            // last row also carries <R, h_out>, which reaches every row)
            const int t = r;
            float v = sh.part[1][t];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_down_sync(0xffffffffu, v, o);
                if (lane + o < 32) v += u;
            }
            if (lane == 0) sh.wsum[q] = v;
            asm volatile("bar.sync 1, 128;" ::: "memory");
            for (int w = q + 1; w < 4; ++w) v += sh.wsum[w];
            float rdot = 0.0f;
#pragma unroll
            for (int w = 0; w < 8; ++w) rdot += sh.rsum[w];
            const float da = v + rdot;
            const float dDelta = fmaf(a.A[h], da, sh.part[0][t]);
            float ddt = 0.0f;
            if (t < len) {
                const float bias = a.dt_bias ? a.dt_bias[h] : 0.0f;
                ddt = dDelta * sigmoid_fast(cdt + bias);
                store_checked(a.ddt_s, &a.ddt[((int64_t)b * a.T + row0 + t) * a.H + h], ddt, status);
            }
            float pa = sh.dl[t] * da, pb = ddt, pc = pdd;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                pa += __shfl_xor_sync(0xffffffffu, pa, o);
                pb += __shfl_xor_sync(0xffffffffu, pb, o);
                pc += __shfl_xor_sync(0xffffffffu, pc, o);
            }
            if (lane == 0) {
                sh.red[q][0] = pa;
                sh.red[q][1] = pb;
                sh.red[q][2] = pc;
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (tid == 0) {
                float sa = 0.0f, sbias = 0.0f, sd = 0.0f;
                for (int w = 0; w < 4; ++w) {
                    sa += sh.red[w][0];
                    sbias += sh.red[w][1];
                    sd += sh.red[w][2];
                }
                atomic_add_checked(a.dA_s, a.dA + h, sa, status);
                if (a.ddt_bias) atomic_add_checked(a.ddtb_s, a.ddt_bias + h, sbias, status);
                if (a.dD) atomic_add_checked(a.dD_s, a.dD + h, sd, status);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
    }

    // ---- dB and dC of the CTA's heads (one group) into global memory (every lane of a
    // warp takes part in the TMEM loads; rows past the sequence add nothing)
    if (!sh.abort) {
        const int t = r;
        const int64_t o = (((int64_t)b * a.T + row0 + t) * a.G + g) * N;
#pragma unroll 1
        for (int n0 = half * (N / 2); n0 < (half + 1) * (N / 2); n0 += 16) {
            uint32_t cv[16], bv[16];
            tc::tmem_ld16_async(tC + lane_base + (uint32_t)n0, cv);
            tc::tmem_ld16_async(tB + lane_base + (uint32_t)n0, bv);
            tc::tmem_wait_ld();
            if (t < len) {
#pragma unroll
                for (int k = 0; k < 16; k += 4) {
                    atomic_add4_checked(a.dC_s, a.dC + o + n0 + k,
                                        make_float4(__uint_as_float(cv[k]), __uint_as_float(cv[k + 1]),
                                                    __uint_as_float(cv[k + 2]), __uint_as_float(cv[k + 3])), status);
                    atomic_add4_checked(a.dB_s, a.dB + o + n0 + k,
                                        make_float4(__uint_as_float(bv[k]), __uint_as_float(bv[k + 1]),
                                                    __uint_as_float(bv[k + 2]), __uint_as_float(bv[k + 3])), status);
                }
            }
        }
    }
    if (sh.abort && tid == 0) atomicExch(status, kStatusTimeout);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ---- host side -----------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 bwd_encode_tiled() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            (void)cudaGetLastError();
            return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 3-D map over a bf16 tensor (inner, T, batch): boxes of 64 inner elements x 128 rows in
// the 128-byte swizzle layout; rows past T read as zero.
bool bwd_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t T, uint64_t batch) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = bwd_encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[3] = {inner, T, batch};
    const cuuint64_t strides[2] = {inner * 2, inner * 2 * T};
    const cuuint32_t box[3] = {64, (cuuint32_t)kQ, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct BwdTcPlan {
    int64_t nchunks;
    size_t o_dl, o_cum, o_fst, o_ast, o_y, o_dyh, o_dyl, total;
};

BwdTcPlan bwd_tc_plan(const ScanArgs& a) {
    BwdTcPlan p;
    p.nchunks = (a.seqlen + kQ - 1) / kQ;
    const size_t vec = (size_t)a.batch * a.nheads * p.nchunks * kQ * sizeof(float);
    const size_t st = (size_t)a.batch * p.nchunks * a.nheads * a.headdim * a.dstate * sizeof(float);
    const size_t el = (size_t)a.batch * a.seqlen * a.nheads * a.headdim * 2;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += align_up(bytes, 256);
        return at;
    };
    p.o_dl = take(vec);
    p.o_cum = take(vec);
    p.o_fst = take(st);
    p.o_ast = take(st);
    p.o_y = take(el);  // with a gate (the size query does not know whether there is one)
    p.o_dyh = take(el);
    p.o_dyl = take(el);
    p.total = o;
    return p;
}

// Heads per CTA of the chunk-gradient kernel: the largest of 16, 8, 4, 2, 1 dividing the
// heads of a group that still gives about four CTAs per SM (one CTA per SM fits).
int bwd_heads_per_cta(const ScanArgs& a, int64_t nchunks) {
    const int64_t hpg = a.nheads / a.ngroups;
    for (int cand : {16, 8, 4, 2})
        if (hpg % cand == 0 && nchunks * (a.nheads / cand) * a.batch >= 4 * (int64_t)sm_count()) return cand;
    return 1;
}

template <int N, bool DYLO>
cudaError_t launch_chunk(const BwdTcArgs& k, const ScanArgs& f, const BwdTcPlan& pl, const void* dyh, const void* dyl,
                         cudaStream_t stream) {
    using Cfg = BwdCfg<N>;
    CUtensorMap tc_, tb_, tx_, tdh, tdl;
    const uint64_t T = (uint64_t)f.seqlen, nb = (uint64_t)f.batch, HP = (uint64_t)f.nheads * kP;
    if (!bwd_map(&tc_, f.C, (uint64_t)f.ngroups * N, T, nb) || !bwd_map(&tb_, f.B, (uint64_t)f.ngroups * N, T, nb) ||
        !bwd_map(&tx_, f.x, HP, T, nb) || !bwd_map(&tdh, dyh, HP, T, nb) || !bwd_map(&tdl, DYLO ? dyl : dyh, HP, T, nb))
        return cudaErrorInvalidValue;
    int* status = nullptr;
    cudaError_t e = device_status_address(&status);
    if (e != cudaSuccess) return e;
    constexpr uint32_t smem_bytes = Cfg::kSmem + (uint32_t)sizeof(BwdShared);
    static_assert(smem_bytes <= 232448, "shared memory");
    auto kern = ssd_bwd_chunk_tc<N, DYLO>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return e;
    const int hpc = bwd_heads_per_cta(f, pl.nchunks);
    cudaEvent_t t0 = timing_begin(stream, "ssd_bwd_chunk_tc");
    kern<<<dim3((unsigned)pl.nchunks, (unsigned)(f.nheads / hpc), (unsigned)f.batch), 256, smem_bytes, stream>>>(
        k, hpc, status, tc_, tb_, tx_, tdh, tdl);
    note_launch("ssd_bwd_chunk_tc", stream, t0);
    return cudaGetLastError();
}

}  // namespace

bool ssd_bwd_tc_supported(const ScanArgs& a) {
    return a.dtype == 1 && a.headdim == kP && (a.dstate == 64 || a.dstate == 128) && a.seqlen > 0 &&
           a.conv_k == 0 && !a.x_f32 && ssd_tc_supported(a, kQ);
}

size_t ssd_bwd_tc_workspace_bytes(const ScanArgs& a) { return bwd_tc_plan(a).total; }

cudaError_t ssd_bwd_tc_launch(const ScanBwdArgs& s, void* ws, cudaStream_t stream) {
    const ScanArgs& f = s.fwd;
    const BwdTcPlan pl = bwd_tc_plan(f);
    char* w = static_cast<char*>(ws);
    float* dl = reinterpret_cast<float*>(w + pl.o_dl);
    float* cum = reinterpret_cast<float*>(w + pl.o_cum);
    float* fst = reinterpret_cast<float*>(w + pl.o_fst);
    float* ast = reinterpret_cast<float*>(w + pl.o_ast);
    __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(w + pl.o_y);
    __nv_bfloat16* dyh = reinterpret_cast<__nv_bfloat16*>(w + pl.o_dyh);
    __nv_bfloat16* dyl = reinterpret_cast<__nv_bfloat16*>(w + pl.o_dyl);
    const int64_t b = f.batch, T = f.seqlen, H = f.nheads, P = f.headdim, N = f.dstate;
    const size_t vec = (size_t)b * H * pl.nchunks * kQ * sizeof(float);
    const size_t stb = (size_t)b * pl.nchunks * H * P * N * sizeof(float);
    const size_t el = (size_t)b * T * H * P;
    int* status = nullptr;
    if (kBoundsCheck) {
        const cudaError_t e = device_status_address(&status);
        if (e != cudaSuccess) return e;
    }

    // forward recompute: Delta, cumulative sums, h_in of every chunk, and with a gate the
    // output before it
    SsdTcArgs t = {};
    t.x = static_cast<const __nv_bfloat16*>(f.x);
    t.x_lo = nullptr;
    t.dt = static_cast<const __nv_bfloat16*>(f.dt);
    t.z = nullptr;
    t.B = static_cast<const __nv_bfloat16*>(f.B);
    t.C = static_cast<const __nv_bfloat16*>(f.C);
    t.A = f.A;
    t.D = f.D;
    t.dt_bias = f.dt_bias;
    t.out = y;
    t.dl = dl;
    t.cum = cum;
    t.states = fst;
    t.T = T;
    t.H = H;
    t.N = N;
    t.G = f.ngroups;
    t.Q = kQ;
    t.nchunks = pl.nchunks;
    t.out_s = span_of(f.z ? y : nullptr, el * 2);
    t.dl_s = span_of(dl, vec);
    t.cum_s = span_of(cum, vec);
    t.states_s = span_of(fst, stb);
    cudaError_t e = ssd_tc_chunk_state(t, b, stream);
    if (e != cudaSuccess) return e;
    e = ssd_tc_forward_carry(f, kQ, pl.nchunks, cum, fst, nullptr, stream);
    if (e != cudaSuccess) return e;
    if (f.z) {
        e = ssd_tc_chunk_scan(t, b, false, stream);
        if (e != cudaSuccess) return e;
    }

    // with a gate: dy planes and dz; without one dy = dout, exact in bf16, read in place
    const bool gate = f.z != nullptr;
    const __nv_bfloat16* dy_hi = gate ? dyh : static_cast<const __nv_bfloat16*>(s.dout);
    const __nv_bfloat16* dy_lo = gate ? dyl : nullptr;
    if (gate) {
        DyArgs d;
        d.dout = static_cast<const __nv_bfloat16*>(s.dout);
        d.z = static_cast<const __nv_bfloat16*>(f.z);
        d.y = y;
        d.dy_hi = dyh;
        d.dy_lo = dyl;
        d.dz = s.dz;
        d.T = T;
        d.HP = H * P;
        d.status = status;
        d.dyh_s = span_of(dyh, el * 2);
        d.dyl_s = span_of(dyl, el * 2);
        d.dz_s = span_of(s.dz, el * 4);
        const dim3 grid((unsigned)((H * P / 8 + 255) / 256), (unsigned)((T + kDyRows - 1) / kDyRows), (unsigned)b);
        cudaEvent_t t0 = timing_begin(stream, "ssd_bwd_dy");
        ssd_bwd_dy<<<grid, 256, 0, stream>>>(d);
        note_launch("ssd_bwd_dy", stream, t0);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    // adjoint chunk states, then R over the chunks in reverse
    SsdTcArgs ta = t;
    ta.x = dy_hi;
    ta.x_lo = dy_lo;
    ta.B = static_cast<const __nv_bfloat16*>(f.C);
    ta.states = ast;
    ta.states_s = span_of(ast, stb);
    e = ssd_tc_chunk_state_adjoint(ta, b, stream);
    if (e != cudaSuccess) return e;
    {
        RevArgs rv;
        rv.ast = ast;
        rv.cum = cum;
        rv.dfinal = s.dfinal;
        rv.dinit = s.dinit;
        rv.T = T;
        rv.H = H;
        rv.P = P;
        rv.N = N;
        rv.Q = kQ;
        rv.nchunks = pl.nchunks;
        rv.status = status;
        rv.ast_s = span_of(ast, stb);
        rv.dinit_s = span_of(s.dinit, (size_t)b * H * P * N * sizeof(float));
        const dim3 grid((unsigned)((P * N / 8 + 255) / 256), (unsigned)H, (unsigned)b);
        cudaEvent_t t0 = timing_begin(stream, "ssd_bwd_reverse_carry");
        ssd_bwd_reverse_carry<<<grid, 256, 0, stream>>>(rv);
        note_launch("ssd_bwd_reverse_carry", stream, t0);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    // the chunk gradients
    BwdTcArgs k;
    k.x = static_cast<const __nv_bfloat16*>(f.x);
    k.dt = static_cast<const __nv_bfloat16*>(f.dt);
    k.A = f.A;
    k.D = f.D;
    k.dt_bias = f.dt_bias;
    k.dl = dl;
    k.cum = cum;
    k.fst = fst;
    k.ast = ast;
    k.dx = s.dx;
    k.ddt = s.ddt;
    k.dA = s.dA;
    k.dB = s.dB;
    k.dC = s.dC;
    k.ddt_bias = s.ddt_bias;
    k.dD = s.dD;
    k.T = T;
    k.H = H;
    k.G = f.ngroups;
    k.nchunks = pl.nchunks;
    k.dx_s = span_of(s.dx, el * 4);
    k.ddt_s = span_of(s.ddt, (size_t)b * T * H * 4);
    k.dA_s = span_of(s.dA, (size_t)H * 4);
    k.dB_s = span_of(s.dB, (size_t)b * T * f.ngroups * N * 4);
    k.dC_s = span_of(s.dC, (size_t)b * T * f.ngroups * N * 4);
    k.ddtb_s = span_of(s.ddt_bias, (size_t)H * 4);
    k.dD_s = span_of(s.dD, (size_t)H * 4);
    if (gate)
        return N == 64 ? launch_chunk<64, true>(k, f, pl, dy_hi, dy_lo, stream)
                       : launch_chunk<128, true>(k, f, pl, dy_hi, dy_lo, stream);
    return N == 64 ? launch_chunk<64, false>(k, f, pl, dy_hi, dy_lo, stream)
                   : launch_chunk<128, false>(k, f, pl, dy_hi, dy_lo, stream);
}

}  // namespace ssm
