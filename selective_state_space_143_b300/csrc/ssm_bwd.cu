// Backward pass of the selective scan: gradients of the inputs from the gradient of the
// output (and optionally of the final state), diagonal (Mamba-1) and SSD (Mamba-2) mode.
//
// The pages give the forward recurrence only ("Mamba-2：把状态空间模型和 Attention 统一到
// 一个数学框架里", 背景问题 / 第一步; training runs it in parallel, "训练时并行化"); the
// reverse-mode derivatives follow from it.  Per channel c, with v_t = dt_t + dt_bias,
// Delta_t = softplus(v_t), a_t[n] = exp(Delta_t A[c,n]) and g_t = dL/dh_t:
//   dy_t   = dout_t SiLU(z_t)                      dz_t = dout_t y_t SiLU'(z_t)
//   g_t    = dy_t C_t + a_{t+1} g_{t+1}            (g starts from dfinal)
//   dx_t   = dy_t D + sum_n g_t Delta_t B_t        dB_t += g_t Delta_t x_t,  dC_t += dy_t h_t
//   dDelta = sum_n g_t (B_t x_t + a_t A h_{t-1})   dA += g_t a_t Delta_t h_{t-1}
//   ddt_t  = dDelta sigmoid(v_t)                   ddt_bias += ddt_t,  dD += dy_t x_t
//   dinit  = a_0 g_0
// SSD mode is the same recurrence per channel c = (head, p) with A, Delta, D and dt_bias
// shared by the head's channels (Mamba-2 explainer, 第二步: a scalar A per head), so
// dA, ddt, dD and ddt_bias of a head are sums over its channels (and, for dA, over n).
//
// Design: LPC lanes of a warp share one channel, each lane R state entries (diagonal
// mode: 4 entries per lane; SSD mode: 8 per lane for dstate above 64; checkpoint
// segments shorten as R grows so that a segment's recomputed states stay in registers).
// A forward sweep stores the state entering every segment of kSeg steps; the reverse
// sweep walks the segments backwards, recomputes each segment's states into registers
// from its checkpoint and runs the adjoint recurrence over them.  With few channels the
// sequence is also cut into time parts: a summary pass gives every part its local end
// state, its local adjoint and its sum of Delta, and the main pass over each part folds
// the earlier parts' states and the later parts' adjoints into its entering state and
// adjoint (see the kernel).
// The per-step scalars of a channel are computed once per segment, spread over its
// lanes, and shuffled to the sweeps; sums over n use shuffles inside the LPC lanes; the
// dB and dC terms of the block's channels (one group) go to shared memory and are summed
// once per segment, then added to global memory once per block and step.  Arithmetic is
// fp32 (CUDA's accurate exp/log1p for fp32 inputs, the SFU exp2 for bf16 inputs, as in
// the forward); every gradient is written in fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>

#include "ssm_device.cuh"
#include "ssd_tc.h"
#include "ssm_internal.h"

namespace ssm {
namespace {

constexpr int kBwdThreads = 256;

// Lanes per channel and entries per lane for a state width N: the width padded to a
// power of two, at most a warp (four entries per lane with fewer lanes measured slower
// on B300: fewer resident warps and a longer per-step chain outweigh the shorter
// reductions); checkpoint segment length by entries per lane.
int bwd_lanes(int64_t N) { return N <= 4 ? 4 : N <= 8 ? 8 : N <= 16 ? 16 : 32; }
int bwd_entries(int64_t N) { return N <= 32 ? 1 : N <= 64 ? 2 : N <= 128 ? 4 : 8; }

// Time parts: the SSM_TUNE_BWD_PARTS override when set.  Otherwise one part when the channels
// give at least 8 warps per SM sub-partition (measured on B300: more parts only add the
// summary pass), else enough parts for ~48 warps per sub-partition, at most 16 and at
// least two checkpoint segments each (c2 backward: 8 parts 11.6 ms, 12 parts 11.2 ms, 16
// parts 11.4 ms; c1: 4 parts 0.40 ms, 12-16 parts 0.34 ms).  Each part is a whole number
// of checkpoint segments; the part count is recomputed from that length.
struct BwdPlan {
    int lpc, r, seg;  // lanes per channel, entries per lane, checkpoint segment length
    int64_t nseg, subs_per_part;
    int parts;
    size_t ckpt_bytes, h_off, q_off, d_off, total;
};
BwdPlan bwd_plan(const ScanArgs& a) {
    const int64_t knob = tuning(2);
    // the SSM_TUNE_BWD_LPC override (4, 8, 16 or 32): lanes per channel (entries per lane
    // follow, at most 4, or 8 with 16 or more lanes)
    const int64_t knob_lpc = tuning(3);
    BwdPlan p;
    p.lpc = bwd_lanes(a.dstate);
    p.r = bwd_entries(a.dstate);
    if (a.headdim == 1 && a.dstate <= 64) {
        // diagonal mode: four entries per lane (fewer per-step reductions; the time parts
        // supply the parallelism): c1 0.49 ms against 0.73 ms with one entry per lane,
        // c2 19.6 ms against 22.2 ms
        p.lpc = a.dstate <= 16 ? 4 : a.dstate <= 32 ? 8 : 16;
        p.r = 1;
        while (p.r * p.lpc < a.dstate) p.r *= 2;
    }
    if (a.dstate > 64 && a.dstate <= 128) {
        // SSD widths: 16 lanes of 8 entries (one shuffle level and half the reductions
        // per entry fewer than 32 x 4): c3 backward 96 ms against 150 ms
        p.lpc = 16;
        p.r = 8;
    }
    if (knob_lpc == 4 || knob_lpc == 8 || knob_lpc == 16 || knob_lpc == 32) {
        int r = 1;
        while (r * knob_lpc < a.dstate) r *= 2;
        if (r <= (knob_lpc >= 16 ? 8 : 4)) {
            p.lpc = (int)knob_lpc;
            p.r = r;
        }
    }
    p.seg = p.r <= 2 ? 16 : p.r == 4 ? 8 : 4;
    const int64_t seg = p.seg;
    p.nseg = (a.seqlen + seg - 1) / seg;
    const int64_t smsp = (int64_t)sm_count() * 4;  // SM sub-partitions
    const int64_t warps = (int64_t)a.batch * a.nheads * a.headdim * p.lpc / 32;
    int64_t rule = 1;
    if (warps > 0 && warps < 8 * smsp)
        rule = std::min<int64_t>({16, (48 * smsp + warps - 1) / warps, std::max<int64_t>(1, p.nseg / 2)});
    const int64_t want = std::max<int64_t>(1, std::min<int64_t>(knob > 0 ? knob : rule, std::max<int64_t>(p.nseg, 1)));
    p.subs_per_part = std::max<int64_t>(1, (p.nseg + want - 1) / want);
    p.parts = (int)std::max<int64_t>(1, (p.nseg + p.subs_per_part - 1) / p.subs_per_part);
    const size_t ch = (size_t)a.batch * a.nheads * a.headdim;
    p.ckpt_bytes = align_up(ch * p.nseg * a.dstate * sizeof(float), 256);
    const size_t hq = p.parts > 1 ? align_up(ch * p.parts * a.dstate * sizeof(float), 256) : 0;
    p.h_off = p.ckpt_bytes;
    p.q_off = p.h_off + hq;
    p.d_off = p.q_off + hq;
    p.total = p.d_off + (p.parts > 1 ? align_up(ch * p.parts * sizeof(float), 256) : 0);
    return p;
}

template <typename T>
struct BwdArgs {
    const T* x;
    const T* dt;
    const T* z;
    const T* B;
    const T* C;
    const T* dout;
    const float* A;
    const float* D;
    const float* dt_bias;
    const float* init;
    const float* dfinal;
    float* dx;
    float* ddt;
    float* dA;
    float* dB;
    float* dC;
    float* dD;
    float* dz;
    float* ddt_bias;
    float* dinit;
    float* ckpt;  // (b, nseg, dim, N): state entering each segment
    // time parts (blockIdx.y), each subs_per_part segments: the parts pass writes, per
    // part k, the local end state Hloc (from zero), the local adjoint Qloc carried out of
    // its first step (from zero at its end), both (b, parts, dim, N), and Dsum (b, parts,
    // dim), the sum of Delta over the part
    float *Hloc, *Qloc, *Dsum;
    int64_t L, dim, N, G, cpg;  // L: sequence length; dim: channels (SSD: heads x P)
    int64_t P;                  // channels per head (SSD headdim; 1 in diagonal mode)
    int nseg, tiles_per_group, subs_per_part;
    // byte ranges of the buffers written (stores checked in SSM_BOUNDS_CHECK builds)
    int* status;
    Span dx_s, ddt_s, dA_s, dB_s, dC_s, dD_s, dz_s, ddtb_s, dinit_s, ckpt_s, hloc_s, qloc_s, dsum_s;
};

template <int LPC>
__device__ __forceinline__ float lane_sum(float v) {
#pragma unroll
    for (int o = LPC / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o, LPC);
    return v;
}

// grid (G * tiles_per_group, parts, batch); LPC lanes x R entries per channel, CPB
// channels, checkpoints every kSeg steps.
// PARTS: the summaries of every time part (forward sweep from zero, adjoint-only reverse
// sweep from zero).  Otherwise the gradients over one part, its entering state folded from
// the earlier parts' summaries, h <- exp(A Dsum_k) h + Hloc_k, and its entering adjoint
// from the later parts', q <- Qloc_k + exp(A Dsum_k) q (the affine combine of the
// parallel-scan formulation, "引言：Attention的天花板" article, 硬件感知算法, run in both
// directions).
// The per-step scalars of a channel (Delta, Delta x, dy, the SiLU' factor, sigmoid(v)) are
// computed once per segment, spread over the channel's lanes (lane j % LPC holds step j),
// and fetched with shuffles inside the sequential sweeps.
template <typename T, int LPC, int R, int kSeg, bool SSD, bool PARTS>
__global__ void __launch_bounds__(kBwdThreads) scan_bwd_kernel(const BwdArgs<T> a) {
    constexpr bool PRECISE = sizeof(T) == 4;
    constexpr int CPB = kBwdThreads / LPC;
    constexpr int NP = LPC * R;                    // padded state width
    // row stride of the dB/dC terms: an odd multiple of LPC, so that the channels of a
    // warp store to distinct banks
    constexpr int SNP = NP + (R > 1 ? LPC : 0);
    constexpr int SPL = (kSeg + LPC - 1) / LPC;    // steps per lane in the per-step pass
    extern __shared__ float s_acc[];               // [2][kSeg][CPB][SNP]: dB and dC terms
    float* s_dB = s_acc;
    float* s_dC = s_acc + kSeg * CPB * SNP;
    // [kSeg][NP]: the segment's B rows (fp32); the part-summary pass has no dB / dC terms
    // and is launched with room for the two row tiles only
    float* s_B = PARTS ? s_acc : s_acc + 2 * kSeg * CPB * SNP;
    float* s_C = s_B + kSeg * NP;                  // [kSeg][NP]: its C rows
    const int tid = threadIdx.x;
    const int lane = tid % LPC;
    const int cc = tid / LPC;  // channel within the block
    const int group = blockIdx.x / a.tiles_per_group;
    const int64_t c_begin = (int64_t)group * a.cpg + (int64_t)(blockIdx.x % a.tiles_per_group) * CPB;
    const int64_t c_end = (int64_t)(group + 1) * a.cpg;
    const int64_t c = c_begin + cc;
    const bool c_ok = c < c_end;
    const int64_t b = blockIdx.z;
    const int64_t L = a.L, dim = a.dim, N = a.N, G = a.G;
    // the index of A's row, Delta, D and dt_bias: the channel, or its head in SSD mode
    const int64_t hd = SSD ? c / a.P : c;
    const int64_t H = SSD ? dim / a.P : dim;

    float Ar[R];
    int nr[R];
    bool nok[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        nr[r] = lane + r * LPC;
        nok[r] = c_ok && nr[r] < N;
        Ar[r] = nok[r] ? a.A[SSD ? hd : c * N + nr[r]] * (PRECISE ? 1.0f : kLog2e) : 0.0f;
    }
    const float bias = (c_ok && a.dt_bias) ? a.dt_bias[hd] : 0.0f;
    const float Dc = (c_ok && a.D) ? a.D[hd] : 0.0f;
    auto decay = [&](float de, int r) { return PRECISE ? expf(de * Ar[r]) : ex2(de * Ar[r]); };
    // the decays of step j for every entry: SSD's scalar A per head makes them one value
    auto decays = [&](float de, float (&av)[R]) {
        if (SSD) {
            const float a0 = decay(de, 0);
#pragma unroll
            for (int r = 0; r < R; ++r) av[r] = a0;
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) av[r] = decay(de, r);
        }
    };
    auto Aval = [&](int r) { return PRECISE ? Ar[r] : Ar[r] * (1.0f / kLog2e); };

    auto row = [&](int64_t t) { return (b * L + t) * dim + c; };
    auto drow = [&](int64_t t) { return (b * L + t) * H + hd; };  // dt and ddt
    auto bc = [&](int64_t t) { return (b * L + t) * G * N + (int64_t)group * N; };
    auto fetch = [&](const float (&v)[SPL], int j) { return __shfl_sync(0xffffffffu, v[j / LPC], j % LPC, LPC); };
    // B and / or C rows t0 .. t0 + len - 1 of the block's group into shared memory as fp32
    // (zero past len and N), read by every channel of the block; the caller's block
    // barrier before it keeps earlier readers safe, the one inside makes the rows visible
    auto stage_bc = [&](int64_t t0, int len, bool withB, bool withC) {
        for (int i = tid; i < kSeg * NP; i += kBwdThreads) {
            const int j = i / NP, n = i % NP;
            const bool ok = j < len && n < N;
            if (withB) s_B[i] = ok ? to_f32<T>(a.B[bc(t0 + j) + n]) : 0.0f;
            if (withC) s_C[i] = ok ? to_f32<T>(a.C[bc(t0 + j) + n]) : 0.0f;
        }
        __syncthreads();
    };

    const int part = blockIdx.y, nparts = gridDim.y;
    const int sub0 = part * a.subs_per_part, sub1 = min(a.nseg, sub0 + a.subs_per_part);
    auto sidx = [&](int k) { return (b * nparts + k) * dim + c; };  // summary of part k

    // forward sweep: checkpoints of the state entering every segment of the part
    float h[R];
#pragma unroll
    for (int r = 0; r < R; ++r) h[r] = (!PARTS && nok[r] && a.init) ? a.init[(b * dim + c) * N + nr[r]] : 0.0f;
    if (!PARTS) {
        for (int k = 0; k < part && c_ok; ++k) {
            const float ds = a.Dsum[sidx(k)];
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (nok[r]) h[r] = fmaf(decay(ds, r), h[r], a.Hloc[sidx(k) * N + nr[r]]);
        }
    }
    float dsum_lane = 0.0f;  // PARTS: this lane's steps of Delta
    // dt and x of a segment, loaded one segment ahead
    float fw_dt[SPL], fw_x[SPL];
    auto prefetch_fw = [&](int sg) {
        const int64_t t0 = (int64_t)sg * kSeg;
        const int len = (int)min((int64_t)kSeg, L - t0);
#pragma unroll
        for (int k = 0; k < SPL; ++k) {
            const int j = lane + LPC * k;
            const bool ok = c_ok && j < len;
            fw_dt[k] = ok ? to_f32<T>(a.dt[drow(t0 + j)]) : 0.0f;
            fw_x[k] = ok ? to_f32<T>(a.x[row(t0 + j)]) : 0.0f;
        }
    };
    if (sub1 > sub0) prefetch_fw(sub0);
    for (int seg = sub0; seg < sub1; ++seg) {
        const int64_t t0 = (int64_t)seg * kSeg;
        float cdt[SPL], cx[SPL];
#pragma unroll
        for (int k = 0; k < SPL; ++k) {
            cdt[k] = fw_dt[k];
            cx[k] = fw_x[k];
        }
        if (seg + 1 < sub1) prefetch_fw(seg + 1);
        __syncthreads();  // every thread is done with the previous segment's rows
        stage_bc(t0, (int)min((int64_t)kSeg, L - t0), true, false);
        if (!PARTS) {
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (nok[r]) store_checked(a.ckpt_s, &a.ckpt[((b * a.nseg + seg) * dim + c) * N + nr[r]], h[r], a.status);
        }
        const int len = (int)min((int64_t)kSeg, L - t0);
        float pde[SPL], pu[SPL];
#pragma unroll
        for (int k = 0; k < SPL; ++k) {
            const int j = lane + LPC * k;
            pde[k] = pu[k] = 0.0f;
            if (c_ok && j < len) {
                pde[k] = softplus_t<PRECISE>(cdt[k] + bias);
                pu[k] = pde[k] * cx[k];
                dsum_lane += pde[k];
            }
        }
#pragma unroll
        for (int j = 0; j < kSeg; ++j) {
            if (j >= len) break;
            const float de = fetch(pde, j), u = fetch(pu, j);
            float av[R];
            decays(de, av);
#pragma unroll
            for (int r = 0; r < R; ++r) h[r] = fmaf(av[r], h[r], u * s_B[j * NP + nr[r]]);
        }
    }

    if (PARTS) {
        // the part's Delta sum and local end state; then its local adjoint, from zero at
        // its end, carried out of its first step (g_t = dy_t C_t + a_{t+1} g_{t+1})
        const float dsum = lane_sum<LPC>(dsum_lane);
        if (c_ok && lane == 0) store_checked(a.dsum_s, &a.Dsum[sidx(part)], dsum, a.status);
        if (part < nparts - 1) {
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (nok[r]) store_checked(a.hloc_s, &a.Hloc[sidx(part) * N + nr[r]], h[r], a.status);
        }
        if (part == 0) return;
        float q[R];
#pragma unroll
        for (int r = 0; r < R; ++r) q[r] = 0.0f;
        for (int seg = sub1 - 1; seg >= sub0; --seg) {
            const int64_t t0 = (int64_t)seg * kSeg;
            const int len = (int)min((int64_t)kSeg, L - t0);
            __syncthreads();
            stage_bc(t0, len, false, true);
            float pde[SPL], pdy[SPL];
#pragma unroll
            for (int k = 0; k < SPL; ++k) {
                const int j = lane + LPC * k;
                pde[k] = pdy[k] = 0.0f;
                if (c_ok && j < len) {
                    const int64_t t = t0 + j;
                    pde[k] = softplus_t<PRECISE>(to_f32<T>(a.dt[drow(t)]) + bias);
                    const float dov = to_f32<T>(a.dout[row(t)]);
                    if (a.z) {
                        const float zv = to_f32<T>(a.z[row(t)]);
                        pdy[k] = dov * zv / (1.0f + __expf(-zv));
                    } else {
                        pdy[k] = dov;
                    }
                }
            }
#pragma unroll
            for (int j = kSeg - 1; j >= 0; --j) {
                if (j >= len) continue;
                const float de = fetch(pde, j), dy = fetch(pdy, j);
                float av[R];
                decays(de, av);
#pragma unroll
                for (int r = 0; r < R; ++r) q[r] = av[r] * fmaf(dy, s_C[j * NP + nr[r]], q[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (nok[r]) store_checked(a.qloc_s, &a.Qloc[sidx(part) * N + nr[r]], q[r], a.status);
    } else {
        // reverse sweep: the adjoint entering the part's last step, folded from the later
        // parts
        float g[R], dA_acc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            g[r] = (nok[r] && a.dfinal) ? a.dfinal[(b * dim + c) * N + nr[r]] : 0.0f;
            dA_acc[r] = 0.0f;
        }
        for (int k = nparts - 1; k > part && c_ok; --k) {
            const float ds = a.Dsum[sidx(k)];
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (nok[r]) g[r] = fmaf(decay(ds, r), g[r], a.Qloc[sidx(k) * N + nr[r]]);
        }
        float dD_acc = 0.0f, dbias_acc = 0.0f;  // this lane's steps
        // the raw per-step inputs and the checkpoint of a segment, loaded one segment ahead
        // so that their latency hides behind the previous segment's sweeps
        float nx_dt[SPL], nx_x[SPL], nx_do[SPL], nx_z[SPL], nx_h0[R];
        auto prefetch_seg = [&](int sg) {
            const int64_t t0 = (int64_t)sg * kSeg;
            const int len = (int)min((int64_t)kSeg, L - t0);
#pragma unroll
            for (int k = 0; k < SPL; ++k) {
                const int j = lane + LPC * k;
                const bool ok = c_ok && j < len;
                const int64_t t = t0 + j;
                nx_dt[k] = ok ? to_f32<T>(a.dt[drow(t)]) : 0.0f;
                nx_x[k] = ok ? to_f32<T>(a.x[row(t)]) : 0.0f;
                nx_do[k] = ok ? to_f32<T>(a.dout[row(t)]) : 0.0f;
                nx_z[k] = (ok && a.z) ? to_f32<T>(a.z[row(t)]) : 0.0f;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) nx_h0[r] = nok[r] ? a.ckpt[((b * a.nseg + sg) * dim + c) * N + nr[r]] : 0.0f;
        };
        if (sub1 > sub0) prefetch_seg(sub1 - 1);
        __syncthreads();  // every thread is done with the forward sweep's last rows
        for (int seg = sub1 - 1; seg >= sub0; --seg) {
            const int64_t t0 = (int64_t)seg * kSeg;
            const int len = (int)min((int64_t)kSeg, L - t0);
            float rdt[SPL], rx[SPL], rdo[SPL], rz[SPL], h0[R];
#pragma unroll
            for (int k = 0; k < SPL; ++k) {
                rdt[k] = nx_dt[k];
                rx[k] = nx_x[k];
                rdo[k] = nx_do[k];
                rz[k] = nx_z[k];
            }
#pragma unroll
            for (int r = 0; r < R; ++r) h0[r] = nx_h0[r];
            if (seg > sub0) prefetch_seg(seg - 1);
            stage_bc(t0, len, true, true);  // the previous segment ended with a block barrier
            // per-step scalars of the segment
            float pde[SPL], pu[SPL], px[SPL], pdy[SPL], pdz[SPL], psig[SPL];
#pragma unroll
            for (int k = 0; k < SPL; ++k) {
                const int j = lane + LPC * k;
                pde[k] = pu[k] = px[k] = pdy[k] = pdz[k] = psig[k] = 0.0f;
                if (c_ok && j < len) {
                    const float v = rdt[k] + bias;
                    pde[k] = softplus_t<PRECISE>(v);
                    psig[k] = 1.0f / (1.0f + __expf(-v));
                    px[k] = rx[k];
                    pu[k] = pde[k] * px[k];
                    const float dov = rdo[k];
                    if (a.z) {
                        const float zv = rz[k];
                        const float sz = 1.0f / (1.0f + __expf(-zv));
                        pdy[k] = dov * zv * sz;
                        pdz[k] = dov * sz * (1.0f + zv * (1.0f - sz));
                    } else {
                        pdy[k] = dov;
                    }
                }
            }
            // the segment's states h_t (after step t), recomputed from the checkpoint
            float hs[kSeg][R];
#pragma unroll
            for (int j = 0; j < kSeg; ++j) {
                if (j < len) {
                    const float de = fetch(pde, j), u = fetch(pu, j);
                    float av[R];
                    decays(de, av);
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        hs[j][r] = fmaf(av[r], j == 0 ? h0[r] : hs[j - 1][r], u * s_B[j * NP + nr[r]]);
                }
            }
#pragma unroll
            for (int j = kSeg - 1; j >= 0; --j) {
                if (j >= len) continue;
                const int64_t t = t0 + j;
                const float de = fetch(pde, j), xv = fetch(px, j), dy = fetch(pdy, j);
                float yp = 0.0f, dxp = 0.0f, ddp = 0.0f;
                float avs[R];
                decays(de, avs);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float Bv = s_B[j * NP + nr[r]];
                    const float Cv = s_C[j * NP + nr[r]];
                    const float av = avs[r];
                    const float hp = j == 0 ? h0[r] : hs[j - 1][r];
                    yp = fmaf(Cv, hs[j][r], yp);
                    g[r] = fmaf(dy, Cv, g[r]);
                    dxp = fmaf(g[r] * de, Bv, dxp);
                    ddp = fmaf(g[r], fmaf(av * Aval(r), hp, Bv * xv), ddp);
                    dA_acc[r] = fmaf(g[r] * av * de, hp, dA_acc[r]);
                    s_dB[(j * CPB + cc) * SNP + r * LPC + lane] = g[r] * de * xv;
                    s_dC[(j * CPB + cc) * SNP + r * LPC + lane] = dy * hs[j][r];
                    g[r] *= av;  // dL/dh_{t-1}
                }
                // three independent reductions over the channel's lanes
#pragma unroll
                for (int o = LPC / 2; o > 0; o >>= 1) {
                    yp += __shfl_xor_sync(0xffffffffu, yp, o, LPC);
                    dxp += __shfl_xor_sync(0xffffffffu, dxp, o, LPC);
                    ddp += __shfl_xor_sync(0xffffffffu, ddp, o, LPC);
                }
                if (c_ok && lane == j % LPC) {  // the lane that holds step j's scalars
                    const int k = j / LPC;
                    store_checked(a.dx_s, &a.dx[row(t)], fmaf(dy, Dc, dxp), a.status);
                    const float dv = ddp * psig[k];
                    if (SSD)
                        atomic_add_checked(a.ddt_s, &a.ddt[drow(t)], dv, a.status);  // the head's channels share Delta_t
                    else
                        store_checked(a.ddt_s, &a.ddt[row(t)], dv, a.status);
                    dbias_acc += dv;
                    dD_acc = fmaf(dy, xv, dD_acc);
                    if (a.z) store_checked(a.dz_s, &a.dz[row(t)], pdz[k] * (yp + Dc * xv), a.status);
                }
            }
            __syncthreads();  // the segment's dB / dC terms are in shared memory
            for (int i = tid; i < len * NP; i += kBwdThreads) {
                const int j = i / NP, n = i % NP;
                if (n < N) {
                    float sb = 0.0f, sc = 0.0f;
                    const int cmax = (int)min((int64_t)CPB, c_end - c_begin);
                    for (int q = 0; q < cmax; ++q) {
                        sb += s_dB[(j * CPB + q) * SNP + n];
                        sc += s_dC[(j * CPB + q) * SNP + n];
                    }
                    const int64_t o = bc(t0 + j) + n;
                    atomic_add_checked(a.dB_s, &a.dB[o], sb, a.status);
                    atomic_add_checked(a.dC_s, &a.dC[o], sc, a.status);
                }
            }
            __syncthreads();  // read before the next segment overwrites them
        }
        dD_acc = lane_sum<LPC>(dD_acc);
        dbias_acc = lane_sum<LPC>(dbias_acc);
        float dA_sum = 0.0f;  // SSD: the head's dA sums every entry of the channel
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (nok[r]) {
                if (a.dinit && part == 0) store_checked(a.dinit_s, &a.dinit[(b * dim + c) * N + nr[r]], g[r], a.status);
                if (SSD)
                    dA_sum += dA_acc[r];
                else
                    atomic_add_checked(a.dA_s, &a.dA[c * N + nr[r]], dA_acc[r], a.status);
            }
        if (SSD) dA_sum = lane_sum<LPC>(dA_sum);
        if (c_ok && lane == 0) {
            if (SSD) atomic_add_checked(a.dA_s, &a.dA[hd], dA_sum, a.status);
            if (a.dD) atomic_add_checked(a.dD_s, &a.dD[hd], dD_acc, a.status);
            if (a.ddt_bias) atomic_add_checked(a.ddtb_s, &a.ddt_bias[hd], dbias_acc, a.status);
        }
    }
}

template <typename T, int LPC, int R, bool SSD>
cudaError_t launch_bwd(const BwdArgs<T>& a, int parts, int64_t batch, cudaStream_t stream) {
    constexpr int kSeg = R <= 2 ? 16 : R == 4 ? 8 : 4;  // as bwd_plan
    constexpr int CPB = kBwdThreads / LPC;
    constexpr size_t kSmem = sizeof(float) * (2 * kSeg * CPB * (LPC * R + (R > 1 ? LPC : 0)) + 2 * kSeg * LPC * R);
    BwdArgs<T> k = a;
    k.tiles_per_group = (int)((a.cpg + CPB - 1) / CPB);
    if (k.nseg != (int)((a.L + kSeg - 1) / kSeg))
        return cudaErrorInvalidValue;  // scratch sized by bwd_plan
    const dim3 grid((unsigned)(a.G * k.tiles_per_group), (unsigned)parts, (unsigned)batch);
    auto kern = scan_bwd_kernel<T, LPC, R, kSeg, SSD, false>;
    if (kSmem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        if (e != cudaSuccess) return e;
    }
    if (parts > 1) {
        constexpr size_t kSmemParts = sizeof(float) * 2 * kSeg * LPC * R;  // B and C rows of a segment
        static_assert(kSmemParts <= 48 * 1024, "part-summary rows");
        cudaEvent_t t1 = timing_begin(stream, "scan_bwd_kernel (part summaries)");
        scan_bwd_kernel<T, LPC, R, kSeg, SSD, true><<<grid, kBwdThreads, kSmemParts, stream>>>(k);
        note_launch("scan_bwd_kernel (part summaries)", stream, t1);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaEvent_t t0 = timing_begin(stream, "scan_bwd_kernel");
    kern<<<grid, kBwdThreads, kSmem, stream>>>(k);
    note_launch("scan_bwd_kernel", stream, t0);
    return cudaGetLastError();
}

// Every (lanes, entries) pair the plans choose: the defaults (one entry per lane up to
// 32 lanes, then 2, 4, 8 entries) and the diagonal-mode tuning knob's (2 or 4 entries
// with 4 to 16 lanes).
template <typename T, bool SSD>
cudaError_t launch_mode(int lpc, int r, const BwdArgs<T>& a, int parts, int64_t batch, cudaStream_t stream) {
    switch (lpc * 10 + r) {
        case 41: return launch_bwd<T, 4, 1, SSD>(a, parts, batch, stream);
        case 42: return launch_bwd<T, 4, 2, SSD>(a, parts, batch, stream);
        case 44: return launch_bwd<T, 4, 4, SSD>(a, parts, batch, stream);
        case 81: return launch_bwd<T, 8, 1, SSD>(a, parts, batch, stream);
        case 82: return launch_bwd<T, 8, 2, SSD>(a, parts, batch, stream);
        case 84: return launch_bwd<T, 8, 4, SSD>(a, parts, batch, stream);
        case 161: return launch_bwd<T, 16, 1, SSD>(a, parts, batch, stream);
        case 162: return launch_bwd<T, 16, 2, SSD>(a, parts, batch, stream);
        case 164: return launch_bwd<T, 16, 4, SSD>(a, parts, batch, stream);
        case 168: return launch_bwd<T, 16, 8, SSD>(a, parts, batch, stream);
        case 321: return launch_bwd<T, 32, 1, SSD>(a, parts, batch, stream);
        case 322: return launch_bwd<T, 32, 2, SSD>(a, parts, batch, stream);
        case 324: return launch_bwd<T, 32, 4, SSD>(a, parts, batch, stream);
        case 328: return launch_bwd<T, 32, 8, SSD>(a, parts, batch, stream);
        default: return cudaErrorInvalidValue;
    }
}
template <typename T>
cudaError_t launch_any(bool ssd, int lpc, int r, const BwdArgs<T>& a, int parts, int64_t batch, cudaStream_t stream) {
    return ssd ? launch_mode<T, true>(lpc, r, a, parts, batch, stream)
               : launch_mode<T, false>(lpc, r, a, parts, batch, stream);
}

template <typename T>
cudaError_t bwd_typed(const ScanBwdArgs& s, void* ws, cudaStream_t stream) {
    const ScanArgs& f = s.fwd;
    BwdArgs<T> a;
    a.x = (const T*)f.x;
    a.dt = (const T*)f.dt;
    a.z = (const T*)f.z;
    a.B = (const T*)f.B;
    a.C = (const T*)f.C;
    a.dout = (const T*)s.dout;
    a.A = f.A;
    a.D = f.D;
    a.dt_bias = f.dt_bias;
    a.init = f.initial_state;
    a.dfinal = s.dfinal;
    a.dx = s.dx;
    a.ddt = s.ddt;
    a.dA = s.dA;
    a.dB = s.dB;
    a.dC = s.dC;
    a.dD = s.dD;
    a.dz = s.dz;
    a.ddt_bias = s.ddt_bias;
    a.dinit = s.dinit;
    const BwdPlan pl = bwd_plan(f);
    a.ckpt = (float*)ws;
    a.Hloc = (float*)((char*)ws + pl.h_off);
    a.Qloc = (float*)((char*)ws + pl.q_off);
    a.Dsum = (float*)((char*)ws + pl.d_off);
    a.nseg = (int)pl.nseg;
    a.subs_per_part = (int)pl.subs_per_part;
    const bool ssd = s.ssd;
    a.L = f.seqlen;
    a.dim = f.nheads * f.headdim;
    a.P = f.headdim;
    a.N = f.dstate;
    a.G = f.ngroups;
    a.cpg = a.dim / f.ngroups;
    a.tiles_per_group = 0;
    a.status = nullptr;
    if (kBoundsCheck) {
        const cudaError_t e = device_status_address(&a.status);
        if (e != cudaSuccess) return e;
    }
    const size_t tok = (size_t)f.batch * f.seqlen;
    const size_t ch = (size_t)f.batch * a.dim;
    a.dx_s = span_of(s.dx, tok * a.dim * 4);
    a.ddt_s = span_of(s.ddt, tok * (ssd ? f.nheads : a.dim) * 4);
    a.dA_s = span_of(s.dA, (size_t)f.nheads * (ssd ? 1 : f.dstate) * 4);
    a.dB_s = span_of(s.dB, tok * f.ngroups * f.dstate * 4);
    a.dC_s = span_of(s.dC, tok * f.ngroups * f.dstate * 4);
    a.dD_s = span_of(s.dD, (size_t)f.nheads * 4);
    a.dz_s = span_of(s.dz, tok * a.dim * 4);
    a.ddtb_s = span_of(s.ddt_bias, (size_t)f.nheads * 4);
    a.dinit_s = span_of(s.dinit, ch * f.dstate * 4);
    a.ckpt_s = span_of(a.ckpt, ch * pl.nseg * f.dstate * 4);
    const size_t hq = pl.parts > 1 ? ch * pl.parts * f.dstate * 4 : 0;
    a.hloc_s = span_of(a.Hloc, hq);
    a.qloc_s = span_of(a.Qloc, hq);
    a.dsum_s = span_of(a.Dsum, pl.parts > 1 ? ch * pl.parts * 4 : 0);
    return launch_any<T>(ssd, pl.lpc, pl.r, a, pl.parts, f.batch, stream);
}

}  // namespace

// The chunked tensor-core backward takes the SSD shapes it supports (bf16, headdim 64,
// dstate 64 or 128) unless SSM_TUNE_SSD_CUDA_CORES keeps SSD on the CUDA cores; every
// other shape runs the recurrence kernel above.
bool use_ssd_tc_bwd(const ScanArgs& a, bool ssd) {
    return ssd && a.batch > 0 && ssd_bwd_tc_supported(a) && tuning(1) != 1;
}

size_t scan_bwd_workspace_bytes(const ScanArgs& a, bool ssd) {
    return use_ssd_tc_bwd(a, ssd) ? ssd_bwd_tc_workspace_bytes(a) : bwd_plan(a).total;
}

cudaError_t scan_bwd_launch(const ScanBwdArgs& s, void* ws, cudaStream_t stream) {
    const ScanArgs& f = s.fwd;
    // accumulated gradients start from zero (SSD: dA per head, and ddt, a sum over the
    // head's channels)
    const size_t acc_bytes[] = {(size_t)f.nheads * (s.ssd ? 1 : f.dstate) * 4,
                                (size_t)f.batch * f.seqlen * f.ngroups * f.dstate * 4,
                                (size_t)f.batch * f.seqlen * f.ngroups * f.dstate * 4, (size_t)f.nheads * 4,
                                (size_t)f.nheads * 4, s.ssd ? (size_t)f.batch * f.seqlen * f.nheads * 4 : 0};
    float* acc[] = {s.dA, s.dB, s.dC, s.dD, s.ddt_bias, s.ddt};
    for (int i = 0; i < 6; ++i)
        if (acc[i] && acc_bytes[i]) {
            const cudaError_t e = cudaMemsetAsync(acc[i], 0, acc_bytes[i], stream);
            if (e != cudaSuccess) return e;
        }
    if (f.batch == 0) return cudaSuccess;
    if (use_ssd_tc_bwd(f, s.ssd)) return ssd_bwd_tc_launch(s, ws, stream);
    if (f.dtype == 1) return bwd_typed<__nv_bfloat16>(s, ws, stream);
    return bwd_typed<float>(s, ws, stream);
}

}  // namespace ssm
