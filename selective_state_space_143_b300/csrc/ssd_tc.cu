// Mamba-2 / SSD chunk kernels on the B300 tensor cores (tcgen05, TMEM accumulators).
//
// Same chunk algebra as ssd_scan.cu ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里",
// 第二步 and 关键技术点 1-3: y = (L o M) x, dense diagonal blocks, low-rank off-diagonal
// blocks through the carried state), with the three matrix products of a chunk issued
// as tcgen05.mma (bf16 operands in shared memory, fp32 accumulators in tensor memory):
//
//   ssd_state_tc : S_c^T for up to 8 heads of a chunk, two at a time:
//                  D[(head, p), n] = sum_s Xd[s, (head, p)] B[s, n]
//                  with Xd[s, :] = exp(s_last - s_s) Delta_s x_s  (M = 128, N = dstate, K = Q)
//   ssd_scan_tc  : per (chunk, 128-row half): G = C_rows B^T once (M = 128, N = rows up to
//                  the half's end, K = dstate), then per head
//                    M'[t, s] = G[t, s] exp(s_t - s_s) Delta_s  (s <= t, else 0) -> bf16 smem
//                    Y_diag   = M' X_h                            (M = 128, N = 64, K = s)
//                    Y_off    = C_rows h_{c-1}^T                  (M = 128, N = 64, K = dstate)
//                    out      = (Y_diag + exp(s_t) Y_off + D x) SiLU(z)
// The carry h_c = exp(s_last) h_{c-1} + S_c runs in between (ssd_state_pass_split in
// ssd_scan.cu): ssd_state_tc stores S_c in a split-ready layout and the carry writes
// h_{c-1} back as the bf16 hi/lo tiles that ssd_scan_tc copies into shared memory.
//
// Shapes taken here: bf16, headdim 64, dstate a multiple of 16 in [32, 256], chunk 128 or
// 256, an even number of heads per group.  Other shapes use the CUDA-core kernels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssd_tc.h"
#include "tc_util.cuh"

namespace ssm {

namespace {

constexpr int kP = 64;         // headdim handled here
constexpr int kThreads = 256;      // state kernel: 8 warps (16 with split x), TMEM lanes 32*(w%4).., column part w/4
constexpr int kScanThreads = 512;  // scan kernel: 16 warps, TMEM lanes 32*(w%4).., column quarter w/4
constexpr int kStatusTimeout = 8;

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* gmem, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// For HPC heads [hbeg, hbeg + HPC) of chunk c at once (one row s per thread; Q <= 256):
// Delta_s, the inclusive cumulative sum cum_s of Delta_s A_h (both to global, for the
// scan kernel) and the chunk-end weights w[h][s] = exp(cum_last - cum_s) Delta_s.  Rows
// past len get Delta 0.  s_warp: [8 warps][HPC].
template <int HPC>
__device__ void delta_cumsum_heads(const SsdTcArgs& a, int64_t b, int64_t hbeg, int64_t c, int len,
                                   float (*s_w)[256], float* s_warp) {
    const int s = threadIdx.x, lane = s & 31, warp = s >> 5;
    float d[HPC], v[HPC];
    const int64_t row = (b * a.T + c * a.Q + s) * a.H + hbeg;
#pragma unroll
    for (int k = 0; k < HPC; ++k) {
        d[k] = 0.0f;
        if (s < len) d[k] = softplus(__bfloat162float(a.dt[row + k]) + (a.dt_bias ? a.dt_bias[hbeg + k] : 0.0f));
        v[k] = d[k] * a.A[hbeg + k];
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int k = 0; k < HPC; ++k) {
            const float u = __shfl_up_sync(0xffffffffu, v[k], o);
            if (lane >= o) v[k] += u;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int k = 0; k < HPC; ++k) s_warp[warp * HPC + k] = v[k];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < HPC; ++k)
        for (int w = 0; w < warp; ++w) v[k] += s_warp[w * HPC + k];
    // cum_last of every head: row len-1 publishes it through s_w (overwritten below)
    if (s == len - 1) {
#pragma unroll
        for (int k = 0; k < HPC; ++k) s_w[k][255] = v[k];
    }
    __syncthreads();
    float last[HPC];
#pragma unroll
    for (int k = 0; k < HPC; ++k) last[k] = s_w[k][255];
    __syncthreads();
    if (s < a.Q) {
#pragma unroll
        for (int k = 0; k < HPC; ++k) {
            const int64_t o = ((b * a.H + hbeg + k) * a.nchunks + c) * a.Q + s;
            a.dl[o] = d[k];
            a.cum[o] = v[k];
            s_w[k][s] = s < len ? __expf(last[k] - v[k]) * d[k] : 0.0f;
        }
    }
}

// Tile fill orders that keep 16-byte shared-memory stores free of bank conflicts: the
// row index inside a core matrix (8 rows x 16 bytes, contiguous) runs fastest.
// K-major tile, KC chunks of 8 elements per row: i -> (row, chunk).
__device__ __forceinline__ void kmajor_item(int i, int KC, int& row, int& kc) {
    row = (i / (8 * KC)) * 8 + (i & 7);
    kc = (i >> 3) % KC;
}
// MN-major tile, MC chunks of 8 elements along M/N: i -> (k, chunk).
__device__ __forceinline__ void mnmajor_item(int i, int MC, int& k, int& mc) {
    k = (i / (8 * MC)) * 8 + (i & 7);
    mc = (i >> 3) % MC;
}

}  // namespace

// Per-device status word: a kernel that gave up a bounded wait records SSM_ERR_TIMEOUT
// here (and returns instead of hanging); the host reads and clears it through
// device_status_take (ssm_device_status).
__device__ int g_device_status = 0;

namespace {

__device__ __forceinline__ void report_timeout() { atomicExch(&g_device_status, kStatusTimeout); }

// One CTA waits on an mbarrier that expects one arrival which nothing makes, giving up
// after max_checks polls: the bounded-wait path of the kernels above, on demand.
__global__ void bounded_wait_selftest(uint32_t max_checks) {
    __shared__ __align__(8) uint64_t mbar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&mbar, 1);
        tc::mbar_fence_init();
    }
    __syncthreads();
    const bool ok = tc::mbar_wait_bounded(&mbar, 0, max_checks);
    if (!ok && threadIdx.x == 0) report_timeout();
}

}  // namespace

// hi/lo split of a scaled operand: v = hi + lo with hi = bf16(v), lo = bf16(v - hi).
// Feeding both halves to accumulating MMAs against the same raw (exact bf16) operand
// keeps ~16 mantissa bits of the scaled operand, so the only rounding left is fp32
// accumulation.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_bf16x2(a - hf.x, b - hf.y);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d));
}

// State kernel configuration: heads per CTA (a divisor of the heads per group, so that
// every head of the CTA reads the same B rows) and the K-part of Q taken per step.
// XS: x arrives as bf16 hi/lo planes (the convolved input); both planes are prefetched,
// so the kernel runs 16 warps to keep the per-thread registers of the prefetch the same.
template <int N, bool XS = false>
struct StateTcCfg {
    static constexpr int NT = XS ? 512 : kThreads;            // threads
    static constexpr int PL = XS ? 2 : 1;                     // x planes
    static constexpr int KS = N > 128 ? 64 : 128;             // rows s per step
    static constexpr size_t kB = (size_t)256 * N * 2;         // B rows [0, Q), resident
    static constexpr size_t kXPart = (size_t)128 * KS * 2;    // one Xd part, hi or lo
    static constexpr size_t kSmem = kB + 4 * kXPart;          // + 2 stages x (hi, lo)
    static constexpr int kMaxHeads = 8;
    static constexpr int XCH = 128 * KS / 8 / NT;             // 8-element x chunks per thread
};

// grid (nchunks, H / hpc, b); 256 threads.  S_c^T for hpc heads of chunk c, two heads
// (128 accumulator rows) per pair:
//   D[(head, p), n] = sum_s Xd[s, (head, p)] B[s, n],  Xd[s, :] = exp(cum_last - cum_s) Delta_s x_s
// B (Q x N) is loaded once.  The pairs' K-parts form one pipeline of steps: the raw x of
// step n+1 is in flight (registers) while step n's weighted, hi/lo-split Xd is written
// to stage buffer n%2 and the MMAs of step n-1 run; a pair's epilogue (TMEM -> states)
// runs once the next pair's first MMAs are queued, from alternating accumulators.
template <int N, bool XS>
__global__ void __launch_bounds__(StateTcCfg<N, XS>::NT) ssd_state_tc(const SsdTcArgs a, int hpc) {
    using Cfg = StateTcCfg<N, XS>;
    constexpr int KS = Cfg::KS, NT = Cfg::NT, PL = Cfg::PL;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ float s_w[Cfg::kMaxHeads][256], s_warp[NT / 32 * Cfg::kMaxHeads];
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_mbar[2];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t c = blockIdx.x, hbeg = (int64_t)blockIdx.y * hpc, b = blockIdx.z;
    const int Q = (int)a.Q;
    const int len = (int)min((int64_t)Q, a.T - c * a.Q);
    const int64_t g = hbeg / (a.H / a.G);
    const int nkp = Q / KS;                  // steps per pair
    const int nsteps = (hpc / 2) * nkp;
    unsigned char* sB = smem;                // MN-major B operand: N_mma = n, K = s
    unsigned char* sX = smem + Cfg::kB;      // [stage][hi, lo], MN-major A: M = (head, p), K = s

    // B rows of the chunk, once
    {
        const uint32_t bb = tc::smem_u32(sB);
        for (int i = tid; i < Q * (N / 8); i += NT) {
            int s, nc;
            mnmajor_item(i, N / 8, s, nc);
            const bool ok = s < len;
            const __nv_bfloat16* src = a.B + (ok ? (((b * a.T + c * a.Q + s) * a.G + g) * a.N + nc * 8) : 0);
            cp_async16(bb + tc::off_mnmajor(nc * 8, s, N), src, ok);
        }
        asm volatile("cp.async.commit_group;\n" ::);
    }
    constexpr uint32_t kCols = 2 * N < 32 ? 32 : 2 * N;  // two accumulators
    if (warp == 0) tc::tmem_alloc(&s_tmem, kCols);
    if (tid == 0) {
        tc::mbar_init(&s_mbar[0], 1);
        tc::mbar_init(&s_mbar[1], 1);
        tc::mbar_fence_init();
    }

    // raw x of step n in registers: rows s in [kp*KS, +KS) of heads (pair, pair+1), each
    // plane; two register sets, so that steps n+1 and n+2 are in flight while step n is
    // built
    uint4 pfa[PL][Cfg::XCH], pfb[PL][Cfg::XCH];
    auto prefetch = [&](int n, uint4 (&pf)[PL][Cfg::XCH]) {
        const int pair = n / nkp, kp = n % nkp;
#pragma unroll
        for (int j = 0; j < Cfg::XCH; ++j) {
            int sl, mc;
            mnmajor_item(tid + j * NT, 16, sl, mc);
            const int s = kp * KS + sl, m0 = mc * 8;
            const int64_t h = hbeg + 2 * pair + m0 / kP;
            const int64_t o = ((b * a.T + c * a.Q + s) * a.H + h) * kP + m0 % kP;
#pragma unroll
            for (int pl = 0; pl < PL; ++pl) {
                pf[pl][j] = make_uint4(0, 0, 0, 0);
                if (s < len) pf[pl][j] = *reinterpret_cast<const uint4*>((pl ? a.x_lo : a.x) + o);
            }
        }
    };
    // Xd of step n -> stage n%2, hi/lo
    auto build = [&](int n, const uint4 (&pf)[PL][Cfg::XCH]) {
        const int pair = n / nkp, kp = n % nkp;
        unsigned char* st = sX + (n & 1) * 2 * Cfg::kXPart;
        const uint32_t bh = tc::smem_u32(st), bl = tc::smem_u32(st + Cfg::kXPart);
#pragma unroll
        for (int j = 0; j < Cfg::XCH; ++j) {
            int sl, mc;
            mnmajor_item(tid + j * NT, 16, sl, mc);
            const int m0 = mc * 8;
            const float w = s_w[2 * pair + m0 / kP][kp * KS + sl];
            const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&pf[0][j]);
            const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&pf[PL - 1][j]);
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float2 f = __bfloat1622float2(r2[k]);
                if (XS) {  // x' = x_hi + x_lo
                    const float2 fl = __bfloat1622float2(l2[k]);
                    f.x += fl.x;
                    f.y += fl.y;
                }
                split2(f.x * w, f.y * w, hi[k], lo[k]);
            }
            const uint32_t off = tc::off_mnmajor(m0, sl, 128);
            st_shared_v4(bh + off, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(bl + off, lo[0], lo[1], lo[2], lo[3]);
        }
    };
    // accumulator of pair -> the (b, c, h) state tile; warp w: lanes 32*(w%4).., column
    // part w/4 (halves with 8 warps, quarters with 16).  Split-ready layout: the 8 values of (p, n..n+7) go as two float4 to the
    // byte offsets that their bf16 hi and lo halves take in the scan kernel's K-major
    // tile (offset o in the first P*N*2 bytes, and o + P*N*2), so that the carry pass can
    // convert every unit in place (see ssd_state_pass_split).
    auto epilogue = [&](uint32_t tmem, int pair) {
        const int q = warp & 3;
        const int m = q * 32 + (tid & 31);
        const int64_t h = hbeg + 2 * pair + m / kP;
        const int p = m % kP;
        char* tile = reinterpret_cast<char*>(a.states + ((b * a.nchunks + c) * a.H + h) * (int64_t)kP * N);
        constexpr uint32_t kHalf = (uint32_t)kP * N * 2;
        const uint32_t acc = tmem + (uint32_t)((pair & 1) * N);
        constexpr int NH = N / (NT / 128) < 16 ? 16 : N / (NT / 128);  // a multiple of 16
#pragma unroll 1
        for (int n0 = (warp >> 2) * NH; n0 < N && n0 < ((warp >> 2) + 1) * NH; n0 += 16) {
            float v[16];
            tc::tmem_ld16(tc::taddr(acc, q * 32, n0), v);
#pragma unroll
            for (int j = 0; j < 16; j += 8) {
                const uint32_t o = tc::off_kmajor(p, n0 + j, N);
                *reinterpret_cast<float4*>(tile + o) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                *reinterpret_cast<float4*>(tile + kHalf + o) = make_float4(v[j + 4], v[j + 5], v[j + 6], v[j + 7]);
            }
        }
    };

    // steps 0 and 1 in flight during the Delta pass; Delta, cumulative sums (to global,
    // for the scan kernel) and chunk-end weights of all the CTA's heads in one pass
    prefetch(0, pfa);
    if (nsteps > 1) prefetch(1, pfb);
    if (hpc == 8)
        delta_cumsum_heads<8>(a, b, hbeg, c, len, s_w, s_warp);
    else if (hpc == 4)
        delta_cumsum_heads<4>(a, b, hbeg, c, len, s_w, s_warp);
    else
        delta_cumsum_heads<2>(a, b, hbeg, c, len, s_w, s_warp);
    asm volatile("cp.async.wait_group 0;\n" ::);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    bool ok = true;
    // commit n arrives on s_mbar[n & 1], phase (n >> 1) & 1; a wait is only ever on the
    // latest commit of its barrier
    auto wait_commit = [&](int n) {
        ok = tc::mbar_wait(&s_mbar[n & 1], (uint32_t)(n >> 1) & 1u) && ok;
        tc::fence_after_sync();
    };
    auto step = [&](int n, uint4 (&pf)[PL][Cfg::XCH]) {
        const int pair = n / nkp, kp = n % nkp;
        if (n >= 2) wait_commit(n - 2);  // stage n%2 free again
        build(n, pf);
        if (n + 2 < nsteps) prefetch(n + 2, pf);
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        if (tid == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16(128, N, 1, 1);
            unsigned char* st = sX + (n & 1) * 2 * Cfg::kXPart;
            const uint64_t dxh = tc::desc_mnmajor(tc::smem_u32(st), 128, 0);
            const uint64_t dxl = tc::desc_mnmajor(tc::smem_u32(st + Cfg::kXPart), 128, 0);
            const uint64_t db = tc::desc_mnmajor(tc::smem_u32(sB), N, kp * (KS / 16));
            const uint32_t d = tmem + (uint32_t)((pair & 1) * N);
#pragma unroll
            for (int ks = 0; ks < KS / 16; ++ks)
                tc::mma_bf16(d, dxh + ks * tc::kstep_mnmajor(128), db + ks * tc::kstep_mnmajor(N), idesc,
                             (kp > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < KS / 16; ++ks)
                tc::mma_bf16(d, dxl + ks * tc::kstep_mnmajor(128), db + ks * tc::kstep_mnmajor(N), idesc, 1u);
            tc::mma_commit(&s_mbar[n & 1]);
        }
        // the previous pair's states, once this pair's first MMAs are queued
        if (kp == 0 && pair > 0) {
            wait_commit(n - 1);
            epilogue(tmem, pair - 1);
            tc::fence_before_sync();
        }
    };
    for (int n = 0; n < nsteps && ok; n += 2) {
        step(n, pfa);
        if (n + 1 < nsteps && ok) step(n + 1, pfb);
    }
    if (ok && nsteps > 0) {
        wait_commit(nsteps - 1);
        epilogue(tmem, hpc / 2 - 1);
    }
    if (!ok && tid == 0) report_timeout();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

// Columns of M' built per K-part (two K-part buffers alternate).
template <int N>
struct ScanTcCfg {
    static constexpr int KPC = N > 128 ? 32 : 64;
    static constexpr size_t kC = (size_t)128 * N * 2;            // C rows, resident
    static constexpr size_t kPhase1 = (size_t)256 * N * 2;       // B rows [0, SW)
    static constexpr size_t kMPart = (size_t)128 * KPC * 2;      // one M' K-part, hi or lo
    static constexpr size_t kX = (size_t)256 * kP * 2;           // one x_h tile
    static constexpr size_t kH = (size_t)kP * N * 2;             // one h tile, hi or lo
    static constexpr int kHBufs = N <= 128 ? 2 : 1;               // (hi, lo) tile sets
    static constexpr size_t kPhase2 = 4 * kMPart + 2 * kX + kHBufs * 2 * kH;
    static constexpr size_t kSmem = kC + (kPhase1 > kPhase2 ? kPhase1 : kPhase2);
};

// grid (nchunks * Q/128, H / HG, b); 512 threads.  Rows [128*rh, 128*rh + 128) of chunk c,
// heads [HG*blockIdx.y, +HG).
// Per head h, pipelined over the CTA's heads:
//   commit   : prefetched inputs of h to shared memory (x_h into its parity buffer, h_{c-1}
//              split hi/lo), inputs of h+1 fetched into registers;
//   K-parts  : M' columns built into alternating buffers while the tensor core runs the
//              previous part's MMAs (Y_diag += M'_hi X + M'_lo X; Y_off with part 0);
//   finish   : the epilogue of head h-1, from its own TMEM accumulators, right after
//              head h's first MMAs are issued.
// XS (x' = x_hi + x_lo, the convolved input): Y_diag adds M'_hi X_lo (M'_lo X_lo is
// below the split's own rounding) and the skip term reads x' from global memory.  With
// 128 rows s (first half) both planes fit in one x buffer and the head pipeline is as
// above; with 256 rows the two buffers hold the current head's planes and the next
// head's planes are copied in once this head's last MMAs are done, while its first M'
// part is built.
template <int N, bool GATE, bool XS>
__global__ void __launch_bounds__(kScanThreads, 1) ssd_scan_tc(const SsdTcArgs a, int heads_per_cta) {
    using Cfg = ScanTcCfg<N>;
    constexpr int KPC = Cfg::KPC;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ float s_cum[256];
    __shared__ __align__(16) float s_beta[256];
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_mbar[3];  // [0], [1]: MMA commits by parity; [2]: G
    const int tid = threadIdx.x, warp = tid >> 5;
    const int Q = (int)a.Q;
    const int halves = Q / 128;
    const int64_t c = blockIdx.x / halves;
    const int rh = blockIdx.x % halves;
    const int64_t b = blockIdx.z;
    const int len = (int)min((int64_t)Q, a.T - c * a.Q);
    const int t0 = 128 * rh;
    if (t0 >= len) return;  // no valid rows in this half (uniform)
    const int SW = t0 + 128;  // columns s of G needed by this half (causal)
    const int nparts = SW / KPC;
    const int64_t hbeg = (int64_t)blockIdx.y * heads_per_cta;
    const int64_t g = hbeg / (a.H / a.G);

    unsigned char* sC = smem;                            // K-major: M = t (128), K = n
    unsigned char* region = smem + Cfg::kC;
    unsigned char* sB = region;                          // phase 1, K-major: N_mma = s, K = n
    unsigned char* sM = region;                          // [2 parts][hi, lo], K-major: M = t, K = KPC
    unsigned char* sX = region + 4 * Cfg::kMPart;        // [2], MN-major: K = s, N_mma = p
    unsigned char* sH = sX + 2 * Cfg::kX;                // [kHBufs][hi, lo], K-major: N_mma = p, K = n

    // phase 1 loads: C rows of this half and B rows [0, SW)
    {
        const uint32_t cb = tc::smem_u32(sC), bb = tc::smem_u32(sB);
        for (int i = tid; i < 128 * (N / 8); i += kScanThreads) {
            int rr, nc;
            kmajor_item(i, N / 8, rr, nc);
            const int s = t0 + rr;
            const bool ok = s < len;
            const __nv_bfloat16* src = a.C + (ok ? (((b * a.T + c * a.Q + s) * a.G + g) * a.N + nc * 8) : 0);
            cp_async16(cb + tc::off_kmajor(rr, nc * 8, N), src, ok);
        }
        for (int i = tid; i < SW * (N / 8); i += kScanThreads) {
            int s, nc;
            kmajor_item(i, N / 8, s, nc);
            const bool ok = s < len;
            const __nv_bfloat16* src = a.B + (ok ? (((b * a.T + c * a.Q + s) * a.G + g) * a.N + nc * 8) : 0);
            cp_async16(bb + tc::off_kmajor(s, nc * 8, N), src, ok);
        }
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) tc::mbar_init(&s_mbar[i], 1);
        tc::mbar_fence_init();
    }
    cp_async_commit_wait_all();
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t tG = tmem;
    bool ok = true;

    // G = C_rows B^T (raw bf16 operands: exact products, fp32 accumulation)
    if (tid == 0) {
        const uint32_t idesc = tc::idesc_bf16(128, SW, 0, 0);
        const uint64_t da = tc::desc_kmajor(tc::smem_u32(sC), N, 0), db = tc::desc_kmajor(tc::smem_u32(sB), N, 0);
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks)
            tc::mma_bf16(tG, da + ks * tc::kstep_kmajor(), db + ks * tc::kstep_kmajor(), idesc, ks > 0);
        tc::mma_commit(&s_mbar[2]);
    }
    ok = tc::mbar_wait(&s_mbar[2], 0);
    tc::fence_after_sync();

    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int cq = warp >> 2;                // column quarter of this warp
    const int r = q * 32 + (tid & 31);       // my row (TMEM lane) within the half
    const int t = t0 + r;                    // row within the chunk
    const bool row_ok = t < len;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int t_warp_max = t0 + q * 32 + 31;  // tcgen05.ld is warp-collective
    constexpr int BC = KPC / 4;              // columns of a K-part built by one warp

    // MMA commits are numbered; commit n arrives on s_mbar[n & 1], phase (n >> 1) & 1.
    uint32_t ncommit = 0;
    auto wait_commit = [&](uint32_t n) {
        ok = tc::mbar_wait(&s_mbar[n & 1], (n >> 1) & 1) && ok;
        tc::fence_after_sync();
    };

    // next head's Delta and cumsum in registers (see commit below); its x_h and its
    // h_{c-1} tiles go straight to shared memory by cp.async (load_x, load_h)
    float pf_dl = 0.0f, pf_cum = 0.0f;
    // h_{c-1} of head hn (bf16 hi and lo tiles, already in this kernel's K-major layout,
    // written by the carry pass) -> tile set hbuf
    auto load_h = [&](int64_t hn, int hbuf) {
        const unsigned char* src = reinterpret_cast<const unsigned char*>(
            a.states + ((b * a.nchunks + c) * a.H + hn) * (int64_t)kP * N);
        const uint32_t dst = tc::smem_u32(sH + hbuf * 2 * Cfg::kH);
        for (int i = tid; i < (int)(2 * Cfg::kH / 16); i += kScanThreads) cp_async16(dst + 16 * i, src + 16 * i, true);
        asm volatile("cp.async.commit_group;\n" ::);
    };
    // XS placement of the planes of head hi: serial (256 rows) x_hi in buffer 0 and x_lo
    // in buffer 1; else both in buffer hi&1, x_lo after the SW rows of x_hi
    const bool xser = XS && SW > 128;
    auto x_hi_tile = [&](int hi_) { return sX + (xser ? 0 : (hi_ & 1)) * Cfg::kX; };
    auto x_lo_tile = [&](int hi_) { return xser ? sX + Cfg::kX : x_hi_tile(hi_) + (size_t)SW * kP * 2; };
    // x_h of head hn (plane: x, or x_lo) -> the tile at xt (MN-major, rows s < SW; rows
    // past len are zero-filled)
    auto load_x = [&](const __nv_bfloat16* plane, int64_t hn, unsigned char* xt) {
        const uint32_t xb = tc::smem_u32(xt);
        for (int i = tid; i < SW * (kP / 8); i += kScanThreads) {
            int s, pc;
            mnmajor_item(i, kP / 8, s, pc);
            const bool okr = s < len;
            const __nv_bfloat16* src = plane + (okr ? ((b * a.T + c * a.Q + s) * a.H + hn) * kP + pc * 8 : 0);
            cp_async16(xb + tc::off_mnmajor(pc * 8, s, kP), src, okr);
        }
        asm volatile("cp.async.commit_group;\n" ::);
    };
    auto prefetch = [&](int64_t hn) {
        if (tid < Q) {
            const int64_t o = ((b * a.H + hn) * a.nchunks + c) * a.Q + tid;
            pf_dl = a.dl[o];
            pf_cum = a.cum[o];
        }
    };
    // prefetched inputs -> shared memory: cumsum and beta_s = log2(Delta_s) - cum_s log2(e)
    // (so that exp(cum_t - cum_s) Delta_s = 2^(cum_t log2(e) + beta_s)); x_h MN-major into
    // buffer xb; h split hi/lo K-major
    auto commit = [&]() {
        if (tid < Q) {
            s_cum[tid] = pf_cum;
            s_beta[tid] = (pf_dl > 0.0f ? lg2(pf_dl) : -INFINITY) - pf_cum * kLog2e;
        }
        // this head's x_h and h tiles (visible after the sync); XS waits before its first MMAs
        if (!XS) asm volatile("cp.async.wait_group 0;\n" ::);
    };
    // epilogue of head hh from accumulator set acc: y = Y_diag + exp(cum_t) Y_off + D x, gate
    auto finish = [&](int64_t hh, int acc, float alpha_h) {
        const unsigned char* xs = sX + acc * Cfg::kX;  // x_h of head hh (buffer parity = acc)
        const uint32_t tYd = tmem + 256 + 128 * acc, tYo = tYd + 64;
        const float et = ex2(alpha_h);
        const float Dh = a.D ? a.D[hh] : 0.0f;
        const int64_t row = ((b * a.T + c * a.Q + t) * a.H + hh) * kP;
        {
            const int p0 = 16 * cq;  // this warp's 16 head channels
            float yd[16], yo[16];
            tc::tmem_ld16(tYd + lane_base + (uint32_t)p0, yd);
            tc::tmem_ld16(tYo + lane_base + (uint32_t)p0, yo);
            if (row_ok) {
                uint32_t pk[8];
#pragma unroll
                for (int j = 0; j < 16; j += 8) {
                    uint4 xr, xl = make_uint4(0, 0, 0, 0);
                    if (XS) {
                        xr = *reinterpret_cast<const uint4*>(a.x + row + p0 + j);
                        xl = *reinterpret_cast<const uint4*>(a.x_lo + row + p0 + j);
                    } else {
                        xr = *reinterpret_cast<const uint4*>(xs + tc::off_mnmajor(p0 + j, t, kP));
                    }
                    const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xr);
                    const __nv_bfloat162* xl2 = reinterpret_cast<const __nv_bfloat162*>(&xl);
                    uint4 zr = make_uint4(0, 0, 0, 0);
                    if (GATE) zr = *reinterpret_cast<const uint4*>(a.z + row + p0 + j);
                    const __nv_bfloat162* z2 = reinterpret_cast<const __nv_bfloat162*>(&zr);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float2 xv = __bfloat1622float2(x2[k]);
                        if (XS) {
                            const float2 lv = __bfloat1622float2(xl2[k]);
                            xv.x += lv.x;
                            xv.y += lv.y;
                        }
                        float y0 = fmaf(et, yo[j + 2 * k], yd[j + 2 * k]) + Dh * xv.x;
                        float y1 = fmaf(et, yo[j + 2 * k + 1], yd[j + 2 * k + 1]) + Dh * xv.y;
                        if (GATE) {
                            const float2 zv = __bfloat1622float2(z2[k]);
                            y0 *= silu(zv.x);
                            y1 *= silu(zv.y);
                        }
                        pk[j / 2 + k] = pack_bf16x2(y0, y1);
                    }
                }
                uint4* dst = reinterpret_cast<uint4*>(a.out + row + p0);
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
        }
    };

    if (ok) {
        prefetch(hbeg);
        load_x(a.x, hbeg, x_hi_tile(0));
        if (XS) load_x(a.x_lo, hbeg, x_lo_tile(0));
        load_h(hbeg, 0);
    }
    uint32_t last_commit_prev = 0;  // the previous head's last commit
    float alpha_prev = 0.0f;
    for (int hi = 0; hi < heads_per_cta && ok; ++hi) {
        const int64_t h = hbeg + hi;
        // every thread is past the previous head's M' builds before s_cum / s_beta change
        // (the h_{c-1} tiles have their own hand-over: two tile sets, or the copy at part 2)
        __syncthreads();
        commit();
        if (hi + 1 < heads_per_cta) prefetch(h + 1);
        tc::fence_async_smem();
        __syncthreads();
        const float alpha = s_cum[min(t, Q - 1)] * kLog2e;
        for (int kp = 0; kp < nparts; ++kp) {
            // this K-part's buffer was last used by commit ncommit - 2
            if (ncommit >= 2) wait_commit(ncommit - 2);
            // one h tile set: part 0's MMAs (the last readers of this head's h tiles) are
            // done once commit ncommit - 2 has arrived at part 2
            if (Cfg::kHBufs == 1 && kp == 2 && hi + 1 < heads_per_cta) load_h(h + 1, 0);
            // M'[t, s] = G[t, s] 2^(alpha_t + beta_s) for s <= t, hi/lo, K-major.  This warp
            // builds BC columns of the part for its 32 rows.
            {
                unsigned char* part = sM + (ncommit & 1) * 2 * Cfg::kMPart;
                const uint32_t mh = tc::smem_u32(part), ml = tc::smem_u32(part + Cfg::kMPart);
                const int s0 = KPC * kp + BC * cq;
                uint32_t ph[BC / 2], pl[BC / 2];
                if (s0 <= t_warp_max) {  // some s <= t for this warp (warp-uniform)
                    uint32_t gv[BC];
                    tc::tmem_ld_async(tG + lane_base + (uint32_t)s0, gv);
                    float bt[BC];
#pragma unroll
                    for (int j = 0; j < BC; j += 4) *reinterpret_cast<float4*>(&bt[j]) = *reinterpret_cast<const float4*>(&s_beta[s0 + j]);
                    const bool full = s0 + BC - 1 <= t0 + q * 32;  // no masked column in this warp
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < BC; j += 2) {
                        float v0 = ex2(alpha + bt[j]) * __uint_as_float(gv[j]);
                        float v1 = ex2(alpha + bt[j + 1]) * __uint_as_float(gv[j + 1]);
                        if (!full) {
                            v0 = s0 + j <= t ? v0 : 0.0f;
                            v1 = s0 + j + 1 <= t ? v1 : 0.0f;
                        }
                        split2(v0, v1, ph[j / 2], pl[j / 2]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < BC / 2; ++j) ph[j] = pl[j] = 0u;
                }
                const int sl = s0 - KPC * kp;
#pragma unroll
                for (int j = 0; j < BC / 8; ++j) {
                    st_shared_v4(mh + tc::off_kmajor(r, sl + 8 * j, KPC), ph[4 * j], ph[4 * j + 1], ph[4 * j + 2], ph[4 * j + 3]);
                    st_shared_v4(ml + tc::off_kmajor(r, sl + 8 * j, KPC), pl[4 * j], pl[4 * j + 1], pl[4 * j + 2], pl[4 * j + 3]);
                }
            }
            // XS: this head's x planes (copied in while the part was built) before its MMAs
            if (XS && kp == 0) asm volatile("cp.async.wait_group 0;\n" ::);
            tc::fence_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            if (tid == 0) {
                unsigned char* part = sM + (ncommit & 1) * 2 * Cfg::kMPart;
                const uint32_t tYd = tmem + 256 + 128 * (hi & 1), tYo = tYd + 64;
                constexpr uint32_t id_diag = tc::idesc_bf16(128, kP, 0, 1);
                const uint64_t dmh = tc::desc_kmajor(tc::smem_u32(part), KPC, 0);
                const uint64_t dml = tc::desc_kmajor(tc::smem_u32(part + Cfg::kMPart), KPC, 0);
                // x_h descriptor at this part's first k-step
                const uint64_t dx = tc::desc_mnmajor(tc::smem_u32(x_hi_tile(hi)), kP, KPC / 16 * kp);
#pragma unroll
                for (int ks = 0; ks < KPC / 16; ++ks)
                    tc::mma_bf16(tYd, dmh + ks * tc::kstep_kmajor(), dx + ks * tc::kstep_mnmajor(kP), id_diag,
                                 (kp > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < KPC / 16; ++ks)
                    tc::mma_bf16(tYd, dml + ks * tc::kstep_kmajor(), dx + ks * tc::kstep_mnmajor(kP), id_diag, 1);
                if (XS) {
                    const uint64_t dxl = tc::desc_mnmajor(tc::smem_u32(x_lo_tile(hi)), kP, KPC / 16 * kp);
#pragma unroll
                    for (int ks = 0; ks < KPC / 16; ++ks)
                        tc::mma_bf16(tYd, dmh + ks * tc::kstep_kmajor(), dxl + ks * tc::kstep_mnmajor(kP), id_diag, 1);
                }
                if (kp == 0) {
                    constexpr uint32_t id_off = tc::idesc_bf16(128, kP, 0, 0);
                    const uint64_t dc = tc::desc_kmajor(tc::smem_u32(sC), N, 0);
                    const unsigned char* hset = sH + (Cfg::kHBufs == 2 ? (hi & 1) : 0) * 2 * Cfg::kH;
                    const uint64_t dhh = tc::desc_kmajor(tc::smem_u32(hset), N, 0);
                    const uint64_t dhl = tc::desc_kmajor(tc::smem_u32(hset + Cfg::kH), N, 0);
#pragma unroll
                    for (int ks = 0; ks < N / 16; ++ks)
                        tc::mma_bf16(tYo, dc + ks * tc::kstep_kmajor(), dhh + ks * tc::kstep_kmajor(), id_off, ks > 0);
#pragma unroll
                    for (int ks = 0; ks < N / 16; ++ks)
                        tc::mma_bf16(tYo, dc + ks * tc::kstep_kmajor(), dhl + ks * tc::kstep_kmajor(), id_off, 1);
                }
                tc::mma_commit(&s_mbar[ncommit & 1]);
            }
            ++ncommit;
            // the previous head's epilogue, once this head's first MMAs are queued; then the
            // previous head's x_h buffer takes the next head's x_h
            if (kp == 0) {
                if (hi > 0) {
                    wait_commit(last_commit_prev);
                    finish(h - 1, (hi - 1) & 1, alpha_prev);
                    tc::fence_before_sync();
                }
                if (hi + 1 < heads_per_cta) {
                    __syncthreads();  // every thread is done reading the buffer in finish
                    if (!xser) load_x(a.x, h + 1, x_hi_tile(hi + 1));
                    if (XS && !xser) load_x(a.x_lo, h + 1, x_lo_tile(hi + 1));
                    // two h tile sets: the previous head's (its MMAs are done) takes the next
                    if (Cfg::kHBufs == 2) load_h(h + 1, (hi + 1) & 1);
                }
            }
            // serial XS: both x buffers are free once this head's last MMAs are done
            if (xser && kp == nparts - 1 && hi + 1 < heads_per_cta) {
                wait_commit(ncommit - 1);
                load_x(a.x, h + 1, x_hi_tile(hi + 1));
                load_x(a.x_lo, h + 1, x_lo_tile(hi + 1));
            }
        }
        last_commit_prev = ncommit - 1;
        alpha_prev = alpha;
    }
    if (ok && heads_per_cta > 0) {
        wait_commit(last_commit_prev);
        finish(hbeg + heads_per_cta - 1, (heads_per_cta - 1) & 1, alpha_prev);
    }
    if (!ok && tid == 0) report_timeout();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ---- host side -----------------------------------------------------------------

bool ssd_tc_supported(const ScanArgs& a, int64_t Q) {
    const int64_t hpg = a.nheads / a.ngroups;
    return a.dtype == 1 && a.headdim == kP && a.dstate % 16 == 0 && a.dstate >= 32 && a.dstate <= 256 &&
           (Q == 128 || Q == 256) && hpg % 2 == 0 && (a.dstate == 32 || a.dstate == 64 || a.dstate == 128 ||
                                                    a.dstate == 256);
}

namespace {

// Heads per CTA: the largest of 8, 4, 2 that divides the heads of a group.
int heads_per_cta(const SsdTcArgs& s, int max_heads) {
    const int hpg = (int)(s.H / s.G);
    for (int cand : {8, 4, 2, 1})
        if (cand <= max_heads && hpg % cand == 0) return cand;
    return 1;
}

template <int N, bool XS>
cudaError_t launch_state(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    using Cfg = StateTcCfg<N, XS>;
    const size_t smem = Cfg::kSmem;
    cudaError_t e = cudaFuncSetAttribute(ssd_state_tc<N, XS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int hpc = heads_per_cta(s, Cfg::kMaxHeads);  // even: heads per group are even here
    cudaEvent_t t0 = timing_begin(stream);
    ssd_state_tc<N, XS><<<dim3((unsigned)s.nchunks, (unsigned)(s.H / hpc), (unsigned)batch), Cfg::NT, smem, stream>>>(s, hpc);
    note_launch("ssd_state_tc", stream, t0);
    return cudaGetLastError();
}

template <int N, bool GATE, bool XS>
cudaError_t launch_scan(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    // at least 116 KB so that one CTA (holding all 512 TMEM columns) runs per SM
    const size_t smem = std::max<size_t>(ScanTcCfg<N>::kSmem, 116 * 1024);
    auto kern = ssd_scan_tc<N, GATE, XS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int hpc = heads_per_cta(s, 8);  // G = C B^T is shared by the CTA's heads
    const dim3 grid((unsigned)(s.nchunks * (s.Q / 128)), (unsigned)(s.H / hpc), (unsigned)batch);
    cudaEvent_t t0 = timing_begin(stream);
    kern<<<grid, kScanThreads, smem, stream>>>(s, hpc);
    note_launch("ssd_scan_tc", stream, t0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t device_status_take(int* status, bool clear, cudaStream_t stream) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_device_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (clear && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return e;
    }
    *status = v;
    return cudaSuccess;
}

cudaError_t bounded_wait_selftest_launch(uint32_t max_checks, cudaStream_t stream) {
    cudaEvent_t t0 = timing_begin(stream);
    bounded_wait_selftest<<<1, 32, 0, stream>>>(max_checks);
    note_launch("bounded_wait_selftest", stream, t0);
    return cudaGetLastError();
}

cudaError_t ssd_tc_chunk_state(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    if (s.x_lo) {
        switch (s.N) {
            case 32: return launch_state<32, true>(s, batch, stream);
            case 64: return launch_state<64, true>(s, batch, stream);
            case 128: return launch_state<128, true>(s, batch, stream);
            default: return launch_state<256, true>(s, batch, stream);
        }
    }
    switch (s.N) {
        case 32: return launch_state<32, false>(s, batch, stream);
        case 64: return launch_state<64, false>(s, batch, stream);
        case 128: return launch_state<128, false>(s, batch, stream);
        default: return launch_state<256, false>(s, batch, stream);
    }
}

cudaError_t ssd_tc_chunk_scan(const SsdTcArgs& s, int64_t batch, bool gate, cudaStream_t stream) {
    if (s.x_lo) {
        switch (s.N) {
            case 32: return gate ? launch_scan<32, true, true>(s, batch, stream) : launch_scan<32, false, true>(s, batch, stream);
            case 64: return gate ? launch_scan<64, true, true>(s, batch, stream) : launch_scan<64, false, true>(s, batch, stream);
            case 128: return gate ? launch_scan<128, true, true>(s, batch, stream) : launch_scan<128, false, true>(s, batch, stream);
            default: return gate ? launch_scan<256, true, true>(s, batch, stream) : launch_scan<256, false, true>(s, batch, stream);
        }
    }
    switch (s.N) {
        case 32: return gate ? launch_scan<32, true, false>(s, batch, stream) : launch_scan<32, false, false>(s, batch, stream);
        case 64: return gate ? launch_scan<64, true, false>(s, batch, stream) : launch_scan<64, false, false>(s, batch, stream);
        case 128: return gate ? launch_scan<128, true, false>(s, batch, stream) : launch_scan<128, false, false>(s, batch, stream);
        default: return gate ? launch_scan<256, true, false>(s, batch, stream) : launch_scan<256, false, false>(s, batch, stream);
    }
}

}  // namespace ssm
