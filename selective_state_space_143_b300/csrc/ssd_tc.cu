// Mamba-2 / SSD chunk-state kernel on the B300 tensor cores (tcgen05, TMEM accumulators),
// the per-device status word of the bounded device-side waits, and the tensor-core shape
// check.
//
// Same chunk algebra as ssd_scan.cu ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里",
// 第二步 and 关键技术点 1-3: y = (L o M) x, dense diagonal blocks, low-rank off-diagonal
// blocks through the carried state), the chunk-state product issued as tcgen05.mma (bf16
// operands in shared memory, fp32 accumulators in tensor memory):
//
//   ssd_state_tc : S_c^T for up to 8 heads of a chunk, two at a time:
//                  D[(head, p), n] = sum_s Xd[s, (head, p)] B[s, n]
//                  with Xd[s, :] = exp(s_last - s_s) Delta_s x_s  (M = 128, N = dstate, K = Q)
// The carry h_c = exp(s_last) h_{c-1} + S_c runs next (ssd_state_pass_split in
// ssd_scan.cu): ssd_state_tc stores S_c in a split-ready layout and the carry writes
// h_{c-1} back as the bf16 hi/lo tiles that the scan kernel (ssd_scan_tc.cu) copies
// into shared memory.
//
// Shapes taken here: bf16, headdim 64, dstate 64, 128 or 256, chunk 128 or 256, an even
// number of heads per group.  Other shapes use the CUDA-core kernels.
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
constexpr int kStatusTimeout = 8;

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* gmem, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr), "l"(gmem), "r"(n));
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

// ---- host side -----------------------------------------------------------------

bool ssd_tc_supported(const ScanArgs& a, int64_t Q) {
    const int64_t hpg = a.nheads / a.ngroups;
    // the scan kernel's tensor maps take 32-bit coordinates; its C and B tiles are rows of
    // 64 elements (dstate a multiple of 64)
    return a.dtype == 1 && a.headdim == kP && a.seqlen < (int64_t(1) << 31) &&
           (a.dstate == 64 || a.dstate == 128 || a.dstate == 256) && (Q == 128 || Q == 256) && hpg % 2 == 0;
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

cudaError_t device_status_address(int** p) {
    constexpr int kMaxDev = 64;
    static int* cache[kMaxDev] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if (!cache[dev]) {
        void* a = nullptr;
        e = cudaGetSymbolAddress(&a, g_device_status);
        if (e != cudaSuccess) return e;
        cache[dev] = static_cast<int*>(a);
    }
    *p = cache[dev];
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
            case 64: return launch_state<64, true>(s, batch, stream);
            case 128: return launch_state<128, true>(s, batch, stream);
            default: return launch_state<256, true>(s, batch, stream);
        }
    }
    switch (s.N) {
        case 64: return launch_state<64, false>(s, batch, stream);
        case 128: return launch_state<128, false>(s, batch, stream);
        default: return launch_state<256, false>(s, batch, stream);
    }
}

}  // namespace ssm
