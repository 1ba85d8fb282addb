// Mamba-2 / SSD chunk kernels on the B300 tensor cores (tcgen05, TMEM accumulators).
//
// Same chunk algebra as ssd_scan.cu ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里",
// 第二步 and 关键技术点 1-3: y = (L o M) x, dense diagonal blocks, low-rank off-diagonal
// blocks through the carried state), with the three matrix products of a chunk issued
// as tcgen05.mma (bf16 operands in shared memory, fp32 accumulators in tensor memory):
//
//   ssd_state_tc : S_c^T for two heads at once:  D[(head, p), n] = sum_s Xd[s, (head, p)] B[s, n]
//                  with Xd[s, :] = exp(s_last - s_s) Delta_s x_s  (M = 128, N = dstate, K = Q)
//   ssd_scan_tc  : per (chunk, 128-row half): G = C_rows B^T once (M = 128, N = rows up to
//                  the half's end, K = dstate), then per head
//                    M'[t, s] = G[t, s] exp(s_t - s_s) Delta_s  (s <= t, else 0) -> bf16 smem
//                    Y_diag   = M' X_h                            (M = 128, N = 64, K = s)
//                    Y_off    = C_rows h_{c-1}^T                  (M = 128, N = 64, K = dstate)
//                    out      = (Y_diag + exp(s_t) Y_off + D x) SiLU(z)
// The carry h_c = exp(s_last) h_{c-1} + S_c runs in between (ssd_state_pass).
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
constexpr int kThreads = 256;  // 8 warps: warp w reads TMEM lanes 32*(w%4).., column half w/4
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

// Inclusive prefix sum of v over the block (one value per thread); s_warp: one float per warp.
__device__ __forceinline__ float block_incl_scan(float v, float* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    __syncthreads();
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    float add = 0.0f;
    for (int w = 0; w < warp; ++w) add += s_warp[w];
    return v + add;
}

// Delta_s and the inclusive cumulative sum of Delta_s A_h for s in [0, Q) of chunk c
// (one row per thread; Q <= 256).  Rows past len get Delta 0.
__device__ void delta_cumsum(const SsdTcArgs& a, int64_t b, int64_t h, int64_t c, int len,
                             float* s_dl, float* s_cum, float* s_warp) {
    const int s = threadIdx.x;
    float d = 0.0f;
    if (s < len) d = softplus(__bfloat162float(a.dt[(b * a.T + c * a.Q + s) * a.H + h]) + (a.dt_bias ? a.dt_bias[h] : 0.0f));
    const float incl = block_incl_scan(d * a.A[h], s_warp);
    if (s < a.Q) {
        s_dl[s] = d;
        s_cum[s] = incl;
    }
    __syncthreads();
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

__device__ __forceinline__ void report_timeout(int* status) {
    if (status) atomicExch(status, kStatusTimeout);
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

// grid (nchunks, H/2, b); 128 threads.
// dynamic smem: Xd hi (128 x Q) | Xd lo (128 x Q) | B column block (Q x NB), NB = min(N, 128)
template <int N>
__global__ void __launch_bounds__(kThreads) ssd_state_tc(const SsdTcArgs a) {
    constexpr int NB = N < 128 ? N : 128;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ float s_dl[2][256], s_cum[2][256], s_w[2][256], s_warp[8];
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_mbar;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t c = blockIdx.x, h0 = 2 * (int64_t)blockIdx.y, b = blockIdx.z;
    const int Q = (int)a.Q;
    const int len = (int)min((int64_t)Q, a.T - c * a.Q);
    const int64_t g = h0 / (a.H / a.G);
    unsigned char* sXh = smem;                         // MN-major A: M = (head, p), K = s
    unsigned char* sXl = smem + (size_t)Q * 128 * 2;
    unsigned char* sB = smem + (size_t)Q * 128 * 4;    // MN-major B: K = s, N = NB columns

    auto load_B = [&](int nb) {
        const uint32_t base = tc::smem_u32(sB);
        for (int i = tid; i < Q * (NB / 8); i += kThreads) {
            int s, nc;
            mnmajor_item(i, NB / 8, s, nc);
            const int n0 = nc * 8;
            const bool ok = s < len;
            const __nv_bfloat16* src = a.B + (ok ? (((b * a.T + c * a.Q + s) * a.G + g) * a.N + nb * NB + n0) : 0);
            cp_async16(base + tc::off_mnmajor(n0, s, NB), src, ok);
        }
    };
    load_B(0);
    // Delta, cumulative sums and the chunk-end weights for both heads
    for (int hl = 0; hl < 2; ++hl) {
        delta_cumsum(a, b, h0 + hl, c, len, s_dl[hl], s_cum[hl], s_warp);
        const float last = s_cum[hl][len - 1];
        for (int s = tid; s < Q; s += kThreads) s_w[hl][s] = s < len ? __expf(last - s_cum[hl][s]) * s_dl[hl][s] : 0.0f;
        for (int s = tid; s < Q; s += kThreads) {
            const int64_t o = ((b * a.H + h0 + hl) * a.nchunks + c) * a.Q + s;
            a.dl[o] = s_dl[hl][s];
            a.cum[o] = s_cum[hl][s];
        }
    }
    __syncthreads();
    // Xd = w_s x_s for both heads, split hi/lo, MN-major (8 consecutive p at one s)
    {
        const uint32_t bh = tc::smem_u32(sXh), bl = tc::smem_u32(sXl);
#pragma unroll 4
        for (int i = tid; i < Q * 16; i += kThreads) {
            int s, mc;
            mnmajor_item(i, 16, s, mc);
            const int m0 = mc * 8;  // m = head_local * 64 + p
            const int hl = m0 / kP, p0 = m0 % kP;
            uint32_t hi[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
            if (s < len) {
                const uint4 raw = *reinterpret_cast<const uint4*>(a.x + ((b * a.T + c * a.Q + s) * a.H + h0 + hl) * kP + p0);
                const float w = s_w[hl][s];
                const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __bfloat1622float2(r2[k]);
                    split2(f.x * w, f.y * w, hi[k], lo[k]);
                }
            }
            const uint32_t off = tc::off_mnmajor(m0, s, 128);
            st_shared_v4(bh + off, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(bl + off, lo[0], lo[1], lo[2], lo[3]);
        }
    }
    constexpr uint32_t kCols = N < 32 ? 32 : N;
    if (warp == 0) tc::tmem_alloc(&s_tmem, kCols);
    if (tid == 0) {
        tc::mbar_init(&s_mbar, 1);
        tc::mbar_fence_init();
    }
    bool ok = true;
    uint32_t phase = 0;
    uint32_t tmem = 0;
    for (int nb = 0; nb < N / NB; ++nb) {
        if (nb > 0) {
            // the previous column block's MMAs must be done with sB before it is reloaded
            ok = tc::mbar_wait(&s_mbar, phase) && ok;
            phase ^= 1;
            tc::fence_after_sync();
            __syncthreads();
            load_B(nb);
        }
        cp_async_commit_wait_all();
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        tmem = s_tmem;
        // D[(head, p), nb*NB + n] = sum_s (Xd_hi + Xd_lo)[s, (head, p)] B[s, nb*NB + n]
        if (tid == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16(128, NB, 1, 1);
            const uint32_t xh = tc::smem_u32(sXh), xl = tc::smem_u32(sXl), ba = tc::smem_u32(sB);
            const uint32_t d = tmem + (uint32_t)(nb * NB);
            for (int ks = 0; ks < Q / 16; ++ks)
                tc::mma_bf16(d, tc::desc_mnmajor(xh, 128, ks), tc::desc_mnmajor(ba, NB, ks), idesc, ks > 0);
            for (int ks = 0; ks < Q / 16; ++ks)
                tc::mma_bf16(d, tc::desc_mnmajor(xl, 128, ks), tc::desc_mnmajor(ba, NB, ks), idesc, 1);
            tc::mma_commit(&s_mbar);
        }
    }
    ok = tc::mbar_wait(&s_mbar, phase) && ok;
    tc::fence_after_sync();
    if (ok) {
        // row m = lane: (head h0 + m/64, p = m%64) -> states[b, c, h, p, :]; warps 4-7 take
        // the upper half of the columns
        const int q = warp & 3;
        const int m = q * 32 + (tid & 31);
        float* dst = a.states + (((b * a.nchunks + c) * a.H + h0 + m / kP) * kP + (m % kP)) * a.N;
        constexpr int NH = N / 2 < 16 ? 16 : N / 2;
#pragma unroll 1
        for (int n0 = (warp >> 2) * NH; n0 < N && n0 < ((warp >> 2) + 1) * NH; n0 += 16) {
            float v[16];
            tc::tmem_ld16(tc::taddr(tmem, q * 32, n0), v);
#pragma unroll
            for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4*>(dst + n0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    } else if (tid == 0) {
        report_timeout(a.status);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

// grid (nchunks * Q/128, H / HG, b); 128 threads.  Rows [128*rh, 128*rh + 128) of chunk c.
// dynamic smem: C rows (128 x N, K-major) | region:
//   phase 1: B rows [0, SW) (K-major)
//   phase 2: M' hi | M' lo (128 x 128 each, one 128-column K-part at a time) | x_h (SW x 64)
//            | h hi | h lo (64 x N each)
template <int N, bool GATE>
__global__ void __launch_bounds__(kThreads) ssd_scan_tc(const SsdTcArgs a, int heads_per_cta) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ float s_dl[256], s_cum[256];
    __shared__ uint32_t s_tmem;
    __shared__ __align__(8) uint64_t s_mbar;
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
    const int64_t hbeg = (int64_t)blockIdx.y * heads_per_cta;
    const int64_t g = hbeg / (a.H / a.G);

    unsigned char* sC = smem;                        // K-major: M = t (128), K = n
    unsigned char* region = smem + 128 * N * 2;
    unsigned char* sB = region;                      // K-major: N_mma = s (SW), K = n
    unsigned char* sMh = region;                     // K-major: M = t, K = 128 columns of s
    unsigned char* sMl = region + 128 * 128 * 2;
    unsigned char* sXh = region + 128 * 128 * 4;     // MN-major: K = s (SW), N_mma = p (64)
    unsigned char* sHh = sXh + 256 * kP * 2;         // K-major: N_mma = p (64), K = n
    unsigned char* sHl = sHh + kP * N * 2;

    // phase 1 loads: C rows of this half and B rows [0, SW)
    {
        const uint32_t cb = tc::smem_u32(sC), bb = tc::smem_u32(sB);
        for (int i = tid; i < 128 * (N / 8); i += kThreads) {
            int r, nc;
            kmajor_item(i, N / 8, r, nc);
            const int n0 = nc * 8;
            const int s = t0 + r;
            const bool ok = s < len;
            const __nv_bfloat16* src = a.C + (ok ? (((b * a.T + c * a.Q + s) * a.G + g) * a.N + n0) : 0);
            cp_async16(cb + tc::off_kmajor(r, n0, N), src, ok);
        }
        for (int i = tid; i < SW * (N / 8); i += kThreads) {
            int s, nc;
            kmajor_item(i, N / 8, s, nc);
            const int n0 = nc * 8;
            const bool ok = s < len;
            const __nv_bfloat16* src = a.B + (ok ? (((b * a.T + c * a.Q + s) * a.G + g) * a.N + n0) : 0);
            cp_async16(bb + tc::off_kmajor(s, n0, N), src, ok);
        }
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 512);
    if (tid == 0) {
        tc::mbar_init(&s_mbar, 1);
        tc::mbar_fence_init();
    }
    cp_async_commit_wait_all();
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t tG = tmem, tYd = tmem + 256, tYo = tmem + 320;
    uint32_t phase = 0;
    bool ok = true;

    // G = C_rows B^T (raw bf16 operands: exact products, fp32 accumulation)
    if (tid == 0) {
        const uint32_t idesc = tc::idesc_bf16(128, SW, 0, 0);
        const uint32_t ca = tc::smem_u32(sC), ba = tc::smem_u32(sB);
        for (int ks = 0; ks < N / 16; ++ks)
            tc::mma_bf16(tG, tc::desc_kmajor(ca, N, ks), tc::desc_kmajor(ba, N, ks), idesc, ks > 0);
        tc::mma_commit(&s_mbar);
    }
    ok = tc::mbar_wait(&s_mbar, phase);
    phase ^= 1;
    tc::fence_after_sync();

    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int chalf = warp >> 2;             // warps 4-7 take the upper half of the columns
    const int r = q * 32 + (tid & 31);       // my row (TMEM lane) within the half
    const int t = t0 + r;                    // row within the chunk
    const bool row_ok = t < len;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int t_warp_max = t0 + q * 32 + 31;  // tcgen05.ld is warp-collective

    for (int hi = 0; hi < heads_per_cta && ok; ++hi) {
        const int64_t h = hbeg + hi;
        __syncthreads();  // every thread is done with the previous head's epilogue
        for (int s = tid; s < Q; s += kThreads) {
            const int64_t o = ((b * a.H + h) * a.nchunks + c) * a.Q + s;
            s_dl[s] = a.dl[o];
            s_cum[s] = a.cum[o];
        }
        __syncthreads();
        // x_h rows [0, SW): raw bf16, MN-major (8 consecutive p at one s)
        {
            const uint32_t xb = tc::smem_u32(sXh);
            for (int i = tid; i < SW * 8; i += kThreads) {
                int s, pc;
                mnmajor_item(i, 8, s, pc);
                const int p0 = pc * 8;
                const bool okr = s < len;
                const __nv_bfloat16* src = a.x + (okr ? (((b * a.T + c * a.Q + s) * a.H + h) * kP + p0) : 0);
                cp_async16(xb + tc::off_mnmajor(p0, s, kP), src, okr);
            }
        }
        // h_{c-1} of this head: fp32 -> bf16 hi/lo, K-major (8 consecutive n at one p)
        {
            const uint32_t hb = tc::smem_u32(sHh), lb = tc::smem_u32(sHl);
            const float* hs = a.states + ((b * a.nchunks + c) * a.H + h) * (int64_t)kP * a.N;
#pragma unroll 2
            for (int i = tid; i < kP * (N / 8); i += kThreads) {
                int p, nc;
                kmajor_item(i, N / 8, p, nc);
                const int n0 = nc * 8;
                const float4 v0 = *reinterpret_cast<const float4*>(hs + (int64_t)p * a.N + n0);
                const float4 v1 = *reinterpret_cast<const float4*>(hs + (int64_t)p * a.N + n0 + 4);
                uint32_t qh[4], ql[4];
                split2(v0.x, v0.y, qh[0], ql[0]);
                split2(v0.z, v0.w, qh[1], ql[1]);
                split2(v1.x, v1.y, qh[2], ql[2]);
                split2(v1.z, v1.w, qh[3], ql[3]);
                const uint32_t off = tc::off_kmajor(p, n0, N);
                st_shared_v4(hb + off, qh[0], qh[1], qh[2], qh[3]);
                st_shared_v4(lb + off, ql[0], ql[1], ql[2], ql[3]);
            }
        }
        const float cum_t = s_cum[min(t, Q - 1)];
        // Y_diag accumulates over K-parts of 128 columns of s; Y_off goes with part 0
        for (int kp = 0; kp < SW / 128; ++kp) {
            if (kp > 0) {
                // the previous part's MMAs must be done with the M' buffers
                ok = tc::mbar_wait(&s_mbar, phase) && ok;
                phase ^= 1;
                tc::fence_after_sync();
                __syncthreads();
            }
            // M'[t, s] = G[t, s] exp(cum_t - cum_s) Delta_s for s <= t, hi/lo, K-major
            {
                const uint32_t mh = tc::smem_u32(sMh), ml = tc::smem_u32(sMl);
                for (int s0 = 128 * kp + 64 * chalf; s0 < 128 * kp + 64 * chalf + 64; s0 += 16) {
                    uint32_t ph[8], pl[8];
                    if (s0 <= t_warp_max) {
                        float gv[16];
                        tc::tmem_ld16(tG + lane_base + (uint32_t)s0, gv);
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            const int s = s0 + j;
                            const float v0 = s <= t ? gv[j] * __expf(cum_t - s_cum[s]) * s_dl[s] : 0.0f;
                            const float v1 = s + 1 <= t ? gv[j + 1] * __expf(cum_t - s_cum[s + 1]) * s_dl[s + 1] : 0.0f;
                            split2(v0, v1, ph[j / 2], pl[j / 2]);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) ph[j] = pl[j] = 0u;
                    }
                    const int sl = s0 - 128 * kp;
                    st_shared_v4(mh + tc::off_kmajor(r, sl, 128), ph[0], ph[1], ph[2], ph[3]);
                    st_shared_v4(mh + tc::off_kmajor(r, sl + 8, 128), ph[4], ph[5], ph[6], ph[7]);
                    st_shared_v4(ml + tc::off_kmajor(r, sl, 128), pl[0], pl[1], pl[2], pl[3]);
                    st_shared_v4(ml + tc::off_kmajor(r, sl + 8, 128), pl[4], pl[5], pl[6], pl[7]);
                }
            }
            cp_async_commit_wait_all();
            tc::fence_async_smem();
            tc::fence_before_sync();
            __syncthreads();
            tc::fence_after_sync();
            if (tid == 0) {
                const uint32_t mh = tc::smem_u32(sMh), ml = tc::smem_u32(sMl), xa = tc::smem_u32(sXh);
                constexpr uint32_t id_diag = tc::idesc_bf16(128, kP, 0, 1);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16(tYd, tc::desc_kmajor(mh, 128, ks), tc::desc_mnmajor(xa, kP, 8 * kp + ks), id_diag,
                                 (kp > 0 || ks > 0) ? 1u : 0u);
                for (int ks = 0; ks < 8; ++ks)
                    tc::mma_bf16(tYd, tc::desc_kmajor(ml, 128, ks), tc::desc_mnmajor(xa, kP, 8 * kp + ks), id_diag, 1);
                if (kp == 0) {
                    const uint32_t ca = tc::smem_u32(sC), hh = tc::smem_u32(sHh), hl = tc::smem_u32(sHl);
                    constexpr uint32_t id_off = tc::idesc_bf16(128, kP, 0, 0);
                    for (int ks = 0; ks < N / 16; ++ks)
                        tc::mma_bf16(tYo, tc::desc_kmajor(ca, N, ks), tc::desc_kmajor(hh, N, ks), id_off, ks > 0);
                    for (int ks = 0; ks < N / 16; ++ks)
                        tc::mma_bf16(tYo, tc::desc_kmajor(ca, N, ks), tc::desc_kmajor(hl, N, ks), id_off, 1);
                }
                tc::mma_commit(&s_mbar);
            }
        }
        ok = tc::mbar_wait(&s_mbar, phase) && ok;
        phase ^= 1;
        tc::fence_after_sync();
        if (!ok) break;
        // epilogue: y = Y_diag + exp(cum_t) Y_off + D x, gate, store 64 bf16
        {
            const float et = __expf(cum_t);
            const float Dh = a.D ? a.D[h] : 0.0f;
            const int64_t row = ((b * a.T + c * a.Q + t) * a.H + h) * kP;
#pragma unroll 1
            for (int p0 = 32 * chalf; p0 < 32 * chalf + 32; p0 += 16) {
                float yd[16], yo[16];
                tc::tmem_ld16(tYd + lane_base + (uint32_t)p0, yd);
                tc::tmem_ld16(tYo + lane_base + (uint32_t)p0, yo);
                if (row_ok) {
                    uint32_t pk[8];
#pragma unroll
                    for (int j = 0; j < 16; j += 8) {
                        const uint4 xr = *reinterpret_cast<const uint4*>(sXh + tc::off_mnmajor(p0 + j, t, kP));
                        const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&xr);
                        uint4 zr = make_uint4(0, 0, 0, 0);
                        if (GATE) zr = *reinterpret_cast<const uint4*>(a.z + row + p0 + j);
                        const __nv_bfloat162* z2 = reinterpret_cast<const __nv_bfloat162*>(&zr);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 xv = __bfloat1622float2(x2[k]);
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
        }
    }
    if (!ok && tid == 0) report_timeout(a.status);
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

template <int N>
cudaError_t launch_state(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    constexpr int NB = N < 128 ? N : 128;
    const size_t smem = (size_t)s.Q * 128 * 4 + (size_t)s.Q * NB * 2;
    cudaError_t e = cudaFuncSetAttribute(ssd_state_tc<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ssd_state_tc<N><<<dim3((unsigned)s.nchunks, (unsigned)(s.H / 2), (unsigned)batch), kThreads, smem, stream>>>(s);
    note_launches(1);
    return cudaGetLastError();
}

template <int N, bool GATE>
cudaError_t launch_scan(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    const size_t phase1 = (size_t)256 * N * 2;  // B rows (up to 256)
    const size_t phase2 = (size_t)128 * 128 * 4 + (size_t)256 * kP * 2 + (size_t)kP * N * 4;
    // at least 116 KB so that one CTA (holding all 512 TMEM columns) runs per SM
    const size_t smem = std::max<size_t>((size_t)128 * N * 2 + std::max(phase1, phase2), 116 * 1024);
    auto kern = ssd_scan_tc<N, GATE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int hpg = (int)(s.H / s.G);
    int hpc = 1;  // heads per CTA: G = C B^T is shared by them (a divisor of heads per group)
    for (int cand : {8, 4, 2, 1})
        if (hpg % cand == 0) {
            hpc = cand;
            break;
        }
    const dim3 grid((unsigned)(s.nchunks * (s.Q / 128)), (unsigned)(s.H / hpc), (unsigned)batch);
    kern<<<grid, kThreads, smem, stream>>>(s, hpc);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t ssd_tc_chunk_state(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    switch (s.N) {
        case 32: return launch_state<32>(s, batch, stream);
        case 64: return launch_state<64>(s, batch, stream);
        case 128: return launch_state<128>(s, batch, stream);
        default: return launch_state<256>(s, batch, stream);
    }
}

cudaError_t ssd_tc_chunk_scan(const SsdTcArgs& s, int64_t batch, bool gate, cudaStream_t stream) {
    switch (s.N) {
        case 32: return gate ? launch_scan<32, true>(s, batch, stream) : launch_scan<32, false>(s, batch, stream);
        case 64: return gate ? launch_scan<64, true>(s, batch, stream) : launch_scan<64, false>(s, batch, stream);
        case 128: return gate ? launch_scan<128, true>(s, batch, stream) : launch_scan<128, false>(s, batch, stream);
        default: return gate ? launch_scan<256, true>(s, batch, stream) : launch_scan<256, false>(s, batch, stream);
    }
}

}  // namespace ssm
