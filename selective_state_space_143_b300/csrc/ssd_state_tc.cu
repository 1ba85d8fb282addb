// SSD chunk states on the B300 tensor cores ("Mamba-2：把状态空间模型和 Attention 统一到一个
// 数学框架里", 第二步 and 关键技术点 1: the off-diagonal blocks of y = (L o M) x are low rank
// and pass through the state carried between chunks).  For every chunk c and head h,
// with cum_s the in-chunk cumulative sum of Delta_s A_h:
//   S_c[p, n] = sum_s w_s x_s[p] B_s[n],   w_s = exp(cum_last - cum_s) Delta_s
// computed as D[(head, p), n] = Xw^T B with two heads (128 accumulator rows) per MMA
// tile: M = 128, N = dstate per MMA, K = rows s.  The weighted
// operand Xw is built by threads and split into bf16 hi + lo halves, both multiplied
// against the exact bf16 B, so it keeps ~16 significant bits.
//
// One CTA per (chunk, group of heads), warp-specialised: a TMA warp (the chunk's B rows
// once, then the heads' x rows in K-parts through a 3-deep ring, all in the 128-byte
// swizzle layout), an MMA warp, and 8 compute warps that first form Delta, the
// cumulative sums (written out for the scan and carry kernels) and the weights w, then
// build the Xw parts (double buffered) and store each head pair's states from one of two
// TMEM accumulators while the next pair's MMAs run.  The states go out in the layout the
// carry pass (ssd_state_pass_split) turns in place into the scan kernel's bf16 hi/lo
// tiles: the 8 values of (p, n..n+7) as two float4 at the byte offsets of their hi and
// lo halves in the scan kernel's K-major h tile.
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

constexpr int kP = 64;
constexpr int kStatusTimeout = 8;
constexpr int kCompute = 8;                 // compute warps
constexpr int kMma = 8, kLoad = 9;          // MMA and TMA warps
constexpr int kCta = 32 * 10;
constexpr int kMaxHeads = 8;
constexpr int kXStagesMax = 5;

template <int N, bool XS>
struct StateCfg {
    static constexpr int KS = (N > 128 || XS) ? 32 : 64;    // rows s per K-part
    static constexpr int PL = XS ? 2 : 1;                    // x planes
    static constexpr uint32_t kB = 256u * N * 2;             // B rows [0, Q): [n/64][s][64] swizzled
    static constexpr uint32_t kXHead = (uint32_t)KS * 128;   // one head's x rows of a part (one plane)
    static constexpr uint32_t kXStage = 2 * PL * kXHead;     // two heads, every plane
    static constexpr uint32_t kXt = 128u * KS * 2;           // one Xw part, hi or lo
    static constexpr uint32_t kW = kMaxHeads * 256 * 4;      // weights w[head][s]
    // x stages in flight: 5 at dstate 256 with one x plane (c4 chunk states 433 -> 410 us
    // against 3), 3 otherwise (more measured slower at dstate 128: c3 154 -> 160 us)
    static constexpr int kXStages = N > 128 && PL == 1 ? 5 : 3;
    static constexpr uint32_t kSmem = kB + kXStages * kXStage + 4 * kXt + kW;
    static constexpr uint32_t kSmemTotal = kSmem + 512;      // + pipeline state
    static_assert(kSmemTotal <= 232448, "shared memory");
};

struct __align__(16) StateShared {
    uint64_t mb_b;              // B rows
    uint64_t x_full[kXStagesMax], x_empty[kXStagesMax];
    uint64_t xt_full[2], xt_empty[2];
    uint64_t acc_full[2], acc_empty[2];
    float warp_sum[kCompute][kMaxHeads];
    uint32_t tmem;
    volatile int abort;
};

__device__ __forceinline__ void wait_or_abort(StateShared& sh, uint64_t* mb, uint32_t phase) {
    if (sh.abort) return;
    if (!tc::mbar_wait(mb, phase)) sh.abort = 1;
}
__device__ __forceinline__ void arrive(uint64_t* mb) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(mb)) : "memory");
}
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ uint32_t bf16pair(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi), two values at a time.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    const float2 l = __ffma2_rn(hf, make_float2(-1.0f, -1.0f), make_float2(a, b));
    lo = bf16pair(l.x, l.y);
}

// grid (nchunks * H / hpc, batch); 10 warps.  Each CTA takes heads [hpc * block, +hpc)
// (hpc even, a divisor of the heads of a group) of one chunk.  At dstate 256, where a
// chunk's B rows are half as many bytes as a CTA's x rows, blockIdx.x = chunk * (H / hpc)
// + head block: the head blocks of a chunk run together and read its B rows once from
// DRAM, then from L2 (c4 434 us against 453 with chunks adjacent).  Below that, blockIdx.x
// = head block * nchunks + chunk (consecutive chunks of the same heads adjacent), which
// measured faster there (c3 152 us against 156).
//
// ADJ: the adjoint chunk states of the backward pass instead,
//   S^g_c[p, n] = sum_t exp(cum_t) dy_t[p] C_t[n]
// with tm_x / tm_xlo the hi / lo planes of dy, tm_b the C rows, and weights exp(cum_t)
// (the gradient carried into the chunk from its outputs); Delta and the cumulative sums
// are recomputed for the weights but not stored (the forward pass stored them).
template <int N, bool XS, bool ADJ>
__global__ void __launch_bounds__(kCta, 1)
    ssd_state_tc(const SsdTcArgs a, const int hpc, int* status, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_xlo, const __grid_constant__ CUtensorMap tm_b) {
    using Cfg = StateCfg<N, XS>;
    constexpr int KS = Cfg::KS, PL = Cfg::PL;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* sB = smem;                                    // [n/64][s 256][64] swizzled
    unsigned char* sXr = smem + Cfg::kB;                         // [stage][head 2][plane][s KS][64] swizzled
    constexpr int kXStages = Cfg::kXStages;
    unsigned char* sXt = sXr + kXStages * Cfg::kXStage;          // [buffer 2][hi, lo] MN-major A, no swizzle
    float* sW = reinterpret_cast<float*>(sXt + 4 * Cfg::kXt);    // [head][s]
    StateShared& sh = *reinterpret_cast<StateShared*>(smem + Cfg::kSmem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Q = (int)a.Q;
    const int nhb = (int)(a.H / hpc);
    constexpr bool kHeadsAdjacent = N > 128;
    const int64_t c = kHeadsAdjacent ? (int64_t)(blockIdx.x / nhb) : (int64_t)blockIdx.x % a.nchunks;
    const int hbeg = (int)(kHeadsAdjacent ? blockIdx.x % nhb : blockIdx.x / a.nchunks) * hpc;
    const int b = blockIdx.y;
    const int len = (int)min((int64_t)Q, a.T - c * a.Q);
    const int g = hbeg / (int)(a.H / a.G);
    const int row0 = (int)(c * a.Q);
    const int npairs = hpc / 2;
    const int nparts = Q / KS;

    if (tid == 0) {
        tc::mbar_init(&sh.mb_b, 1);
        for (int i = 0; i < kXStages; ++i) {
            tc::mbar_init(&sh.x_full[i], 1);
            tc::mbar_init(&sh.x_empty[i], kCompute);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sh.xt_full[i], kCompute);
            tc::mbar_init(&sh.xt_empty[i], 1);
            tc::mbar_init(&sh.acc_full[i], 1);
            tc::mbar_init(&sh.acc_empty[i], kCompute);
        }
        sh.abort = 0;
        tc::mbar_fence_init();
    }
    constexpr uint32_t kCols = 2 * N < 32 ? 32 : 2 * N;  // two accumulators
    if (warp == 0) tc::tmem_alloc(&sh.tmem, kCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh.tmem;

    if (warp == kLoad) {
        // ---- TMA: B rows once, then x rows of each pair's K-parts through the ring
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(&sh.mb_b, (uint32_t)Q * N * 2);
            for (int j = 0; j < N / 64; ++j)
                for (int rb = 0; rb < Q / 128; ++rb)
                    tc::tma_load_3d(sB + (j * 256 + rb * 128) * 128, &tm_b, g * N + 64 * j, row0 + 128 * rb, b, &sh.mb_b);
            uint32_t n = 0;
            for (int pr = 0; pr < npairs && !sh.abort; ++pr) {
                for (int kp = 0; kp < nparts; ++kp, ++n) {
                    const uint32_t st = n % kXStages, use = n / kXStages;
                    if (use > 0) wait_or_abort(sh, &sh.x_empty[st], (use - 1) & 1);
                    if (sh.abort) break;
                    tc::mbar_arrive_expect_tx(&sh.x_full[st], Cfg::kXStage);
                    unsigned char* dst = sXr + st * Cfg::kXStage;
                    for (int hh = 0; hh < 2; ++hh)
                        for (int pl = 0; pl < PL; ++pl)
                            tc::tma_load_3d(dst + (hh * PL + pl) * Cfg::kXHead, pl ? &tm_xlo : &tm_x,
                                            (hbeg + 2 * pr + hh) * kP, row0 + kp * KS, b, &sh.x_full[st]);
                }
            }
        }
    } else if (warp == kMma) {
        // ---- MMA: D[(head, p), n] += Xw^T B per K-part, all N columns per MMA.  A
        // shared-memory access by this thread waits behind the operand reads of the MMAs
        // it has issued (the tensor pipe idles meanwhile), so it makes one barrier wait
        // per K-part and keeps its give-up state in a register; a wait given up elsewhere
        // stops the arrivals, and its own bounded waits then end.
        if (lane == 0) {
            bool ok = tc::mbar_wait(&sh.mb_b, 0);
            tc::fence_after_sync();
            constexpr uint32_t idesc = tc::idesc_bf16(128, N, 1, 1);
            uint32_t n = 0;
            for (int pr = 0; pr < npairs && ok; ++pr) {
                const int ab = pr & 1;
                const uint32_t acc = tmem + (uint32_t)(ab * N);
                if (pr >= 2) ok = tc::mbar_wait(&sh.acc_empty[ab], ((pr - 2) >> 1) & 1);
                for (int kp = 0; kp < nparts && ok; ++kp, ++n) {
                    const uint32_t xb = n & 1;
                    ok = tc::mbar_wait(&sh.xt_full[xb], (n >> 1) & 1);
                    tc::fence_after_sync();
                    if (!ok) break;
                    const uint32_t ah = tc::smem_u32(sXt + xb * 2 * Cfg::kXt);
                    // Xw^T: MN-major no-swizzle, M = 128 contiguous in 16-byte rows; K steps
                    // of 16 rows are two core-matrix rows (2 * 16 * 128 bytes) apart
                    const uint64_t dah = tc::desc_mnmajor(ah, 128, 0), dal = tc::desc_mnmajor(ah + Cfg::kXt, 128, 0);
                    // B: all N columns in one MMA, the 64-column rows of the swizzle layout
                    // 256 * 128 bytes apart (lbo), 8-row groups 1024 bytes apart (sbo)
                    const uint64_t db = tc::desc_sw128(tc::smem_u32(sB) + (uint32_t)(kp * KS) * 128, 256 * 128, 1024);
#pragma unroll
                    for (int ks = 0; ks < KS / 16; ++ks) {
                        tc::mma_bf16(acc, dah + ks * tc::kstep_mnmajor(128), db + ks * 128u, idesc, (kp > 0 || ks > 0) ? 1u : 0u);
                        tc::mma_bf16(acc, dal + ks * tc::kstep_mnmajor(128), db + ks * 128u, idesc, 1u);
                    }
                    tc::mma_commit(&sh.xt_empty[xb]);
                }
                if (!ok) break;
                tc::mma_commit(&sh.acc_full[ab]);
            }
            if (!ok) sh.abort = 1;
        }
    } else {
        // ---- compute warps (256 threads)
        // Delta, the inclusive cumulative sum of Delta A_h within the chunk (both to
        // global, for the scan and carry kernels) and the weights w[h][s] of the CTA's
        // heads; one row s per thread (Q <= 256), rows past len get Delta 0.
        {
            const int s = tid;
            float d[kMaxHeads], v[kMaxHeads];
#pragma unroll
            for (int k = 0; k < kMaxHeads; ++k) {
                d[k] = 0.0f;
                if (k < hpc && s < len) {
                    const float dtv = __bfloat162float(a.dt[((int64_t)b * a.T + row0 + s) * a.H + hbeg + k]);
                    d[k] = softplus(dtv + (a.dt_bias ? a.dt_bias[hbeg + k] : 0.0f));
                }
                v[k] = k < hpc ? d[k] * a.A[hbeg + k] : 0.0f;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                for (int k = 0; k < kMaxHeads; ++k) {
                    const float u = __shfl_up_sync(0xffffffffu, v[k], o);
                    if (lane >= o) v[k] += u;
                }
            }
            if (lane == 31) {
#pragma unroll
                for (int k = 0; k < kMaxHeads; ++k) sh.warp_sum[warp][k] = v[k];
            }
            compute_sync();
#pragma unroll
            for (int k = 0; k < kMaxHeads; ++k)
                for (int w = 0; w < warp; ++w) v[k] += sh.warp_sum[w][k];
            // the chunk's last cumulative sum of every head: row len-1 publishes it
            if (s == len - 1) {
#pragma unroll
                for (int k = 0; k < kMaxHeads; ++k) sW[k * 256 + 255] = v[k];
            }
            compute_sync();
            float last[kMaxHeads];
#pragma unroll
            for (int k = 0; k < kMaxHeads; ++k) last[k] = sW[k * 256 + 255];
            compute_sync();
            if (s < Q) {
#pragma unroll
                for (int k = 0; k < kMaxHeads; ++k) {
                    if (k >= hpc) break;
                    if (ADJ) {
                        sW[k * 256 + s] = s < len ? __expf(v[k]) : 0.0f;
                    } else {
                        const int64_t o = (((int64_t)b * a.H + hbeg + k) * a.nchunks + c) * a.Q + s;
                        store_checked(a.dl_s, &a.dl[o], d[k], status);
                        store_checked(a.cum_s, &a.cum[o], v[k], status);
                        sW[k * 256 + s] = s < len ? __expf(last[k] - v[k]) * d[k] : 0.0f;
                    }
                }
            }
            compute_sync();
        }

        // Xw part n (pair pr, rows kp*KS ..): every 16-byte piece of 8 (head, p) values at
        // one row s, read from the swizzled x stage and written MN-major (no swizzle).
        // Piece i: s = i % 8 + 8 * (i / 128), m-chunk (i / 8) % 16, so that 8 consecutive
        // lanes write one contiguous 128-byte core matrix and read 8 distinct swizzle rows.
        constexpr int kPieces = KS * 16 / 256;  // per thread
        auto build = [&](int pr, int kp, uint32_t n) {
            const uint32_t st = n % kXStages;
            const unsigned char* xs = sXr + st * Cfg::kXStage;
            const uint32_t ah = tc::smem_u32(sXt + (n & 1) * 2 * Cfg::kXt), al = ah + Cfg::kXt;
#pragma unroll
            for (int k = 0; k < kPieces; ++k) {
                const int i = tid + 256 * k;
                const int s = (i & 7) + 8 * (i >> 7);
                const int mc = (i >> 3) & 15;
                const int hh = mc >> 3, pc = mc & 7;
                const float w = sW[(2 * pr + hh) * 256 + kp * KS + s];
                const unsigned char* row = xs + hh * PL * Cfg::kXHead + s * 128;
                const uint4 raw = *reinterpret_cast<const uint4*>(row + ((pc ^ (s & 7)) * 16));
                const __nv_bfloat162* r2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
                uint4 rawl = make_uint4(0, 0, 0, 0);
                if (XS) rawl = *reinterpret_cast<const uint4*>(row + Cfg::kXHead + ((pc ^ (s & 7)) * 16));
                const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&rawl);
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float2 f = __bfloat1622float2(r2[j]);
                    if (XS) f = __fadd2_rn(f, __bfloat1622float2(l2[j]));  // x' = x_hi + x_lo
                    f = __fmul2_rn(f, make_float2(w, w));
                    split_pair(f.x, f.y, hw[j], lw[j]);
                }
                const uint32_t off = (uint32_t)((s >> 3) * 2048 + mc * 128 + (s & 7) * 16);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(ah + off), "r"(hw[0]), "r"(hw[1]), "r"(hw[2]), "r"(hw[3]));
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(al + off), "r"(lw[0]), "r"(lw[1]), "r"(lw[2]), "r"(lw[3]));
            }
        };

        // states of pair pr from accumulator pr & 1: warp w has TMEM lanes 32*(w%4)..
        // (rows m = (head, p)) and the column half w/4
        const int q = warp & 3, chalf = warp >> 2;
        const int m = q * 32 + lane;
        constexpr uint32_t kHalf = (uint32_t)kP * N * 2;  // bytes of a tile's hi (or lo) half
        auto store_states = [&](int pr) {
            const int ab = pr & 1;
            wait_or_abort(sh, &sh.acc_full[ab], (pr >> 1) & 1);
            tc::fence_after_sync();
            const int h = hbeg + 2 * pr + (m >> 6), p = m & 63;
            char* tile = reinterpret_cast<char*>(a.states + ((((int64_t)b * a.nchunks + c) * a.H + h) * (int64_t)kP) * N);
            const uint32_t accb = tmem + (uint32_t)(ab * N) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
            for (int n0 = chalf * (N / 2); n0 < (chalf + 1) * (N / 2); n0 += 16) {
                uint32_t v[16];
                tc::tmem_ld16_async(accb + (uint32_t)n0, v);
                tc::tmem_wait_ld();
                if (sh.abort) continue;
#pragma unroll
                for (int j = 0; j < 16; j += 8) {
                    const uint32_t o = (uint32_t)((p >> 3) * (N / 8) * 128 + ((n0 + j) >> 3) * 128 + (p & 7) * 16);
                    store_checked(a.states_s, reinterpret_cast<uint4*>(tile + o), make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]), status);
                    store_checked(a.states_s, reinterpret_cast<uint4*>(tile + kHalf + o), make_uint4(v[j + 4], v[j + 5], v[j + 6], v[j + 7]), status);
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) arrive(&sh.acc_empty[ab]);
        };

        uint32_t n = 0;
        for (int pr = 0; pr < npairs; ++pr) {
            for (int kp = 0; kp < nparts; ++kp, ++n) {
                const uint32_t st = n % kXStages;
                wait_or_abort(sh, &sh.x_full[st], (n / kXStages) & 1);
                if (n >= 2) wait_or_abort(sh, &sh.xt_empty[n & 1], ((n - 2) >> 1) & 1);
                tc::fence_after_sync();
                build(pr, kp, n);
                tc::fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    arrive(&sh.x_empty[st]);
                    arrive(&sh.xt_full[n & 1]);
                }
            }
            if (pr > 0) store_states(pr - 1);
        }
        if (npairs > 0) store_states(npairs - 1);
    }
    if (sh.abort && tid == 0) atomicExch(status, kStatusTimeout);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}

// ---- host side -----------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 state_encode_tiled() {
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

// 3-D map over a bf16 tensor (inner, T, batch) with boxes of 64 inner elements x `rows`
// rows in the 128-byte swizzle layout; rows past T read as zero.
bool state_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t T, uint64_t batch, uint32_t rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = state_encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[3] = {inner, T, batch};
    const cuuint64_t strides[2] = {inner * 2, inner * 2 * T};
    const cuuint32_t box[3] = {64, rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Heads per CTA: the largest of 8, 4, 2 that divides the heads of a group (every head
// of the CTA reads the same B rows).
int state_heads_per_cta(const SsdTcArgs& s) {
    const int hpg = (int)(s.H / s.G);
    for (int cand : {8, 4, 2})
        if (hpg % cand == 0) return cand;
    return 2;
}

template <int N, bool XS, bool ADJ>
cudaError_t launch_state(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    using Cfg = StateCfg<N, XS>;
    CUtensorMap tx, txl, tb;
    const uint64_t T = (uint64_t)s.T, nb = (uint64_t)batch;
    if (!state_map(&tx, s.x, (uint64_t)s.H * kP, T, nb, Cfg::KS) ||
        !state_map(&txl, XS ? s.x_lo : s.x, (uint64_t)s.H * kP, T, nb, Cfg::KS) ||
        !state_map(&tb, s.B, (uint64_t)s.G * N, T, nb, 128))
        return cudaErrorInvalidValue;
    int* status = nullptr;
    cudaError_t e = device_status_address(&status);
    if (e != cudaSuccess) return e;
    auto kern = ssd_state_tc<N, XS, ADJ>;
    static_assert(sizeof(StateShared) <= 512, "pipeline state");
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmemTotal);
    if (e != cudaSuccess) return e;
    const int hpc = state_heads_per_cta(s);
    cudaEvent_t t0 = timing_begin(stream, ADJ ? "ssd_state_tc (adjoint)" : "ssd_state_tc");
    kern<<<dim3((unsigned)(s.nchunks * (s.H / hpc)), (unsigned)batch), kCta, Cfg::kSmemTotal, stream>>>(
        s, hpc, status, tx, txl, tb);
    note_launch(ADJ ? "ssd_state_tc (adjoint)" : "ssd_state_tc", stream, t0);
    return cudaGetLastError();
}

template <bool XS>
cudaError_t launch_state_n(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    switch (s.N) {
        case 64: return launch_state<64, XS, false>(s, batch, stream);
        case 128: return launch_state<128, XS, false>(s, batch, stream);
        default: return launch_state<256, XS, false>(s, batch, stream);
    }
}

}  // namespace

cudaError_t ssd_tc_chunk_state(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    return s.x_lo ? launch_state_n<true>(s, batch, stream) : launch_state_n<false>(s, batch, stream);
}

cudaError_t ssd_tc_chunk_state_adjoint(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    switch (s.N) {
        case 64: return s.x_lo ? launch_state<64, true, true>(s, batch, stream) : launch_state<64, false, true>(s, batch, stream);
        case 128: return s.x_lo ? launch_state<128, true, true>(s, batch, stream) : launch_state<128, false, true>(s, batch, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ssm
