// SSD chunk scan on the B300 tensor cores: the output of every chunk from the chunk's
// own inputs and the state carried into it ("Mamba-2：把状态空间模型和 Attention 统一到一个
// 数学框架里", 第二步 and 关键技术点 1-3: y = (L o M) x, dense diagonal blocks, low-rank
// off-diagonal blocks through the carried state).  Per (chunk, 128-row half, up to 32
// heads of one group), with s_t the in-chunk cumulative sum of Delta_t A_h:
//   G        = C_rows B^T                                   (M = 128, N = rows s of the half's causal range, K = dstate)
//   M'[t, s] = G[t, s] exp(s_t - s_s) Delta_s  (s < t),  G[t, t] Delta_t + D  (s = t),  0  (s > t)
//   Y_diag   = M' X_h                                       (M = 128, N = 64, K = s)
//   Y_off    = C_rows h_{c-1}^T                              (M = 128, N = 64, K = dstate)
//   out      = (Y_diag + exp(s_t) Y_off) SiLU(z)
// The skip term D x rides on M's diagonal, so the epilogue reads only the accumulators
// (and z).  M' is the one operand built by threads: scaled, masked and split into bf16
// hi + lo halves, both multiplied against the exact bf16 X, so that the scaled operand
// keeps ~16 significant bits.  Every other operand arrives by TMA / bulk copies: C and
// B rows and x tiles through 3-D tensor maps with 128-byte rows in the 128-byte swizzle
// layout (C, B K-major; x MN-major), h_{c-1} (already split hi/lo by the carry pass) as
// one contiguous bulk copy.  Up to dstate 128 the output tiles go back by TMA stores
// from shared memory.  Copies complete on mbarriers; every wait is bounded.
//
// One CTA per SM, warp-specialised: a TMA warp, an MMA warp and 16 compute warps that
// build M' and run the epilogues, handing work over on mbarriers (two M' parts in
// flight, x tiles double buffered, one h tile set refilled once a head's Y_off MMAs
// have read it, two sets of Y accumulators so that a head's epilogue overlaps the next
// head's MMAs).  512 TMEM columns: G, and the two accumulator sets.  Compute warp w
// owns TMEM lanes 32*(w%4).. (rows) and 16 columns of the M' parts it builds.
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

constexpr int kP = 64;            // headdim handled here
constexpr int kStatusTimeout = 8;

template <int N, bool XS>
struct ScanCfg {
    static_assert(N % 64 == 0, "C and B rows are 128-byte swizzle rows of 64 elements");
    static constexpr int KPC = N > 128 ? 32 : 64;           // columns of M' per K-part
    static constexpr int BC = 16;                            // columns of a part per warp
    static constexpr int NCG = KPC / BC;                     // column groups of a part (4 or 2)
    static constexpr int NG = 4 / NCG;                       // warp groups taking alternate parts
    static constexpr int kPartWarps = 4 * NCG;               // warps that build one part
    static constexpr uint32_t kC = 128u * N * 2;             // C rows of the half
    static constexpr uint32_t kB = 256u * N * 2;             // B rows [0, SW), prologue only
    static constexpr uint32_t kMPart = 128u * KPC * 2;       // one M' part, hi or lo
    static constexpr uint32_t kX = 256u * kP * 2;            // one x buffer (256 rows)
    static constexpr uint32_t kH = (uint32_t)kP * N * 2;     // one h_{c-1} tile, hi or lo
    // two M' parts in flight, one h_{c-1} tile set; up to dstate 128 also a staging area
    // for the output tiles (1 KB per compute warp), written to global memory by TMA
    static constexpr int kParts = 2;
    static constexpr int kHBufs = 1;
    static constexpr bool kStageOut = N <= 128;
    static constexpr uint32_t kOut = kStageOut ? 16u * 1024 : 0u;
    static constexpr uint32_t kPhase2 = kParts * 2 * kMPart + 2 * kX + kHBufs * 2 * kH + kOut;
    static constexpr uint32_t kRegion = kB > kPhase2 ? kB : kPhase2;
    static constexpr uint32_t kSmem = kC + kRegion;   // operands; the pipeline state follows
    static constexpr uint32_t kSmemTotal = kSmem + 2304;
    static_assert(kSmemTotal <= 232448, "shared memory");
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// v = hi + lo with hi = bf16(v) and lo = bf16(v - hi), two values at a time.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    const float2 l = __ffma2_rn(hf, make_float2(-1.0f, -1.0f), make_float2(a, b));
    lo = pack_bf16x2(l.x, l.y);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d));
}

// Shared state of one CTA's pipeline (after the operand buffers in dynamic shared memory).
struct __align__(16) ScanShared {
    float beta[2][256];     // per head parity: log2(Delta_s) - cum_s log2(e), so that
                            // exp(cum_t - cum_s) Delta_s = 2^(alpha_t + beta_s)
    uint64_t mb_load;       // C and B rows (prologue TMA)
    uint64_t mb_g;          // G = C B^T in TMEM
    uint64_t full_part[2];  // M' part built (one arrival per building warp)
    uint64_t empty_part[2]; // M' part consumed by its MMAs
    uint64_t acc_full[2];   // a head's Y accumulators complete
    uint64_t acc_empty[2];  // a head's Y accumulators read by the epilogue (one arrival per compute warp)
    uint64_t x_full[2], x_empty[2];
    uint64_t h_full[2], h_empty[2];
    uint32_t tmem;
    volatile int abort;     // a bounded wait gave up: every later wait returns at once
};

constexpr int kComputeWarps = 16;
constexpr int kMmaWarp = 16;
constexpr int kLoadWarp = 17;
constexpr int kCtaThreads = 32 * 18;

// Bounded wait that gives up at once when another wait of the CTA already gave up.
__device__ __forceinline__ void pipe_wait(ScanShared& sh, uint64_t* mb, uint32_t phase) {
    if (sh.abort) return;
    if (!tc::mbar_wait(mb, phase)) sh.abort = 1;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* mb) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(mb)) : "memory");
}
// Named barrier of the compute warps only.
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// grid (nchunks * Q/128 * H / heads_per_cta, batch): blockIdx.x = (chunk * Q/128 + half) *
// (H / heads_per_cta) + head block; 18 warps; one CTA per SM.
// Warps 0-15 build M' and run the epilogues (warp w: TMEM lanes 32*(w%4).., column
// quarter w/4 of each part); warp 16 issues the MMAs; warp 17 issues the TMA copies.
template <int N, bool GATE, bool XS>
__global__ void __launch_bounds__(kCtaThreads, 1)
    ssd_scan_tc(const SsdTcArgs a, const int heads_per_cta, int* status, const __grid_constant__ CUtensorMap tm_x,
                const __grid_constant__ CUtensorMap tm_xlo, const __grid_constant__ CUtensorMap tm_c,
                const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_out) {
    using Cfg = ScanCfg<N, XS>;
    constexpr int KPC = Cfg::KPC, BC = Cfg::BC, NCG = Cfg::NCG, NG = Cfg::NG;
    extern __shared__ __align__(1024) unsigned char smem[];
    ScanShared& sh = *reinterpret_cast<ScanShared*>(smem + Cfg::kSmem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Q = (int)a.Q;
    const int halves = Q / 128;
    const int nhb = (int)(a.H / heads_per_cta);
    const int64_t c = (blockIdx.x / nhb) / halves;
    const int rh = (int)((blockIdx.x / nhb) % halves);
    const int b = blockIdx.y;
    const int len = (int)min((int64_t)Q, a.T - c * a.Q);
    const int t0 = 128 * rh;
    if (t0 >= len) return;      // no valid rows in this half (uniform over the CTA)
    const int SW = t0 + 128;    // columns s of G this half needs (causal)
    const int nparts = SW / KPC;
    const int hbeg = (int)(blockIdx.x % nhb) * heads_per_cta;
    const int nh = heads_per_cta;
    const int g = hbeg / (int)(a.H / a.G);
    const int row0 = (int)(c * a.Q);  // first token of the chunk within its sequence
    // XS with 256 rows: a head's two x planes take both x buffers (one head at a time)
    const bool xser = XS && SW > 128;

    // TMA-written operands use the 128-byte swizzle layout (rows of 64 elements):
    unsigned char* sC = smem;                               // [n/64][t 128][64], K-major A
    unsigned char* region = smem + Cfg::kC;
    unsigned char* sB = region;                             // [n/64][s SW][64], K-major B (prologue)
    // thread- and carry-written operands use the no-swizzle core-matrix layout:
    unsigned char* sM = region;                             // [part kParts][hi, lo] [t/8][s/8 of KPC][8][8]
    unsigned char* sX = region + Cfg::kParts * 2 * Cfg::kMPart;  // [buffer 2] [s SW][64] (+ lo plane), MN-major B
    unsigned char* sH = sX + 2 * Cfg::kX;                   // [set kHBufs][hi, lo] [p/8][n/8][8][8]
    unsigned char* sOut = sH + Cfg::kHBufs * 2 * Cfg::kH;   // [compute warp][row 32][16 p] output staging

    if (tid == 0) {
        tc::mbar_init(&sh.mb_load, 1);
        tc::mbar_init(&sh.mb_g, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&sh.full_part[i], Cfg::kPartWarps);
            tc::mbar_init(&sh.empty_part[i], 1);
            tc::mbar_init(&sh.acc_full[i], 1);
            tc::mbar_init(&sh.acc_empty[i], kComputeWarps);
            tc::mbar_init(&sh.x_full[i], 1);
            tc::mbar_init(&sh.x_empty[i], 1);
            tc::mbar_init(&sh.h_full[i], 1);
            tc::mbar_init(&sh.h_empty[i], 1);
        }
        sh.abort = 0;
        tc::mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(&sh.tmem, 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sh.tmem;
    const uint32_t tG = tmem;
    // TMEM columns: G = C B^T in [0, SW), and two sets of {Y_diag, Y_off} at 256 + 128 *
    // set.  At dstate 256 a first half (SW = 128) uses its 128 spare columns instead:
    // Y_diag sets at 128 + 64 * set, and Y_off sets of 128 columns at 256 + 128 * set
    // holding C h_hi and C h_lo side by side from one N = 128 MMA over the stacked
    // [h_hi; h_lo] tile (half the MMAs and C reads of two N = 64 products; c4 scan
    // 1005 -> 899 us).  At dstate 128 the extra epilogue load costs more than the 8
    // MMAs it saves (c3 scan 348 -> 354 us), so those keep the narrow layout.
    const bool wide_off = N > 128 && SW == 128;
    auto t_yd = [&](int set) { return wide_off ? tmem + 128 + 64 * set : tmem + 256 + 128 * set; };
    auto t_yo = [&](int set) { return wide_off ? tmem + 256 + 128 * set : tmem + 256 + 128 * set + 64; };

    // Buffer schedule: x buffer and its use count for head hi (serial planes: buffer 0 every
    // head); h set likewise.
    auto xbuf = [&](int hi) { return xser ? 0 : (hi & 1); };
    auto xuse = [&](int hi) { return xser ? hi : (hi >> 1); };
    auto hbuf = [&](int hi) { return Cfg::kHBufs == 2 ? (hi & 1) : 0; };
    auto huse = [&](int hi) { return Cfg::kHBufs == 2 ? (hi >> 1) : hi; };
    auto x_tile = [&](int hi, int plane) -> uint32_t {
        if (xser) return tc::smem_u32(sX + plane * Cfg::kX);
        return tc::smem_u32(sX + (hi & 1) * Cfg::kX + plane * (uint32_t)SW * kP * 2);
    };

    if (warp == kLoadWarp) {
        // ---- TMA producer (one thread)
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(&sh.mb_load, Cfg::kC + (uint32_t)SW * N * 2);
            for (int j = 0; j < N / 64; ++j) {
                tc::tma_load_3d(sC + j * 128 * 128, &tm_c, g * N + 64 * j, row0 + t0, b, &sh.mb_load);
                for (int rb = 0; rb < SW / 128; ++rb)
                    tc::tma_load_3d(sB + (j * SW + rb * 128) * 128, &tm_b, g * N + 64 * j, row0 + 128 * rb, b, &sh.mb_load);
            }
            pipe_wait(sh, &sh.mb_g, 0);  // G's MMAs are done: B's region takes the head tiles
            for (int hi = 0; hi < nh && !sh.abort; ++hi) {
                const int hn = hbeg + hi;
                const int xb = xbuf(hi), ux = xuse(hi);
                if (ux > 0) pipe_wait(sh, &sh.x_empty[xb], (ux - 1) & 1);
                const uint32_t planes = XS ? 2 : 1;
                tc::mbar_arrive_expect_tx(&sh.x_full[xb], planes * (uint32_t)SW * kP * 2);
                for (int pl = 0; pl < (int)planes; ++pl) {
                    unsigned char* base = xser ? sX + pl * Cfg::kX : sX + xb * Cfg::kX + pl * (uint32_t)SW * kP * 2;
                    const CUtensorMap* tm = pl ? &tm_xlo : &tm_x;
                    for (int rb = 0; rb < SW / 128; ++rb)
                        tc::tma_load_3d(base + rb * 128 * 128, tm, hn * kP, row0 + 128 * rb, b, &sh.x_full[xb]);
                }
                const int hs = hbuf(hi), uh = huse(hi);
                if (uh > 0) pipe_wait(sh, &sh.h_empty[hs], (uh - 1) & 1);
                const unsigned char* src = reinterpret_cast<const unsigned char*>(
                    a.states + (((int64_t)b * a.nchunks + c) * a.H + hn) * (int64_t)kP * N);
                tc::mbar_arrive_expect_tx(&sh.h_full[hs], 2 * Cfg::kH);
                tc::bulk_load(sH + hs * 2 * Cfg::kH, src, 2 * Cfg::kH, &sh.h_full[hs]);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---- MMA issuer (one thread).  A shared-memory access by this thread (a barrier
        // test, a flag read) waits behind the operand reads of the MMAs it has issued, so
        // the tensor pipe idles while it completes: the loop makes one barrier wait per
        // M' part and keeps its own give-up state in a register (a wait given up
        // elsewhere in the CTA stops the arrivals, and its own bounded waits then end).
        if (lane == 0) {
            bool ok = tc::mbar_wait(&sh.mb_load, 0);
            tc::fence_after_sync();
            if (ok) {
                const uint32_t idesc = tc::idesc_bf16(128, SW, 0, 0);
#pragma unroll 1
                for (int ks = 0; ks < N / 16; ++ks) {
                    const uint32_t in_row = (uint32_t)(ks & 3) * 32;  // K offset inside a 128-byte row
                    const uint64_t da = tc::desc_sw128(tc::smem_u32(sC + (ks >> 2) * 128 * 128) + in_row, 16, 1024);
                    const uint64_t db = tc::desc_sw128(tc::smem_u32(sB + (ks >> 2) * SW * 128) + in_row, 16, 1024);
                    tc::mma_bf16(tG, da, db, idesc, ks > 0);
                }
                tc::mma_commit(&sh.mb_g);
            }
            constexpr uint32_t id_diag = tc::idesc_bf16(128, kP, 0, 1);
            constexpr uint32_t id_off = tc::idesc_bf16(128, kP, 0, 0);
            constexpr uint32_t id_off_wide = tc::idesc_bf16(128, 2 * kP, 0, 0);
            uint32_t n = 0;  // M' parts consumed so far
            for (int hi = 0; hi < nh && ok; ++hi) {
                const int ab = hi & 1;
                const uint32_t tYd = t_yd(ab), tYo = t_yo(ab);
                if (hi >= 2) ok = tc::mbar_wait(&sh.acc_empty[ab], ((hi - 2) >> 1) & 1);  // head hi-2's epilogue read them
                ok = ok && tc::mbar_wait(&sh.h_full[hbuf(hi)], huse(hi) & 1);
                tc::fence_after_sync();
                if (!ok) break;
                {
                    // Y_off = C h_hi + C h_lo first: it needs no M' part, so the tensor pipe
                    // runs it while the compute warps finish the previous heads and build
                    // this head's first part
                    const uint32_t cb = tc::smem_u32(sC);
                    const uint32_t hs = tc::smem_u32(sH + hbuf(hi) * 2 * Cfg::kH);
                    // the lo tile continues the hi tile's 8-row groups (kH = 8 group strides),
                    // so one descriptor spans both as 128 rows
                    const uint64_t dhh = tc::desc_strided(hs, 128, (N / 8) * 128);
                    const uint64_t dhl = tc::desc_strided(hs + Cfg::kH, 128, (N / 8) * 128);
                    if (wide_off) {
#pragma unroll
                        for (int ks = 0; ks < N / 16; ++ks) {
                            const uint64_t dc = tc::desc_sw128(cb + (uint32_t)(ks >> 2) * 128 * 128 + (uint32_t)(ks & 3) * 32, 16, 1024);
                            tc::mma_bf16(tYo, dc, dhh + ks * 16u, id_off_wide, ks > 0 ? 1u : 0u);
                        }
                    } else {
#pragma unroll
                        for (int ks = 0; ks < N / 16; ++ks) {
                            const uint64_t dc = tc::desc_sw128(cb + (uint32_t)(ks >> 2) * 128 * 128 + (uint32_t)(ks & 3) * 32, 16, 1024);
                            tc::mma_bf16(tYo, dc, dhh + ks * 16u, id_off, ks > 0 ? 1u : 0u);
                            tc::mma_bf16(tYo, dc, dhl + ks * 16u, id_off, 1u);
                        }
                    }
                    tc::mma_commit(&sh.h_empty[hbuf(hi)]);  // the h tiles may be replaced
                }
                ok = tc::mbar_wait(&sh.x_full[xbuf(hi)], xuse(hi) & 1);
                for (int kp = 0; kp < nparts && ok; ++kp, ++n) {
                    const uint32_t pb = n % Cfg::kParts;
                    ok = tc::mbar_wait(&sh.full_part[pb], (n / Cfg::kParts) & 1);
                    tc::fence_after_sync();
                    if (!ok) break;
                    const uint32_t mh = tc::smem_u32(sM + pb * 2 * Cfg::kMPart);
                    const uint64_t dmh = tc::desc_strided(mh, 128, (KPC / 8) * 128);
                    const uint64_t dml = tc::desc_strided(mh + Cfg::kMPart, 128, (KPC / 8) * 128);
                    // x: rows s of this part, 128 bytes each; K steps of 16 rows are 2048
                    // bytes (128 in descriptor units) apart
                    const uint64_t dx = tc::desc_sw128(x_tile(hi, 0) + (uint32_t)(kp * KPC) * 128, 1024, 1024);
#pragma unroll
                    for (int ks = 0; ks < KPC / 16; ++ks)
                        tc::mma_bf16(tYd, dmh + ks * 16u, dx + ks * 128u, id_diag, (kp > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                    for (int ks = 0; ks < KPC / 16; ++ks) tc::mma_bf16(tYd, dml + ks * 16u, dx + ks * 128u, id_diag, 1u);
                    if (XS) {
                        const uint64_t dxl = tc::desc_sw128(x_tile(hi, 1) + (uint32_t)(kp * KPC) * 128, 1024, 1024);
#pragma unroll
                        for (int ks = 0; ks < KPC / 16; ++ks) tc::mma_bf16(tYd, dmh + ks * 16u, dxl + ks * 128u, id_diag, 1u);
                    }
                    tc::mma_commit(&sh.empty_part[pb]);  // the part buffer may be rebuilt
                }
                if (!ok) break;
                tc::mma_commit(&sh.acc_full[ab]);   // the epilogue may read this head's accumulators
                tc::mma_commit(&sh.x_empty[xbuf(hi)]);
            }
            if (!ok) sh.abort = 1;
        }
    } else {
        // ---- compute warps: M' builds and epilogues
        const int q = warp & 3;             // TMEM lane quarter
        const int cq = warp >> 2;           // column quarter of the epilogue's outputs
        const int cg = (warp >> 2) % NCG;   // column group of a part
        const int gi = warp / (4 * NCG);    // warp group: builds the parts kp with kp % NG == gi
        const int r = q * 32 + lane;        // row (TMEM lane) within the half
        const int t = t0 + r;               // row within the chunk
        const bool row_ok = t < len;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int t_warp_min = t0 + q * 32;  // tcgen05.ld and the part blocks are per warp
        const int t_warp_max = t_warp_min + 31;
        const uint32_t row_off = (uint32_t)((r >> 3) * (KPC / 8) * 128 + (r & 7) * 16);
        const int tq = min(t, Q - 1);

        // per-head scalars: Delta and the cumulative sum of row tid (for beta), the
        // cumulative sum of this thread's row (alpha), D; fetched a head ahead
        float pf_dl = 0.0f, pf_cum = 0.0f, pf_row = 0.0f, pf_D = 0.0f;
        auto prefetch = [&](int hn) {
            const int64_t base = (((int64_t)b * a.H + hn) * a.nchunks + c) * a.Q;
            if (tid < Q) {
                pf_dl = a.dl[base + tid];
                pf_cum = a.cum[base + tid];
            }
            pf_row = a.cum[base + tq];
            pf_D = a.D ? a.D[hn] : 0.0f;
        };
        auto publish_beta = [&](int parity) {
            if (tid < Q) sh.beta[parity][tid] = (pf_dl > 0.0f ? lg2(pf_dl) : -INFINITY) - pf_cum * kLog2e;
        };
        prefetch(hbeg);
        publish_beta(0);
        float cur_alpha = pf_row * kLog2e, cur_D = pf_D;  // head hbeg
        if (nh > 1) prefetch(hbeg + 1);

        // this thread's BC columns of M' part kp into part buffer pb: row t, columns
        // s0 .. s0 + BC - 1.  Blocks wholly above the diagonal are zero; blocks that reach
        // it are masked and take D on the diagonal.
        auto build = [&](int kp, int pb, const float* beta, float alpha, float Dh) {
            const int s0 = KPC * kp + BC * cg;
            uint32_t hw[BC / 2], lw[BC / 2];
            if (s0 > t_warp_max) {
#pragma unroll
                for (int j = 0; j < BC / 2; ++j) hw[j] = lw[j] = 0u;
            } else {
                uint32_t gv[BC];
                tc::tmem_ld_async(tG + lane_base + (uint32_t)s0, gv);
                float bt[BC];
#pragma unroll
                for (int j = 0; j < BC; j += 4) *reinterpret_cast<float4*>(&bt[j]) = *reinterpret_cast<const float4*>(&beta[s0 + j]);
                tc::tmem_wait_ld();
                if (s0 + BC - 1 < t_warp_min) {
                    // every column of the block lies left of every row's diagonal
#pragma unroll
                    for (int j = 0; j < BC; j += 2) {
                        const float v0 = ex2(alpha + bt[j]) * __uint_as_float(gv[j]);
                        const float v1 = ex2(alpha + bt[j + 1]) * __uint_as_float(gv[j + 1]);
                        split_pair(v0, v1, hw[j / 2], lw[j / 2]);
                    }
                } else {
                    // the block reaches the diagonal: zero right of it, D on it
                    const int dg = t - s0;
#pragma unroll
                    for (int j = 0; j < BC; j += 2) {
                        float v0 = ex2(alpha + bt[j]) * __uint_as_float(gv[j]);
                        float v1 = ex2(alpha + bt[j + 1]) * __uint_as_float(gv[j + 1]);
                        v0 = j < dg ? v0 : (j == dg ? v0 + Dh : 0.0f);
                        v1 = j + 1 < dg ? v1 : (j + 1 == dg ? v1 + Dh : 0.0f);
                        split_pair(v0, v1, hw[j / 2], lw[j / 2]);
                    }
                }
            }
            const uint32_t ph = tc::smem_u32(sM + pb * 2 * Cfg::kMPart) + row_off + (uint32_t)(cg * BC / 8) * 128;
            const uint32_t pl = ph + Cfg::kMPart;
#pragma unroll
            for (int j = 0; j < BC / 8; ++j) {
                sts128(ph + j * 128, hw[4 * j], hw[4 * j + 1], hw[4 * j + 2], hw[4 * j + 3]);
                sts128(pl + j * 128, lw[4 * j], lw[4 * j + 1], lw[4 * j + 2], lw[4 * j + 3]);
            }
        };

        // epilogue of head hi (accumulator set hi & 1): out = Y_diag + exp(cum_t) Y_off, gate
        auto finish = [&](int hi, float alpha_h) {
            const int ab = hi & 1;
            pipe_wait(sh, &sh.acc_full[ab], (hi >> 1) & 1);
            tc::fence_after_sync();
            const uint32_t tYd = t_yd(ab), tYo = t_yo(ab);
            const int p0 = 16 * cq;
            uint32_t yd[16], yo[16];
            tc::tmem_ld16_async(tYd + lane_base + (uint32_t)p0, yd);
            tc::tmem_ld16_async(tYo + lane_base + (uint32_t)p0, yo);
            tc::tmem_wait_ld();
            if (wide_off) {
                // C h_lo sits 64 columns after C h_hi
                uint32_t yl[16];
                tc::tmem_ld16_async(tYo + 64 + lane_base + (uint32_t)p0, yl);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) yo[j] = __float_as_uint(__uint_as_float(yo[j]) + __uint_as_float(yl[j]));
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.acc_empty[ab]);  // the MMAs of head hi + 2 may overwrite them
            if (sh.abort || (!Cfg::kStageOut && !row_ok)) return;
            const float e = ex2(alpha_h);
            const int64_t row = (((int64_t)b * a.T + row0 + t) * a.H + hbeg + hi) * kP + p0;
            uint4 zr[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            if (GATE) {
                zr[0] = *reinterpret_cast<const uint4*>(a.z + row);
                zr[1] = *reinterpret_cast<const uint4*>(a.z + row + 8);
            }
            const __nv_bfloat162* z2 = reinterpret_cast<const __nv_bfloat162*>(zr);
            uint32_t pk[8];
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                float2 y = __ffma2_rn(make_float2(e, e), make_float2(__uint_as_float(yo[j]), __uint_as_float(yo[j + 1])),
                                      make_float2(__uint_as_float(yd[j]), __uint_as_float(yd[j + 1])));
                if (GATE) y = __fmul2_rn(y, silu2_fma(__bfloat1622float2(z2[j / 2])));
                pk[j / 2] = pack_bf16x2(y.x, y.y);
            }
            if (Cfg::kStageOut) {
                // this warp's 32 rows x 16 columns through shared memory, one TMA store
                // (rows past the sequence's end are clipped by the tensor map)
                unsigned char* st = sOut + warp * 1024;
                if (lane == 0) tc::bulk_wait_read_all();  // the previous head's store has read it
                __syncwarp();
                sts128(tc::smem_u32(st + lane * 32), pk[0], pk[1], pk[2], pk[3]);
                sts128(tc::smem_u32(st + lane * 32 + 16), pk[4], pk[5], pk[6], pk[7]);
                tc::fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_3d(&tm_out, st, (hbeg + hi) * kP + p0, row0 + t0 + q * 32, b);
                    tc::bulk_commit();
                }
            } else {
                uint4* dst = reinterpret_cast<uint4*>(a.out + row);
                store_checked(a.out_s, dst, make_uint4(pk[0], pk[1], pk[2], pk[3]), status);
                store_checked(a.out_s, dst + 1, make_uint4(pk[4], pk[5], pk[6], pk[7]), status);
            }
        };

        pipe_wait(sh, &sh.mb_g, 0);  // G is in TMEM
        tc::fence_after_sync();
        uint32_t n = 0;  // M' parts built so far
        float alpha_prev = 0.0f;
        for (int hi = 0; hi < nh; ++hi) {
            // every compute warp is done with head hi-1's builds (so the beta buffer of
            // head hi + 1 is free) and head hi's beta is visible
            compute_sync();
            const float alpha = cur_alpha, Dh = cur_D;
            if (hi + 1 < nh) {
                publish_beta((hi + 1) & 1);
                cur_alpha = pf_row * kLog2e;
                cur_D = pf_D;
                if (hi + 2 < nh) prefetch(hbeg + hi + 2);
            }
            const float* beta = sh.beta[hi & 1];
            for (int kp = 0; kp < nparts; ++kp, ++n) {
                if (kp % NG != gi) continue;  // the other warp group builds this part
                const uint32_t pb = n % Cfg::kParts;
                if (n >= (uint32_t)Cfg::kParts) pipe_wait(sh, &sh.empty_part[pb], ((n - Cfg::kParts) / Cfg::kParts) & 1);
                tc::fence_after_sync();
                build(kp, pb, beta, alpha, Dh);
                tc::fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.full_part[pb]);
            }
            if (hi > 0) finish(hi - 1, alpha_prev);
            alpha_prev = alpha;
        }
        if (nh > 0) finish(nh - 1, alpha_prev);
        if (Cfg::kStageOut && lane == 0) tc::bulk_wait_all();  // the output stores are done
    }
    if (sh.abort && tid == 0) atomicExch(status, kStatusTimeout);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ---- host side -----------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
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

// 3-D store map over the bf16 output (inner, T, batch): boxes of 16 columns x 32 rows
// (one compute warp's part of an epilogue), no swizzle; rows past T are not written.
bool make_out_map(CUtensorMap* m, void* base, uint64_t inner, uint64_t T, uint64_t batch) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[3] = {inner, T, batch};
    const cuuint64_t strides[2] = {inner * 2, inner * 2 * T};
    const cuuint32_t box[3] = {16, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over a bf16 tensor (inner, T, batch), row-major and contiguous, with boxes of
// 64 inner elements x 128 rows x 1 in the 128-byte swizzle layout: each box lands as 128
// rows of 128 bytes, the operand layout of desc_sw128.  Rows past T read as zero.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t T, uint64_t batch) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[3] = {inner, T, batch};
    const cuuint64_t strides[2] = {inner * 2, inner * 2 * T};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Heads per CTA: G = C B^T and the C and B rows are shared by the CTA's heads, and each
// CTA pays a prologue (the C and B copies, G's MMAs) that nothing overlaps, so a CTA takes
// as many heads of its group as keep at least six waves of CTAs on the GPU, up to 16 (32
// measured slower: c4 scan 900 us against 882 with 16; c3 353 against 348; 8 on c3 357).
int scan_heads_per_cta(const SsdTcArgs& s, int64_t batch) {
    const int hpg = (int)(s.H / s.G);
    const int64_t halves = s.nchunks * (s.Q / 128) * batch;
    const int64_t want = 6 * (int64_t)sm_count();
    int best = 1;
    for (int cand : {1, 2, 4, 8, 16})
        if (hpg % cand == 0 && (cand == 1 || halves * (s.H / cand) >= want)) best = cand;
    return best;
}

template <int N, bool GATE, bool XS>
cudaError_t launch_scan(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    using Cfg = ScanCfg<N, XS>;
    CUtensorMap tx, txl, tmc, tmb, tmo;
    const uint64_t T = (uint64_t)s.T, nb = (uint64_t)batch;
    if (!make_map(&tx, s.x, (uint64_t)s.H * kP, T, nb) || !make_map(&txl, XS ? s.x_lo : s.x, (uint64_t)s.H * kP, T, nb) ||
        !make_map(&tmc, s.C, (uint64_t)s.G * N, T, nb) || !make_map(&tmb, s.B, (uint64_t)s.G * N, T, nb) ||
        !make_out_map(&tmo, s.out, (uint64_t)s.H * kP, T, nb))
        return cudaErrorInvalidValue;
    int* status = nullptr;
    cudaError_t e = device_status_address(&status);
    if (e != cudaSuccess) return e;
    auto kern = ssd_scan_tc<N, GATE, XS>;
    static_assert(sizeof(ScanShared) <= 2304, "pipeline state");
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmemTotal);
    if (e != cudaSuccess) return e;
    const int hpc = scan_heads_per_cta(s, batch);
    // the head blocks of a chunk half are adjacent in launch order: they run together and
    // read its C and B rows once from DRAM and then from L2
    const dim3 grid((unsigned)(s.nchunks * (s.Q / 128) * (s.H / hpc)), (unsigned)batch);
    cudaEvent_t t0 = timing_begin(stream, "ssd_scan_tc");
    kern<<<grid, kCtaThreads, Cfg::kSmemTotal, stream>>>(s, hpc, status, tx, txl, tmc, tmb, tmo);
    note_launch("ssd_scan_tc", stream, t0);
    return cudaGetLastError();
}

template <bool GATE, bool XS>
cudaError_t launch_scan_n(const SsdTcArgs& s, int64_t batch, cudaStream_t stream) {
    switch (s.N) {
        case 64: return launch_scan<64, GATE, XS>(s, batch, stream);
        case 128: return launch_scan<128, GATE, XS>(s, batch, stream);
        default: return launch_scan<256, GATE, XS>(s, batch, stream);
    }
}

}  // namespace

cudaError_t ssd_tc_chunk_scan(const SsdTcArgs& s, int64_t batch, bool gate, cudaStream_t stream) {
    if (s.x_lo) return gate ? launch_scan_n<true, true>(s, batch, stream) : launch_scan_n<false, true>(s, batch, stream);
    return gate ? launch_scan_n<true, false>(s, batch, stream) : launch_scan_n<false, false>(s, batch, stream);
}

}  // namespace ssm
