/*
 * fp64 CPU oracle for the selective state-space scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package's smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant with the CUDA
 * library; the two meet only at the seeded input generator.
 *
 * Sources (web pages, cited by title and section):
 *   [Mamba-2 explainer] "Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里"
 *       section 背景问题: discrete recurrence h_t = Abar h_{t-1} + Bbar x_t, y_t = C h_t
 *       section 核心思路 / 第一步: Delta_t = softplus(Linear(x_t)); Abar obtained from Delta
 *       section 第二步: unrolled form y = (L o M) x with a lower-triangular M
 *       section 关键技术点 1: semiseparable M, low-rank off-diagonal blocks
 *   [SSM engineering article] "引言：Attention的天花板 ... State Space Model：序列建模的另一条路"
 *       section 基本原理: y(t) = C h(t) + D x(t)
 *   [Mamba paper digest] "论文解读：Mamba — 线性时间的序列建模革命"
 *       section 五 Mamba块架构: SSM output multiplied by SiLU of the z branch
 *   [Mamba / hybrid overview] "基础知识：Mamba 与混合 SSM 架构"
 *       section 2 从 SSM 到 Selective SSM: h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t
 *       section 3 Mamba block 里发生了什么: a depthwise convolution adds local context
 *       before the selective scan
 *   [Mamba paper digest] section 五 Mamba块架构: the x branch runs Conv1d, then SiLU,
 *       then the selective SSM; [SSM engineering article] 工程实践: kernel width d_conv = 4
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - discretisation: Abar = exp(Delta * A) and Bbar = Delta * B (exponential decay,
 *     Euler input term); the pages only say that Abar comes from Delta;
 *   - initial state zero unless an initial state is passed;
 *   - y_t reads the state after the update (so M[t,t] = C_t . Delta_t B_t);
 *   - softplus(v) = ln(1 + e^v), evaluated as max(v,0) + log1p(exp(-|v|)), with the
 *     optional dt_bias added before the softplus;
 *   - out = (C.h + D x) * SiLU(z) with SiLU(z) = z / (1 + e^-z);
 *   - B and C are shared by groups: channel group g = head / (nheads / ngroups).
 *   - the convolution ahead of the scan (oracle_conv_silu) is causal and depthwise,
 *     x'_t = SiLU(bias + sum_k w[k] x_{t-K+1+k}), so w[K-1] weights the current input;
 *     inputs before t = 0 come from the previous call (x_prev) or are zero.  The scan
 *     then reads x' wherever it reads x, the skip term included.
 *
 * Layouts (row-major, token-major, all float64 here):
 *   x, z, out      (batch, seqlen, nheads, headdim)   -- DIAG: headdim == 1
 *   dt             (batch, seqlen, nheads)
 *   A              DIAG: (nheads, dstate)             SSD: (nheads,)
 *   B, C           (batch, seqlen, ngroups, dstate)
 *   D, dt_bias     (nheads,)                          nullable
 *   initial_state, final_state (batch, nheads, headdim, dstate), nullable
 *
 * Parity status: pinned (brute-force semiseparable matrix, closed-form LTI responses,
 * masked linear attention at A = 0, hand-worked golden values, invariants; the
 * convolution against numpy's convolution; the backward pass against central finite
 * differences of the forward; the complex scan against the real scan with zero
 * imaginary parts, its own materialised matrix, closed-form damped-oscillator
 * responses and pure-rotation invariants).
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MODE_DIAG 0
#define ORACLE_MODE_SSD 1

/* softplus(v) = ln(1 + e^v), overflow-free form. */
static double oracle_softplus(double v) { return fmax(v, 0.0) + log1p(exp(-fabs(v))); }

/* SiLU(z) = z * sigmoid(z). */
static double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

typedef struct {
    int mode;
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups;
    const double *x, *dt, *A, *B, *C, *D, *z, *dt_bias, *initial_state;
    double *out, *final_state;
} oracle_problem;

static int oracle_check(const oracle_problem* p) {
    if (!p->x || !p->dt || !p->A || !p->B || !p->C || !p->out) return 1;
    if (p->batch < 0 || p->seqlen < 0 || p->nheads <= 0 || p->headdim <= 0 || p->dstate <= 0 ||
        p->ngroups <= 0)
        return 2;
    if (p->nheads % p->ngroups != 0) return 2;
    if (p->mode == ORACLE_MODE_DIAG && p->headdim != 1) return 2;
    if (p->mode != ORACLE_MODE_DIAG && p->mode != ORACLE_MODE_SSD) return 2;
    return 0;
}

/* Decay coefficient A for channel head h and state index n. */
static double oracle_acoef(const oracle_problem* p, int64_t h, int64_t n) {
    return p->mode == ORACLE_MODE_DIAG ? p->A[h * p->dstate + n] : p->A[h];
}

/* Plain sequential recurrence for one channel (b, h, q); q indexes headdim. */
static void oracle_channel_sequential(const oracle_problem* p, int64_t b, int64_t h, int64_t q,
                                      double* state) {
    const int64_t T = p->seqlen, H = p->nheads, P = p->headdim, N = p->dstate, G = p->ngroups;
    const int64_t g = h / (H / G);
    const int64_t sidx = ((b * H + h) * P + q) * N;
    for (int64_t n = 0; n < N; ++n) state[n] = p->initial_state ? p->initial_state[sidx + n] : 0.0;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t bt = b * T + t;
        const double v = p->dt[bt * H + h] + (p->dt_bias ? p->dt_bias[h] : 0.0);
        const double delta = oracle_softplus(v);
        const int64_t xi = (bt * H + h) * P + q;
        const double xv = p->x[xi];
        const double* Bt = p->B + (bt * G + g) * N;
        const double* Ct = p->C + (bt * G + g) * N;
        double y = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double abar = exp(delta * oracle_acoef(p, h, n));
            state[n] = abar * state[n] + delta * Bt[n] * xv;
            y += Ct[n] * state[n];
        }
        if (p->D) y += p->D[h] * xv;
        if (p->z) y *= oracle_silu(p->z[xi]);
        p->out[xi] = y;
    }
    if (p->final_state)
        for (int64_t n = 0; n < N; ++n) p->final_state[sidx + n] = state[n];
}

/*
 * Chunked evaluation of the same operator, following the semiseparable block
 * structure ([Mamba-2 explainer] 第二步 and 关键技术点 1): inside a chunk of Q steps
 * the diagonal block is summed directly,
 *     y_t += sum_{s<=t} C_t[n] exp(A_n (S_t - S_s)) B_s[n] Delta_s x_s,
 * with S the in-chunk inclusive cumulative sum of Delta, and the off-diagonal
 * blocks enter through the state carried across the chunk boundary,
 *     y_t += C_t[n] exp(A_n S_t) h_prev[n],
 *     h_next[n] = exp(A_n S_last) h_prev[n] + sum_s exp(A_n (S_last - S_s)) B_s[n] Delta_s x_s.
 * A different summation order from the sequential recurrence, used to pin that
 * the result does not depend on the chunk length.
 */
static void oracle_channel_chunked(const oracle_problem* p, int64_t b, int64_t h, int64_t q,
                                   int64_t Q, double* state, double* scratch) {
    const int64_t T = p->seqlen, H = p->nheads, P = p->headdim, N = p->dstate, G = p->ngroups;
    const int64_t g = h / (H / G);
    const int64_t sidx = ((b * H + h) * P + q) * N;
    double* delta = scratch;     /* Q */
    double* cum = scratch + Q;   /* Q */
    double* hnext = scratch + 2 * Q; /* N */
    for (int64_t n = 0; n < N; ++n) state[n] = p->initial_state ? p->initial_state[sidx + n] : 0.0;
    for (int64_t c0 = 0; c0 < T; c0 += Q) {
        const int64_t len = (T - c0 < Q) ? (T - c0) : Q;
        double run = 0.0;
        for (int64_t i = 0; i < len; ++i) {
            const int64_t bt = b * T + c0 + i;
            delta[i] = oracle_softplus(p->dt[bt * H + h] + (p->dt_bias ? p->dt_bias[h] : 0.0));
            run += delta[i];
            cum[i] = run;
        }
        for (int64_t i = 0; i < len; ++i) {
            const int64_t bt = b * T + c0 + i;
            const double* Ct = p->C + (bt * G + g) * N;
            double y = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double an = oracle_acoef(p, h, n);
                double acc = exp(an * cum[i]) * state[n];
                for (int64_t s = 0; s <= i; ++s) {
                    const int64_t bs = b * T + c0 + s;
                    const double* Bs = p->B + (bs * G + g) * N;
                    const double xs = p->x[(bs * H + h) * P + q];
                    acc += exp(an * (cum[i] - cum[s])) * Bs[n] * delta[s] * xs;
                }
                y += Ct[n] * acc;
            }
            const int64_t xi = (bt * H + h) * P + q;
            if (p->D) y += p->D[h] * p->x[xi];
            if (p->z) y *= oracle_silu(p->z[xi]);
            p->out[xi] = y;
        }
        for (int64_t n = 0; n < N; ++n) {
            const double an = oracle_acoef(p, h, n);
            double acc = exp(an * cum[len - 1]) * state[n];
            for (int64_t s = 0; s < len; ++s) {
                const int64_t bs = b * T + c0 + s;
                const double* Bs = p->B + (bs * G + g) * N;
                const double xs = p->x[(bs * H + h) * P + q];
                acc += exp(an * (cum[len - 1] - cum[s])) * Bs[n] * delta[s] * xs;
            }
            hnext[n] = acc;
        }
        for (int64_t n = 0; n < N; ++n) state[n] = hnext[n];
    }
    if (p->final_state)
        for (int64_t n = 0; n < N; ++n) p->final_state[sidx + n] = state[n];
}

static int oracle_run(const oracle_problem* p, int64_t chunk, const int64_t* sel, int64_t nsel,
                      int nthreads) {
    int rc = oracle_check(p);
    if (rc) return rc;
    const int64_t H = p->nheads, P = p->headdim, N = p->dstate;
    const int64_t nchan = p->batch * H * P;
    const int64_t count = sel ? nsel : nchan;
    if (sel)
        for (int64_t i = 0; i < nsel; ++i)
            if (sel[i] < 0 || sel[i] >= nchan) return 2;
    const int64_t Q = chunk > 0 ? chunk : 1;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double* state = (double*)malloc(sizeof(double) * (size_t)(N + 2 * Q + N));
        if (!state) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t i = 0; i < count; ++i) {
            if (!state) continue;
            const int64_t ch = sel ? sel[i] : i;
            const int64_t b = ch / (H * P), h = (ch / P) % H, q = ch % P;
            if (chunk > 0)
                oracle_channel_chunked(p, b, h, q, Q, state, state + N);
            else
                oracle_channel_sequential(p, b, h, q, state);
        }
        free(state);
    }
    return failed ? 6 : 0;
}

/*
 * Exported entry points (called through ctypes by the tests and the benchmark's
 * CPU leg).  Return 0 on success, 1 for a missing required pointer, 2 for a bad
 * shape or selection, 6 when a per-thread buffer cannot be allocated.
 *
 * sel / nsel: optional list of flat channel indices b*H*P + h*P + q to evaluate;
 * outputs of channels not listed are left untouched.  nthreads <= 0 keeps the
 * OpenMP default.
 */
int oracle_scan(int mode, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                int64_t dstate, int64_t ngroups, const double* x, const double* dt,
                const double* A, const double* B, const double* C, const double* D,
                const double* z, const double* dt_bias, const double* initial_state,
                double* out, double* final_state, const int64_t* sel, int64_t nsel,
                int nthreads) {
    oracle_problem p = {mode, batch, seqlen, nheads, headdim, dstate, ngroups, x, dt, A, B, C,
                        D, z, dt_bias, initial_state, out, final_state};
    return oracle_run(&p, 0, sel, nsel, nthreads);
}

int oracle_scan_chunked(int mode, int64_t batch, int64_t seqlen, int64_t nheads,
                        int64_t headdim, int64_t dstate, int64_t ngroups, int64_t chunk,
                        const double* x, const double* dt, const double* A, const double* B,
                        const double* C, const double* D, const double* z,
                        const double* dt_bias, const double* initial_state, double* out,
                        double* final_state, const int64_t* sel, int64_t nsel, int nthreads) {
    if (chunk <= 0) return 2;
    oracle_problem p = {mode, batch, seqlen, nheads, headdim, dstate, ngroups, x, dt, A, B, C,
                        D, z, dt_bias, initial_state, out, final_state};
    return oracle_run(&p, chunk, sel, nsel, nthreads);
}

/*
 * Causal depthwise convolution followed by SiLU, per batch b, time t and channel c
 * (channels = nheads * headdim, innermost):
 *   x'[b,t,c] = SiLU( bias[c] + sum_{k=0..K-1} w[c,k] * x[b, t-K+1+k, c] )
 * where x at a time s < 0 is x_prev[b, K-1+s, c] (NULL: zero).  x_last, if given,
 * receives the K-1 inputs that precede time T: x_last[b, j, c] = x at time T-K+1+j
 * (taken from x_prev where that time is negative).
 * Layouts: x, xc (batch, T, channels); w (channels, K); bias (channels,) nullable;
 * x_prev, x_last (batch, K-1, channels) nullable.
 */
int oracle_conv_silu(int64_t batch, int64_t seqlen, int64_t channels, int64_t width,
                     const double* x, const double* w, const double* bias,
                     const double* x_prev, double* xc, double* x_last) {
    if (!x || !w || !xc || batch < 0 || seqlen < 0 || channels <= 0 || width < 1) return 2;
    const int64_t K = width;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t t = 0; t < seqlen; ++t) {
            for (int64_t c = 0; c < channels; ++c) {
                double acc = bias ? bias[c] : 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const int64_t s = t - K + 1 + k;
                    double v = 0.0;
                    if (s >= 0)
                        v = x[(b * seqlen + s) * channels + c];
                    else if (x_prev)
                        v = x_prev[(b * (K - 1) + (K - 1 + s)) * channels + c];
                    acc += w[c * K + k] * v;
                }
                xc[(b * seqlen + t) * channels + c] = oracle_silu(acc);
            }
        }
        if (x_last) {
            for (int64_t j = 0; j < K - 1; ++j) {
                const int64_t s = seqlen - K + 1 + j;
                for (int64_t c = 0; c < channels; ++c) {
                    double v = 0.0;
                    if (s >= 0)
                        v = x[(b * seqlen + s) * channels + c];
                    else if (x_prev)
                        v = x_prev[(b * (K - 1) + (K - 1 + s)) * channels + c];
                    x_last[(b * (K - 1) + j) * channels + c] = v;
                }
            }
        }
    }
    return 0;
}

/*
 * Backward pass of the scan (reverse-mode derivatives), written from the recurrence;
 * the pages give none.  With v_t = dt_t + dt_bias, Delta_t = softplus(v_t),
 * a_t[n] = exp(Delta_t A_n), h_t = a_t h_{t-1} + Delta_t B_t x_t, y_t = C_t.h_t + D x_t,
 * out_t = y_t SiLU(z_t), and the incoming gradients dout (of out) and dfinal (of the
 * final state, nullable), per channel from t = T-1 down to 0:
 *   dy_t     = dout_t SiLU(z_t)                  dz_t += dout_t y_t SiLU'(z_t)
 *   g_t      = dy_t C_t + a_{t+1} g_{t+1}        (g_T-1 starts from dfinal) = dL/dh_t
 *   dx_t    += dy_t D + sum_n g_t[n] Delta_t B_t[n]
 *   dB_t    += g_t Delta_t x_t                   dC_t += dy_t h_t
 *   dDelta_t = sum_n g_t[n] (B_t[n] x_t + a_t[n] A_n h_{t-1}[n])
 *   dA_n    += g_t[n] a_t[n] Delta_t h_{t-1}[n]  dD   += dy_t x_t
 *   ddt_t   += dDelta_t sigmoid(v_t)             ddt_bias += dDelta_t sigmoid(v_t)
 * and dinit = a_0 g_0.  Parameters shared by channels (B, C by group; A, D, dt and
 * dt_bias by head in SSD mode) receive the sum over those channels.  Every output is
 * overwritten (zeroed first).  Each channel keeps its whole state history (T x N).
 * Layouts as the forward; dA as A; ddt as dt; dinit as initial_state.  dz, dD,
 * ddt_bias and dinit may be NULL (not computed); z, D, dt_bias, initial_state and
 * dfinal may be NULL as in the forward.
 */
int oracle_scan_bwd(int mode, int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                    int64_t dstate, int64_t ngroups, const double* x, const double* dt,
                    const double* A, const double* B, const double* C, const double* D,
                    const double* z, const double* dt_bias, const double* initial_state,
                    const double* dout, const double* dfinal, double* dx, double* ddt, double* dA,
                    double* dB, double* dC, double* dD, double* dz, double* ddt_bias,
                    double* dinit) {
    double dummy = 0.0;
    oracle_problem p = {mode, batch, seqlen, nheads, headdim, dstate, ngroups, x, dt, A, B, C,
                        D, z, dt_bias, initial_state, &dummy, NULL};
    int rc = oracle_check(&p);
    if (rc) return rc;
    if (!dout || !dx || !ddt || !dA || !dB || !dC) return 1;
    const int64_t T = seqlen, H = nheads, P = headdim, N = dstate, G = ngroups;
    memset(dx, 0, sizeof(double) * (size_t)(batch * T * H * P));
    memset(ddt, 0, sizeof(double) * (size_t)(batch * T * H));
    memset(dA, 0, sizeof(double) * (size_t)(mode == ORACLE_MODE_DIAG ? H * N : H));
    memset(dB, 0, sizeof(double) * (size_t)(batch * T * G * N));
    memset(dC, 0, sizeof(double) * (size_t)(batch * T * G * N));
    if (dD) memset(dD, 0, sizeof(double) * (size_t)H);
    if (dz) memset(dz, 0, sizeof(double) * (size_t)(batch * T * H * P));
    if (ddt_bias) memset(ddt_bias, 0, sizeof(double) * (size_t)H);
    double* hist = (double*)malloc(sizeof(double) * (size_t)((T + 1) * N));
    double* g = (double*)malloc(sizeof(double) * (size_t)N);
    if (!hist || !g) {
        free(hist);
        free(g);
        return 6;
    }
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t q = 0; q < P; ++q) {
                const int64_t grp = h / (H / G);
                const int64_t sidx = ((b * H + h) * P + q) * N;
                /* forward, keeping h_{t-1} in hist[t] (hist[0] = initial state) */
                for (int64_t n = 0; n < N; ++n) hist[n] = initial_state ? initial_state[sidx + n] : 0.0;
                for (int64_t t = 0; t < T; ++t) {
                    const int64_t bt = b * T + t;
                    const double delta = oracle_softplus(dt[bt * H + h] + (dt_bias ? dt_bias[h] : 0.0));
                    const double xv = x[(bt * H + h) * P + q];
                    const double* Bt = B + (bt * G + grp) * N;
                    for (int64_t n = 0; n < N; ++n)
                        hist[(t + 1) * N + n] = exp(delta * oracle_acoef(&p, h, n)) * hist[t * N + n] + delta * Bt[n] * xv;
                }
                /* reverse */
                for (int64_t n = 0; n < N; ++n) g[n] = dfinal ? dfinal[sidx + n] : 0.0;
                for (int64_t t = T - 1; t >= 0; --t) {
                    const int64_t bt = b * T + t;
                    const int64_t xi = (bt * H + h) * P + q;
                    const double v = dt[bt * H + h] + (dt_bias ? dt_bias[h] : 0.0);
                    const double delta = oracle_softplus(v);
                    const double sig_v = 1.0 / (1.0 + exp(-v));
                    const double xv = x[xi];
                    const double* Bt = B + (bt * G + grp) * N;
                    const double* Ct = C + (bt * G + grp) * N;
                    const double* hprev = hist + t * N;
                    const double* hcur = hist + (t + 1) * N;
                    double y = 0.0;
                    for (int64_t n = 0; n < N; ++n) y += Ct[n] * hcur[n];
                    if (D) y += D[h] * xv;
                    double gate = 1.0;
                    if (z) {
                        const double zv = z[xi];
                        const double sz = 1.0 / (1.0 + exp(-zv));
                        gate = zv * sz;
                        if (dz) dz[xi] = dout[xi] * y * sz * (1.0 + zv * (1.0 - sz));
                    }
                    const double dy = dout[xi] * gate;
                    double dxv = D ? dy * D[h] : 0.0;
                    double ddelta = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        const double an = oracle_acoef(&p, h, n);
                        const double abar = exp(delta * an);
                        g[n] += dy * Ct[n];
                        dxv += g[n] * delta * Bt[n];
                        dB[(bt * G + grp) * N + n] += g[n] * delta * xv;
                        dC[(bt * G + grp) * N + n] += dy * hcur[n];
                        ddelta += g[n] * (Bt[n] * xv + abar * an * hprev[n]);
                        const double da = g[n] * abar * delta * hprev[n];
                        if (mode == ORACLE_MODE_DIAG)
                            dA[h * N + n] += da;
                        else
                            dA[h] += da;
                        g[n] *= abar; /* now dL/dh_{t-1} */
                    }
                    dx[xi] = dxv;
                    if (dD) dD[h] += dy * xv;
                    ddt[bt * H + h] += ddelta * sig_v;
                    if (ddt_bias) ddt_bias[h] += ddelta * sig_v;
                }
                if (dinit)
                    for (int64_t n = 0; n < N; ++n) dinit[sidx + n] = g[n];
            }
    free(hist);
    free(g);
    return 0;
}

/*
 * Complex diagonal scan: the state update of Mamba-3 read as a complex-valued, rotating
 * recurrence.  Sources: [SSM/Mamba primer] "状态空间模型与 Mamba：不用注意力读取长序列的方法",
 * the paragraph on Mamba-3's oscillatory dynamics (an input-dependent rotation in the
 * state update, read as underdamped oscillation); [Mamba / hybrid overview] section 6
 * Mamba-3：新的推理优先视角 (keywords: complex-valued state update, SSM discretization).
 * The pages print no formula.  Reading (listed in the design notes): A[c,n] is complex,
 * Re A the decay rate and Im A the angular frequency; the same discretisation as the
 * real scan, Abar = exp(Delta A) = e^{Delta Re A} (cos(Delta Im A) + i sin(Delta Im A)),
 * so the rotation angle Delta_t Im A follows the input through Delta_t; B and C are
 * complex; the output reads the real part of the plain (unconjugated) product:
 *   h_t[n] = exp(Delta_t A[c,n]) h_{t-1}[n] + Delta_t B_t[n] x_t          (complex)
 *   y_t    = (Re(sum_n C_t[n] h_t[n]) + D x_t) * SiLU(z_t)
 * Layouts (complex numbers as (re, im) pairs of doubles):
 *   x, z, out, dt (batch, seqlen, nheads); A (nheads, dstate, 2); B, C (batch, seqlen,
 *   ngroups, dstate, 2); D, dt_bias (nheads,) nullable; initial_state, final_state
 *   (batch, nheads, dstate, 2) nullable.  sel/nsel: flat channels b*nheads + c.
 */
static void oracle_channel_complex(int64_t T, int64_t H, int64_t N, int64_t G, int64_t b,
                                   int64_t c, const double* x, const double* dt, const double* A,
                                   const double* B, const double* C, const double* D,
                                   const double* z, const double* dt_bias,
                                   const double* initial_state, double* out, double* final_state,
                                   double complex* state) {
    const int64_t g = c / (H / G);
    const int64_t sidx = (b * H + c) * N;
    for (int64_t n = 0; n < N; ++n)
        state[n] = initial_state ? initial_state[2 * (sidx + n)] + I * initial_state[2 * (sidx + n) + 1] : 0.0;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t bt = b * T + t;
        const double delta = oracle_softplus(dt[bt * H + c] + (dt_bias ? dt_bias[c] : 0.0));
        const double xv = x[bt * H + c];
        const double* Bt = B + 2 * (bt * G + g) * N;
        const double* Ct = C + 2 * (bt * G + g) * N;
        double complex acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            const double complex an = A[2 * (c * N + n)] + I * A[2 * (c * N + n) + 1];
            const double complex bn = Bt[2 * n] + I * Bt[2 * n + 1];
            const double complex cn = Ct[2 * n] + I * Ct[2 * n + 1];
            state[n] = cexp(delta * an) * state[n] + delta * bn * xv;
            acc += cn * state[n];
        }
        double y = creal(acc);
        if (D) y += D[c] * xv;
        if (z) y *= oracle_silu(z[bt * H + c]);
        out[bt * H + c] = y;
    }
    if (final_state)
        for (int64_t n = 0; n < N; ++n) {
            final_state[2 * (sidx + n)] = creal(state[n]);
            final_state[2 * (sidx + n) + 1] = cimag(state[n]);
        }
}

int oracle_scan_complex(int64_t batch, int64_t seqlen, int64_t nheads, int64_t dstate,
                        int64_t ngroups, const double* x, const double* dt, const double* A,
                        const double* B, const double* C, const double* D, const double* z,
                        const double* dt_bias, const double* initial_state, double* out,
                        double* final_state, const int64_t* sel, int64_t nsel, int nthreads) {
    if (!x || !dt || !A || !B || !C || !out) return 1;
    if (batch < 0 || seqlen < 0 || nheads <= 0 || dstate <= 0 || ngroups <= 0 || nheads % ngroups) return 2;
    const int64_t nchan = batch * nheads;
    const int64_t count = sel ? nsel : nchan;
    if (sel)
        for (int64_t i = 0; i < nsel; ++i)
            if (sel[i] < 0 || sel[i] >= nchan) return 2;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double complex* state = (double complex*)malloc(sizeof(double complex) * (size_t)dstate);
        if (!state) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t i = 0; i < count; ++i) {
            if (!state) continue;
            const int64_t ch = sel ? sel[i] : i;
            oracle_channel_complex(seqlen, nheads, dstate, ngroups, ch / nheads, ch % nheads, x, dt,
                                   A, B, C, D, z, dt_bias, initial_state, out, final_state, state);
        }
        free(state);
    }
    return failed ? 6 : 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
