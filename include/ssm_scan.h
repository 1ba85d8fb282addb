/*
 * ssm_scan.h -- C ABI of the B300 selective state-space scan library (libssmscan.so).
 *
 * The operation (cited by web-page title and section):
 *   "Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里", 背景问题 / 第一步:
 *       h_t = Abar_t h_{t-1} + Bbar_t x_t,  y_t = C_t h_t,  Delta_t = softplus(.),
 *       Abar from Delta (selective, input-dependent parameters);
 *   "引言：Attention的天花板" (SSM engineering article), 基本原理: y = C h + D x;
 *   "论文解读：Mamba — 线性时间的序列建模革命", 五 Mamba块架构: y * SiLU(z);
 *   "Mamba-2 ..." explainer, 第二步 / 关键技术点 1-3: with A scalar per head the same
 *       operator is y = (L o M) x with a semiseparable M, evaluated in chunks by
 *       matrix multiplications (the SSD form).
 * Discretisation: Abar = exp(Delta * A), Bbar = Delta * B, with
 *   Delta = softplus(dt + dt_bias) = ln(1 + exp(dt + dt_bias)).
 * Per channel c (SSD: c = (head h, p), A_c = A_h, Delta_c = Delta_h), group g:
 *   h_t[n] = exp(Delta_t A[c,n]) h_{t-1}[n] + Delta_t B_t[g,n] x_t[c]
 *   out_t[c] = (sum_n C_t[g,n] h_t[n] + D[c] x_t[c]) * SiLU(z_t[c])
 * with h_{-1} = 0, D and the gate optional.  final_state = h_{T-1}.
 *
 * Layouts: row-major, contiguous, token-major (channels innermost).
 *   mode DIAG (Mamba-1, A per channel and state):
 *     x, z, out : (batch, seqlen, nheads)        nheads = d_inner, headdim must be 1
 *     dt        : (batch, seqlen, nheads)
 *     A         : (nheads, dstate) fp32
 *     D, dt_bias: (nheads,) fp32
 *     final_state: (batch, nheads, dstate) fp32
 *   mode SSD (Mamba-2, scalar A per head):
 *     x, z, out : (batch, seqlen, nheads, headdim)
 *     dt        : (batch, seqlen, nheads)
 *     A, D, dt_bias: (nheads,) fp32
 *     final_state: (batch, nheads, headdim, dstate) fp32
 *   mode CDIAG (complex diagonal A: the rotating, complex-valued state update read for
 *   Mamba-3 -- "状态空间模型与 Mamba：不用注意力读取长序列的方法", the Mamba-3 paragraph: an
 *   input-dependent rotation in the state update, read as underdamped oscillation;
 *   "基础知识：Mamba 与混合 SSM 架构", 6 Mamba-3: complex-valued state update):
 *     h_t[n] = exp(Delta_t A[c,n]) h_{t-1}[n] + Delta_t B_t[g,n] x_t[c]   (complex)
 *     out_t[c] = (Re(sum_n C_t[g,n] h_t[n]) + D[c] x_t[c]) * SiLU(z_t[c])
 *     with exp(Delta A) = e^{Delta Re A} (cos(Delta Im A) + i sin(Delta Im A)); every
 *     complex number is stored as an (re, im) pair:
 *     x, z, out, dt, D, dt_bias as DIAG (headdim must be 1);
 *     A          : (nheads, dstate, 2) fp32
 *     B, C       : (batch, seqlen, ngroups, dstate, 2) in the input dtype
 *     final_state, initial_state: (batch, nheads, dstate, 2) fp32
 *     dstate (complex entries) 1..32, dstate*2 elements a multiple of 16 bytes; chunk: 0
 *     or the time-segment length (multiple of 16).  Supported by ssm_scan_fwd, _ws,
 *     _noalloc and _state; the convolution, step and backward entry points return
 *     SSM_ERR_UNSUPPORTED for it.
 *   DIAG and SSD: B, C : (batch, seqlen, ngroups, dstate); head h reads group
 *   h / (nheads/ngroups).
 *   SSD also needs headdim * dstate to be a multiple of 4 (the state moves in 16-byte
 *   pieces).
 *   x, dt, B, C, z and out share the element type `dtype` (fp32 or bf16; bf16 output
 *   is rounded to nearest even).  State and accumulation are fp32.
 *
 * Ownership: every pointer is device memory owned by the caller; the library keeps
 * no reference after the call returns.  Calls are asynchronous on `stream`; results
 * are valid after the caller synchronises with it.  Kernel faults surface at that
 * synchronisation, not in the return value.
 *
 * Errors: every argument is checked on the host before any work is queued; on an
 * error nothing is launched and the status says why (see ssm_strerror).  There is
 * no CPU fallback: without a usable CUDA device the call returns SSM_ERR_CUDA.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SSM_OK = 0,
    SSM_ERR_NULL = 1,        /* a required pointer is NULL                          */
    SSM_ERR_SHAPE = 2,       /* a size is out of range or inconsistent              */
    SSM_ERR_DTYPE = 3,       /* unknown mode or dtype                                */
    SSM_ERR_ALIGN = 4,       /* a pointer or a row is not 16-byte aligned            */
    SSM_ERR_UNSUPPORTED = 5, /* valid but unsupported (dstate too large, flags != 0) */
    SSM_ERR_ALLOC = 6,       /* workspace allocation failed or workspace too small   */
    SSM_ERR_CUDA = 7,        /* a CUDA call failed (launch error, no device)         */
    SSM_ERR_TIMEOUT = 8,     /* a bounded device-side wait ran out (ssm_device_status) */
    SSM_ERR_BOUNDS = 9       /* a store address fell outside its buffer: builds with
                                SSM_BOUNDS_CHECK only (ssm_device_status)              */
} ssm_status;

typedef enum { SSM_MODE_DIAG = 0, SSM_MODE_SSD = 1, SSM_MODE_CDIAG = 2 } ssm_mode;
typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

typedef struct ssm_shape {
    int32_t mode;     /* ssm_mode                                                        */
    int32_t dtype;    /* ssm_dtype of x, dt, B, C, z, out                                */
    int64_t batch;    /* >= 0                                                            */
    int64_t seqlen;   /* >= 0                                                            */
    int64_t nheads;   /* DIAG: d_inner; SSD: heads; >= 1                                 */
    int64_t headdim;  /* DIAG: 1; SSD: channels per head, 1..256                         */
    int64_t dstate;   /* N: DIAG 1..64; SSD 1..256; CDIAG 1..32 complex entries          */
    int64_t ngroups;  /* >= 1, divides nheads                                            */
    int64_t chunk;    /* 0 = default.  DIAG: time-segment length (multiple of 32) used to
                         split the sequence across thread blocks; SSD: chunk length Q
                         (multiple of 16, <= 256).  Results agree within rounding for any
                         valid value.                                                    */
    uint32_t flags;   /* reserved, must be 0                                             */
} ssm_shape;

/* A cudaStream_t passed as an opaque handle (NULL = the legacy default stream). */
typedef struct CUstream_st* ssm_stream_t;

/*
 * Forward scan.  x, dt, A, B, C and out are required (x, dt, B, C, out may be NULL
 * when batch or seqlen is 0, since they then hold no elements); D, z, dt_bias and
 * final_state may be NULL (no skip term, no gate, no bias, no final state written).
 * With seqlen 0 and batch > 0 the final state is written as zeros.
 * Alignment: every non-NULL pointer 16-byte aligned, and the innermost row of x/z/out
 * (DIAG: nheads elements; SSD: nheads*headdim elements) and of B/C (ngroups*dstate)
 * a multiple of 16 bytes.
 * Workspace: when the chosen schedule needs device scratch (see
 * ssm_scan_workspace_size) this call takes it from the stream-ordered allocator
 * (cudaMallocAsync / cudaFreeAsync on `stream`); SSM_ERR_ALLOC if that fails.
 * Returns an ssm_status.
 */
int ssm_scan_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* dt_bias, void* out,
                 float* final_state, const ssm_shape* shape, ssm_stream_t stream);

/* Bytes of device scratch the call needs for `shape` (0 when none; (size_t)-1 when the
 * shape is invalid).  Depends on the shape, the current device's SM count (the
 * schedule fills the GPU; 148 is assumed when no device is visible) and the plan
 * overrides of ssm_tuning_set. */
size_t ssm_scan_workspace_size(const ssm_shape* shape);

/*
 * As ssm_scan_fwd, with caller-provided scratch: `workspace` (device, 256-byte aligned)
 * of at least ssm_scan_workspace_size(shape) bytes; it may be NULL when that size is 0.
 * The workspace must not be used by anything else until the call's work on `stream`
 * has finished.  SSM_ERR_ALLOC if it is too small.
 */
int ssm_scan_fwd_ws(const void* x, const void* dt, const float* A, const void* B, const void* C,
                    const float* D, const void* z, const float* dt_bias, void* out,
                    float* final_state, const ssm_shape* shape, void* workspace,
                    size_t workspace_bytes, ssm_stream_t stream);

/*
 * As ssm_scan_fwd, but the call allocates no device memory.  (This entry point has
 * no counterpart in the papers: it is a deployment variant of the same scan.)
 * It is for callers that must not allocate during a scan -- for example an
 * application that reserves all device memory up front for its own allocator, or a
 * latency-critical loop where an allocation could synchronise the device or fail
 * under memory pressure.  Inputs and outputs are passed as for ssm_scan_fwd.
 * Scratch: a fixed 64 MiB device array inside the library, held by every GPU that
 * uses it until the process exits.  Shapes whose scratch
 * (ssm_scan_workspace_size) exceeds 64 MiB are rejected with SSM_ERR_ALLOC before
 * anything is queued; shapes that need no scratch always run.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before any
 * stream capture.  Every call shares the one array per device, so calls that can
 * overlap on the GPU (different streams, or host threads without ordering) race on
 * it; order them on one stream.  Nothing in the array needs clearing between calls.
 */
int ssm_scan_fwd_noalloc(const void* x, const void* dt, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* dt_bias,
                         void* out, float* final_state, const ssm_shape* shape,
                         ssm_stream_t stream);

/*
 * Forward scan that starts from a given state instead of zero: h_{-1} = initial_state.
 * Together with final_state this lets a long sequence be scanned in pieces, each call
 * resuming where the previous one stopped (the recurrent form needs only the previous
 * state: "Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里", 背景问题; the
 * streaming example of "引言：Attention的天花板" passes the state between calls).
 * Arguments as ssm_scan_fwd, plus:
 *   initial_state: NULL (start from zero) or device fp32 of the final_state layout
 *     (DIAG (batch, nheads, dstate); SSD (batch, nheads, headdim, dstate)), 16-byte
 *     aligned.  It must not overlap final_state (SSM_ERR_SHAPE): with the sequence split
 *     across thread blocks, some blocks read it after others have written the final
 *     state.  With seqlen 0 the final state is a copy of the initial state.
 *   workspace, workspace_bytes: both NULL/0 to draw scratch from the stream-ordered
 *     allocator as ssm_scan_fwd does; otherwise caller scratch as for ssm_scan_fwd_ws.
 */
int ssm_scan_fwd_state(const void* x, const void* dt, const float* A, const void* B, const void* C,
                       const float* D, const void* z, const float* dt_bias,
                       const float* initial_state, void* out, float* final_state,
                       const ssm_shape* shape, void* workspace, size_t workspace_bytes,
                       ssm_stream_t stream);

/*
 * One token of recurrent decoding for a batch of sequences, the state carried in place:
 *   Delta = softplus(dt + dt_bias); h <- exp(Delta A) h + Delta B x;
 *   out = (C . h + D x) * SiLU(z)
 * (the recurrent form of "Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里",
 * 背景问题: constant memory per generated token).  The result equals ssm_scan_fwd_state
 * over a sequence of length 1 with initial_state = state, final_state = state.
 *   shape: as for the scan with seqlen == 1 (SSM_ERR_SHAPE otherwise); chunk is not used
 *     beyond the scan's checks; dstate must be a multiple of 4 (SSM_ERR_ALIGN).
 *   x, z, out: (batch, nheads, headdim) (DIAG: headdim 1); dt: (batch, nheads);
 *   B, C: (batch, ngroups, dstate); A, D, dt_bias as for the scan.
 *   state: device fp32, (batch, nheads, headdim, dstate) (DIAG: (batch, nheads, dstate)),
 *     read and overwritten with the new state.  It must not overlap out (SSM_ERR_SHAPE).
 * Needs no scratch and allocates nothing.  Calls on one stream apply in order, so a
 * loop of calls is a decode of one token per call.
 */
int ssm_step(const void* x, const void* dt, const float* A, const void* B, const void* C,
             const float* D, const void* z, const float* dt_bias, float* state, void* out,
             const ssm_shape* shape, ssm_stream_t stream);

/*
 * Causal depthwise convolution + SiLU applied to x ahead of the scan: the x branch of the
 * Mamba block runs Conv1d, then SiLU, then the selective SSM ("论文解读：Mamba — 线性时间的
 * 序列建模革命", 五 Mamba块架构; "基础知识：Mamba 与混合 SSM 架构", 3 Mamba block 里发生了
 * 什么: a depthwise convolution adds local context; width d_conv = 4 in the example of
 * "引言：Attention的天花板", 工程实践).  With channels = nheads * headdim (x's innermost
 * dimensions) and K = width:
 *   x'[b,t,c] = SiLU( bias[c] + sum_{k=0..K-1} weight[c,k] * x[b, t-K+1+k, c] )
 * so weight[c, K-1] multiplies the current input.  x at times before 0 is x_prev (or
 * zero).  The scan then uses x' wherever it uses x, the skip term D*x' included.
 */
typedef struct ssm_conv {
    const float* weight; /* (channels, width) fp32, required                               */
    const float* bias;   /* (channels,) fp32, or NULL for none                              */
    const void* x_prev;  /* (batch, width-1, channels) in the input dtype: the inputs that
                            precede this call's first token, oldest first; NULL = zeros    */
    void* x_last;        /* (batch, width-1, channels) in the input dtype, or NULL: receives
                            the width-1 raw inputs before the end of this call, the x_prev
                            of a following call                                             */
    int32_t width;       /* K, 1..4 (SSM_ERR_UNSUPPORTED otherwise)                        */
} ssm_conv;

/*
 * Forward scan with the convolution ahead of it; otherwise as ssm_scan_fwd_state
 * (initial_state nullable; workspace NULL/0 = stream-ordered allocation).
 * Diagonal mode fuses the convolution into the scan kernels (x is read once).  SSD mode
 * runs it as a separate pass into scratch that the SSD kernels then read, with x' kept in
 * fp32 (rounding it to bf16 would exceed the scan's tolerance); the SSD kernels that read
 * an fp32 x are the CUDA-core ones, slower than the tensor-core kernels used otherwise.
 * Its scratch is ssm_scan_conv_workspace_size(shape).
 * All conv pointers 16-byte aligned.  x_last must not overlap x_prev, x or out
 * (SSM_ERR_SHAPE): thread blocks still reading them may run after it is written.
 */
int ssm_scan_fwd_conv(const void* x, const void* dt, const float* A, const void* B, const void* C,
                      const float* D, const void* z, const float* dt_bias, const ssm_conv* conv,
                      const float* initial_state, void* out, float* final_state,
                      const ssm_shape* shape, void* workspace, size_t workspace_bytes,
                      ssm_stream_t stream);

/* Scratch bytes of ssm_scan_fwd_conv for `shape` ((size_t)-1 when the shape is invalid). */
size_t ssm_scan_conv_workspace_size(const ssm_shape* shape);

/*
 * ssm_step with the convolution ahead of it: x' is formed from the width-1 carried inputs
 * in conv->x_prev and this token's x, and conv->x_last (if non-NULL) receives the carried
 * inputs shifted by one token.  x_last may be the same pointer as x_prev (the state is then
 * updated in place) but must not otherwise overlap it, state, out or x (SSM_ERR_SHAPE).
 */
int ssm_step_conv(const void* x, const void* dt, const float* A, const void* B, const void* C,
                  const float* D, const void* z, const float* dt_bias, const ssm_conv* conv,
                  float* state, void* out, const ssm_shape* shape, ssm_stream_t stream);

/*
 * Backward pass of the scan (both modes): the gradients of every input from the
 * gradient of out (and, optionally, of the final state).  The pages give the forward
 * recurrence only ("Mamba-2：把状态空间模型和 Attention 统一到一个数学框架里", 背景问题 and
 * 第一步; training runs the recurrence in parallel, "训练时并行化"); the derivatives are
 * taken from it, per channel from the last step to the first, with g_t = dL/dh_t:
 *   dy_t = dout_t SiLU(z_t);  g_t = dy_t C_t + exp(Delta_{t+1} A) g_{t+1};
 *   dx_t = dy_t D + sum_n g_t Delta_t B_t;  dB_t += g_t Delta_t x_t;  dC_t += dy_t h_t;
 *   ddt_t = sigmoid(dt_t + dt_bias) sum_n g_t (B_t x_t + exp(Delta_t A) A h_{t-1});
 *   dA += g_t exp(Delta_t A) Delta_t h_{t-1};  dD += dy_t x_t;  ddt_bias += ddt_t;
 *   dz_t = dout_t y_t SiLU'(z_t);  dinitial_state = exp(Delta_0 A) g_0.
 * In SSD mode a channel is (head, p) and A, Delta, D and dt_bias belong to the head
 * (the same page, 第二步), so their gradients sum over the head's channels (dA also over
 * n).  Shapes and forward arguments as ssm_scan_fwd_state (initial_state nullable).
 *   dout: the gradient of out, x's layout and dtype (required unless batch or seqlen is 0);
 *   dfinal_state: gradient of the final state, fp32, the final state's layout
 *     (DIAG (batch, nheads, dstate); SSD (batch, nheads, headdim, dstate)), or NULL (zero).
 * Outputs, all fp32 and in the layout of the matching input: dx, ddt (required; SSD
 * (batch, seqlen, nheads)), dA (required; DIAG (nheads, dstate), SSD (nheads,)), dB, dC
 * (required; (batch, seqlen, ngroups, dstate)), dD, dz, ddt_bias, dinitial_state (NULL:
 * not computed; dD, dz and ddt_bias are also skipped when D, z or dt_bias is NULL).
 * dA, dB, dC, dD and ddt_bias (and, in SSD mode, ddt) are sums over channels and batch:
 * the call zeroes them first.  No output may overlap an input or another output.
 * Scratch: ssm_scan_bwd_workspace_size(shape) bytes: the state every 8 steps in diagonal
 * mode (16 for dstate 8 or less), every 16 in SSD mode (4 for dstate above 64); with few
 * channels the sequence is also cut into up to 16 time parts, each with
 * a local end state, a local adjoint and a Delta sum.  Workspace NULL/0 draws it from
 * the stream-ordered allocator, as ssm_scan_fwd does.
 * The sums over channels use floating-point atomics, so dA, dB, dC, dD and ddt_bias (and
 * SSD's ddt) may differ between runs in the last bits.
 */
int ssm_scan_bwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* dt_bias, const float* initial_state,
                 const void* dout, const float* dfinal_state, float* dx, float* ddt, float* dA,
                 float* dB, float* dC, float* dD, float* dz, float* ddt_bias,
                 float* dinitial_state, const ssm_shape* shape, void* workspace,
                 size_t workspace_bytes, ssm_stream_t stream);

/* Scratch bytes of ssm_scan_bwd ((size_t)-1 for an invalid shape). */
size_t ssm_scan_bwd_workspace_size(const ssm_shape* shape);

/*
 * Launch timing, for measurement (this has no counterpart in the pages: it instruments
 * the library's own launches).  While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on the launch's own stream;
 * ssm_timing_collect waits for the recorded events, fills `out` (up to `max_entries`,
 * sorted by name) with each kernel's launch count and summed device time in
 * milliseconds, clears the records and returns the number of distinct kernels (which
 * may exceed max_entries; out may be NULL), or -SSM_ERR_CUDA if an event failed.
 * Enabling adds two event records per launch; the library's results do not change.
 * Process-wide; thread-safe.
 */
typedef struct ssm_kernel_time {
    char name[64];     /* kernel name and role, NUL-terminated */
    int64_t launches;  /* launches recorded since the last collect */
    double total_ms;   /* summed event-to-event time of those launches */
} ssm_kernel_time;
void ssm_timing_enable(int on);
int ssm_timing_collect(ssm_kernel_time* out, int max_entries);

/*
 * Device-side wait status (this has no counterpart in the pages: it is how the library's
 * own kernels report a wait that did not end).  The tensor-core SSD kernels wait on
 * mbarriers for their MMAs; every such wait is bounded (about one second, or 2^24
 * polls), and a kernel whose wait ran out records SSM_ERR_TIMEOUT in a per-device status
 * word, releases its tensor memory and returns, so the context stays usable and its
 * outputs are not valid.  Launches are asynchronous, so the entry points cannot return
 * this status themselves: ssm_device_status synchronizes `stream`, then returns SSM_OK,
 * SSM_ERR_TIMEOUT or SSM_ERR_BOUNDS (below) for the current device (SSM_ERR_CUDA if the
 * read fails), and clears the word when `clear` is non-zero.  The first code a kernel
 * records stays until cleared.
 *
 * Bounds-checked build (compiled with -DSSM_BOUNDS_CHECK; the debugging stand-in for a
 * memory checker): every kernel checks the address of each global store against the
 * byte range of the buffer it writes (derived from the shape); an address outside it is
 * not written and SSM_ERR_BOUNDS is recorded in the same status word.  The kernels do
 * not trap.  Normal builds compile the checks away.
 */
int ssm_device_status(int clear, ssm_stream_t stream);

/* 1 if this library was built with SSM_BOUNDS_CHECK, else 0. */
int ssm_bounds_check_enabled(void);

/*
 * Self-test of the bounds-check path: one thread stores to buf[index] through the check
 * against [buf, buf + bytes); with index * 4 >= bytes the store is skipped and
 * SSM_ERR_BOUNDS recorded (read it with ssm_device_status).  buf is a device buffer
 * owned by the caller that must hold element `index` either way, so the address stays
 * valid whatever the check does.  SSM_ERR_UNSUPPORTED in builds without the checks,
 * SSM_ERR_NULL for a NULL buf, SSM_ERR_SHAPE for index < 0 or bytes not a multiple of 4.
 */
int ssm_selftest_bounds(float* buf, size_t bytes, int64_t index, ssm_stream_t stream);

/*
 * Self-test of the bounded-wait path: one thread block waits on an mbarrier that expects
 * an arrival nothing makes, gives up after `max_checks` polls (at most one second) and
 * records SSM_ERR_TIMEOUT in the status word, exactly as the SSD kernels would.  Returns
 * SSM_OK once launched on `stream` (SSM_ERR_CUDA on a launch error); read the outcome
 * with ssm_device_status.
 */
int ssm_selftest_bounded_wait(uint32_t max_checks, ssm_stream_t stream);

/*
 * Plan overrides for measurement sweeps (this has no counterpart in the pages: it
 * selects among the library's own kernel schedules; results agree within rounding for
 * every setting, within the stated error for SSM_TUNE_DIAG_EXP_POLY).  Process-wide, thread-safe; 0 restores the library's own choice.
 * A setting changes the scratch size that the *_workspace_size queries report, so query
 * after setting it.  Values out of a knob's range are ignored by the planner.
 *   SSM_TUNE_DIAG_NPT       state entries per lane of the diagonal scan: 4 or 8
 *   SSM_TUNE_SSD_CUDA_CORES 1: run SSD on the CUDA-core kernels (a cross-check of the
 *                           tensor-core ones)
 *   SSM_TUNE_BWD_PARTS      time parts of the backward pass, 1..16
 *   SSM_TUNE_BWD_LPC        lanes per channel of the backward pass: 4, 8, 16 or 32
 *   SSM_TUNE_DIAG_EXP_POLY  diagonal scan, bf16 with dstate <= 16 and no convolution: of
 *                           each 4 state entries per step, the decays of 1 or 2 pairs from
 *                           a polynomial exp2 on the FMA pipe instead of the SFU (results
 *                           agree within the polynomial's 2.5e-7 relative error)
 * ssm_tuning_set returns SSM_ERR_UNSUPPORTED for an unknown knob and SSM_ERR_SHAPE for a
 * negative value; ssm_tuning_get returns the current setting (0 for an unknown knob).
 */
typedef enum {
    SSM_TUNE_DIAG_NPT = 0,
    SSM_TUNE_SSD_CUDA_CORES = 1,
    SSM_TUNE_BWD_PARTS = 2,
    SSM_TUNE_BWD_LPC = 3,
    SSM_TUNE_DIAG_EXP_POLY = 4
} ssm_tuning_knob;
int ssm_tuning_set(int knob, int64_t value);
int64_t ssm_tuning_get(int knob);

/*
 * Host-side fault injection for tests (this has no counterpart in the pages): the next
 * `count` device-scratch allocations made by the entry points that allocate
 * (ssm_scan_fwd, ssm_scan_fwd_state/_conv and ssm_scan_bwd with no workspace) report
 * failure without allocating, so those calls return SSM_ERR_ALLOC with nothing queued.
 * 0 clears pending failures.  Process-wide.
 */
void ssm_inject_alloc_failures(int count);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* ssm_strerror(int status);

/* Number of kernels this library has launched in the calling process so far.  Used to
 * count launches inside a timed region.  Thread-safe. */
uint64_t ssm_kernel_launch_count(void);

/* Library ABI version: (major << 16) | minor. */
int ssm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
