// Internal interface between the C-ABI entry points and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssm {

// Everything a launcher needs, already validated by the entry point.
struct ScanArgs {
    const void* x;
    const void* dt;
    const float* A;
    const void* B;
    const void* C;
    const float* D;
    const void* z;
    const float* dt_bias;
    const float* initial_state;  // nullable: state entering t = 0 (zero when NULL)
    // causal depthwise convolution + SiLU applied to x ahead of the scan (conv_k 0: none)
    const float* conv_w;         // (channels, conv_k)
    const float* conv_b;         // (channels,) nullable
    const void* x_prev;          // (batch, conv_k-1, channels) nullable: inputs before t = 0
    void* x_last;                // (batch, conv_k-1, channels) nullable: last inputs, written
    int conv_k;
    int x_f32;                   // x is stored as fp32 whatever dtype says (the convolved
                                 // input on the CUDA-core SSD kernels)
    const void* x_lo;            // nullable: x is bf16 x_hi (at x) + x_lo (here), the
                                 // convolved input on the tensor-core SSD kernels
    void* out;
    float* final_state;
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk;
    int dtype;  // 0 fp32, 1 bf16
};

// Launch bookkeeping.  Around every kernel launch:
//   cudaEvent_t t0 = timing_begin(stream, "name");  kernel<<<...>>>(...);  note_launch("name", stream, t0);
// timing_begin opens an NVTX range named after the kernel on the calling thread (so a
// profiler can select a launch by range, e.g. ncu --nvtx --nvtx-include "ssd_scan_tc/")
// and note_launch closes it; a launcher that gives up between the two calls
// launch_failed instead.  note_launch counts the launch; when timing is enabled
// (ssm_timing_enable) timing_begin records an event before the launch and note_launch one
// after it, on the same stream, for ssm_timing_collect.
cudaEvent_t timing_begin(cudaStream_t stream, const char* name);
void note_launch(const char* name, cudaStream_t stream, cudaEvent_t start);
void launch_failed(cudaEvent_t start);

// Diagonal (Mamba-1) path.
size_t diag_workspace_bytes(const ScanArgs& a);
cudaError_t diag_launch(const ScanArgs& a, void* ws, cudaStream_t stream);

// Complex diagonal path (the rotating state update read for Mamba-3): A (nheads, dstate, 2),
// B/C (batch, seqlen, ngroups, dstate, 2), states (batch, nheads, dstate, 2).
size_t cdiag_workspace_bytes(const ScanArgs& a);
cudaError_t cdiag_launch(const ScanArgs& a, void* ws, cudaStream_t stream);

// SSD (Mamba-2) path.
size_t ssd_workspace_bytes(const ScanArgs& a);
cudaError_t ssd_launch(const ScanArgs& a, void* ws, cudaStream_t stream);
// True when the SSD launcher takes the convolved input of this shape on the tensor-core
// kernels, i.e. as bf16 hi/lo planes (else as fp32, on the CUDA-core kernels).
bool ssd_conv_split(const ScanArgs& a);

// Single-token step: the state (batch, nheads, headdim, dstate) is updated in place and
// out (batch, nheads, headdim) written; diag_a selects A of shape (nheads, dstate).
cudaError_t step_launch(const ScanArgs& a, bool diag_a, float* state, cudaStream_t stream);

// Backward pass of the scan: the forward arguments plus the incoming gradients and the
// gradient outputs (fp32; dA, dB, dC, dD and ddt_bias, and in SSD mode ddt, are zeroed,
// then summed).
struct ScanBwdArgs {
    ScanArgs fwd;
    bool ssd;  // SSD mode: A, Delta, D and dt_bias per head
    const void* dout;
    const float* dfinal;
    float *dx, *ddt, *dA, *dB, *dC, *dD, *dz, *ddt_bias, *dinit;
};
size_t scan_bwd_workspace_bytes(const ScanArgs& a, bool ssd);
cudaError_t scan_bwd_launch(const ScanBwdArgs& s, void* ws, cudaStream_t stream);

// Convolution + SiLU of x into xc, and the last conv_k-1 inputs into a.x_last; used
// ahead of the SSD kernels.  x' keeps fp32 precision: it is an intermediate, and
// rounding it to bf16 would add an input error the scan's tolerance does not allow.  xc
// holds either fp32 x' (split false) or two bf16 planes of the same total size, x_hi =
// bf16(x') followed by x_lo = bf16(x' - x_hi) (split true), so that x_hi + x_lo carries
// 16 significant bits into bf16 tensor-core products.
cudaError_t conv_prepass_launch(const ScanArgs& a, void* xc, bool split, cudaStream_t stream);
cudaError_t conv_tail_launch(const ScanArgs& a, cudaStream_t stream);

// Per-device status word of bounded device-side waits and bounds checks: read into
// *status (0, SSM_ERR_TIMEOUT or SSM_ERR_BOUNDS) after the stream's work, cleared when
// `clear`.
cudaError_t device_status_take(int* status, bool clear, cudaStream_t stream);
// Device address of that status word for the current device (looked up once per device),
// for kernels in other translation units, which record SSM_ERR_TIMEOUT through it.
cudaError_t device_status_address(int** p);
// One CTA waiting on an mbarrier that nothing completes, giving up after max_checks polls.
cudaError_t bounded_wait_selftest_launch(uint32_t max_checks, cudaStream_t stream);
// One thread storing to buf + index * 4 through the bounds check against [buf, buf + bytes).
cudaError_t bounds_selftest_launch(float* buf, size_t bytes, int64_t index, cudaStream_t stream);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Streaming multiprocessors of the current device, read once per device and cached
// (148 when no device is visible, so that workspace queries still answer on a host
// without a GPU).  Schedules that size their grids to fill the GPU use this.
int sm_count();

// Plan overrides set through ssm_tuning_set (0 = the library's own choice).  Indexed by
// the ssm_tuning_knob values of include/ssm_scan.h.
int64_t tuning(int knob);

// Stream-ordered scratch allocation for the entry points that allocate.  Reports
// failure (and allocates nothing) while an injected failure is pending
// (ssm_inject_alloc_failures).
cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream);

}  // namespace ssm
