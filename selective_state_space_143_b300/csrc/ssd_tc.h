// Tensor-core (tcgen05) SSD chunk kernels: arguments and launchers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

struct SsdTcArgs {
    const __nv_bfloat16* x;     // x, or x_hi of the split convolved input
    const __nv_bfloat16* x_lo;  // null, or x_lo: x' = x_hi + x_lo
    const __nv_bfloat16* dt;
    const __nv_bfloat16* z;
    const __nv_bfloat16* B;
    const __nv_bfloat16* C;
    const float* A;
    const float* D;
    const float* dt_bias;
    __nv_bfloat16* out;
    float* dl;      // (b, H, nchunks, Q) Delta
    float* cum;     // (b, H, nchunks, Q) inclusive cumsum of Delta*A_h within the chunk
    float* states;  // (b, nchunks, H, P, N): S_c, then (after the carry pass) h_{c-1}
    int64_t T, H, N, G, Q, nchunks;
    // byte ranges of the buffers written (stores checked in SSM_BOUNDS_CHECK builds)
    Span out_s, dl_s, cum_s, states_s;
};

// True when the shape is one the tensor-core kernels take (bf16, headdim 64,
// dstate 64, 128 or 256, chunk 128 or 256, even heads per group).
bool ssd_tc_supported(const ScanArgs& a, int64_t Q);

// S_c for every (chunk, head) into states; also writes dl and cum.
cudaError_t ssd_tc_chunk_state(const SsdTcArgs& s, int64_t batch, cudaStream_t stream);

// Adjoint chunk states of the backward pass, S^g_c = sum_t exp(cum_t) dy_t C_t^T for
// every (chunk, head) into states (split-ready layout), with x / x_lo the hi / lo planes
// of dy (x_lo null when dy is exact in bf16) and B the C rows; reads dt for the weights,
// writes neither dl nor cum.  dstate 64 or 128.
cudaError_t ssd_tc_chunk_state_adjoint(const SsdTcArgs& s, int64_t batch, cudaStream_t stream);

// out for every chunk, reading h_{c-1} from states (after the carry pass).
cudaError_t ssd_tc_chunk_scan(const SsdTcArgs& s, int64_t batch, bool gate, cudaStream_t stream);

// The tensor-core path's carry over chunks of length Q (states in the split-ready layout
// of ssd_tc_chunk_state, rewritten in place as h_{c-1} bf16 hi/lo tiles), from
// a.initial_state; final_state (b, H, P, N) fp32 or null.
cudaError_t ssd_tc_forward_carry(const ScanArgs& a, int64_t Q, int64_t nchunks, const float* cum, float* states,
                                 float* final_state, cudaStream_t stream);

// Backward pass of the SSD scan in chunk form on the tensor cores (ssd_bwd_tc.cu): bf16,
// headdim 64, dstate 64 or 128, the tensor-core forward's head grouping, no convolution.
bool ssd_bwd_tc_supported(const ScanArgs& a);
size_t ssd_bwd_tc_workspace_bytes(const ScanArgs& a);
// Every gradient of ScanBwdArgs; dA, dB, dC, dD and ddt_bias must be zero on entry (they
// are accumulated); dx, ddt, dz and dinit are written.
cudaError_t ssd_bwd_tc_launch(const ScanBwdArgs& s, void* ws, cudaStream_t stream);

}  // namespace ssm
