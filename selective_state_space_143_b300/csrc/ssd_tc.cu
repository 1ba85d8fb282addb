// Support code of the tensor-core SSD kernels (ssd_state_tc.cu, ssd_scan_tc.cu): the
// shape check that routes a call to them, the per-device status word through which their
// bounded device-side waits report a wait that ran out, and the self-test of that path.
//
// Shapes taken by the tensor-core kernels: bf16, headdim 64, dstate 64, 128 or 256, chunk
// 128 or 256, an even number of heads per group.  Other shapes use the CUDA-core kernels
// (ssd_scan.cu).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "ssm_device.cuh"
#include "ssm_internal.h"
#include "ssd_tc.h"
#include "tc_util.cuh"

namespace ssm {

namespace {

constexpr int kP = 64;  // headdim handled by the tensor-core kernels
constexpr int kStatusTimeout = 8;

}  // namespace

// Per-device status word: a kernel that gave up a bounded wait records SSM_ERR_TIMEOUT
// here (and returns instead of hanging), a store that failed its bounds check (builds
// with SSM_BOUNDS_CHECK) SSM_ERR_BOUNDS; the host reads and clears it through
// device_status_take (ssm_device_status).
__device__ int g_device_status = 0;

namespace {

__device__ __forceinline__ void report_timeout() { atomicExch(&g_device_status, kStatusTimeout); }

// One CTA waits on an mbarrier that expects one arrival which nothing makes, giving up
// after max_checks polls: the bounded-wait path of the tensor-core kernels, on demand.
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

// One thread stores to buf[index] through the bounds check against [buf, buf + bytes):
// the check's path (record the status, skip the store) on demand.  The caller's buffer
// holds index, so the address is valid either way.
__global__ void bounds_selftest(float* buf, Span s, int64_t index) {
    float* p = buf + index;
    if (span_ok(s, p, 4, &g_device_status)) *p = 1.0f;
}

}  // namespace

// ---- host side -----------------------------------------------------------------

bool ssd_tc_supported(const ScanArgs& a, int64_t Q) {
    const int64_t hpg = a.nheads / a.ngroups;
    // the scan kernel's tensor maps take 32-bit coordinates; its C and B tiles are rows of
    // 64 elements (dstate a multiple of 64)
    return a.dtype == 1 && a.headdim == kP && a.seqlen < (int64_t(1) << 31) &&
           (a.dstate == 64 || a.dstate == 128 || a.dstate == 256) && (Q == 128 || Q == 256) && hpg % 2 == 0;
}

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

cudaError_t bounds_selftest_launch(float* buf, size_t bytes, int64_t index, cudaStream_t stream) {
    cudaEvent_t t0 = timing_begin(stream, "bounds_selftest");
    bounds_selftest<<<1, 1, 0, stream>>>(buf, span_of(buf, bytes), index);
    note_launch("bounds_selftest", stream, t0);
    return cudaGetLastError();
}

cudaError_t bounded_wait_selftest_launch(uint32_t max_checks, cudaStream_t stream) {
    cudaEvent_t t0 = timing_begin(stream, "bounded_wait_selftest");
    bounded_wait_selftest<<<1, 32, 0, stream>>>(max_checks);
    note_launch("bounded_wait_selftest", stream, t0);
    return cudaGetLastError();
}

}  // namespace ssm
