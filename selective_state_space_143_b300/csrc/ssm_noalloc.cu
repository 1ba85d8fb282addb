// ssm_scan_fwd_noalloc: the forward scan with its scratch taken from a fixed device
// array that is part of the library image, so the call itself allocates nothing.
//
// Who needs it: callers that must not allocate device memory during a scan, such as
// an application that reserves all device memory up front for its own allocator, or
// a latency-critical loop where an allocation could synchronise the device or fail
// under memory pressure.  They pass inputs and outputs as usual; the scratch is the
// array below.
#include <cuda_runtime.h>

#include <mutex>

#include "ssm_scan.h"
#include "ssm_internal.h"

namespace ssm {
namespace {

// Largest scratch the no-allocation entry point can serve.  Every GPU that loads this
// part of the library keeps the array for the life of the process.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array for the current device, looked up once per device
// (with that device current) and cached.  In host code the array's name is only a
// host-side handle, so the kernels must be given this address.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return SSM_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SSM_OK;
}

}  // namespace
}  // namespace ssm

extern "C" int ssm_scan_fwd_noalloc(const void* x, const void* dt, const float* A, const void* B,
                                    const void* C, const float* D, const void* z,
                                    const float* dt_bias, void* out, float* final_state,
                                    const ssm_shape* shape, ssm_stream_t stream) {
    // An invalid shape gets its status from ssm_scan_fwd_ws below, before any work.
    const size_t need = ssm_scan_workspace_size(shape);
    const bool valid = need != (size_t)-1;
    if (valid && need > ssm::kStaticScratchBytes) return SSM_ERR_ALLOC;  // beyond the fixed scratch
    void* scratch = nullptr;
    if (valid && need > 0) {
        const int rc = ssm::scratch_address(&scratch);
        if (rc != SSM_OK) return rc;
    }
    // The scratch keeps whatever the previous call left.  Nothing in it has to start at
    // zero: every scratch entry the scan reads is written earlier in the same call.
    return ssm_scan_fwd_ws(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape, scratch,
                           ssm::kStaticScratchBytes, stream);
}
