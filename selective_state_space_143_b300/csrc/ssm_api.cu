// C-ABI entry points of libssmscan.so: argument checks, workspace, dispatch.
// The operation and the argument contract are stated in include/ssm_scan.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "ssm_scan.h"
#include "ssm_internal.h"

namespace ssm {

static std::atomic<uint64_t> g_launches{0};

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {

constexpr int64_t kMaxGridYZ = 65535;

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int32_t dtype) { return dtype == SSM_BF16 ? 2 : 4; }

// Shape checks shared by every entry point.  Returns SSM_OK or the status to report.
int check_shape(const ssm_shape* s) {
    if (!s) return SSM_ERR_NULL;
    if (s->mode != SSM_MODE_DIAG && s->mode != SSM_MODE_SSD) return SSM_ERR_DTYPE;
    if (s->dtype != SSM_F32 && s->dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (s->flags != 0) return SSM_ERR_UNSUPPORTED;
    if (s->batch < 0 || s->seqlen < 0 || s->nheads < 1 || s->headdim < 1 || s->dstate < 1 ||
        s->ngroups < 1 || s->chunk < 0)
        return SSM_ERR_SHAPE;
    if (s->nheads % s->ngroups != 0) return SSM_ERR_SHAPE;
    if (s->batch > kMaxGridYZ / 4) return SSM_ERR_UNSUPPORTED;
    if (s->seqlen > (int64_t(1) << 40) || s->nheads > (int64_t(1) << 24)) return SSM_ERR_UNSUPPORTED;
    const int E = elem_size(s->dtype);
    if (s->mode == SSM_MODE_DIAG) {
        if (s->headdim != 1) return SSM_ERR_SHAPE;
        if (s->dstate > 64) return SSM_ERR_UNSUPPORTED;
        if (s->chunk != 0 && s->chunk % 32 != 0) return SSM_ERR_SHAPE;
        // each group's channel run and each B/C row are whole 16-byte chunks
        if (((s->nheads / s->ngroups) * E) % 16 != 0) return SSM_ERR_ALIGN;
        if ((s->dstate * E) % 16 != 0) return SSM_ERR_ALIGN;
        if (s->chunk > 0 && (s->seqlen + s->chunk - 1) / s->chunk > kMaxGridYZ) return SSM_ERR_UNSUPPORTED;
    } else {
        if (s->dstate > 256 || s->headdim > 256) return SSM_ERR_UNSUPPORTED;
        if (s->chunk != 0 && (s->chunk % 16 != 0 || s->chunk > 256)) return SSM_ERR_SHAPE;
        if ((s->nheads * s->headdim * E) % 16 != 0) return SSM_ERR_ALIGN;
        if ((s->ngroups * s->dstate * E) % 16 != 0) return SSM_ERR_ALIGN;
        if (s->nheads * ((s->headdim + 63) / 64) * ((s->dstate + 63) / 64) > kMaxGridYZ)
            return SSM_ERR_UNSUPPORTED;
    }
    return SSM_OK;
}

int check_args(const void* x, const void* dt, const float* A, const void* B, const void* C,
               const float* D, const void* z, const float* dt_bias, const void* out,
               const float* final_state, const ssm_shape* s) {
    const int rc = check_shape(s);
    if (rc != SSM_OK) return rc;
    // x, dt, B, C and out may be NULL only when they hold no elements
    const bool empty = s->batch == 0 || s->seqlen == 0;
    if (!A || (!empty && (!x || !dt || !B || !C || !out))) return SSM_ERR_NULL;
    const void* ptrs[] = {x, dt, A, B, C, D, z, dt_bias, out, final_state};
    for (const void* p : ptrs)
        if (!aligned16(p)) return SSM_ERR_ALIGN;
    return SSM_OK;
}

ScanArgs make_args(const void* x, const void* dt, const float* A, const void* B, const void* C,
                   const float* D, const void* z, const float* dt_bias, void* out,
                   float* final_state, const ssm_shape* s) {
    ScanArgs a;
    a.x = x;
    a.dt = dt;
    a.A = A;
    a.B = B;
    a.C = C;
    a.D = D;
    a.z = z;
    a.dt_bias = dt_bias;
    a.initial_state = nullptr;
    a.out = out;
    a.final_state = final_state;
    a.batch = s->batch;
    a.seqlen = s->seqlen;
    a.nheads = s->nheads;
    a.headdim = s->headdim;
    a.dstate = s->dstate;
    a.ngroups = s->ngroups;
    a.chunk = s->chunk;
    a.dtype = s->dtype;
    return a;
}

size_t workspace_for(const ScanArgs& a, int mode) {
    return mode == SSM_MODE_DIAG ? diag_workspace_bytes(a) : ssd_workspace_bytes(a);
}

int run(const ScanArgs& a, int mode, void* ws, cudaStream_t stream) {
    if (a.batch == 0) return SSM_OK;
    const cudaError_t e = mode == SSM_MODE_DIAG ? diag_launch(a, ws, stream) : ssd_launch(a, ws, stream);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace
}  // namespace ssm

using namespace ssm;

extern "C" {

int ssm_abi_version(void) { return (1 << 16) | 0; }

uint64_t ssm_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* ssm_strerror(int status) {
    switch (status) {
        case SSM_OK: return "success";
        case SSM_ERR_NULL: return "a required pointer is NULL";
        case SSM_ERR_SHAPE: return "a size is out of range or inconsistent";
        case SSM_ERR_DTYPE: return "unknown mode or dtype";
        case SSM_ERR_ALIGN: return "a pointer or a row is not 16-byte aligned";
        case SSM_ERR_UNSUPPORTED: return "valid but unsupported shape or flags";
        case SSM_ERR_ALLOC: return "workspace allocation failed or workspace too small";
        case SSM_ERR_CUDA: return "a CUDA call failed";
        case SSM_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        default: return "unknown status";
    }
}

size_t ssm_scan_workspace_size(const ssm_shape* shape) {
    if (check_shape(shape) != SSM_OK) return (size_t)-1;
    const ScanArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, shape);
    return workspace_for(a, shape->mode);
}

int ssm_scan_fwd_ws(const void* x, const void* dt, const float* A, const void* B, const void* C,
                    const float* D, const void* z, const float* dt_bias, void* out,
                    float* final_state, const ssm_shape* shape, void* workspace,
                    size_t workspace_bytes, ssm_stream_t stream) {
    const int rc = check_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape);
    if (rc != SSM_OK) return rc;
    const ScanArgs a = make_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape);
    const size_t need = workspace_for(a, shape->mode);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return SSM_ERR_ALLOC;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SSM_ERR_ALIGN;
    return run(a, shape->mode, workspace, (cudaStream_t)stream);
}

int ssm_scan_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* dt_bias, void* out,
                 float* final_state, const ssm_shape* shape, ssm_stream_t stream) {
    const int rc = check_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape);
    if (rc != SSM_OK) return rc;
    const ScanArgs a = make_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape);
    const size_t need = workspace_for(a, shape->mode);
    void* ws = nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    if (need > 0 && a.batch > 0) {
        if (cudaMallocAsync(&ws, need, st) != cudaSuccess) {
            (void)cudaGetLastError();
            return SSM_ERR_ALLOC;
        }
    }
    const int r = run(a, shape->mode, ws, st);
    if (ws) {
        if (cudaFreeAsync(ws, st) != cudaSuccess && r == SSM_OK) return SSM_ERR_CUDA;
    }
    return r;
}

}  // extern "C"
