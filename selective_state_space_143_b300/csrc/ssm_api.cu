// C-ABI entry points of libssmscan.so: argument checks, workspace, dispatch.
// The operation and the argument contract are stated in include/ssm_scan.h.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "ssm_scan.h"
#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

static std::atomic<uint64_t> g_launches{0};

// Launch timing: events recorded around each launch while enabled, summed per kernel
// name by ssm_timing_collect.
namespace {
struct TimedLaunch {
    const char* name;
    cudaEvent_t start, end;
};
std::atomic<int> g_timing{0};
std::mutex g_timing_mutex;
std::vector<TimedLaunch> g_timed;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return e;
}
}  // namespace

cudaEvent_t timing_begin(cudaStream_t stream, const char* name) {
    nvtxRangePushA(name);
    if (!g_timing.load(std::memory_order_relaxed)) return nullptr;
    cudaEvent_t e = take_event();
    if (e && cudaEventRecord(e, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return e;
}

void launch_failed(cudaEvent_t start) {
    nvtxRangePop();
    if (!start) return;
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    g_event_pool.push_back(start);
}

void note_launch(const char* name, cudaStream_t stream, cudaEvent_t start) {
    nvtxRangePop();
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (!start) return;
    cudaEvent_t end = take_event();
    if (!end || cudaEventRecord(end, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return;
    }
    std::lock_guard<std::mutex> lock(g_timing_mutex);
    g_timed.push_back({name, start, end});
}

// Plan overrides (ssm_tuning_set), one slot per ssm_tuning_knob.
namespace {
constexpr int kKnobs = 5;
std::atomic<int64_t> g_tuning[kKnobs] = {};
std::atomic<int> g_alloc_failures{0};
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices] = {};
}  // namespace

int64_t tuning(int knob) { return knob >= 0 && knob < kKnobs ? g_tuning[knob].load(std::memory_order_relaxed) : 0; }

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return 148;
    }
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 148;
    }
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t scratch_alloc(void** p, size_t bytes, cudaStream_t stream) {
    int pending = g_alloc_failures.load(std::memory_order_relaxed);
    while (pending > 0) {
        if (g_alloc_failures.compare_exchange_weak(pending, pending - 1, std::memory_order_relaxed)) {
            *p = nullptr;
            return cudaErrorMemoryAllocation;
        }
    }
    return cudaMallocAsync(p, bytes, stream);
}

namespace {

constexpr int64_t kMaxGridYZ = 65535;

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_size(int32_t dtype) { return dtype == SSM_BF16 ? 2 : 4; }

// Shape checks shared by every entry point.  Returns SSM_OK or the status to report.
int check_shape(const ssm_shape* s) {
    if (!s) return SSM_ERR_NULL;
    if (s->mode != SSM_MODE_DIAG && s->mode != SSM_MODE_SSD && s->mode != SSM_MODE_CDIAG) return SSM_ERR_DTYPE;
    if (s->dtype != SSM_F32 && s->dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (s->flags != 0) return SSM_ERR_UNSUPPORTED;
    if (s->batch < 0 || s->seqlen < 0 || s->nheads < 1 || s->headdim < 1 || s->dstate < 1 ||
        s->ngroups < 1 || s->chunk < 0)
        return SSM_ERR_SHAPE;
    if (s->nheads % s->ngroups != 0) return SSM_ERR_SHAPE;
    if (s->batch > kMaxGridYZ / 4) return SSM_ERR_UNSUPPORTED;
    if (s->seqlen > (int64_t(1) << 40) || s->nheads > (int64_t(1) << 24)) return SSM_ERR_UNSUPPORTED;
    const int E = elem_size(s->dtype);
    if (s->mode == SSM_MODE_CDIAG) {
        if (s->headdim != 1) return SSM_ERR_SHAPE;
        if (s->dstate > 32) return SSM_ERR_UNSUPPORTED;
        if (s->chunk != 0 && s->chunk % 16 != 0) return SSM_ERR_SHAPE;
        // each group's channel run and each complex B/C row are whole 16-byte chunks
        if (((s->nheads / s->ngroups) * E) % 16 != 0) return SSM_ERR_ALIGN;
        if ((s->dstate * 2 * E) % 16 != 0) return SSM_ERR_ALIGN;
        if (s->chunk > 0 && (s->seqlen + s->chunk - 1) / s->chunk > kMaxGridYZ) return SSM_ERR_UNSUPPORTED;
    } else if (s->mode == SSM_MODE_DIAG) {
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
        // the state of one head moves in 16-byte pieces
        if ((s->headdim * s->dstate) % 4 != 0) return SSM_ERR_ALIGN;
        if (s->nheads * ((s->headdim + 63) / 64) * ((s->dstate + 63) / 64) > kMaxGridYZ)
            return SSM_ERR_UNSUPPORTED;
    }
    return SSM_OK;
}

int check_args(const void* x, const void* dt, const float* A, const void* B, const void* C,
               const float* D, const void* z, const float* dt_bias, const void* out,
               const float* final_state, const ssm_shape* s, const float* initial_state = nullptr) {
    const int rc = check_shape(s);
    if (rc != SSM_OK) return rc;
    // x, dt, B, C and out may be NULL only when they hold no elements
    const bool empty = s->batch == 0 || s->seqlen == 0;
    if (!A || (!empty && (!x || !dt || !B || !C || !out))) return SSM_ERR_NULL;
    const void* ptrs[] = {x, dt, A, B, C, D, z, dt_bias, out, final_state, initial_state};
    for (const void* p : ptrs)
        if (!aligned16(p)) return SSM_ERR_ALIGN;
    return SSM_OK;
}

// Bytes of the fp32 state of all sequences: (batch, nheads, headdim, dstate), times two
// (re, im) in the complex mode.
size_t state_bytes(const ssm_shape* s) {
    return (size_t)s->batch * s->nheads * s->headdim * s->dstate * sizeof(float) *
           (s->mode == SSM_MODE_CDIAG ? 2 : 1);
}

bool overlaps(const void* p, size_t pn, const void* q, size_t qn) {
    if (!p || !q || pn == 0 || qn == 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + qn && b < a + pn;
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
    a.conv_w = nullptr;
    a.conv_b = nullptr;
    a.x_prev = nullptr;
    a.x_last = nullptr;
    a.conv_k = 0;
    a.x_f32 = 0;
    a.x_lo = nullptr;
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

// Bytes of the convolved input the SSD path keeps in scratch (the diagonal path fuses
// the convolution and needs none).
size_t conv_buffer_bytes(const ScanArgs& a, int mode) {
    if (a.conv_k == 0 || mode != SSM_MODE_SSD || a.batch == 0) return 0;
    return align_up((size_t)a.batch * a.seqlen * a.nheads * a.headdim * sizeof(float), 256);
}

size_t workspace_for(const ScanArgs& a, int mode) {
    const size_t base = mode == SSM_MODE_DIAG    ? diag_workspace_bytes(a)
                        : mode == SSM_MODE_CDIAG ? cdiag_workspace_bytes(a)
                                                 : ssd_workspace_bytes(a);
    const size_t conv = conv_buffer_bytes(a, mode);
    return conv ? align_up(base, 256) + conv : base;
}

int run(const ScanArgs& a, int mode, void* ws, cudaStream_t stream) {
    if (a.batch == 0) return SSM_OK;
    cudaError_t e;
    if (mode == SSM_MODE_DIAG) {
        e = diag_launch(a, ws, stream);
    } else if (mode == SSM_MODE_CDIAG) {
        e = cdiag_launch(a, ws, stream);
    } else if (a.conv_k > 0) {
        // convolution pass into scratch, then the SSD kernels on the convolved input
        void* xc = (char*)ws + align_up(ssd_workspace_bytes(a), 256);
        const bool split = ssd_conv_split(a);
        e = conv_prepass_launch(a, xc, split, stream);
        if (e == cudaSuccess) {
            ScanArgs b = a;
            b.x = xc;
            if (split)
                b.x_lo = (const char*)xc + (size_t)a.batch * a.seqlen * a.nheads * a.headdim * 2;
            else
                b.x_f32 = 1;
            b.conv_k = 0;
            e = ssd_launch(b, ws, stream);
        }
        if (e == cudaSuccess) e = conv_tail_launch(a, stream);
    } else {
        e = ssd_launch(a, ws, stream);
    }
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

int check_conv(const ssm_conv* cv) {
    if (!cv || !cv->weight) return SSM_ERR_NULL;
    if (cv->width < 1 || cv->width > 4) return SSM_ERR_UNSUPPORTED;
    const void* ptrs[] = {cv->weight, cv->bias, cv->x_prev, cv->x_last};
    for (const void* p : ptrs)
        if (!aligned16(p)) return SSM_ERR_ALIGN;
    return SSM_OK;
}

void set_conv(ScanArgs& a, const ssm_conv* cv) {
    a.conv_w = cv->weight;
    a.conv_b = cv->bias;
    a.x_prev = cv->x_prev;
    a.x_last = cv->x_last;
    a.conv_k = cv->width;
}

// Bytes of one convolution state (batch, width-1, channels) in the input dtype.
size_t conv_state_bytes(const ssm_shape* s, int width) {
    return (size_t)s->batch * (width - 1) * s->nheads * s->headdim * elem_size(s->dtype);
}

// Caller-provided scratch.
int run_with(const ScanArgs& a, int mode, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    const size_t need = workspace_for(a, mode);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return SSM_ERR_ALLOC;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SSM_ERR_ALIGN;
    return run(a, mode, workspace, stream);
}

// Scratch from the stream-ordered allocator, freed on the same stream.
int run_allocating(const ScanArgs& a, int mode, cudaStream_t st) {
    const size_t need = workspace_for(a, mode);
    void* ws = nullptr;
    if (need > 0 && a.batch > 0) {
        if (scratch_alloc(&ws, need, st) != cudaSuccess) {
            (void)cudaGetLastError();
            return SSM_ERR_ALLOC;
        }
    }
    const int r = run(a, mode, ws, st);
    if (ws) {
        if (cudaFreeAsync(ws, st) != cudaSuccess && r == SSM_OK) return SSM_ERR_CUDA;
    }
    return r;
}

int step_common(const void* x, const void* dt, const float* A, const void* B, const void* C,
                const float* D, const void* z, const float* dt_bias, const ssm_conv* conv,
                float* state, void* out, const ssm_shape* shape, cudaStream_t stream) {
    const int rc = check_shape(shape);
    if (rc != SSM_OK) return rc;
    if (shape->mode == SSM_MODE_CDIAG) return SSM_ERR_UNSUPPORTED;
    if (shape->seqlen != 1) return SSM_ERR_SHAPE;
    if (shape->dstate % 4 != 0) return SSM_ERR_ALIGN;  // state rows move in 16-byte pieces
    // one grid row per sequence, 32-bit channel indices within a sequence
    if (shape->batch > 65535 || shape->nheads * shape->headdim > (int64_t(1) << 30)) return SSM_ERR_UNSUPPORTED;
    if (!A || (shape->batch > 0 && (!x || !dt || !B || !C || !out || !state))) return SSM_ERR_NULL;
    const void* ptrs[] = {x, dt, A, B, C, D, z, dt_bias, out, state};
    for (const void* p : ptrs)
        if (!aligned16(p)) return SSM_ERR_ALIGN;
    const size_t out_bytes = (size_t)shape->batch * shape->nheads * shape->headdim * elem_size(shape->dtype);
    const size_t sb = state_bytes(shape);
    if (overlaps(state, sb, out, out_bytes)) return SSM_ERR_SHAPE;
    ScanArgs a = make_args(x, dt, A, B, C, D, z, dt_bias, out, nullptr, shape);
    if (conv) {
        // the convolution state may be updated in place (x_last == x_prev), but must not
        // overlap anything else the step writes or reads
        const size_t cb = conv_state_bytes(shape, conv->width);
        if ((conv->x_last != conv->x_prev && overlaps(conv->x_last, cb, conv->x_prev, cb)) ||
            overlaps(conv->x_last, cb, state, sb) || overlaps(conv->x_last, cb, out, out_bytes) ||
            overlaps(conv->x_last, cb, x, out_bytes))
            return SSM_ERR_SHAPE;
        set_conv(a, conv);
    }
    if (shape->batch == 0) return SSM_OK;
    const cudaError_t e = step_launch(a, shape->mode == SSM_MODE_DIAG, state, stream);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace
}  // namespace ssm

using namespace ssm;

extern "C" {

int ssm_abi_version(void) { return (1 << 16) | 6; }

int ssm_tuning_set(int knob, int64_t value) {
    if (knob < 0 || knob >= ssm::kKnobs) return SSM_ERR_UNSUPPORTED;
    if (value < 0) return SSM_ERR_SHAPE;
    ssm::g_tuning[knob].store(value, std::memory_order_relaxed);
    return SSM_OK;
}

int64_t ssm_tuning_get(int knob) { return ssm::tuning(knob); }

void ssm_inject_alloc_failures(int count) {
    ssm::g_alloc_failures.store(count > 0 ? count : 0, std::memory_order_relaxed);
}

int ssm_device_status(int clear, ssm_stream_t stream) {
    int v = 0;
    if (ssm::device_status_take(&v, clear != 0, (cudaStream_t)stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    if (v == 0) return SSM_OK;
    return v == ssm::kStatusBounds ? SSM_ERR_BOUNDS : SSM_ERR_TIMEOUT;
}

int ssm_bounds_check_enabled(void) { return ssm::kBoundsCheck ? 1 : 0; }

int ssm_selftest_bounds(float* buf, size_t bytes, int64_t index, ssm_stream_t stream) {
    if (!ssm::kBoundsCheck) return SSM_ERR_UNSUPPORTED;
    if (!buf) return SSM_ERR_NULL;
    if (index < 0 || bytes % 4 != 0) return SSM_ERR_SHAPE;
    if (ssm::bounds_selftest_launch(buf, bytes, index, (cudaStream_t)stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

int ssm_selftest_bounded_wait(uint32_t max_checks, ssm_stream_t stream) {
    if (ssm::bounded_wait_selftest_launch(max_checks, (cudaStream_t)stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

uint64_t ssm_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void ssm_timing_enable(int on) { g_timing.store(on ? 1 : 0, std::memory_order_relaxed); }

int ssm_timing_collect(ssm_kernel_time* out, int max_entries) {
    std::vector<TimedLaunch> recs;
    {
        std::lock_guard<std::mutex> lock(g_timing_mutex);
        recs.swap(g_timed);
    }
    std::map<std::string, std::pair<int64_t, double>> agg;
    int status = 0;
    for (const TimedLaunch& r : recs) {
        float ms = 0.0f;
        if (cudaEventSynchronize(r.end) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.end) != cudaSuccess) {
            (void)cudaGetLastError();
            status = -SSM_ERR_CUDA;
        }
        auto& a = agg[r.name];
        a.first += 1;
        a.second += ms;
    }
    {
        std::lock_guard<std::mutex> lock(g_timing_mutex);
        for (const TimedLaunch& r : recs) {
            g_event_pool.push_back(r.start);
            g_event_pool.push_back(r.end);
        }
    }
    if (status < 0) return status;
    int n = 0;
    for (const auto& kv : agg) {
        if (out && n < max_entries) {
            std::memset(out[n].name, 0, sizeof(out[n].name));
            std::strncpy(out[n].name, kv.first.c_str(), sizeof(out[n].name) - 1);
            out[n].launches = kv.second.first;
            out[n].total_ms = kv.second.second;
        }
        ++n;
    }
    return n;
}

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
        case SSM_ERR_BOUNDS: return "a store address fell outside its buffer (bounds-checked build)";
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
    return run_with(a, shape->mode, workspace, workspace_bytes, (cudaStream_t)stream);
}

int ssm_scan_fwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* dt_bias, void* out,
                 float* final_state, const ssm_shape* shape, ssm_stream_t stream) {
    const int rc = check_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape);
    if (rc != SSM_OK) return rc;
    const ScanArgs a = make_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape);
    return run_allocating(a, shape->mode, (cudaStream_t)stream);
}

int ssm_scan_fwd_state(const void* x, const void* dt, const float* A, const void* B, const void* C,
                       const float* D, const void* z, const float* dt_bias,
                       const float* initial_state, void* out, float* final_state,
                       const ssm_shape* shape, void* workspace, size_t workspace_bytes,
                       ssm_stream_t stream) {
    const int rc = check_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape, initial_state);
    if (rc != SSM_OK) return rc;
    // the initial state is read by blocks that may start after the final state is written
    if (overlaps(initial_state, state_bytes(shape), final_state, state_bytes(shape))) return SSM_ERR_SHAPE;
    ScanArgs a = make_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape);
    a.initial_state = initial_state;
    if (workspace == nullptr && workspace_bytes == 0) return run_allocating(a, shape->mode, (cudaStream_t)stream);
    return run_with(a, shape->mode, workspace, workspace_bytes, (cudaStream_t)stream);
}

size_t ssm_scan_conv_workspace_size(const ssm_shape* shape) {
    if (check_shape(shape) != SSM_OK || shape->mode == SSM_MODE_CDIAG) return (size_t)-1;
    ScanArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                           nullptr, nullptr, shape);
    a.conv_k = 4;  // any width: the scratch does not depend on it
    return workspace_for(a, shape->mode);
}

int ssm_scan_fwd_conv(const void* x, const void* dt, const float* A, const void* B, const void* C,
                      const float* D, const void* z, const float* dt_bias, const ssm_conv* conv,
                      const float* initial_state, void* out, float* final_state,
                      const ssm_shape* shape, void* workspace, size_t workspace_bytes,
                      ssm_stream_t stream) {
    int rc = check_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape, initial_state);
    if (rc != SSM_OK) return rc;
    rc = check_conv(conv);
    if (rc != SSM_OK) return rc;
    if (shape->mode == SSM_MODE_CDIAG) return SSM_ERR_UNSUPPORTED;
    const size_t sb = state_bytes(shape);
    const size_t cb = conv_state_bytes(shape, conv->width);
    const size_t xb = (size_t)shape->batch * shape->seqlen * shape->nheads * shape->headdim * elem_size(shape->dtype);
    // x_last is written while other thread blocks may still read x, x_prev or out
    if (overlaps(initial_state, sb, final_state, sb) || overlaps(conv->x_last, cb, conv->x_prev, cb) ||
        overlaps(conv->x_last, cb, x, xb) || overlaps(conv->x_last, cb, out, xb))
        return SSM_ERR_SHAPE;
    ScanArgs a = make_args(x, dt, A, B, C, D, z, dt_bias, out, final_state, shape);
    a.initial_state = initial_state;
    set_conv(a, conv);
    if (workspace == nullptr && workspace_bytes == 0) return run_allocating(a, shape->mode, (cudaStream_t)stream);
    return run_with(a, shape->mode, workspace, workspace_bytes, (cudaStream_t)stream);
}

size_t ssm_scan_bwd_workspace_size(const ssm_shape* shape) {
    if (check_shape(shape) != SSM_OK || shape->mode == SSM_MODE_CDIAG) return (size_t)-1;
    const ScanArgs a = make_args(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, shape);
    return scan_bwd_workspace_bytes(a, shape->mode == SSM_MODE_SSD);
}

int ssm_scan_bwd(const void* x, const void* dt, const float* A, const void* B, const void* C,
                 const float* D, const void* z, const float* dt_bias, const float* initial_state,
                 const void* dout, const float* dfinal_state, float* dx, float* ddt, float* dA,
                 float* dB, float* dC, float* dD, float* dz, float* ddt_bias,
                 float* dinitial_state, const ssm_shape* shape, void* workspace,
                 size_t workspace_bytes, ssm_stream_t stream) {
    int rc = check_args(x, dt, A, B, C, D, z, dt_bias, dx, nullptr, shape, initial_state);
    if (rc != SSM_OK) return rc;
    if (shape->mode == SSM_MODE_CDIAG) return SSM_ERR_UNSUPPORTED;
    const bool empty = shape->batch == 0 || shape->seqlen == 0;
    if (!dA || (!empty && (!dout || !dx || !ddt || !dB || !dC))) return SSM_ERR_NULL;
    const void* outs[] = {dout, dfinal_state, dx, ddt, dA, dB, dC, dD, dz, ddt_bias, dinitial_state};
    for (const void* p : outs)
        if (!aligned16(p)) return SSM_ERR_ALIGN;
    ScanBwdArgs s;
    s.fwd = make_args(x, dt, A, B, C, D, z, dt_bias, nullptr, nullptr, shape);
    s.ssd = shape->mode == SSM_MODE_SSD;
    s.fwd.initial_state = initial_state;
    s.dout = dout;
    s.dfinal = dfinal_state;
    s.dx = dx;
    s.ddt = ddt;
    s.dA = dA;
    s.dB = dB;
    s.dC = dC;
    s.dD = D ? dD : nullptr;
    s.dz = z ? dz : nullptr;
    s.ddt_bias = dt_bias ? ddt_bias : nullptr;
    s.dinit = dinitial_state;
    const size_t need = scan_bwd_workspace_bytes(s.fwd, s.ssd);
    cudaStream_t st = (cudaStream_t)stream;
    void* ws = workspace;
    bool owned = false;
    if (need > 0 && !empty) {
        if (workspace == nullptr && workspace_bytes == 0) {
            if (scratch_alloc(&ws, need, st) != cudaSuccess) {
                (void)cudaGetLastError();
                return SSM_ERR_ALLOC;
            }
            owned = true;
        } else if (workspace == nullptr || workspace_bytes < need) {
            return SSM_ERR_ALLOC;
        } else if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) {
            return SSM_ERR_ALIGN;
        }
    }
    const cudaError_t e = scan_bwd_launch(s, ws, st);
    int r = e == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
    if (owned && cudaFreeAsync(ws, st) != cudaSuccess && r == SSM_OK) r = SSM_ERR_CUDA;
    return r;
}

int ssm_step_conv(const void* x, const void* dt, const float* A, const void* B, const void* C,
                  const float* D, const void* z, const float* dt_bias, const ssm_conv* conv,
                  float* state, void* out, const ssm_shape* shape, ssm_stream_t stream) {
    const int rc = check_conv(conv);
    if (rc != SSM_OK) return rc;
    return step_common(x, dt, A, B, C, D, z, dt_bias, conv, state, out, shape, (cudaStream_t)stream);
}

int ssm_step(const void* x, const void* dt, const float* A, const void* B, const void* C,
             const float* D, const void* z, const float* dt_bias, float* state, void* out,
             const ssm_shape* shape, ssm_stream_t stream) {
    return step_common(x, dt, A, B, C, D, z, dt_bias, nullptr, state, out, shape, (cudaStream_t)stream);
}

}  // extern "C"
