// noalloc.cu -- rm_cp_backward_noalloc: the whole backward (prepare, suffix,
// apply) with its per-token scratch taken from a fixed device array that the
// library owns, for callers that cannot allocate device memory.
//
// The backward needs one fp32 value per (row, token, head) between its two
// sweeps (q.dq minus its same-token term, read by the gate-gradient scan).
// The regular entry points take that as the caller's workspace; this one
// keeps it in kScratchFloats floats of file-scope device memory instead.
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace {

// 4 Mi floats (16 MiB): enough for B * T * H <= 4,194,304, e.g. one row of
// 262,144 tokens with 16 heads.  The array is placed on a device when this
// file's module is loaded there; under CUDA's default lazy module loading
// that is the first rm_cp_backward_noalloc call on the device (its address
// lookup), after which the device holds it until the process exits.
constexpr size_t kScratchFloats = size_t(1) << 22;
static __device__ __align__(256) float g_backward_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_lock[kMaxDevices];
float* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// g_backward_scratch names a host-side shadow, never the device memory, so
// the address is looked up with that device current.  Only a successful
// lookup is kept: a failed one (e.g. attempted during stream capture, where
// a module cannot be loaded) clears its error and is retried by the next call.
rm_status scratch_for_current_device(float** out, cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) {
        cudaGetLastError();
        return RM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return RM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> guard(g_lock[dev]);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_backward_scratch);
        if (*err != cudaSuccess || p == nullptr) {
            cudaGetLastError();  // leave no error pending for later checks
            if (*err == cudaSuccess) *err = cudaErrorInvalidSymbol;
            return RM_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return RM_OK;
}

}  // namespace

#define RM_NEED_NA(ptr)                                      \
    do {                                                     \
        rm_status s_ = rmcp::api_need((ptr), #ptr);          \
        if (s_ != RM_OK) return s_;                          \
    } while (0)

extern "C" rm_status rm_cp_backward_noalloc(const rm_cp_problem* p, const void* q, const void* k,
                                            const void* v, const float* g, const float* S_in,
                                            const float* M, const void* dO, float* gamma,
                                            float* dS_out, void* dq, void* dk, void* dv,
                                            float* dg, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status st = rmcp::api_check_problem(p, &d);
    if (st != RM_OK) return st;
    RM_NEED_NA(q);
    RM_NEED_NA(k);
    RM_NEED_NA(v);
    RM_NEED_NA(g);
    RM_NEED_NA(S_in);
    RM_NEED_NA(M);
    RM_NEED_NA(dO);
    RM_NEED_NA(gamma);
    RM_NEED_NA(dS_out);
    RM_NEED_NA(dq);
    RM_NEED_NA(dk);
    RM_NEED_NA(dv);
    RM_NEED_NA(dg);
    // one scratch value per (row, token, head), or per key dimension with vector gates
    if (size_t(d.B) * size_t(d.T) * size_t(d.H) * (d.vg ? size_t(d.Dk) : 1) > kScratchFloats)
        return rmcp::api_fail(RM_ERR_SHAPE,
                              "rm_cp_backward_noalloc: B*T*H (times Dk with vector gates) exceeds "
                              "its fixed scratch of 4194304 entries; use "
                              "rm_cp_backward_prepare/apply with a workspace");
    float* scratch = nullptr;
    cudaError_t err = cudaSuccess;
    if (scratch_for_current_device(&scratch, &err) != RM_OK) {
        char msg[256];
        std::snprintf(msg, sizeof(msg),
                      "rm_cp_backward_noalloc: scratch address lookup failed (%s); the next "
                      "call retries it",
                      cudaGetErrorString(err));
        return rmcp::api_fail(RM_ERR_CUDA, msg);
    }

    // the per-token partials are fully written by the prepare sweep before the
    // apply sweep reads them, so the array needs no clearing between calls
    rmcp::Ptrs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = g;
    a.S_in = S_in;
    a.dO = dO;
    a.sum_out = gamma;
    a.out0 = dq;
    a.ws_f32 = scratch;
    st = rmcp::api_launch(rmcp::Op::kBackwardPrepare, p, d, a, stream);
    if (st != RM_OK) return st;
    st = rmcp::launch_compose_suffix(d, M, gamma, dS_out, reinterpret_cast<cudaStream_t>(stream));
    if (st != RM_OK) {
        char msg[192];
        std::snprintf(msg, sizeof(msg), "rm_cp_backward_noalloc: suffix launch failed: %s", rmcp::cuda_error_text());
        return rmcp::api_fail(st, msg);
    }
    rmcp::Ptrs b;
    b.q = q;
    b.k = k;
    b.v = v;
    b.g = g;
    b.dO = dO;
    b.S_in = S_in;
    b.dS_out = dS_out;
    b.out0 = dk;
    b.out1 = dv;
    b.dg = dg;
    b.ws_f32 = scratch;
    return rmcp::api_launch(rmcp::Op::kBackwardApply, p, d, b, stream);
}
