// noalloc.cu -- rm_cp_backward_noalloc: the whole backward (prepare, suffix,
// apply) with its per-token scratch taken from a fixed device array that the
// library owns, for callers that cannot allocate device memory.
//
// The backward needs one fp32 value per (row, token, head) between its two
// sweeps (q.dq minus its same-token term, read by the gate-gradient scan).
// The regular entry points take that as the caller's workspace; this one
// keeps it in kScratchFloats floats of file-scope device memory instead.
#include <mutex>

#include "internal.h"

namespace {

// 4 Mi floats (16 MiB): enough for B * T * H <= 4,194,304, e.g. one row of
// 262,144 tokens with 16 heads.  Every device that loads the library holds
// this array until the process exits.
constexpr size_t kScratchFloats = size_t(1) << 22;
static __device__ __align__(256) float g_backward_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
float* g_scratch_ptr[kMaxDevices] = {};
cudaError_t g_scratch_err[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// g_backward_scratch names a host-side shadow, never the device memory, so
// the address is looked up once per device with that device current.
rm_status scratch_for_current_device(float** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RM_ERR_CUDA;
    std::call_once(g_once[dev], [dev] {
        void* p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_backward_scratch);
        g_scratch_ptr[dev] = static_cast<float*>(p);
    });
    if (g_scratch_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) return RM_ERR_CUDA;
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
    if (size_t(d.B) * size_t(d.T) * size_t(d.H) > kScratchFloats)
        return rmcp::api_fail(RM_ERR_SHAPE,
                              "rm_cp_backward_noalloc: B*T*H exceeds its fixed scratch of "
                              "4194304 entries; use rm_cp_backward_prepare/apply with a workspace");
    float* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != RM_OK)
        return rmcp::api_fail(RM_ERR_CUDA, "rm_cp_backward_noalloc: scratch address lookup failed");

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
    if (st != RM_OK) return rmcp::api_fail(st, "rm_cp_backward_noalloc: suffix launch failed");
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
