// rm_cp_host.cu -- the C ABI (include/rm_cp.h): host-side validation, path
// dispatch, the packed-sequence metadata builder and error reporting.
// Nothing here allocates device memory or synchronises; every compute call
// validates all of its arguments before it enqueues anything.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "internal.h"

namespace rmcp {
namespace {
std::atomic<uint64_t> g_launches{0};
}
void note_launch(int n) { g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed); }
}  // namespace rmcp

namespace rmcp {
namespace {
thread_local cudaError_t g_launch_error = cudaSuccess;
}
void begin_launches() {
    g_launch_error = cudaSuccess;
    tc::clear_map_result();
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) (void)cudaSetDevice(dev);  // initialises and binds the context
    (void)cudaGetLastError();
}
bool launch_ok() {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return true;
    g_launch_error = e;
    return false;
}
const char* cuda_error_text() {
    cudaError_t e = g_launch_error;
    g_launch_error = cudaSuccess;
    if (e == cudaSuccess) e = cudaGetLastError();
    return cudaGetErrorString(e);
}
}  // namespace rmcp

namespace {

thread_local char g_last_error[512] = "";

rm_status fail(rm_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks the problem and fills the launch dimensions.
rm_status check_problem(const rm_cp_problem* p, rmcp::Dims* d) {
    if (p == nullptr) return fail(RM_ERR_INVALID_ARG, "problem pointer is NULL");
    if (p->B <= 0 || p->T <= 0 || p->H <= 0 || p->Dk <= 0 || p->Dv <= 0 ||
        p->num_segments <= 0 || p->chunk <= 0)
        return fail(RM_ERR_INVALID_ARG,
                    "sizes must be positive (B=%d T=%d H=%d Dk=%d Dv=%d num_segments=%d chunk=%d)",
                    p->B, p->T, p->H, p->Dk, p->Dv, p->num_segments, p->chunk);
    if (p->dtype != RM_F32 && p->dtype != RM_BF16)
        return fail(RM_ERR_INVALID_ARG, "dtype %d is neither RM_F32 nor RM_BF16", (int)p->dtype);
    if (!std::isfinite(p->scale)) return fail(RM_ERR_INVALID_ARG, "scale is not finite");
    if (p->T % p->num_segments != 0)
        return fail(RM_ERR_SHAPE, "T=%d is not a multiple of num_segments=%d", p->T,
                    p->num_segments);
    const int L = p->T / p->num_segments;
    if (L % p->chunk != 0)
        return fail(RM_ERR_SHAPE, "segment length %d is not a multiple of chunk=%d", L, p->chunk);
    // every element count must fit comfortably in int64 and every token index in int32
    const double big = double(p->B) * p->T * p->H * (p->Dk > p->Dv ? p->Dk : p->Dv);
    const double sum = double(p->num_segments) * p->B * p->H * p->Dk * p->Dv;
    if (big > 4.0e18 || sum > 4.0e18 || double(p->B) * p->H > 2.0e9)
        return fail(RM_ERR_SHAPE, "problem too large");
    if (!aligned16(p->seq_idx) || !aligned16(p->preceding_start) || !aligned16(p->following_stop))
        return fail(RM_ERR_ALIGNMENT, "metadata arrays must be 16-byte aligned");
    d->B = p->B;
    d->T = p->T;
    d->H = p->H;
    d->Dk = p->Dk;
    d->Dv = p->Dv;
    d->nseg = p->num_segments;
    d->L = L;
    d->scale = p->scale;
    d->seq_idx = p->seq_idx;
    d->preceding_start = p->preceding_start;
    d->following_stop = p->following_stop;
    if (p->q_heads < 0 || (p->q_heads > 0 && p->H % p->q_heads != 0))
        return fail(RM_ERR_INVALID_ARG, "q_heads=%d does not divide H=%d", p->q_heads, p->H);
    d->qh = p->q_heads > 0 ? p->q_heads : p->H;
    d->qdiv = p->H / d->qh;
    if (p->vector_gates != 0 && p->vector_gates != 1)
        return fail(RM_ERR_INVALID_ARG, "vector_gates=%d is neither 0 nor 1", p->vector_gates);
    d->vg = p->vector_gates;
    if (d->vg && !rmcp::generic_supports(*d))
        return fail(RM_ERR_UNSUPPORTED,
                    "vector gates: unsupported head dims Dk=%d Dv=%d (need Dk in {16,32,64,128}, Dv "
                    "a multiple of 8 in [8,256], segment length a multiple of 16)",
                    p->Dk, p->Dv);
    if (!rmcp::tc_supports(*d, p->dtype) && !rmcp::generic_supports(*d))
        return fail(RM_ERR_UNSUPPORTED,
                    "unsupported head dims Dk=%d Dv=%d (need Dk in {16,32,64,128}, Dv a multiple "
                    "of 8 in [8,256], segment length a multiple of 16)",
                    p->Dk, p->Dv);
    return RM_OK;
}

rm_status need(const void* ptr, const char* name) {
    if (ptr == nullptr) return fail(RM_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(ptr)) return fail(RM_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
    return RM_OK;
}

#define RM_NEED(ptr)                                       \
    do {                                                   \
        rm_status s_ = need((ptr), #ptr);                  \
        if (s_ != RM_OK) return s_;                        \
    } while (0)

size_t workspace_bytes(const rmcp::Dims& d, rm_dtype dt) {
    // the backward: one fp32 per (row, token, head), or per key dimension with
    // vector gates; the fused forward: its flags and inclusive prefixes (the
    // two are never in use at the same time)
    const size_t per_tok = size_t(d.B) * d.T * d.H * sizeof(float) * (d.vg ? d.Dk : 1);
    const size_t bwd = (per_tok + 255) / 256 * 256;
    const size_t fused = rmcp::tc_fused_bytes(d, dt);
    return bwd > fused ? bwd : fused;
}

rm_status launch(rmcp::Op op, const rm_cp_problem* p, const rmcp::Dims& d, const rmcp::Ptrs& ptrs,
                 rm_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rmcp::begin_launches();
    rm_status st = d.vg ? (rmcp::vgtc_supports(d, p->dtype) ? rmcp::launch_vgtc(op, d, ptrs, s)
                                                            : rmcp::launch_vg(op, d, p->dtype, ptrs, s))
                   : rmcp::tc_supports_op(op, d, p->dtype)
                       ? rmcp::launch_tc(op, d, ptrs, s)
                       : rmcp::launch_generic(op, d, p->dtype, ptrs, s);
    if (st == RM_ERR_CUDA) {
        const int mr = rmcp::tc::last_map_result();
        if (mr != 0)
            return fail(RM_ERR_CUDA, "kernel launch failed: no tensor map (CUresult %d; bases 16-byte aligned?)", mr);
        return fail(RM_ERR_CUDA, "kernel launch failed: %s", rmcp::cuda_error_text());
    }
    if (st != RM_OK) return fail(st, "launch refused");
    return RM_OK;
}

}  // namespace

namespace rmcp {
// host-side checks and launches shared with noalloc.cu
rm_status api_check_problem(const rm_cp_problem* p, Dims* d) { return check_problem(p, d); }
rm_status api_need(const void* ptr, const char* name) { return need(ptr, name); }
rm_status api_fail(rm_status s, const char* msg) { return fail(s, "%s", msg); }
rm_status api_launch(Op op, const rm_cp_problem* p, const Dims& d, const Ptrs& ptrs,
                     rm_stream_t stream) {
    return launch(op, p, d, ptrs, stream);
}
}  // namespace rmcp

extern "C" {

const char* rm_cp_status_string(rm_status s) {
    switch (s) {
        case RM_OK: return "RM_OK";
        case RM_ERR_INVALID_ARG: return "RM_ERR_INVALID_ARG";
        case RM_ERR_SHAPE: return "RM_ERR_SHAPE";
        case RM_ERR_ALIGNMENT: return "RM_ERR_ALIGNMENT";
        case RM_ERR_UNSUPPORTED: return "RM_ERR_UNSUPPORTED";
        case RM_ERR_METADATA: return "RM_ERR_METADATA";
        case RM_ERR_CUDA: return "RM_ERR_CUDA";
        case RM_ERR_TIMEOUT: return "RM_ERR_TIMEOUT";
    }
    return "RM_ERR_UNKNOWN";
}

const char* rm_cp_last_error(void) { return g_last_error; }

uint64_t rm_cp_launch_count(void) { return rmcp::g_launches.load(std::memory_order_relaxed); }

rm_status rm_cp_device_status(int32_t* dev_scratch, int32_t clear, rm_stream_t stream) {
    RM_NEED(dev_scratch);
    // each tensor-core translation unit keeps its own flag
    int flag = 0, vflag = 0, gflag = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rm_status st = rmcp::tc_read_timeout_flag(&flag, clear, dev_scratch, s);
    if (st == RM_OK) st = rmcp::vgtc_read_timeout_flag(&vflag, clear, dev_scratch, s);
    if (st == RM_OK) st = rmcp::gdrtc_read_timeout_flag(&gflag, clear, dev_scratch, s);
    if (st != RM_OK)
        return fail(st, "device status read failed: %s", rmcp::cuda_error_text());
    if (flag || vflag || gflag) return fail(RM_ERR_TIMEOUT, "a bounded device-side wait ran out");
    return RM_OK;
}

rm_status rm_cp_selftest_wait_timeout(uint32_t limit_us, rm_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000)
        return fail(RM_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
    rm_status st = rmcp::tc_selftest_wait(limit_us, reinterpret_cast<cudaStream_t>(stream));
    if (st != RM_OK) return fail(st, "self-test launch failed");
    return RM_OK;
}

rm_status rm_cp_validate(const rm_cp_problem* p) {
    rmcp::Dims d;
    return check_problem(p, &d);
}

int32_t rm_cp_path(const rm_cp_problem* p) {
    rmcp::Dims d;
    if (check_problem(p, &d) != RM_OK) return -1;
    if (d.vg) return rmcp::vgtc_supports(d, p->dtype) ? 1 : 0;
    int n = 0;
    for (rmcp::Op op : {rmcp::Op::kForwardPrepare, rmcp::Op::kForwardApply,
                        rmcp::Op::kBackwardPrepare, rmcp::Op::kBackwardApply})
        n += rmcp::tc_supports_op(op, d, p->dtype) ? 1 : 0;
    return n == 4 ? 1 : (n == 0 ? 0 : 2);
}

size_t rm_cp_workspace_size(const rm_cp_problem* p) {
    rmcp::Dims d;
    if (check_problem(p, &d) != RM_OK) return 0;
    return workspace_bytes(d, p->dtype);
}

rm_status rm_cp_build_packed_metadata(const int32_t* cu, int32_t num_seqs, int32_t T,
                                      int32_t num_segments, int32_t* seq_idx,
                                      int32_t* local_cu, int32_t* local_off, int32_t* pre,
                                      int32_t* fol) {
    if (!cu || !seq_idx || !local_cu || !local_off || !pre || !fol)
        return fail(RM_ERR_INVALID_ARG, "metadata builder: NULL pointer");
    if (num_seqs <= 0 || T <= 0 || num_segments <= 0)
        return fail(RM_ERR_INVALID_ARG, "metadata builder: sizes must be positive");
    if (T % num_segments != 0)
        return fail(RM_ERR_SHAPE, "metadata builder: T=%d not a multiple of num_segments=%d", T,
                    num_segments);
    if (cu[0] != 0 || cu[num_seqs] != T)
        return fail(RM_ERR_METADATA, "cu_seqlens must start at 0 and end at T=%d", T);
    for (int32_t i = 0; i < num_seqs; ++i)
        if (cu[i + 1] <= cu[i])
            return fail(RM_ERR_METADATA, "cu_seqlens not strictly increasing at %d", i);
    const int32_t L = T / num_segments;
    // one pass over the sequences fills the per-token ids
    for (int32_t i = 0; i < num_seqs; ++i)
        for (int32_t t = cu[i]; t < cu[i + 1]; ++t) seq_idx[t] = i;
    // one merge pass of segment boundaries against sequence starts
    int32_t n = 0, next_seq = 1;  // cu[next_seq] is the first start not yet placed
    for (int32_t j = 0; j < num_segments; ++j) {
        const int32_t a = j * L, e = a + L;
        local_off[j] = n;
        local_cu[n++] = 0;
        while (next_seq < num_seqs && cu[next_seq] <= a) ++next_seq;
        while (next_seq < num_seqs && cu[next_seq] < e) local_cu[n++] = cu[next_seq++] - a;
        local_cu[n++] = L;
        pre[j] = cu[seq_idx[a]] / L;                 // segment of the start of a's sequence
        fol[j] = (cu[seq_idx[e - 1] + 1] - 1) / L + 1;  // 1 + segment of its last token
    }
    local_off[num_segments] = n;
    return RM_OK;
}

rm_status rm_cp_forward_prepare(const rm_cp_problem* p, const void* k, const void* v,
                                const float* g, float* M, float* dS, void* ws,
                                rm_stream_t stream) {
    (void)ws;
    rmcp::Dims d;
    rm_status st = check_problem(p, &d);
    if (st != RM_OK) return st;
    RM_NEED(k);
    RM_NEED(v);
    RM_NEED(g);
    RM_NEED(M);
    RM_NEED(dS);
    rmcp::Ptrs x;
    x.k = k;
    x.v = v;
    x.g = g;
    x.M = M;
    x.sum_out = dS;
    return launch(rmcp::Op::kForwardPrepare, p, d, x, stream);
}

rm_status rm_cp_compose_prefix(const rm_cp_problem* p, const float* M, const float* dS,
                               float* S_in, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status st = check_problem(p, &d);
    if (st != RM_OK) return st;
    RM_NEED(M);
    RM_NEED(dS);
    RM_NEED(S_in);
    rmcp::begin_launches();
    st = rmcp::launch_compose_prefix(d, M, dS, S_in, reinterpret_cast<cudaStream_t>(stream));
    if (st != RM_OK) return fail(st, "compose_prefix launch failed: %s",
                                 rmcp::cuda_error_text());
    return RM_OK;
}

rm_status rm_cp_forward_apply(const rm_cp_problem* p, const void* q, const void* k,
                              const void* v, const float* g, const float* S_in, void* o,
                              void* ws, rm_stream_t stream) {
    (void)ws;
    rmcp::Dims d;
    rm_status st = check_problem(p, &d);
    if (st != RM_OK) return st;
    RM_NEED(q);
    RM_NEED(k);
    RM_NEED(v);
    RM_NEED(g);
    RM_NEED(S_in);
    RM_NEED(o);
    rmcp::Ptrs x;
    x.q = q;
    x.k = k;
    x.v = v;
    x.g = g;
    x.S_in = S_in;
    x.out0 = o;
    return launch(rmcp::Op::kForwardApply, p, d, x, stream);
}

rm_status rm_cp_forward_fused(const rm_cp_problem* p, const void* q, const void* k,
                              const void* v, const float* g, float* M, float* dS, float* S_in,
                              void* o, void* ws, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status st = check_problem(p, &d);
    if (st != RM_OK) return st;
    RM_NEED(q);
    RM_NEED(k);
    RM_NEED(v);
    RM_NEED(g);
    RM_NEED(M);
    RM_NEED(dS);
    RM_NEED(S_in);
    RM_NEED(o);
    if (!rmcp::tc_supports(d, p->dtype)) {
        // the generic kernels: the three calls in order
        st = rm_cp_forward_prepare(p, k, v, g, M, dS, ws, stream);
        if (st == RM_OK) st = rm_cp_compose_prefix(p, M, dS, S_in, stream);
        if (st == RM_OK) st = rm_cp_forward_apply(p, q, k, v, g, S_in, o, ws, stream);
        return st;
    }
    RM_NEED(ws);
    rmcp::Ptrs x;
    x.q = q;
    x.k = k;
    x.v = v;
    x.g = g;
    x.M = M;
    x.sum_out = dS;
    x.S_in_out = S_in;
    x.out0 = o;
    x.ws = ws;
    rmcp::begin_launches();
    st = rmcp::tc_launch_fused_forward(d, x, reinterpret_cast<cudaStream_t>(stream));
    if (st == RM_ERR_CUDA) {
        const int mr = rmcp::tc::last_map_result();
        if (mr != 0)
            return fail(RM_ERR_CUDA, "fused forward launch failed: no tensor map (CUresult %d)", mr);
        return fail(RM_ERR_CUDA, "fused forward launch failed: %s", rmcp::cuda_error_text());
    }
    return st;
}

rm_status rm_cp_backward_prepare(const rm_cp_problem* p, const void* q, const void* k,
                                 const void* v, const float* g, const float* S_in,
                                 const void* dO, float* gamma, void* dq, void* ws,
                                 rm_stream_t stream) {
    rmcp::Dims d;
    rm_status st = check_problem(p, &d);
    if (st != RM_OK) return st;
    RM_NEED(q);
    RM_NEED(k);
    RM_NEED(v);
    RM_NEED(g);
    RM_NEED(S_in);
    RM_NEED(dO);
    RM_NEED(gamma);
    RM_NEED(dq);
    RM_NEED(ws);
    rmcp::Ptrs x;
    x.q = q;
    x.k = k;
    x.v = v;
    x.g = g;
    x.S_in = S_in;
    x.dO = dO;
    x.sum_out = gamma;
    x.out0 = dq;
    x.ws_f32 = static_cast<float*>(ws);
    return launch(rmcp::Op::kBackwardPrepare, p, d, x, stream);
}

rm_status rm_cp_compose_suffix(const rm_cp_problem* p, const float* M, const float* gamma,
                               float* dS_out, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status st = check_problem(p, &d);
    if (st != RM_OK) return st;
    RM_NEED(M);
    RM_NEED(gamma);
    RM_NEED(dS_out);
    rmcp::begin_launches();
    st = rmcp::launch_compose_suffix(d, M, gamma, dS_out, reinterpret_cast<cudaStream_t>(stream));
    if (st != RM_OK) return fail(st, "compose_suffix launch failed: %s",
                                 rmcp::cuda_error_text());
    return RM_OK;
}

rm_status rm_cp_backward_apply(const rm_cp_problem* p, const void* q, const void* k,
                               const void* v, const float* g, const void* dO,
                               const float* S_in, const float* dS_out, void* dk, void* dv,
                               float* dg, void* ws, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status st = check_problem(p, &d);
    if (st != RM_OK) return st;
    RM_NEED(q);
    RM_NEED(k);
    RM_NEED(v);
    RM_NEED(g);
    RM_NEED(dO);
    RM_NEED(S_in);
    RM_NEED(dS_out);
    RM_NEED(dk);
    RM_NEED(dv);
    RM_NEED(dg);
    RM_NEED(ws);
    rmcp::Ptrs x;
    x.q = q;
    x.k = k;
    x.v = v;
    x.g = g;
    x.dO = dO;
    x.S_in = S_in;
    x.dS_out = dS_out;
    x.out0 = dk;
    x.out1 = dv;
    x.dg = dg;
    x.ws_f32 = static_cast<float*>(ws);
    return launch(rmcp::Op::kBackwardApply, p, d, x, stream);
}

}  // extern "C"
