// host_step.cu -- rm_cp_step_host: one step of the path from host buffers.
//
// The inputs go in on one stream, the six compute calls run on another and
// the results come back on a third, ordered by three events per device
// buffer set so that successive steps on alternating sets overlap their
// copies with each other's kernels.  Host-side orchestration only: every
// arithmetic step is one of the library's own compute calls.
#include <cstdio>

#include "internal.h"

namespace {

// device pointers: non-null and 16-byte aligned, as for every compute call
#define RM_NEED_HS(ptr)                                      \
    do {                                                     \
        rm_status s_ = rmcp::api_need((ptr), #ptr);          \
        if (s_ != RM_OK) return s_;                          \
    } while (0)
// host buffers, events and the argument structs: non-null
#define RM_NONNULL_HS(ptr)                                                         \
    do {                                                                           \
        if ((ptr) == nullptr) return rmcp::api_fail(RM_ERR_INVALID_ARG, #ptr " is NULL"); \
    } while (0)

struct Copy {
    void* dst;
    const void* src;
    size_t bytes;
};

rm_status cuda_fail(cudaError_t e, const char* what) {
    char buf[160];
    snprintf(buf, sizeof(buf), "rm_cp_step_host: %s: %s", what, cudaGetErrorString(e));
    return rmcp::api_fail(RM_ERR_CUDA, buf);
}

}  // namespace

extern "C" rm_status rm_cp_event_create(void** event) {
    if (event == nullptr) return rmcp::api_fail(RM_ERR_INVALID_ARG, "event is NULL");
    cudaEvent_t e = nullptr;
    const cudaError_t err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (err != cudaSuccess) return rmcp::api_fail(RM_ERR_CUDA, cudaGetErrorString(err));
    *event = static_cast<void*>(e);
    return RM_OK;
}

extern "C" rm_status rm_cp_event_destroy(void* event) {
    if (event == nullptr) return rmcp::api_fail(RM_ERR_INVALID_ARG, "event is NULL");
    const cudaError_t err = cudaEventDestroy(static_cast<cudaEvent_t>(event));
    if (err != cudaSuccess) return rmcp::api_fail(RM_ERR_CUDA, cudaGetErrorString(err));
    return RM_OK;
}

extern "C" rm_status rm_cp_step_host(const rm_cp_problem* p, const rm_cp_host_io* host,
                                     const rm_cp_step_set* set, const rm_cp_step_state* st,
                                     rm_stream_t compute, rm_stream_t h2d, rm_stream_t d2h) {
    rmcp::Dims d;
    rm_status s = rmcp::api_check_problem(p, &d);
    if (s != RM_OK) return s;
    RM_NONNULL_HS(host);
    RM_NONNULL_HS(set);
    RM_NONNULL_HS(st);
    const bool bwd = host->dO != nullptr;
    RM_NONNULL_HS(host->q);
    RM_NONNULL_HS(host->k);
    RM_NONNULL_HS(host->v);
    RM_NONNULL_HS(host->g);
    RM_NONNULL_HS(host->o);
    RM_NEED_HS(set->q);
    RM_NEED_HS(set->k);
    RM_NEED_HS(set->v);
    RM_NEED_HS(set->g);
    RM_NEED_HS(set->o);
    RM_NONNULL_HS(set->loaded);
    RM_NONNULL_HS(set->computed);
    RM_NONNULL_HS(set->drained);
    RM_NEED_HS(st->M);
    RM_NEED_HS(st->dS);
    RM_NEED_HS(st->S_in);
    if (bwd) {
        RM_NONNULL_HS(host->dq);
        RM_NONNULL_HS(host->dk);
        RM_NONNULL_HS(host->dv);
        RM_NONNULL_HS(host->dg);
        RM_NEED_HS(set->dO);
        RM_NEED_HS(set->dq);
        RM_NEED_HS(set->dk);
        RM_NEED_HS(set->dv);
        RM_NEED_HS(set->dg);
        RM_NEED_HS(st->gamma);
        RM_NEED_HS(st->dS_out);
        RM_NEED_HS(st->ws);
    }

    const size_t e = p->dtype == RM_BF16 ? 2 : 4;
    const size_t ntok = size_t(d.B) * size_t(d.T) * size_t(d.H);
    const size_t bk = ntok * size_t(d.Dk) * e, bv = ntok * size_t(d.Dv) * e;
    const size_t bg = ntok * 4 * (d.vg ? size_t(d.Dk) : 1);  // g, dg: one per key dim with vector gates
    const size_t bq = size_t(d.B) * size_t(d.T) * size_t(d.qh) * size_t(d.Dk) * e;
    const Copy ins[5] = {{set->q, host->q, bq}, {set->k, host->k, bk}, {set->v, host->v, bv},
                         {set->g, host->g, bg}, {set->dO, host->dO, bv}};
    const Copy outs[5] = {{host->o, set->o, bv}, {host->dq, set->dq, bk}, {host->dk, set->dk, bk},
                          {host->dv, set->dv, bv}, {host->dg, set->dg, bg}};
    const int nin = bwd ? 5 : 4, nout = bwd ? 5 : 1;
    auto cs = reinterpret_cast<cudaStream_t>(compute);
    auto hs = reinterpret_cast<cudaStream_t>(h2d);
    auto ds = reinterpret_cast<cudaStream_t>(d2h);
    auto loaded = static_cast<cudaEvent_t>(set->loaded);
    auto computed = static_cast<cudaEvent_t>(set->computed);
    auto drained = static_cast<cudaEvent_t>(set->drained);

    // inputs: once this set's previous kernels have read the old ones
    cudaError_t err = cudaStreamWaitEvent(hs, computed, 0);
    for (int i = 0; i < nin && err == cudaSuccess; ++i)
        err = cudaMemcpyAsync(ins[i].dst, ins[i].src, ins[i].bytes, cudaMemcpyHostToDevice, hs);
    if (err == cudaSuccess) err = cudaEventRecord(loaded, hs);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(cs, loaded, 0);
    // outputs are overwritten once this set's previous results have left
    if (err == cudaSuccess) err = cudaStreamWaitEvent(cs, drained, 0);
    if (err != cudaSuccess) return cuda_fail(err, "input copies");

    s = rm_cp_forward_prepare(p, set->k, set->v, set->g, st->M, st->dS, st->ws, compute);
    if (s == RM_OK) s = rm_cp_compose_prefix(p, st->M, st->dS, st->S_in, compute);
    if (s == RM_OK)
        s = rm_cp_forward_apply(p, set->q, set->k, set->v, set->g, st->S_in, set->o, st->ws, compute);
    if (bwd) {
        if (s == RM_OK)
            s = rm_cp_backward_prepare(p, set->q, set->k, set->v, set->g, st->S_in, set->dO, st->gamma,
                                       set->dq, st->ws, compute);
        if (s == RM_OK) s = rm_cp_compose_suffix(p, st->M, st->gamma, st->dS_out, compute);
        if (s == RM_OK)
            s = rm_cp_backward_apply(p, set->q, set->k, set->v, set->g, set->dO, st->S_in, st->dS_out,
                                     set->dk, set->dv, set->dg, st->ws, compute);
    }
    if (s != RM_OK) return s;

    err = cudaEventRecord(computed, cs);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(ds, computed, 0);
    for (int i = 0; i < nout && err == cudaSuccess; ++i)
        err = cudaMemcpyAsync(outs[i].dst, outs[i].src, outs[i].bytes, cudaMemcpyDeviceToHost, ds);
    if (err == cudaSuccess) err = cudaEventRecord(drained, ds);
    if (err != cudaSuccess) return cuda_fail(err, "output copies");
    return RM_OK;
}
