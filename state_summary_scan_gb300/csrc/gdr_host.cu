// gdr_host.cu -- C ABI of the gated delta rule (include/rm_cp.h, rm_gdr_*):
// host-side validation and launches.  Nothing here allocates or synchronises.
#include <cstdio>

#include "internal.h"

namespace {

using rmcp::api_fail;

rm_status check_gdr(const rm_cp_problem* p, rmcp::Dims* d) {
    rm_status s = rmcp::api_check_problem(p, d);
    if (s != RM_OK) return s;
    if (d->vg) return api_fail(RM_ERR_INVALID_ARG, "the gated delta rule takes one gate per head");
    if (!rmcp::gdr_supports(*d))
        return api_fail(RM_ERR_UNSUPPORTED,
                        "the gated delta rule takes Dk in {16, 32, 64, 128}, Dv a multiple of 8 in "
                        "[8, 128] and segment lengths that are multiples of 16");
    return RM_OK;
}

rm_status run(rmcp::GdrOp op, const rm_cp_problem* p, const rmcp::Dims& d, const rmcp::GdrPtrs& x,
              rm_stream_t stream) {
    // the four sweeps take the tensor cores where they can (the folds stay generic)
    const bool tc = op != rmcp::GdrOp::kComposePrefix && op != rmcp::GdrOp::kComposeSuffix &&
                    rmcp::gdrtc_supports(d, p->dtype);
    rmcp::begin_launches();
    if (tc) return rmcp::launch_gdrtc(op, d, x, reinterpret_cast<cudaStream_t>(stream));  // reports its own failures
    rm_status st = rmcp::launch_gdr(op, d, p->dtype, x, reinterpret_cast<cudaStream_t>(stream));
    if (st == RM_ERR_CUDA) {
        char msg[256];
        std::snprintf(msg, sizeof(msg), "gated delta rule launch failed: %s",
                      rmcp::cuda_error_text());
        return api_fail(RM_ERR_CUDA, msg);
    }
    if (st != RM_OK) return api_fail(st, "gated delta rule launch refused");
    return RM_OK;
}

}  // namespace

#define RM_NEED_GDR(ptr)                                \
    do {                                                \
        rm_status s_ = rmcp::api_need((ptr), #ptr);     \
        if (s_ != RM_OK) return s_;                     \
    } while (0)

extern "C" {

int32_t rm_gdr_path(const rm_cp_problem* p) {
    rmcp::Dims d;
    if (rmcp::api_check_problem(p, &d) != RM_OK || d.vg || !rmcp::gdr_supports(d)) return -1;
    return rmcp::gdrtc_supports(d, p->dtype) ? 1 : 0;
}

size_t rm_gdr_workspace_size(const rm_cp_problem* p) {
    rmcp::Dims d;
    if (rmcp::api_check_problem(p, &d) != RM_OK || d.vg || !rmcp::gdr_supports(d)) return 0;
    return rmcp::gdr_workspace_bytes(d);
}

rm_status rm_gdr_forward_prepare(const rm_cp_problem* p, const void* k, const void* v,
                                 const float* g, const float* beta, float* M, float* dS, void* ws,
                                 rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = check_gdr(p, &d);
    if (s != RM_OK) return s;
    RM_NEED_GDR(k);
    RM_NEED_GDR(v);
    RM_NEED_GDR(g);
    RM_NEED_GDR(beta);
    RM_NEED_GDR(M);
    RM_NEED_GDR(dS);
    RM_NEED_GDR(ws);
    rmcp::GdrPtrs x;
    x.k = k;
    x.v = v;
    x.g = g;
    x.beta = beta;
    x.M = M;
    x.dS = dS;
    x.ws = static_cast<float*>(ws);
    return run(rmcp::GdrOp::kPrepare, p, d, x, stream);
}

rm_status rm_gdr_compose_prefix(const rm_cp_problem* p, const float* M, const float* dS,
                                float* S_in, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = check_gdr(p, &d);
    if (s != RM_OK) return s;
    RM_NEED_GDR(M);
    RM_NEED_GDR(dS);
    RM_NEED_GDR(S_in);
    rmcp::GdrPtrs x;
    x.M = const_cast<float*>(M);
    x.dS = const_cast<float*>(dS);
    x.S_in_out = S_in;
    return run(rmcp::GdrOp::kComposePrefix, p, d, x, stream);
}

rm_status rm_gdr_forward_apply(const rm_cp_problem* p, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, const float* S_in, void* o, void* ws,
                               rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = check_gdr(p, &d);
    if (s != RM_OK) return s;
    RM_NEED_GDR(q);
    RM_NEED_GDR(k);
    RM_NEED_GDR(v);
    RM_NEED_GDR(g);
    RM_NEED_GDR(beta);
    RM_NEED_GDR(S_in);
    RM_NEED_GDR(o);
    RM_NEED_GDR(ws);
    rmcp::GdrPtrs x;
    x.q = q;
    x.k = k;
    x.v = v;
    x.g = g;
    x.beta = beta;
    x.S_in = S_in;
    x.o = o;
    x.ws = static_cast<float*>(ws);
    return run(rmcp::GdrOp::kApply, p, d, x, stream);
}

rm_status rm_gdr_backward_prepare(const rm_cp_problem* p, const void* q, const void* k,
                                  const void* v, const float* g, const float* beta,
                                  const float* S_in, const void* dO, float* gamma, void* dq,
                                  void* ws, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = check_gdr(p, &d);
    if (s != RM_OK) return s;
    RM_NEED_GDR(q);
    RM_NEED_GDR(k);
    RM_NEED_GDR(v);
    RM_NEED_GDR(g);
    RM_NEED_GDR(beta);
    RM_NEED_GDR(S_in);
    RM_NEED_GDR(dO);
    RM_NEED_GDR(gamma);
    RM_NEED_GDR(dq);
    RM_NEED_GDR(ws);
    rmcp::GdrPtrs x;
    x.q = q;
    x.k = k;
    x.v = v;
    x.g = g;
    x.beta = beta;
    x.S_in = S_in;
    x.dO = dO;
    x.gamma_out = gamma;
    x.dq = dq;
    x.ws = static_cast<float*>(ws);
    return run(rmcp::GdrOp::kBackwardPrepare, p, d, x, stream);
}

rm_status rm_gdr_compose_suffix(const rm_cp_problem* p, const float* M, const float* gamma,
                                float* dS_out, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = check_gdr(p, &d);
    if (s != RM_OK) return s;
    RM_NEED_GDR(M);
    RM_NEED_GDR(gamma);
    RM_NEED_GDR(dS_out);
    rmcp::GdrPtrs x;
    x.M = const_cast<float*>(M);
    x.gamma = gamma;
    x.dS_out_out = dS_out;
    return run(rmcp::GdrOp::kComposeSuffix, p, d, x, stream);
}

rm_status rm_gdr_backward_apply(const rm_cp_problem* p, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, const void* dO,
                                const float* dS_out, void* dk, void* dv, float* dg, float* dbeta,
                                void* ws, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = check_gdr(p, &d);
    if (s != RM_OK) return s;
    RM_NEED_GDR(q);
    RM_NEED_GDR(k);
    RM_NEED_GDR(v);
    RM_NEED_GDR(g);
    RM_NEED_GDR(beta);
    RM_NEED_GDR(dO);
    RM_NEED_GDR(dS_out);
    RM_NEED_GDR(dk);
    RM_NEED_GDR(dv);
    RM_NEED_GDR(dg);
    RM_NEED_GDR(dbeta);
    RM_NEED_GDR(ws);
    rmcp::GdrPtrs x;
    x.q = q;
    x.k = k;
    x.v = v;
    x.g = g;
    x.beta = beta;
    x.dO = dO;
    x.dS_out = dS_out;
    x.dk = dk;
    x.dv = dv;
    x.dg = dg;
    x.dbeta = dbeta;
    x.ws = static_cast<float*>(ws);
    return run(rmcp::GdrOp::kBackwardApply, p, d, x, stream);
}

}  // extern "C"
