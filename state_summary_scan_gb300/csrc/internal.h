// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace rmcp {

enum class Op { kForwardPrepare, kForwardApply, kBackwardPrepare, kBackwardApply };

// Device pointers of one call; unused ones are null.
struct Ptrs {
    const void* q = nullptr;
    const void* k = nullptr;
    const void* v = nullptr;
    const float* g = nullptr;
    const void* dO = nullptr;
    const float* S_in = nullptr;
    const float* dS_out = nullptr;
    float* M = nullptr;
    float* sum_out = nullptr;  // dS (forward prepare) or gamma (backward prepare)
    void* out0 = nullptr;      // o / dq / dk
    void* out1 = nullptr;      // dv
    float* dg = nullptr;
    float* ws_f32 = nullptr;   // per-token q.dq [B,T,H]
    void* ws = nullptr;        // the call's workspace (fused forward)
    float* S_in_out = nullptr; // S_in written by the fused forward
};

// adds n to the process-wide launch counter (rm_cp_launch_count)
void note_launch(int n);

// generic fp32 SIMT path (simt_kernels.cu)
bool generic_supports(const Dims& d);
rm_status launch_generic(Op op, const Dims& d, rm_dtype dt, const Ptrs& p, cudaStream_t s);

// gated delta rule (gdr_kernels.cu)
enum class GdrOp { kPrepare, kComposePrefix, kApply, kBackwardPrepare, kComposeSuffix, kBackwardApply };
struct GdrPtrs {
    const void* q = nullptr;
    const void* k = nullptr;
    const void* v = nullptr;
    const void* dO = nullptr;
    const float* g = nullptr;
    const float* beta = nullptr;
    float* M = nullptr;           // [nseg,B,H,Dk,Dk]: written by kPrepare, read by the folds
    float* dS = nullptr;          // written by kPrepare, read by kComposePrefix
    const float* S_in = nullptr;  // read by kApply, kBackwardPrepare
    float* S_in_out = nullptr;    // written by kComposePrefix
    const float* gamma = nullptr; // read by kComposeSuffix
    float* gamma_out = nullptr;   // written by kBackwardPrepare
    const float* dS_out = nullptr;  // read by kBackwardApply
    float* dS_out_out = nullptr;  // written by kComposeSuffix
    void* o = nullptr;
    void* dq = nullptr;
    void* dk = nullptr;
    void* dv = nullptr;
    float* dg = nullptr;
    float* dbeta = nullptr;
    float* ws = nullptr;          // the step's workspace: saved states (kBackwardPrepare ->
                                  // kBackwardApply) and, on the tensor cores, the per-chunk
                                  // factors (kPrepare -> the other sweeps)
};
bool gdr_supports(const Dims& d);
size_t gdr_workspace_bytes(const Dims& d);
rm_status launch_gdr(GdrOp op, const Dims& d, rm_dtype dt, const GdrPtrs& p, cudaStream_t s);
// its forward and backward sweeps on the tensor cores (gdrtc_kernels.cu)
bool gdrtc_supports(const Dims& d, rm_dtype dt);
rm_status launch_gdrtc(GdrOp op, const Dims& d, const GdrPtrs& p, cudaStream_t s);
rm_status gdrtc_read_timeout_flag(int* host_flag, int clear, int* dev_scratch, cudaStream_t s);

// vector (per key dimension) gates on the generic path (vg_kernels.cu)
rm_status launch_vg(Op op, const Dims& d, rm_dtype dt, const Ptrs& p, cudaStream_t s);
// vector gates on the tensor-core path (vgtc_kernels.cu)
bool vgtc_supports(const Dims& d, rm_dtype dt);
rm_status launch_vgtc(Op op, const Dims& d, const Ptrs& p, cudaStream_t s);
rm_status vgtc_read_timeout_flag(int* host_flag, int clear, int* dev_scratch, cudaStream_t s);

// host-side checks and launches of rm_cp_host.cu, for other entry points
rm_status api_check_problem(const rm_cp_problem* p, Dims* d);
rm_status api_need(const void* ptr, const char* name);
rm_status api_fail(rm_status s, const char* msg);
// Every compute entry point calls begin_launches() before its first CUDA
// call.  It makes the current device's primary context current on the calling
// thread (a thread that has made no runtime call yet, such as the thread
// PyTorch's autograd runs backward calls on, may have none, and the tensor-map
// encoder is a driver call that needs one) and clears a non-sticky error that
// an earlier, unrelated runtime call on the thread left pending
// (cudaGetLastError is per thread); a faulted context still fails the launches
// themselves.  launch_ok() checks the launch just made and keeps its error for
// the message cuda_error_text() gives.
void begin_launches();
bool launch_ok();
const char* cuda_error_text();
namespace tc {
int last_map_result();   // CUresult of the thread's last tensor-map encode
void clear_map_result();
}  // namespace tc
rm_status api_launch(Op op, const rm_cp_problem* p, const Dims& d, const Ptrs& ptrs,
                     rm_stream_t stream);

// summary scans (compose_kernels.cu)
rm_status launch_compose_prefix(const Dims& d, const float* M, const float* dS, float* S_in,
                                cudaStream_t s);
rm_status launch_compose_suffix(const Dims& d, const float* M, const float* gamma,
                                float* dS_out, cudaStream_t s);

// tensor-core path (tc_kernels.cu)
bool tc_supports(const Dims& d, rm_dtype dt);
bool tc_supports_op(Op op, const Dims& d, rm_dtype dt);
rm_status launch_tc(Op op, const Dims& d, const Ptrs& p, cudaStream_t s);
// the forward in one launch (prepare, composition, apply) and its workspace
size_t tc_fused_bytes(const Dims& d, rm_dtype dt);
rm_status tc_launch_fused_forward(const Dims& d, const Ptrs& p, cudaStream_t s);
rm_status tc_selftest_wait(uint32_t limit_us, cudaStream_t s);
rm_status tc_read_timeout_flag(int* host_flag, int clear, int* dev_scratch, cudaStream_t s);

}  // namespace rmcp
