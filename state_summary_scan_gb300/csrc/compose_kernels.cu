// compose_kernels.cu -- the summary scans of chunkwise_cp_forward and
// chunkwise_cp_backward (Megatron-Core page "core.ssm.context_parallel.chunkwise"):
//   prefix  S_in[j]   = summaries of segments [pre_j, j) applied in order to 0,
//           each one S <- M_i S + dS_i          (CPForwardUnpackedSummary)
//   suffix  dS_out[j] = summaries of segments (j, fol_j) applied from the
//           last one down, D <- M_i D + gamma_i  (CPBackwardUnpackedSummary)
// M is one scalar per (segment, row, head), or with vector gates one value
// per key dimension (a diagonal M, applied to state row i as M[i]).  Every
// thread owns four adjacent fp32 elements of one (row, head) state (always in
// one state row: Dv is a multiple of 8) and walks the segments serially;
// consecutive threads touch consecutive 16-byte words, so each segment step is
// one fully coalesced 128-bit stream over [B,H,Dk,Dv].  The loads of the next
// kPrefetch segments are issued before the dependent multiply-adds.
#include "internal.h"

namespace rmcp {

namespace {

constexpr int kThreads = 256;
constexpr int kPrefetch = 4;

__device__ __forceinline__ float4 axpy4(float m, float4 s, float4 x) {
    return make_float4(fmaf(m, s.x, x.x), fmaf(m, s.y, x.y), fmaf(m, s.z, x.z), fmaf(m, s.w, x.w));
}

__device__ __forceinline__ float4 ld4(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void st4(float* p, float4 x) {
    __stcs(reinterpret_cast<float4*>(p), x);
}

// Clamp metadata so that a bad value can never index outside [0, nseg).
__device__ __forceinline__ int clamp_i(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

// Offset of M for segment j of (row, head) bh: mstride = 1 (scalar gates) or
// Dk (vector gates, mrow = the state row of the thread's elements).
__device__ __forceinline__ int64_t m_at(int j, int BH, int bh, int mstride, int mrow) {
    return (int64_t(j) * BH + bh) * mstride + mrow;
}

__global__ void __launch_bounds__(kThreads) compose_prefix_kernel(
    int nseg, int BH, int64_t vec_per_state, int Dv, int mstride, const float* __restrict__ M,
    const float* __restrict__ dS, const int32_t* __restrict__ pre, float* __restrict__ S_in) {
    const int64_t gid = int64_t(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t per_seg = int64_t(BH) * vec_per_state;  // float4s per segment slab
    if (gid >= per_seg) return;
    const int bh = int(gid / vec_per_state);
    const int64_t e = gid * 4;                            // element offset inside a slab
    const int64_t slab = per_seg * 4;
    const int mrow = mstride > 1 ? int((gid - int64_t(bh) * vec_per_state) * 4 / Dv) : 0;

    float4 S = make_float4(0.f, 0.f, 0.f, 0.f);
    int start = 0;  // S = composition over [start, j)
    for (int j0 = 0; j0 < nseg; j0 += kPrefetch) {
        float4 x[kPrefetch];
        float m[kPrefetch];
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            if (j0 + u < nseg) {
                x[u] = ld4(dS + int64_t(j0 + u) * slab + e);
                m[u] = __ldg(M + m_at(j0 + u, BH, bh, mstride, mrow));
            }
        }
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int j = j0 + u;
            if (j >= nseg) break;
            const int pj = pre ? clamp_i(__ldg(pre + j), 0, j) : 0;
            if (pj != start) {
                // the prefix of segment j starts elsewhere: rebuild it from pj
                S = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int i = pj; i < j; ++i)
                    S = axpy4(__ldg(M + m_at(i, BH, bh, mstride, mrow)), S, ld4(dS + int64_t(i) * slab + e));
                start = pj;
            }
            st4(S_in + int64_t(j) * slab + e, S);
            S = axpy4(m[u], S, x[u]);
        }
    }
}

__global__ void __launch_bounds__(kThreads) compose_suffix_kernel(
    int nseg, int BH, int64_t vec_per_state, int Dv, int mstride, const float* __restrict__ M,
    const float* __restrict__ gamma, const int32_t* __restrict__ fol, float* __restrict__ dS_out) {
    const int64_t gid = int64_t(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t per_seg = int64_t(BH) * vec_per_state;
    if (gid >= per_seg) return;
    const int bh = int(gid / vec_per_state);
    const int64_t e = gid * 4;
    const int64_t slab = per_seg * 4;
    const int mrow = mstride > 1 ? int((gid - int64_t(bh) * vec_per_state) * 4 / Dv) : 0;

    float4 D = make_float4(0.f, 0.f, 0.f, 0.f);
    int stop = nseg;  // D = composition over (j, stop)
    for (int j0 = nseg - 1; j0 >= 0; j0 -= kPrefetch) {
        float4 x[kPrefetch];
        float m[kPrefetch];
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            if (j0 - u >= 0) {
                x[u] = ld4(gamma + int64_t(j0 - u) * slab + e);
                m[u] = __ldg(M + m_at(j0 - u, BH, bh, mstride, mrow));
            }
        }
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int j = j0 - u;
            if (j < 0) break;
            const int fj = fol ? clamp_i(__ldg(fol + j), j + 1, nseg) : nseg;
            if (fj != stop) {
                D = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int i = fj - 1; i > j; --i)
                    D = axpy4(__ldg(M + m_at(i, BH, bh, mstride, mrow)), D, ld4(gamma + int64_t(i) * slab + e));
                stop = fj;
            }
            st4(dS_out + int64_t(j) * slab + e, D);
            D = axpy4(m[u], D, x[u]);
        }
    }
}

}  // namespace

rm_status launch_compose_prefix(const Dims& d, const float* M, const float* dS, float* S_in,
                                cudaStream_t s) {
    const int64_t vps = int64_t(d.Dk) * d.Dv / 4;
    const int64_t n = int64_t(d.B) * d.H * vps;
    const int blocks = int((n + kThreads - 1) / kThreads);
    compose_prefix_kernel<<<blocks, kThreads, 0, s>>>(d.nseg, d.B * d.H, vps, d.Dv, d.vg ? d.Dk : 1,
                                                      M, dS, d.preceding_start, S_in);
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(1);
    return RM_OK;
}

rm_status launch_compose_suffix(const Dims& d, const float* M, const float* gamma,
                                float* dS_out, cudaStream_t s) {
    const int64_t vps = int64_t(d.Dk) * d.Dv / 4;
    const int64_t n = int64_t(d.B) * d.H * vps;
    const int blocks = int((n + kThreads - 1) / kThreads);
    compose_suffix_kernel<<<blocks, kThreads, 0, s>>>(d.nseg, d.B * d.H, vps, d.Dv, d.vg ? d.Dk : 1,
                                                      M, gamma, d.following_stop, dS_out);
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(1);
    return RM_OK;
}

}  // namespace rmcp
