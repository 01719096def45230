// common.cuh -- device helpers and launch-parameter block shared by the
// kernels of the chunkwise gated linear attention library (internal header).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rm_cp.h"

namespace rmcp {

// Launch parameters derived from rm_cp_problem on the host.
struct Dims {
    int B, T, H, Dk, Dv;
    int nseg;   // segments per row
    int L;      // tokens per segment
    float scale;
    const int32_t* seq_idx;          // device [T] or nullptr
    const int32_t* preceding_start;  // device [nseg] or nullptr
    const int32_t* following_stop;   // device [nseg] or nullptr
    int qh;     // query heads (rows of q per token)
    int qdiv;   // H / qh: head h reads query row h / qdiv
    int vg;     // 1: one gate per key dimension (g [B,T,H,Dk], M [nseg,B,H,Dk])
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Token t of a row starts a sequence: the row's first token or a change of id.
__device__ __forceinline__ bool starts_sequence(const int32_t* seq_idx, int t) {
    if (t == 0) return true;
    if (seq_idx == nullptr) return false;
    return __ldg(seq_idx + t) != __ldg(seq_idx + t - 1);
}

__device__ __forceinline__ bool same_sequence(const int32_t* seq_idx, int s, int t) {
    if (seq_idx == nullptr) return true;
    return __ldg(seq_idx + s) == __ldg(seq_idx + t);
}

__device__ __forceinline__ int64_t qk_off(const Dims& d, int b, int t, int h) {
    return ((int64_t(b) * d.T + t) * d.H + h) * d.Dk;
}
// q row of head h (heads share query rows when qh < H)
__device__ __forceinline__ int64_t q_off(const Dims& d, int b, int t, int h) {
    return ((int64_t(b) * d.T + t) * d.qh + h / d.qdiv) * d.Dk;
}
__device__ __forceinline__ int64_t v_off(const Dims& d, int b, int t, int h) {
    return ((int64_t(b) * d.T + t) * d.H + h) * d.Dv;
}
__device__ __forceinline__ int64_t g_off(const Dims& d, int b, int t, int h) {
    return (int64_t(b) * d.T + t) * d.H + h;
}
// summary [nseg, B, H, Dk, Dv]
__device__ __forceinline__ int64_t sum_off(const Dims& d, int j, int b, int h) {
    return ((int64_t(j) * d.B + b) * d.H + h) * int64_t(d.Dk) * d.Dv;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace rmcp
