// vg_kernels.cu -- the path with one gate per key dimension ("vector
// gates"): per row b and head h,
//     S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,   o_t = scale S_t^T q_t,
// alpha_t[i] = exp(g_t[i]) (all 0 when token t starts a sequence), so a
// segment's transition is the diagonal matrix M = diag(prod of alpha) of the
// general summary S_out = M S_in + delta_S (CPForwardUnpackedSummary on the
// Megatron-Core page "core.ssm.context_parallel.chunkwise"); M^T = M in the
// backward's dS_in = M^T dS_out + gamma.  The compositions of the summaries
// are the shared scan kernels (compose_kernels.cu) with M applied row by row.
//
// Like the scalar-gate generic path, one CTA walks one (segment, row, head)
// token by token in fp32 (both storage types), with the same two ownership
// patterns: a column owner keeps column j of the state in registers (the
// forward sweeps and gamma), a row owner keeps row i in shared memory (dq,
// and the adjoint for dk).  Per key dimension i the gate gradient is the
// reverse running sum, within a sequence, of q_t[i] dq_t[i] - k_t[i] dk_t[i]
// (the oracle's identity for vector gates), plus <S_out[i,:], dS_out[i,:]>
// for the segment's last sequence; the same-token term of the two products
// cancels exactly and is left out of both, as on the scalar path.
#include "internal.h"

namespace rmcp {

namespace {

constexpr int kTok = 16;  // tokens staged per tile

enum VgMode { kVgPrepare = 0, kVgApply = 1, kVgGamma = 2 };

// [B,T,H,Dk] offset of token t's gates (and of the per-dimension workspace)
__device__ __forceinline__ int64_t gv_off(const Dims& d, int b, int t, int h) {
    return ((int64_t(b) * d.T + t) * d.H + h) * d.Dk;
}

// ---------------------------------------------------------------------------
// Forward sweep, column owner (thread = column j of the state).
//   PREPARE: S from 0; writes dS and M[i] = prod alpha[i] (0 after a start).
//   APPLY  : S from S_in; writes o.
//   GAMMA  : gamma[:, j] = sum_t diag(P_t) scale q_t dO_t[j] with
//            P_t[i] = alpha_a[i] ... alpha_t[i] (0 once a sequence starts).
// grid (nseg, B*H, ceil(Dv / blockDim.x)); block 32..128 threads.  The
// per-dimension running products (P for GAMMA, M for PREPARE) are kept in
// shared memory by dimension owners (thread i takes dimensions i, i + block).
// ---------------------------------------------------------------------------
template <int DK, int MODE, typename T>
__global__ void __launch_bounds__(128) vg_column_sweep(Dims d, const T* __restrict__ q,
                                                       const T* __restrict__ k,
                                                       const T* __restrict__ v,
                                                       const float* __restrict__ g,
                                                       const T* __restrict__ dO,
                                                       const float* __restrict__ S_in,
                                                       T* __restrict__ o, float* __restrict__ M,
                                                       float* __restrict__ sum_out) {
    __shared__ float vec_s[kTok][DK];    // k (PREPARE/APPLY) or q (GAMMA)
    __shared__ float q_s[kTok][DK];      // q (APPLY)
    __shared__ float alpha_s[kTok][DK];  // alpha_t[i]; GAMMA: P_t[i]
    __shared__ float run_s[DK];          // running product over the tiles walked

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int col = blockIdx.z * blockDim.x + threadIdx.x;
    const bool active = col < d.Dv;
    const int a0 = seg * d.L;

    float st[DK];
    if (MODE == kVgApply && active) {
        const float* src = S_in + sum_off(d, seg, b, h);
#pragma unroll
        for (int i = 0; i < DK; ++i) st[i] = src[int64_t(i) * d.Dv + col];
    } else {
#pragma unroll
        for (int i = 0; i < DK; ++i) st[i] = 0.f;
    }
    for (int i = threadIdx.x; i < DK; i += blockDim.x) run_s[i] = 1.f;

    for (int t0 = a0; t0 < a0 + d.L; t0 += kTok) {
        __syncthreads();
        for (int e = threadIdx.x; e < kTok * DK; e += blockDim.x) {
            const int tt = e / DK, i = e % DK;
            const int t = t0 + tt;
            vec_s[tt][i] = to_f32(MODE == kVgGamma ? q[q_off(d, b, t, h) + i] : k[qk_off(d, b, t, h) + i]);
            if (MODE == kVgApply) q_s[tt][i] = to_f32(q[q_off(d, b, t, h) + i]);
            alpha_s[tt][i] = starts_sequence(d.seq_idx, t) ? 0.f : expf(g[gv_off(d, b, t, h) + i]);
        }
        float vr[kTok];
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt)
            vr[tt] = active ? to_f32((MODE == kVgGamma ? dO : v)[v_off(d, b, t0 + tt, h) + col]) : 0.f;
        __syncthreads();
        if (MODE != kVgApply) {
            // dimension owners: PREPARE multiplies M along; GAMMA turns the
            // tile's alphas into the prefix products P_t[i] (from the segment start)
            for (int i = threadIdx.x; i < DK; i += blockDim.x) {
                float r = run_s[i];
                for (int tt = 0; tt < kTok; ++tt) {
                    r *= alpha_s[tt][i];
                    if (MODE == kVgGamma) alpha_s[tt][i] = r;
                }
                run_s[i] = r;
            }
            __syncthreads();
        }
#pragma unroll 1
        for (int tt = 0; tt < kTok; ++tt) {
            if (MODE == kVgGamma) {
                const float w = d.scale * vr[tt];
#pragma unroll
                for (int i = 0; i < DK; ++i) st[i] = fmaf(alpha_s[tt][i] * w, vec_s[tt][i], st[i]);
            } else {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < DK; ++i) {
                    st[i] = fmaf(alpha_s[tt][i], st[i], vec_s[tt][i] * vr[tt]);
                    if (MODE == kVgApply) acc = fmaf(st[i], q_s[tt][i], acc);
                }
                if (MODE == kVgApply && active)
                    o[v_off(d, b, t0 + tt, h) + col] = from_f32<T>(d.scale * acc);
            }
        }
    }

    if (MODE != kVgApply) {
        if (active) {
            float* dst = sum_out + sum_off(d, seg, b, h);
#pragma unroll
            for (int i = 0; i < DK; ++i) dst[int64_t(i) * d.Dv + col] = st[i];
        }
        if (MODE == kVgPrepare && blockIdx.z == 0) {
            __syncthreads();
            float* m = M + ((int64_t(seg) * d.B + b) * d.H + h) * DK;
            for (int i = threadIdx.x; i < DK; i += blockDim.x) m[i] = run_s[i];
        }
    }
}

// ---------------------------------------------------------------------------
// dq sweep, row owner (thread = row i of the state, S in shared memory):
// dq_t[i] = scale (alpha_t[i] S_{t-1}[i,:] . dO_t + k_t[i] (v_t . dO_t)),
// qdq[t, i] = q_t[i] times the first part (the gate gradient's q.dq without
// its same-token term).  grid (nseg, B*H); block DK threads (>= 32).
// ---------------------------------------------------------------------------
template <int DK, typename T>
__global__ void __launch_bounds__(128) vg_dq_sweep(Dims d, const T* __restrict__ q,
                                                   const T* __restrict__ k,
                                                   const T* __restrict__ v,
                                                   const float* __restrict__ g,
                                                   const T* __restrict__ dO,
                                                   const float* __restrict__ S_in,
                                                   T* __restrict__ dq, float* __restrict__ qdq) {
    extern __shared__ float smem[];
    const int pitch = d.Dv + 1;
    float* S = smem;                  // [DK][pitch]
    float* v_s = S + DK * pitch;      // [kTok][Dv]
    float* do_s = v_s + kTok * d.Dv;  // [kTok][Dv]
    __shared__ float vdo_s[kTok];

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int i = threadIdx.x;
    const int a0 = seg * d.L;

    const float* src = S_in + sum_off(d, seg, b, h);
    for (int e = threadIdx.x; e < DK * d.Dv; e += blockDim.x) S[(e / d.Dv) * pitch + e % d.Dv] = src[e];

    for (int t0 = a0; t0 < a0 + d.L; t0 += kTok) {
        __syncthreads();
        for (int e = threadIdx.x; e < kTok * d.Dv; e += blockDim.x) {
            const int tt = e / d.Dv, j = e % d.Dv;
            const int64_t off = v_off(d, b, t0 + tt, h) + j;
            v_s[e] = to_f32(v[off]);
            do_s[e] = to_f32(dO[off]);
        }
        __syncthreads();
        for (int tt = threadIdx.x >> 5; tt < kTok; tt += blockDim.x >> 5) {
            float x = 0.f;
            for (int j = threadIdx.x & 31; j < d.Dv; j += 32) x = fmaf(v_s[tt * d.Dv + j], do_s[tt * d.Dv + j], x);
            x = warp_sum(x);
            if ((threadIdx.x & 31) == 0) vdo_s[tt] = x;
        }
        __syncthreads();
        if (i < DK) {
            float* row = S + i * pitch;
#pragma unroll 1
            for (int tt = 0; tt < kTok; ++tt) {
                const int t = t0 + tt;
                const float alpha = starts_sequence(d.seq_idx, t) ? 0.f : expf(g[gv_off(d, b, t, h) + i]);
                const float kr = to_f32(k[qk_off(d, b, t, h) + i]);
                const float qr = to_f32(q[q_off(d, b, t, h) + i]);
                const float* vv = v_s + tt * d.Dv;
                const float* dd = do_s + tt * d.Dv;
                float old_acc = 0.f;
                for (int j = 0; j < d.Dv; ++j) {
                    const float s_old = row[j];
                    row[j] = fmaf(alpha, s_old, kr * vv[j]);
                    old_acc = fmaf(s_old, dd[j], old_acc);
                }
                const float hist = d.scale * alpha * old_acc;
                dq[qk_off(d, b, t, h) + i] = from_f32<T>(fmaf(d.scale * kr, vdo_s[tt], hist));
                qdq[gv_off(d, b, t, h) + i] = qr * hist;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Reverse sweep: the adjoint D (row owners, shared memory) from dS_out at the
// segment's last token, D_t[i,:] = scale q_t[i] dO_t + alpha_{t+1}[i] D_{t+1}[i,:];
// dk (row owners), dv (column owners), and per dimension the gate gradient's
// reverse running sum, kept by the row owner of that dimension.
// grid (nseg, B*H); block max(DK, Dv) rounded up to 32 (<= 256).
// ---------------------------------------------------------------------------
template <int DK, typename T>
__global__ void __launch_bounds__(256) vg_reverse_sweep(Dims d, const T* __restrict__ q,
                                                        const T* __restrict__ k,
                                                        const T* __restrict__ v,
                                                        const float* __restrict__ g,
                                                        const T* __restrict__ dO,
                                                        const float* __restrict__ S_in,
                                                        const float* __restrict__ dS_out,
                                                        const float* __restrict__ qdq,
                                                        T* __restrict__ dk, T* __restrict__ dv,
                                                        float* __restrict__ dg) {
    extern __shared__ float smem[];
    const int pitch = d.Dv + 1;
    float* D = smem;                  // [DK][pitch]
    float* v_s = D + DK * pitch;      // [kTok][Dv]
    float* do_s = v_s + kTok * d.Dv;  // [kTok][Dv]
    float* k_s = do_s + kTok * d.Dv;  // [kTok][DK]
    __shared__ float vdo_s[kTok];

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int a0 = seg * d.L, e0 = a0 + d.L;
    const int i = threadIdx.x;  // row owner for i < DK

    // D <- dS_out[seg]; run[i] = <S_out[i,:], dS_out[i,:]> with S_out read as S_in[seg+1]
    const float* dso = dS_out + sum_off(d, seg, b, h);
    for (int e = threadIdx.x; e < DK * d.Dv; e += blockDim.x) D[(e / d.Dv) * pitch + e % d.Dv] = dso[e];
    float run = 0.f;
    if (i < DK && seg + 1 < d.nseg) {
        const float* so = S_in + sum_off(d, seg + 1, b, h) + int64_t(i) * d.Dv;
        const float* dr = dso + int64_t(i) * d.Dv;
        for (int j = 0; j < d.Dv; ++j) run = fmaf(so[j], dr[j], run);
    }

    for (int t0 = e0 - kTok; t0 >= a0; t0 -= kTok) {
        __syncthreads();
        for (int e = threadIdx.x; e < kTok * d.Dv; e += blockDim.x) {
            const int tt = e / d.Dv, j = e % d.Dv;
            const int64_t off = v_off(d, b, t0 + tt, h) + j;
            v_s[e] = to_f32(v[off]);
            do_s[e] = to_f32(dO[off]);
        }
        for (int e = threadIdx.x; e < kTok * DK; e += blockDim.x) {
            const int tt = e / DK, r = e % DK;
            k_s[e] = to_f32(k[qk_off(d, b, t0 + tt, h) + r]);
        }
        __syncthreads();
        for (int tt = threadIdx.x >> 5; tt < kTok; tt += blockDim.x >> 5) {
            float x = 0.f;
            for (int j = threadIdx.x & 31; j < d.Dv; j += 32) x = fmaf(v_s[tt * d.Dv + j], do_s[tt * d.Dv + j], x);
            x = warp_sum(x);
            if ((threadIdx.x & 31) == 0) vdo_s[tt] = x;
        }
        __syncthreads();
#pragma unroll 1
        for (int tt = kTok - 1; tt >= 0; --tt) {
            const int t = t0 + tt;
            // phase 1: row owners update D, form dk and the gate gradient
            if (i < DK) {
                // beta multiplies D_{t+1}: alpha_{t+1}[i] inside the segment,
                // 1 at its last token (D starts as dS_out there)
                const float beta = (t + 1 < e0)
                    ? (starts_sequence(d.seq_idx, t + 1) ? 0.f : expf(g[gv_off(d, b, t + 1, h) + i]))
                    : 1.f;
                float* row = D + i * pitch;
                const float qi = d.scale * to_f32(q[q_off(d, b, t, h) + i]);
                const float* vv = v_s + tt * d.Dv;
                const float* dd = do_s + tt * d.Dv;
                float old_acc = 0.f;
                for (int j = 0; j < d.Dv; ++j) {
                    const float x_old = row[j];
                    row[j] = fmaf(beta, x_old, qi * dd[j]);
                    old_acc = fmaf(x_old, vv[j], old_acc);
                }
                const float fut = beta * old_acc;
                dk[qk_off(d, b, t, h) + i] = from_f32<T>(fmaf(qi, vdo_s[tt], fut));
                run += __ldg(qdq + gv_off(d, b, t, h) + i) - k_s[tt * DK + i] * fut;
                const bool start = starts_sequence(d.seq_idx, t);
                dg[gv_off(d, b, t, h) + i] = start ? 0.f : run;
                if (start) run = 0.f;  // earlier tokens belong to another sequence
            }
            __syncthreads();
            // phase 2: column owners form dv
            if (threadIdx.x < d.Dv) {
                const int j = threadIdx.x;
                float acc = 0.f;
                for (int r = 0; r < DK; ++r) acc = fmaf(D[r * pitch + j], k_s[tt * DK + r], acc);
                dv[v_off(d, b, t, h) + j] = from_f32<T>(acc);
            }
            __syncthreads();
        }
    }
}

template <typename T>
rm_status launch_vg_T(Op op, const Dims& d, const Ptrs& p, cudaStream_t s) {
    const int BH = d.B * d.H;
    const int colthreads = d.Dv >= 128 ? 128 : ((d.Dv + 31) / 32) * 32;
    const dim3 cgrid(d.nseg, BH, (d.Dv + colthreads - 1) / colthreads);
    const T* q = static_cast<const T*>(p.q);
    const T* k = static_cast<const T*>(p.k);
    const T* v = static_cast<const T*>(p.v);
    const T* dO = static_cast<const T*>(p.dO);

#define RMCP_VG_DK_SWITCH(...)                                    \
    switch (d.Dk) {                                               \
        case 16: { constexpr int DK = 16; __VA_ARGS__; break; }   \
        case 32: { constexpr int DK = 32; __VA_ARGS__; break; }   \
        case 64: { constexpr int DK = 64; __VA_ARGS__; break; }   \
        case 128: { constexpr int DK = 128; __VA_ARGS__; break; } \
        default: return RM_ERR_UNSUPPORTED;                       \
    }

    switch (op) {
        case Op::kForwardPrepare:
            RMCP_VG_DK_SWITCH((vg_column_sweep<DK, kVgPrepare, T><<<cgrid, colthreads, 0, s>>>(
                d, nullptr, k, v, p.g, nullptr, nullptr, nullptr, p.M, p.sum_out)));
            break;
        case Op::kForwardApply:
            RMCP_VG_DK_SWITCH((vg_column_sweep<DK, kVgApply, T><<<cgrid, colthreads, 0, s>>>(
                d, q, k, v, p.g, nullptr, p.S_in, static_cast<T*>(p.out0), nullptr, nullptr)));
            break;
        case Op::kBackwardPrepare: {
            RMCP_VG_DK_SWITCH((vg_column_sweep<DK, kVgGamma, T><<<cgrid, colthreads, 0, s>>>(
                d, q, nullptr, nullptr, p.g, dO, nullptr, nullptr, nullptr, p.sum_out)));
            if (!rmcp::launch_ok()) return RM_ERR_CUDA;
            const int threads = d.Dk < 32 ? 32 : d.Dk;
            const size_t smem = sizeof(float) * (size_t(d.Dk) * (d.Dv + 1) + 2 * kTok * d.Dv);
            RMCP_VG_DK_SWITCH({
                auto fn = vg_dq_sweep<DK, T>;
                if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                    return RM_ERR_CUDA;
                fn<<<dim3(d.nseg, BH), threads, smem, s>>>(d, q, k, v, p.g, dO, p.S_in,
                                                           static_cast<T*>(p.out0), p.ws_f32);
            });
            break;
        }
        case Op::kBackwardApply: {
            int threads = d.Dk > d.Dv ? d.Dk : d.Dv;
            threads = ((threads + 31) / 32) * 32;
            const size_t smem =
                sizeof(float) * (size_t(d.Dk) * (d.Dv + 1) + 2 * kTok * d.Dv + kTok * d.Dk);
            RMCP_VG_DK_SWITCH({
                auto fn = vg_reverse_sweep<DK, T>;
                if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                    return RM_ERR_CUDA;
                fn<<<dim3(d.nseg, BH), threads, smem, s>>>(
                    d, q, k, v, p.g, dO, p.S_in, p.dS_out, p.ws_f32,
                    static_cast<T*>(p.out0), static_cast<T*>(p.out1), p.dg);
            });
            break;
        }
        default:
            return RM_ERR_INVALID_ARG;
    }
#undef RMCP_VG_DK_SWITCH
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(op == Op::kBackwardPrepare ? 2 : 1);
    return RM_OK;
}

}  // namespace

rm_status launch_vg(Op op, const Dims& d, rm_dtype dt, const Ptrs& p, cudaStream_t s) {
    return dt == RM_F32 ? launch_vg_T<float>(op, d, p, s) : launch_vg_T<__nv_bfloat16>(op, d, p, s);
}

}  // namespace rmcp
