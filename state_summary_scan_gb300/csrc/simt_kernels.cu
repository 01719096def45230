// simt_kernels.cu -- generic fp32 SIMT path: one CTA per (segment, row, head)
// walks the segment token by token with the gated recurrence
//     S_t = alpha_t S_{t-1} + k_t v_t^T,   o_t = scale S_t^T q_t
// (alpha_t = exp(g_t), 0 at a sequence start), which is the plain form of the
// chunkwise method whose segment summaries the Megatron-Core page
// "core.ssm.context_parallel.chunkwise" describes.  It serves every supported
// head size and both storage types; the fp32 tolerance is met because all
// arithmetic is fp32 FMA.  The tensor-core path covers the large bf16 shapes.
//
// Two ownership patterns keep the inner loops free of block barriers:
//  - column owner: thread j holds column j of the Dk x Dv state in registers
//    (o_t = S^T q, the state update and gamma are column-local);
//  - row owner: thread i holds row i of the state in shared memory
//    (dq_t = S dO and dk_t = D v are row-local).
#include "internal.h"

namespace rmcp {

namespace {

constexpr int kTok = 16;  // tokens staged per tile

// ---------------------------------------------------------------------------
// Forward sweep, column owner.
//   PREPARE: S starts at 0; writes dS (end state) and M = exp(sum g) or 0.
//   APPLY  : S starts at S_in; writes o.
//   GAMMA  : accumulates gamma = sum_t P_t scale q_t dO_t^T, P_t = alpha_a..alpha_t
//            (column j of gamma in the register array instead of the state).
// grid (nseg, B*H, ceil(Dv / blockDim.x)); block = 32..128 threads, one column each.
// ---------------------------------------------------------------------------
enum SweepMode { kPrepare = 0, kApply = 1, kGamma = 2 };

template <int DK, int MODE, typename T>
__global__ void __launch_bounds__(128) simt_column_sweep(Dims d, const T* __restrict__ q,
                                                         const T* __restrict__ k,
                                                         const T* __restrict__ v,
                                                         const float* __restrict__ g,
                                                         const T* __restrict__ dO,
                                                         const float* __restrict__ S_in,
                                                         T* __restrict__ o, float* __restrict__ M,
                                                         float* __restrict__ sum_out) {
    __shared__ float vec_s[kTok][DK];   // k (PREPARE/APPLY) or q (GAMMA)
    __shared__ float q_s[kTok][DK];     // q (APPLY)
    __shared__ float alpha_s[kTok];
    __shared__ float g_s[kTok];
    __shared__ int start_s[kTok];

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int col = blockIdx.z * blockDim.x + threadIdx.x;
    const bool active = col < d.Dv;
    const int a0 = seg * d.L;

    float st[DK];
    if (MODE == kApply && active) {
        const float* src = S_in + sum_off(d, seg, b, h);
#pragma unroll
        for (int i = 0; i < DK; ++i) st[i] = src[int64_t(i) * d.Dv + col];
    } else {
#pragma unroll
        for (int i = 0; i < DK; ++i) st[i] = 0.f;
    }
    float P = 1.f;        // GAMMA: running product of alphas since the segment start
    float gsum = 0.f;     // PREPARE: sum of gates
    bool reset = false;   // PREPARE: a sequence starts inside the segment

    for (int t0 = a0; t0 < a0 + d.L; t0 += kTok) {
        __syncthreads();
        for (int e = threadIdx.x; e < kTok * DK; e += blockDim.x) {
            const int tt = e / DK, i = e % DK;
            const int64_t off = qk_off(d, b, t0 + tt, h) + i;
            const int64_t qo = q_off(d, b, t0 + tt, h) + i;
            vec_s[tt][i] = to_f32(MODE == kGamma ? q[qo] : k[off]);
            if (MODE == kApply) q_s[tt][i] = to_f32(q[qo]);
        }
        if (threadIdx.x < kTok) {
            const int t = t0 + threadIdx.x;
            const float gv = g[g_off(d, b, t, h)];
            const bool s = starts_sequence(d.seq_idx, t);
            g_s[threadIdx.x] = gv;
            start_s[threadIdx.x] = s;
            alpha_s[threadIdx.x] = s ? 0.f : expf(gv);
        }
        float vr[kTok];
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt)
            vr[tt] = active ? to_f32((MODE == kGamma ? dO : v)[v_off(d, b, t0 + tt, h) + col]) : 0.f;
        __syncthreads();

#pragma unroll 1
        for (int tt = 0; tt < kTok; ++tt) {
            const float alpha = alpha_s[tt];
            if (MODE == kGamma) {
                P = (t0 + tt == a0) ? alpha : P * alpha;
                const float w = P * d.scale * vr[tt];
#pragma unroll
                for (int i = 0; i < DK; ++i) st[i] = fmaf(w, vec_s[tt][i], st[i]);
            } else {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < DK; ++i) {
                    st[i] = fmaf(alpha, st[i], vec_s[tt][i] * vr[tt]);
                    if (MODE == kApply) acc = fmaf(st[i], q_s[tt][i], acc);
                }
                if (MODE == kApply && active)
                    o[v_off(d, b, t0 + tt, h) + col] = from_f32<T>(d.scale * acc);
                if (MODE == kPrepare) {
                    gsum += g_s[tt];
                    reset = reset || start_s[tt];
                }
            }
        }
    }

    if (MODE != kApply) {
        if (active) {
            float* dst = sum_out + sum_off(d, seg, b, h);
#pragma unroll
            for (int i = 0; i < DK; ++i) dst[int64_t(i) * d.Dv + col] = st[i];
        }
        if (MODE == kPrepare && blockIdx.z == 0 && threadIdx.x == 0)
            M[(int64_t(seg) * d.B + b) * d.H + h] = reset ? 0.f : expf(gsum);
    }
}

// ---------------------------------------------------------------------------
// dq sweep, row owner: dq_t = scale S_t dO_t, S carried from S_in; also
// qdq_t = q_t . dq_t (fp32 per token) into the workspace.
// grid (nseg, B*H); block = DK threads (rounded up to 32); dynamic smem holds
// S with an odd row pitch (conflict-free row and column walks) and the v/dO tiles.
// ---------------------------------------------------------------------------
template <int DK, typename T>
__global__ void __launch_bounds__(128) simt_dq_sweep(Dims d, const T* __restrict__ q,
                                                     const T* __restrict__ k,
                                                     const T* __restrict__ v,
                                                     const float* __restrict__ g,
                                                     const T* __restrict__ dO,
                                                     const float* __restrict__ S_in,
                                                     T* __restrict__ dq, float* __restrict__ qdq) {
    extern __shared__ float smem[];
    const int pitch = d.Dv + 1;
    float* S = smem;                         // [DK][pitch]
    float* v_s = S + DK * pitch;             // [kTok][Dv]
    float* do_s = v_s + kTok * d.Dv;         // [kTok][Dv]
    __shared__ float alpha_s[kTok];
    __shared__ float vdo_s[kTok];
    __shared__ float part_s[kTok][DK / 32 > 0 ? DK / 32 : 1];

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int i = threadIdx.x;  // row
    const int a0 = seg * d.L;
    const int nwarp = (DK + 31) / 32;

    const float* src = S_in + sum_off(d, seg, b, h);
    for (int e = threadIdx.x; e < DK * d.Dv; e += blockDim.x)
        S[(e / d.Dv) * pitch + e % d.Dv] = src[e];

    for (int t0 = a0; t0 < a0 + d.L; t0 += kTok) {
        __syncthreads();
        for (int e = threadIdx.x; e < kTok * d.Dv; e += blockDim.x) {
            const int tt = e / d.Dv, j = e % d.Dv;
            const int64_t off = v_off(d, b, t0 + tt, h) + j;
            v_s[e] = to_f32(v[off]);
            do_s[e] = to_f32(dO[off]);
        }
        if (threadIdx.x < kTok) {
            const int t = t0 + threadIdx.x;
            alpha_s[threadIdx.x] = starts_sequence(d.seq_idx, t) ? 0.f : expf(g[g_off(d, b, t, h)]);
        }
        __syncthreads();
        // v_t . dO_t per token: one warp per token
        for (int tt = threadIdx.x >> 5; tt < kTok; tt += blockDim.x >> 5) {
            float x = 0.f;
            for (int j = threadIdx.x & 31; j < d.Dv; j += 32) x = fmaf(v_s[tt * d.Dv + j], do_s[tt * d.Dv + j], x);
            x = warp_sum(x);
            if ((threadIdx.x & 31) == 0) vdo_s[tt] = x;
        }
        float kr[kTok], qr[kTok];
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt) {
            kr[tt] = i < DK ? to_f32(k[qk_off(d, b, t0 + tt, h) + i]) : 0.f;
            qr[tt] = i < DK ? to_f32(q[q_off(d, b, t0 + tt, h) + i]) : 0.f;
        }
        __syncthreads();
#pragma unroll 1
        for (int tt = 0; tt < kTok; ++tt) {
            const float alpha = alpha_s[tt];
            float acc = 0.f;
            if (i < DK) {
                // dq_t = scale (alpha_t S_{t-1} dO_t + k_t (v_t . dO_t)); the gate
                // gradient takes only the first part (q_t . dq_t minus its
                // same-token term, which cancels against k_t . dk_t exactly)
                float* row = S + i * pitch;
                const float* vv = v_s + tt * d.Dv;
                const float* dd = do_s + tt * d.Dv;
                float old_acc = 0.f;
                for (int j = 0; j < d.Dv; ++j) {
                    const float s_old = row[j];
                    row[j] = fmaf(alpha, s_old, kr[tt] * vv[j]);
                    old_acc = fmaf(s_old, dd[j], old_acc);
                }
                const float hist = d.scale * alpha * old_acc;
                const float dqi = fmaf(d.scale * kr[tt], vdo_s[tt], hist);
                dq[qk_off(d, b, t0 + tt, h) + i] = from_f32<T>(dqi);
                acc = qr[tt] * hist;
            }
            acc = warp_sum(acc);
            if ((threadIdx.x & 31) == 0) part_s[tt][threadIdx.x >> 5] = acc;
        }
        __syncthreads();
        if (threadIdx.x < kTok) {
            float s = 0.f;
            for (int w = 0; w < nwarp; ++w) s += part_s[threadIdx.x][w];
            qdq[g_off(d, b, t0 + threadIdx.x, h)] = s;
        }
    }
}

// ---------------------------------------------------------------------------
// Reverse sweep of cp_backward_apply: D carried from dS_out at the segment's
// last token; dk (row owners), dv (column owners), dg (reverse running sum).
// grid (nseg, B*H); block = max(DK, Dv) rounded up to 32 (<= 256).
// ---------------------------------------------------------------------------
template <int DK, typename T>
__global__ void __launch_bounds__(256) simt_reverse_sweep(Dims d, const T* __restrict__ q,
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
    float* D = smem;                        // [DK][pitch]
    float* v_s = D + DK * pitch;            // [kTok][Dv]
    float* do_s = v_s + kTok * d.Dv;        // [kTok][Dv]
    float* q_s = do_s + kTok * d.Dv;        // [kTok][DK]
    float* k_s = q_s + kTok * DK;           // [kTok][DK]
    __shared__ float beta_s[kTok];
    __shared__ float vdo_s[kTok];
    __shared__ int start_s[kTok];
    __shared__ float part_s[kTok][DK / 32 > 0 ? DK / 32 : 1];
    __shared__ float red_s[8];
    __shared__ float run_s;

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int a0 = seg * d.L, e0 = a0 + d.L;
    const int nwarp_rows = (DK + 31) / 32;

    // D <- dS_out[seg]; ext = <S_out, dS_out> with S_out read as S_in[seg+1]
    const float* dso = dS_out + sum_off(d, seg, b, h);
    const float* sout = seg + 1 < d.nseg ? S_in + sum_off(d, seg + 1, b, h) : nullptr;
    float ext = 0.f;
    for (int e = threadIdx.x; e < DK * d.Dv; e += blockDim.x) {
        const float x = dso[e];
        D[(e / d.Dv) * pitch + e % d.Dv] = x;
        if (sout) ext = fmaf(sout[e], x, ext);
    }
    ext = warp_sum(ext);
    if ((threadIdx.x & 31) == 0) red_s[threadIdx.x >> 5] = ext;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red_s[w];
        run_s = s;
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
            const int tt = e / DK, i = e % DK;
            const int64_t off = qk_off(d, b, t0 + tt, h) + i;
            q_s[e] = to_f32(q[q_off(d, b, t0 + tt, h) + i]);
            k_s[e] = to_f32(k[off]);
        }
        if (threadIdx.x < kTok) {
            const int t = t0 + threadIdx.x;
            // beta_t multiplies D_{t+1}: alpha_{t+1} inside the segment, 1 at its
            // last token (D starts as dS_out there).
            beta_s[threadIdx.x] = (t + 1 < e0)
                ? (starts_sequence(d.seq_idx, t + 1) ? 0.f : expf(g[g_off(d, b, t + 1, h)]))
                : 1.f;
            start_s[threadIdx.x] = starts_sequence(d.seq_idx, t);
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
            const float beta = beta_s[tt];
            // phase 1: row owners update D and form dk
            float kdk = 0.f;
            if (threadIdx.x < DK) {
                const int i = threadIdx.x;
                // dk_t = beta D_{t+1} v_t + scale q_t (dO_t . v_t); the gate
                // gradient takes only the first part (see the dq sweep)
                float* row = D + i * pitch;
                const float qi = d.scale * q_s[tt * DK + i];
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
                kdk = k_s[tt * DK + i] * fut;
            }
            if (threadIdx.x < nwarp_rows * 32) {
                kdk = warp_sum(kdk);
                if ((threadIdx.x & 31) == 0) part_s[tt][threadIdx.x >> 5] = kdk;
            }
            __syncthreads();
            // phase 2: column owners form dv
            if (threadIdx.x < d.Dv) {
                const int j = threadIdx.x;
                float acc = 0.f;
                for (int i = 0; i < DK; ++i) acc = fmaf(D[i * pitch + j], k_s[tt * DK + i], acc);
                dv[v_off(d, b, t, h) + j] = from_f32<T>(acc);
            }
            __syncthreads();
        }
        // gate gradient of the tile, newest token first
        if (threadIdx.x == 0) {
            float run = run_s;
            for (int tt = kTok - 1; tt >= 0; --tt) {
                const int t = t0 + tt;
                float kdk = 0.f;
                for (int w = 0; w < nwarp_rows; ++w) kdk += part_s[tt][w];
                run += qdq[g_off(d, b, t, h)] - kdk;
                dg[g_off(d, b, t, h)] = start_s[tt] ? 0.f : run;
                if (start_s[tt]) run = 0.f;  // earlier tokens belong to another sequence
            }
            run_s = run;
        }
    }
}

template <typename T>
rm_status launch_generic_T(Op op, const Dims& d, const Ptrs& p, cudaStream_t s) {
    const int BH = d.B * d.H;
    const int colthreads = d.Dv >= 128 ? 128 : ((d.Dv + 31) / 32) * 32;
    const dim3 cgrid(d.nseg, BH, (d.Dv + colthreads - 1) / colthreads);
    const T* q = static_cast<const T*>(p.q);
    const T* k = static_cast<const T*>(p.k);
    const T* v = static_cast<const T*>(p.v);
    const T* dO = static_cast<const T*>(p.dO);

#define RMCP_DK_SWITCH(...)                                 \
    switch (d.Dk) {                                         \
        case 16: { constexpr int DK = 16; __VA_ARGS__; break; }   \
        case 32: { constexpr int DK = 32; __VA_ARGS__; break; }   \
        case 64: { constexpr int DK = 64; __VA_ARGS__; break; }   \
        case 128: { constexpr int DK = 128; __VA_ARGS__; break; } \
        default: return RM_ERR_UNSUPPORTED;                 \
    }

    switch (op) {
        case Op::kForwardPrepare:
            RMCP_DK_SWITCH((simt_column_sweep<DK, kPrepare, T><<<cgrid, colthreads, 0, s>>>(
                d, nullptr, k, v, p.g, nullptr, nullptr, nullptr, p.M, p.sum_out)));
            break;
        case Op::kForwardApply:
            RMCP_DK_SWITCH((simt_column_sweep<DK, kApply, T><<<cgrid, colthreads, 0, s>>>(
                d, q, k, v, p.g, nullptr, p.S_in, static_cast<T*>(p.out0), nullptr, nullptr)));
            break;
        case Op::kBackwardPrepare: {
            RMCP_DK_SWITCH((simt_column_sweep<DK, kGamma, T><<<cgrid, colthreads, 0, s>>>(
                d, q, nullptr, nullptr, p.g, dO, nullptr, nullptr, nullptr, p.sum_out)));
            if (!rmcp::launch_ok()) return RM_ERR_CUDA;
            const int threads = d.Dk < 32 ? 32 : d.Dk;
            const size_t smem = sizeof(float) * (size_t(d.Dk) * (d.Dv + 1) + 2 * kTok * d.Dv);
            RMCP_DK_SWITCH({
                auto fn = simt_dq_sweep<DK, T>;
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
            const size_t smem = sizeof(float) * (size_t(d.Dk) * (d.Dv + 1) + 2 * kTok * d.Dv +
                                                 2 * kTok * d.Dk);
            RMCP_DK_SWITCH({
                auto fn = simt_reverse_sweep<DK, T>;
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
#undef RMCP_DK_SWITCH
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(op == Op::kBackwardPrepare ? 2 : 1);
    return RM_OK;
}

}  // namespace

// The generic path needs L to be a multiple of the staging tile.
bool generic_supports(const Dims& d) {
    return (d.Dk == 16 || d.Dk == 32 || d.Dk == 64 || d.Dk == 128) && d.Dv % 8 == 0 &&
           d.Dv >= 8 && d.Dv <= 256 && d.L % kTok == 0;
}

rm_status launch_generic(Op op, const Dims& d, rm_dtype dt, const Ptrs& p, cudaStream_t s) {
    return dt == RM_F32 ? launch_generic_T<float>(op, d, p, s)
                        : launch_generic_T<__nv_bfloat16>(op, d, p, s);
}

}  // namespace rmcp
