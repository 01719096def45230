// ssd_map.cu -- the Mamba2 SSD scan on the gated-linear-attention path: the
// elementwise maps of its arguments onto q, k, g (q = C, k = dt B, g = dt A,
// v = x, scale 1), the output y = o + D x, and the maps of the path's
// gradients back onto the SSD arguments with per-head sums in a fixed order.
//
// Every kernel moves 16-byte vectors (8 bf16 or 4 fp32 values).  Rows of N
// (or P) values are split over N / VEC consecutive lanes of one warp, so a
// row's dot products reduce with warp shuffles.
#include <cstdio>

#include "internal.h"

namespace rmcp {
namespace {

constexpr int kThreads = 256;
constexpr int kRedBlocks = 1024;  // blocks of the per-head reduction

template <typename T>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int n = 4;
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int n = 8;
};

__device__ __forceinline__ void load16(const float* p, float* x) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
}
__device__ __forceinline__ void store16(float* p, const float* x) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float* x) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void store16(__nv_bfloat16* p, const float* x) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// sum over the `width` consecutive lanes that share a row (width divides 32)
__device__ __forceinline__ float row_sum(float v, int width) {
    for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// k (and q) of every head and g; block = one (row, token), its threads take
// the H * NC (head, 16-byte chunk) items, NC = N / VEC a power of two
template <typename T>
__global__ void __launch_bounds__(kThreads) ssd_map_inputs_kernel(
    int H, int G, int N, int lnc, const float* __restrict__ dt, const float* __restrict__ A,
    const T* __restrict__ Bm, const T* __restrict__ Cm, T* __restrict__ q, T* __restrict__ k,
    float* __restrict__ g) {
    constexpr int VE = Vec<T>::n;
    const int64_t bt = blockIdx.x;
    const int hpg = H / G, nc = 1 << lnc;
    for (int j = threadIdx.x; j < (H << lnc); j += kThreads) {
        const int h = j >> lnc, c = j & (nc - 1), gi = h / hpg;
        const float d = __ldg(dt + bt * H + h);
        const int64_t src = (bt * G + gi) * N + c * VE;
        float bv[VE];
        load16(Bm + src, bv);
#pragma unroll
        for (int e = 0; e < VE; ++e) bv[e] *= d;
        const int64_t row = (bt * H + h) * N + c * VE;
        if (q != nullptr) {
            float cv[VE];
            load16(Cm + src, cv);
            store16(q + row, cv);
        }
        store16(k + row, bv);
        if (c == 0) g[bt * H + h] = d * __ldg(A + h);
    }
}

// y = o + D_h x over [B,T,H,P], in place; block = one (row, token)
template <typename T>
__global__ void __launch_bounds__(kThreads) ssd_finish_forward_kernel(
    int H, int lpc, const T* __restrict__ x, const float* __restrict__ D, T* o) {
    constexpr int VE = Vec<T>::n;
    const int64_t base = int64_t(blockIdx.x) * (int64_t(H) << lpc);
    for (int j = threadIdx.x; j < (H << lpc); j += kThreads) {
        const float dh = __ldg(D + (j >> lpc));
        const int64_t i = base + j;
        float xv[VE], ov[VE];
        load16(x + i * VE, xv);
        load16(o + i * VE, ov);
#pragma unroll
        for (int e = 0; e < VE; ++e) ov[e] = fmaf(dh, xv[e], ov[e]);
        store16(o + i * VE, ov);
    }
}

// dC, dB of a (row, token, group) and ddt of its heads; item = (bt * G + gi) * NC + c.
// Every lane runs the head loop (the shuffles need the whole warp); lanes past
// the end work on zeros and store nothing.
template <typename T>
__global__ void __launch_bounds__(kThreads) ssd_grad_bc_kernel(
    int64_t items, int H, int G, int N, const float* __restrict__ dt, const float* __restrict__ A,
    const T* __restrict__ Bm, const T* __restrict__ dq, const T* __restrict__ dk,
    const float* __restrict__ dg, float* __restrict__ ddt, T* __restrict__ dB, T* __restrict__ dC) {
    constexpr int VE = Vec<T>::n;
    const int i = blockIdx.x * kThreads + threadIdx.x;  // items < 2^31 (checked on the host)
    const bool live = i < items;
    const int NC = N / VE, hpg = H / G;
    const int c = i & (NC - 1);
    const int btg32 = live ? i / NC : 0;
    const int gi = btg32 % G;
    const int64_t btg = btg32, bt = btg32 / G;
    float bv[VE], sb[VE], sc[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) {
        bv[e] = 0.f;
        sb[e] = 0.f;
        sc[e] = 0.f;
    }
    if (live) load16(Bm + btg * N + c * VE, bv);
#pragma unroll 4
    for (int hh = 0; hh < hpg; ++hh) {
        const int h = gi * hpg + hh;
        float qv[VE], kv[VE];
        float d = 0.f;
        if (live) {
            const int64_t row = (bt * H + h) * N + c * VE;
            load16(dq + row, qv);
            load16(dk + row, kv);
            d = __ldg(dt + bt * H + h);
        } else {
#pragma unroll
            for (int e = 0; e < VE; ++e) qv[e] = kv[e] = 0.f;
        }
        float pd = 0.f;
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            sc[e] += qv[e];
            sb[e] = fmaf(d, kv[e], sb[e]);
            pd = fmaf(bv[e], kv[e], pd);
        }
        pd = row_sum(pd, NC);
        if (live && c == 0) ddt[bt * H + h] = fmaf(__ldg(A + h), __ldg(dg + bt * H + h), pd);
    }
    if (live) {
        store16(dB + btg * N + c * VE, sb);
        store16(dC + btg * N + c * VE, sc);
    }
}

// dx = dv + D_h dy in place over dv (D may be null), and part[row] = x . dy
// per (row, token, head); block = one (row, token), its threads take the
// H * PC items (PC = P / VEC lanes per head row, a power of two up to 32).
// The loop runs the same number of times in every lane of a warp (the row
// sums shuffle across lanes); lanes past the end work on zeros.
template <typename T>
__global__ void __launch_bounds__(kThreads) ssd_grad_x_kernel(
    int H, int lpc, const T* __restrict__ x, const T* __restrict__ dy, const float* __restrict__ D,
    T* dv, float* __restrict__ part) {
    constexpr int VE = Vec<T>::n;
    const int n = H << lpc, pc = 1 << lpc;
    const int64_t base = int64_t(blockIdx.x) * n;
    for (int j0 = 0; j0 < n; j0 += kThreads) {
        const int j = j0 + threadIdx.x;
        const bool live = j < n;
        float s = 0.f;
        if (live) {
            const int64_t i = base + j;
            float xv[VE], yv[VE], vv[VE];
            load16(x + i * VE, xv);
            load16(dy + i * VE, yv);
            load16(dv + i * VE, vv);
            const float dh = D != nullptr ? __ldg(D + (j >> lpc)) : 0.f;
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                vv[e] = fmaf(dh, yv[e], vv[e]);
                s = fmaf(xv[e], yv[e], s);
            }
            store16(dv + i * VE, vv);
        }
        s = row_sum(s, pc);
        if (live && (j & (pc - 1)) == 0) part[(base >> lpc) + (j >> lpc)] = s;
    }
}

// per-head partial sums of dt dg and of part over the flattened [B*T, H]
// arrays: block r takes rows r, r + kRedBlocks, ...; thread tid < S (S the
// largest multiple of H not above kThreads) always sees head tid % H.
__global__ void __launch_bounds__(kThreads) ssd_reduce_heads_kernel(
    int64_t rows, int H, const float* __restrict__ dt, const float* __restrict__ dg,
    const float* __restrict__ part, float* __restrict__ pa, float* __restrict__ pd) {
    __shared__ float sa[kThreads], sd[kThreads];
    const int S = (kThreads / H) * H;
    const int tid = threadIdx.x;
    float a = 0.f, dd = 0.f;
    if (tid < S) {
        const int rpb = S / H;  // rows per step of one block
        for (int64_t r0 = int64_t(blockIdx.x) * rpb; r0 < rows; r0 += int64_t(kRedBlocks) * rpb) {
            const int64_t r = r0 + tid / H;
            if (r < rows) {
                const int64_t e = r * H + tid % H;
                a = fmaf(__ldg(dt + e), __ldg(dg + e), a);
                dd += __ldg(part + e);
            }
        }
    }
    sa[tid] = a;
    sd[tid] = dd;
    __syncthreads();
    if (tid < H) {
        float ta = 0.f, td = 0.f;
        for (int j = tid; j < S; j += H) {
            ta += sa[j];
            td += sd[j];
        }
        pa[blockIdx.x * H + tid] = ta;
        pd[blockIdx.x * H + tid] = td;
    }
}

// dA, dD from the block partials: block h sums head h; thread t adds partials
// t, t + 256, ... (independent loads), then warps and the block finish the
// sum in a fixed order
__global__ void __launch_bounds__(kThreads) ssd_reduce_final_kernel(
    int H, const float* __restrict__ pa, const float* __restrict__ pd, float* __restrict__ dA,
    float* __restrict__ dD) {
    __shared__ float wa[kThreads / 32], wd[kThreads / 32];
    const int h = blockIdx.x, tid = threadIdx.x;
    float a = 0.f, d = 0.f;
#pragma unroll
    for (int r = tid; r < kRedBlocks; r += kThreads) {
        a += __ldg(pa + r * H + h);
        d += __ldg(pd + r * H + h);
    }
    a = row_sum(a, 32);
    d = row_sum(d, 32);
    if ((tid & 31) == 0) {
        wa[tid >> 5] = a;
        wd[tid >> 5] = d;
    }
    __syncthreads();
    if (tid == 0) {
        float sa = 0.f, sd = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) {
            sa += wa[w];
            sd += wd[w];
        }
        dA[h] = sa;
        dD[h] = sd;
    }
}

int blocks_for(int64_t items) { return int((items + kThreads - 1) / kThreads); }
int log2i(int n) {
    int l = 0;
    while ((1 << l) < n) ++l;
    return l;
}

#define RM_NEED_SSD(ptr)                                     \
    do {                                                     \
        rm_status s_ = api_need((ptr), #ptr);                \
        if (s_ != RM_OK) return s_;                          \
    } while (0)

rm_status check_ssd(const rm_cp_problem* p, int G, Dims* d) {
    rm_status s = api_check_problem(p, d);
    if (s != RM_OK) return s;
    if (p->scale != 1.0f) return api_fail(RM_ERR_INVALID_ARG, "the SSD scan needs scale = 1");
    if (d->vg) return api_fail(RM_ERR_INVALID_ARG, "the SSD scan has one gate per head (vector_gates = 0)");
    if (G < 1 || d->H % G != 0) return api_fail(RM_ERR_INVALID_ARG, "G must divide H");
    if (d->H > kThreads) return api_fail(RM_ERR_UNSUPPORTED, "the SSD reductions take H <= 256");
    // rows of N and P values split into 16-byte vectors over 1..32 lanes of a warp
    const int ve = p->dtype == RM_BF16 ? 8 : 4;
    auto lanes_ok = [ve](int n) {
        const int w = n / ve;
        return n % ve == 0 && w >= 1 && w <= 32 && (w & (w - 1)) == 0;
    };
    if (!lanes_ok(d->Dk) || !lanes_ok(d->Dv))
        return api_fail(RM_ERR_UNSUPPORTED,
                        "the SSD maps take N and P with N/v and P/v a power of two up to 32 "
                        "(v = 8 for bf16, 4 for fp32)");
    // one block per (row, token); flat (row, token, group, lane) indices in int32
    const double tokens = double(d->B) * d->T;
    if (tokens > 2.0e9 || tokens * G * (d->Dk / ve) > 2.0e9)
        return api_fail(RM_ERR_SHAPE, "B*T too large for the SSD maps");
    return RM_OK;
}

size_t ssd_ws_bytes(const Dims& d) {
    return sizeof(float) * (size_t(d.B) * d.T * d.H + 2 * size_t(kRedBlocks) * d.H);
}

}  // namespace
}  // namespace rmcp

using rmcp::api_fail;
using rmcp::api_need;

extern "C" size_t rm_ssd_workspace_size(const rm_cp_problem* p) {
    rmcp::Dims d;
    if (rmcp::api_check_problem(p, &d) != RM_OK) return 0;
    return rmcp::ssd_ws_bytes(d);
}

extern "C" rm_status rm_ssd_map_inputs(const rm_cp_problem* p, int32_t G, const float* dt,
                                       const float* A, const void* Bm, const void* Cm, void* q,
                                       void* k, float* g, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = rmcp::check_ssd(p, G, &d);
    if (s != RM_OK) return s;
    RM_NEED_SSD(dt);
    RM_NEED_SSD(A);
    RM_NEED_SSD(Bm);
    if (q != nullptr) {
        RM_NEED_SSD(Cm);
        RM_NEED_SSD(q);
    }
    RM_NEED_SSD(k);
    RM_NEED_SSD(g);
    auto st = reinterpret_cast<cudaStream_t>(stream);
    rmcp::begin_launches();
    const int64_t bt = int64_t(d.B) * d.T;
    if (p->dtype == RM_BF16) {
        rmcp::ssd_map_inputs_kernel<__nv_bfloat16><<<unsigned(bt), rmcp::kThreads, 0, st>>>(
            d.H, G, d.Dk, rmcp::log2i(d.Dk / 8), dt, A, static_cast<const __nv_bfloat16*>(Bm),
            static_cast<const __nv_bfloat16*>(Cm), static_cast<__nv_bfloat16*>(q),
            static_cast<__nv_bfloat16*>(k), g);
    } else {
        rmcp::ssd_map_inputs_kernel<float><<<unsigned(bt), rmcp::kThreads, 0, st>>>(
            d.H, G, d.Dk, rmcp::log2i(d.Dk / 4), dt, A, static_cast<const float*>(Bm), static_cast<const float*>(Cm),
            static_cast<float*>(q), static_cast<float*>(k), g);
    }
    if (!rmcp::launch_ok()) {
        char msg[192];
        std::snprintf(msg, sizeof(msg), "rm_ssd_map_inputs: launch failed: %s", rmcp::cuda_error_text());
        return api_fail(RM_ERR_CUDA, msg);
    }
    rmcp::note_launch(1);
    return RM_OK;
}

extern "C" rm_status rm_ssd_finish_forward(const rm_cp_problem* p, const void* x, const float* D,
                                           void* o, rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = rmcp::check_ssd(p, 1, &d);
    if (s != RM_OK) return s;
    RM_NEED_SSD(x);
    RM_NEED_SSD(o);
    if (D == nullptr) return RM_OK;
    RM_NEED_SSD(D);
    auto st = reinterpret_cast<cudaStream_t>(stream);
    rmcp::begin_launches();
    const unsigned bt = unsigned(int64_t(d.B) * d.T);
    if (p->dtype == RM_BF16) {
        rmcp::ssd_finish_forward_kernel<__nv_bfloat16><<<bt, rmcp::kThreads, 0, st>>>(
            d.H, rmcp::log2i(d.Dv / 8), static_cast<const __nv_bfloat16*>(x), D, static_cast<__nv_bfloat16*>(o));
    } else {
        rmcp::ssd_finish_forward_kernel<float><<<bt, rmcp::kThreads, 0, st>>>(
            d.H, rmcp::log2i(d.Dv / 4), static_cast<const float*>(x), D, static_cast<float*>(o));
    }
    if (!rmcp::launch_ok()) {
        char msg[192];
        std::snprintf(msg, sizeof(msg), "rm_ssd_finish_forward: launch failed: %s", rmcp::cuda_error_text());
        return api_fail(RM_ERR_CUDA, msg);
    }
    rmcp::note_launch(1);
    return RM_OK;
}

extern "C" rm_status rm_ssd_finish_backward(const rm_cp_problem* p, int32_t G, const void* x,
                                            const float* dt, const float* A, const void* Bm,
                                            const void* dy, const float* D, const void* dq,
                                            const void* dk, void* dv, const float* dg, float* ddt,
                                            float* dA, void* dB, void* dC, float* dD, void* ws,
                                            rm_stream_t stream) {
    rmcp::Dims d;
    rm_status s = rmcp::check_ssd(p, G, &d);
    if (s != RM_OK) return s;
    RM_NEED_SSD(x);
    RM_NEED_SSD(dt);
    RM_NEED_SSD(A);
    RM_NEED_SSD(Bm);
    RM_NEED_SSD(dy);
    RM_NEED_SSD(dq);
    RM_NEED_SSD(dk);
    RM_NEED_SSD(dv);
    RM_NEED_SSD(dg);
    RM_NEED_SSD(ddt);
    RM_NEED_SSD(dA);
    RM_NEED_SSD(dB);
    RM_NEED_SSD(dC);
    RM_NEED_SSD(dD);
    RM_NEED_SSD(ws);
    if (D != nullptr) RM_NEED_SSD(D);
    auto st = reinterpret_cast<cudaStream_t>(stream);
    rmcp::begin_launches();
    const int64_t bt = int64_t(d.B) * d.T, rows = bt * d.H;
    float* part = static_cast<float*>(ws);
    float* pa = part + rows;
    float* pd = pa + size_t(rmcp::kRedBlocks) * d.H;
    int launches = 0;
    if (p->dtype == RM_BF16) {
        using T = __nv_bfloat16;
        const int64_t nbc = bt * G * (d.Dk / 8);
        rmcp::ssd_grad_bc_kernel<T><<<rmcp::blocks_for(nbc), rmcp::kThreads, 0, st>>>(
            nbc, d.H, G, d.Dk, dt, A, static_cast<const T*>(Bm), static_cast<const T*>(dq),
            static_cast<const T*>(dk), dg, ddt, static_cast<T*>(dB), static_cast<T*>(dC));
        ++launches;
        rmcp::ssd_grad_x_kernel<T><<<unsigned(bt), rmcp::kThreads, 0, st>>>(
            d.H, rmcp::log2i(d.Dv / 8), static_cast<const T*>(x), static_cast<const T*>(dy), D,
            static_cast<T*>(dv), part);
        ++launches;
    } else {
        using T = float;
        const int64_t nbc = bt * G * (d.Dk / 4);
        rmcp::ssd_grad_bc_kernel<T><<<rmcp::blocks_for(nbc), rmcp::kThreads, 0, st>>>(
            nbc, d.H, G, d.Dk, dt, A, static_cast<const T*>(Bm), static_cast<const T*>(dq),
            static_cast<const T*>(dk), dg, ddt, static_cast<T*>(dB), static_cast<T*>(dC));
        ++launches;
        rmcp::ssd_grad_x_kernel<T><<<unsigned(bt), rmcp::kThreads, 0, st>>>(
            d.H, rmcp::log2i(d.Dv / 4), static_cast<const T*>(x), static_cast<const T*>(dy), D,
            static_cast<T*>(dv), part);
        ++launches;
    }
    rmcp::ssd_reduce_heads_kernel<<<rmcp::kRedBlocks, rmcp::kThreads, 0, st>>>(
        bt, d.H, dt, dg, part, pa, pd);
    rmcp::ssd_reduce_final_kernel<<<d.H, rmcp::kThreads, 0, st>>>(d.H, pa, pd, dA, dD);
    launches += 2;
    if (!rmcp::launch_ok()) {
        char msg[192];
        std::snprintf(msg, sizeof(msg), "rm_ssd_finish_backward: launch failed: %s", rmcp::cuda_error_text());
        return api_fail(RM_ERR_CUDA, msg);
    }
    rmcp::note_launch(launches);
    return RM_OK;
}
