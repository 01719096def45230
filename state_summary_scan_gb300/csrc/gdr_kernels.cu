// gdr_kernels.cu -- the gated delta rule on the segment-summary path.
//
// Per row b and head h, with a scalar gate g_t and write strength beta_t
// ([B,T,H] fp32 each), alpha_t = exp(g_t) (0 when token t starts a sequence)
// and A_t = alpha_t (I - beta_t k_t k_t^T):
//     S_t = A_t S_{t-1} + beta_t k_t v_t^T,      o_t = scale S_t^T q_t.
// A segment's summary is then the general affine map of the Megatron-Core
// page "core.ssm.context_parallel.chunkwise": S_out = M S_in + delta_S
// (CPForwardUnpackedSummary) with the Dk x Dk transition M = A_last ... A_first
// (0 when a token of the segment starts a sequence), and the backward's
// dS_in = M^T dS_out + gamma (CPBackwardUnpackedSummary); A_t is symmetric.
//
// Kernels (fp32 arithmetic, both storage types; one CTA per (segment, row,
// head) unless noted):
//   gdr_column_sweep  forward walks by column owners (thread = one column of
//                     the state in registers: k^T S, the rank-one correction
//                     and the readout are all column-local).  PREPARE also
//                     walks M's columns as extra columns with v = 0 from the
//                     identity; APPLY starts from S_in and writes o.
//   gdr_gamma_sweep   gamma = A_a D_a of the local adjoint walked back from
//                     the segment end with a zero outgoing gradient (column
//                     owners of D, column-local for the same reason).
//   gdr_compose       the prefix fold S <- M_i S + dS_i over [pre_j, j), or
//                     the suffix fold D <- M_i^T D + gamma_i over (j, fol_j),
//                     one CTA per (row, head, block of 4 columns), the
//                     carried block in shared memory, each lane's part of a
//                     row of M_i in registers (a row per lane up to Dk = 64,
//                     half a row at Dk = 128).
//   gdr_dq_sweep      the state in shared memory from S_in (k^T S by column
//                     partitions, the update over all elements, dq_t = scale
//                     S_t dO_t by row owners); writes the state before every
//                     16-token block to the workspace.  Each block's token
//                     vectors are staged in shared memory by one coalesced load.
//   gdr_reverse_sweep the adjoint D in shared memory from dS_out at the
//                     segment end (D_t = scale q_t dO_t^T + A_{t+1} D_{t+1});
//                     the states S_{t-1} of each group of four tokens are
//                     rebuilt once, into a stack in shared memory, from the
//                     block's saved state; dv, dk, dbeta and dg per token:
//                       dv_t    = beta_t D_t^T k_t
//                       dk_t    = beta_t D_t v_t - alpha_t beta_t (S_{t-1} D_t^T + D_t S_{t-1}^T) k_t
//                       dbeta_t = k_t^T D_t v_t - alpha_t k_t^T D_t S_{t-1}^T k_t
//                       dg_t    = alpha_t <D_t, (I - beta_t k_t k_t^T) S_{t-1}>  (0 at a start)
#include "internal.h"

namespace rmcp {

namespace {

constexpr int kBlk = 16;  // tokens per saved state of the dq sweep (and per rebuild)
constexpr int kSweepThreads = 256;  // threads of the backward sweeps' CTAs

__device__ __forceinline__ float gdr_alpha(const Dims& d, const float* g, int b, int t, int h) {
    return starts_sequence(d.seq_idx, t) ? 0.f : expf(__ldg(g + g_off(d, b, t, h)));
}

// store(e, load(e)) for e in [0, n) over the CTA's threads, with eight loads
// in flight ahead of their stores: a global load and a shared store in the
// same step of a loop would otherwise wait out each load's latency in turn.
template <class Load, class Store>
__device__ __forceinline__ void batched_copy(int n, Load load, Store store) {
    for (int e0 = threadIdx.x; e0 < n; e0 += 8 * blockDim.x) {
        float x[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int e = e0 + m * blockDim.x;
            x[m] = e < n ? load(e) : 0.f;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int e = e0 + m * blockDim.x;
            if (e < n) store(e, x[m]);
        }
    }
}

// ---------------------------------------------------------------------------
// Forward column sweep.  Column c < Dv is column c of the state (value v_c);
// PREPARE adds columns Dv + c' for column c' of M (value 0, start e_c').
// grid (nseg, B*H, ceil(ncol / blockDim)); block 32..128 threads.
// ---------------------------------------------------------------------------
enum GdrMode { kGdrPrepare = 0, kGdrApply = 1 };

template <int DK, int MODE, typename T>
__global__ void __launch_bounds__(128) gdr_column_sweep(Dims d, const T* __restrict__ q,
                                                        const T* __restrict__ k,
                                                        const T* __restrict__ v,
                                                        const float* __restrict__ g,
                                                        const float* __restrict__ beta,
                                                        const float* __restrict__ S_in,
                                                        T* __restrict__ o, float* __restrict__ M,
                                                        float* __restrict__ dS) {
    constexpr int kTok = 16;
    __shared__ float k_s[kTok][DK];
    __shared__ float q_s[kTok][DK];
    __shared__ float a_s[kTok], b_s[kTok];

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int col = blockIdx.z * blockDim.x + threadIdx.x;
    const int ncol = MODE == kGdrPrepare ? d.Dv + DK : d.Dv;
    const bool active = col < ncol;
    const bool is_m = MODE == kGdrPrepare && col >= d.Dv;  // a column of M
    const int a0 = seg * d.L;

    float st[DK];
    if (MODE == kGdrApply && active) {
        const float* src = S_in + sum_off(d, seg, b, h);
#pragma unroll
        for (int i = 0; i < DK; ++i) st[i] = src[int64_t(i) * d.Dv + col];
    } else {
#pragma unroll
        for (int i = 0; i < DK; ++i) st[i] = (is_m && i == col - d.Dv) ? 1.f : 0.f;
    }

    for (int t0 = a0; t0 < a0 + d.L; t0 += kTok) {
        __syncthreads();
        batched_copy(kTok * DK, [&](int e) { return to_f32(k[qk_off(d, b, t0 + e / DK, h) + e % DK]); },
                     [&](int e, float x) { k_s[e / DK][e % DK] = x; });
        if (MODE == kGdrApply)
            batched_copy(kTok * DK, [&](int e) { return to_f32(q[q_off(d, b, t0 + e / DK, h) + e % DK]); },
                         [&](int e, float x) { q_s[e / DK][e % DK] = x; });
        if (threadIdx.x < kTok) {
            const int t = t0 + threadIdx.x;
            a_s[threadIdx.x] = gdr_alpha(d, g, b, t, h);
            b_s[threadIdx.x] = __ldg(beta + g_off(d, b, t, h));
        }
        float vr[kTok];
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt)
            vr[tt] = (active && !is_m) ? to_f32(v[v_off(d, b, t0 + tt, h) + col]) : 0.f;
        __syncthreads();
#pragma unroll 1
        for (int tt = 0; tt < kTok; ++tt) {
            const float al = a_s[tt], be = b_s[tt];
            float ka[4] = {0.f, 0.f, 0.f, 0.f};  // k_t^T S[:, col], four sums
#pragma unroll
            for (int i = 0; i < DK; ++i) ka[i & 3] = fmaf(k_s[tt][i], st[i], ka[i & 3]);
            const float ks = (ka[0] + ka[1]) + (ka[2] + ka[3]);
            // S = alpha (S - beta k (k^T S)) + beta k v^T, column col
            const float c1 = be * ks, c2 = be * vr[tt];
            float oa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < DK; ++i) {
                const float ki = k_s[tt][i];
                st[i] = fmaf(al, fmaf(-c1, ki, st[i]), c2 * ki);
                if (MODE == kGdrApply) oa[i & 3] = fmaf(st[i], q_s[tt][i], oa[i & 3]);
            }
            if (MODE == kGdrApply && active)
                o[v_off(d, b, t0 + tt, h) + col] = from_f32<T>(d.scale * ((oa[0] + oa[1]) + (oa[2] + oa[3])));
        }
    }
    if (MODE == kGdrPrepare && active) {
        if (is_m) {
            float* dst = M + ((int64_t(seg) * d.B + b) * d.H + h) * DK * DK + (col - d.Dv);
#pragma unroll
            for (int i = 0; i < DK; ++i) dst[int64_t(i) * DK] = st[i];
        } else {
            float* dst = dS + sum_off(d, seg, b, h) + col;
#pragma unroll
            for (int i = 0; i < DK; ++i) dst[int64_t(i) * d.Dv] = st[i];
        }
    }
}

// ---------------------------------------------------------------------------
// gamma: column owners of the local adjoint D, walked back from the segment
// end with zero outgoing gradient: per token D += scale q_t dO_t[col] (now
// D_t), then D <- A_t D (the carry into token t - 1); after the segment's
// first token a, D = A_a D_a = gamma[:, col].
// grid (nseg, B*H, ceil(Dv / blockDim)); block 32..128 threads.
// ---------------------------------------------------------------------------
template <int DK, typename T>
__global__ void __launch_bounds__(128) gdr_gamma_sweep(Dims d, const T* __restrict__ q,
                                                       const T* __restrict__ k,
                                                       const float* __restrict__ g,
                                                       const float* __restrict__ beta,
                                                       const T* __restrict__ dO,
                                                       float* __restrict__ gamma) {
    constexpr int kTok = 16;
    __shared__ float k_s[kTok][DK];  // k of the tile's tokens
    __shared__ float q_s[kTok][DK];
    __shared__ float a_s[kTok], b_s[kTok];

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int col = blockIdx.z * blockDim.x + threadIdx.x;
    const bool active = col < d.Dv;
    const int a0 = seg * d.L, e0 = a0 + d.L;

    float D[DK];
#pragma unroll
    for (int i = 0; i < DK; ++i) D[i] = 0.f;

    for (int t0 = e0 - kTok; t0 >= a0; t0 -= kTok) {
        __syncthreads();
        batched_copy(kTok * DK, [&](int e) { return to_f32(k[qk_off(d, b, t0 + e / DK, h) + e % DK]); },
                     [&](int e, float x) { k_s[e / DK][e % DK] = x; });
        batched_copy(kTok * DK, [&](int e) { return to_f32(q[q_off(d, b, t0 + e / DK, h) + e % DK]); },
                     [&](int e, float x) { q_s[e / DK][e % DK] = x; });
        if (threadIdx.x < kTok) {
            const int t = t0 + threadIdx.x;
            a_s[threadIdx.x] = gdr_alpha(d, g, b, t, h);
            b_s[threadIdx.x] = __ldg(beta + g_off(d, b, t, h));
        }
        float dor[kTok];
#pragma unroll
        for (int tt = 0; tt < kTok; ++tt) dor[tt] = active ? to_f32(dO[v_off(d, b, t0 + tt, h) + col]) : 0.f;
        __syncthreads();
#pragma unroll 1
        for (int tt = kTok - 1; tt >= 0; --tt) {
            // D holds A_{t+1} D_{t+1} (0 past the segment end): D_t = scale
            // q_t dO_t + D, then the carry A_t D_t into token t - 1
            const float w = d.scale * dor[tt];
#pragma unroll
            for (int i = 0; i < DK; ++i) D[i] = fmaf(w, q_s[tt][i], D[i]);
            const float al = a_s[tt], be = b_s[tt];
            float ka[4] = {0.f, 0.f, 0.f, 0.f};  // k_t^T D, four sums
#pragma unroll
            for (int i = 0; i < DK; ++i) ka[i & 3] = fmaf(k_s[tt][i], D[i], ka[i & 3]);
            const float c1 = be * ((ka[0] + ka[1]) + (ka[2] + ka[3]));
#pragma unroll
            for (int i = 0; i < DK; ++i) D[i] = al * fmaf(-c1, k_s[tt][i], D[i]);
        }
    }
    // after the segment's first token: D = A_a D_a, i.e. gamma
    if (active) {
        float* dst = gamma + sum_off(d, seg, b, h) + col;
#pragma unroll
        for (int i = 0; i < DK; ++i) dst[int64_t(i) * d.Dv] = D[i];
    }
}

// ---------------------------------------------------------------------------
// Summary folds with matrix transitions: each column of the carried state
// folds on its own (S <- M S + X acts column by column), so one CTA takes
// kFoldCols = 4 columns of one (row, head), fold_parts(DK) consecutive lanes
// per state row r.  Lane part p holds the entries [NT p, NT p + NT) of row r
// of M_i (of column r for the suffix's M_i^T; NT = DK / parts) in registers,
// loaded two segments ahead, and reads those rows of the carried block as
// 16-byte vectors from shared memory, so each loaded entry serves four
// multiply-adds; the parts' sums meet by lane exchanges and part 0 writes row
// r of the result.  Up to DK = 64 a lane takes the whole row; at DK = 128 two
// lanes share it, so that the two segments' entries stay in registers.
//   prefix: S_in[j] = fold over [pre_j, j) of S <- M_i S + dS_i  (from 0)
//   suffix: dS_out[j] = fold over (j, fol_j) of D <- M_i^T D + gamma_i,
//           from the last segment down (from 0)
// grid (B*H, Dv / kFoldCols); block DK * fold_parts(DK).
// ---------------------------------------------------------------------------
constexpr int kFoldCols = 4;
__host__ __device__ constexpr int fold_parts(int dk) { return dk > 64 ? 2 : 1; }

template <int DK, bool SUFFIX>
__global__ void __launch_bounds__(DK * fold_parts(DK)) gdr_compose(Dims d, const float* __restrict__ M,
                                                  const float* __restrict__ X,
                                                  const int32_t* __restrict__ range,
                                                  float* __restrict__ out) {
    constexpr int PARTS = fold_parts(DK);
    constexpr int NT = DK / PARTS;  // entries of a row a lane multiplies
    // the carried block: row c, the CTA's four columns, at c + c / NT (one
    // vector of padding per part, so that the parts read distinct banks)
    __shared__ float4 s_s[2][DK + PARTS];
    const int bh = blockIdx.x;
    const int b = bh / d.H, h = bh % d.H;
    const int r = threadIdx.x / PARTS;        // state row
    const int part = threadIdx.x % PARTS;     // rows [NT part, +NT) of the product
    const int rs = r + r / NT;                // padded slot of row r
    const int c0 = blockIdx.y * kFoldCols;    // first column (Dv is a multiple of 8)
    const int n = d.nseg;
    int buf = 0;  // s_s[buf] holds the carried block
    // two segments in flight: slot i & 1 holds segment i's row of M_i and X_i
    // (the folds walk the segments in order, so i + 2 refills the slot i frees)
    float mpa[NT], mpb[NT];
    float4 xpa = make_float4(0.f, 0.f, 0.f, 0.f), xpb = xpa;  // X_i's row (part 0)
    int pfa = -1, pfb = -1;  // the segment in each slot (the same in every thread)
    auto fetch = [&](int i, float (&mp)[NT], float4& xp) {
        const float* mi = M + ((int64_t(i) * d.B + b) * d.H + h) * DK * DK;
        if (SUFFIX) {
#pragma unroll
            for (int c = 0; c < NT; ++c) mp[c] = __ldg(mi + (NT * part + c) * DK + r);
        } else {
#pragma unroll
            for (int c = 0; c < NT; c += 4) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(mi + r * DK + NT * part + c));
                mp[c] = v.x; mp[c + 1] = v.y; mp[c + 2] = v.z; mp[c + 3] = v.w;
            }
        }
        if (part == 0)
            xp = __ldg(reinterpret_cast<const float4*>(X + sum_off(d, i, b, h) + int64_t(r) * d.Dv + c0));
    };
    auto prefetch = [&](int i) {
        if (i < 0 || i >= n) return;
        if (i & 1) {
            fetch(i, mpb, xpb);
            pfb = i;
        } else {
            fetch(i, mpa, xpa);
            pfa = i;
        }
    };
    auto clear = [&]() {
        if (part == 0) s_s[buf][rs] = make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto step = [&](const float (&m)[NT], float4 a0) {
        float4 a1 = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4* src = &s_s[buf][(NT + 1) * part];
#pragma unroll
        for (int c = 0; c < NT; c += 2) {
            const float4 s0 = src[c], s1 = src[c + 1];
            a0.x = fmaf(m[c], s0.x, a0.x); a0.y = fmaf(m[c], s0.y, a0.y);
            a0.z = fmaf(m[c], s0.z, a0.z); a0.w = fmaf(m[c], s0.w, a0.w);
            a1.x = fmaf(m[c + 1], s1.x, a1.x); a1.y = fmaf(m[c + 1], s1.y, a1.y);
            a1.z = fmaf(m[c + 1], s1.z, a1.z); a1.w = fmaf(m[c + 1], s1.w, a1.w);
        }
        float4 a = make_float4(a0.x + a1.x, a0.y + a1.y, a0.z + a1.z, a0.w + a1.w);
#pragma unroll
        for (int o = 1; o < PARTS; o <<= 1) {  // the parts of row r
            a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
            a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
            a.z += __shfl_xor_sync(0xffffffffu, a.z, o);
            a.w += __shfl_xor_sync(0xffffffffu, a.w, o);
        }
        if (part == 0) s_s[buf ^ 1][rs] = a;
    };
    // s_s[buf ^ 1] = M_i s_s[buf] + X_i (M_i^T for the suffix); buf flips
    auto fold = [&](int i) {
        const bool odd = i & 1;
        if ((odd ? pfb : pfa) != i) prefetch(i);
        __syncthreads();  // the carried block is complete
        if (odd)
            step(mpb, xpb);
        else
            step(mpa, xpa);
        buf ^= 1;
        prefetch(SUFFIX ? i - 2 : i + 2);  // into the slot just read
    };
    // the fold for segment j restarts whenever its range start (end) moves;
    // the next segment's bound is loaded a segment ahead
    int cur = SUFFIX ? n : 0;
    clear();
    prefetch(SUFFIX ? n - 1 : 0);
    prefetch(SUFFIX ? n - 2 : 1);
    int rnext = range ? __ldg(range + (SUFFIX ? n - 1 : 0)) : (SUFFIX ? n : 0);
    for (int u = 0; u < n; ++u) {
        const int j = SUFFIX ? n - 1 - u : u;
        int lim = rnext;
        if (range && u + 1 < n) rnext = __ldg(range + (SUFFIX ? j - 1 : j + 1));
        if (SUFFIX)
            lim = lim < j + 1 ? j + 1 : (lim > n ? n : lim);
        else
            lim = lim < 0 ? 0 : (lim > j ? j : lim);
        if (lim != cur) {  // rebuild the fold over the new range
            __syncthreads();  // every thread has read the old carried block
            clear();
            const int i0 = SUFFIX ? lim - 1 : lim;
            for (int i = i0; SUFFIX ? i > j : i < j; i += SUFFIX ? -1 : 1) fold(i);
            cur = lim;
        }
        // row r of the carried block is part 0's own last write
        if (part == 0) *reinterpret_cast<float4*>(out + sum_off(d, j, b, h) + int64_t(r) * d.Dv + c0) = s_s[buf][rs];
        fold(j);  // extend the fold by segment j for the next segment's range
    }
}

// ---------------------------------------------------------------------------
// One step of the recurrence between states in shared memory (pitch Dv + 1):
// dst = alpha (src - beta k (k^T src)) + beta k v^T; dst may equal src.  The
// column sums k^T src are split over nprt = blockDim / Dv row partitions
// (partial sums in ksp [nprt][Dv]); the update runs over all elements with
// every thread.  Two CTA barriers; all threads of the CTA take part.
// ---------------------------------------------------------------------------
template <int DK>
__device__ __forceinline__ void gdr_step(const float* src, float* dst, int pitch, int Dv, const float* kt,
                                         const float* vt, float al, float be, float* ksp, int nprt) {
    const int tid = threadIdx.x;
    const int j = tid % Dv, part = tid / Dv;
    const bool act = tid < nprt * Dv;
    if (act) {
        // four independent sums (named, so that they stay in registers)
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        int i = part;
        for (; i + 3 * nprt < DK; i += 4 * nprt) {
            a0 = fmaf(kt[i], src[i * pitch + j], a0);
            a1 = fmaf(kt[i + nprt], src[(i + nprt) * pitch + j], a1);
            a2 = fmaf(kt[i + 2 * nprt], src[(i + 2 * nprt) * pitch + j], a2);
            a3 = fmaf(kt[i + 3 * nprt], src[(i + 3 * nprt) * pitch + j], a3);
        }
        for (; i < DK; i += nprt) a0 = fmaf(kt[i], src[i * pitch + j], a0);
        ksp[part * Dv + j] = (a0 + a1) + (a2 + a3);
    }
    __syncthreads();
    if (act) {
        float ks = 0.f;
        for (int pp = 0; pp < nprt; ++pp) ks += ksp[pp * Dv + j];
        const float bv = be * vt[j];
        // rows i = part + nprt m: four loads ahead of four stores
        for (int i0 = part; i0 < DK; i0 += 4 * nprt) {
            float x[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int i = i0 + m * nprt;
                x[m] = i < DK ? src[i * pitch + j] : 0.f;
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int i = i0 + m * nprt;
                if (i < DK) dst[i * pitch + j] = fmaf(al, fmaf(-be * kt[i], ks, x[m]), kt[i] * bv);
            }
        }
    }
    __syncthreads();
}

// X[i][j] = f(i, j, X[i][j]) over a [DK][Dv] state (pitch), every thread on
// column j = tid % Dv and rows part, part + nprt, ... (part = tid / Dv), four
// loads ahead of four stores.  No barrier.
template <int DK, class F>
__device__ __forceinline__ void gdr_map(float* X, int pitch, int Dv, int nprt, F f) {
    const int tid = threadIdx.x;
    if (tid >= nprt * Dv) return;
    const int j = tid % Dv, part = tid / Dv;
    for (int i0 = part; i0 < DK; i0 += 4 * nprt) {
        float x[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int i = i0 + m * nprt;
            x[m] = i < DK ? X[i * pitch + j] : 0.f;
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int i = i0 + m * nprt;
            if (i < DK) X[i * pitch + j] = f(i, j, x[m]);
        }
    }
}

// The kBlk tokens of a block starting at t0: the x rows ([B,T,heads,D], head
// index hx) as fp32 in dst [kBlk][D]; a warp reads consecutive elements.
template <typename T>
__device__ __forceinline__ void stage_rows(const T* __restrict__ x, const Dims& d, int b, int t0, int heads,
                                           int hx, int D, float* dst) {
    batched_copy(kBlk * D,
                 [&](int e) {
                     const int tt = e / D, c = e - tt * D;
                     return to_f32(x[((int64_t(b) * d.T + t0 + tt) * heads + hx) * D + c]);
                 },
                 [&](int e, float v) { dst[e] = v; });
}

// ---------------------------------------------------------------------------
// dq sweep: S from S_in in shared memory; per token the state step, then
// dq_t[i] = scale S_t[i,:] . dO_t by row owners.  Before every kBlk-token
// block the state is saved to ckpt (the block's starting state), and the
// block's k, v, dO, alpha and beta are staged in shared memory.
// grid (nseg, B*H); block kSweepThreads.
// ---------------------------------------------------------------------------
template <int DK, typename T>
__global__ void __launch_bounds__(kSweepThreads) gdr_dq_sweep(Dims d, const T* __restrict__ q,
                                                    const T* __restrict__ k,
                                                    const T* __restrict__ v,
                                                    const float* __restrict__ g,
                                                    const float* __restrict__ beta,
                                                    const T* __restrict__ dO,
                                                    const float* __restrict__ S_in,
                                                    T* __restrict__ dq, float* __restrict__ ckpt) {
    extern __shared__ float smem[];
    const int pitch = d.Dv + 1;
    const int nprt = blockDim.x / d.Dv > 0 ? int(blockDim.x) / d.Dv : 1;
    float* S = smem;                   // [DK][pitch]
    float* kb = S + DK * pitch;        // [kBlk][DK]
    float* vb = kb + kBlk * DK;        // [kBlk][Dv]
    float* ob = vb + kBlk * d.Dv;      // [kBlk][Dv]
    float* ksp = ob + kBlk * d.Dv;     // [nprt][Dv]
    __shared__ float alb[kBlk], beb[kBlk];

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int a0 = seg * d.L;
    const int nblk = d.L / kBlk;
    float* ck = ckpt + (((int64_t(seg) * d.B + b) * d.H + h) * nblk) * int64_t(DK) * d.Dv;

    const float* src = S_in + sum_off(d, seg, b, h);
    batched_copy(DK * d.Dv, [&](int e) { return __ldg(src + e); },
                 [&](int e, float x) { S[(e / d.Dv) * pitch + e % d.Dv] = x; });
    for (int c = a0; c < a0 + d.L; c += kBlk) {
        __syncthreads();  // the state is complete and the last block's vectors are read
        float* dst = ck + int64_t((c - a0) / kBlk) * DK * d.Dv;
        for (int e = threadIdx.x; e < DK * d.Dv; e += blockDim.x) dst[e] = S[(e / d.Dv) * pitch + e % d.Dv];
        stage_rows(k, d, b, c, d.H, h, DK, kb);
        stage_rows(v, d, b, c, d.H, h, d.Dv, vb);
        stage_rows(dO, d, b, c, d.H, h, d.Dv, ob);
        if (threadIdx.x < kBlk) {
            alb[threadIdx.x] = gdr_alpha(d, g, b, c + threadIdx.x, h);
            beb[threadIdx.x] = __ldg(beta + g_off(d, b, c + threadIdx.x, h));
        }
        __syncthreads();
        for (int r = 0; r < kBlk; ++r) {
            gdr_step<DK>(S, S, pitch, d.Dv, kb + r * DK, vb + r * d.Dv, alb[r], beb[r], ksp, nprt);
            // the next step's first barrier orders these reads before its update
            for (int i = threadIdx.x; i < DK; i += blockDim.x) {
                const float* row = S + i * pitch;
                const float* dr = ob + r * d.Dv;
                float a0 = 0.f, a1 = 0.f;
                for (int j = 0; j < d.Dv; j += 2) {
                    a0 = fmaf(row[j], dr[j], a0);
                    a1 = fmaf(row[j + 1], dr[j + 1], a1);
                }
                dq[qk_off(d, b, c + r, h) + i] = from_f32<T>(d.scale * (a0 + a1));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Reverse sweep.  Shared memory: D, a stack of kSlots states (pitch Dv + 1),
// the block's staged vectors and scratch.  For each kBlk-token block (last
// first) and each group of kSlots tokens of it (last first), the states
// S_{t-1} of the group are rebuilt once from the block's saved state (the
// first slot advanced in place to the group's start, the others one step
// apart), then for each token t of the group (last first):
// D_t = scale q_t dO_t^T + (t at the segment end ? dS_out : A_{t+1} D_{t+1}),
// and the gradients follow.  The stack holds four states, or fewer where
// four do not fit in shared memory.  The value columns are independent given
// k, so where four states of all Dv columns do not fit (Dk = 128, Dv > 64)
// the sweep runs twice, on columns [0, Dv/2) and then [Dv/2, Dv): dv is
// written per half, and the first launch leaves its partial dk, dbeta and dg
// (sums over the columns) in fp32 in the workspace, where the second adds
// its own before writing them.  grid (nseg, B*H); block kSweepThreads.
// ---------------------------------------------------------------------------
constexpr int kSlots = 4;
constexpr size_t kRevSmemLimit = 227 * 1024;

size_t rev_smem_bytes(int Dk, int ncol, int slots) {
    const int nprt = kSweepThreads / ncol > 0 ? kSweepThreads / ncol : 1;
    return sizeof(float) * ((1 + size_t(slots)) * size_t(Dk) * (ncol + 1) +
                            size_t(kBlk) * (2 * Dk + 2 * ncol) + size_t(nprt + 2) * ncol);
}
int rev_slots(int Dk, int ncol) {
    int s = kSlots;
    while (s > 1 && rev_smem_bytes(Dk, ncol, s) > kRevSmemLimit) s /= 2;  // kBlk stays a multiple
    return s;
}
// column parts of the reverse sweep: 2 where four states of all columns do
// not fit but four of half of them do
int rev_parts(const Dims& d) {
    return rev_slots(d.Dk, d.Dv) < kSlots && d.Dv % 16 == 0 && rev_slots(d.Dk, d.Dv / 2) == kSlots ? 2 : 1;
}
// bytes of the partial sums a two-part reverse sweep keeps: per (row, token,
// head) Dk values of dk, then dbeta's and dg's sums
size_t rev_part_bytes(const Dims& d) {
    return rev_parts(d) > 1 ? size_t(d.B) * d.T * d.H * (d.Dk + 2) * sizeof(float) : 0;
}

template <int DK, typename T>
__global__ void __launch_bounds__(kSweepThreads) gdr_reverse_sweep(Dims d, const T* __restrict__ q,
                                                         const T* __restrict__ k,
                                                         const T* __restrict__ v,
                                                         const float* __restrict__ g,
                                                         const float* __restrict__ beta,
                                                         const T* __restrict__ dO,
                                                         const float* __restrict__ dS_out,
                                                         const float* __restrict__ ckpt,
                                                         T* __restrict__ dk, T* __restrict__ dv,
                                                         float* __restrict__ dg,
                                                         float* __restrict__ dbeta, int nslots, int col0,
                                                         int ncol, int mode, float* __restrict__ part) {
    // columns [col0, col0 + ncol) of the state (d.Dv is the storage stride);
    // mode 0: every column, 1: the first part (partial sums to part), 2: the
    // last part (adds part's partial sums)
    extern __shared__ float smem[];
    const int pitch = ncol + 1;
    const int spitch = DK * pitch;     // floats per state
    const int nprt = blockDim.x / ncol > 0 ? int(blockDim.x) / ncol : 1;
    float* D = smem;                   // [DK][pitch]
    float* St = D + spitch;            // [nslots][DK][pitch]
    float* kb = St + nslots * spitch;  // [kBlk][DK]
    float* qb = kb + kBlk * DK;        // [kBlk][DK]
    float* vb = qb + kBlk * DK;        // [kBlk][ncol]
    float* ob = vb + kBlk * ncol;      // [kBlk][ncol]
    float* ksp = ob + kBlk * ncol;     // [nprt][ncol]
    float* ks = ksp + nprt * ncol;     // [ncol]  S_{t-1}^T k
    float* w = ks + ncol;              // [ncol]  D^T k
    __shared__ float alb[kBlk], beb[kBlk];
    __shared__ float red[2][kSweepThreads / 32];  // per-warp partials: k.u - alpha k.s2, <D, S>

    const int seg = blockIdx.x;
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int a0 = seg * d.L, e0 = a0 + d.L;
    const int nblk = d.L / kBlk;
    const float* ck = ckpt + (((int64_t(seg) * d.B + b) * d.H + h) * nblk) * int64_t(DK) * d.Dv;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;

    // D carries A_{t+1} D_{t+1} between tokens; it starts as dS_out
    const float* dso = dS_out + sum_off(d, seg, b, h) + col0;
    batched_copy(DK * ncol, [&](int e) { return __ldg(dso + (e / ncol) * d.Dv + e % ncol); },
                 [&](int e, float x) { D[(e / ncol) * pitch + e % ncol] = x; });
    // lanes per column (cp) and per row (rp) of the per-token phases: the
    // largest power of two up to 32 that keeps all kSweepThreads busy
    auto lanes_per = [](int n) {
        int l = 1;
        while (l < 32 && 2 * l * n <= kSweepThreads) l *= 2;
        return l;
    };
    const int cp = lanes_per(ncol), rp = lanes_per(DK);
    const int col_iters = (ncol + kSweepThreads / cp - 1) / (kSweepThreads / cp);
    const int row_iters = (DK + kSweepThreads / rp - 1) / (kSweepThreads / rp);
    // the block's value-side rows, columns [col0, col0 + ncol)
    auto stage_cols = [&](const T* __restrict__ x, int t0, float* dst) {
        batched_copy(kBlk * ncol,
                     [&](int e) {
                         const int tt = e / ncol, cc = e - tt * ncol;
                         return to_f32(x[v_off(d, b, t0 + tt, h) + col0 + cc]);
                     },
                     [&](int e, float val) { dst[e] = val; });
    };

    for (int c = e0 - kBlk; c >= a0; c -= kBlk) {
        const float* cs = ck + int64_t((c - a0) / kBlk) * DK * d.Dv;
        __syncthreads();  // the previous block's vectors are read
        stage_rows(k, d, b, c, d.H, h, DK, kb);
        stage_rows(q, d, b, c, d.qh, h / d.qdiv, DK, qb);
        stage_cols(v, c, vb);
        stage_cols(dO, c, ob);
        if (threadIdx.x < kBlk) {
            alb[threadIdx.x] = gdr_alpha(d, g, b, c + threadIdx.x, h);
            beb[threadIdx.x] = __ldg(beta + g_off(d, b, c + threadIdx.x, h));
        }
        for (int grp = kBlk / nslots - 1; grp >= 0; --grp) {
            const int r0 = grp * nslots;  // block index of the group's first token
            // slot 0 <- S_{c + r0 - 1}: the saved S_{c-1} advanced over tokens c .. c + r0 - 1
            batched_copy(DK * ncol, [&](int e) { return __ldg(cs + (e / ncol) * d.Dv + col0 + e % ncol); },
                         [&](int e, float x) { St[(e / ncol) * pitch + e % ncol] = x; });
            __syncthreads();
            for (int r = 0; r < r0; ++r)
                gdr_step<DK>(St, St, pitch, ncol, kb + r * DK, vb + r * ncol, alb[r], beb[r], ksp, nprt);
            // slot j <- S_{c + r0 + j - 1}
            for (int j = 1; j < nslots; ++j) {
                const int r = r0 + j - 1;
                gdr_step<DK>(St + (j - 1) * spitch, St + j * spitch, pitch, ncol, kb + r * DK, vb + r * ncol,
                             alb[r], beb[r], ksp, nprt);
            }
            for (int j = nslots - 1; j >= 0; --j) {
                const int r = r0 + j, t = c + r;
                const float* S = St + j * spitch;  // S_{t-1}
                const float* kt = kb + r * DK;
                const float* qt = qb + r * DK;
                const float* vt = vb + r * ncol;
                const float* dot = ob + r * ncol;
                const float al = alb[r], be = beb[r];
                // D_t = scale q_t dO_t^T + (A_{t+1} D_{t+1}, already in D)
                gdr_map<DK>(D, pitch, ncol, nprt,
                            [&](int i, int jj, float x) { return fmaf(d.scale * qt[i], dot[jj], x); });
                __syncthreads();
                // column owners: w = D_t^T k_t, kS = S_{t-1}^T k_t; dv = beta w.
                // cp consecutive lanes share a column (rows p, p + cp, ...) and
                // meet by lane exchanges; every lane of a warp runs the same
                // iterations
                for (int it = 0; it < col_iters; ++it) {
                    const int jj = threadIdx.x / cp + it * (kSweepThreads / cp), pp = threadIdx.x % cp;
                    const bool live = jj < ncol;
                    float a1 = 0.f, a2 = 0.f;
                    if (live) {
#pragma unroll 4
                        for (int i = pp; i < DK; i += cp) {
                            a1 = fmaf(kt[i], D[i * pitch + jj], a1);
                            a2 = fmaf(kt[i], S[i * pitch + jj], a2);
                        }
                    }
                    for (int o = 1; o < cp; o <<= 1) {
                        a1 += __shfl_xor_sync(0xffffffffu, a1, o);
                        a2 += __shfl_xor_sync(0xffffffffu, a2, o);
                    }
                    if (live && pp == 0) {
                        w[jj] = a1;
                        ks[jj] = a2;
                        dv[v_off(d, b, t, h) + col0 + jj] = from_f32<T>(be * a1);
                    }
                }
                __syncthreads();
                // row owners: u = D_t v_t, s1 = S_{t-1} w, s2 = D_t kS, <D, S> row
                // part; rp consecutive lanes share a row (columns p, p + rp, ...)
                float p_kb = 0.f, p_ds = 0.f;
                float* prow = part + ((int64_t(b) * d.T + t) * d.H + h) * (DK + 2);  // modes 1, 2
                for (int it = 0; it < row_iters; ++it) {
                    const int i = threadIdx.x / rp + it * (kSweepThreads / rp), pp = threadIdx.x % rp;
                    const bool live = i < DK;
                    float u = 0.f, s1 = 0.f, s2 = 0.f, ds = 0.f;
                    if (live) {
                        const float* dr = D + i * pitch;
                        const float* sr = S + i * pitch;
                        for (int jj = pp; jj < ncol; jj += rp) {
                            u = fmaf(dr[jj], vt[jj], u);
                            s1 = fmaf(sr[jj], w[jj], s1);
                            s2 = fmaf(dr[jj], ks[jj], s2);
                            ds = fmaf(dr[jj], sr[jj], ds);
                        }
                    }
                    for (int o = 1; o < rp; o <<= 1) {
                        u += __shfl_xor_sync(0xffffffffu, u, o);
                        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                        s2 += __shfl_xor_sync(0xffffffffu, s2, o);
                        ds += __shfl_xor_sync(0xffffffffu, ds, o);
                    }
                    if (live && pp == 0) {
                        const float dki = be * u - al * be * (s1 + s2);
                        if (mode == 1)
                            prow[i] = dki;
                        else
                            dk[qk_off(d, b, t, h) + i] = from_f32<T>(mode == 2 ? prow[i] + dki : dki);
                        p_kb = fmaf(kt[i], u - al * s2, p_kb);
                        p_ds += ds - be * kt[i] * s2;
                    }
                }
                p_kb = warp_sum(p_kb);
                p_ds = warp_sum(p_ds);
                if (lane == 0) {
                    red[0][wid] = p_kb;
                    red[1][wid] = p_ds;
                }
                __syncthreads();
                if (threadIdx.x == 0) {
                    float s_kb = 0.f, s_ds = 0.f;
                    for (int u2 = 0; u2 < int(blockDim.x >> 5); ++u2) {
                        s_kb += red[0][u2];
                        s_ds += red[1][u2];
                    }
                    if (mode == 1) {
                        prow[DK] = s_kb;
                        prow[DK + 1] = s_ds;
                    } else {
                        if (mode == 2) {
                            s_kb += prow[DK];
                            s_ds += prow[DK + 1];
                        }
                        dbeta[g_off(d, b, t, h)] = s_kb;
                        dg[g_off(d, b, t, h)] = starts_sequence(d.seq_idx, t) ? 0.f : al * s_ds;
                    }
                }
                // D <- A_t D_t = alpha (D - beta k w^T), the carry into token t-1
                gdr_map<DK>(D, pitch, ncol, nprt,
                            [&](int i, int jj, float x) { return al * fmaf(-be * kt[i], w[jj], x); });
                __syncthreads();
            }
        }
    }
}

template <typename T>
rm_status launch_gdr_T(GdrOp op, const Dims& d, const GdrPtrs& p, cudaStream_t s) {
    const int BH = d.B * d.H;
    const T* q = static_cast<const T*>(p.q);
    const T* k = static_cast<const T*>(p.k);
    const T* v = static_cast<const T*>(p.v);
    const T* dO = static_cast<const T*>(p.dO);
    int launches = 1;

#define RMCP_GDR_DK_SWITCH(...)                                   \
    switch (d.Dk) {                                               \
        case 16: { constexpr int DK = 16; __VA_ARGS__; break; }   \
        case 32: { constexpr int DK = 32; __VA_ARGS__; break; }   \
        case 64: { constexpr int DK = 64; __VA_ARGS__; break; }   \
        case 128: { constexpr int DK = 128; __VA_ARGS__; break; } \
        default: return RM_ERR_UNSUPPORTED;                       \
    }

    auto colgrid = [&](int ncol, int* threads) {
        *threads = ncol >= 128 ? 128 : ((ncol + 31) / 32) * 32;
        return dim3(d.nseg, BH, (ncol + *threads - 1) / *threads);
    };
    switch (op) {
        case GdrOp::kPrepare: {
            int th;
            const dim3 grid = colgrid(d.Dv + d.Dk, &th);
            RMCP_GDR_DK_SWITCH((gdr_column_sweep<DK, kGdrPrepare, T><<<grid, th, 0, s>>>(
                d, nullptr, k, v, p.g, p.beta, nullptr, nullptr, p.M, p.dS)));
            break;
        }
        case GdrOp::kApply: {
            int th;
            const dim3 grid = colgrid(d.Dv, &th);
            RMCP_GDR_DK_SWITCH((gdr_column_sweep<DK, kGdrApply, T><<<grid, th, 0, s>>>(
                d, q, k, v, p.g, p.beta, p.S_in, static_cast<T*>(p.o), nullptr, nullptr)));
            break;
        }
        case GdrOp::kComposePrefix:
        case GdrOp::kComposeSuffix: {
            const dim3 grid(BH, d.Dv / kFoldCols);
            if (op == GdrOp::kComposePrefix) {
                RMCP_GDR_DK_SWITCH((gdr_compose<DK, false><<<grid, DK * fold_parts(DK), 0, s>>>(
                    d, p.M, p.dS, d.preceding_start, p.S_in_out)));
            } else {
                RMCP_GDR_DK_SWITCH((gdr_compose<DK, true><<<grid, DK * fold_parts(DK), 0, s>>>(
                    d, p.M, p.gamma, d.following_stop, p.dS_out_out)));
            }
            break;
        }
        case GdrOp::kBackwardPrepare: {
            int th;
            const dim3 grid = colgrid(d.Dv, &th);
            RMCP_GDR_DK_SWITCH((gdr_gamma_sweep<DK, T><<<grid, th, 0, s>>>(d, q, k, p.g, p.beta, dO, p.gamma_out)));
            if (!rmcp::launch_ok()) return RM_ERR_CUDA;
            const int nprt = kSweepThreads / d.Dv > 0 ? kSweepThreads / d.Dv : 1;
            const size_t smem = sizeof(float) * (size_t(d.Dk) * (d.Dv + 1) + size_t(kBlk) * (d.Dk + 2 * d.Dv) +
                                                 size_t(nprt) * d.Dv);
            RMCP_GDR_DK_SWITCH({
                auto fn = gdr_dq_sweep<DK, T>;
                if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
                    return RM_ERR_CUDA;
                fn<<<dim3(d.nseg, BH), kSweepThreads, smem, s>>>(d, q, k, v, p.g, p.beta, dO, p.S_in,
                                                       static_cast<T*>(p.dq), p.ws);
            });
            launches = 2;
            break;
        }
        case GdrOp::kBackwardApply: {
            const int parts = rev_parts(d), ncol = d.Dv / parts;
            const int nslots = rev_slots(d.Dk, ncol);
            const size_t smem = rev_smem_bytes(d.Dk, ncol, nslots);
            // the partial sums follow the saved states in the workspace
            float* part = p.ws + (gdr_workspace_bytes(d) - rev_part_bytes(d)) / sizeof(float);
            RMCP_GDR_DK_SWITCH({
                auto fn = gdr_reverse_sweep<DK, T>;
                if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
                    return RM_ERR_CUDA;
                for (int pt = 0; pt < parts; ++pt) {
                    const int mode = parts == 1 ? 0 : (pt == 0 ? 1 : 2);
                    fn<<<dim3(d.nseg, BH), kSweepThreads, smem, s>>>(
                        d, q, k, v, p.g, p.beta, dO, p.dS_out, p.ws, static_cast<T*>(p.dk),
                        static_cast<T*>(p.dv), p.dg, p.dbeta, nslots, pt * ncol, ncol, mode, part);
                    if (pt + 1 < parts && !rmcp::launch_ok()) return RM_ERR_CUDA;
                }
            });
            launches = parts;
            break;
        }
    }
#undef RMCP_GDR_DK_SWITCH
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(launches);
    return RM_OK;
}

}  // namespace

bool gdr_supports(const Dims& d) {
    return (d.Dk == 16 || d.Dk == 32 || d.Dk == 64 || d.Dk == 128) && d.Dv % 8 == 0 && d.Dv >= 8 &&
           d.Dv <= 128 &&
           d.L % kBlk == 0 && !d.vg;
}

size_t gdr_workspace_bytes(const Dims& d) {
    // the saved states (every kBlk tokens), then the two-part reverse sweep's
    // partial sums (where it runs in two parts)
    const size_t b = size_t(d.B) * d.H * (size_t(d.T) / kBlk) * d.Dk * d.Dv * sizeof(float);
    return (b + 255) / 256 * 256 + rev_part_bytes(d);
}

rm_status launch_gdr(GdrOp op, const Dims& d, rm_dtype dt, const GdrPtrs& p, cudaStream_t s) {
    return dt == RM_F32 ? launch_gdr_T<float>(op, d, p, s) : launch_gdr_T<__nv_bfloat16>(op, d, p, s);
}

}  // namespace rmcp
