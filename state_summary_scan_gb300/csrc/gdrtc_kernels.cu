// gdrtc_kernels.cu -- tensor-core sweeps (sm_103a, tcgen05 + TMA) of the
// gated delta rule: bf16 storage, Dk = Dv = 64, segment lengths that are
// multiples of 64.  Per row b and head h,
//     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
//     o_t = scale S_t^T q_t,
// alpha_t = exp(g_t) (0 when token t starts a sequence): the summary
// S_out = M S_in + delta_S of CPForwardUnpackedSummary on the Megatron-Core
// page "core.ssm.context_parallel.chunkwise" with a Dk x Dk transition M.
//
// Chunkwise (WY/UT) form.  In a chunk of 64 tokens with S_prev the state
// before it, let b_t be the running sum of the gates, Gam[t][r] =
// exp(b_t - b_r) for r <= t in one sequence (else 0), gam_t = exp(b_t) while
// no sequence starts in [0, t] (else 0).  Unrolling the recurrence one token
// at a time gives S_t = gam_t S_prev + sum_{r<=t} Gam[t][r] k_r D_r^T with
//     D_t = beta_t (v_t - gam_t S_prev^T k_t - sum_{r<t} Gam[t][r] (k_r.k_t) D_r),
// i.e. (I + A) D = diag(beta) (V - (K o gam) S_prev) with the strictly lower
// A[t][r] = beta_t (k_t.k_r) Gam[t][r].  With T = (I + A)^{-1} diag(beta):
//     D      = T V - T (K o gam) S_prev          (U = T V, W = T (K o gam))
//     O      = scale ((Q o gam) S_prev + mask(Q K^T o Gam) D)
//     S_next = gam_63 S_prev + (K o Gam[63][.])^T D
// Every product is a tcgen05.mma of bf16 tiles in 128-byte-swizzled shared
// memory with an fp32 accumulator in tensor memory; T is formed on the CUDA
// cores in fp32 (the inverse of a unit lower-triangular matrix by 16 x 16
// blocks) once per chunk, for every chunk at once, and the walks read it from
// the workspace; the fp32 state lives in registers (16 values a thread).
//
// Kernels (256 threads a CTA; thread 0 issues the TMA loads and stores and
// the products, and the CTA steps through each chunk together):
//   gdrtc_factor_kernel       one CTA per (chunk, row, head): the chunk's T
//                             and (I + A)^{-1} into the workspace (the forward
//                             prepare's first launch)
// and the walks, one CTA per (segment, row, head):
//   gdrtc_prepare_kernel      the recurrence on [S | M] from [0 | I] with
//                             values [V | 0]: delta_S and the transition M
//   gdrtc_apply_kernel        o from S_in (T from the workspace)
//   gdrtc_bwd_prepare_kernel  dq by a forward walk that saves each chunk's
//                             incoming state, and gamma by a reverse walk of
//                             the state adjoint (two CTA roles, one launch)
//   gdrtc_adjoint_kernel      the state adjoint E of each chunk by a reverse
//                             walk from dS_out (the backward apply's first launch)
// and, one CTA per (chunk, row, head), every chunk at once:
//   gdrtc_chunk_grad_kernel   dk, dv, dbeta and dg of the chunk from its
//                             saved S_prev and E (the backward apply's second)
#include <cstdio>

#include "tc_tiles.cuh"

namespace rmcp {
namespace gdrtc {

using namespace tc;

namespace {

constexpr int kD = 64;                 // Dk = Dv
constexpr uint32_t T8 = kTileBytes;    // one [64][64] bf16 tile
constexpr int kP = kD + 1;             // pitch of the fp32 [64][64] A (and scratch) arrays
constexpr int kQ = kD + 4;             // pitch of the fp32 inverse and its partial sums (16-byte rows)
constexpr size_t kF32Bytes = (kD * kP + 2 * kD * kQ) * sizeof(float);  // A, X, Y

// Row t of a [64][64] bf16 tile times w[t] (times mul), from src into dst:
// 512 chunks of 16 bytes, two a thread (a row's scale does not depend on the
// swizzle).
__device__ __forceinline__ void rows_scaled(const uint8_t* src, uint8_t* dst, const float* w, float mul,
                                            int tid) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int n = tid + 256 * k;
        const int r = n >> 3;
        const uint32_t off = uint32_t(r * 128 + (n & 7) * 16);
        float x[8];
        unpack8(*reinterpret_cast<const uint4*>(src + off), x);
        const float f = mul * w[r];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= f;
        *reinterpret_cast<uint4*>(dst + off) = pack8(x);
    }
}

// Xs = (I + La)^{-1} for the strictly lower La (fp32, pitch kP; Xs and the
// scratch Ys pitch kQ): a unit lower triangular inverse by 16 x 16 blocks.
// The four diagonal blocks by forward substitution with the 16 rows of a
// column in 16 lanes (x_k reaches the rows below it by a shuffle; four columns
// a thread, every thread of the CTA busy), then the blocks below the diagonal
// by their distance from it, X_ij = -X_ii sum_{k=j}^{i-1} A_ik X_kj (Ys holds
// the sums), four adjacent columns a thread so that each loaded A or X entry
// serves four products.  Entries above the diagonal are 0.  All 256 threads of
// the CTA call it.
__device__ __noinline__ void tri_inverse(const float* La, float* Xs, float* Ys) {
    const int tid = threadIdx.x;
    for (int e = tid; e < kD * kD / 4; e += blockDim.x) {  // the six blocks above the diagonal
        const int r = e >> 4, c = (e & 15) * 4;
        if ((c >> 4) > (r >> 4)) *reinterpret_cast<float4*>(Xs + r * kQ + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    {
        // warp w: diagonal block w / 2; lane: row r, column group (w % 2, lane / 16)
        const int w = tid >> 5, lane = tid & 31;
        const int o = 16 * (w >> 1), r = lane & 15, grp = ((w & 1) << 1) | (lane >> 4);
        float x[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) x[m] = r == 4 * grp + m ? 1.f : 0.f;
        const float* lrow = La + (o + r) * kP + o;
#pragma unroll
        for (int k = 0; k < 15; ++k) {
            const float l = lrow[k];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float xk = __shfl_sync(kFull, x[m], (lane & 16) | k);
                if (r > k) x[m] = fmaf(-l, xk, x[m]);
            }
        }
        *reinterpret_cast<float4*>(Xs + (o + r) * kQ + o + 4 * grp) = make_float4(x[0], x[1], x[2], x[3]);
    }
    __syncthreads();
    for (int dist = 1; dist < 4; ++dist) {
        // thread: block (j + dist, j), row r, columns 4 q .. 4 q + 3 of the block
        const bool act = tid < 64 * (4 - dist);
        const int j = tid >> 6, r = (tid >> 2) & 15, q = tid & 3, i = j + dist;
        if (act) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            const float* arow = La + (16 * i + r) * kP;
            const float* xc = Xs + 16 * j + 4 * q;
#pragma unroll 16
            for (int kk = 16 * j; kk < 16 * i; ++kk) {
                const float a = arow[kk];
                const float4 xv = *reinterpret_cast<const float4*>(xc + kk * kQ);
                a0 = fmaf(a, xv.x, a0);
                a1 = fmaf(a, xv.y, a1);
                a2 = fmaf(a, xv.z, a2);
                a3 = fmaf(a, xv.w, a3);
            }
            *reinterpret_cast<float4*>(Ys + (16 * i + r) * kQ + 16 * j + 4 * q) = make_float4(a0, a1, a2, a3);
        }
        __syncthreads();
        if (act) {
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
            const float* xrow = Xs + (16 * i + r) * kQ + 16 * i;
            const float* yc = Ys + 16 * i * kQ + 16 * j + 4 * q;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const float a = xrow[kk];
                const float4 yv = *reinterpret_cast<const float4*>(yc + kk * kQ);
                a0 = fmaf(a, yv.x, a0);
                a1 = fmaf(a, yv.y, a1);
                a2 = fmaf(a, yv.z, a2);
                a3 = fmaf(a, yv.w, a3);
            }
            *reinterpret_cast<float4*>(Xs + (16 * i + r) * kQ + 16 * j + 4 * q) = make_float4(-a0, -a1, -a2, -a3);
        }
        __syncthreads();
    }
}

// Columns c0..c0+15 of row tau of the inverse (pitch kQ).
__device__ __forceinline__ void xs_row16(const float* Xs, int tau, int c0, float* x) {
    const float* row = Xs + tau * kQ + c0;
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
        const float4 v = *reinterpret_cast<const float4*>(row + e);
        x[e] = v.x; x[e + 1] = v.y; x[e + 2] = v.z; x[e + 3] = v.w;
    }
}

// The next chunk's gates (warp 0) and write strengths (threads 0..63), loaded
// into registers while the current chunk runs, then published to shared
// memory at the top of the chunk that uses them.
struct GateFetch {
    GateRegs gr;
    float be;
};
__device__ __forceinline__ GateFetch gates_fetch(const Dims& d, const float* __restrict__ g,
                                                 const float* __restrict__ beta, int b, int h, int t0,
                                                 const Geo& G) {
    GateFetch f{};
    if (G.warp == 0) f.gr = gate_load(d, g, b, h, t0, G.lane);
    if (G.tid < kChunk) f.be = __ldg(beta + g_off(d, b, t0 + G.tid, h));
    return f;
}
__device__ __forceinline__ void gates_commit(const GateFetch& f, GateSmem& gs, float* beta_s, const Geo& G) {
    if (G.warp == 0) gate_prep(f.gr, &gs, G.lane);
    if (G.tid < kChunk) beta_s[G.tid] = f.be;
}

// Row tau, columns c0..c0+15 of the within-sequence decay Gam[tau][r] =
// exp(b_tau - b_r) for r < tau (strict) or r <= tau, 0 elsewhere.  Branch
// free: the gate table is read by 16-byte loads and every exponential is
// taken (those outside the mask may overflow; the select drops them).
__device__ __forceinline__ void decay16(const GateSmem& gs, int tau, int c0, bool strict, float* m) {
    const int lt = gs.lid[tau];
    const float bt = gs.b[tau];
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
        const float4 bv = *reinterpret_cast<const float4*>(gs.b + c0 + e);
        const int4 lv = *reinterpret_cast<const int4*>(gs.lid + c0 + e);
        const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
        const int ll[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = c0 + e + u;
            const float x = __expf(bt - bb[u]);
            m[e + u] = ((strict ? r < tau : r <= tau) && ll[u] == lt) ? x : 0.f;
        }
    }
}

// A (strictly lower, fp32) from this thread's 16 columns r = c0..c0+15 of
// row tau of K K^T and of the inclusive decay m: A[tau][r] = beta_tau
// (k_tau.k_r) Gam[tau][r], r < tau.
__device__ __forceinline__ void a_row16(const float* beta_s, const float* kk, const float* m, int tau, int c0,
                                        float* La) {
    const float be = beta_s[tau];
#pragma unroll
    for (int e = 0; e < 16; ++e) La[tau * kP + c0 + e] = c0 + e < tau ? be * kk[e] * m[e] : 0.f;
}

// The state row tau, columns c0..c0+15, of a [64][64] fp32 block at src.
__device__ __forceinline__ void load_row16(const float* src, int tau, int c0, float* x) {
    const float* p = src + tau * kD + c0;
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
        const float4 v = *reinterpret_cast<const float4*>(p + e);
        x[e] = v.x; x[e + 1] = v.y; x[e + 2] = v.z; x[e + 3] = v.w;
    }
}
__device__ __forceinline__ void save_row16(float* dst, int tau, int c0, const float* x) {
    float* p = dst + tau * kD + c0;
#pragma unroll
    for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4*>(p + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
}

// One synchronous step: fence shared-memory writes for the tensor core and
// make every thread's tensor-memory reads and shared writes visible.
__device__ __forceinline__ void cta_sync_tc() {
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Commit the products issued so far (thread 0) and wait for them (everyone).
__device__ __forceinline__ void commit_wait(uint64_t* mbar, uint32_t& mph, int tid) {
    if (tid == 0) mma_commit(smem_u32(mbar));
    mbar_wait(smem_u32(mbar), mph);
    mph ^= 1;
    tc_fence_after();
}

constexpr uint32_t idKK = idesc_bf16(64, 64, 0, 0);  // A K-major, B K-major
constexpr uint32_t idKM = idesc_bf16(64, 64, 0, 1);  // A K-major, B MN-major
constexpr uint32_t idMM = idesc_bf16(64, 64, 1, 1);  // A MN-major, B MN-major

// D (+)= A B over K = 64 for [64][64] tiles (four K-steps of 16).
__device__ __forceinline__ void mma_kk(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(d, desc_plus(a, k * 32), desc_plus(b, k * 32), idKK, (acc || k > 0) ? 1u : 0u);
}
__device__ __forceinline__ void mma_km(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(d, desc_plus(a, k * 32), desc_plus(b, k * 2048), idKM, (acc || k > 0) ? 1u : 0u);
}
__device__ __forceinline__ void mma_mm(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
#pragma unroll
    for (int k = 0; k < 4; ++k) mma_bf16(d, desc_plus(a, k * 2048), desc_plus(b, k * 2048), idMM, (acc || k > 0) ? 1u : 0u);
}

// ===========================================================================
// The per-chunk factors.  The forward prepare forms, for every chunk, T =
// (I + A)^{-1} diag(beta) and (I + A)^{-1} (they depend on k, beta and the
// gates only) and leaves them in the workspace after the saved states: a
// bf16 table of [chunks][2][64][64] rows, chunk index ((seg B + b) H + h)
// (L / 64) + c.  The apply and the backward load them by TMA instead of
// forming them again.
// ===========================================================================
__device__ __forceinline__ int64_t chunk_base(const Dims& d, int seg, int b, int h) {
    return ((int64_t(seg) * d.B + b) * d.H + h) * (d.L / kChunk);
}
// first row of factor f (0: T, 1: the inverse) of chunk ci in the factor table
__device__ __forceinline__ int fac_row(int64_t ci, int f) { return int((2 * ci + f) * kD); }

// ===========================================================================
// forward apply: o from S_in.  Two CTAs a SM: one input stage, refilled with
// the next chunk as soon as the chunk's first products (the last readers of
// Q, K, V and T) are done.
// Shared memory (8 KB tiles): Q|K|V|T; scale Q o gam, K o gam (then -W),
// K o Gam[63], P, D (then o staging), S (bf16).
// Tensor memory: [0,64) the state product; [64,128) Q K^T, then O; [128,192)
// W; [192,256) U, then D.
// ===========================================================================
constexpr uint32_t AP_STAGE = 4 * T8;
constexpr uint32_t AP_QG = AP_STAGE, AP_KG = AP_QG + T8, AP_KC = AP_KG + T8, AP_P = AP_KC + T8;
constexpr uint32_t AP_DL = AP_P + T8, AP_S = AP_DL + T8;
constexpr uint32_t AP_WN = AP_KG;  // -W over K o gam, which dies with W
constexpr uint32_t AP_O = AP_DL;   // o over D, which dies with O and the state product
constexpr size_t kApplySmem = AP_S + T8 + 1024;

__global__ void __launch_bounds__(256, 2)
    gdrtc_apply_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                       const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                       const __grid_constant__ CUtensorMap mf, const __grid_constant__ CUtensorMap mo,
                       const float* __restrict__ g, const float* __restrict__ beta,
                       const float* __restrict__ S_in) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ GateSmem gsb[2];
    __shared__ __align__(16) float bsb[2][kChunk];
    __shared__ __align__(8) uint64_t full, mbar;
    __shared__ uint32_t tmem_slot;
    constexpr uint32_t TKK = 0, TQK = 64, TW = 128, TD = 192;

    const Geo G = geo();
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    const int c0 = 32 * G.grp + 16 * G.hi;  // this thread's 16 columns of a [64][64] product
    const int64_t cb = chunk_base(d, seg, b, h);

    if (G.tid == 0) {
        mbar_init(smem_u32(&full), 1);
        mbar_init(smem_u32(&mbar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 256);
    // the state row tau, columns c0..c0+15, in registers; its bf16 copy in the S tile
    float Sr[16];
    load_row16(S_in + sum_off(d, seg, b, h), G.tau, c0, Sr);
    store_row16(smem + AP_S, G.tau, c0, Sr);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    auto load = [&](int c) {
        const int row = b * d.T + a0 + c * kChunk;
        const uint32_t bar = smem_u32(&full);
        uint8_t* st = smem;
        mbar_expect_tx(bar, AP_STAGE);
        tma_load_3d(smem_u32(st), &mq, 0, h / d.qdiv, row, bar);
        tma_load_3d(smem_u32(st + T8), &mk, 0, h, row, bar);
        tma_load_3d(smem_u32(st + 2 * T8), &mv, 0, h, row, bar);
        tma_load_3d(smem_u32(st + 3 * T8), &mf, 0, 0, fac_row(cb + c, 0), bar);
    };
    if (G.tid == 0) load(0);
    const uint32_t sb0 = smem_u32(smem);
    const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, T8, 1024);
    GateFetch gf = gates_fetch(d, g, beta, b, h, a0, G);
    gates_commit(gf, gsb[0], bsb[0], G);
    if (nch > 1) gf = gates_fetch(d, g, beta, b, h, a0 + kChunk, G);
    uint32_t mph = 0;
    for (int c = 0; c < nch; ++c) {
        const int t0 = a0 + c * kChunk;
        constexpr uint32_t sq = 0, sk = T8, sv = 2 * T8, st = 3 * T8;
        GateSmem& gs = gsb[c & 1];
        __syncthreads();
        mbar_wait(smem_u32(&full), c & 1);
        tc_fence_after();
        if (G.tid == 0) mma_kk(tmem + TQK, desc_plus(DK, sq), desc_plus(DK, sk), 0);  // Q K^T
        rows_scaled(smem + sq, smem + AP_QG, gs.win, d.scale, G.tid);  // scale Q o gam
        rows_scaled(smem + sk, smem + AP_KG, gs.win, 1.f, G.tid);      // K o gam
        rows_scaled(smem + sk, smem + AP_KC, gs.wout, 1.f, G.tid);     // K o Gam[63]
        cta_sync_tc();
        if (G.tid == 0) {  // W = T (K o gam), U = T V
            mma_km(tmem + TW, desc_plus(DK, st), desc_plus(DM, AP_KG), 0);
            mma_km(tmem + TD, desc_plus(DK, st), desc_plus(DM, sv), 0);
        }
        if (c + 1 < nch) {  // the next chunk's gate tables, while the products run
            gates_commit(gf, gsb[(c + 1) & 1], bsb[(c + 1) & 1], G);
            if (c + 2 < nch) gf = gates_fetch(d, g, beta, b, h, t0 + 2 * kChunk, G);
        }
        commit_wait(&mbar, mph, G.tid);
        if (G.tid == 0 && c + 1 < nch) load(c + 1);  // Q, K, V and T are read
        {
            float qk[16], w[16], m[16];
            tok16x2(tmem, G, TQK + 32 * G.grp, TW + 32 * G.grp, qk, w);
            decay16(gs, G.tau, c0, false, m);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                qk[e] *= d.scale * m[e];  // P = scale (Q K^T o Gam), r <= tau
                w[e] = -w[e];
            }
            store_row16(smem + AP_P, G.tau, c0, qk);
            store_row16(smem + AP_WN, G.tau, c0, w);
        }
        if (G.tid == 0) bulk_wait_read();  // the previous o store has read its tile (over D)
        cta_sync_tc();
        if (G.tid == 0)  // D = U - W S_prev
            mma_km(tmem + TD, desc_plus(DK, AP_WN), desc_plus(DM, AP_S), 1);
        commit_wait(&mbar, mph, G.tid);
        {
            float x[16];
            tok16(tmem, G, TD + 32 * G.grp, x);
            store_row16(smem + AP_DL, G.tau, c0, x);
        }
        cta_sync_tc();
        if (G.tid == 0) {
            mma_km(tmem + TQK, desc_plus(DK, AP_QG), desc_plus(DM, AP_S), 0);  // O = (scale Q o gam) S_prev
            mma_km(tmem + TQK, desc_plus(DK, AP_P), desc_plus(DM, AP_DL), 1);  //   + P D
            mma_mm(tmem + TKK, desc_plus(DM, AP_KC), desc_plus(DM, AP_DL), 0); // (K o Gam[63])^T D
        }
        commit_wait(&mbar, mph, G.tid);
        {
            float x[16], y[16];
            tok16x2(tmem, G, TQK + 32 * G.grp, TKK + 32 * G.grp, x, y);
            store_row16(smem + AP_O, G.tau, c0, x);
#pragma unroll
            for (int e = 0; e < 16; ++e) Sr[e] = fmaf(gs.W, Sr[e], y[e]);
            store_row16(smem + AP_S, G.tau, c0, Sr);
        }
        cta_sync_tc();
        if (G.tid == 0) {
            tma_store_3d(&mo, smem_u32(smem + AP_O), 0, h, b * d.T + t0);
            bulk_commit();
        }
    }
    if (G.tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// per-chunk factors (the first launch of the forward prepare): one CTA per
// (chunk, row, head), every chunk at once (they do not depend on the state).
// K K^T on the tensor cores, A from it and the chunk's gates, the fp32
// inverse, then T = (I + A)^{-1} diag(beta) and (I + A)^{-1} (bf16) to the
// factor table.
// Shared memory: K (bf16); fp32 A, X, Y.  Tensor memory: K K^T.
// ===========================================================================
constexpr uint32_t FA_F32 = T8;
constexpr size_t kFactorSmem = FA_F32 + kF32Bytes + 1024;

__global__ void __launch_bounds__(256, 3)
    gdrtc_factor_kernel(const Dims d, const __grid_constant__ CUtensorMap mk, const float* __restrict__ g,
                        const float* __restrict__ beta, __nv_bfloat16* __restrict__ fac) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    float* La = reinterpret_cast<float*>(smem + FA_F32);
    float* Xs = La + kD * kP;
    float* Ys = Xs + kD * kQ;
    __shared__ GateSmem gs;
    __shared__ __align__(16) float beta_s[kChunk];
    __shared__ __align__(8) uint64_t full, mbar;
    __shared__ uint32_t tmem_slot;

    const Geo G = geo();
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int t0 = blockIdx.x * kChunk;
    const int seg = t0 / d.L, c = (t0 % d.L) / kChunk;
    const int64_t ci = chunk_base(d, seg, b, h) + c;
    const int c0 = 32 * G.grp + 16 * G.hi;

    if (G.tid == 0) {
        mbar_init(smem_u32(&full), 1);
        mbar_init(smem_u32(&mbar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (G.tid == 0) {
        mbar_expect_tx(smem_u32(&full), T8);
        tma_load_3d(smem_u32(smem), &mk, 0, h, b * d.T + t0, smem_u32(&full));
    }
    gates_commit(gates_fetch(d, g, beta, b, h, t0, G), gs, beta_s, G);
    mbar_wait(smem_u32(&full), 0);
    tc_fence_after();
    const uint64_t DK = sdesc(smem_u32(smem), 16, 1024);
    if (G.tid == 0) mma_kk(tmem, DK, DK, 0);  // K K^T
    uint32_t mph = 0;
    commit_wait(&mbar, mph, G.tid);
    __syncthreads();  // the gate tables are complete
    {
        float kk[16], m[16];
        tok16(tmem, G, 32 * G.grp, kk);
        decay16(gs, G.tau, c0, false, m);
        a_row16(beta_s, kk, m, G.tau, c0, La);
    }
    __syncthreads();
    tri_inverse(La, Xs, Ys);
    {
        float x[16], t[16];
        xs_row16(Xs, G.tau, c0, x);
#pragma unroll
        for (int e = 0; e < 16; ++e) t[e] = x[e] * beta_s[c0 + e];
        __nv_bfloat16* f = fac + (int64_t(fac_row(ci, 0)) + G.tau) * kD + c0;
        store_bf16x16(f, t);
        store_bf16x16(f + kD * kD, x);
    }
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 64);
}

// ===========================================================================
// forward prepare walk (the second launch): the recurrence on [S | M] from
// [0 | I] with values [V | 0] over one segment: S_out = M S_in + delta_S
// with delta_S = S and M its last state.  Per chunk, with T from the factor
// table: D_S = T V - W S, D_M = -W M, then S = gam_63 S + (K o Gam[63])^T D_S
// and M likewise.  Two CTAs a SM: one input stage, refilled once the
// chunk's first products are done.
// Shared memory: K|V|T; K o gam (then -W), K o Gam[63], D_S, D_M, S, M (bf16).
// Tensor memory: [0,64) the S product; [64,128) W, then the M product;
// [128,192) U, then D_S; [192,256) D_M.
// ===========================================================================
constexpr uint32_t PR_STAGE = 3 * T8;
constexpr uint32_t PR_KG = PR_STAGE, PR_KC = PR_KG + T8, PR_DS = PR_KC + T8, PR_DM = PR_DS + T8;
constexpr uint32_t PR_S = PR_DM + T8, PR_M = PR_S + T8;
constexpr uint32_t PR_WN = PR_KG;  // -W over K o gam, which dies with W
constexpr size_t kPrepSmem = PR_M + T8 + 1024;

__global__ void __launch_bounds__(256, 2)
    gdrtc_prepare_kernel(const Dims d, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mf,
                         const float* __restrict__ g, const float* __restrict__ beta, float* __restrict__ M,
                         float* __restrict__ dS) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ GateSmem gsb[2];
    __shared__ __align__(16) float bsb[2][kChunk];
    __shared__ __align__(8) uint64_t full, mbar;
    __shared__ uint32_t tmem_slot;
    constexpr uint32_t TKK = 0, TW = 64, TU = 128, TDM = 192;

    const Geo G = geo();
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    const int c0 = 32 * G.grp + 16 * G.hi;
    const int64_t cb = chunk_base(d, seg, b, h);

    if (G.tid == 0) {
        mbar_init(smem_u32(&full), 1);
        mbar_init(smem_u32(&mbar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 256);
    float Sr[16], Mr[16];  // row tau, columns c0..c0+15 of S and of M
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        Sr[e] = 0.f;
        Mr[e] = (c0 + e == G.tau) ? 1.f : 0.f;
    }
    store_row16(smem + PR_S, G.tau, c0, Sr);
    store_row16(smem + PR_M, G.tau, c0, Mr);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    auto load = [&](int c) {
        const int row = b * d.T + a0 + c * kChunk;
        const uint32_t bar = smem_u32(&full);
        mbar_expect_tx(bar, PR_STAGE);
        tma_load_3d(smem_u32(smem), &mk, 0, h, row, bar);
        tma_load_3d(smem_u32(smem + T8), &mv, 0, h, row, bar);
        tma_load_3d(smem_u32(smem + 2 * T8), &mf, 0, 0, fac_row(cb + c, 0), bar);
    };
    if (G.tid == 0) load(0);
    const uint32_t sb0 = smem_u32(smem);
    const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, T8, 1024);
    GateFetch gf = gates_fetch(d, g, beta, b, h, a0, G);
    gates_commit(gf, gsb[0], bsb[0], G);
    if (nch > 1) gf = gates_fetch(d, g, beta, b, h, a0 + kChunk, G);
    uint32_t mph = 0;
    for (int c = 0; c < nch; ++c) {
        const int t0 = a0 + c * kChunk;
        GateSmem& gs = gsb[c & 1];
        __syncthreads();
        mbar_wait(smem_u32(&full), c & 1);
        tc_fence_after();
        rows_scaled(smem, smem + PR_KG, gs.win, 1.f, G.tid);   // K o gam
        rows_scaled(smem, smem + PR_KC, gs.wout, 1.f, G.tid);  // K o Gam[63]
        cta_sync_tc();
        if (G.tid == 0) {  // W = T (K o gam), U = T V
            const uint64_t t = desc_plus(DK, 2 * T8);
            mma_km(tmem + TW, t, desc_plus(DM, PR_KG), 0);
            mma_km(tmem + TU, t, desc_plus(DM, T8), 0);
        }
        if (c + 1 < nch) {  // the next chunk's gate tables, while the products run
            gates_commit(gf, gsb[(c + 1) & 1], bsb[(c + 1) & 1], G);
            if (c + 2 < nch) gf = gates_fetch(d, g, beta, b, h, t0 + 2 * kChunk, G);
        }
        commit_wait(&mbar, mph, G.tid);
        if (G.tid == 0 && c + 1 < nch) load(c + 1);  // K, V and T are read
        {
            float w[16];
            tok16(tmem, G, TW + 32 * G.grp, w);
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = -w[e];
            store_row16(smem + PR_WN, G.tau, c0, w);
        }
        cta_sync_tc();
        if (G.tid == 0) {
            const uint64_t wn = desc_plus(DK, PR_WN);
            mma_km(tmem + TU, wn, desc_plus(DM, PR_S), 1);   // D_S = U - W S
            mma_km(tmem + TDM, wn, desc_plus(DM, PR_M), 0);  // D_M = -W M
        }
        commit_wait(&mbar, mph, G.tid);
        {
            float x[16], y[16];
            tok16x2(tmem, G, TU + 32 * G.grp, TDM + 32 * G.grp, x, y);
            store_row16(smem + PR_DS, G.tau, c0, x);
            store_row16(smem + PR_DM, G.tau, c0, y);
        }
        cta_sync_tc();
        if (G.tid == 0) {
            const uint64_t kc = desc_plus(DM, PR_KC);
            mma_mm(tmem + TKK, kc, desc_plus(DM, PR_DS), 0);  // (K o Gam[63])^T D_S
            mma_mm(tmem + TW, kc, desc_plus(DM, PR_DM), 0);   // (K o Gam[63])^T D_M
        }
        commit_wait(&mbar, mph, G.tid);
        {
            float x[16], y[16];
            tok16x2(tmem, G, TKK + 32 * G.grp, TW + 32 * G.grp, x, y);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                Sr[e] = fmaf(gs.W, Sr[e], x[e]);
                Mr[e] = fmaf(gs.W, Mr[e], y[e]);
            }
            store_row16(smem + PR_S, G.tau, c0, Sr);
            store_row16(smem + PR_M, G.tau, c0, Mr);
        }
        cta_sync_tc();
    }
    save_row16(dS + sum_off(d, seg, b, h), G.tau, c0, Sr);
    save_row16(M + ((int64_t(seg) * d.B + b) * d.H + h) * kD * kD, G.tau, c0, Mr);
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 256);
}


// Per-block state of the backward kernels (static shared memory).
struct BwdShared {
    GateSmem gsb[2];                   // gate tables, by chunk parity
    alignas(16) float bsb[2][kChunk];  // write strengths, by chunk parity
    float red[3][2][kChunk];  // row partials of the gate, key-norm and beta terms, by column half
    float dbm[kChunk];        // row sum minus column sum of the score-gradient products
    float red_se[8];          // per-warp <S_prev, E>
    alignas(8) uint64_t full[2];
    alignas(8) uint64_t mbar;
    uint32_t tmem_slot;
};

__device__ __forceinline__ void bwd_setup(BwdShared& sh, const Geo& G, int cols) {
    if (G.tid == 0) {
        mbar_init(smem_u32(&sh.full[0]), 1);
        mbar_init(smem_u32(&sh.full[1]), 1);
        mbar_init(smem_u32(&sh.mbar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&sh.tmem_slot), cols);
}

// ===========================================================================
// backward prepare, dq walk (blockIdx.z == 0): the forward recurrence again
// from S_in with dO in place of the queries,
//     dq = scale (gam o (dO S_prev^T) + mask(dO D^T o Gam) K),
// (dq_t = scale S_t dO_t with S_t = gam_t S_prev + sum_{r<=t} Gam[t][r] k_r D_r^T)
// and S_prev saved to the workspace before each chunk.
// Shared memory: two stages of K|V|dO|T; K o gam (then -W), K o Gam[63],
// scale dO o gam, D (then P, then dq staging), S (bf16).
// Tensor memory: [0,64) dO D^T; [64,128) dq; [128,192) W, then the state
// product; [192,256) U, then D.
// ===========================================================================
constexpr uint32_t DQ_STAGE = 4 * T8;
constexpr uint32_t DQ_KG = 2 * DQ_STAGE, DQ_KC = DQ_KG + T8, DQ_OG = DQ_KC + T8, DQ_DL = DQ_OG + T8;
constexpr uint32_t DQ_S = DQ_DL + T8;
constexpr uint32_t DQ_WN = DQ_KG;  // -W over K o gam, which dies with W
constexpr uint32_t DQ_P = DQ_DL;   // P over D, which dies with dO D^T and the state product
constexpr uint32_t DQ_O = DQ_DL;   // dq over P, which dies with P K
constexpr size_t kDqSmem = DQ_S + T8 + 1024;

__device__ __forceinline__ void dq_walk(const Dims& d, const CUtensorMap* mk, const CUtensorMap* mv,
                                        const CUtensorMap* mo, const CUtensorMap* mf, const CUtensorMap* mdq,
                                        const float* __restrict__ g, const float* __restrict__ beta,
                                        const float* __restrict__ S_in, float* __restrict__ ws,
                                        uint8_t* smem, BwdShared& sh, uint32_t tmem, const Geo& G) {
    constexpr uint32_t TKK = 0, TQ = 64, TW = 128, TD = 192;
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    const int c0 = 32 * G.grp + 16 * G.hi;
    const int64_t cb = chunk_base(d, seg, b, h);
    float* ck = ws + cb * int64_t(kD * kD);

    float Sr[16];
    load_row16(S_in + sum_off(d, seg, b, h), G.tau, c0, Sr);
    store_row16(smem + DQ_S, G.tau, c0, Sr);
    auto load = [&](int c, int s) {
        const int row = b * d.T + a0 + c * kChunk;
        const uint32_t bar = smem_u32(&sh.full[s]);
        uint8_t* st = smem + s * DQ_STAGE;
        mbar_expect_tx(bar, DQ_STAGE);
        tma_load_3d(smem_u32(st), mk, 0, h, row, bar);
        tma_load_3d(smem_u32(st + T8), mv, 0, h, row, bar);
        tma_load_3d(smem_u32(st + 2 * T8), mo, 0, h, row, bar);
        tma_load_3d(smem_u32(st + 3 * T8), mf, 0, 0, fac_row(cb + c, 0), bar);
    };
    if (G.tid == 0) {
        load(0, 0);
        if (nch > 1) load(1, 1);
    }
    const uint32_t sb0 = smem_u32(smem);
    const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, T8, 1024);
    GateFetch gf = gates_fetch(d, g, beta, b, h, a0, G);
    gates_commit(gf, sh.gsb[0], sh.bsb[0], G);
    if (nch > 1) gf = gates_fetch(d, g, beta, b, h, a0 + kChunk, G);
    uint32_t mph = 0;
    for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        const int t0 = a0 + c * kChunk;
        const uint32_t sk = s * DQ_STAGE, sv = sk + T8, so = sk + 2 * T8, st = sk + 3 * T8;
        save_row16(ck + int64_t(c) * kD * kD, G.tau, c0, Sr);
        GateSmem& gs = sh.gsb[c & 1];
        if (G.tid == 0 && c >= 1 && c + 1 < nch) load(c + 1, s ^ 1);  // the previous chunk's products are done
        __syncthreads();
        mbar_wait(smem_u32(&sh.full[s]), (c >> 1) & 1);
        tc_fence_after();
        rows_scaled(smem + sk, smem + DQ_KG, gs.win, 1.f, G.tid);      // K o gam
        rows_scaled(smem + sk, smem + DQ_KC, gs.wout, 1.f, G.tid);     // K o Gam[63]
        rows_scaled(smem + so, smem + DQ_OG, gs.win, d.scale, G.tid);  // scale dO o gam
        cta_sync_tc();
        if (G.tid == 0) {
            mma_kk(tmem + TQ, desc_plus(DK, DQ_OG), desc_plus(DK, DQ_S), 0);  // (scale dO o gam) S^T
            mma_km(tmem + TW, desc_plus(DK, st), desc_plus(DM, DQ_KG), 0);    // W = T (K o gam)
            mma_km(tmem + TD, desc_plus(DK, st), desc_plus(DM, sv), 0);       // U = T V
        }
        if (c + 1 < nch) {  // the next chunk's gate tables, while the products run
            gates_commit(gf, sh.gsb[(c + 1) & 1], sh.bsb[(c + 1) & 1], G);
            if (c + 2 < nch) gf = gates_fetch(d, g, beta, b, h, t0 + 2 * kChunk, G);
        }
        commit_wait(&sh.mbar, mph, G.tid);
        {
            float w[16];
            tok16(tmem, G, TW + 32 * G.grp, w);
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = -w[e];
            store_row16(smem + DQ_WN, G.tau, c0, w);
        }
        if (G.tid == 0) bulk_wait_read();  // the previous dq store has read its tile (over D)
        cta_sync_tc();
        if (G.tid == 0) mma_km(tmem + TD, desc_plus(DK, DQ_WN), desc_plus(DM, DQ_S), 1);  // D = U - W S_prev
        commit_wait(&sh.mbar, mph, G.tid);
        {
            float x[16];
            tok16(tmem, G, TD + 32 * G.grp, x);
            store_row16(smem + DQ_DL, G.tau, c0, x);
        }
        cta_sync_tc();
        if (G.tid == 0) {
            mma_kk(tmem + TKK, desc_plus(DK, so), desc_plus(DK, DQ_DL), 0);     // dO D^T
            mma_mm(tmem + TW, desc_plus(DM, DQ_KC), desc_plus(DM, DQ_DL), 0);  // (K o Gam[63])^T D
        }
        commit_wait(&sh.mbar, mph, G.tid);
        {
            float p[16], m[16], y[16];
            tok16x2(tmem, G, TKK + 32 * G.grp, TW + 32 * G.grp, p, y);
            decay16(gs, G.tau, c0, false, m);
#pragma unroll
            for (int e = 0; e < 16; ++e) p[e] *= d.scale * m[e];
            store_row16(smem + DQ_P, G.tau, c0, p);
#pragma unroll
            for (int e = 0; e < 16; ++e) Sr[e] = fmaf(gs.W, Sr[e], y[e]);
            store_row16(smem + DQ_S, G.tau, c0, Sr);
        }
        cta_sync_tc();
        if (G.tid == 0) mma_km(tmem + TQ, desc_plus(DK, DQ_P), desc_plus(DM, sk), 1);  // + P K
        commit_wait(&sh.mbar, mph, G.tid);
        {
            float x[16];
            tok16(tmem, G, TQ + 32 * G.grp, x);
            store_row16(smem + DQ_O, G.tau, c0, x);
        }
        cta_sync_tc();
        if (G.tid == 0) {
            tma_store_3d(mdq, smem_u32(smem + DQ_O), 0, h, b * d.T + t0);
            bulk_commit();
        }
    }
    if (G.tid == 0) bulk_wait_all();
}

// ===========================================================================
// backward prepare, gamma walk (blockIdx.z == 1): the adjoint E of the state
// walked back from the segment end with E = 0 there, chunk by chunk,
//     dD = P^T dO + (K o Gam[63]) E,   dX = T^T dD,
//     E <- scale (Q o gam)^T dO + gam_63 E - (K o gam)^T dX,
// gamma = E at the segment start.  No state is needed.
// Shared memory: two stages of Q|K|dO|T; K o gam, K o Gam[63] (then dD),
// scale Q o gam (then P, then -dX), E (bf16).
// Tensor memory: [0,64) dX; [64,128) Q K^T; [128,192) dD; [192,256) the E
// product.
// ===========================================================================
constexpr uint32_t GA_STAGE = 4 * T8;
constexpr uint32_t GA_KG = 2 * GA_STAGE, GA_KC = GA_KG + T8, GA_QG = GA_KC + T8, GA_E = GA_QG + T8;
constexpr uint32_t GA_P = GA_QG;   // P over scale Q o gam, which dies with its E product
constexpr uint32_t GA_DD = GA_KC;  // dD over K o Gam[63], which dies with its dD product
constexpr uint32_t GA_DX = GA_QG;  // -dX over P, which dies with P^T dO
constexpr size_t kGaSmem = GA_E + T8 + 1024;
constexpr size_t kBwdPrepSmem = kDqSmem > kGaSmem ? kDqSmem : kGaSmem;

// E0 (the segments' dS_out, or NULL for 0) starts the walk; Esave (or NULL)
// receives each chunk's E, the adjoint of the state after the chunk, before the
// chunk updates it; gamma (or NULL) receives E at the segment start.
__device__ __forceinline__ void gamma_walk(const Dims& d, const CUtensorMap* mq, const CUtensorMap* mk,
                                           const CUtensorMap* mo, const CUtensorMap* mf,
                                           const float* __restrict__ g, const float* __restrict__ beta,
                                           const float* __restrict__ E0, float* __restrict__ Esave,
                                           float* __restrict__ gamma, uint8_t* smem, BwdShared& sh,
                                           uint32_t tmem, const Geo& G) {
    constexpr uint32_t TX = 0, TQK = 64, TDD = 128, TE = 192;
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    const int c0 = 32 * G.grp + 16 * G.hi;
    const int64_t cb = chunk_base(d, seg, b, h);

    float Er[16];
    if (E0 != nullptr) {
        load_row16(E0 + sum_off(d, seg, b, h), G.tau, c0, Er);
    } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) Er[e] = 0.f;
    }
    store_row16(smem + GA_E, G.tau, c0, Er);
    auto load = [&](int c, int s) {
        const int row = b * d.T + a0 + c * kChunk;
        const uint32_t bar = smem_u32(&sh.full[s]);
        uint8_t* st = smem + s * GA_STAGE;
        mbar_expect_tx(bar, GA_STAGE);
        tma_load_3d(smem_u32(st), mq, 0, h / d.qdiv, row, bar);
        tma_load_3d(smem_u32(st + T8), mk, 0, h, row, bar);
        tma_load_3d(smem_u32(st + 2 * T8), mo, 0, h, row, bar);
        tma_load_3d(smem_u32(st + 3 * T8), mf, 0, 0, fac_row(cb + c, 0), bar);
    };
    if (G.tid == 0) {
        load(nch - 1, 0);
        if (nch > 1) load(nch - 2, 1);
    }
    const uint32_t sb0 = smem_u32(smem);
    const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, T8, 1024);
    GateFetch gf = gates_fetch(d, g, beta, b, h, a0 + (nch - 1) * kChunk, G);
    gates_commit(gf, sh.gsb[0], sh.bsb[0], G);
    if (nch > 1) gf = gates_fetch(d, g, beta, b, h, a0 + (nch - 2) * kChunk, G);
    uint32_t mph = 0;
    for (int it = 0; it < nch; ++it) {
        const int c = nch - 1 - it, s = it & 1;
        const int t0 = a0 + c * kChunk;
        const uint32_t sq = s * GA_STAGE, sk = sq + T8, so = sq + 2 * T8, st = sq + 3 * T8;
        GateSmem& gs = sh.gsb[it & 1];
        if (Esave != nullptr) save_row16(Esave + (cb + c) * int64_t(kD * kD), G.tau, c0, Er);
        if (G.tid == 0 && it >= 1 && it + 1 < nch) load(c - 1, s ^ 1);  // the previous chunk's products are done
        __syncthreads();
        mbar_wait(smem_u32(&sh.full[s]), (it >> 1) & 1);
        tc_fence_after();
        if (G.tid == 0) mma_kk(tmem + TQK, desc_plus(DK, sq), desc_plus(DK, sk), 0);  // Q K^T
        rows_scaled(smem + sk, smem + GA_KG, gs.win, 1.f, G.tid);      // K o gam
        rows_scaled(smem + sk, smem + GA_KC, gs.wout, 1.f, G.tid);     // K o Gam[63]
        rows_scaled(smem + sq, smem + GA_QG, gs.win, d.scale, G.tid);  // scale Q o gam
        cta_sync_tc();
        if (G.tid == 0) {
            mma_km(tmem + TDD, desc_plus(DK, GA_KC), desc_plus(DM, GA_E), 0);  // (K o Gam[63]) E
            mma_mm(tmem + TE, desc_plus(DM, GA_QG), desc_plus(DM, so), 0);     // (scale Q o gam)^T dO
        }
        if (it + 1 < nch) {  // the next chunk's gate tables, while the products run
            gates_commit(gf, sh.gsb[(it + 1) & 1], sh.bsb[(it + 1) & 1], G);
            if (it + 2 < nch) gf = gates_fetch(d, g, beta, b, h, t0 - 2 * kChunk, G);
        }
        commit_wait(&sh.mbar, mph, G.tid);
        {
            float qk[16], m[16];
            tok16(tmem, G, TQK + 32 * G.grp, qk);
            decay16(gs, G.tau, c0, false, m);
#pragma unroll
            for (int e = 0; e < 16; ++e) qk[e] *= d.scale * m[e];
            store_row16(smem + GA_P, G.tau, c0, qk);
        }
        cta_sync_tc();
        if (G.tid == 0) mma_mm(tmem + TDD, desc_plus(DM, GA_P), desc_plus(DM, so), 1);  // + P^T dO
        commit_wait(&sh.mbar, mph, G.tid);
        {
            float x[16];
            tok16(tmem, G, TDD + 32 * G.grp, x);
            store_row16(smem + GA_DD, G.tau, c0, x);
        }
        cta_sync_tc();
        if (G.tid == 0) mma_mm(tmem + TX, desc_plus(DM, st), desc_plus(DM, GA_DD), 0);  // dX = T^T dD
        commit_wait(&sh.mbar, mph, G.tid);
        {
            float x[16];
            tok16(tmem, G, TX + 32 * G.grp, x);
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = -x[e];
            store_row16(smem + GA_DX, G.tau, c0, x);
        }
        cta_sync_tc();
        if (G.tid == 0) mma_mm(tmem + TE, desc_plus(DM, GA_KG), desc_plus(DM, GA_DX), 1);  // - (K o gam)^T dX
        commit_wait(&sh.mbar, mph, G.tid);
        {
            float x[16];
            tok16(tmem, G, TE + 32 * G.grp, x);
#pragma unroll
            for (int e = 0; e < 16; ++e) Er[e] = fmaf(gs.W, Er[e], x[e]);
            store_row16(smem + GA_E, G.tau, c0, Er);
        }
        cta_sync_tc();
    }
    if (gamma != nullptr) save_row16(gamma + sum_off(d, seg, b, h), G.tau, c0, Er);
}

__global__ void __launch_bounds__(256, 2)
    gdrtc_bwd_prepare_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                             const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                             const __grid_constant__ CUtensorMap mo, const __grid_constant__ CUtensorMap mf,
                             const __grid_constant__ CUtensorMap mdq,
                             const float* __restrict__ g, const float* __restrict__ beta,
                             const float* __restrict__ S_in, float* __restrict__ gamma, float* __restrict__ ws) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ BwdShared sh;
    const Geo G = geo();
    bwd_setup(sh, G, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_slot;
    if (blockIdx.z == 0)
        dq_walk(d, &mk, &mv, &mo, &mf, &mdq, g, beta, S_in, ws, smem, sh, tmem, G);
    else
        gamma_walk(d, &mq, &mk, &mo, &mf, g, beta, nullptr, nullptr, gamma, smem, sh, tmem, G);
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// backward apply, first launch: the adjoint walk of gamma_walk from dS_out,
// saving each chunk's E (the adjoint of the state after the chunk) to the
// workspace.  Two CTAs a SM.
// ===========================================================================
__global__ void __launch_bounds__(256, 2)
    gdrtc_adjoint_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                         const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mo,
                         const __grid_constant__ CUtensorMap mf, const float* __restrict__ g,
                         const float* __restrict__ beta, const float* __restrict__ dS_out,
                         float* __restrict__ Esave) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ BwdShared sh;
    const Geo G = geo();
    bwd_setup(sh, G, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_slot;
    gamma_walk(d, &mq, &mk, &mo, &mf, g, beta, dS_out, Esave, nullptr, smem, sh, tmem, G);
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// backward apply, second launch: the gradients of every chunk at once, one
// CTA per (chunk, row, head), from the chunk's S_prev (saved by the dq walk),
// its E (saved by the adjoint walk) and its factors T and L^{-1} = (I + A)^-1.
// With L = I + A, P = scale mask(Q K^T o Gam), X = V - (K o gam) S_prev,
// D = T X and G = K K^T:
//     dD  = P^T dO + (K o Gam[63]) E,   dZ = L^{-T} dD,   dv = dX = beta o dZ
//     dA  = -strict_lower(dZ D^T),     dG = dA o beta_t o Gam
//     dk  = DW E^T + XG S_prev^T + P2^T Q + (dG + dG^T) K,  with
//           DW = Gam[63] o D, XG = -gam o dX, P2 = scale mask(dO D^T o Gam)
//     dbeta_t = dZ_t . X_t + sum_r dA[t][r] G[t][r] Gam[t][r]
// and the gradient db_t of the running gate sums: the row sum minus the
// column sum of M1 + M2 (M1 = P o (dO D^T), M2 = dA o A), + scale gam_t
// q_t . (S_prev dO_t) + k_t . (XG S_prev^T)_t - w_t, w_t = k_t . (DW E^T)_t,
// and at t = 63 + gam_63 <S_prev, E> + sum_r w_r; dg_u = sum_{t >= u} db_t
// inside the chunk (0 where a sequence starts).
// Two CTAs a SM.  Shared memory (8 KB tiles): Q|K|V|dO|T|L^{-1} (dk staged in
// Q and dv in V once they are dead), and seven work tiles reused by lifetime:
//   W0 S_prev, then dG + dG^T      W1 E, then P2
//   W2 K o gam, then dD            W3 K o Gam[63], then DW
//   W4 P, then dZ                  W5 X, then XG          W6 D
// with the fp32 M1 + M2 over W2|W3 from the third products on and the fp32
// dG over W4|W5 from the fourth (rows of 64 values, the column index
// swizzled by the row so that row and column walks avoid bank conflicts).
// Tensor memory, four 64-column slots: Q K^T, then dD, then dZ, then dZ D^T;
// (K o gam) S_prev, then D, then dO D^T, then XG S_prev^T; dO S_prev^T,
// then the dk product; Q K^T again, then K K^T.
// ===========================================================================
constexpr uint32_t CG_Q = 0, CG_K = T8, CG_V = 2 * T8, CG_O = 3 * T8, CG_T = 4 * T8, CG_L = 5 * T8;
constexpr uint32_t CG_W0 = 6 * T8, CG_W1 = 7 * T8, CG_W2 = 8 * T8, CG_W3 = 9 * T8;
constexpr uint32_t CG_W4 = 10 * T8, CG_W5 = 11 * T8, CG_W6 = 12 * T8;
constexpr size_t kChunkGradSmem = 13 * T8 + 1024;

// element (t, c) of a [64][64] fp32 array of unpadded rows, column swizzled by the row
__device__ __forceinline__ int swz(int t, int c) { return t * kD + (c ^ (t & 31)); }

__global__ void __launch_bounds__(256, 2)
    gdrtc_chunk_grad_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                            const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                            const __grid_constant__ CUtensorMap mo, const __grid_constant__ CUtensorMap mf,
                            const __grid_constant__ CUtensorMap mdk, const __grid_constant__ CUtensorMap mdv,
                            const float* __restrict__ g, const float* __restrict__ beta,
                            const float* __restrict__ Ssave, const float* __restrict__ Esave,
                            float* __restrict__ dg, float* __restrict__ dbeta) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    float* Mm = reinterpret_cast<float*>(smem + CG_W2);  // M1 + M2
    float* dG = reinterpret_cast<float*>(smem + CG_W4);
    __shared__ BwdShared sh;
    constexpr uint32_t SA = 0, SB = 64, SC = 128, SD = 192;
    GateSmem& gs = sh.gsb[0];
    const float* beta_s = sh.bsb[0];

    const Geo G = geo();
    const int b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int t0 = blockIdx.x * kChunk;
    const int seg = t0 / d.L, c = (t0 % d.L) / kChunk;
    const int64_t ci = chunk_base(d, seg, b, h) + c;
    const int c0 = 32 * G.grp + 16 * G.hi;

    // every load of the chunk in flight at once: the TMA tiles (thread 0, as
    // soon as its barrier exists), the fp32 S_prev and E rows, the gates
    if (G.tid == 0) {
        mbar_init(smem_u32(&sh.full[0]), 1);
        mbar_init(smem_u32(&sh.mbar), 1);
        mbar_fence_init();
        const uint32_t bar = smem_u32(&sh.full[0]);
        const int row = b * d.T + t0;
        mbar_expect_tx(bar, 6 * T8);
        tma_load_3d(smem_u32(smem + CG_Q), &mq, 0, h / d.qdiv, row, bar);
        tma_load_3d(smem_u32(smem + CG_K), &mk, 0, h, row, bar);
        tma_load_3d(smem_u32(smem + CG_V), &mv, 0, h, row, bar);
        tma_load_3d(smem_u32(smem + CG_O), &mo, 0, h, row, bar);
        tma_load_3d(smem_u32(smem + CG_T), &mf, 0, 0, fac_row(ci, 0), bar);
        tma_load_3d(smem_u32(smem + CG_L), &mf, 0, 0, fac_row(ci, 1), bar);
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&sh.tmem_slot), 256);
    const GateFetch gf = gates_fetch(d, g, beta, b, h, t0, G);
    float pse = 0.f;  // this thread's part of <S_prev, E>
    {
        float Sr[16], Er[16];
        load_row16(Ssave + ci * int64_t(kD * kD), G.tau, c0, Sr);
        load_row16(Esave + ci * int64_t(kD * kD), G.tau, c0, Er);
#pragma unroll
        for (int e = 0; e < 16; ++e) pse = fmaf(Sr[e], Er[e], pse);
        store_row16(smem + CG_W0, G.tau, c0, Sr);
        store_row16(smem + CG_W1, G.tau, c0, Er);
    }
    gates_commit(gf, gs, sh.bsb[0], G);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_slot;
    mbar_wait(smem_u32(&sh.full[0]), 0);
    tc_fence_after();
    const uint32_t sb0 = smem_u32(smem);
    const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, T8, 1024);
    uint32_t mph = 0;
    if (G.tid == 0) mma_kk(tmem + SA, desc_plus(DK, CG_Q), desc_plus(DK, CG_K), 0);  // Q K^T
    rows_scaled(smem + CG_K, smem + CG_W2, gs.win, 1.f, G.tid);   // K o gam
    rows_scaled(smem + CG_K, smem + CG_W3, gs.wout, 1.f, G.tid);  // K o Gam[63]
    cta_sync_tc();
    if (G.tid == 0) {
        mma_km(tmem + SB, desc_plus(DK, CG_W2), desc_plus(DM, CG_W0), 0);  // (K o gam) S_prev
        mma_kk(tmem + SC, desc_plus(DK, CG_O), desc_plus(DK, CG_W0), 0);   // dO S_prev^T
    }
    commit_wait(&sh.mbar, mph, G.tid);
    float Xr[16], pq = 0.f;  // X (fp32) and this thread's part of q_t . (dO S_prev^T)_t
    {
        float qk[16], tx[16], os[16], qv[16], m[16];
        tok16x2(tmem, G, SA + 32 * G.grp, SB + 32 * G.grp, qk, tx);
        tok16(tmem, G, SC + 32 * G.grp, os);
        tile_row_get16(smem + CG_V, G.tau, c0, Xr);
        tile_row_get16(smem + CG_Q, G.tau, c0, qv);
        decay16(gs, G.tau, c0, false, m);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            qk[e] *= d.scale * m[e];
            Xr[e] -= tx[e];
            pq = fmaf(qv[e], os[e], pq);
        }
        store_row16(smem + CG_W4, G.tau, c0, qk);  // P
        store_row16(smem + CG_W5, G.tau, c0, Xr);  // X
    }
    cta_sync_tc();
    if (G.tid == 0) {
        mma_km(tmem + SA, desc_plus(DK, CG_W3), desc_plus(DM, CG_W1), 0);  // (K o Gam[63]) E
        mma_mm(tmem + SA, desc_plus(DM, CG_W4), desc_plus(DM, CG_O), 1);   //   + P^T dO = dD
        mma_km(tmem + SB, desc_plus(DK, CG_T), desc_plus(DM, CG_W5), 0);   // D = T X
    }
    commit_wait(&sh.mbar, mph, G.tid);
    {
        float x[16], y[16];
        tok16x2(tmem, G, SA + 32 * G.grp, SB + 32 * G.grp, x, y);
        store_row16(smem + CG_W2, G.tau, c0, x);  // dD
        store_row16(smem + CG_W6, G.tau, c0, y);  // D
        const float wo = gs.wout[G.tau];
#pragma unroll
        for (int e = 0; e < 16; ++e) y[e] *= wo;
        store_row16(smem + CG_W3, G.tau, c0, y);  // DW = Gam[63] o D
    }
    cta_sync_tc();
    if (G.tid == 0) {
        mma_mm(tmem + SA, desc_plus(DM, CG_L), desc_plus(DM, CG_W2), 0);   // dZ = L^{-T} dD
        mma_kk(tmem + SB, desc_plus(DK, CG_O), desc_plus(DK, CG_W6), 0);   // dO D^T
        mma_kk(tmem + SC, desc_plus(DK, CG_W3), desc_plus(DK, CG_W1), 0);  // DW E^T (the dk product)
        mma_kk(tmem + SD, desc_plus(DK, CG_Q), desc_plus(DK, CG_K), 0);    // Q K^T again
    }
    commit_wait(&sh.mbar, mph, G.tid);
    float pb = 0.f, pw = 0.f;  // this thread's parts of dbeta_t and of w_t
    {
        float z[16], od[16], qk[16], kw[16], kv[16], m[16], x[16];
        tok16x2(tmem, G, SA + 32 * G.grp, SB + 32 * G.grp, z, od);
        tok16x2(tmem, G, SC + 32 * G.grp, SD + 32 * G.grp, kw, qk);
        tile_row_get16(smem + CG_K, G.tau, c0, kv);
        decay16(gs, G.tau, c0, false, m);
        const float be = beta_s[G.tau], gm = gs.win[G.tau];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            pb = fmaf(z[e], Xr[e], pb);
            pw = fmaf(kv[e], kw[e], pw);
            x[e] = be * z[e];
        }
        store_row16(smem + CG_W4, G.tau, c0, z);  // dZ
        store_row16(smem + CG_V, G.tau, c0, x);   // dv = dX, staged over V
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] *= -gm;
        store_row16(smem + CG_W5, G.tau, c0, x);  // XG = -gam o dX
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float p2 = d.scale * m[e] * od[e];
            Mm[swz(G.tau, c0 + e)] = p2 * qk[e];  // M1 = P o (dO D^T)
            od[e] = p2;
        }
        store_row16(smem + CG_W1, G.tau, c0, od);  // P2 = scale mask(dO D^T o Gam)
    }
    cta_sync_tc();
    if (G.tid == 0) {
        tma_store_3d(&mdv, smem_u32(smem + CG_V), 0, h, b * d.T + t0);
        bulk_commit();
        mma_kk(tmem + SA, desc_plus(DK, CG_W4), desc_plus(DK, CG_W6), 0);  // dZ D^T
        mma_kk(tmem + SB, desc_plus(DK, CG_W5), desc_plus(DK, CG_W0), 0);  // XG S_prev^T
        mma_kk(tmem + SC, desc_plus(DK, CG_W5), desc_plus(DK, CG_W0), 1);  // dk += XG S_prev^T
        mma_mm(tmem + SC, desc_plus(DM, CG_W1), desc_plus(DM, CG_Q), 1);   // dk += P2^T Q
        mma_kk(tmem + SD, desc_plus(DK, CG_K), desc_plus(DK, CG_K), 0);    // K K^T
    }
    commit_wait(&sh.mbar, mph, G.tid);
    float pk = 0.f;  // this thread's part of k_t . (XG S_prev^T)_t
    {
        float da[16], kk[16], xs[16], kv[16], m[16];
        tok16x2(tmem, G, SA + 32 * G.grp, SD + 32 * G.grp, da, kk);
        tok16(tmem, G, SB + 32 * G.grp, xs);
        tile_row_get16(smem + CG_K, G.tau, c0, kv);
        decay16(gs, G.tau, c0, true, m);
        const float be = beta_s[G.tau];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int r = c0 + e;
            const float a = r < G.tau ? -da[e] : 0.f;  // dA
            const float kg = kk[e] * m[e];           // G o Gam, strictly lower within a sequence
            pb = fmaf(a, kg, pb);
            Mm[swz(G.tau, r)] += a * be * kg;        // M2 = dA o A
            dG[swz(G.tau, r)] = a * be * m[e];
            pk = fmaf(kv[e], xs[e], pk);
        }
    }
    __syncthreads();
    {
        float x[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = dG[swz(G.tau, c0 + e)] + dG[swz(c0 + e, G.tau)];
        store_row16(smem + CG_W0, G.tau, c0, x);  // dG + dG^T
        const int t = G.tid >> 2, part = G.tid & 3;
        float rs = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) rs += Mm[swz(t, 16 * part + e)] - Mm[swz(16 * part + e, t)];
        rs += __shfl_xor_sync(kFull, rs, 1);
        rs += __shfl_xor_sync(kFull, rs, 2);
        if (part == 0) sh.dbm[t] = rs;
    }
    cta_sync_tc();
    if (G.tid == 0) mma_km(tmem + SC, desc_plus(DK, CG_W0), desc_plus(DM, CG_K), 1);  // dk += (dG + dG^T) K
    commit_wait(&sh.mbar, mph, G.tid);
    {
        float ka[16];
        tok16(tmem, G, SC + 32 * G.grp, ka);
        store_row16(smem + CG_Q, G.tau, c0, ka);  // dk, staged over Q
        const float gm = gs.win[G.tau];
        float rw = pw;
        float rdb = d.scale * gm * pq + pk - rw;
        rdb += __shfl_xor_sync(kFull, rdb, 16);
        rw += __shfl_xor_sync(kFull, rw, 16);
        pb += __shfl_xor_sync(kFull, pb, 16);
        if (!G.hi) {
            sh.red[0][G.grp][G.tau] = rdb;
            sh.red[1][G.grp][G.tau] = rw;
            sh.red[2][G.grp][G.tau] = pb;
        }
        pse = warp_sum(pse);
        if (G.lane == 0) sh.red_se[G.warp] = pse;
    }
    cta_sync_tc();
    if (G.tid == 0) {
        tma_store_3d(&mdk, smem_u32(smem + CG_Q), 0, h, b * d.T + t0);
        bulk_commit();
    }
    if (G.warp == 0) {  // tokens 2 lane and 2 lane + 1: db, the in-chunk suffix sums, dbeta
        const int u0 = 2 * G.lane, u1 = u0 + 1;
        float db0 = sh.red[0][0][u0] + sh.red[0][1][u0] + sh.dbm[u0];
        float db1 = sh.red[0][0][u1] + sh.red[0][1][u1] + sh.dbm[u1];
        const float wsum = warp_sum(sh.red[1][0][u0] + sh.red[1][1][u0] + sh.red[1][0][u1] + sh.red[1][1][u1]);
        const float se = warp_sum(G.lane < 8 ? sh.red_se[G.lane] : 0.f);
        if (u1 == kChunk - 1) db1 += gs.W * se + wsum;
        float suf = db0 + db1;  // inclusive suffix sum over lanes >= lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float x = __shfl_down_sync(kFull, suf, o);
            if (G.lane + o < 32) suf += x;
        }
        const int ta = t0 + u0, tb = t0 + u1;
        dg[g_off(d, b, ta, h)] = starts_sequence(d.seq_idx, ta) ? 0.f : suf;
        dg[g_off(d, b, tb, h)] = starts_sequence(d.seq_idx, tb) ? 0.f : suf - db0;
        dbeta[g_off(d, b, ta, h)] = sh.red[2][0][u0] + sh.red[2][1][u0];
        dbeta[g_off(d, b, tb, h)] = sh.red[2][0][u1] + sh.red[2][1][u1];
    }
    if (G.tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 256);
}

__global__ void read_flag_kernel(int* out, int clear) {
    *out = g_timeout_flag;
    if (clear) g_timeout_flag = 0;
}

}  // namespace
}  // namespace gdrtc

bool gdrtc_supports(const Dims& d, rm_dtype dt) {
    return !d.vg && dt == RM_BF16 && d.Dk == gdrtc::kD && d.Dv == gdrtc::kD && d.L % tc::kChunk == 0 &&
           d.T >= tc::kChunk;
}

namespace {

// Failures of launch_gdrtc, reported with the step that failed.
rm_status map_fail(const char* what) {
    char msg[192];
    std::snprintf(msg, sizeof(msg), "gated delta rule (tensor cores): no tensor map for %s (CUresult %d)", what,
                  tc::last_map_result());
    return api_fail(RM_ERR_CUDA, msg);
}

rm_status cuda_fail(const char* what) {
    char msg[256];
    std::snprintf(msg, sizeof(msg), "gated delta rule (tensor cores): %s failed: %s", what,
                  cuda_error_text());
    return api_fail(RM_ERR_CUDA, msg);
}

}  // namespace

rm_status launch_gdrtc(GdrOp op, const Dims& d, const GdrPtrs& p, cudaStream_t s) {
    using namespace gdrtc;
    if (!gdrtc_supports(d, RM_BF16)) return RM_ERR_UNSUPPORTED;
    const dim3 grid(d.nseg, d.B * d.H);
    // the factor table follows the saved states (one fp32 state per chunk) in the workspace
    const int64_t nchunks = int64_t(d.B) * d.H * (d.T / kChunk);
    __nv_bfloat16* fac = reinterpret_cast<__nv_bfloat16*>(p.ws + nchunks * kD * kD);
    Dims fd = d;  // the factor table as a [2 nchunks 64][64] bf16 matrix
    fd.B = 1;
    fd.T = int(2 * nchunks * kD);
    CUtensorMap mq, mk, mv, mo, mf, mx, my;
    if (!make_map(&mk, p.k, d, kD)) return map_fail("k");
    if (op != GdrOp::kBackwardPrepare && !make_map(&mv, p.v, d, kD)) return map_fail("v");
    if (op != GdrOp::kPrepare && !make_map(&mq, p.q, d, kD, d.qh)) return map_fail("q");
    if (op != GdrOp::kPrepare && !make_map(&mf, fac, fd, kD, 1)) return map_fail("the factor table");
    if (op == GdrOp::kPrepare) {
        // every chunk's factors at once, then the walk over each segment's chunks
        if (!make_map(&mf, fac, fd, kD, 1)) return map_fail("the factor table");
        auto ff = gdrtc_factor_kernel;
        if (!set_smem(ff, kFactorSmem)) return cuda_fail("shared-memory attribute of the factor kernel");
        ff<<<dim3(d.T / kChunk, d.B * d.H), 256, kFactorSmem, s>>>(d, mk, p.g, p.beta, fac);
        if (!launch_ok()) return cuda_fail("launch of the factor kernel");
        note_launch(1);
        auto fn = gdrtc_prepare_kernel;
        if (!set_smem(fn, kPrepSmem)) return cuda_fail("shared-memory attribute of the prepare kernel");
        fn<<<grid, 256, kPrepSmem, s>>>(d, mk, mv, mf, p.g, p.beta, p.M, p.dS);
    } else if (op == GdrOp::kApply) {
        if (!make_map(&mo, p.o, d, kD)) return map_fail("o");
        auto fn = gdrtc_apply_kernel;
        if (!set_smem(fn, kApplySmem)) return cuda_fail("shared-memory attribute of the apply kernel");
        fn<<<grid, 256, kApplySmem, s>>>(d, mq, mk, mv, mf, mo, p.g, p.beta, p.S_in);
    } else if (op == GdrOp::kBackwardPrepare) {
        // z = 0: the dq walk (which also needs v); z = 1: the gamma walk
        if (!make_map(&mv, p.v, d, kD)) return map_fail("v");
        if (!make_map(&mo, p.dO, d, kD)) return map_fail("dO");
        if (!make_map(&mx, p.dq, d, kD)) return map_fail("dq");
        auto fn = gdrtc_bwd_prepare_kernel;
        if (!set_smem(fn, kBwdPrepSmem)) return cuda_fail("shared-memory attribute of the backward prepare kernel");
        fn<<<dim3(d.nseg, d.B * d.H, 2), 256, kBwdPrepSmem, s>>>(d, mq, mk, mv, mo, mf, mx, p.g, p.beta, p.S_in,
                                                                p.gamma_out, p.ws);
    } else if (op == GdrOp::kBackwardApply) {
        // the adjoint walk saves each chunk's E after the states and the factors,
        // then the gradients of every chunk at once
        if (!make_map(&mo, p.dO, d, kD)) return map_fail("dO");
        if (!make_map(&mx, p.dk, d, kD)) return map_fail("dk");
        if (!make_map(&my, p.dv, d, kD)) return map_fail("dv");
        float* Esave = p.ws + 2 * nchunks * kD * kD;
        auto fa = gdrtc_adjoint_kernel;
        if (!set_smem(fa, kGaSmem)) return cuda_fail("shared-memory attribute of the adjoint kernel");
        fa<<<grid, 256, kGaSmem, s>>>(d, mq, mk, mo, mf, p.g, p.beta, p.dS_out, Esave);
        if (!launch_ok()) return cuda_fail("launch of the adjoint kernel");
        note_launch(1);
        auto fc = gdrtc_chunk_grad_kernel;
        if (!set_smem(fc, kChunkGradSmem)) return cuda_fail("shared-memory attribute of the chunk-gradient kernel");
        fc<<<dim3(d.T / kChunk, d.B * d.H), 256, kChunkGradSmem, s>>>(d, mq, mk, mv, mo, mf, mx, my, p.g, p.beta,
                                                                     p.ws, Esave, p.dg, p.dbeta);
    } else {
        return RM_ERR_INVALID_ARG;
    }
    if (!launch_ok()) return cuda_fail("kernel launch");
    note_launch(1);
    return RM_OK;
}

rm_status gdrtc_read_timeout_flag(int* host_flag, int clear, int* dev_scratch, cudaStream_t s) {
    gdrtc::read_flag_kernel<<<1, 1, 0, s>>>(dev_scratch, clear);
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(1);
    if (cudaMemcpyAsync(host_flag, dev_scratch, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RM_ERR_CUDA;
    return RM_OK;
}

}  // namespace rmcp
