// tc_kernels.cu -- tensor-core path (sm_103a, tcgen05 + TMA) for bf16 storage,
// Dk = 128, Dv in {128, 256}, segment lengths that are multiples of 64.
//
// The segment is walked in chunks of C = 64 tokens.  With b the chunk-local
// running sum of the gates and Gam[t][s] = exp(b_t - b_s) for s <= t in the
// same sequence (0 otherwise), the chunkwise form of the gated recurrence is
//   O       = scale (Gam o Q K^T) V + diag(scale win) Q S_prev
//   S_next  = W S_prev + (diag(wout) K)^T V
// (win = decay from the chunk's incoming state, wout = decay to its last
// state, W = whole-chunk decay), and the backward mirrors it.  Every product
// above is a tcgen05.mma with bf16 operands in 128-byte-swizzled shared memory
// (loaded by TMA) and fp32 accumulators in tensor memory; the fp32 master
// state lives in registers, one state row per thread, and is re-quantised to
// a bf16 shared-memory copy for the next chunk's products.
//
// Kernels (one CTA per (segment, row, head[, value block])):
//   tc_outer_kernel     sum_t w_t x_t y_t^T over a segment: delta_S of
//                       cp_forward_prepare (x = k, y = v, w = decay to the
//                       segment end) and gamma of cp_backward_prepare (x = q,
//                       y = dO, w = scale * decay from the segment start)
//   tc_fwd_apply_kernel the forward sweep from S_in: o
//   tc_dq_kernel        the forward sweep of the backward: dq and, per token,
//                       q.dq minus its same-token term (for the gate gradient)
//   tc_rev_kernel       the reverse sweep from dS_out: dk, dv, dg
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "tc_common.cuh"

namespace rmcp {
namespace tc {

namespace {

constexpr uint32_t kTileBytes = kChunk * 64 * 2;  // one [64 rows][64 cols] bf16 block: 8 KB

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t a = smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}

// Loads a [64 tokens][ncol] bf16 tile (ncol/64 swizzled blocks) with TMA.
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, int col0, int ncol,
                                          int h, int row, uint32_t bar) {
    for (int c = 0; c < ncol; c += 64)
        tma_load_3d(smem_u32(dst + (c / 64) * kTileBytes), map, col0 + c, h, row, bar);
}

// ===========================================================================
// sum_t w_t x_t y_t^T over one segment (x: Dk = 128 columns, y: DV columns)
// ===========================================================================
template <int DV, bool GAMMA>
__global__ void __launch_bounds__(128, 1)
    tc_outer_kernel(const Dims d, const __grid_constant__ CUtensorMap mx,
                    const __grid_constant__ CUtensorMap my, const float* __restrict__ g,
                    float* __restrict__ M, float* __restrict__ out) {
    constexpr int STAGES = DV == 128 ? 3 : 2;
    constexpr uint32_t XBYTES = 2 * kTileBytes;
    constexpr uint32_t YBYTES = (DV / 64) * kTileBytes;
    constexpr uint32_t SBYTES = XBYTES + YBYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ GateSmem gs;
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t done_bar;
    __shared__ uint32_t tmem_slot;

    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&done_bar), 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), DV);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    // gamma walks forward from the segment start, delta_S backward from its end
    auto chunk_of = [&](int it) { return GAMMA ? it : nch - 1 - it; };
    auto issue = [&](int it, int s) {
        const int row = b * d.T + a0 + chunk_of(it) * kChunk;
        const uint32_t bar = smem_u32(&full_bar[s]);
        uint8_t* st = smem + s * SBYTES;
        mbar_expect_tx(bar, SBYTES);
        load_tile(st, &mx, 0, 128, h, row, bar);
        load_tile(st + XBYTES, &my, 0, DV, h, row, bar);
    };
    if (tid == 0)
        for (int it = 0; it < STAGES && it < nch; ++it) issue(it, it);

    float run = 0.f;  // sum of the gates of the chunks already walked
    int seen = 0;     // a sequence starts in the chunks already walked
    GateRegs gr;
    if (warp == 0) gr = gate_load(d, g, b, h, a0 + chunk_of(0) * kChunk, lane);
    for (int it = 0; it < nch; ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (warp == 0) {
            gate_prep(gr, &gs, lane);
            if (it + 1 < nch) gr = gate_load(d, g, b, h, a0 + chunk_of(it + 1) * kChunk, lane);
        }
        mbar_wait(smem_u32(&full_bar[s]), ph);
        __syncthreads();
        {
            // row weight w_t, applied to x_t in place
            const int r = tid >> 1, blk = tid & 1;
            float w;
            if (GAMMA)  // scale * alpha_a ... alpha_t: no start in [a, t]
                w = (!seen && !gs.first && gs.lid[r] == 0) ? d.scale * expf(run + gs.b[r]) : 0.f;
            else        // alpha_{t+1} ... alpha_end: no start in (t, end]
                w = (!seen && gs.lid[r] == gs.lid[kChunk - 1]) ? expf(run + gs.btot - gs.b[r]) : 0.f;
            scale_row128(smem + s * SBYTES + blk * kTileBytes + r * 128, w);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t xa = smem_u32(smem + s * SBYTES), ya = xa + XBYTES;
            constexpr uint32_t idesc = idesc_bf16(128, DV, 1, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, sdesc(xa + k * 2048, kTileBytes, 1024),
                         sdesc(ya + k * 2048, kTileBytes, 1024), idesc, (it > 0 || k > 0) ? 1u : 0u);
            mma_commit(smem_u32(&empty_bar[s]));
            if (it + STAGES < nch) {
                mbar_wait(smem_u32(&empty_bar[s]), ph);
                issue(it + STAGES, s);
            }
        }
        run += gs.btot;
        seen |= gs.any;
        __syncthreads();
    }
    if (tid == 0) mma_commit(smem_u32(&done_bar));
    mbar_wait(smem_u32(&done_bar), 0);
    tc_fence_after();
    float* dst = out + sum_off(d, seg, b, h) + int64_t(warp * 32 + lane) * DV;
#pragma unroll 1
    for (int c = 0; c < DV; c += 32) {
        float v[32];
        tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + c, v);
#pragma unroll
        for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
    if (!GAMMA && tid == 0) M[(int64_t(seg) * d.B + b) * d.H + h] = seen ? 0.f : expf(run);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, DV);
}

// ---------------------------------------------------------------------------
// helpers shared by the sweeps
// ---------------------------------------------------------------------------

// Writes row i (128 fp32 values) of a state as bf16 into a [128][128] tile.
__device__ __forceinline__ void store_state_row(uint8_t* tile, int i, const float* s) {
#pragma unroll
    for (int ch = 0; ch < 16; ++ch)
        *reinterpret_cast<uint4*>(tile + sw_chunk(128, i, ch)) = pack8(s + ch * 8);
}

// Masked score row: out[s] = scale * x[s] * exp(b_t - b_s) for s <= t (s < t if
// strict) in t's sequence, else 0; written as bf16 row t of a [64][64] tile.
// diag receives x[t].
__device__ __forceinline__ void masked_row(uint8_t* tile, const GateSmem& gs, int t, const float* x,
                                           float scale, bool strict, float* diag) {
    const float bt = gs.b[t];
    const int lt = gs.lid[t];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int s = ch * 8 + e;
            const bool keep = (strict ? s < t : s <= t) && gs.lid[s] == lt;
            y[e] = keep ? scale * x[s] * expf(bt - gs.b[s]) : 0.f;
            if (s == t) *diag = x[s];
        }
        *reinterpret_cast<uint4*>(tile + sw_chunk(64, t, ch)) = pack8(y);
    }
}

// 32 values of row t of a [64][128] bf16 tile, columns [col0, col0 + 32)
__device__ __forceinline__ void tile_row_get32(const uint8_t* tile, int t, int col0, float* x) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
        unpack8(*reinterpret_cast<const uint4*>(tile + sw_chunk(64, t, (col0 >> 3) + ch)), x + ch * 8);
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) *reinterpret_cast<uint4*>(dst + i) = pack8(v + i);
}

// ===========================================================================
// forward sweep: o for one (segment, row, head, 128-wide value block)
// ===========================================================================
__global__ void __launch_bounds__(128, 1)
    tc_fwd_apply_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                        const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                        const float* __restrict__ g, const float* __restrict__ S_in,
                        __nv_bfloat16* __restrict__ o) {
    constexpr uint32_t OFF_Q = 0, OFF_K = 2 * kTileBytes, OFF_V = 4 * kTileBytes;
    constexpr uint32_t OFF_P = 6 * kTileBytes, OFF_S = 7 * kTileBytes;  // S tile: 32 KB
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Qs = smem + OFF_Q;
    uint8_t* Ks = smem + OFF_K;
    uint8_t* Vs = smem + OFF_V;
    uint8_t* Ps = smem + OFF_P;
    uint8_t* Sb = smem + OFF_S;
    __shared__ GateSmem gs;
    __shared__ __align__(8) uint64_t full_bar;
    __shared__ __align__(8) uint64_t mma_bar;
    __shared__ uint32_t tmem_slot;

    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H, vb = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tau = warp * 16 + lane;  // token row of the M = 64 tiles (lanes 0-15)
    const bool tok = lane < 16;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    const uint32_t fb = smem_u32(&full_bar), mb = smem_u32(&mma_bar);

    if (tid == 0) {
        mbar_init(fb, 1);
        mbar_init(mb, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 256);

    // fp32 master state row i = tid, columns [128 vb, 128 vb + 128)
    float S[128];
    {
        const float* src = S_in + sum_off(d, seg, b, h) + int64_t(tid) * d.Dv + vb * 128;
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + j);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
        store_state_row(Sb, tid, S);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t t_lane = uint32_t(warp * 32) << 16;
    auto issue = [&](int c) {
        const int row = b * d.T + a0 + c * kChunk;
        mbar_expect_tx(fb, 6 * kTileBytes);
        load_tile(Qs, &mq, 0, 128, h, row, fb);
        load_tile(Ks, &mk, 0, 128, h, row, fb);
        load_tile(Vs, &mv, vb * 128, 128, h, row, fb);
    };
    if (tid == 0) issue(0);
    GateRegs gr;
    if (warp == 0) gr = gate_load(d, g, b, h, a0, lane);
    uint32_t mph = 0;
    for (int c = 0; c < nch; ++c) {
        const int t0 = a0 + c * kChunk;
        if (warp == 0) {
            gate_prep(gr, &gs, lane);
            if (c + 1 < nch) gr = gate_load(d, g, b, h, t0 + kChunk, lane);
        }
        mbar_wait(fb, c & 1);
        __syncthreads();
        const uint32_t qa = smem_u32(Qs), ka = smem_u32(Ks), va = smem_u32(Vs);
        const uint32_t pa = smem_u32(Ps), sa = smem_u32(Sb);
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t off = (s >> 2) * kTileBytes + (s & 3) * 32;
                mma_bf16(tmem, sdesc(qa + off, 16, 1024), sdesc(ka + off, 16, 1024), id1, s > 0);
            }
            mma_commit(mb);
        }
        mbar_wait(mb, mph);
        mph ^= 1;
        tc_fence_after();
        {
            float x[64];
            tmem_ld32(tmem + t_lane, x);
            tmem_ld32(tmem + t_lane + 32, x + 32);
            float dummy;
            if (tok) masked_row(Ps, gs, tau, x, d.scale, false, &dummy);
            const int r = tid >> 1, blk = tid & 1;
            scale_row128(Qs + blk * kTileBytes + r * 128, d.scale * gs.win[r]);
            scale_row128(Ks + blk * kTileBytes + r * 128, gs.wout[r]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_o = idesc_bf16(64, 128, 0, 1);
            constexpr uint32_t id_s = idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // O = P V
                mma_bf16(tmem, sdesc(pa + k * 32, 16, 1024), sdesc(va + k * 2048, kTileBytes, 1024),
                         id_o, k > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)  // O += Q~ S_prev
                mma_bf16(tmem, sdesc(qa + (s >> 2) * kTileBytes + (s & 3) * 32, 16, 1024),
                         sdesc(sa + s * 2048, 2 * kTileBytes, 1024), id_o, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // dS = K~^T V
                mma_bf16(tmem + 128, sdesc(ka + k * 2048, kTileBytes, 1024),
                         sdesc(va + k * 2048, kTileBytes, 1024), id_s, k > 0);
            mma_commit(mb);
        }
        mbar_wait(mb, mph);
        mph ^= 1;
        if (tid == 0 && c + 1 < nch) issue(c + 1);
        tc_fence_after();
        {
            __nv_bfloat16* orow = o + (((int64_t)b * d.T + t0 + tau) * d.H + h) * d.Dv + vb * 128;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(tmem + t_lane + cb * 32, x);
                if (tok) store_bf16x32(orow + cb * 32, x);
            }
            const float W = gs.W;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(tmem + t_lane + 128 + cb * 32, x);
#pragma unroll
                for (int e = 0; e < 32; ++e) S[cb * 32 + e] = fmaf(W, S[cb * 32 + e], x[e]);
            }
            store_state_row(Sb, tid, S);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
    }
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// forward sweep of the backward: dq and q.dq' for one (segment, row, head), Dv = 128
// ===========================================================================
__global__ void __launch_bounds__(128, 1)
    tc_dq_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                 const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                 const __grid_constant__ CUtensorMap mdo, const float* __restrict__ g,
                 const float* __restrict__ S_in, __nv_bfloat16* __restrict__ dq,
                 float* __restrict__ qdq) {
    constexpr uint32_t OFF_Q = 0, OFF_K = 2 * kTileBytes, OFF_V = 4 * kTileBytes;
    constexpr uint32_t OFF_DO = 6 * kTileBytes, OFF_P = 8 * kTileBytes, OFF_S = 9 * kTileBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Qs = smem + OFF_Q;
    uint8_t* Ks = smem + OFF_K;
    uint8_t* Vs = smem + OFF_V;
    uint8_t* Ds = smem + OFF_DO;
    uint8_t* Ps = smem + OFF_P;
    uint8_t* Sb = smem + OFF_S;
    __shared__ GateSmem gs;
    __shared__ __align__(8) uint64_t full_bar;
    __shared__ __align__(8) uint64_t mma_bar;
    __shared__ uint32_t tmem_slot;

    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tau = warp * 16 + lane;
    const bool tok = lane < 16;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    const uint32_t fb = smem_u32(&full_bar), mb = smem_u32(&mma_bar);

    if (tid == 0) {
        mbar_init(fb, 1);
        mbar_init(mb, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 256);
    float S[128];
    {
        const float* src = S_in + sum_off(d, seg, b, h) + int64_t(tid) * 128;
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + j);
            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
        }
        store_state_row(Sb, tid, S);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t t_lane = uint32_t(warp * 32) << 16;
    auto issue = [&](int c) {
        const int row = b * d.T + a0 + c * kChunk;
        mbar_expect_tx(fb, 8 * kTileBytes);
        load_tile(Qs, &mq, 0, 128, h, row, fb);
        load_tile(Ks, &mk, 0, 128, h, row, fb);
        load_tile(Vs, &mv, 0, 128, h, row, fb);
        load_tile(Ds, &mdo, 0, 128, h, row, fb);
    };
    if (tid == 0) issue(0);
    GateRegs gr;
    if (warp == 0) gr = gate_load(d, g, b, h, a0, lane);
    uint32_t mph = 0;
    for (int c = 0; c < nch; ++c) {
        const int t0 = a0 + c * kChunk;
        if (warp == 0) {
            gate_prep(gr, &gs, lane);
            if (c + 1 < nch) gr = gate_load(d, g, b, h, t0 + kChunk, lane);
        }
        mbar_wait(fb, c & 1);
        __syncthreads();
        const uint32_t qa = smem_u32(Qs), ka = smem_u32(Ks), va = smem_u32(Vs), da = smem_u32(Ds);
        const uint32_t pa = smem_u32(Ps), sa = smem_u32(Sb);
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
#pragma unroll
            for (int s = 0; s < 8; ++s) {  // dA = dO V^T
                const uint32_t off = (s >> 2) * kTileBytes + (s & 3) * 32;
                mma_bf16(tmem, sdesc(da + off, 16, 1024), sdesc(va + off, 16, 1024), id1, s > 0);
            }
            mma_commit(mb);
        }
        mbar_wait(mb, mph);
        mph ^= 1;
        tc_fence_after();
        float diag = 0.f;  // dO_t . v_t
        {
            float x[64];
            tmem_ld32(tmem + t_lane, x);
            tmem_ld32(tmem + t_lane + 32, x + 32);
            if (tok) masked_row(Ps, gs, tau, x, d.scale, true, &diag);
            const int r = tid >> 1, blk = tid & 1;
            scale_row128(Ds + blk * kTileBytes + r * 128, d.scale * gs.win[r]);
            scale_row128(Vs + blk * kTileBytes + r * 128, gs.wout[r]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_a = idesc_bf16(64, 128, 0, 1);
            constexpr uint32_t id_b = idesc_bf16(64, 128, 0, 0);
            constexpr uint32_t id_s = idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // dq' = P K  (strictly causal part)
                mma_bf16(tmem, sdesc(pa + k * 32, 16, 1024), sdesc(ka + k * 2048, kTileBytes, 1024),
                         id_a, k > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)  // dq' += dO~ S_prev^T
                mma_bf16(tmem, sdesc(da + (s >> 2) * kTileBytes + (s & 3) * 32, 16, 1024),
                         sdesc(sa + (s >> 2) * 2 * kTileBytes + (s & 3) * 32, 16, 1024), id_b, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // dS = K^T V~
                mma_bf16(tmem + 128, sdesc(ka + k * 2048, kTileBytes, 1024),
                         sdesc(va + k * 2048, kTileBytes, 1024), id_s, k > 0);
            mma_commit(mb);
        }
        mbar_wait(mb, mph);
        mph ^= 1;
        tc_fence_after();
        {
            const int64_t tok_off = ((int64_t)b * d.T + t0 + tau) * d.H + h;
            float a = 0.f;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(tmem + t_lane + cb * 32, x);
                if (tok) {
                    float qv[32], kv[32];
                    tile_row_get32(Qs, tau, cb * 32, qv);
                    tile_row_get32(Ks, tau, cb * 32, kv);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        a = fmaf(qv[e], x[e], a);
                        x[e] = fmaf(d.scale * diag, kv[e], x[e]);
                    }
                    store_bf16x32(dq + tok_off * 128 + cb * 32, x);
                }
            }
            if (tok) qdq[tok_off] = a;
            const float W = gs.W;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(tmem + t_lane + 128 + cb * 32, x);
#pragma unroll
                for (int e = 0; e < 32; ++e) S[cb * 32 + e] = fmaf(W, S[cb * 32 + e], x[e]);
            }
            store_state_row(Sb, tid, S);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && c + 1 < nch) issue(c + 1);
    }
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ===========================================================================
// reverse sweep of the backward: dk, dv, dg for one (segment, row, head), Dv = 128
// ===========================================================================
__global__ void __launch_bounds__(128, 1)
    tc_rev_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                  const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                  const __grid_constant__ CUtensorMap mdo, const float* __restrict__ g,
                  const float* __restrict__ S_in, const float* __restrict__ dS_out,
                  const float* __restrict__ qdq, __nv_bfloat16* __restrict__ dk,
                  __nv_bfloat16* __restrict__ dv, float* __restrict__ dg) {
    constexpr uint32_t STAGE = 8 * kTileBytes;  // Q | K | V | dO
    constexpr uint32_t OFF_QT = 2 * STAGE, OFF_KT = OFF_QT + 2 * kTileBytes;
    constexpr uint32_t OFF_PA = OFF_KT + 2 * kTileBytes, OFF_PD = OFF_PA + kTileBytes;
    constexpr uint32_t OFF_E = OFF_PD + kTileBytes;  // E tile: 32 KB
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Qt = smem + OFF_QT;
    uint8_t* Kt = smem + OFF_KT;
    uint8_t* PA = smem + OFF_PA;
    uint8_t* PD = smem + OFF_PD;
    uint8_t* Eb = smem + OFF_E;
    __shared__ GateSmem gs;
    __shared__ __align__(8) uint64_t full_bar[2];
    __shared__ __align__(8) uint64_t mma_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ float cbuf[kChunk];
    __shared__ float dgbuf[kChunk];
    __shared__ float red[4];
    __shared__ float carry_s;

    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tau = warp * 16 + lane;
    const bool tok = lane < 16;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    const uint32_t mb = smem_u32(&mma_bar);

    if (tid == 0) {
        mbar_init(smem_u32(&full_bar[0]), 1);
        mbar_init(smem_u32(&full_bar[1]), 1);
        mbar_init(mb, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
    // E (adjoint arriving at the last state of the current chunk) starts as dS_out;
    // ext = <S_out, dS_out> with S_out read as S_in[seg+1]
    float E[128];
    float ext = 0.f;
    {
        const float* src = dS_out + sum_off(d, seg, b, h) + int64_t(tid) * 128;
        const float* so = seg + 1 < d.nseg ? S_in + sum_off(d, seg + 1, b, h) + int64_t(tid) * 128 : nullptr;
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + j);
            E[j] = x.x; E[j + 1] = x.y; E[j + 2] = x.z; E[j + 3] = x.w;
            if (so) {
                const float4 y = *reinterpret_cast<const float4*>(so + j);
                ext = fmaf(x.x, y.x, ext); ext = fmaf(x.y, y.y, ext);
                ext = fmaf(x.z, y.z, ext); ext = fmaf(x.w, y.w, ext);
            }
        }
        store_state_row(Eb, tid, E);
        ext = warp_sum(ext);
        if (lane == 0) red[warp] = ext;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) carry_s = red[0] + red[1] + red[2] + red[3];
    const uint32_t tmem = tmem_slot;
    const uint32_t t_lane = uint32_t(warp * 32) << 16;
    auto stage_ptr = [&](int s) { return smem + s * STAGE; };
    auto issue = [&](int it, int s) {
        const int c = nch - 1 - it;
        const int row = b * d.T + a0 + c * kChunk;
        const uint32_t bar = smem_u32(&full_bar[s]);
        uint8_t* st = stage_ptr(s);
        mbar_expect_tx(bar, STAGE);
        load_tile(st, &mq, 0, 128, h, row, bar);
        load_tile(st + 2 * kTileBytes, &mk, 0, 128, h, row, bar);
        load_tile(st + 4 * kTileBytes, &mv, 0, 128, h, row, bar);
        load_tile(st + 6 * kTileBytes, &mdo, 0, 128, h, row, bar);
    };
    if (tid == 0) {
        issue(0, 0);
        if (nch > 1) issue(1, 1);
    }
    GateRegs gr;
    if (warp == 0) gr = gate_load(d, g, b, h, a0 + (nch - 1) * kChunk, lane);
    uint32_t mph = 0;
    for (int it = 0; it < nch; ++it) {
        const int c = nch - 1 - it;
        const int t0 = a0 + c * kChunk;
        const int s = it & 1;
        uint8_t* Qs = stage_ptr(s);
        uint8_t* Ks = Qs + 2 * kTileBytes;
        uint8_t* Vs = Qs + 4 * kTileBytes;
        uint8_t* Ds = Qs + 6 * kTileBytes;
        if (warp == 0) {
            gate_prep(gr, &gs, lane);
            if (it + 1 < nch) gr = gate_load(d, g, b, h, t0 - kChunk, lane);
        }
        mbar_wait(smem_u32(&full_bar[s]), (it >> 1) & 1);
        __syncthreads();
        const uint32_t qa = smem_u32(Qs), ka = smem_u32(Ks), va = smem_u32(Vs), da = smem_u32(Ds);
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                mma_bf16(tmem, sdesc(qa + off, 16, 1024), sdesc(ka + off, 16, 1024), id1, k > 0);
                mma_bf16(tmem + 64, sdesc(da + off, 16, 1024), sdesc(va + off, 16, 1024), id1, k > 0);
            }
            mma_commit(mb);
        }
        mbar_wait(mb, mph);
        mph ^= 1;
        tc_fence_after();
        float diag = 0.f;
        {
            float x[64];
            tmem_ld32(tmem + t_lane, x);
            tmem_ld32(tmem + t_lane + 32, x + 32);
            float dummy;
            if (tok) masked_row(PA, gs, tau, x, d.scale, false, &dummy);
            tmem_ld32(tmem + t_lane + 64, x);
            tmem_ld32(tmem + t_lane + 96, x + 32);
            if (tok) masked_row(PD, gs, tau, x, d.scale, true, &diag);
            const int r = tid >> 1, blk = tid & 1;
            const uint32_t ro = blk * kTileBytes + r * 128;
            // Q~ = scale win Q and K~ = wout K into their own tiles; V~ = wout V in place
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                float xq[8], xk[8];
                unpack8(*reinterpret_cast<const uint4*>(Qs + ro + ch * 16), xq);
                unpack8(*reinterpret_cast<const uint4*>(Ks + ro + ch * 16), xk);
                const float wq = d.scale * gs.win[r], wk = gs.wout[r];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    xq[e] *= wq;
                    xk[e] *= wk;
                }
                *reinterpret_cast<uint4*>(Qt + ro + ch * 16) = pack8(xq);
                *reinterpret_cast<uint4*>(Kt + ro + ch * 16) = pack8(xk);
            }
            scale_row128(Vs + ro, gs.wout[r]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t pa = smem_u32(PA), pd = smem_u32(PD), ea = smem_u32(Eb);
            const uint32_t qta = smem_u32(Qt), kta = smem_u32(Kt);
            constexpr uint32_t id_mm = idesc_bf16(64, 128, 1, 1);
            constexpr uint32_t id_kk = idesc_bf16(64, 128, 0, 0);
            constexpr uint32_t id_km = idesc_bf16(64, 128, 0, 1);
            constexpr uint32_t id_e = idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // dk' = PdA^T Q
                mma_bf16(tmem + 128, sdesc(pd + k * 2048, kTileBytes, 1024),
                         sdesc(qa + k * 2048, kTileBytes, 1024), id_mm, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k)  // dk' += V~ E^T
                mma_bf16(tmem + 128, sdesc(va + (k >> 2) * kTileBytes + (k & 3) * 32, 16, 1024),
                         sdesc(ea + (k >> 2) * 2 * kTileBytes + (k & 3) * 32, 16, 1024), id_kk, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // dv = PA^T dO
                mma_bf16(tmem + 256, sdesc(pa + k * 2048, kTileBytes, 1024),
                         sdesc(da + k * 2048, kTileBytes, 1024), id_mm, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k)  // dv += K~ E
                mma_bf16(tmem + 256, sdesc(kta + (k >> 2) * kTileBytes + (k & 3) * 32, 16, 1024),
                         sdesc(ea + k * 2048, 2 * kTileBytes, 1024), id_km, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // dE = Q~^T dO
                mma_bf16(tmem + 384, sdesc(qta + k * 2048, kTileBytes, 1024),
                         sdesc(da + k * 2048, kTileBytes, 1024), id_e, k > 0);
            mma_commit(mb);
        }
        mbar_wait(mb, mph);
        mph ^= 1;
        tc_fence_after();
        {
            const int64_t tok_off = ((int64_t)b * d.T + t0 + tau) * d.H + h;
            float bk = 0.f;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(tmem + t_lane + 128 + cb * 32, x);
                if (tok) {
                    float qv[32], kv[32];
                    tile_row_get32(Qs, tau, cb * 32, qv);
                    tile_row_get32(Ks, tau, cb * 32, kv);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        bk = fmaf(kv[e], x[e], bk);
                        x[e] = fmaf(d.scale * diag, qv[e], x[e]);
                    }
                    store_bf16x32(dk + tok_off * 128 + cb * 32, x);
                }
            }
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(tmem + t_lane + 256 + cb * 32, x);
                if (tok) store_bf16x32(dv + tok_off * 128 + cb * 32, x);
            }
            if (tok) cbuf[tau] = qdq[tok_off] - bk;
            const float W = gs.W;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
                float x[32];
                tmem_ld32(tmem + t_lane + 384 + cb * 32, x);
#pragma unroll
                for (int e = 0; e < 32; ++e) E[cb * 32 + e] = fmaf(W, E[cb * 32 + e], x[e]);
            }
            store_state_row(Eb, tid, E);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            // gate gradient of the chunk, newest token first: sums restart where
            // a sequence starts; tokens that start one get exactly 0
            float run = carry_s;
            for (int t = kChunk - 1; t >= 0; --t) {
                if (t + 1 < kChunk && gs.lid[t + 1] != gs.lid[t]) run = 0.f;
                run += cbuf[t];
                const bool start = t == 0 ? gs.first != 0 : gs.lid[t] != gs.lid[t - 1];
                dgbuf[t] = start ? 0.f : run;
            }
            carry_s = gs.first ? 0.f : run;
            if (it + 2 < nch) issue(it + 2, s);
        }
        __syncthreads();
        if (tid < kChunk) dg[((int64_t)b * d.T + t0 + tid) * d.H + h] = dgbuf[tid];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Failure-detection self test: waits on an mbarrier that nothing arrives on,
// with the given bound, so that the timeout path and its host-side status can
// be exercised without faulting or hanging the device.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    mbar_fence_init();
    mbar_wait(b, 0, limit_ns);
}

__global__ void read_flag_kernel(int* out, int clear) {
    *out = g_timeout_flag;
    if (clear) g_timeout_flag = 0;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [B*T rows][H][D] bf16 viewed as a 3-D tensor; boxes of 64 tokens x 64 columns.
bool make_map(CUtensorMap* m, const void* base, const Dims& d, int D) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(d.H), cuuint64_t(d.B) * cuuint64_t(d.T)};
    cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(d.H) * D * 2};
    cuuint32_t box[3] = {64, 1, uint32_t(kChunk)};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K>
bool set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) ==
           cudaSuccess;
}

constexpr size_t kOuterSmem = 96 * 1024 + 1024;
constexpr size_t kFwdSmem = 11 * kTileBytes + 1024;   // Q K V P (7 tiles) + S (4 tiles)
constexpr size_t kDqSmem = 13 * kTileBytes + 1024;    // Q K V dO P (9) + S (4)
constexpr size_t kRevSmem = 26 * kTileBytes + 1024;   // 2 stages x 8 + Q~ K~ (4) + PA PdA (2) + E (4)

}  // namespace

}  // namespace tc

rm_status tc_selftest_wait(uint32_t limit_us, cudaStream_t s) {
    tc::selftest_wait_kernel<<<1, 1, 0, s>>>(uint64_t(limit_us) * 1000ull);
    if (cudaGetLastError() != cudaSuccess) return RM_ERR_CUDA;
    note_launch(1);
    return RM_OK;
}

rm_status tc_read_timeout_flag(int* host_flag, int clear, int* dev_scratch, cudaStream_t s) {
    tc::read_flag_kernel<<<1, 1, 0, s>>>(dev_scratch, clear);
    if (cudaGetLastError() != cudaSuccess) return RM_ERR_CUDA;
    note_launch(1);
    if (cudaMemcpyAsync(host_flag, dev_scratch, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RM_ERR_CUDA;
    return RM_OK;
}

bool tc_supports(const Dims& d, rm_dtype dt) {
    return dt == RM_BF16 && d.Dk == 128 && (d.Dv == 128 || d.Dv == 256) && d.L % tc::kChunk == 0 &&
           d.T >= tc::kChunk;
}

bool tc_supports_op(Op op, const Dims& d, rm_dtype dt) {
    if (!tc_supports(d, dt)) return false;
    if (op == Op::kBackwardPrepare || op == Op::kBackwardApply) return d.Dv == 128;
    return true;
}

rm_status launch_tc(Op op, const Dims& d, const Ptrs& p, cudaStream_t s) {
    using namespace tc;
    if (!tc_supports_op(op, d, RM_BF16)) return RM_ERR_UNSUPPORTED;
    const dim3 grid(d.nseg, d.B * d.H);
    CUtensorMap mq, mk, mv, mdo;
    switch (op) {
        case Op::kForwardPrepare: {
            if (!make_map(&mk, p.k, d, 128) || !make_map(&mv, p.v, d, d.Dv)) return RM_ERR_CUDA;
            if (d.Dv == 128) {
                auto fn = tc_outer_kernel<128, false>;
                if (!set_smem(fn, kOuterSmem)) return RM_ERR_CUDA;
                fn<<<grid, 128, kOuterSmem, s>>>(d, mk, mv, p.g, p.M, p.sum_out);
            } else {
                auto fn = tc_outer_kernel<256, false>;
                if (!set_smem(fn, kOuterSmem)) return RM_ERR_CUDA;
                fn<<<grid, 128, kOuterSmem, s>>>(d, mk, mv, p.g, p.M, p.sum_out);
            }
            if (cudaGetLastError() != cudaSuccess) return RM_ERR_CUDA;
            note_launch(1);
            return RM_OK;
        }
        case Op::kForwardApply: {
            if (!make_map(&mq, p.q, d, 128) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, d.Dv))
                return RM_ERR_CUDA;
            if (!set_smem(tc_fwd_apply_kernel, kFwdSmem)) return RM_ERR_CUDA;
            tc_fwd_apply_kernel<<<dim3(d.nseg, d.B * d.H, d.Dv / 128), 128, kFwdSmem, s>>>(
                d, mq, mk, mv, p.g, p.S_in, static_cast<__nv_bfloat16*>(p.out0));
            if (cudaGetLastError() != cudaSuccess) return RM_ERR_CUDA;
            note_launch(1);
            return RM_OK;
        }
        case Op::kBackwardPrepare: {
            if (!make_map(&mq, p.q, d, 128) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, 128) || !make_map(&mdo, p.dO, d, 128))
                return RM_ERR_CUDA;
            auto fo = tc_outer_kernel<128, true>;
            if (!set_smem(fo, kOuterSmem) || !set_smem(tc_dq_kernel, kDqSmem)) return RM_ERR_CUDA;
            fo<<<grid, 128, kOuterSmem, s>>>(d, mq, mdo, p.g, nullptr, p.sum_out);
            if (cudaGetLastError() != cudaSuccess) return RM_ERR_CUDA;
            tc_dq_kernel<<<grid, 128, kDqSmem, s>>>(d, mq, mk, mv, mdo, p.g, p.S_in,
                                                    static_cast<__nv_bfloat16*>(p.out0), p.ws_f32);
            if (cudaGetLastError() != cudaSuccess) return RM_ERR_CUDA;
            note_launch(2);
            return RM_OK;
        }
        case Op::kBackwardApply: {
            if (!make_map(&mq, p.q, d, 128) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, 128) || !make_map(&mdo, p.dO, d, 128))
                return RM_ERR_CUDA;
            if (!set_smem(tc_rev_kernel, kRevSmem)) return RM_ERR_CUDA;
            tc_rev_kernel<<<grid, 128, kRevSmem, s>>>(
                d, mq, mk, mv, mdo, p.g, p.S_in, p.dS_out, p.ws_f32,
                static_cast<__nv_bfloat16*>(p.out0), static_cast<__nv_bfloat16*>(p.out1), p.dg);
            if (cudaGetLastError() != cudaSuccess) return RM_ERR_CUDA;
            note_launch(1);
            return RM_OK;
        }
    }
    return RM_ERR_INVALID_ARG;
}

}  // namespace rmcp
