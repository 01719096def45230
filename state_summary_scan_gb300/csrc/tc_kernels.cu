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
// (loaded by TMA) and fp32 accumulators in tensor memory.  The fp32 master
// state of a sweep lives in tensor memory in the forward sweep and in the
// Dv = 256 dq and reverse sweeps, and in registers (one state row per pair of
// threads) in the Dv = 128 dq and reverse sweeps; either way it is
// re-quantised to a bf16 shared-memory copy for the next chunk's products.
//
// Kernels (one CTA per (segment, row, head[, value block])):
//   tc_outer2_kernel    (Dv = 128, barrier-paced) and tc_outer_kernel (Dv = 256):
//                       sum_t w_t x_t y_t^T over a segment: delta_S of
//                       cp_forward_prepare (x = k, y = v, w = decay to the
//                       segment end) and gamma of cp_backward_prepare (x = q,
//                       y = dO, w = scale * decay from the segment start)
//   tc_fwd2_kernel      the forward sweep from S_in: o
//   tc_dqg128_kernel    the forward sweep of the backward for Dv = 128: dq,
//                       per token q.dq minus its same-token term (for the
//                       gate gradient), and gamma
//   tc_dq256_kernel     the same for Dv = 256, without gamma
//   tc_rev128_kernel    the reverse sweep from dS_out: dk, dv, dg (Dv = 128)
//   tc_rev256_kernel    the same for Dv = 256
#include <cudaTypedefs.h>

#include <mutex>

#include "tc_tiles.cuh"

namespace rmcp {
namespace tc {

namespace {

constexpr int kRev3Threads = kThreads + 96;       // + an MMA warp, a gate/scan warp and a copy warp

// S[e] = W S[e] + acc[srow][64 grp + e] for e < 64, accumulator at column col;
// then row srow's columns [64 grp, +64) are written as bf16 into a [128][128] tile.
__device__ __forceinline__ void state_update(uint32_t tmem, const Geo& g, int col, float W, float* S,
                                             uint8_t* tile);

// Writes columns [64 grp, +64) of state row i as bf16 into a [128][128] tile.

__device__ __forceinline__ void state_update(uint32_t tmem, const Geo& g, int col, float W, float* S,
                                             uint8_t* tile) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        float y[32];
        tmem_ld32(tmem + g.tl + col + 64 * g.grp + 32 * hf, y);
#pragma unroll
        for (int e = 0; e < 32; ++e) S[32 * hf + e] = fmaf(W, S[32 * hf + e], y[e]);
    }
    store_state_half(tile, g.srow, g.grp, S);
}

// S[e] = W (S[e] + acc[srow][64 grp + e]): the update of a factored chunk
__device__ __forceinline__ void state_update_scaled(uint32_t tmem, const Geo& g, int col, float W, float* S,
                                                    uint8_t* tile) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        float y[32];
        tmem_ld32(tmem + g.tl + col + 64 * g.grp + 32 * hf, y);
#pragma unroll
        for (int e = 0; e < 32; ++e) S[32 * hf + e] = W * (S[32 * hf + e] + y[e]);
    }
    store_state_half(tile, g.srow, g.grp, S);
}

// S[64 hh + e] = W S[64 hh + e] + acc[srow][col + 64 grp + e] (accumulator
// holding state columns [128 hh, +128) at column col), with both 32-column
// tensor-memory loads in flight together; writes those columns as bf16.
__device__ __forceinline__ void state_update_half2(uint32_t tmem, const Geo& g, int col, int hh, float W,
                                                   float* S, uint8_t* tile) {
    uint32_t r0[32], r1[32];
    tmem_ld32_nowait(tmem + g.tl + col + 64 * g.grp, r0);
    tmem_ld32_nowait(tmem + g.tl + col + 64 * g.grp + 32, r1);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        S[64 * hh + e] = fmaf(W, S[64 * hh + e], __uint_as_float(r0[e]));
        S[64 * hh + 32 + e] = fmaf(W, S[64 * hh + 32 + e], __uint_as_float(r1[e]));
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(tile + sw_chunk(128, g.srow, 16 * hh + 8 * g.grp + c)) =
            pack8(S + 64 * hh + c * 8);
}

// State rows of width DV split over the two column groups: thread (srow, grp)
// owns columns 128 h + 64 grp + [0, 64) for h < DV / 128, stored in S[64 h + e].
template <int DV>
__device__ __forceinline__ void load_state_rows(const float* __restrict__ src, const Geo& g, float* S,
                                                uint8_t* tile) {
#pragma unroll
    for (int hh = 0; hh < DV / 128; ++hh) {
        const float* p = src + int64_t(g.srow) * DV + 128 * hh + 64 * g.grp;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
            const float4 x = *reinterpret_cast<const float4*>(p + j);
            S[64 * hh + j] = x.x; S[64 * hh + j + 1] = x.y; S[64 * hh + j + 2] = x.z; S[64 * hh + j + 3] = x.w;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(tile + sw_chunk(128, g.srow, 16 * hh + 8 * g.grp + c)) =
                pack8(S + 64 * hh + c * 8);
    }
}

// dst row r = w[r] * src row r for the [64][128] tile (dst may equal src)
__device__ __forceinline__ void scale_tile(const uint8_t* src, uint8_t* dst, const float* w, float mul,
                                           int tid) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        int r;
        const uint32_t off = scale_off(tid, k, &r);
        scale_chunk(src + off, dst + off, mul * w[r]);
    }
}

// Decay mask for this thread's 16 columns c0..c0+15 of row tau:
// gam[e] = exp(b_tau - b_s) if s <= tau (s < tau when strict) in tau's sequence.
// When the chunk's decays are moderate the exponential factors through the
// chunk end, exp(b_tau - b_63) exp(b_63 - b_s), and costs one multiply.
__device__ __forceinline__ void decay_row16(const GateSmem& gs, int tau, int c0, bool strict, float* gam) {
    const int lt = gs.lid[tau];
    float bb[16], en[16];
    int ll[16];
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
        const float4 x = *reinterpret_cast<const float4*>(&gs.b[c0 + e]);
        const float4 y = *reinterpret_cast<const float4*>(&gs.en[c0 + e]);
        const int4 z = *reinterpret_cast<const int4*>(&gs.lid[c0 + e]);
        bb[e] = x.x; bb[e + 1] = x.y; bb[e + 2] = x.z; bb[e + 3] = x.w;
        en[e] = y.x; en[e + 1] = y.y; en[e + 2] = y.z; en[e + 3] = y.w;
        ll[e] = z.x; ll[e + 1] = z.y; ll[e + 2] = z.z; ll[e + 3] = z.w;
    }
    if (gs.fast) {
        const float et = gs.ep[tau];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int s = c0 + e;
            const bool keep = (strict ? s < tau : s <= tau) && ll[e] == lt;
            gam[e] = keep ? et * en[e] : 0.f;
        }
    } else {
        const float bt = gs.b[tau];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int s = c0 + e;
            const bool keep = (strict ? s < tau : s <= tau) && ll[e] == lt;
            gam[e] = keep ? __expf(bt - bb[e]) : 0.f;
        }
    }
}

// ===========================================================================
// sum_t w_t x_t y_t^T over one segment (x: Dk = 128 columns, y: DV columns)
// ===========================================================================
template <int DV, bool GAMMA>
__global__ void __launch_bounds__(kThreads, 1)
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

    const Geo G = geo();
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        mbar_init(smem_u32(&done_bar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), DV);
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
        load_tile(st, &mx, 0, 128, GAMMA ? h / d.qdiv : h, row, bar);  // x = q or k
        load_tile(st + XBYTES, &my, 0, DV, h, row, bar);
    };
    if (G.tid == 0)
        for (int it = 0; it < STAGES && it < nch; ++it) issue(it, it);

    float run = 0.f;  // sum of the gates of the chunks already walked
    int seen = 0;     // a sequence starts in the chunks already walked
    GateRegs gr;
    if (G.warp == 0) gr = gate_load(d, g, b, h, a0 + chunk_of(0) * kChunk, G.lane);
    for (int it = 0; it < nch; ++it) {
        const int s = it % STAGES;
        if (G.warp == 0) {
            gate_prep(gr, &gs, G.lane);
            if (it + 1 < nch) gr = gate_load(d, g, b, h, a0 + chunk_of(it + 1) * kChunk, G.lane);
        }
        mbar_wait(smem_u32(&full_bar[s]), (it / STAGES) & 1);
        __syncthreads();
        {
            // row weight w_t, applied to x_t in place
            uint8_t* xt = smem + s * SBYTES;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                int r;
                const uint32_t off = scale_off(G.tid, k, &r);
                float w;
                if (GAMMA)  // scale * alpha_a ... alpha_t: no start in [a, t]
                    w = (!seen && !gs.first && gs.lid[r] == 0) ? d.scale * expf(run + gs.b[r]) : 0.f;
                else        // alpha_{t+1} ... alpha_end: no start in (t, end]
                    w = (!seen && gs.lid[r] == gs.lid[kChunk - 1]) ? expf(run + gs.btot - gs.b[r]) : 0.f;
                scale_chunk(xt + off, xt + off, w);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (G.tid == 0) {
            tc_fence_after();
            const uint32_t xa = smem_u32(smem + s * SBYTES), ya = xa + XBYTES;
            constexpr uint32_t idesc = idesc_bf16(128, DV, 1, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, sdesc(xa + k * 2048, kTileBytes, 1024),
                         sdesc(ya + k * 2048, kTileBytes, 1024), idesc, (it > 0 || k > 0) ? 1u : 0u);
            mma_commit(smem_u32(&empty_bar[s]));
            // refill the stage the previous chunk's products have finished with
            const int prev = it - 1;
            if (prev >= 0 && prev + STAGES < nch) {
                const int ps = prev % STAGES;
                mbar_wait(smem_u32(&empty_bar[ps]), (prev / STAGES) & 1);
                issue(prev + STAGES, ps);
            }
        }
        run += gs.btot;
        seen |= gs.any;
        __syncthreads();
    }
    if (G.tid == 0) mma_commit(smem_u32(&done_bar));
    mbar_wait(smem_u32(&done_bar), 0);
    tc_fence_after();
    {
        float* dst = out + sum_off(d, seg, b, h) + int64_t(G.srow) * DV;
#pragma unroll 1
        for (int c = G.grp * (DV / 2); c < (G.grp + 1) * (DV / 2); c += 64) {
            float v[64];
            state_cols64(tmem, G, c - 64 * G.grp, v);
#pragma unroll
            for (int i = 0; i < 64; i += 4)
                *reinterpret_cast<float4*>(dst + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
    }
    if (!GAMMA && G.tid == 0) M[(int64_t(seg) * d.B + b) * d.H + h] = seen ? 0.f : expf(run);
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, DV);
}

// dst = f * src for a [64][128] bf16 tile (uniform factor), 4 chunks per thread
__device__ __forceinline__ void copy_scaled_tile(const uint8_t* src, uint8_t* dst, float f, int tid) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        int r;
        const uint32_t off = scale_off(tid, k, &r);
        scale_chunk(src + off, dst + off, f);
    }
}

// ===========================================================================
// forward sweep of the backward for Dv = 128: dq, q.dq' per token and
// gamma = sum_t (alpha_a..alpha_t) scale q_t dO_t^T, accumulated in tensor
// memory over the segment (one pass over q, k, v, dO).  Warp-specialised and
// paced by mbarriers:
//   warps 0-7 (epilogues), per chunk:
//     E1  score mask P; K^ in place (factored) or dO~, V~ (general) -> p_ready
//         gamma's copy of Q with its row weights                   -> q_ready
//     E2  dq rows into their staging tile, q.dq' partials           -> dq_staged
//         state update into the S tile                              -> in_dead, a_ready
//   warp 8 (one thread): dq' = P K + dO S^T (in factored chunks dO S^T is
//     issued as soon as the previous state is in the S tile), dS = K^T V,
//     gamma += Qh^T dO, then the next chunk's dO V^T.
//   warp 9: per-token q.dq' sums and the gate tables two chunks ahead.
//   warp 10 (one thread): TMA loads (a stage is refilled once its chunk is
//     done) and the dq stores.
// Every barrier completes once per chunk (parity-indexed pairs once per two
// chunks), and each waiter is paced so that it cannot fall a phase behind.
// ===========================================================================
__global__ void __launch_bounds__(kRev3Threads, 1)
    tc_dqg128_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                     const __grid_constant__ CUtensorMap mdo, const __grid_constant__ CUtensorMap mdq,
                     const float* __restrict__ g, const float* __restrict__ S_in,
                     float* __restrict__ gamma, float* __restrict__ qdq) {
    constexpr uint32_t STAGE = 8 * kTileBytes;  // Q | K | V | dO
    constexpr uint32_t OFF_P = 2 * STAGE, OFF_S = OFF_P + kTileBytes;  // S tile 32 KB
    constexpr uint32_t OFF_QH = OFF_S + 4 * kTileBytes;               // gamma's Q
    constexpr uint32_t OFF_DQ = OFF_QH + 2 * kTileBytes;              // dq staging
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Ps = smem + OFF_P;
    uint8_t* Sb = smem + OFF_S;
    uint8_t* Qh = smem + OFF_QH;
    uint8_t* DQ = smem + OFF_DQ;
    __shared__ GateSmem gsb[2];
    __shared__ __align__(8) uint64_t full_bar[2];
    __shared__ __align__(8) uint64_t score_bar, dq_done, st_done;          // tensor-core commits
    __shared__ __align__(8) uint64_t p_ready, q_ready, dq_staged, in_dead;  // epilogue -> warps 8, 10
    __shared__ __align__(8) uint64_t a_ready[2];     // epilogue -> warps 8, 9: chunk done
    __shared__ __align__(8) uint64_t a_done[2];      // warp 9 -> epilogue: q.dq' partials read
    __shared__ __align__(8) uint64_t gate_ready[2];  // warp 9 -> epilogue, warp 8: gate tables
    __shared__ __align__(8) uint64_t stg_free;       // warp 10 -> epilogue: dq store has read DQ
    __shared__ uint32_t tmem_slot;
    __shared__ float diag_s[2][kChunk];  // dO_t . v_t by chunk parity
    __shared__ float apart[2][2][kChunk];  // [chunk parity][column group][token]

    const Geo G = geo();
    const bool epi = G.warp < 8;
    const bool ctl = G.warp == 8;
    const bool gat = G.warp == 9;
    const bool cpy = G.warp == 10;
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&a_ready[i]), 8);
            mbar_init(smem_u32(&a_done[i]), 1);
            mbar_init(smem_u32(&gate_ready[i]), 1);
        }
        mbar_init(smem_u32(&score_bar), 1);
        mbar_init(smem_u32(&dq_done), 1);
        mbar_init(smem_u32(&st_done), 1);
        mbar_init(smem_u32(&p_ready), 8);
        mbar_init(smem_u32(&q_ready), 8);
        mbar_init(smem_u32(&dq_staged), 8);
        mbar_init(smem_u32(&in_dead), 8);
        mbar_init(smem_u32(&stg_free), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
    float S[64];
    GateRegs gr;
    if (epi) {
        load_state_rows<128>(S_in + sum_off(d, seg, b, h), G, S, Sb);
    } else if (gat) {  // gate tables of the first two chunks; registers for the third
        gr = gate_load(d, g, b, h, a0, G.lane);
        gate_prep(gr, &gsb[0], G.lane);
        if (nch > 1) {
            gr = gate_load(d, g, b, h, a0 + kChunk, G.lane);
            gate_prep(gr, &gsb[1], G.lane);
        }
        if (nch > 2) gr = gate_load(d, g, b, h, a0 + 2 * kChunk, G.lane);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (ctl) {
        if (G.lane == 0) {
            // operand descriptors as offsets from those of the start of
            // shared memory (K-major; MN-major with blocks one tile apart)
            const uint32_t sb0 = smem_u32(smem);
            const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, kTileBytes, 1024);
            const uint64_t pa = desc_plus(DK, OFF_P), sa = desc_plus(DK, OFF_S), qh = desc_plus(DM, OFF_QH);
            constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
            constexpr uint32_t id_a = idesc_bf16(64, 128, 0, 1);
            constexpr uint32_t id_b = idesc_bf16(64, 128, 0, 0);
            constexpr uint32_t id_s = idesc_bf16(128, 128, 1, 1);
            auto issue_scores = [&](int s) {  // dA = dO V^T of the chunk in stage s
                const uint64_t v = desc_plus(DK, s * STAGE + 4 * kTileBytes);
                const uint64_t o = desc_plus(DK, s * STAGE + 6 * kTileBytes);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                    mma_bf16(tmem, desc_plus(o, off), desc_plus(v, off), id1, k > 0);
                }
                mma_commit(smem_u32(&score_bar));
            };
            // dq' (+)= dO S_prev^T: first in a factored chunk, after P K otherwise
            auto issue_state_side = [&](int s, bool first) {
                const uint64_t o = desc_plus(DK, s * STAGE + 6 * kTileBytes);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16(tmem + 128, desc_plus(o, (k >> 2) * kTileBytes + (k & 3) * 32),
                             desc_plus(sa, (k >> 2) * 2 * kTileBytes + (k & 3) * 32), id_b,
                             (first && k == 0) ? 0u : 1u);
            };
            mbar_wait(smem_u32(&full_bar[0]), 0);
            tc_fence_after();
            issue_scores(0);
            bool fact = gsb[0].fact != 0;
            if (fact) issue_state_side(0, true);
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                const uint32_t ph = c & 1;
                const uint64_t km = desc_plus(DM, s * STAGE + 2 * kTileBytes);
                const uint64_t vm = desc_plus(DM, s * STAGE + 4 * kTileBytes);
                const uint64_t om = desc_plus(DM, s * STAGE + 6 * kTileBytes);
                mbar_wait(smem_u32(&p_ready), ph);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // dq' (+)= P K  (strictly causal part)
                    mma_bf16(tmem + 128, desc_plus(pa, k * 32), desc_plus(km, k * 2048), id_a,
                             (fact || k > 0) ? 1u : 0u);
                if (!fact) issue_state_side(s, false);
                mma_commit(smem_u32(&dq_done));
#pragma unroll
                for (int k = 0; k < 4; ++k)  // dS = K^T V  (K^ or V~ carry the weights)
                    mma_bf16(tmem + 256, desc_plus(km, k * 2048), desc_plus(vm, k * 2048), id_s, k > 0);
                mbar_wait(smem_u32(&q_ready), ph);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // gamma += Qh^T dO
                    mma_bf16(tmem + 384, desc_plus(qh, k * 2048), desc_plus(om, k * 2048), id_s,
                             (c > 0 || k > 0) ? 1u : 0u);
                mma_commit(smem_u32(&st_done));
                if (c + 1 < nch) {
                    mbar_wait(smem_u32(&full_bar[s ^ 1]), ((c + 1) >> 1) & 1);
                    tc_fence_after();
                    issue_scores(s ^ 1);
                    // the state after this chunk is in the S tile once its
                    // epilogue is done: the next factored chunk's dO S^T
                    mbar_wait(smem_u32(&a_ready[s]), (c >> 1) & 1);
                    if (c + 1 >= 2) mbar_wait(smem_u32(&gate_ready[s ^ 1]), ((c - 1) >> 1) & 1);
                    fact = gsb[s ^ 1].fact != 0;
                    if (fact) {
                        tc_fence_after();
                        issue_state_side(s ^ 1, true);
                    }
                }
            }
        }
    } else if (cpy) {
        if (G.lane == 0) {
            auto issue = [&](int c, int s) {
                const int row = b * d.T + a0 + c * kChunk;
                const uint32_t bar = smem_u32(&full_bar[s]);
                uint8_t* st = smem + s * STAGE;
                mbar_expect_tx(bar, STAGE);
                load_tile(st, &mq, 0, 128, h / d.qdiv, row, bar);
                load_tile(st + 2 * kTileBytes, &mk, 0, 128, h, row, bar);
                load_tile(st + 4 * kTileBytes, &mv, 0, 128, h, row, bar);
                load_tile(st + 6 * kTileBytes, &mdo, 0, 128, h, row, bar);
            };
            issue(0, 0);
            if (nch > 1) issue(1, 1);
            for (int c = 0; c < nch; ++c) {
                const uint32_t ph = c & 1;
                const int row = b * d.T + a0 + c * kChunk;
                mbar_wait(smem_u32(&dq_staged), ph);
                tma_store_3d(&mdq, smem_u32(DQ), 0, h, row);
                tma_store_3d(&mdq, smem_u32(DQ + kTileBytes), 64, h, row);
                bulk_commit();
                mbar_wait(smem_u32(&in_dead), ph);  // every read of the chunk's stage is done
                if (c + 2 < nch) issue(c + 2, c & 1);
                bulk_wait_read();
                mbar_arrive(smem_u32(&stg_free));
            }
            bulk_wait_all();
        }
    } else if (gat) {
        for (int c = 0; c < nch; ++c) {
            const int p = c & 1;
            const int t0 = a0 + c * kChunk;
            mbar_wait(smem_u32(&a_ready[p]), (c >> 1) & 1);
            const int64_t base = ((int64_t)b * d.T + t0) * d.H + h;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = 2 * G.lane + u;
                qdq[base + int64_t(t) * d.H] = apart[p][0][t] + apart[p][1][t];
            }
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&a_done[p]));
            if (c + 2 < nch) {  // the tables of chunk c + 2 replace this chunk's
                gate_prep(gr, &gsb[p], G.lane);
                if (c + 3 < nch) gr = gate_load(d, g, b, h, t0 + 3 * kChunk, G.lane);
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&gate_ready[p]));
            }
        }
    } else {  // epilogue warps
        uint32_t sph = 0, dph = 0, tph = 0;
        float P = 1.f;  // alpha product from the segment start to this chunk's start
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            const int p = c & 1;
            const GateSmem& gs = gsb[p];
            uint8_t* Qs = smem + s * STAGE;
            uint8_t* Ks = Qs + 2 * kTileBytes;
            uint8_t* Vs = Qs + 4 * kTileBytes;
            uint8_t* Ds = Qs + 6 * kTileBytes;
            // ---- E1
            if (c >= 2) mbar_wait(smem_u32(&gate_ready[p]), ((c - 2) >> 1) & 1);
            mbar_wait(smem_u32(&score_bar), sph);
            sph ^= 1;
            mbar_wait(smem_u32(&full_bar[s]), (c >> 1) & 1);
            tc_fence_after();
            // Factored chunks (no sequence start, moderate decays) take the
            // decays as K^ = exp(-b) K:  dq'_t = scale win_t (sum_{s<t}
            // (dO_t . v_s) k^_s + dO_t S_prev^T),  dS = W K^T^ V,  and gamma's
            // row weights go on its copy of Q; dO and V stay unscaled.
            const bool fact = gs.fact != 0;
            {
                float x[16];
                tok16(tmem, G, 32 * G.grp, x);
                const int c0 = 32 * G.grp + 16 * G.hi;
                if (fact) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (c0 + e == G.tau) diag_s[p][G.tau] = x[e];  // dO_t . v_t
                        x[e] = c0 + e < G.tau ? x[e] : 0.f;
                    }
                } else {
                    float gam[16];
                    decay_row16(gs, G.tau, c0, true, gam);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (c0 + e == G.tau) diag_s[p][G.tau] = x[e];  // dO_t . v_t
                        x[e] *= d.scale * gam[e];
                    }
                }
                store_row16(Ps, G.tau, c0, x);
            }
            if (fact) {
                scale_tile(Ks, Ks, gs.nb, 1.f, G.tid);  // K^
            } else {
                scale_tile(Ds, Ds, gs.win, d.scale, G.tid);  // dO~
                scale_tile(Vs, Vs, gs.wout, 1.f, G.tid);     // V~
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&p_ready));
            if (fact)
                scale_tile(Qs, Qh, gs.win, P * d.scale, G.tid);  // gamma's A operand
            else
                copy_scaled_tile(Qs, Qh, P, G.tid);
            fence_async_smem();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&q_ready));
            P *= gs.W;
            // ---- E2: dq rows
            mbar_wait(smem_u32(&dq_done), dph);
            dph ^= 1;
            if (c >= 1) mbar_wait(smem_u32(&stg_free), (c - 1) & 1);      // DQ tile free
            if (c >= 2) mbar_wait(smem_u32(&a_done[p]), ((c - 2) >> 1) & 1);  // apart[p] free
            // diag_s of this chunk comes from the other warp of the quadrant:
            // every epilogue warp arrived on p_ready after writing it
            mbar_wait(smem_u32(&p_ready), c & 1);
            tc_fence_after();
            {
                // factored: dq' = scale win_t acc and k_t = win_t k^_t
                const float wr = fact ? d.scale * gs.win[G.tau] : 1.f;
                const float cd = d.scale * diag_s[p][G.tau] * (fact ? gs.win[G.tau] : 1.f);
                float a = 0.f;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float x[16], qv[16], kv[16];
                    const int col = 64 * G.grp + 32 * k;
                    const int cc = col + 16 * G.hi;
                    tok16(tmem, G, 128 + col, x);
                    tile_row_get16(Qs, G.tau, cc, qv);
                    tile_row_get16(Ks, G.tau, cc, kv);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        x[e] *= wr;
                        a = fmaf(qv[e], x[e], a);
                        x[e] = fmaf(cd, kv[e], x[e]);
                    }
                    store_row16(DQ, G.tau, cc, x);
                }
                a += __shfl_xor_sync(kFull, a, 16);
                if (!G.hi) apart[p][G.grp][G.tau] = a;
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&dq_staged));
            // ---- E2: state update
            mbar_wait(smem_u32(&st_done), tph);
            tph ^= 1;
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&in_dead));  // the stage's last reader is done
            tc_fence_after();
            if (fact)
                state_update_scaled(tmem, G, 256, gs.W, S, Sb);
            else
                state_update(tmem, G, 256, gs.W, S, Sb);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&a_ready[p]));
        }
        // gamma rows (every product has completed: the last st_done wait)
        tc_fence_after();
        float* dst = gamma + sum_off(d, seg, b, h) + int64_t(G.srow) * 128 + 64 * G.grp;
        float v[64];
        state_cols64(tmem, G, 384, v);
#pragma unroll
        for (int i = 0; i < 64; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 512);
}

// Gate gradient of one chunk (warp 0): reverse running sums of q.dq' - k.dk'
// that restart where a sequence starts, plus the carry from later chunks for
// the sequence open at the chunk's end.  Lane l holds tokens 63 - 2l and
// 62 - 2l; a segmented warp scan runs over the lanes in that (reverse) order.
// bp[grp][t] are the two column groups' partials of k.dk'; qd0/qd1 are q.dq'
// of the lane's tokens; dgc points at dg of the chunk's token 0 (stride H).
// Returns the carry into the previous chunk.
__device__ __forceinline__ float dg_scan(const GateSmem& gs, const float (*bp)[kChunk], float qd0,
                                         float qd1, float carry, int lane, float* dgc, int H) {
    const int tA = 63 - 2 * lane, tB = 62 - 2 * lane;
    const float cA = qd0 - (bp[0][tA] + bp[1][tA]);
    const float cB = qd1 - (bp[0][tB] + bp[1][tB]);
    const bool hA = tA < 63 && gs.lid[tA + 1] != gs.lid[tA];  // t + 1 starts a sequence
    const bool hB = gs.lid[tB + 1] != gs.lid[tB];
    float v = hB ? cB : cA + cB;  // pair summary
    bool f = hA || hB;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float vp = __shfl_up_sync(kFull, v, o);
        const bool fp = __shfl_up_sync(kFull, f, o);
        if (lane >= o) {
            if (!f) v += vp;
            f = f || fp;
        }
    }
    float vx = __shfl_up_sync(kFull, v, 1);
    bool fx = __shfl_up_sync(kFull, f, 1);
    if (lane == 0) {
        vx = 0.f;
        fx = false;
    }
    const float X = fx ? vx : carry + vx;
    const float sA = cA + (hA ? 0.f : X);
    const float sB = cB + (hB ? 0.f : sA);
    const bool stA = gs.lid[tA] != gs.lid[tA - 1];  // tA >= 1
    const bool stB = tB == 0 ? gs.first != 0 : gs.lid[tB] != gs.lid[tB - 1];
    dgc[int64_t(tA) * H] = stA ? 0.f : sA;
    dgc[int64_t(tB) * H] = stB ? 0.f : sB;
    const float last = __shfl_sync(kFull, sB, 31);  // value at token 0
    return gs.first ? 0.f : last;
}

// ===========================================================================
// reverse sweep for Dv = 128, warp-specialised, paced by mbarriers instead of
// CTA-wide barriers so that the tensor products overlap the epilogues:
//   warps 0-7 (epilogues), per chunk:
//     E1  score masks PA, PdA; V~ in place          -> pv_ready
//         K~ and Q~ copies                            -> kq_ready
//     E2  dk rows (staged in the dead V~ tile)        -> dk_staged
//         dv rows (in the K~ tile), adjoint E          -> dv_staged, b_ready
//   warp 8 (one thread) issues the tensor products: dk' = PdA^T Q + V~ E^T
//     at pv_ready, dv = PA^T dO + K~ E and dE = Q~^T dO at kq_ready, then
//     the next chunk's scores.  Chunks without sequence starts and with
//     moderate decays are "factored": their weights sit in the score masks,
//     on dO and on the output rows, so V E^T and K E need no epilogue work:
//     V E^T is issued as soon as the adjoint of the chunk after is in place,
//     K E right behind the chunk's dk' products.
//   warp 10 (one thread): the bulk stores of dk and dv, the refill of the
//     stage with the chunk after next as its tiles die (Q, K, dO at
//     in_dead, V once the dk store has read it), and stg_free once the dv
//     store has read the K~ tile.
//   warp 9: the gate-gradient scan of a chunk once its b' rows are in, and
//     the gate tables two chunks ahead.
// Every barrier completes once per chunk (or once per two chunks for the
// parity-indexed pairs) and each waiter is paced so that it cannot fall a
// full phase behind.
// ===========================================================================

__global__ void __launch_bounds__(kRev3Threads, 1)
    tc_rev128_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                     const __grid_constant__ CUtensorMap mdo, const __grid_constant__ CUtensorMap mdk,
                     const __grid_constant__ CUtensorMap mdv, const float* __restrict__ g,
                     const float* __restrict__ S_in, const float* __restrict__ dS_out,
                     const float* __restrict__ qdq, float* __restrict__ dg) {
    constexpr int DV = 128;
    constexpr uint32_t STAGE = 8 * kTileBytes;  // Q | K | V | dO
    constexpr uint32_t OFF_QT = 2 * STAGE, OFF_KT = OFF_QT + 2 * kTileBytes;
    constexpr uint32_t OFF_PA = OFF_KT + 2 * kTileBytes, OFF_PD = OFF_PA + kTileBytes;
    constexpr uint32_t OFF_E = OFF_PD + kTileBytes;  // E tile [128][128]
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Qt = smem + OFF_QT;
    uint8_t* Kt = smem + OFF_KT;
    uint8_t* PA = smem + OFF_PA;
    uint8_t* PD = smem + OFF_PD;
    uint8_t* Eb = smem + OFF_E;
    __shared__ GateSmem gsb[2];  // gate tables by chunk parity
    __shared__ __align__(8) uint64_t full_bar[2];
    __shared__ __align__(8) uint64_t score_bar, dk_done, dve_done;  // tensor-core commits
    __shared__ __align__(8) uint64_t pv_ready, kq_ready, dk_staged, dv_staged;  // epilogue -> warp 8
    __shared__ __align__(8) uint64_t b_ready[2];     // epilogue -> warp 9, by chunk parity
    __shared__ __align__(8) uint64_t scan_done[2];   // warp 9 -> epilogue (b' rows free)
    __shared__ __align__(8) uint64_t gate_ready[2];  // warp 9 -> epilogue (gate tables)
    __shared__ __align__(8) uint64_t stg_free;       // copy warp -> epilogue: dv store has read K~
    __shared__ __align__(8) uint64_t in_dead;        // epilogue -> copy warp: Q, K, dO of the stage dead
    __shared__ uint32_t tmem_slot;
    __shared__ float diag_s[2][kChunk];  // dO_t . v_t by chunk parity
    __shared__ float bpart[2][2][kChunk];  // [chunk parity][column group][token]
    __shared__ float red[8];

    const Geo G = geo();
    const bool epi = G.warp < 8;
    const bool ctl = G.warp == 8;
    const bool scn = G.warp == 9;
    const bool tma = G.warp == 10;
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&b_ready[i]), 8);
            mbar_init(smem_u32(&scan_done[i]), 1);
            mbar_init(smem_u32(&gate_ready[i]), 1);
        }
        mbar_init(smem_u32(&score_bar), 1);
        mbar_init(smem_u32(&dk_done), 1);
        mbar_init(smem_u32(&dve_done), 1);
        mbar_init(smem_u32(&pv_ready), 8);
        mbar_init(smem_u32(&kq_ready), 8);
        mbar_init(smem_u32(&dk_staged), 8);
        mbar_init(smem_u32(&dv_staged), 8);
        mbar_init(smem_u32(&stg_free), 1);
        mbar_init(smem_u32(&in_dead), 8);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
    auto issue = [&](int it, int s) {
        const int row = b * d.T + a0 + (nch - 1 - it) * kChunk;
        const uint32_t bar = smem_u32(&full_bar[s]);
        uint8_t* st = smem + s * STAGE;
        mbar_expect_tx(bar, STAGE);
        load_tile(st, &mq, 0, 128, h / d.qdiv, row, bar);
        load_tile(st + 2 * kTileBytes, &mk, 0, 128, h, row, bar);
        load_tile(st + 4 * kTileBytes, &mv, 0, DV, h, row, bar);
        load_tile(st + 6 * kTileBytes, &mdo, 0, DV, h, row, bar);
    };
    // E (adjoint arriving at the last state of the current chunk) starts as
    // dS_out; ext = <S_out, dS_out> with S_out read as S_in[seg+1]
    float E[DV / 2];
    GateRegs gr;
    if (epi) {
        load_state_rows<DV>(dS_out + sum_off(d, seg, b, h), G, E, Eb);
        float ext = 0.f;
        if (seg + 1 < d.nseg) {
            const float* so = S_in + sum_off(d, seg + 1, b, h) + int64_t(G.srow) * DV + 64 * G.grp;
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
                const float4 y = *reinterpret_cast<const float4*>(so + j);
                ext = fmaf(E[j], y.x, ext);
                ext = fmaf(E[j + 1], y.y, ext);
                ext = fmaf(E[j + 2], y.z, ext);
                ext = fmaf(E[j + 3], y.w, ext);
            }
        }
        ext = warp_sum(ext);
        if (G.lane == 0) red[G.warp] = ext;
    } else if (scn) {  // gate tables of the first two chunks; registers for the third
        gr = gate_load(d, g, b, h, a0 + (nch - 1) * kChunk, G.lane);
        gate_prep(gr, &gsb[0], G.lane);
        if (nch > 1) {
            gr = gate_load(d, g, b, h, a0 + (nch - 2) * kChunk, G.lane);
            gate_prep(gr, &gsb[1], G.lane);
        }
        if (nch > 2) gr = gate_load(d, g, b, h, a0 + (nch - 3) * kChunk, G.lane);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (ctl) {
        if (G.lane == 0) {
            // Descriptors of the shared-memory operands: the three layouts
            // (K-major, MN-major with 64-column blocks one or two tiles apart)
            // at the start of shared memory; every operand is an offset from it.
            const uint32_t sb0 = smem_u32(smem);
            const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, kTileBytes, 1024);
            const uint64_t DM2 = sdesc(sb0, 2 * kTileBytes, 1024);
            // score products A = Q K^T and dA = dO V^T of the chunk in stage s
            auto issue_scores = [&](int s) {
                const uint64_t q = desc_plus(DK, s * STAGE), kk = desc_plus(q, 2 * kTileBytes);
                const uint64_t v = desc_plus(q, 4 * kTileBytes), o = desc_plus(q, 6 * kTileBytes);
                constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                    mma_bf16(tmem, desc_plus(q, off), desc_plus(kk, off), id1, k > 0);
                    mma_bf16(tmem + 64, desc_plus(o, off), desc_plus(v, off), id1, k > 0);
                }
                mma_commit(smem_u32(&score_bar));
            };
            const uint64_t pa = desc_plus(DM, OFF_PA), pd = desc_plus(DM, OFF_PD);
            const uint64_t ek = desc_plus(DK, OFF_E), em = desc_plus(DM2, OFF_E);
            const uint64_t qt = desc_plus(DM, OFF_QT), kt = desc_plus(DK, OFF_KT);
            constexpr uint32_t id_mm = idesc_bf16(64, 128, 1, 1);
            constexpr uint32_t id_kk = idesc_bf16(64, 128, 0, 0);
            constexpr uint32_t id_km = idesc_bf16(64, 128, 0, 1);
            constexpr uint32_t id_e = idesc_bf16(128, 128, 1, 1);
            // The E-side products of a factored chunk, dk' = V E^T and
            // dv = K E, use unscaled tiles and the adjoint of the chunk after
            // it: they are issued as soon as that adjoint is in the E tile,
            // ahead of the chunk's score masks.
            auto issue_ve = [&](int s, uint32_t acc) {  // dk' (+)= V~ E^T
                const uint64_t v = desc_plus(DK, s * STAGE + 4 * kTileBytes);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                    mma_bf16(tmem + 128, desc_plus(v, off), desc_plus(ek, 2 * off - (k & 3) * 32), id_kk,
                             (acc || k > 0) ? 1u : 0u);
                }
            };
            auto issue_ke = [&](uint64_t kk, uint32_t acc) {  // dv (+)= K E
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16(tmem + 256, desc_plus(kk, (k >> 2) * kTileBytes + (k & 3) * 32),
                             desc_plus(em, k * 2048), id_km, (acc || k > 0) ? 1u : 0u);
            };
            mbar_wait(smem_u32(&full_bar[0]), 0);
            tc_fence_after();
            issue_scores(0);
            // factored chunks keep K, Q and V unscaled (the weights sit in the
            // score masks, on dO and on the output rows)
            bool fact = gsb[0].fact != 0;
            if (fact) issue_ve(0, 0);
            for (int it = 0; it < nch; ++it) {
                const int s = it & 1;
                const uint32_t ph = it & 1;
                const uint64_t q = desc_plus(DM, s * STAGE), o = desc_plus(DM, s * STAGE + 6 * kTileBytes);
                mbar_wait(smem_u32(&pv_ready), ph);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // dk' (+)= PdA^T Q
                    mma_bf16(tmem + 128, desc_plus(pd, k * 2048), desc_plus(q, k * 2048), id_mm,
                             (fact || k > 0) ? 1u : 0u);
                if (!fact) issue_ve(s, 1);  // dk' += V~ E^T
                mma_commit(smem_u32(&dk_done));
                if (fact) issue_ke(desc_plus(DK, s * STAGE + 2 * kTileBytes), 0);  // behind the dk' products
                mbar_wait(smem_u32(&kq_ready), ph);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // dv (+)= PA^T dO
                    mma_bf16(tmem + 256, desc_plus(pa, k * 2048), desc_plus(o, k * 2048), id_mm,
                             (fact || k > 0) ? 1u : 0u);
                if (!fact) issue_ke(kt, 1);  // dv += K~ E
                const uint64_t qx = fact ? q : qt;
#pragma unroll
                for (int k = 0; k < 4; ++k)  // dE = Q~^T dO
                    mma_bf16(tmem + 384, desc_plus(qx, k * 2048), desc_plus(o, k * 2048), id_e, k > 0);
                mma_commit(smem_u32(&dve_done));
                // the next chunk's scores: their accumulator columns were read
                // before pv_ready, their tiles were loaded into the other stage
                if (it + 1 < nch) {
                    mbar_wait(smem_u32(&full_bar[s ^ 1]), ((it + 1) >> 1) & 1);
                    tc_fence_after();
                    issue_scores(s ^ 1);
                }
                // the adjoint of this chunk is in the E tile and its dk', dv
                // rows have been read: the next chunk's E-side products
                if (it + 1 < nch) {
                    mbar_wait(smem_u32(&dv_staged), ph);
                    if (it + 1 >= 2) mbar_wait(smem_u32(&gate_ready[(it + 1) & 1]), ((it - 1) >> 1) & 1);
                    fact = gsb[(it + 1) & 1].fact != 0;
                    if (fact) {
                        tc_fence_after();
                        issue_ve(s ^ 1, 0);
                    }
                }
            }
        }
    } else if (tma) {
        if (G.lane == 0) {
            issue(0, 0);
            if (nch > 1) issue(1, 1);
            const uint32_t kta = smem_u32(Kt);
            for (int it = 0; it < nch; ++it) {
                const int s = it & 1;
                const uint32_t ph = it & 1;
                const int row = b * d.T + a0 + (nch - 1 - it) * kChunk;
                uint8_t* st = smem + s * STAGE;
                uint8_t* Vs = st + 4 * kTileBytes;
                mbar_wait(smem_u32(&dk_staged), ph);
                tma_store_3d(&mdk, smem_u32(Vs), 0, h, row);
                tma_store_3d(&mdk, smem_u32(Vs + kTileBytes), 64, h, row);
                bulk_commit();
                // in_dead: the output products are done and the dk rows have
                // read Q and K, so Q, K and dO of this stage are dead; V is
                // dead once the dk store has read it
                const int nrow = b * d.T + a0 + (nch - 3 - it) * kChunk;
                const uint32_t fb = smem_u32(&full_bar[s]);
                mbar_wait(smem_u32(&in_dead), ph);
                if (it + 2 < nch) {
                    mbar_expect_tx(fb, STAGE);
                    load_tile(st, &mq, 0, 128, h / d.qdiv, nrow, fb);
                    load_tile(st + 2 * kTileBytes, &mk, 0, 128, h, nrow, fb);
                    load_tile(st + 6 * kTileBytes, &mdo, 0, DV, h, nrow, fb);
                }
                mbar_wait(smem_u32(&dv_staged), ph);
                tma_store_3d(&mdv, kta, 0, h, row);
                tma_store_3d(&mdv, kta + kTileBytes, 64, h, row);
                bulk_commit();
                if (it + 2 < nch) {
                    bulk_wait_read1();  // the dk store has read V's tile
                    load_tile(Vs, &mv, 0, DV, h, nrow, fb);
                }
                bulk_wait_read();  // the dv store has read the K~ tile
                mbar_arrive(smem_u32(&stg_free));
            }
            bulk_wait_all();
        }
    } else if (scn) {
        float carry = 0.f;  // gate-gradient sum carried from later chunks
#pragma unroll
        for (int w = 0; w < 8; ++w) carry += red[w];
        for (int it = 0; it < nch; ++it) {
            const int c = nch - 1 - it;
            const int t0 = a0 + c * kChunk;
            const int p = it & 1;
            const float qd0 = __ldg(qdq + ((int64_t)b * d.T + t0 + 63 - 2 * G.lane) * d.H + h);
            const float qd1 = __ldg(qdq + ((int64_t)b * d.T + t0 + 62 - 2 * G.lane) * d.H + h);
            mbar_wait(smem_u32(&b_ready[p]), (it >> 1) & 1);
            carry = dg_scan(gsb[p], bpart[p], qd0, qd1, carry, G.lane,
                            dg + ((int64_t)b * d.T + t0) * d.H + h, d.H);
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&scan_done[p]));
            if (it + 2 < nch) {  // the tables of chunk it + 2 replace this chunk's
                gate_prep(gr, &gsb[p], G.lane);
                if (it + 3 < nch) gr = gate_load(d, g, b, h, t0 - 3 * kChunk, G.lane);
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&gate_ready[p]));
            }
        }
    } else {  // epilogue warps
        uint32_t sph = 0, kph = 0, vph = 0;
        for (int it = 0; it < nch; ++it) {
            const int s = it & 1;
            const int p = it & 1;
            const GateSmem& gs = gsb[p];
            uint8_t* Qs = smem + s * STAGE;
            uint8_t* Ks = Qs + 2 * kTileBytes;
            uint8_t* Vs = Qs + 4 * kTileBytes;
            uint8_t* Ds = Qs + 6 * kTileBytes;
            // ---- E1
            if (it >= 2) mbar_wait(smem_u32(&gate_ready[p]), ((it - 2) >> 1) & 1);
            mbar_wait(smem_u32(&score_bar), sph);
            sph ^= 1;
            mbar_wait(smem_u32(&full_bar[s]), (it >> 1) & 1);  // its tiles, for the scaling
            tc_fence_after();
            const bool fact = gs.fact != 0;
            if (fact) {
                // dk = wout (Pd^T Q + V E^T) with Pd = scale ep_t dA (s < t);
                // dv = wout (Pa^T dO~ + K E) with Pa = e^(-b_63) A (s <= t);
                // dE = Q^T dO~, dO~ = scale win dO
                float xa[16], xd[16];
                tok16x2(tmem, G, 32 * G.grp, 64 + 32 * G.grp, xa, xd);
                const int c0 = 32 * G.grp + 16 * G.hi;
                const float fd = d.scale * gs.ep[G.tau], fa = gs.emb;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int sidx = c0 + e;
                    if (sidx == G.tau) diag_s[p][G.tau] = xd[e];  // dO_t . v_t
                    xa[e] = sidx <= G.tau ? xa[e] * fa : 0.f;
                    xd[e] = sidx < G.tau ? xd[e] * fd : 0.f;
                }
                store_row16(PA, G.tau, c0, xa);
                store_row16(PD, G.tau, c0, xd);
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&pv_ready));
                scale_tile(Ds, Ds, gs.win, d.scale, G.tid);
                fence_async_smem();
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&kq_ready));
            } else {
                {
                    float xa[16], xd[16], gam[16];
                    tok16x2(tmem, G, 32 * G.grp, 64 + 32 * G.grp, xa, xd);
                    const int c0 = 32 * G.grp + 16 * G.hi;
                    decay_row16(gs, G.tau, c0, false, gam);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int sidx = c0 + e;
                        if (sidx == G.tau) diag_s[p][G.tau] = xd[e];  // dO_t . v_t
                        xa[e] *= d.scale * gam[e];
                        xd[e] = sidx < G.tau ? xd[e] * d.scale * gam[e] : 0.f;
                    }
                    store_row16(PA, G.tau, c0, xa);
                    store_row16(PD, G.tau, c0, xd);
                }
                scale_tile(Vs, Vs, gs.wout, 1.f, G.tid);
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&pv_ready));
                if (it >= 1) mbar_wait(smem_u32(&stg_free), (it - 1) & 1);  // K~ tile free
                scale_tile(Ks, Kt, gs.wout, 1.f, G.tid);
                scale_tile(Qs, Qt, gs.win, d.scale, G.tid);
                fence_async_smem();
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&kq_ready));
            }
            // ---- E2: dk rows
            mbar_wait(smem_u32(&dk_done), kph);
            kph ^= 1;
            if (it >= 2) mbar_wait(smem_u32(&scan_done[p]), ((it - 2) >> 1) & 1);
            // the copy warp has stored the previous chunk (K~ tile free); this
            // also keeps dk_staged and dv_staged within one phase of it
            if (it >= 1) mbar_wait(smem_u32(&stg_free), (it - 1) & 1);
            // diag_s of this chunk comes from the other warp of the quadrant:
            // every epilogue warp arrived on pv_ready after writing it
            mbar_wait(smem_u32(&pv_ready), it & 1);
            tc_fence_after();
            {
                float bk = 0.f;
                const float cd = d.scale * diag_s[p][G.tau];
                const float wr = fact ? gs.wout[G.tau] : 1.f;
                float xx[2][16];
                tok16x2(tmem, G, 128 + 64 * G.grp, 128 + 64 * G.grp + 32, xx[0], xx[1]);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float qv[16], kv[16];
                    float* x = xx[k];
                    const int col = 64 * G.grp + 32 * k;
                    const int c0 = col + 16 * G.hi;
                    tile_row_get16(Qs, G.tau, c0, qv);
                    tile_row_get16(Ks, G.tau, c0, kv);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        x[e] *= wr;
                        bk = fmaf(kv[e], x[e], bk);
                        x[e] = fmaf(cd, qv[e], x[e]);
                    }
                    store_row16(Vs, G.tau, c0, x);  // V~ is dead: stage dk there
                }
                bk += __shfl_xor_sync(kFull, bk, 16);
                if (!G.hi) bpart[p][G.grp][G.tau] = bk;
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&dk_staged));
            // ---- E2: dv rows and the adjoint update
            mbar_wait(smem_u32(&dve_done), vph);
            vph ^= 1;
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&in_dead));  // after the dk rows and the products
            tc_fence_after();
            {
                float xx[2][16];
                tok16x2(tmem, G, 256 + 64 * G.grp, 256 + 64 * G.grp + 32, xx[0], xx[1]);
                const float wr = fact ? gs.wout[G.tau] : 1.f;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) xx[k][e] *= wr;
                    store_row16(Kt, G.tau, 64 * G.grp + 32 * k + 16 * G.hi, xx[k]);  // K~ is dead: stage dv there
                }
            }
            state_update_half2(tmem, G, 384, 0, gs.W, E, Eb);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) {
                mbar_arrive(smem_u32(&dv_staged));
                mbar_arrive(smem_u32(&b_ready[p]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 512);
}

// ===========================================================================
// reverse sweep for Dv = 256, warp-specialised like the Dv = 128 sweep.  At
// Dv = 256 the fp32 adjoint E (128 x 256) would take 128 registers a thread,
// so it lives in tensor memory instead, where dE = Q~^T dO accumulates into
// it; the epilogue snapshots it to the bf16 E tile that the next chunk's
// products read and, in the same pass, scales the tensor-memory copy by W of
// that chunk ahead of its dE.
// Tensor memory: [0,128) the scores, then dv half 0; [128,256) dk', then dv
// half 1; [256,512) E.
// Shared memory: Q|K by chunk parity (2 x 32 KB), V and dO (32 KB each,
// refilled as soon as their last reader is done), E as bf16 (64 KB), PA, PD.
//   warps 0-7 (epilogues), per chunk:
//     E1  score masks; factored: dO~ in place          -> pv_ready, kq_ready
//                      general: V~ in place           -> pv_ready
//     E2  dk rows                                     -> v_dead
//         general: K~, Q~ in place                    -> kq_ready
//         (dk' read                                   -> dk_read)
//         dv rows of half 0                           -> dv0_read
//         dv rows of half 1                           -> in_dead
//         E snapshot (and E *= W of the next chunk)   -> e_ready, b_ready
//   warp 8 (one thread): the tensor products; in factored chunks V E^T and
//     K E need no epilogue work, V E^T is issued as soon as E is in place.
//   warp 9: the gate-gradient scan and the gate tables two chunks ahead.
//   warp 10 (one thread): V, dO and Q|K loads as the tiles die (dO at the
//     commit of the chunk's last products).
// ===========================================================================
__global__ void __launch_bounds__(kRev3Threads, 1)
    tc_rev256_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                     const __grid_constant__ CUtensorMap mdo, const float* __restrict__ g,
                     const float* __restrict__ S_in, const float* __restrict__ dS_out,
                     const float* __restrict__ qdq, __nv_bfloat16* __restrict__ dk,
                     __nv_bfloat16* __restrict__ dv, float* __restrict__ dg) {
    constexpr int DV = 256;
    constexpr uint32_t QKB = 4 * kTileBytes;  // Q | K
    constexpr uint32_t OFF_V = 2 * QKB, OFF_D = OFF_V + 4 * kTileBytes, OFF_E = OFF_D + 4 * kTileBytes;
    constexpr uint32_t OFF_PA = OFF_E + 8 * kTileBytes, OFF_PD = OFF_PA + kTileBytes;
    constexpr uint32_t TE = 256;  // tensor-memory column of E
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Vs = smem + OFF_V;
    uint8_t* Ds = smem + OFF_D;
    uint8_t* Eb = smem + OFF_E;
    uint8_t* PA = smem + OFF_PA;
    uint8_t* PD = smem + OFF_PD;
    __shared__ GateSmem gsb[2];
    __shared__ __align__(8) uint64_t qk_full[2], v_full, d_full;
    __shared__ __align__(8) uint64_t score_bar, dk_done, dv0_done, dv1_done;  // tensor-core commits
    __shared__ __align__(8) uint64_t pv_ready, kq_ready, dk_read, dv0_read, e_ready;  // epilogue -> warp 8
    __shared__ __align__(8) uint64_t v_dead, in_dead;  // epilogue -> warp 10
    __shared__ __align__(8) uint64_t b_ready[2], scan_done[2], gate_ready[2];
    __shared__ uint32_t tmem_slot;
    __shared__ float diag_s[2][kChunk];
    __shared__ float bpart[2][2][kChunk];
    __shared__ float red[8];

    const Geo G = geo();
    const bool epi = G.warp < 8;
    const bool ctl = G.warp == 8;
    const bool scn = G.warp == 9;
    const bool cpy = G.warp == 10;
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&qk_full[i]), 1);
            mbar_init(smem_u32(&b_ready[i]), 8);
            mbar_init(smem_u32(&scan_done[i]), 1);
            mbar_init(smem_u32(&gate_ready[i]), 1);
        }
        mbar_init(smem_u32(&v_full), 1);
        mbar_init(smem_u32(&d_full), 1);
        mbar_init(smem_u32(&score_bar), 1);
        mbar_init(smem_u32(&dk_done), 1);
        mbar_init(smem_u32(&dv0_done), 1);
        mbar_init(smem_u32(&dv1_done), 1);
        for (uint64_t* bar : {&pv_ready, &kq_ready, &dk_read, &dv0_read, &e_ready, &v_dead, &in_dead})
            mbar_init(smem_u32(bar), 8);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
    GateRegs gr;
    if (scn) {  // gate tables of the first two chunks; registers for the third
        gr = gate_load(d, g, b, h, a0 + (nch - 1) * kChunk, G.lane);
        gate_prep(gr, &gsb[0], G.lane);
        if (nch > 1) {
            gr = gate_load(d, g, b, h, a0 + (nch - 2) * kChunk, G.lane);
            gate_prep(gr, &gsb[1], G.lane);
        }
        if (nch > 2) gr = gate_load(d, g, b, h, a0 + (nch - 3) * kChunk, G.lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (epi) {
        // E starts as dS_out: into tensor memory and the bf16 tile; thread
        // (srow, grp) owns columns [128 grp, +128).  ext = <S_out, dS_out>,
        // S_out read as S_in[seg + 1].
        const float* src = dS_out + sum_off(d, seg, b, h) + int64_t(G.srow) * DV + 128 * G.grp;
        const float* so = S_in + sum_off(d, seg + 1, b, h) + int64_t(G.srow) * DV + 128 * G.grp;
        // the tensor-memory E is kept scaled by W of the chunk about to
        // accumulate into it (the bf16 tile holds it unscaled)
        const float W0 = gsb[0].W;
        float ext = 0.f;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + 32 * j + i);
                r[i] = __float_as_uint(x.x); r[i + 1] = __float_as_uint(x.y);
                r[i + 2] = __float_as_uint(x.z); r[i + 3] = __float_as_uint(x.w);
                if (seg + 1 < d.nseg) {
                    const float4 y = *reinterpret_cast<const float4*>(so + 32 * j + i);
                    ext = fmaf(x.x, y.x, ext); ext = fmaf(x.y, y.y, ext);
                    ext = fmaf(x.z, y.z, ext); ext = fmaf(x.w, y.w, ext);
                }
            }
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                f[i] = __uint_as_float(r[i]);
                r[i] = __float_as_uint(W0 * f[i]);
            }
            tmem_st32(tmem + G.tl + TE + 128 * G.grp + 32 * j, r);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(Eb + sw_chunk(128, G.srow, 16 * G.grp + 4 * j + c)) = pack8(f + 8 * c);
        }
        tmem_wait_st();
        ext = warp_sum(ext);
        if (G.lane == 0) red[G.warp] = ext;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (ctl) {
        if (G.lane == 0) {
            const uint32_t sb0 = smem_u32(smem);
            const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, kTileBytes, 1024);
            const uint64_t DM2 = sdesc(sb0, 2 * kTileBytes, 1024);
            const uint64_t pa = desc_plus(DM, OFF_PA), pd = desc_plus(DM, OFF_PD);
            const uint64_t ek = desc_plus(DK, OFF_E), em = desc_plus(DM2, OFF_E);
            const uint64_t vk = desc_plus(DK, OFF_V), dk16 = desc_plus(DK, OFF_D), dm = desc_plus(DM, OFF_D);
            constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
            constexpr uint32_t id_mm = idesc_bf16(64, 128, 1, 1);
            constexpr uint32_t id_kk = idesc_bf16(64, 128, 0, 0);
            constexpr uint32_t id_km = idesc_bf16(64, 128, 0, 1);
            constexpr uint32_t id_e = idesc_bf16(128, 256, 1, 1);
            auto issue_scores = [&](int p) {  // A = Q K^T, dA = dO V^T
                const uint64_t q = desc_plus(DK, p * QKB), kk = desc_plus(q, 2 * kTileBytes);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                    mma_bf16(tmem, desc_plus(q, off), desc_plus(kk, off), id1, k > 0);
                }
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                    mma_bf16(tmem + 64, desc_plus(dk16, off), desc_plus(vk, off), id1, k > 0);
                }
                mma_commit(smem_u32(&score_bar));
            };
            auto issue_ve = [&](bool first) {  // dk' (+)= V E^T
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    mma_bf16(tmem + 128, desc_plus(vk, (k >> 2) * kTileBytes + (k & 3) * 32),
                             desc_plus(ek, (k >> 2) * 2 * kTileBytes + (k & 3) * 32), id_kk,
                             (first && k == 0) ? 0u : 1u);
            };
            // dv_hh = PA^T dO_hh + K E_hh, half 0 into the scores' columns, half 1
            // into dk''s (free once the dk rows have been read)
            auto issue_dv = [&](int hh, uint64_t kx) {
                const uint64_t dah = desc_plus(dm, 2 * hh * kTileBytes), eah = desc_plus(em, 4 * hh * kTileBytes);
                const uint32_t acc = tmem + 128 * hh;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(acc, desc_plus(pa, k * 2048), desc_plus(dah, k * 2048), id_mm, k > 0);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16(acc, desc_plus(kx, (k >> 2) * kTileBytes + (k & 3) * 32), desc_plus(eah, k * 2048),
                             id_km, 1);
            };
            mbar_wait(smem_u32(&qk_full[0]), 0);
            mbar_wait(smem_u32(&v_full), 0);
            mbar_wait(smem_u32(&d_full), 0);
            tc_fence_after();
            issue_scores(0);
            bool fact = gsb[0].fact != 0;
            if (fact) issue_ve(true);
            for (int it = 0; it < nch; ++it) {
                const int p = it & 1;
                const uint32_t ph = it & 1;
                const uint64_t qm = desc_plus(DM, p * QKB), kx = desc_plus(DK, p * QKB + 2 * kTileBytes);
                mbar_wait(smem_u32(&pv_ready), ph);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // dk' (+)= PdA^T Q
                    mma_bf16(tmem + 128, desc_plus(pd, k * 2048), desc_plus(qm, k * 2048), id_mm,
                             (fact || k > 0) ? 1u : 0u);
                if (!fact) issue_ve(false);  // V~ E^T
                mma_commit(smem_u32(&dk_done));
                mbar_wait(smem_u32(&kq_ready), ph);  // dO~ or K~, Q~ in place; E scaled by W
                tc_fence_after();
                issue_dv(0, kx);
                mma_commit(smem_u32(&dv0_done));
#pragma unroll
                for (int k = 0; k < 4; ++k)  // E += Q~^T dO (all 256 columns)
                    mma_bf16(tmem + TE, desc_plus(qm, k * 2048), desc_plus(dm, k * 2048), id_e, 1u);
                mbar_wait(smem_u32(&dk_read), ph);  // dk' columns read: dv half 1 goes there
                tc_fence_after();
                issue_dv(1, kx);
                mma_commit(smem_u32(&dv1_done));
                if (it + 1 < nch) {
                    mbar_wait(smem_u32(&dv0_read), ph);  // the scores overwrite dv half 0
                    mbar_wait(smem_u32(&qk_full[p ^ 1]), ((it + 1) >> 1) & 1);
                    mbar_wait(smem_u32(&v_full), (it + 1) & 1);
                    mbar_wait(smem_u32(&d_full), (it + 1) & 1);
                    tc_fence_after();
                    issue_scores(p ^ 1);
                    // E of the chunk before is in the bf16 tile: the next chunk's V E^T
                    mbar_wait(smem_u32(&e_ready), ph);
                    if (it + 1 >= 2) mbar_wait(smem_u32(&gate_ready[p ^ 1]), ((it - 1) >> 1) & 1);
                    fact = gsb[p ^ 1].fact != 0;
                    if (fact) {
                        tc_fence_after();
                        issue_ve(true);
                    }
                }
            }
        }
    } else if (cpy) {
        if (G.lane == 0) {
            auto load_qk = [&](int it, int p) {
                const int row = b * d.T + a0 + (nch - 1 - it) * kChunk;
                const uint32_t bar = smem_u32(&qk_full[p]);
                uint8_t* st = smem + p * QKB;
                mbar_expect_tx(bar, QKB);
                load_tile(st, &mq, 0, 128, h / d.qdiv, row, bar);
                load_tile(st + 2 * kTileBytes, &mk, 0, 128, h, row, bar);
            };
            auto load_one = [&](int it, uint8_t* dst, const CUtensorMap* map, uint64_t* barp) {
                const int row = b * d.T + a0 + (nch - 1 - it) * kChunk;
                const uint32_t bar = smem_u32(barp);
                mbar_expect_tx(bar, 4 * kTileBytes);
                load_tile(dst, map, 0, DV, h, row, bar);
            };
            load_qk(0, 0);
            load_one(0, Vs, &mv, &v_full);
            load_one(0, Ds, &mdo, &d_full);
            if (nch > 1) load_qk(1, 1);
            for (int it = 0; it + 1 < nch; ++it) {
                const uint32_t ph = it & 1;
                mbar_wait(smem_u32(&v_dead), ph);  // dk' and the scores are done with V
                load_one(it + 1, Vs, &mv, &v_full);
                mbar_wait(smem_u32(&dv1_done), ph);  // the chunk's last products (dO's readers) are done
                load_one(it + 1, Ds, &mdo, &d_full);
                mbar_wait(smem_u32(&in_dead), ph);  // ... and the dk rows have read Q and K
                if (it + 2 < nch) load_qk(it + 2, it & 1);
            }
        }
    } else if (scn) {
        float carry = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) carry += red[w];
        for (int it = 0; it < nch; ++it) {
            const int c = nch - 1 - it;
            const int t0 = a0 + c * kChunk;
            const int p = it & 1;
            const float qd0 = __ldg(qdq + ((int64_t)b * d.T + t0 + 63 - 2 * G.lane) * d.H + h);
            const float qd1 = __ldg(qdq + ((int64_t)b * d.T + t0 + 62 - 2 * G.lane) * d.H + h);
            mbar_wait(smem_u32(&b_ready[p]), (it >> 1) & 1);
            carry = dg_scan(gsb[p], bpart[p], qd0, qd1, carry, G.lane,
                            dg + ((int64_t)b * d.T + t0) * d.H + h, d.H);
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&scan_done[p]));
            if (it + 2 < nch) {
                gate_prep(gr, &gsb[p], G.lane);
                if (it + 3 < nch) gr = gate_load(d, g, b, h, t0 - 3 * kChunk, G.lane);
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&gate_ready[p]));
            }
        }
    } else {  // epilogue warps
        uint32_t sph = 0, kph = 0, v0ph = 0, v1ph = 0;
        for (int it = 0; it < nch; ++it) {
            const int c = nch - 1 - it;
            const int t0 = a0 + c * kChunk;
            const int p = it & 1;
            const GateSmem& gs = gsb[p];
            uint8_t* Qs = smem + p * QKB;
            uint8_t* Ks = Qs + 2 * kTileBytes;
            const int64_t tok = ((int64_t)b * d.T + t0 + G.tau) * d.H + h;
            // ---- E1
            if (it >= 2) mbar_wait(smem_u32(&gate_ready[p]), ((it - 2) >> 1) & 1);
            mbar_wait(smem_u32(&score_bar), sph);
            sph ^= 1;
            mbar_wait(smem_u32(&qk_full[p]), (it >> 1) & 1);
            mbar_wait(smem_u32(&v_full), it & 1);
            mbar_wait(smem_u32(&d_full), it & 1);
            tc_fence_after();
            const bool fact = gs.fact != 0;
            {
                float xa[16], xd[16];
                tok16x2(tmem, G, 32 * G.grp, 64 + 32 * G.grp, xa, xd);
                const int c0 = 32 * G.grp + 16 * G.hi;
                if (fact) {
                    // dk = wout (Pd^T Q + V E^T) with Pd = scale ep_t dA (s < t);
                    // dv = wout (Pa^T dO~ + K E) with Pa = e^(-b_63) A (s <= t);
                    // dE = Q^T dO~, dO~ = scale win dO
                    const float fd = d.scale * gs.ep[G.tau], fa = gs.emb;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int sidx = c0 + e;
                        if (sidx == G.tau) diag_s[p][G.tau] = xd[e];  // dO_t . v_t
                        xa[e] = sidx <= G.tau ? xa[e] * fa : 0.f;
                        xd[e] = sidx < G.tau ? xd[e] * fd : 0.f;
                    }
                } else {
                    float gam[16];
                    decay_row16(gs, G.tau, c0, false, gam);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int sidx = c0 + e;
                        if (sidx == G.tau) diag_s[p][G.tau] = xd[e];  // dO_t . v_t
                        xa[e] *= d.scale * gam[e];
                        xd[e] = sidx < G.tau ? xd[e] * d.scale * gam[e] : 0.f;
                    }
                }
                store_row16(PA, G.tau, c0, xa);
                store_row16(PD, G.tau, c0, xd);
            }
            if (!fact) {  // V~ = wout V in place
                scale_tile(Vs, Vs, gs.wout, 1.f, G.tid);
                scale_tile(Vs + 2 * kTileBytes, Vs + 2 * kTileBytes, gs.wout, 1.f, G.tid);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&pv_ready));
            if (fact) {
                scale_tile(Ds, Ds, gs.win, d.scale, G.tid);
                scale_tile(Ds + 2 * kTileBytes, Ds + 2 * kTileBytes, gs.win, d.scale, G.tid);
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&kq_ready));
            }
            // ---- E2: dk rows
            mbar_wait(smem_u32(&dk_done), kph);
            kph ^= 1;
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&v_dead));
            if (it >= 2) mbar_wait(smem_u32(&scan_done[p]), ((it - 2) >> 1) & 1);
            mbar_wait(smem_u32(&pv_ready), it & 1);  // diag_s from the other warp of the quadrant
            tc_fence_after();
            const float wr = fact ? gs.wout[G.tau] : 1.f;
            {
                float bk = 0.f;
                const float cd = d.scale * diag_s[p][G.tau];
                float xx[2][16];
                tok16x2(tmem, G, 128 + 64 * G.grp, 128 + 64 * G.grp + 32, xx[0], xx[1]);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float qv[16], kv[16];
                    float* x = xx[k];
                    const int c0 = 64 * G.grp + 32 * k + 16 * G.hi;
                    tile_row_get16(Qs, G.tau, c0, qv);
                    tile_row_get16(Ks, G.tau, c0, kv);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        x[e] *= wr;
                        bk = fmaf(kv[e], x[e], bk);
                        x[e] = fmaf(cd, qv[e], x[e]);
                    }
                    store_bf16x16(dk + tok * 128 + c0, x);
                }
                bk += __shfl_xor_sync(kFull, bk, 16);
                if (!G.hi) bpart[p][G.grp][G.tau] = bk;
            }
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&dk_read));
            if (!fact) {
                // K~ = wout K and Q~ = scale win Q in place, once every epilogue
                // warp has read its q, k rows
                asm volatile("bar.sync 1, 256;" ::: "memory");
                scale_tile(Ks, Ks, gs.wout, 1.f, G.tid);
                scale_tile(Qs, Qs, gs.win, d.scale, G.tid);
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&kq_ready));
            }
            // ---- E2: dv rows, half 0 then half 1
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                mbar_wait(smem_u32(hh == 0 ? &dv0_done : &dv1_done), hh == 0 ? v0ph : v1ph);
                if (hh == 0) v0ph ^= 1; else v1ph ^= 1;
                tc_fence_after();
                if (hh == 1) {
                    __syncwarp();
                    if (G.lane == 0) mbar_arrive(smem_u32(&in_dead));
                }
                float xx[2][16];
                tok16x2(tmem, G, 128 * hh + 64 * G.grp, 128 * hh + 64 * G.grp + 32, xx[0], xx[1]);
                if (hh == 0) {
                    tc_fence_before();
                    __syncwarp();
                    if (G.lane == 0) mbar_arrive(smem_u32(&dv0_read));
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) xx[k][e] *= wr;
                    store_bf16x16(dv + tok * DV + 128 * hh + 64 * G.grp + 32 * k + 16 * G.hi, xx[k]);
                }
            }
            // ---- E2: E snapshot (the chunk's products are done with the E tile);
            // the tensor-memory copy is scaled by W of the next chunk, ahead
            // of that chunk's dE
            float Wn = 1.f;
            if (it + 1 < nch) {
                if (it + 1 >= 2) mbar_wait(smem_u32(&gate_ready[p ^ 1]), ((it - 1) >> 1) & 1);
                Wn = gsb[p ^ 1].W;
            }
#pragma unroll 1
            for (int j = 0; j < 4; j += 2) {  // two 32-column loads in flight at a time
                uint32_t r0[32], r1[32];
                tmem_ld32_nowait(tmem + G.tl + TE + 128 * G.grp + 32 * j, r0);
                tmem_ld32_nowait(tmem + G.tl + TE + 128 * G.grp + 32 * (j + 1), r1);
                tmem_wait_ld();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    *reinterpret_cast<uint4*>(Eb + sw_chunk(128, G.srow, 16 * G.grp + 4 * j + cc)) =
                        pack8(reinterpret_cast<const float*>(r0) + 8 * cc);
                    *reinterpret_cast<uint4*>(Eb + sw_chunk(128, G.srow, 16 * G.grp + 4 * (j + 1) + cc)) =
                        pack8(reinterpret_cast<const float*>(r1) + 8 * cc);
                }
                if (it + 1 < nch) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        r0[i] = __float_as_uint(Wn * __uint_as_float(r0[i]));
                        r1[i] = __float_as_uint(Wn * __uint_as_float(r1[i]));
                    }
                    tmem_st32(tmem + G.tl + TE + 128 * G.grp + 32 * j, r0);
                    tmem_st32(tmem + G.tl + TE + 128 * G.grp + 32 * (j + 1), r1);
                }
            }
            tmem_wait_st();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) {
                mbar_arrive(smem_u32(&e_ready));
                mbar_arrive(smem_u32(&b_ready[p]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 512);
}

// ===========================================================================
// forward sweep of the backward for Dv = 256: dq and q.dq' per token.  The
// fp32 state S (128 x 256) lives in tensor memory, where dS accumulates; the
// epilogue scales it by W (after dS in factored chunks, before it otherwise)
// and snapshots it to the bf16 S tile for the next chunk's dO S^T.  Gamma
// keeps its own pass at Dv = 256 (its accumulator would not fit beside S).
// Tensor memory: [0,64) dA, [128,256) dq', [256,512) S.
// Shared memory: Q|K by chunk parity (2 x 32 KB), V and dO (32 KB each), S as
// bf16 (64 KB), P.  dS = K^T V is issued first once the chunk's operands are
// ready, so V dies early and the next chunk's V load overlaps dq' and the dq
// rows; dO dies with dq'.
//   warps 0-7 (epilogues): E1 score mask, K^ (factored) or dO~, V~ and
//     S *= W (general) -> p_ready;  E2 dq rows -> in_dead, state snapshot
//     -> s_ready, a_ready.
//   warp 8 (one thread): the tensor products.  warp 9: q.dq' sums and gate
//   tables.  warp 10 (one thread): V at v_dead, dO at dq_done, Q|K at in_dead.
// ===========================================================================
__global__ void __launch_bounds__(kRev3Threads, 1)
    tc_dq256_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                    const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                    const __grid_constant__ CUtensorMap mdo, const float* __restrict__ g,
                    const float* __restrict__ S_in, __nv_bfloat16* __restrict__ dq,
                    float* __restrict__ qdq) {
    constexpr int DV = 256;
    constexpr uint32_t QKB = 4 * kTileBytes;  // Q | K
    constexpr uint32_t OFF_V = 2 * QKB, OFF_D = OFF_V + 4 * kTileBytes, OFF_S = OFF_D + 4 * kTileBytes;
    constexpr uint32_t OFF_P = OFF_S + 8 * kTileBytes;
    constexpr uint32_t TS = 256;  // tensor-memory column of S
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Vs = smem + OFF_V;
    uint8_t* Ds = smem + OFF_D;
    uint8_t* Sb = smem + OFF_S;
    uint8_t* Ps = smem + OFF_P;
    __shared__ GateSmem gsb[2];
    __shared__ __align__(8) uint64_t qk_full[2], v_full, d_full;
    __shared__ __align__(8) uint64_t score_bar, v_dead, dq_done;  // tensor-core commits
    __shared__ __align__(8) uint64_t p_ready, s_ready;           // epilogue -> warp 8
    __shared__ __align__(8) uint64_t in_dead[2];                 // epilogue -> warp 10, by chunk parity
    __shared__ __align__(8) uint64_t a_ready[2], a_done[2], gate_ready[2];
    __shared__ uint32_t tmem_slot;
    __shared__ float diag_s[2][kChunk];
    __shared__ float apart[2][2][kChunk];

    const Geo G = geo();
    const bool epi = G.warp < 8;
    const bool ctl = G.warp == 8;
    const bool gat = G.warp == 9;
    const bool cpy = G.warp == 10;
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&qk_full[i]), 1);
            mbar_init(smem_u32(&a_ready[i]), 8);
            mbar_init(smem_u32(&a_done[i]), 1);
            mbar_init(smem_u32(&gate_ready[i]), 1);
            mbar_init(smem_u32(&in_dead[i]), 8);
        }
        mbar_init(smem_u32(&v_full), 1);
        mbar_init(smem_u32(&d_full), 1);
        mbar_init(smem_u32(&score_bar), 1);
        mbar_init(smem_u32(&v_dead), 1);
        mbar_init(smem_u32(&dq_done), 1);
        mbar_init(smem_u32(&p_ready), 8);
        mbar_init(smem_u32(&s_ready), 8);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
    GateRegs gr;
    if (gat) {  // gate tables of the first two chunks; registers for the third
        gr = gate_load(d, g, b, h, a0, G.lane);
        gate_prep(gr, &gsb[0], G.lane);
        if (nch > 1) {
            gr = gate_load(d, g, b, h, a0 + kChunk, G.lane);
            gate_prep(gr, &gsb[1], G.lane);
        }
        if (nch > 2) gr = gate_load(d, g, b, h, a0 + 2 * kChunk, G.lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (epi) {  // S_in into tensor memory and the bf16 tile; thread (srow, grp) owns columns [128 grp, +128)
        const float* src = S_in + sum_off(d, seg, b, h) + int64_t(G.srow) * DV + 128 * G.grp;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            float f[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + 32 * j + i);
                f[i] = x.x; f[i + 1] = x.y; f[i + 2] = x.z; f[i + 3] = x.w;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(f[i]);
            tmem_st32(tmem + G.tl + TS + 128 * G.grp + 32 * j, r);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(Sb + sw_chunk(128, G.srow, 16 * G.grp + 4 * j + c)) = pack8(f + 8 * c);
        }
        tmem_wait_st();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (ctl) {
        if (G.lane == 0) {
            const uint32_t sb0 = smem_u32(smem);
            const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, kTileBytes, 1024);
            const uint64_t pa = desc_plus(DK, OFF_P), sa = desc_plus(DK, OFF_S);
            const uint64_t vk = desc_plus(DK, OFF_V), vm = desc_plus(DM, OFF_V), dk16 = desc_plus(DK, OFF_D);
            constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
            constexpr uint32_t id_a = idesc_bf16(64, 128, 0, 1);
            constexpr uint32_t id_b = idesc_bf16(64, 128, 0, 0);
            constexpr uint32_t id_s = idesc_bf16(128, 256, 1, 1);
            auto issue_scores = [&]() {  // dA = dO V^T
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                    mma_bf16(tmem, desc_plus(dk16, off), desc_plus(vk, off), id1, k > 0);
                }
                mma_commit(smem_u32(&score_bar));
            };
            auto issue_state_side = [&](bool first) {  // dq' (+)= dO S_prev^T
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    mma_bf16(tmem + 128, desc_plus(dk16, (k >> 2) * kTileBytes + (k & 3) * 32),
                             desc_plus(sa, (k >> 2) * 2 * kTileBytes + (k & 3) * 32), id_b,
                             (first && k == 0) ? 0u : 1u);
            };
            mbar_wait(smem_u32(&v_full), 0);
            mbar_wait(smem_u32(&d_full), 0);
            tc_fence_after();
            issue_scores();
            bool fact = gsb[0].fact != 0;
            if (fact) issue_state_side(true);
            for (int c = 0; c < nch; ++c) {
                const int p = c & 1;
                const uint32_t ph = c & 1;
                const uint64_t km = desc_plus(DM, p * QKB + 2 * kTileBytes);
                mbar_wait(smem_u32(&p_ready), ph);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // S += K^T V  (K^ or V~ carry the weights)
                    mma_bf16(tmem + TS, desc_plus(km, k * 2048), desc_plus(vm, k * 2048), id_s, 1u);
                mma_commit(smem_u32(&v_dead));
#pragma unroll
                for (int k = 0; k < 4; ++k)  // dq' (+)= P K  (strictly causal part)
                    mma_bf16(tmem + 128, desc_plus(pa, k * 32), desc_plus(km, k * 2048), id_a,
                             (fact || k > 0) ? 1u : 0u);
                if (!fact) issue_state_side(false);  // dO~ S_prev^T
                mma_commit(smem_u32(&dq_done));
                if (c + 1 < nch) {
                    mbar_wait(smem_u32(&v_full), (c + 1) & 1);
                    mbar_wait(smem_u32(&d_full), (c + 1) & 1);
                    tc_fence_after();
                    issue_scores();
                    // the state after this chunk is in the S tile: the next
                    // factored chunk's dO S^T
                    mbar_wait(smem_u32(&s_ready), ph);
                    if (c + 1 >= 2) mbar_wait(smem_u32(&gate_ready[p ^ 1]), ((c - 1) >> 1) & 1);
                    fact = gsb[p ^ 1].fact != 0;
                    if (fact) {
                        tc_fence_after();
                        issue_state_side(true);
                    }
                }
            }
        }
    } else if (cpy) {
        if (G.lane == 0) {
            auto load_qk = [&](int c, int p) {
                const int row = b * d.T + a0 + c * kChunk;
                const uint32_t bar = smem_u32(&qk_full[p]);
                uint8_t* st = smem + p * QKB;
                mbar_expect_tx(bar, QKB);
                load_tile(st, &mq, 0, 128, h / d.qdiv, row, bar);
                load_tile(st + 2 * kTileBytes, &mk, 0, 128, h, row, bar);
            };
            auto load_one = [&](int c, uint8_t* dst, const CUtensorMap* map, uint64_t* barp) {
                const int row = b * d.T + a0 + c * kChunk;
                const uint32_t bar = smem_u32(barp);
                mbar_expect_tx(bar, 4 * kTileBytes);
                load_tile(dst, map, 0, DV, h, row, bar);
            };
            load_one(0, Vs, &mv, &v_full);
            load_one(0, Ds, &mdo, &d_full);
            load_qk(0, 0);
            if (nch > 1) load_qk(1, 1);
            for (int c = 0; c + 1 < nch; ++c) {
                const uint32_t ph = c & 1;
                mbar_wait(smem_u32(&v_dead), ph);  // the scores and dS are done with V
                load_one(c + 1, Vs, &mv, &v_full);
                mbar_wait(smem_u32(&dq_done), ph);  // the scores and dq' are done with dO
                load_one(c + 1, Ds, &mdo, &d_full);
                // the dq rows are done with Q and K (parity-indexed: its next
                // completion needs the Q|K this load brings)
                mbar_wait(smem_u32(&in_dead[c & 1]), (c >> 1) & 1);
                if (c + 2 < nch) load_qk(c + 2, c & 1);
            }
        }
    } else if (gat) {
        for (int c = 0; c < nch; ++c) {
            const int p = c & 1;
            const int t0 = a0 + c * kChunk;
            mbar_wait(smem_u32(&a_ready[p]), (c >> 1) & 1);
            const int64_t base = ((int64_t)b * d.T + t0) * d.H + h;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = 2 * G.lane + u;
                qdq[base + int64_t(t) * d.H] = apart[p][0][t] + apart[p][1][t];
            }
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&a_done[p]));
            if (c + 2 < nch) {
                gate_prep(gr, &gsb[p], G.lane);
                if (c + 3 < nch) gr = gate_load(d, g, b, h, t0 + 3 * kChunk, G.lane);
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&gate_ready[p]));
            }
        }
    } else {  // epilogue warps
        uint32_t sph = 0, dph = 0;
        for (int c = 0; c < nch; ++c) {
            const int p = c & 1;
            const int t0 = a0 + c * kChunk;
            const GateSmem& gs = gsb[p];
            uint8_t* Qs = smem + p * QKB;
            uint8_t* Ks = Qs + 2 * kTileBytes;
            // ---- E1
            if (c >= 2) mbar_wait(smem_u32(&gate_ready[p]), ((c - 2) >> 1) & 1);
            mbar_wait(smem_u32(&score_bar), sph);
            sph ^= 1;
            mbar_wait(smem_u32(&qk_full[p]), (c >> 1) & 1);
            mbar_wait(smem_u32(&v_full), c & 1);
            mbar_wait(smem_u32(&d_full), c & 1);
            tc_fence_after();
            // Factored chunks take the decays as K^ = exp(-b) K:  dq'_t =
            // scale win_t (sum_{s<t} (dO_t . v_s) k^_s + dO_t S_prev^T) and
            // S = W (S_prev + K^T^ V); dO and V stay unscaled.
            const bool fact = gs.fact != 0;
            {
                float x[16];
                tok16(tmem, G, 32 * G.grp, x);
                const int c0 = 32 * G.grp + 16 * G.hi;
                if (fact) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (c0 + e == G.tau) diag_s[p][G.tau] = x[e];  // dO_t . v_t
                        x[e] = c0 + e < G.tau ? x[e] : 0.f;
                    }
                } else {
                    float gam[16];
                    decay_row16(gs, G.tau, c0, true, gam);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        if (c0 + e == G.tau) diag_s[p][G.tau] = x[e];  // dO_t . v_t
                        x[e] *= d.scale * gam[e];
                    }
                }
                store_row16(Ps, G.tau, c0, x);
            }
            if (fact) {
                scale_tile(Ks, Ks, gs.nb, 1.f, G.tid);  // K^
            } else {
                scale_tile(Ds, Ds, gs.win, d.scale, G.tid);  // dO~
                scale_tile(Ds + 2 * kTileBytes, Ds + 2 * kTileBytes, gs.win, d.scale, G.tid);
                scale_tile(Vs, Vs, gs.wout, 1.f, G.tid);  // V~
                scale_tile(Vs + 2 * kTileBytes, Vs + 2 * kTileBytes, gs.wout, 1.f, G.tid);
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {  // S *= W ahead of S += K^T V~
                    uint32_t r[32];
                    tmem_ld32_nowait(tmem + G.tl + TS + 128 * G.grp + 32 * j, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(gs.W * __uint_as_float(r[i]));
                    tmem_st32(tmem + G.tl + TS + 128 * G.grp + 32 * j, r);
                }
                tmem_wait_st();
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&p_ready));
            // ---- E2: dq rows
            mbar_wait(smem_u32(&dq_done), dph);
            dph ^= 1;
            if (c >= 2) mbar_wait(smem_u32(&a_done[p]), ((c - 2) >> 1) & 1);  // apart[p] free
            mbar_wait(smem_u32(&p_ready), c & 1);  // diag_s from the other warp of the quadrant
            tc_fence_after();
            {
                // factored: dq' = scale win_t acc and k_t = win_t k^_t
                const float wr = fact ? d.scale * gs.win[G.tau] : 1.f;
                const float cd = d.scale * diag_s[p][G.tau] * (fact ? gs.win[G.tau] : 1.f);
                const int64_t tok = ((int64_t)b * d.T + t0 + G.tau) * d.H + h;
                float a = 0.f;
                float xx[2][16];
                tok16x2(tmem, G, 128 + 64 * G.grp, 128 + 64 * G.grp + 32, xx[0], xx[1]);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float qv[16], kv[16];
                    float* x = xx[k];
                    const int cc = 64 * G.grp + 32 * k + 16 * G.hi;
                    tile_row_get16(Qs, G.tau, cc, qv);
                    tile_row_get16(Ks, G.tau, cc, kv);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        x[e] *= wr;
                        a = fmaf(qv[e], x[e], a);
                        x[e] = fmaf(cd, kv[e], x[e]);
                    }
                    store_bf16x16(dq + tok * 128 + cc, x);
                }
                a += __shfl_xor_sync(kFull, a, 16);
                if (!G.hi) apart[p][G.grp][G.tau] = a;
            }
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&in_dead[p]));
            // ---- E2: state snapshot (dS has accumulated: it precedes dq' in
            // the commit that dq_done tracks)
            {  // two 32-column loads in flight at a time
                const float Wf = fact ? gs.W : 1.f;  // S = W (S_prev + K^T^ V) in factored chunks
#pragma unroll 1
                for (int j = 0; j < 4; j += 2) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32_nowait(tmem + G.tl + TS + 128 * G.grp + 32 * j, r0);
                    tmem_ld32_nowait(tmem + G.tl + TS + 128 * G.grp + 32 * (j + 1), r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        r0[i] = __float_as_uint(Wf * __uint_as_float(r0[i]));
                        r1[i] = __float_as_uint(Wf * __uint_as_float(r1[i]));
                    }
                    if (fact) {
                        tmem_st32(tmem + G.tl + TS + 128 * G.grp + 32 * j, r0);
                        tmem_st32(tmem + G.tl + TS + 128 * G.grp + 32 * (j + 1), r1);
                    }
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        *reinterpret_cast<uint4*>(Sb + sw_chunk(128, G.srow, 16 * G.grp + 4 * j + cc)) =
                            pack8(reinterpret_cast<const float*>(r0) + 8 * cc);
                        *reinterpret_cast<uint4*>(Sb + sw_chunk(128, G.srow, 16 * G.grp + 4 * (j + 1) + cc)) =
                            pack8(reinterpret_cast<const float*>(r1) + 8 * cc);
                    }
                }
            }
            tmem_wait_st();
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) {
                mbar_arrive(smem_u32(&s_ready));
                mbar_arrive(smem_u32(&a_ready[p]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 512);
}

// ===========================================================================
// forward sweep, warp-specialised: o for one (segment, row, head, 128-wide
// value block).  The fp32 state block S (128 x 128) lives in tensor memory,
// where dS accumulates; the epilogue scales it by W and snapshots it to the
// bf16 state tile that the next chunk's Q S reads.
// Factored chunks (no sequence start, every |b| < 60) take the decays as
// V^ = exp(-b) V in place:
//   o_t = scale win_t (sum_{s<=t} (q_t . k_s) v^_s + q_t S_prev),
//   S   = W (S_prev + K^T V^),
// so the score mask is plain causal, Q and K stay unscaled, and Q S_prev is
// issued as soon as the previous state is in place.  Other chunks scale Q~ and
// K~ in place and pre-scale S by W.
// Tensor memory: [0,64) scores, [64,192) O, [256,384) S.
// Shared memory: Q|K and V double-buffered by chunk parity, P, S (bf16), o
// staging (written by bulk tensor stores).
//   warps 0-7: E1 score mask (+ V^, or Q~, K~, S *= W) -> p_ready;
//              E2 o rows -> o_read, o_staged; state snapshot -> s_ready,
//              in_dead, g_free
//   warp 8 (one thread): the tensor products; warp 9: gate tables;
//   warp 10 (one thread): loads (a stage refilled once its chunk is done)
//              and the o stores.
// ===========================================================================
// The sweep as a device body: value block vb of segment seg, row b, head h,
// from S_in.  tmem_slot holds the address of the tensor-memory columns
// (256 with TWO, else 512) the caller allocated (read after the body's first
// barrier).
template <bool TWO>
__device__ __forceinline__ void fwd2_body(const Dims& d, const CUtensorMap* mq, const CUtensorMap* mk,
                                          const CUtensorMap* mv, const CUtensorMap* mo,
                                          const float* __restrict__ g, const float* __restrict__ S_in,
                                          int seg, int vb, int b, int h, const uint32_t* tmem_slot) {
    constexpr uint32_t QKB = 4 * kTileBytes;  // Q | K
    constexpr uint32_t VB = 2 * kTileBytes;   // V block (128 columns)
    constexpr int NST = TWO ? 1 : 2;          // input stages
    constexpr uint32_t OFF_V = NST * QKB, OFF_P = OFF_V + NST * VB, OFF_S = OFF_P + kTileBytes;
    constexpr uint32_t OFF_O = OFF_S + 4 * kTileBytes;
    // tensor-memory columns of O and S; two CTAs a SM share the 512 columns,
    // so there O aliases the scores (issued after the scores were read)
    constexpr uint32_t TO = TWO ? 0 : 64, TS = TWO ? 128 : 256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Ps = smem + OFF_P;
    uint8_t* Sb = smem + OFF_S;
    uint8_t* Os = smem + OFF_O;
    __shared__ GateSmem gsb[2];
    __shared__ __align__(8) uint64_t qk_full[NST], v_full[NST];
    __shared__ __align__(8) uint64_t score_bar, o_done, s_done;            // tensor-core commits
    __shared__ __align__(8) uint64_t p_ready, s_ready, o_read, o_staged;   // epilogue -> warps 8, 10
    __shared__ __align__(8) uint64_t in_dead[NST], g_free[2], gate_ready[2];
    __shared__ __align__(8) uint64_t stg_free;                             // warp 10 -> epilogue

    const Geo G = geo();
    const bool epi = G.warp < 8;
    const bool ctl = G.warp == 8;
    const bool gat = G.warp == 9;
    const bool cpy = G.warp == 10;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(smem_u32(&qk_full[i]), 1);
            mbar_init(smem_u32(&v_full[i]), 1);
            mbar_init(smem_u32(&in_dead[i]), 8);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&g_free[i]), 8);
            mbar_init(smem_u32(&gate_ready[i]), 1);
        }
        mbar_init(smem_u32(&score_bar), 1);
        mbar_init(smem_u32(&o_done), 1);
        mbar_init(smem_u32(&s_done), 1);
        mbar_init(smem_u32(&p_ready), 8);
        mbar_init(smem_u32(&s_ready), 8);
        mbar_init(smem_u32(&o_read), 8);
        mbar_init(smem_u32(&o_staged), 8);
        mbar_init(smem_u32(&stg_free), 1);
        mbar_fence_init();
    }
    GateRegs gr;
    if (gat) {  // gate tables of the first two chunks; registers for the third
        gr = gate_load(d, g, b, h, a0, G.lane);
        gate_prep(gr, &gsb[0], G.lane);
        if (nch > 1) {
            gr = gate_load(d, g, b, h, a0 + kChunk, G.lane);
            gate_prep(gr, &gsb[1], G.lane);
        }
        if (nch > 2) gr = gate_load(d, g, b, h, a0 + 2 * kChunk, G.lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (epi) {  // S_in block into tensor memory and the bf16 tile: row srow, columns [64 grp, +64)
        const float* src = S_in + sum_off(d, seg, b, h) + int64_t(G.srow) * d.Dv + vb * 128 + 64 * G.grp;
        float f[64];
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + j);
            f[j] = x.x; f[j + 1] = x.y; f[j + 2] = x.z; f[j + 3] = x.w;
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(f[32 * hf + i]);
            tmem_st32(tmem + G.tl + TS + 64 * G.grp + 32 * hf, r);
        }
        tmem_wait_st();
        store_state_half(Sb, G.srow, G.grp, f);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (ctl) {
        if (G.lane == 0) {
            const uint32_t sb0 = smem_u32(smem);
            const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, kTileBytes, 1024);
            const uint64_t pa = desc_plus(DK, OFF_P), sa = desc_plus(sdesc(sb0, 2 * kTileBytes, 1024), OFF_S);
            constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
            constexpr uint32_t id_o = idesc_bf16(64, 128, 0, 1);
            constexpr uint32_t id_s = idesc_bf16(128, 128, 1, 1);
            auto issue_scores = [&](int p) {  // scores = Q K^T
                const uint64_t q = desc_plus(DK, p * QKB), kk = desc_plus(q, 2 * kTileBytes);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * kTileBytes + (k & 3) * 32;
                    mma_bf16(tmem, desc_plus(q, off), desc_plus(kk, off), id1, k > 0);
                }
                mma_commit(smem_u32(&score_bar));
            };
            auto issue_qs = [&](int p, bool first) {  // O (+)= Q S_prev
                const uint64_t q = desc_plus(DK, p * QKB);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_bf16(tmem + TO, desc_plus(q, (k >> 2) * kTileBytes + (k & 3) * 32), desc_plus(sa, k * 2048),
                             id_o, (first && k == 0) ? 0u : 1u);
            };
            mbar_wait(smem_u32(&qk_full[0]), 0);
            tc_fence_after();
            issue_scores(0);
            bool fact = gsb[0].fact != 0;
            if (!TWO && fact) issue_qs(0, true);
            for (int c = 0; c < nch; ++c) {
                const int p = c & 1;
                const int st = TWO ? 0 : p;
                const uint32_t ph = c & 1;
                const uint64_t km = desc_plus(DM, st * QKB + 2 * kTileBytes);
                const uint64_t vm = desc_plus(DM, OFF_V + st * VB);
                mbar_wait(smem_u32(&p_ready), ph);
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)  // O (+)= P V
                    mma_bf16(tmem + TO, desc_plus(pa, k * 32), desc_plus(vm, k * 2048), id_o,
                             ((!TWO && fact) || k > 0) ? 1u : 0u);
                if (TWO || !fact) issue_qs(st, false);  // O += Q S_prev (Q~ in general chunks)
                mma_commit(smem_u32(&o_done));
#pragma unroll
                for (int k = 0; k < 4; ++k)  // S += K^T V  (V^ or K~ carry the weights)
                    mma_bf16(tmem + TS, desc_plus(km, k * 2048), desc_plus(vm, k * 2048), id_s, 1u);
                mma_commit(smem_u32(&s_done));
                if (c + 1 < nch) {
                    if (TWO) {
                        mbar_wait(smem_u32(&o_read), ph);  // the scores overwrite O
                        mbar_wait(smem_u32(&qk_full[0]), (c + 1) & 1);
                        tc_fence_after();
                        issue_scores(0);
                        if (c + 1 >= 2) mbar_wait(smem_u32(&gate_ready[p ^ 1]), ((c - 1) >> 1) & 1);
                        fact = gsb[p ^ 1].fact != 0;
                        continue;
                    }
                    mbar_wait(smem_u32(&qk_full[p ^ 1]), ((c + 1) >> 1) & 1);
                    tc_fence_after();
                    issue_scores(p ^ 1);
                    // the next factored chunk's Q S once the state is in its
                    // tile and this chunk's o rows have left tensor memory
                    mbar_wait(smem_u32(&o_read), ph);
                    mbar_wait(smem_u32(&s_ready), ph);
                    if (c + 1 >= 2) mbar_wait(smem_u32(&gate_ready[p ^ 1]), ((c - 1) >> 1) & 1);
                    fact = gsb[p ^ 1].fact != 0;
                    if (fact) {
                        tc_fence_after();
                        issue_qs(p ^ 1, true);
                    }
                }
            }
        }
    } else if (cpy) {
        if (G.lane == 0) {
            auto load = [&](int c, int p) {
                const int row = b * d.T + a0 + c * kChunk;
                uint8_t* st = smem + p * QKB;
                const uint32_t qb = smem_u32(&qk_full[p]), vbar = smem_u32(&v_full[p]);
                mbar_expect_tx(qb, QKB);
                load_tile(st, mq, 0, 128, h / d.qdiv, row, qb);
                load_tile(st + 2 * kTileBytes, mk, 0, 128, h, row, qb);
                mbar_expect_tx(vbar, VB);
                load_tile(smem + OFF_V + p * VB, mv, vb * 128, 128, h, row, vbar);
            };
            load(0, 0);
            if (!TWO && nch > 1) load(1, 1);
            for (int c = 0; c < nch; ++c) {
                const int p = c & 1;
                const int row = b * d.T + a0 + c * kChunk;
                if (TWO && c + 1 < nch) {
                    // one stage: every product of the chunk has read it once
                    // S += K^T V is done (the scores of the next chunk come later)
                    mbar_wait(smem_u32(&s_done), c & 1);
                    load(c + 1, 0);
                }
                mbar_wait(smem_u32(&o_staged), c & 1);
                tma_store_3d(mo, smem_u32(Os), vb * 128, h, row);
                tma_store_3d(mo, smem_u32(Os + kTileBytes), vb * 128 + 64, h, row);
                bulk_commit();
                if (!TWO) {
                    mbar_wait(smem_u32(&in_dead[p]), (c >> 1) & 1);  // every read of the stage is done
                    if (c + 2 < nch) load(c + 2, p);
                }
                bulk_wait_read();
                mbar_arrive(smem_u32(&stg_free));
            }
            bulk_wait_all();
        }
    } else if (gat) {
        for (int c = 0; c + 2 < nch; ++c) {
            const int p = c & 1;
            mbar_wait(smem_u32(&g_free[p]), (c >> 1) & 1);
            gate_prep(gr, &gsb[p], G.lane);
            if (c + 3 < nch) gr = gate_load(d, g, b, h, a0 + (c + 3) * kChunk, G.lane);
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&gate_ready[p]));
        }
    } else {  // epilogue warps
        uint32_t sph = 0, oph = 0, tph = 0;
        for (int c = 0; c < nch; ++c) {
            const int p = c & 1;
            const int st = TWO ? 0 : p;
            const GateSmem& gs = gsb[p];
            uint8_t* Qs = smem + st * QKB;
            uint8_t* Ks = Qs + 2 * kTileBytes;
            uint8_t* Vs = smem + OFF_V + st * VB;
            // ---- E1
            if (c >= 2) mbar_wait(smem_u32(&gate_ready[p]), ((c - 2) >> 1) & 1);
            mbar_wait(smem_u32(&score_bar), sph);
            sph ^= 1;
            mbar_wait(smem_u32(&qk_full[st]), TWO ? (c & 1) : ((c >> 1) & 1));
            mbar_wait(smem_u32(&v_full[st]), TWO ? (c & 1) : ((c >> 1) & 1));
            tc_fence_after();
            const bool fact = gs.fact != 0;
            {
                float x[16];
                tok16(tmem, G, 32 * G.grp, x);
                const int c0 = 32 * G.grp + 16 * G.hi;
                if (fact) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = c0 + e <= G.tau ? x[e] : 0.f;
                } else {
                    float gam[16];
                    decay_row16(gs, G.tau, c0, false, gam);
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] *= d.scale * gam[e];
                }
                store_row16(Ps, G.tau, c0, x);
            }
            if (fact) {
                scale_tile(Vs, Vs, gs.nb, 1.f, G.tid);  // V^
            } else {
                scale_tile(Qs, Qs, gs.win, d.scale, G.tid);  // Q~
                scale_tile(Ks, Ks, gs.wout, 1.f, G.tid);     // K~
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {  // S *= W ahead of S += K~^T V
                    uint32_t r[32];
                    tmem_ld32_nowait(tmem + G.tl + TS + 64 * G.grp + 32 * hf, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(gs.W * __uint_as_float(r[i]));
                    tmem_st32(tmem + G.tl + TS + 64 * G.grp + 32 * hf, r);
                }
                tmem_wait_st();
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&p_ready));
            // ---- E2: o rows
            mbar_wait(smem_u32(&o_done), oph);
            oph ^= 1;
            if (c >= 1) mbar_wait(smem_u32(&stg_free), (c - 1) & 1);  // o staging free
            tc_fence_after();
            {
                float xx[2][16];
                tok16x2(tmem, G, TO + 64 * G.grp, TO + 64 * G.grp + 32, xx[0], xx[1]);
                tc_fence_before();
                __syncwarp();
                if (G.lane == 0) mbar_arrive(smem_u32(&o_read));
                const float wr = fact ? d.scale * gs.win[G.tau] : 1.f;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) xx[k][e] *= wr;
                    store_row16(Os, G.tau, 64 * G.grp + 32 * k + 16 * G.hi, xx[k]);
                }
            }
            fence_async_smem();
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&o_staged));
            // ---- E2: state snapshot
            mbar_wait(smem_u32(&s_done), tph);
            tph ^= 1;
            tc_fence_after();
            {
                float f[64];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t r[32];
                    tmem_ld32_nowait(tmem + G.tl + TS + 64 * G.grp + 32 * hf, r);
                    tmem_wait_ld();
                    if (fact) {  // S = W (S_prev + K^T V^)
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            f[32 * hf + i] = gs.W * __uint_as_float(r[i]);
                            r[i] = __float_as_uint(f[32 * hf + i]);
                        }
                        tmem_st32(tmem + G.tl + TS + 64 * G.grp + 32 * hf, r);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) f[32 * hf + i] = __uint_as_float(r[i]);
                    }
                }
                tmem_wait_st();
                store_state_half(Sb, G.srow, G.grp, f);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (G.lane == 0) {
                mbar_arrive(smem_u32(&s_ready));
                if (!TWO) mbar_arrive(smem_u32(&in_dead[p]));
                mbar_arrive(smem_u32(&g_free[p]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
}

template <bool TWO>
__global__ void __launch_bounds__(kRev3Threads, TWO ? 2 : 1)
    tc_fwd2_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                   const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                   const __grid_constant__ CUtensorMap mo, const float* __restrict__ g,
                   const float* __restrict__ S_in) {
    constexpr uint32_t TCOLS = TWO ? 256 : 512;
    __shared__ uint32_t tmem_slot;
    const int nvb = d.Dv / 128;
    const int seg = blockIdx.x / nvb, vb = blockIdx.x % nvb, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    if (threadIdx.x < 32) tmem_alloc(smem_u32(&tmem_slot), TCOLS);
    fwd2_body<TWO>(d, &mq, &mk, &mv, &mo, g, S_in, seg, vb, b, h, &tmem_slot);
    if (threadIdx.x < 32) tmem_dealloc(tmem_slot, TCOLS);
}

// ===========================================================================
// sum_t w_t x_t y_t^T over a segment (delta_S of forward prepare: x = k, y = v,
// w = decay to the segment end, chunks walked from the last one; gamma of
// backward prepare: x = q, y = dO, w = scale * decay from the segment start),
// paced by mbarriers: warps 0-7 scale each chunk's x rows by w in place as soon
// as it lands (xready), warp 8 (one thread) issues the chunk's products and the
// stage refills, warp 9 builds the gate tables two chunks ahead.  The scaling
// of one chunk overlaps the products of the one before.
// ===========================================================================
// The sweep itself, as a device body: segment seg of row b and head h, value
// columns [vcol0, vcol0 + DV) of y, written to out with row stride ostride.
// Warps 0-9 take the roles above; any further warp only takes part in the
// CTA barriers.  tmem_slot holds the address of DV tensor-memory columns the
// caller allocated (read after the body's first barrier).  M (if not null)
// receives exp(sum g) or 0 at (seg, b, h), and mval (if not null, shared
// memory) the same value for the caller.
template <int DV, bool GAMMA>
__device__ __forceinline__ void outer2_body(const Dims& d, const CUtensorMap* mx, const CUtensorMap* my,
                                            const float* __restrict__ g, float* __restrict__ M,
                                            float* __restrict__ out, int seg, int b, int h, int vcol0,
                                            int ostride, const uint32_t* tmem_slot, float* mval) {
    constexpr int NS = DV == 128 ? 3 : 2;
    constexpr uint32_t XBYTES = 2 * kTileBytes;
    constexpr uint32_t YBYTES = (DV / 64) * kTileBytes;
    constexpr uint32_t SBYTES = XBYTES + YBYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    __shared__ GateSmem gsb[2];
    __shared__ __align__(8) uint64_t full_bar[NS], empty_bar[NS], xready[NS];
    __shared__ __align__(8) uint64_t done_bar, gate_ready[2], g_free[2];

    const Geo G = geo();
    const bool ctl = G.warp == 8;  // warps 0-7 scale, warp 8 issues, warp 9 prepares gates
    const bool gat = G.warp == 9;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    // gamma walks forward from the segment start, delta_S backward from its end
    auto chunk_of = [&](int it) { return GAMMA ? it : nch - 1 - it; };

    if (G.tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), 1);
            mbar_init(smem_u32(&xready[i]), 8);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&gate_ready[i]), 1);
            mbar_init(smem_u32(&g_free[i]), 8);
        }
        mbar_init(smem_u32(&done_bar), 1);
        mbar_fence_init();
    }
    GateRegs gr;
    if (gat) {
        gr = gate_load(d, g, b, h, a0 + chunk_of(0) * kChunk, G.lane);
        gate_prep(gr, &gsb[0], G.lane);
        if (nch > 1) {
            gr = gate_load(d, g, b, h, a0 + chunk_of(1) * kChunk, G.lane);
            gate_prep(gr, &gsb[1], G.lane);
        }
        if (nch > 2) gr = gate_load(d, g, b, h, a0 + chunk_of(2) * kChunk, G.lane);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (ctl) {
        if (G.lane == 0) {
            auto issue = [&](int it, int s) {
                const int row = b * d.T + a0 + chunk_of(it) * kChunk;
                const uint32_t bar = smem_u32(&full_bar[s]);
                uint8_t* st = smem + s * SBYTES;
                mbar_expect_tx(bar, SBYTES);
                load_tile(st, mx, 0, 128, GAMMA ? h / d.qdiv : h, row, bar);  // x = q or k
                load_tile(st + XBYTES, my, vcol0, DV, h, row, bar);
            };
            for (int it = 0; it < NS && it < nch; ++it) issue(it, it);
            constexpr uint32_t idesc = idesc_bf16(128, DV, 1, 1);
            for (int it = 0; it < nch; ++it) {
                const int s = it % NS;
                mbar_wait(smem_u32(&xready[s]), (it / NS) & 1);
                tc_fence_after();
                const uint32_t xa = smem_u32(smem + s * SBYTES), ya = xa + XBYTES;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_bf16(tmem, sdesc(xa + k * 2048, kTileBytes, 1024), sdesc(ya + k * 2048, kTileBytes, 1024),
                             idesc, (it > 0 || k > 0) ? 1u : 0u);
                mma_commit(smem_u32(&empty_bar[s]));
                // refill the stage the previous chunk's products have finished with
                const int prev = it - 1;
                if (prev >= 0 && prev + NS < nch) {
                    const int ps = prev % NS;
                    mbar_wait(smem_u32(&empty_bar[ps]), (prev / NS) & 1);
                    issue(prev + NS, ps);
                }
            }
            mma_commit(smem_u32(&done_bar));
        }
    } else if (gat) {
        for (int it = 0; it + 2 < nch; ++it) {
            const int p = it & 1;
            mbar_wait(smem_u32(&g_free[p]), (it >> 1) & 1);
            gate_prep(gr, &gsb[p], G.lane);
            if (it + 3 < nch) gr = gate_load(d, g, b, h, a0 + chunk_of(it + 3) * kChunk, G.lane);
            __syncwarp();
            if (G.lane == 0) mbar_arrive(smem_u32(&gate_ready[p]));
        }
    } else if (G.warp < 8) {  // epilogue warps
        float run = 0.f;  // sum of the gates of the chunks already walked
        int seen = 0;     // a sequence starts in the chunks already walked
        for (int it = 0; it < nch; ++it) {
            const int s = it % NS, p = it & 1;
            const GateSmem& gs = gsb[p];
            if (it >= 2) mbar_wait(smem_u32(&gate_ready[p]), ((it - 2) >> 1) & 1);
            mbar_wait(smem_u32(&full_bar[s]), (it / NS) & 1);
            uint8_t* xt = smem + s * SBYTES;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                int r;
                const uint32_t off = scale_off(G.tid, k, &r);
                float w;
                if (GAMMA)  // scale * alpha_a ... alpha_t: no start in [a, t]
                    w = (!seen && !gs.first && gs.lid[r] == 0) ? d.scale * expf(run + gs.b[r]) : 0.f;
                else        // alpha_{t+1} ... alpha_end: no start in (t, end]
                    w = (!seen && gs.lid[r] == gs.lid[kChunk - 1]) ? expf(run + gs.btot - gs.b[r]) : 0.f;
                scale_chunk(xt + off, xt + off, w);
            }
            run += gs.btot;
            seen |= gs.any;
            fence_async_smem();
            __syncwarp();
            if (G.lane == 0) {
                mbar_arrive(smem_u32(&xready[s]));
                mbar_arrive(smem_u32(&g_free[p]));
            }
        }
        mbar_wait(smem_u32(&done_bar), 0);
        tc_fence_after();
        float* dst = out + sum_off(d, seg, b, h) + int64_t(G.srow) * ostride + vcol0;
#pragma unroll 1
        for (int c = G.grp * (DV / 2); c < (G.grp + 1) * (DV / 2); c += 64) {
            float v[64];
            state_cols64(tmem, G, c - 64 * G.grp, v);
#pragma unroll
            for (int i = 0; i < 64; i += 4)
                *reinterpret_cast<float4*>(dst + c + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
        if (!GAMMA && G.tid == 0) {
            const float m = seen ? 0.f : expf(run);
            if (M != nullptr) M[(int64_t(seg) * d.B + b) * d.H + h] = m;
            if (mval != nullptr) *mval = m;
        }
    }
    tc_fence_before();
    __syncthreads();
}

template <int DV, bool GAMMA>
__global__ void __launch_bounds__(kThreads + 64, 2)
    tc_outer2_kernel(const Dims d, const __grid_constant__ CUtensorMap mx,
                     const __grid_constant__ CUtensorMap my, const float* __restrict__ g,
                     float* __restrict__ M, float* __restrict__ out) {
    __shared__ uint32_t tmem_slot;
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    if (threadIdx.x < 32) tmem_alloc(smem_u32(&tmem_slot), DV);
    outer2_body<DV, GAMMA>(d, &mx, &my, g, M, out, seg, b, h, 0, DV, &tmem_slot, nullptr);
    if (threadIdx.x < 32) tmem_dealloc(tmem_slot, DV);
}

// ===========================================================================
// The forward in one launch: chunkwise_cp_forward's prepare, composition of
// the preceding summaries and apply ("compose the preceding summaries and
// compute the local output", cp_forward_apply), for one (segment j, row b,
// head h, value block vb) per CTA.  CTAs take tickets in the order they
// start; ticket t is (j, b H + h, vb) in segment-major order, so every CTA
// whose results a CTA waits for started earlier, and none of them waits
// before it has published what is waited for.
//   1. prepare (outer2_body on the block's 128 value columns): dS_j, M_j;
//      published with the block's "aggregate" flag.
//   2. compose: S_in[j] = the fold S <- M_i S + dS_i over i in [p_j, j) from
//      0, started instead after the last segment i in that range whose
//      inclusive prefix (= S_in[i+1]) is already published (flags read
//      without waiting); the aggregates folded after the start are waited
//      for, each wait bounded.  Every start gives the same values: an
//      inclusive prefix is the same chain of multiply-adds, and the chain
//      from p_j equals the one through it because segment p_j holds a
//      sequence start (M = 0).  The CTA writes S_in[j], then publishes its
//      own inclusive prefix M_j S_in[j] + dS_j.
//   3. apply (fwd2_body): o from S_in[j], with the same sweep variant the
//      separate apply call picks (two CTAs a SM when there are more CTAs
//      than SMs, else one with two stages).
// The multiply-adds are those of compose_prefix_kernel, in the same order,
// so M, dS, S_in and o equal those of the three separate calls.
// ===========================================================================
struct FusedWs {
    int* ticket;     // one counter
    int* agg;        // [n] aggregate published
    int* inc;        // [n] inclusive prefix published
    float* mval;     // [n] M_j of each CTA's segment
    float* incl;     // [nseg,B,H,Dk,Dv] inclusive prefixes: incl[j] = S_in[j+1]
};

template <bool TWO>
__global__ void __launch_bounds__(kRev3Threads, TWO ? 2 : 1)
    tc_fused_fwd_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                        const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                        const __grid_constant__ CUtensorMap mo, const float* __restrict__ g,
                        float* __restrict__ M, float* __restrict__ dS, float* __restrict__ S_in,
                        const FusedWs w) {
    constexpr uint32_t TCOLS = TWO ? 256 : 512;
    __shared__ uint32_t tmem_slot;
    __shared__ int tk_s, start_s, from_inc_s;
    __shared__ float m_self;
    if (threadIdx.x == 0) tk_s = atomicAdd(w.ticket, 1);
    if (threadIdx.x < 32) tmem_alloc(smem_u32(&tmem_slot), TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int nvb = d.Dv / 128, per = d.B * d.H * nvb;
    const int tk = tk_s;
    const int j = tk / per, bhv = tk % per, bh = bhv / nvb, vb = bhv % nvb;
    const int b = bh / d.H, h = bh % d.H;
    auto slot_of = [&](int i) { return (i * d.B * d.H + bh) * nvb + vb; };  // = ticket of (i, bh, vb)

    // ---- 1. prepare
    outer2_body<128, false>(d, &mk, &mv, g, vb == 0 ? M : nullptr, dS, j, b, h, vb * 128, d.Dv,
                            &tmem_slot, &m_self);
    const Geo G = geo();
    if (G.tid == 0) {  // the body's closing barrier ordered every write of dS_j before this
        w.mval[tk] = m_self;
        flag_release(w.agg + tk);
    }

    // ---- 2. compose
    if (G.warp == 0) {
        const int pj = d.preceding_start ? min(max(__ldg(d.preceding_start + j), 0), j) : 0;
        // the last i in [pj, j) with a published inclusive prefix, 32 at a time
        int start = pj, from_inc = 0;
        for (int top = j - 1; top >= pj; top -= 32) {
            const int i = top - G.lane;
            const bool ok = i >= pj && flag_acquire(w.inc + slot_of(i));
            const unsigned m = __ballot_sync(kFull, ok);
            if (m != 0u) {
                start = top - (__ffs(m) - 1) + 1;
                from_inc = 1;
                break;
            }
        }
        if (G.lane == 0) {
            for (int l = start; l < j; ++l) flag_wait(w.agg + slot_of(l));
            start_s = start;
            from_inc_s = from_inc;
        }
    }
    __syncthreads();
    if (G.warp < 8) {
        const int start = start_s;
        const int64_t col = int64_t(G.srow) * d.Dv + vb * 128 + 64 * G.grp;
        const float* dsj = dS + sum_off(d, j, b, h) + col;
        const float mj = m_self;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            float S[32];
            if (from_inc_s) {
                const float* src = w.incl + sum_off(d, start - 1, b, h) + col + 32 * hf;
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4*>(src + e));
                    S[e] = x.x; S[e + 1] = x.y; S[e + 2] = x.z; S[e + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) S[e] = 0.f;
            }
#pragma unroll 1
            for (int l = start; l < j; ++l) {
                const float m = __ldcg(w.mval + slot_of(l));
                const float* src = dS + sum_off(d, l, b, h) + col + 32 * hf;
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4*>(src + e));
                    S[e] = fmaf(m, S[e], x.x);
                    S[e + 1] = fmaf(m, S[e + 1], x.y);
                    S[e + 2] = fmaf(m, S[e + 2], x.z);
                    S[e + 3] = fmaf(m, S[e + 3], x.w);
                }
            }
            float* so = S_in + sum_off(d, j, b, h) + col + 32 * hf;
            float* io = w.incl + sum_off(d, j, b, h) + col + 32 * hf;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                *reinterpret_cast<float4*>(so + e) = make_float4(S[e], S[e + 1], S[e + 2], S[e + 3]);
                const float4 x = *reinterpret_cast<const float4*>(dsj + 32 * hf + e);
                *reinterpret_cast<float4*>(io + e) =
                    make_float4(fmaf(mj, S[e], x.x), fmaf(mj, S[e + 1], x.y), fmaf(mj, S[e + 2], x.z),
                                fmaf(mj, S[e + 3], x.w));
            }
        }
    }
    __syncthreads();  // every inclusive-prefix write is ordered before the release
    if (G.tid == 0) flag_release(w.inc + tk);

    // ---- 3. apply (reads S_in[j] back: each thread reads the elements it wrote)
    fwd2_body<TWO>(d, &mq, &mk, &mv, &mo, g, S_in, j, vb, b, h, &tmem_slot);
    if (threadIdx.x < 32) tmem_dealloc(tmem_slot, TCOLS);
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

}  // namespace

namespace {
thread_local int g_map_result = 0;  // CUresult of the calling thread's last make_map
}
int last_map_result() { return g_map_result; }
void clear_map_result() { g_map_result = 0; }

// [B*T rows][H][D] bf16 viewed as a 3-D tensor; boxes of 64 tokens x 64 columns.
bool make_map(CUtensorMap* m, const void* base, const Dims& d, int D, int heads) {
    auto fn = encode_fn();
    g_map_result = -1;  // no encoder
    if (!fn) return false;
    if (heads <= 0) heads = d.H;
    cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(heads), cuuint64_t(d.B) * cuuint64_t(d.T)};
    cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(heads) * D * 2};
    cuuint32_t box[3] = {64, 1, uint32_t(kChunk)};
    cuuint32_t estr[3] = {1, 1, 1};
    g_map_result = int(fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
    return g_map_result == int(CUDA_SUCCESS);
}

// multiprocessors of the current device (cached per device)
int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

namespace {

constexpr size_t kOuterSmem = 96 * 1024 + 1024;
// Q|K x 2 (8) + V x 2 (4) + P (1) + S (4) + o staging (2)
constexpr size_t kFwd2Smem = 19 * kTileBytes + 1024;
// two CTAs a SM: Q|K (4) + V (2) + P (1) + S (4) + o staging (2)
constexpr size_t kFwd2TwoSmem = 13 * kTileBytes + 1024;
// Q|K x 2 (8) + V (4) + dO (4) + S (8) + P (1)
constexpr size_t kDq256Smem = 25 * kTileBytes + 1024;
// 2 stages x 8 + P (1) + S (4) + gamma's Q (2) + dq staging (2)
constexpr size_t kDqg128Smem = 25 * kTileBytes + 1024;
// Dv = 128: 2 stages x 8 + Q~ K~ (4) + PA PdA (2) + E (4);
// Dv = 256: Q|K x 2 (8) + V (4) + dO (4) + E (8) + PA PdA (2): 26 tiles either way
constexpr size_t rev_smem(int dv) {
    return size_t((dv == 128 ? 2 : 1) * (4 + 2 * (dv / 64)) + 6 + 2 * (dv / 64)) * kTileBytes + 1024;
}

// Workspace of the fused forward: ticket, the two flag arrays and the M
// values (each in its own 256-byte-aligned block), then the inclusive prefixes.
size_t fused_flags_bytes(const Dims& d) {
    const size_t n = size_t(d.nseg) * d.B * d.H * (d.Dv / 128);
    const size_t blk = (n * 4 + 255) / 256 * 256;
    return 256 + 3 * blk;
}
size_t fused_bytes_for(const Dims& d) {
    return fused_flags_bytes(d) + size_t(d.nseg) * d.B * d.H * d.Dk * d.Dv * sizeof(float);
}

}  // namespace

}  // namespace tc

size_t tc_fused_bytes(const Dims& d, rm_dtype dt) {
    return tc_supports(d, dt) ? tc::fused_bytes_for(d) : 0;
}

rm_status tc_launch_fused_forward(const Dims& d, const Ptrs& p, cudaStream_t s) {
    using namespace tc;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, p.q, d, 128, d.qh) || !make_map(&mk, p.k, d, 128) ||
        !make_map(&mv, p.v, d, d.Dv) || !make_map(&mo, p.out0, d, d.Dv))
        return RM_ERR_CUDA;
    const size_t n = size_t(d.nseg) * d.B * d.H * (d.Dv / 128);
    const size_t blk = (n * 4 + 255) / 256 * 256;
    char* base = static_cast<char*>(p.ws);
    FusedWs w;
    w.ticket = reinterpret_cast<int*>(base);
    w.agg = reinterpret_cast<int*>(base + 256);
    w.inc = reinterpret_cast<int*>(base + 256 + blk);
    w.mval = reinterpret_cast<float*>(base + 256 + 2 * blk);
    w.incl = reinterpret_cast<float*>(base + fused_flags_bytes(d));
    // ticket and flags start at zero for every launch
    if (cudaMemsetAsync(base, 0, 256 + 2 * blk, s) != cudaSuccess) return RM_ERR_CUDA;
    // the apply variant of rm_cp_forward_apply for this grid (same arithmetic)
    const bool two = int64_t(n) > sm_count();
    auto fk = two ? tc_fused_fwd_kernel<true> : tc_fused_fwd_kernel<false>;
    const size_t fsm = two ? kFwd2TwoSmem : kFwd2Smem;
    if (!set_smem(fk, fsm)) return RM_ERR_CUDA;
    fk<<<unsigned(n), kRev3Threads, fsm, s>>>(d, mq, mk, mv, mo, p.g, p.M, p.sum_out, p.S_in_out, w);
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(1);
    return RM_OK;
}

rm_status tc_selftest_wait(uint32_t limit_us, cudaStream_t s) {
    tc::selftest_wait_kernel<<<1, 1, 0, s>>>(uint64_t(limit_us) * 1000ull);
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(1);
    return RM_OK;
}

rm_status tc_read_timeout_flag(int* host_flag, int clear, int* dev_scratch, cudaStream_t s) {
    tc::read_flag_kernel<<<1, 1, 0, s>>>(dev_scratch, clear);
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(1);
    if (cudaMemcpyAsync(host_flag, dev_scratch, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RM_ERR_CUDA;
    return RM_OK;
}

bool tc_supports(const Dims& d, rm_dtype dt) {
    return !d.vg && dt == RM_BF16 && d.Dk == 128 && (d.Dv == 128 || d.Dv == 256) && d.L % tc::kChunk == 0 &&
           d.T >= tc::kChunk;
}

bool tc_supports_op(Op op, const Dims& d, rm_dtype dt) {
    (void)op;
    return tc_supports(d, dt);
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
                auto fn = tc_outer2_kernel<128, false>;
                if (!set_smem(fn, kOuterSmem)) return RM_ERR_CUDA;
                fn<<<grid, kThreads + 64, kOuterSmem, s>>>(d, mk, mv, p.g, p.M, p.sum_out);
            } else {
                // at Dv = 256 (two stages) the barrier-paced variant measured
                // no faster than the original one
                auto fn = tc_outer_kernel<256, false>;
                if (!set_smem(fn, kOuterSmem)) return RM_ERR_CUDA;
                fn<<<grid, kThreads, kOuterSmem, s>>>(d, mk, mv, p.g, p.M, p.sum_out);
            }
            if (!rmcp::launch_ok()) return RM_ERR_CUDA;
            note_launch(1);
            return RM_OK;
        }
        case Op::kForwardApply: {
            CUtensorMap mo;
            if (!make_map(&mq, p.q, d, 128, d.qh) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, d.Dv) || !make_map(&mo, p.out0, d, d.Dv))
                return RM_ERR_CUDA;
            // more CTAs than SMs: two a SM (single-stage, 256 tensor-memory
            // columns) so that each hides the other's latencies; otherwise one
            // a SM with two stages
            const dim3 fgrid(d.nseg * (d.Dv / 128), d.B * d.H);
            const bool two = int64_t(fgrid.x) * fgrid.y > sm_count();
            auto ff = two ? tc_fwd2_kernel<true> : tc_fwd2_kernel<false>;
            const size_t fsm = two ? kFwd2TwoSmem : kFwd2Smem;
            if (!set_smem(ff, fsm)) return RM_ERR_CUDA;
            ff<<<fgrid, kRev3Threads, fsm, s>>>(
                d, mq, mk, mv, mo, p.g, p.S_in);
            if (!rmcp::launch_ok()) return RM_ERR_CUDA;
            note_launch(1);
            return RM_OK;
        }
        case Op::kBackwardPrepare: {
            if (!make_map(&mq, p.q, d, 128, d.qh) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, d.Dv) || !make_map(&mdo, p.dO, d, d.Dv))
                return RM_ERR_CUDA;
            CUtensorMap mdq;
            if (!make_map(&mdq, p.out0, d, 128)) return RM_ERR_CUDA;
            if (d.Dv == 128) {
                auto fq = tc_dqg128_kernel;
                if (!set_smem(fq, kDqg128Smem)) return RM_ERR_CUDA;
                fq<<<grid, kRev3Threads, kDqg128Smem, s>>>(d, mq, mk, mv, mdo, mdq, p.g, p.S_in, p.sum_out,
                                                          p.ws_f32);
                if (!rmcp::launch_ok()) return RM_ERR_CUDA;
                note_launch(1);
                return RM_OK;
            } else {
                auto fo = tc_outer_kernel<256, true>;
                auto fq = tc_dq256_kernel;
                if (!set_smem(fo, kOuterSmem) || !set_smem(fq, kDq256Smem)) return RM_ERR_CUDA;
                fo<<<grid, kThreads, kOuterSmem, s>>>(d, mq, mdo, p.g, nullptr, p.sum_out);
                if (!rmcp::launch_ok()) return RM_ERR_CUDA;
                fq<<<grid, kRev3Threads, kDq256Smem, s>>>(d, mq, mk, mv, mdo, p.g, p.S_in,
                                                          static_cast<__nv_bfloat16*>(p.out0), p.ws_f32);
            }
            if (!rmcp::launch_ok()) return RM_ERR_CUDA;
            note_launch(2);
            return RM_OK;
        }
        case Op::kBackwardApply: {
            if (!make_map(&mq, p.q, d, 128, d.qh) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, d.Dv) || !make_map(&mdo, p.dO, d, d.Dv))
                return RM_ERR_CUDA;
            auto* dko = static_cast<__nv_bfloat16*>(p.out0);
            auto* dvo = static_cast<__nv_bfloat16*>(p.out1);
            CUtensorMap mdk, mdv;
            if (!make_map(&mdk, p.out0, d, 128) || !make_map(&mdv, p.out1, d, d.Dv)) return RM_ERR_CUDA;
            if (d.Dv == 128) {
                auto fr = tc_rev128_kernel;
                if (!set_smem(fr, rev_smem(128))) return RM_ERR_CUDA;
                fr<<<grid, kRev3Threads, rev_smem(128), s>>>(d, mq, mk, mv, mdo, mdk, mdv, p.g, p.S_in, p.dS_out,
                                                          p.ws_f32, p.dg);
            } else {
                auto fr = tc_rev256_kernel;
                if (!set_smem(fr, rev_smem(256))) return RM_ERR_CUDA;
                fr<<<grid, kRev3Threads, rev_smem(256), s>>>(d, mq, mk, mv, mdo, p.g, p.S_in, p.dS_out,
                                                             p.ws_f32, dko, dvo, p.dg);
            }
            if (!rmcp::launch_ok()) return RM_ERR_CUDA;
            note_launch(1);
            return RM_OK;
        }
    }
    return RM_ERR_INVALID_ARG;
}

}  // namespace rmcp
