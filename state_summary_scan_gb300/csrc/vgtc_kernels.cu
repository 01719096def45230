// vgtc_kernels.cu -- tensor-core path (sm_103a, tcgen05 + TMA) for vector
// (per key dimension) gates: bf16 storage, Dk = Dv = 128, segment lengths
// that are multiples of 64.  Per row b and head h,
//     S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,   o_t = scale S_t^T q_t,
// alpha_t[i] = exp(g_t[i]) (0 when token t starts a sequence): the summary
// S_out = M S_in + delta_S of CPForwardUnpackedSummary on the Megatron-Core
// page "core.ssm.context_parallel.chunkwise" with a diagonal M.
//
// Chunkwise form.  In a chunk of 64 tokens let b_t[i] = g_0[i] + ... + g_t[i]
// and B[i] = b_63[i].  For tokens s <= t of one sequence the state carries
// k_s v_s^T to t with the factor exp(b_t[i] - b_s[i]) on row i, which splits
// through the chunk end as exp(b_t - B) exp(B - b_s).  So, with
//     Q~ = scale Q o exp(b - B),   K~ = K o exp(B - b),   S' = diag(W) S_prev,
// W[i] = exp(B[i]) (0 once a token of the chunk starts a sequence):
//     O      = mask(Q~ K~^T) V + Q~ S'
//     S_next = S' + K~^T V
// and the backward mirrors it (dq and dk take the per-element factor
// exp(b - B) or exp(B - b) on their accumulators).  Every product is a
// tcgen05.mma of bf16 tiles in 128-byte-swizzled shared memory with an fp32
// accumulator in tensor memory; the element-wise factors are applied while
// the tiles sit in shared memory.  A chunk is "factored" when no sequence
// starts at positions 1..63 and every |b_t[i] - B[i]| < 60 (all factors
// within e^60 in fp32 and bf16).  Other chunks take the intra-chunk scores,
// dq and dk terms directly, sum_i x y exp(b_t[i] - b_s[i]) on the CUDA
// cores, and keep the tensor-core products only for the stable terms
// (Q o win against S_prev, K o wout for the state, the adjoint products).
//
// Kernels, one CTA of 256 threads per (segment, row, head); thread 0 issues
// the TMA loads and stores and the tensor-core products, and the CTA steps
// through each chunk together (two input stages, so the next chunk's tiles
// load during this one; the apply on a grid wider than the GPU runs two CTAs
// a SM with one stage each):
//   vgtc_prepare_kernel  delta_S = sum_t diag(w_t) k_t v_t^T over the
//                        segment (w = decay to the segment end) and M
//                        (cp_forward_prepare)
//   vgtc_apply_kernel    o from S_in (cp_forward_apply)
//   vgtc_dq_kernel       cp_backward_prepare in one sweep: dq, gamma =
//                        sum_t diag(w_t) scale q_t dO_t^T (w = decay from the
//                        segment start) and, per key dimension, q_t[i] times
//                        dq_t[i] without its same-token term (for dg)
//   vgtc_rev_kernel      dk, dv and dg from dS_out (cp_backward_apply);
//                        dg is the reverse running sum, within a sequence,
//                        of q.dq - k.dk per dimension, taken as a product
//                        with a 0/1 upper-triangular matrix on the tensor
//                        cores (the summands split into two bf16 parts),
//                        plus <S_out, dS_out>.
#include "tc_tiles.cuh"

namespace rmcp {
namespace vgtc {

using namespace tc;

namespace {

constexpr int kDk = 128;
constexpr uint32_t T8 = kTileBytes;   // one [64][64] bf16 block
constexpr float kFactLimit = 60.f;

// Per-chunk gate quantities shared by the CTA (16-byte aligned: btot is
// read as float4).
struct alignas(16) VgGate {
    int lid[kChunk];    // number of sequence starts at chunk positions 1..tau
    float btot[kDk];    // B[i] = b_63[i]
    float tot0[kDk];    // g_0[i] + ... + g_31[i]
    int first;          // position 0 starts a sequence
    int any;            // some position of the chunk starts a sequence
    int ltot;           // lid[63]
};

// [B,T,H,Dk] offset of token t's per-dimension values
__device__ __forceinline__ int64_t gv_off(const Dims& d, int b, int t, int h) {
    return ((int64_t(b) * d.T + t) * d.H + h) * kDk;
}

// Gates of the chunk at t0 for this thread's dimension i = tid % 128 and
// tokens t0 + 32 hf + [0, 32), hf = tid / 128 (a warp reads 128 contiguous
// bytes per token).
__device__ __forceinline__ void gate_fetch(const Dims& d, const float* __restrict__ g, int b, int h,
                                           int t0, int tid, float* gp) {
    const int i = tid & 127, hf = tid >> 7;
    const float* src = g + gv_off(d, b, t0 + 32 * hf, h) + i;
    const int64_t stride = int64_t(d.H) * kDk;
#pragma unroll
    for (int u = 0; u < 32; ++u) gp[u] = __ldg(src + u * stride);
}

// The chunk's gate tables from the fetched gates: bt[tau][i] = b_tau[i] (fp32
// [64][128] in shared memory), gs.btot, and the sequence tables (warp 0).
// bl receives this thread's 32 values b_tau[i].  Returns whether the chunk
// is factored.  Three CTA barriers: every thread of the CTA calls it.
__device__ __forceinline__ bool gate_build(const Dims& d, int t0, const float* gp, float* bt, VgGate& gs,
                                           int tid, float* bl) {
    const int i = tid & 127, hf = tid >> 7;
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        acc += gp[u];
        bl[u] = acc;
    }
    if (hf == 0) gs.tot0[i] = acc;
    if (tid < 32) {
        const int lane = tid;
        const int t = t0 + 2 * lane;
        const int s0 = starts_sequence(d.seq_idx, t) ? 1 : 0;
        const int s1 = starts_sequence(d.seq_idx, t + 1) ? 1 : 0;
        const int c0 = lane > 0 ? s0 : 0;  // starts at positions >= 1
        const int c = c0 + s1;
        int cs = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int cc = __shfl_up_sync(kFull, cs, o);
            if (lane >= o) cs += cc;
        }
        gs.lid[2 * lane] = cs - c + c0;
        gs.lid[2 * lane + 1] = cs;
        const int ltot = __shfl_sync(kFull, cs, 31);
        const int first = __shfl_sync(kFull, s0, 0);
        if (lane == 0) {
            gs.ltot = ltot;
            gs.first = first;
            gs.any = (first || ltot > 0) ? 1 : 0;
        }
    }
    __syncthreads();
    const float off = hf ? gs.tot0[i] : 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        bl[u] += off;
        bt[(32 * hf + u) * kDk + i] = bl[u];
    }
    if (hf == 1) gs.btot[i] = bl[31];
    __syncthreads();
    const float B = gs.btot[i];
    float dev = 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) dev = fmaxf(dev, fabsf(bl[u] - B));
    return __syncthreads_and(dev < kFactLimit && gs.ltot == 0) != 0;
}

// In place: the [64][128] bf16 tile's element (r, c) times a factor.  The
// 256 threads take four 16-byte chunks each (eight consecutive threads on
// the eight chunks of a 128-byte row); f(r, c, x) scales x[0..7], the
// columns c..c+7 of row r.
template <class F>
__device__ __forceinline__ void scale_el(uint8_t* tile, int tid, F f) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int n = tid + 256 * k;
        const int r = (n >> 3) & 63, blk = n >> 9, pch = n & 7;
        const int c = 64 * blk + 8 * (pch ^ (r & 7));  // logical column of the physical chunk
        uint8_t* p = tile + blk * T8 + r * 128 + pch * 16;
        float x[8];
        unpack8(*reinterpret_cast<const uint4*>(p), x);
        f(r, c, x);
        *reinterpret_cast<uint4*>(p) = pack8(x);
    }
}

__device__ __forceinline__ void ld8(const float* p, float* x) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Factors of one 8-column chunk of row r (columns c..c+7).
struct Fac {
    const float* bt;
    const VgGate* gs;
    float scale;
    // exp(b_r - B) scale (the factored Q~)
    __device__ __forceinline__ void q_fact(int r, int c, float* x) const {
        float b[8], B[8];
        ld8(bt + r * kDk + c, b);
        ld8(gs->btot + c, B);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= scale * __expf(b[e] - B[e]);
    }
    // scale win = scale exp(b_r) if no sequence starts at positions 0..r, else 0
    __device__ __forceinline__ void q_win(int r, int c, float* x) const {
        const bool keep = !gs->first && gs->lid[r] == 0;
        float b[8];
        ld8(bt + r * kDk + c, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = keep ? x[e] * scale * __expf(b[e]) : 0.f;
    }
    // wout = exp(B - b_r) if no sequence starts at positions r+1..63, else 0
    __device__ __forceinline__ void k_wout(int r, int c, float* x) const {
        const bool keep = gs->lid[r] == gs->ltot;
        float b[8], B[8];
        ld8(bt + r * kDk + c, b);
        ld8(gs->btot + c, B);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = keep ? x[e] * __expf(B[e] - b[e]) : 0.f;
    }
};

// Rows of an M = 128 accumulator at column col (state row srow, columns
// [64 grp, +64)) times w, written back; the bf16 tile receives w S or S.
__device__ __forceinline__ void state_pass(uint32_t tmem, const Geo& G, int col, float w, bool tile_scaled,
                                           uint8_t* tile) {
    float f[64];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t r[32];
        tmem_ld32_nowait(tmem + G.tl + col + 64 * G.grp + 32 * hf, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float s = __uint_as_float(r[e]);
            const float ws = w * s;
            f[32 * hf + e] = tile_scaled ? ws : s;
            r[e] = __float_as_uint(ws);
        }
        tmem_st32(tmem + G.tl + col + 64 * G.grp + 32 * hf, r);
    }
    tmem_wait_st();
    store_state_half(tile, G.srow, G.grp, f);
}

// fp32 state rows [128][128] from global memory into tensor memory at col
// and (if tile) the bf16 tile.
__device__ __forceinline__ void state_load(const float* __restrict__ src, uint32_t tmem, const Geo& G, int col,
                                           uint8_t* tile) {
    const float* p = src + int64_t(G.srow) * kDk + 64 * G.grp;
    float f[64];
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
        const float4 x = *reinterpret_cast<const float4*>(p + j);
        f[j] = x.x; f[j + 1] = x.y; f[j + 2] = x.z; f[j + 3] = x.w;
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        uint32_t r[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(f[32 * hf + e]);
        tmem_st32(tmem + G.tl + col + 64 * G.grp + 32 * hf, r);
    }
    tmem_wait_st();
    if (tile != nullptr) store_state_half(tile, G.srow, G.grp, f);
}

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Element (r, c) of a [64][64] or [64][128] bf16 tile.
__device__ __forceinline__ float tile_el(const uint8_t* tile, int r, int c) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + sw_off(64, r, c)));
}

// Intra-chunk scores of a general chunk for this thread's 16 columns s =
// c0..c0+15 of row tau: scale sum_i q[tau][i] k[s][i] exp(b_tau[i] - b_s[i])
// for s <= tau in tau's sequence, else 0 (raw Q and K tiles).
__device__ __noinline__ void exact_scores(const uint8_t* Qs, const uint8_t* Ks, const float* bt,
                                          const VgGate& gs, int tau, int c0, float scale, uint8_t* Ps) {
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    const int lt = gs.lid[tau];
#pragma unroll 1
    for (int ic = 0; ic < 16; ++ic) {
        float qv[8], bq[8];
        unpack8(*reinterpret_cast<const uint4*>(Qs + sw_chunk(64, tau, ic)), qv);
        ld8(bt + tau * kDk + 8 * ic, bq);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int s = c0 + e;
            if (s <= tau && gs.lid[s] == lt) {
                float kv[8], bs[8];
                unpack8(*reinterpret_cast<const uint4*>(Ks + sw_chunk(64, s, ic)), kv);
                ld8(bt + s * kDk + 8 * ic, bs);
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[e] = fmaf(qv[u] * kv[u], __expf(bq[u] - bs[u]), acc[e]);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] *= scale;
    store_row16(Ps, tau, c0, acc);
}

// TMA store of a [64][128] bf16 tile to rows row.. of the [B*T][H][128] map.
__device__ __forceinline__ void store_tile(const CUtensorMap* map, const uint8_t* tile, int h, int row) {
    tma_store_3d(map, smem_u32(tile), 0, h, row);
    tma_store_3d(map, smem_u32(tile + T8), 64, h, row);
}

// ===========================================================================
// forward prepare: delta_S = sum_t diag(w_t) k_t v_t^T over a segment, chunks
// walked from the segment end, w_t[i] = exp(sum of g[i] over (t, end]) with
// no sequence start in (t, end]; M[i] = exp(sum of g[i] over the segment), 0
// if a sequence starts in it.
// Shared memory: two stages of K|V (32 KB each), the gate table (32 KB).
// Tensor memory: the 128 x 128 accumulator.
// ===========================================================================
constexpr uint32_t O_STAGE = 4 * T8;
constexpr uint32_t O_OFF_BT = 2 * O_STAGE;
constexpr size_t kPrepSmem = O_OFF_BT + 4 * T8 + 1024;

__global__ void __launch_bounds__(256, 2)
    vgtc_prepare_kernel(const Dims d, const __grid_constant__ CUtensorMap mx,
                      const __grid_constant__ CUtensorMap my, const float* __restrict__ g,
                      float* __restrict__ M, float* __restrict__ out) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    float* bt = reinterpret_cast<float*>(smem + O_OFF_BT);
    __shared__ VgGate gs;
    __shared__ __align__(8) uint64_t full[2], mbar;
    __shared__ uint32_t tmem_slot;

    const Geo G = geo();
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;
    const int i = G.tid & 127, hf = G.tid >> 7;
    auto chunk_of = [&](int it) { return nch - 1 - it; };

    if (G.tid == 0) {
        mbar_init(smem_u32(&full[0]), 1);
        mbar_init(smem_u32(&full[1]), 1);
        mbar_init(smem_u32(&mbar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 128);
    float gp[32], bl[32];
    gate_fetch(d, g, b, h, a0 + chunk_of(0) * kChunk, G.tid, gp);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    auto load = [&](int it, int s) {
        const int row = b * d.T + a0 + chunk_of(it) * kChunk;
        const uint32_t bar = smem_u32(&full[s]);
        uint8_t* st = smem + s * O_STAGE;
        mbar_expect_tx(bar, O_STAGE);
        load_tile(st, &mx, 0, 128, h, row, bar);
        load_tile(st + 2 * T8, &my, 0, 128, h, row, bar);
    };
    if (G.tid == 0) {
        load(0, 0);
        if (nch > 1) load(1, 1);
    }
    float run = 0.f;  // sum of g[i] over the chunks already walked
    int seen = 0;     // a sequence starts in the chunks already walked
    for (int it = 0; it < nch; ++it) {
        const int s = it & 1;
        const int t0 = a0 + chunk_of(it) * kChunk;
        gate_build(d, t0, gp, bt, gs, G.tid, bl);
        if (it + 1 < nch) gate_fetch(d, g, b, h, a0 + chunk_of(it + 1) * kChunk, G.tid, gp);
        // this thread's weights replace its entries of the table
        const float B = gs.btot[i];
        const int lend = gs.ltot;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int t = 32 * hf + u;
            bt[t * kDk + i] = (!seen && gs.lid[t] == lend) ? __expf(run + B - bl[u]) : 0.f;
        }
        run += B;
        seen |= gs.any;
        __syncthreads();
        if (G.tid == 0 && it >= 1) {
            // the previous chunk's products are done: its stage takes chunk it + 1
            mbar_wait(smem_u32(&mbar), (it - 1) & 1);
            if (it + 1 < nch) load(it + 1, s ^ 1);
        }
        mbar_wait(smem_u32(&full[s]), (it >> 1) & 1);
        uint8_t* xs = smem + s * O_STAGE;
        scale_el(xs, G.tid, [&](int r, int c, float* x) {
            float w[8];
            ld8(bt + r * kDk + c, w);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] *= w[e];
        });
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (G.tid == 0) {
            const uint32_t xa = smem_u32(xs), ya = xa + 2 * T8;
            constexpr uint32_t idesc = idesc_bf16(128, 128, 1, 1);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16(tmem, sdesc(xa + k * 2048, T8, 1024), sdesc(ya + k * 2048, T8, 1024), idesc,
                         (it > 0 || k > 0) ? 1u : 0u);
            mma_commit(smem_u32(&mbar));
        }
    }
    mbar_wait(smem_u32(&mbar), (nch - 1) & 1);
    tc_fence_after();
    {
        float* dst = out + sum_off(d, seg, b, h) + int64_t(G.srow) * kDk + 64 * G.grp;
        float v[64];
        state_cols64(tmem, G, 0, v);
#pragma unroll
        for (int e = 0; e < 64; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    }
    if (hf == 0) M[((int64_t(seg) * d.B + b) * d.H + h) * kDk + i] = seen ? 0.f : expf(run);
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 128);
}

// ===========================================================================
// forward apply: o from S_in.
// Shared memory: two stages of Q|K|V (48 KB each), P, S (bf16), the gate table.
// Tensor memory: [0,64) scores, [64,192) O, [256,384) S.
// With TWO (more CTAs than SMs): two CTAs a SM, each with one input stage,
// the gate table in the S tile's bytes (the table's last reader, the
// scaling, is done before the state pass writes the tile) and O over the
// scores in 256 tensor-memory columns ([0,128) O, [128,256) S); a stage is
// refilled once the chunk's o rows have left it.
// Per chunk: gate tables; general chunks: exact scores into P; Q~, K~ in
// place; S *= W (bf16 tile: W S in factored chunks, S otherwise); factored
// chunks: scores = Q~ K~^T, causal mask into P; O = P V + Q~ S_tile,
// S += K~^T V; o rows into the dead Q tile and out by TMA.
// ===========================================================================
constexpr uint32_t A_STAGE = 6 * T8;
template <bool TWO> struct ApplyLayout {
    static constexpr int NST = TWO ? 1 : 2;
    static constexpr uint32_t OFF_P = NST * A_STAGE;
    static constexpr uint32_t OFF_S = OFF_P + T8;
    static constexpr uint32_t OFF_BT = TWO ? OFF_S : OFF_S + 4 * T8;
    static constexpr size_t SMEM = OFF_BT + 4 * T8 + 1024;
    static constexpr uint32_t TO = TWO ? 0 : 64, TS = TWO ? 128 : 256, TCOLS = TWO ? 256 : 512;
};

template <bool TWO>
__global__ void __launch_bounds__(256, TWO ? 2 : 1)
    vgtc_apply_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                      const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                      const __grid_constant__ CUtensorMap mo, const float* __restrict__ g,
                      const float* __restrict__ S_in) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    using LY = ApplyLayout<TWO>;
    uint8_t* Ps = smem + LY::OFF_P;
    uint8_t* Sb = smem + LY::OFF_S;
    float* bt = reinterpret_cast<float*>(smem + LY::OFF_BT);
    __shared__ VgGate gs;
    __shared__ __align__(8) uint64_t full[2], mbar;
    __shared__ uint32_t tmem_slot;
    constexpr uint32_t TO = LY::TO, TS = LY::TS;

    const Geo G = geo();
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        mbar_init(smem_u32(&full[0]), 1);
        mbar_init(smem_u32(&full[1]), 1);
        mbar_init(smem_u32(&mbar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), LY::TCOLS);
    float gp[32], bl[32];
    gate_fetch(d, g, b, h, a0, G.tid, gp);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    state_load(S_in + sum_off(d, seg, b, h), tmem, G, TS, nullptr);
    auto load = [&](int c, int s) {
        const int row = b * d.T + a0 + c * kChunk;
        const uint32_t bar = smem_u32(&full[s]);
        uint8_t* st = smem + s * A_STAGE;
        mbar_expect_tx(bar, A_STAGE);
        load_tile(st, &mq, 0, 128, h / d.qdiv, row, bar);
        load_tile(st + 2 * T8, &mk, 0, 128, h, row, bar);
        load_tile(st + 4 * T8, &mv, 0, 128, h, row, bar);
    };
    if (G.tid == 0) {
        load(0, 0);
        if (!TWO && nch > 1) load(1, 1);
    }
    const uint32_t sb0 = smem_u32(smem);
    const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, T8, 1024);
    const uint64_t pa = desc_plus(DK, LY::OFF_P), sa = desc_plus(sdesc(sb0, 2 * T8, 1024), LY::OFF_S);
    constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
    constexpr uint32_t id_o = idesc_bf16(64, 128, 0, 1);
    constexpr uint32_t id_s = idesc_bf16(128, 128, 1, 1);
    const Fac fac{bt, &gs, d.scale};
    uint32_t mph = 0;
    for (int c = 0; c < nch; ++c) {
        const int s = TWO ? 0 : (c & 1);
        uint8_t* Qs = smem + s * A_STAGE;
        uint8_t* Ks = Qs + 2 * T8;
        const bool fact = gate_build(d, a0 + c * kChunk, gp, bt, gs, G.tid, bl);
        if (!TWO && G.tid == 0 && c >= 1 && c + 1 < nch) {
            bulk_wait_read();  // the o store of chunk c - 1 has read its stage
            load(c + 1, s ^ 1);
        }
        mbar_wait(smem_u32(&full[s]), TWO ? (c & 1) : ((c >> 1) & 1));
        if (!fact) {  // from the raw tiles, before any thread scales them
            exact_scores(Qs, Ks, bt, gs, G.tau, 32 * G.grp + 16 * G.hi, d.scale, Ps);
            __syncthreads();
        }
        if (fact)
            scale_el(Qs, G.tid, [&](int r, int cc, float* x) { fac.q_fact(r, cc, x); });
        else
            scale_el(Qs, G.tid, [&](int r, int cc, float* x) { fac.q_win(r, cc, x); });
        scale_el(Ks, G.tid, [&](int r, int cc, float* x) { fac.k_wout(r, cc, x); });
        if (TWO) __syncthreads();  // the gate table's last reads before the S tile takes its bytes
        state_pass(tmem, G, TS, gs.any ? 0.f : expf(gs.btot[G.srow]), fact, Sb);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (fact) {
            if (G.tid == 0) {
                const uint64_t q = desc_plus(DK, s * A_STAGE), kk = desc_plus(q, 2 * T8);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t off = (k >> 2) * T8 + (k & 3) * 32;
                    mma_bf16(tmem, desc_plus(q, off), desc_plus(kk, off), id1, k > 0);
                }
                mma_commit(smem_u32(&mbar));
            }
            mbar_wait(smem_u32(&mbar), mph);
            mph ^= 1;
            tc_fence_after();
            float x[16];
            tok16(tmem, G, 32 * G.grp, x);
            const int c0 = 32 * G.grp + 16 * G.hi;
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = c0 + e <= G.tau ? x[e] : 0.f;
            store_row16(Ps, G.tau, c0, x);
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }
        if (G.tid == 0) {
            const uint64_t q = desc_plus(DK, s * A_STAGE);
            const uint64_t km = desc_plus(DM, s * A_STAGE + 2 * T8), vm = desc_plus(DM, s * A_STAGE + 4 * T8);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // O = P V
                mma_bf16(tmem + TO, desc_plus(pa, k * 32), desc_plus(vm, k * 2048), id_o, k > 0);
#pragma unroll
            for (int k = 0; k < 8; ++k)  // O += Q~ S_tile
                mma_bf16(tmem + TO, desc_plus(q, (k >> 2) * T8 + (k & 3) * 32), desc_plus(sa, k * 2048), id_o, 1u);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // S += K~^T V
                mma_bf16(tmem + TS, desc_plus(km, k * 2048), desc_plus(vm, k * 2048), id_s, 1u);
            mma_commit(smem_u32(&mbar));
        }
        // the next chunk's gates, loaded while the products run
        if (c + 1 < nch) gate_fetch(d, g, b, h, a0 + (c + 1) * kChunk, G.tid, gp);
        mbar_wait(smem_u32(&mbar), mph);
        mph ^= 1;
        tc_fence_after();
        {
            float xx[2][16];
            tok16x2(tmem, G, TO + 64 * G.grp, TO + 64 * G.grp + 32, xx[0], xx[1]);
#pragma unroll
            for (int k = 0; k < 2; ++k) store_row16(Qs, G.tau, 64 * G.grp + 32 * k + 16 * G.hi, xx[k]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (G.tid == 0) {
            store_tile(&mo, Qs, h, b * d.T + a0 + c * kChunk);
            bulk_commit();
            if (TWO && c + 1 < nch) {
                bulk_wait_read();  // the o store has read the stage
                load(c + 1, 0);
            }
        }
    }
    if (G.tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, LY::TCOLS);
}

// ===========================================================================
// backward prepare in one sweep from S_in: dq, gamma and qdq[t][i] = q_t[i]
// (dq_t[i] minus its same-token term scale (dO_t . v_t) k_t[i]).
//   factored: X = mask(A) K~ + dO S'^T with A = dO V^T (s <= t), K~ and
//             S' = W S_prev as in the forward; dq = scale exp(b_t - B) X
//   general:  X = dO S_prev^T; dq = scale (win X + sum_{s <= t} A k_s
//             exp(b_t - b_s)) with the sum taken directly
//   gamma += Qh^T dO, Qh = Q scaled in place by scale exp(sum of g over
//             [segment start, t]) (0 once a sequence starts there); the
//             epilogue reads raw q from global memory
// Shared memory: two stages of Q|K|V|dO (64 KB each), K~ (16 KB), A (bf16),
// S (bf16), the gate table.  dq is staged in the dead V tile.
// Tensor memory: [0,64) A, [128,256) X, [256,384) S, [384,512) gamma.
// ===========================================================================
constexpr uint32_t Q_STAGE = 8 * T8;
constexpr uint32_t Q_OFF_KT = 2 * Q_STAGE;
constexpr uint32_t Q_OFF_P = Q_OFF_KT + 2 * T8;
constexpr uint32_t Q_OFF_S = Q_OFF_P + T8;
constexpr uint32_t Q_OFF_BT = Q_OFF_S + 4 * T8;
constexpr size_t kDqSmem = Q_OFF_BT + 4 * T8 + 1024;

// Direct intra-chunk dq terms of a general chunk for 16 columns i = cc..cc+15
// of row tau: hist[u] = sum_{s < tau, same sequence} A[tau][s] k_s[i]
// exp(b_tau[i] - b_s[i]) (A from the masked bf16 tile) and the s = tau term
// diag[u] = A[tau][tau] k_tau[i].
__device__ __noinline__ void exact_dq16(const uint8_t* Ps, const uint8_t* Ks, const float* bt,
                                        const VgGate& gs, int tau, int cc, float* hist, float* diag) {
    float bq[16];
    ld8(bt + tau * kDk + cc, bq);
    ld8(bt + tau * kDk + cc + 8, bq + 8);
#pragma unroll
    for (int u = 0; u < 16; ++u) hist[u] = 0.f;
    const int lt = gs.lid[tau];
#pragma unroll 1
    for (int s = 0; s < tau; ++s) {
        if (gs.lid[s] != lt) continue;
        const float a = tile_el(Ps, tau, s);
        float kv[16], bs[16];
        tile_row_get16(Ks, s, cc, kv);
        ld8(bt + s * kDk + cc, bs);
        ld8(bt + s * kDk + cc + 8, bs + 8);
#pragma unroll
        for (int u = 0; u < 16; ++u) hist[u] = fmaf(a * kv[u], __expf(bq[u] - bs[u]), hist[u]);
    }
    float kt[16];
    tile_row_get16(Ks, tau, cc, kt);
    const float att = tile_el(Ps, tau, tau);
#pragma unroll
    for (int u = 0; u < 16; ++u) diag[u] = att * kt[u];
}

__global__ void __launch_bounds__(256, 1)
    vgtc_dq_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                   const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                   const __grid_constant__ CUtensorMap mdo, const __grid_constant__ CUtensorMap mdq,
                   const __nv_bfloat16* __restrict__ q, const float* __restrict__ g,
                   const float* __restrict__ S_in, float* __restrict__ gamma, float* __restrict__ qdq) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Kt = smem + Q_OFF_KT;
    uint8_t* Ps = smem + Q_OFF_P;
    uint8_t* Sb = smem + Q_OFF_S;
    float* bt = reinterpret_cast<float*>(smem + Q_OFF_BT);
    __shared__ VgGate gs;
    __shared__ __align__(8) uint64_t full[2], abar, mbar;
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(16) float run_s[kDk];  // sum of g[i] over the segment's chunks before this one (read as float4)
    constexpr uint32_t TX = 128, TS = 256, TG = 384;

    const Geo G = geo();
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        mbar_init(smem_u32(&full[0]), 1);
        mbar_init(smem_u32(&full[1]), 1);
        mbar_init(smem_u32(&abar), 1);
        mbar_init(smem_u32(&mbar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
    float gp[32], bl[32];
    gate_fetch(d, g, b, h, a0, G.tid, gp);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    state_load(S_in + sum_off(d, seg, b, h), tmem, G, TS, nullptr);
    auto load = [&](int c, int s) {
        const int row = b * d.T + a0 + c * kChunk;
        const uint32_t bar = smem_u32(&full[s]);
        uint8_t* st = smem + s * Q_STAGE;
        mbar_expect_tx(bar, Q_STAGE);
        load_tile(st, &mq, 0, 128, h / d.qdiv, row, bar);
        load_tile(st + 2 * T8, &mk, 0, 128, h, row, bar);
        load_tile(st + 4 * T8, &mv, 0, 128, h, row, bar);
        load_tile(st + 6 * T8, &mdo, 0, 128, h, row, bar);
    };
    if (G.tid == 0) {
        load(0, 0);
        if (nch > 1) load(1, 1);
    }
    const uint32_t sb0 = smem_u32(smem);
    const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, T8, 1024);
    const uint64_t pa = desc_plus(DK, Q_OFF_P), sa = desc_plus(DK, Q_OFF_S), ktm = desc_plus(DM, Q_OFF_KT);
    constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
    constexpr uint32_t id_a = idesc_bf16(64, 128, 0, 1);
    constexpr uint32_t id_b = idesc_bf16(64, 128, 0, 0);
    constexpr uint32_t id_s = idesc_bf16(128, 128, 1, 1);
    const Fac fac{bt, &gs, d.scale};
    if (G.tid < kDk) run_s[G.tid] = 0.f;
    int seen = 0;  // a sequence starts in the segment's chunks before this one
    uint32_t aph = 0, mph = 0;
    for (int c = 0; c < nch; ++c) {
        const int s = c & 1;
        uint8_t* Qs = smem + s * Q_STAGE;
        uint8_t* Ks = Qs + 2 * T8;
        uint8_t* Vs = Qs + 4 * T8;
        const bool fact = gate_build(d, a0 + c * kChunk, gp, bt, gs, G.tid, bl);
        if (G.tid == 0) {
            if (c >= 1 && c + 1 < nch) {
                bulk_wait_read();  // the dq store of chunk c - 1 has read its stage
                load(c + 1, s ^ 1);
            }
            mbar_wait(smem_u32(&full[s]), (c >> 1) & 1);
            tc_fence_after();
            const uint64_t v = desc_plus(DK, s * Q_STAGE + 4 * T8), o = desc_plus(DK, s * Q_STAGE + 6 * T8);
#pragma unroll
            for (int k = 0; k < 8; ++k) {  // A = dO V^T
                const uint32_t off = (k >> 2) * T8 + (k & 3) * 32;
                mma_bf16(tmem, desc_plus(o, off), desc_plus(v, off), id1, k > 0);
            }
            mma_commit(smem_u32(&abar));
        }
        mbar_wait(smem_u32(&full[s]), (c >> 1) & 1);
        // K~ (for the state, and for A K~ in factored chunks) into its own tile
        {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int n = G.tid + 256 * k;
                const uint32_t off = (n >> 9) * T8 + ((n >> 3) & 63) * 128 + (n & 7) * 16;
                *reinterpret_cast<uint4*>(Kt + off) = *reinterpret_cast<const uint4*>(Ks + off);
            }
            scale_el(Kt, G.tid, [&](int r, int cc, float* x) { fac.k_wout(r, cc, x); });
            // gamma's A operand in place of Q: scale exp(sum of g over [segment start, t])
            // while no sequence starts in [segment start, t], else 0
            const bool open = !seen && !gs.first;
            scale_el(Qs, G.tid, [&](int r, int cc, float* x) {
                const bool keep = open && gs.lid[r] == 0;
                float bb[8], rr[8];
                ld8(bt + r * kDk + cc, bb);
                ld8(run_s + cc, rr);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = keep ? x[e] * d.scale * __expf(rr[e] + bb[e]) : 0.f;
            });
        }
        state_pass(tmem, G, TS, gs.any ? 0.f : expf(gs.btot[G.srow]), fact, Sb);
        mbar_wait(smem_u32(&abar), aph);
        aph ^= 1;
        tc_fence_after();
        {
            float x[16];
            tok16(tmem, G, 32 * G.grp, x);
            const int c0 = 32 * G.grp + 16 * G.hi;
            const int lt = gs.lid[G.tau];
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = (c0 + e <= G.tau && gs.lid[c0 + e] == lt) ? x[e] : 0.f;
            store_row16(Ps, G.tau, c0, x);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (G.tid == 0) {
            const uint64_t o = desc_plus(DK, s * Q_STAGE + 6 * T8), vm = desc_plus(DM, s * Q_STAGE + 4 * T8);
            if (fact) {
#pragma unroll
                for (int k = 0; k < 4; ++k)  // X = A K~
                    mma_bf16(tmem + TX, desc_plus(pa, k * 32), desc_plus(ktm, k * 2048), id_a, k > 0);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k)  // X += dO S_tile^T
                mma_bf16(tmem + TX, desc_plus(o, (k >> 2) * T8 + (k & 3) * 32),
                         desc_plus(sa, (k >> 2) * 2 * T8 + (k & 3) * 32), id_b, (fact || k > 0) ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // S += K~^T V
                mma_bf16(tmem + TS, desc_plus(ktm, k * 2048), desc_plus(vm, k * 2048), id_s, 1u);
            const uint64_t qhm = desc_plus(DM, s * Q_STAGE), om = desc_plus(DM, s * Q_STAGE + 6 * T8);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // gamma += Qh^T dO
                mma_bf16(tmem + TG, desc_plus(qhm, k * 2048), desc_plus(om, k * 2048), id_s,
                         (c > 0 || k > 0) ? 1u : 0u);
            mma_commit(smem_u32(&mbar));
        }
        if (G.tid < kDk) run_s[G.tid] += gs.btot[G.tid];  // every scaling has read run_s
        seen |= gs.any;
        // the next chunk's gates and this thread's raw q (the Q tile holds
        // gamma's operand), loaded while the products run
        if (c + 1 < nch) gate_fetch(d, g, b, h, a0 + (c + 1) * kChunk, G.tid, gp);
        uint4 q4[2][2];
        {
            const __nv_bfloat16* qp = q + q_off(d, b, a0 + c * kChunk + G.tau, h) + 64 * G.grp + 16 * G.hi;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                q4[k][0] = *reinterpret_cast<const uint4*>(qp + 32 * k);
                q4[k][1] = *reinterpret_cast<const uint4*>(qp + 32 * k + 8);
            }
        }
        mbar_wait(smem_u32(&mbar), mph);
        mph ^= 1;
        tc_fence_after();
        {
            const int t = a0 + c * kChunk + G.tau;
            float* qrow = qdq + gv_off(d, b, t, h);
            const float att = tile_el(Ps, G.tau, G.tau);  // as the product saw it
            const bool keep_in = !gs.first && gs.lid[G.tau] == 0;
            float xx[2][16];
            tok16x2(tmem, G, TX + 64 * G.grp, TX + 64 * G.grp + 32, xx[0], xx[1]);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int cc = 64 * G.grp + 32 * k + 16 * G.hi;
                float* x = xx[k];
                float qv[16], bq[16], out[16];
                unpack8(q4[k][0], qv);
                unpack8(q4[k][1], qv + 8);
                ld8(bt + G.tau * kDk + cc, bq);
                ld8(bt + G.tau * kDk + cc + 8, bq + 8);
                if (fact) {
                    float kt[16], B[16];
                    tile_row_get16(Kt, G.tau, cc, kt);
                    ld8(gs.btot + cc, B);
                    ld8(gs.btot + cc + 8, B + 8);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float f = d.scale * __expf(bq[u] - B[u]);
                        out[u] = qv[u] * f * (x[u] - att * kt[u]);
                        x[u] *= f;
                    }
                } else {
                    float hist[16], diag[16];
                    exact_dq16(Ps, Ks, bt, gs, G.tau, cc, hist, diag);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float hi = hist[u] + (keep_in ? __expf(bq[u]) * x[u] : 0.f);
                        out[u] = qv[u] * d.scale * hi;
                        x[u] = d.scale * (hi + diag[u]);
                    }
                }
                store_row16(Vs, G.tau, cc, x);
#pragma unroll
                for (int u = 0; u < 16; u += 4)
                    *reinterpret_cast<float4*>(qrow + cc + u) = make_float4(out[u], out[u + 1], out[u + 2], out[u + 3]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (G.tid == 0) {
            store_tile(&mdq, Vs, h, b * d.T + a0 + c * kChunk);
            bulk_commit();
        }
    }
    {   // gamma rows (every product has completed)
        float* dst = gamma + sum_off(d, seg, b, h) + int64_t(G.srow) * kDk + 64 * G.grp;
        float v[64];
        state_cols64(tmem, G, TG, v);
#pragma unroll
        for (int e = 0; e < 64; e += 4)
            *reinterpret_cast<float4*>(dst + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    }
    if (G.tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 512);
}

// ===========================================================================
// backward apply, the reverse sweep: dk, dv, dg from dS_out (chunks walked
// from the segment end).  E is the adjoint arriving at the chunk's last
// state (dS_out at the segment end).
//   factored: P = mask(Q~ K~^T), A' = dO V^T (r >= s, as A'^T);
//             dk = exp(B - b_s) (A'^T Q~ + V E^T), dv = P^T dO + K~ E,
//             E <- W (E + Q~^T dO)
//   general:  P and the intra-chunk dk terms directly; dk = intra + wout V E^T,
//             dv = P^T dO + K~ E, E <- W E + (scale Q o win)^T dO
// dg: c_s[i] = qdq[s][i] - k_s[i] (dk_s[i] - scale A'[s][s] q_s[i]); the
// running sums R = U c (U[s][r] = 1 for r >= s in s's sequence) on the tensor
// cores with c split as bf16 c_hi + c_lo, plus the carry from later chunks.
// Shared memory: two stages of Q|K|V|dO (64 KB each), P (then U), A', E
// (bf16), the gate table.  dk is staged in the dead V tile, dv in dO, c_hi
// and c_lo in Q and K.
// Tensor memory: [0,64) P, [64,128) A', [128,256) dk (then R), [256,384) dv,
// [384,512) E.
// ===========================================================================
constexpr uint32_t R_STAGE = 8 * T8;
constexpr uint32_t R_OFF_P = 2 * R_STAGE;
constexpr uint32_t R_OFF_PD = R_OFF_P + T8;
constexpr uint32_t R_OFF_E = R_OFF_PD + T8;
constexpr uint32_t R_OFF_BT = R_OFF_E + 4 * T8;
constexpr size_t kRevSmem = R_OFF_BT + 4 * T8 + 1024;

// Direct intra-chunk dk terms of a general chunk for 16 columns i = cc..cc+15
// of row s = tau: sum_{r >= tau, same sequence} A'[r][tau] scale q_r[i]
// exp(b_r[i] - b_tau[i]) (A' from the masked bf16 tile; q read from global
// memory, since the Q tile holds Q o win by now).
__device__ __noinline__ void exact_dk16(const Dims& d, const __nv_bfloat16* __restrict__ q, int b, int h,
                                        int t0, const uint8_t* PD, const float* bt, const VgGate& gs, int tau,
                                        int cc, float* acc) {
    float bs[16];
    ld8(bt + tau * kDk + cc, bs);
    ld8(bt + tau * kDk + cc + 8, bs + 8);
#pragma unroll
    for (int u = 0; u < 16; ++u) acc[u] = 0.f;
    const int lt = gs.lid[tau];
#pragma unroll 1
    for (int r = tau; r < kChunk; ++r) {
        if (gs.lid[r] != lt) break;  // later tokens belong to later sequences
        const float a = tile_el(PD, r, tau) * d.scale;
        const __nv_bfloat16* qr = q + q_off(d, b, t0 + r, h) + cc;
        float qv[16], br[16];
        unpack8(*reinterpret_cast<const uint4*>(qr), qv);
        unpack8(*reinterpret_cast<const uint4*>(qr + 8), qv + 8);
        ld8(bt + r * kDk + cc, br);
        ld8(bt + r * kDk + cc + 8, br + 8);
#pragma unroll
        for (int u = 0; u < 16; ++u) acc[u] = fmaf(a * qv[u], __expf(br[u] - bs[u]), acc[u]);
    }
}

__global__ void __launch_bounds__(256, 1)
    vgtc_rev_kernel(const Dims d, const __grid_constant__ CUtensorMap mq,
                    const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                    const __grid_constant__ CUtensorMap mdo, const __grid_constant__ CUtensorMap mdk,
                    const __grid_constant__ CUtensorMap mdv, const __nv_bfloat16* __restrict__ q,
                    const __nv_bfloat16* __restrict__ k, const float* __restrict__ g,
                    const float* __restrict__ S_in, const float* __restrict__ dS_out,
                    const float* __restrict__ qdq, float* __restrict__ dg) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* Ps = smem + R_OFF_P;
    uint8_t* PD = smem + R_OFF_PD;
    uint8_t* Eb = smem + R_OFF_E;
    float* bt = reinterpret_cast<float*>(smem + R_OFF_BT);
    __shared__ VgGate gs;
    __shared__ __align__(8) uint64_t full[2], abar, mbar;
    __shared__ uint32_t tmem_slot;
    __shared__ float carry[2][kDk];   // running dg sum carried into the chunk, by parity
    __shared__ float ext_part[2][kDk];
    constexpr uint32_t TP = 0, TA = 64, TK = 128, TV = 256, TE = 384;

    const Geo G = geo();
    const int seg = blockIdx.x, b = blockIdx.y / d.H, h = blockIdx.y % d.H;
    const int nch = d.L / kChunk;
    const int a0 = seg * d.L;

    if (G.tid == 0) {
        mbar_init(smem_u32(&full[0]), 1);
        mbar_init(smem_u32(&full[1]), 1);
        mbar_init(smem_u32(&abar), 1);
        mbar_init(smem_u32(&mbar), 1);
        mbar_fence_init();
    }
    if (G.warp == 0) tmem_alloc(smem_u32(&tmem_slot), 512);
    float gp[32], bl[32];
    gate_fetch(d, g, b, h, a0 + (nch - 1) * kChunk, G.tid, gp);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    state_load(dS_out + sum_off(d, seg, b, h), tmem, G, TE, Eb);
    {   // carry into the last chunk: <S_out[i,:], dS_out[i,:]> (S_out read as S_in[seg+1])
        float e = 0.f;
        if (seg + 1 < d.nseg) {
            const float* so = S_in + sum_off(d, seg + 1, b, h) + int64_t(G.srow) * kDk + 64 * G.grp;
            const float* dso = dS_out + sum_off(d, seg, b, h) + int64_t(G.srow) * kDk + 64 * G.grp;
#pragma unroll 4
            for (int j = 0; j < 64; j += 4) {
                const float4 x = *reinterpret_cast<const float4*>(so + j);
                const float4 y = *reinterpret_cast<const float4*>(dso + j);
                e = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, e))));
            }
        }
        ext_part[G.grp][G.srow] = e;
    }
    auto load = [&](int it, int s) {
        const int row = b * d.T + a0 + (nch - 1 - it) * kChunk;
        const uint32_t bar = smem_u32(&full[s]);
        uint8_t* st = smem + s * R_STAGE;
        mbar_expect_tx(bar, R_STAGE);
        load_tile(st, &mq, 0, 128, h / d.qdiv, row, bar);
        load_tile(st + 2 * T8, &mk, 0, 128, h, row, bar);
        load_tile(st + 4 * T8, &mv, 0, 128, h, row, bar);
        load_tile(st + 6 * T8, &mdo, 0, 128, h, row, bar);
    };
    if (G.tid == 0) {
        load(0, 0);
        if (nch > 1) load(1, 1);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (G.tid < kDk) carry[0][G.tid] = ext_part[0][G.tid] + ext_part[1][G.tid];
    const uint32_t sb0 = smem_u32(smem);
    const uint64_t DK = sdesc(sb0, 16, 1024), DM = sdesc(sb0, T8, 1024), DM2 = sdesc(sb0, 2 * T8, 1024);
    const uint64_t pk = desc_plus(DK, R_OFF_P), pm = desc_plus(DM, R_OFF_P), pdm = desc_plus(DM, R_OFF_PD);
    const uint64_t ek = desc_plus(DK, R_OFF_E), em = desc_plus(DM2, R_OFF_E);
    constexpr uint32_t id1 = idesc_bf16(64, 64, 0, 0);
    constexpr uint32_t id_mm = idesc_bf16(64, 128, 1, 1);
    constexpr uint32_t id_kk = idesc_bf16(64, 128, 0, 0);
    constexpr uint32_t id_km = idesc_bf16(64, 128, 0, 1);
    constexpr uint32_t id_e = idesc_bf16(128, 128, 1, 1);
    const Fac fac{bt, &gs, d.scale};
    uint32_t aph = 0, mph = 0;
    for (int it = 0; it < nch; ++it) {
        const int s = it & 1, p = it & 1;
        const int cidx = nch - 1 - it;
        const int t0 = a0 + cidx * kChunk;
        uint8_t* Qs = smem + s * R_STAGE;
        uint8_t* Ks = Qs + 2 * T8;
        uint8_t* Vs = Qs + 4 * T8;
        uint8_t* Ds = Qs + 6 * T8;
        const bool fact = gate_build(d, t0, gp, bt, gs, G.tid, bl);
        if (G.tid == 0) {
            if (it >= 1 && it + 1 < nch) {
                bulk_wait_read();  // the dk, dv stores of the previous chunk have read its stage
                load(it + 1, s ^ 1);
            }
            mbar_wait(smem_u32(&full[s]), (it >> 1) & 1);
            tc_fence_after();
            const uint64_t v = desc_plus(DK, s * R_STAGE + 4 * T8), o = desc_plus(DK, s * R_STAGE + 6 * T8);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // A' = dO V^T
                const uint32_t off = (kk >> 2) * T8 + (kk & 3) * 32;
                mma_bf16(tmem + TA, desc_plus(o, off), desc_plus(v, off), id1, kk > 0);
            }
            mma_commit(smem_u32(&abar));
        }
        mbar_wait(smem_u32(&full[s]), (it >> 1) & 1);
        if (!fact) {  // from the raw tiles, before any thread scales them
            exact_scores(Qs, Ks, bt, gs, G.tau, 32 * G.grp + 16 * G.hi, d.scale, Ps);
            __syncthreads();
        }
        if (fact)
            scale_el(Qs, G.tid, [&](int r, int cc, float* x) { fac.q_fact(r, cc, x); });
        else
            scale_el(Qs, G.tid, [&](int r, int cc, float* x) { fac.q_win(r, cc, x); });
        scale_el(Ks, G.tid, [&](int r, int cc, float* x) { fac.k_wout(r, cc, x); });
        if (!fact) {  // E *= W ahead of E += (scale Q o win)^T dO; the bf16 tile keeps E
            const float w = gs.any ? 0.f : expf(gs.btot[G.srow]);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t r[32];
                tmem_ld32_nowait(tmem + G.tl + TE + 64 * G.grp + 32 * hf, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(w * __uint_as_float(r[e]));
                tmem_st32(tmem + G.tl + TE + 64 * G.grp + 32 * hf, r);
            }
            tmem_wait_st();
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (fact && G.tid == 0) {
            const uint64_t qq = desc_plus(DK, s * R_STAGE), kk2 = desc_plus(qq, 2 * T8);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // P = Q~ K~^T
                const uint32_t off = (kk >> 2) * T8 + (kk & 3) * 32;
                mma_bf16(tmem + TP, desc_plus(qq, off), desc_plus(kk2, off), id1, kk > 0);
            }
            mma_commit(smem_u32(&mbar));
        }
        mbar_wait(smem_u32(&abar), aph);
        aph ^= 1;
        if (fact) {
            mbar_wait(smem_u32(&mbar), mph);
            mph ^= 1;
        }
        tc_fence_after();
        {
            const int c0 = 32 * G.grp + 16 * G.hi;
            const int lt = gs.lid[G.tau];
            float xa[16];
            tok16(tmem, G, TA + 32 * G.grp, xa);
            // A' stored as [r][s] with r = tau: keep s <= r in r's sequence
#pragma unroll
            for (int e = 0; e < 16; ++e) xa[e] = (c0 + e <= G.tau && gs.lid[c0 + e] == lt) ? xa[e] : 0.f;
            store_row16(PD, G.tau, c0, xa);
            if (fact) {
                float xp[16];
                tok16(tmem, G, TP + 32 * G.grp, xp);
#pragma unroll
                for (int e = 0; e < 16; ++e) xp[e] = c0 + e <= G.tau ? xp[e] : 0.f;
                store_row16(Ps, G.tau, c0, xp);
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (G.tid == 0) {
            const uint64_t qm = desc_plus(DM, s * R_STAGE), om = desc_plus(DM, s * R_STAGE + 6 * T8);
            const uint64_t vk = desc_plus(DK, s * R_STAGE + 4 * T8), kk2 = desc_plus(DK, s * R_STAGE + 2 * T8);
            if (fact) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // dk = A'^T Q~
                    mma_bf16(tmem + TK, desc_plus(pdm, kk * 2048), desc_plus(qm, kk * 2048), id_mm, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // dk += V E^T
                const uint32_t off = (kk >> 2) * T8 + (kk & 3) * 32;
                mma_bf16(tmem + TK, desc_plus(vk, off), desc_plus(ek, 2 * off - (kk & 3) * 32), id_kk,
                         (fact || kk > 0) ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // dv = P^T dO
                mma_bf16(tmem + TV, desc_plus(pm, kk * 2048), desc_plus(om, kk * 2048), id_mm, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // dv += K~ E
                mma_bf16(tmem + TV, desc_plus(kk2, (kk >> 2) * T8 + (kk & 3) * 32), desc_plus(em, kk * 2048),
                         id_km, 1u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // E += Q~^T dO
                mma_bf16(tmem + TE, desc_plus(qm, kk * 2048), desc_plus(om, kk * 2048), id_e, 1u);
            mma_commit(smem_u32(&mbar));
        }
        // the previous chunk's gates and this thread's q.dq values, loaded
        // while the products run
        if (it + 1 < nch) gate_fetch(d, g, b, h, t0 - kChunk, G.tid, gp);
        float4 qd4[2][4];
        {
            const float* qrow = qdq + gv_off(d, b, t0 + G.tau, h);
#pragma unroll
            for (int kq = 0; kq < 2; ++kq)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    qd4[kq][u] = *reinterpret_cast<const float4*>(qrow + 64 * G.grp + 32 * kq + 16 * G.hi + 4 * u);
        }
        mbar_wait(smem_u32(&mbar), mph);
        mph ^= 1;
        tc_fence_after();
        {   // dk rows (staged in V), the dg summands c (split into Q and K)
            const int t = t0 + G.tau;
            const float att = tile_el(PD, G.tau, G.tau);  // as the products saw it
            const bool keep_out = gs.lid[G.tau] == gs.ltot;
            float xx[2][16];
            tok16x2(tmem, G, TK + 64 * G.grp, TK + 64 * G.grp + 32, xx[0], xx[1]);
#pragma unroll
            for (int kq = 0; kq < 2; ++kq) {
                const int cc = 64 * G.grp + 32 * kq + 16 * G.hi;
                float* x = xx[kq];
                float bq[16], B[16], qd[16], cs[16];
                ld8(bt + G.tau * kDk + cc, bq);
                ld8(bt + G.tau * kDk + cc + 8, bq + 8);
                ld8(gs.btot + cc, B);
                ld8(gs.btot + cc + 8, B + 8);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 y = qd4[kq][u];
                    qd[4 * u] = y.x; qd[4 * u + 1] = y.y; qd[4 * u + 2] = y.z; qd[4 * u + 3] = y.w;
                }
                if (fact) {
                    float qt[16], kt[16];
                    tile_row_get16(Qs, G.tau, cc, qt);
                    tile_row_get16(Ks, G.tau, cc, kt);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        cs[u] = qd[u] - kt[u] * (x[u] - att * qt[u]);
                        x[u] *= __expf(B[u] - bq[u]);
                    }
                } else {
                    float intra[16], qr[16], kr[16];
                    exact_dk16(d, q, b, h, t0, PD, bt, gs, G.tau, cc, intra);
                    const __nv_bfloat16* qp = q + q_off(d, b, t, h) + cc;
                    const __nv_bfloat16* kp = k + qk_off(d, b, t, h) + cc;
                    unpack8(*reinterpret_cast<const uint4*>(qp), qr);
                    unpack8(*reinterpret_cast<const uint4*>(qp + 8), qr + 8);
                    unpack8(*reinterpret_cast<const uint4*>(kp), kr);
                    unpack8(*reinterpret_cast<const uint4*>(kp + 8), kr + 8);
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const float dk = intra[u] + (keep_out ? __expf(B[u] - bq[u]) * x[u] : 0.f);
                        cs[u] = qd[u] - kr[u] * (dk - att * d.scale * qr[u]);
                        x[u] = dk;
                    }
                }
                store_row16(Vs, G.tau, cc, x);
                float hi[16], lo[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    hi[u] = bf16_round(cs[u]);
                    lo[u] = cs[u] - hi[u];
                }
                store_row16(Qs, G.tau, cc, hi);
                store_row16(Ks, G.tau, cc, lo);
            }
        }
        {   // dv rows (staged in dO)
            float xx[2][16];
            tok16x2(tmem, G, TV + 64 * G.grp, TV + 64 * G.grp + 32, xx[0], xx[1]);
#pragma unroll
            for (int kq = 0; kq < 2; ++kq) store_row16(Ds, G.tau, 64 * G.grp + 32 * kq + 16 * G.hi, xx[kq]);
        }
        // adjoint for the chunk before: factored E <- W E (tensor memory and tile);
        // general: E already carries W, the tile takes it as is
        state_pass(tmem, G, TE, fact ? (gs.any ? 0.f : expf(gs.btot[G.srow])) : 1.f, true, Eb);
        {   // U[s][r] = 1 for r >= s in s's sequence, into the P tile
            const int c0 = 32 * G.grp + 16 * G.hi;
            const int lt = gs.lid[G.tau];
            float u16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) u16[e] = (c0 + e >= G.tau && gs.lid[c0 + e] == lt) ? 1.f : 0.f;
            store_row16(Ps, G.tau, c0, u16);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (G.tid == 0) {
            const int row = b * d.T + t0;
            store_tile(&mdk, Vs, h, row);
            store_tile(&mdv, Ds, h, row);
            bulk_commit();
            const uint64_t chm = desc_plus(DM, s * R_STAGE), clm = desc_plus(DM, s * R_STAGE + 2 * T8);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // R = U c_hi
                mma_bf16(tmem + TK, desc_plus(pk, kk * 32), desc_plus(chm, kk * 2048), id_km, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // R += U c_lo
                mma_bf16(tmem + TK, desc_plus(pk, kk * 32), desc_plus(clm, kk * 2048), id_km, 1u);
            mma_commit(smem_u32(&mbar));
        }
        mbar_wait(smem_u32(&mbar), mph);
        mph ^= 1;
        tc_fence_after();
        {   // dg rows: R plus the carry for the sequence open at the chunk end
            const int t = t0 + G.tau;
            float* drow = dg + gv_off(d, b, t, h);
            const bool open = gs.lid[G.tau] == gs.ltot;
            const bool start = G.tau == 0 ? gs.first != 0 : gs.lid[G.tau] != gs.lid[G.tau - 1];
            float xx[2][16];
            tok16x2(tmem, G, TK + 64 * G.grp, TK + 64 * G.grp + 32, xx[0], xx[1]);
#pragma unroll
            for (int kq = 0; kq < 2; ++kq) {
                const int cc = 64 * G.grp + 32 * kq + 16 * G.hi;
                float* x = xx[kq];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float v = x[u] + (open ? carry[p][cc + u] : 0.f);
                    x[u] = start ? 0.f : v;
                    if (G.tau == 0) carry[p ^ 1][cc + u] = x[u];  // 0 when position 0 starts a sequence
                }
#pragma unroll
                for (int u = 0; u < 16; u += 4)
                    *reinterpret_cast<float4*>(drow + cc + u) = make_float4(x[u], x[u + 1], x[u + 2], x[u + 3]);
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (G.tid == 0) bulk_wait_all();
    tc_fence_before();
    __syncthreads();
    if (G.warp == 0) tmem_dealloc(tmem, 512);
}

__global__ void read_flag_kernel(int* out, int clear) {
    *out = g_timeout_flag;
    if (clear) g_timeout_flag = 0;
}

}  // namespace
}  // namespace vgtc

bool vgtc_supports(const Dims& d, rm_dtype dt) {
    return d.vg && dt == RM_BF16 && d.Dk == 128 && d.Dv == 128 && d.L % tc::kChunk == 0 &&
           d.T >= tc::kChunk;
}

rm_status launch_vgtc(Op op, const Dims& d, const Ptrs& p, cudaStream_t s) {
    using namespace vgtc;
    if (!vgtc_supports(d, RM_BF16)) return RM_ERR_UNSUPPORTED;
    const dim3 grid(d.nseg, d.B * d.H);
    CUtensorMap mq, mk, mv, mdo;
    switch (op) {
        case Op::kForwardPrepare: {
            if (!make_map(&mk, p.k, d, 128) || !make_map(&mv, p.v, d, 128)) return RM_ERR_CUDA;
            auto fn = vgtc_prepare_kernel;
            if (!set_smem(fn, kPrepSmem)) return RM_ERR_CUDA;
            fn<<<grid, 256, kPrepSmem, s>>>(d, mk, mv, p.g, p.M, p.sum_out);
            break;
        }
        case Op::kForwardApply: {
            CUtensorMap mo;
            if (!make_map(&mq, p.q, d, 128, d.qh) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, 128) || !make_map(&mo, p.out0, d, 128))
                return RM_ERR_CUDA;
            // more CTAs than SMs: two a SM (one input stage each), else one
            // with two stages
            const bool two = int64_t(grid.x) * grid.y > sm_count();
            auto fn = two ? vgtc_apply_kernel<true> : vgtc_apply_kernel<false>;
            const size_t sm = two ? ApplyLayout<true>::SMEM : ApplyLayout<false>::SMEM;
            if (!set_smem(fn, sm)) return RM_ERR_CUDA;
            fn<<<grid, 256, sm, s>>>(d, mq, mk, mv, mo, p.g, p.S_in);
            break;
        }
        case Op::kBackwardPrepare: {
            CUtensorMap mdq;
            if (!make_map(&mq, p.q, d, 128, d.qh) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, 128) || !make_map(&mdo, p.dO, d, 128) || !make_map(&mdq, p.out0, d, 128))
                return RM_ERR_CUDA;
            auto fq = vgtc_dq_kernel;
            if (!set_smem(fq, kDqSmem)) return RM_ERR_CUDA;
            fq<<<grid, 256, kDqSmem, s>>>(d, mq, mk, mv, mdo, mdq, static_cast<const __nv_bfloat16*>(p.q), p.g,
                                          p.S_in, p.sum_out, p.ws_f32);
            break;
        }
        case Op::kBackwardApply: {
            CUtensorMap mdk, mdv;
            if (!make_map(&mq, p.q, d, 128, d.qh) || !make_map(&mk, p.k, d, 128) ||
                !make_map(&mv, p.v, d, 128) || !make_map(&mdo, p.dO, d, 128) ||
                !make_map(&mdk, p.out0, d, 128) || !make_map(&mdv, p.out1, d, 128))
                return RM_ERR_CUDA;
            auto fn = vgtc_rev_kernel;
            if (!set_smem(fn, kRevSmem)) return RM_ERR_CUDA;
            fn<<<grid, 256, kRevSmem, s>>>(d, mq, mk, mv, mdo, mdk, mdv,
                                           static_cast<const __nv_bfloat16*>(p.q),
                                           static_cast<const __nv_bfloat16*>(p.k), p.g, p.S_in, p.dS_out,
                                           p.ws_f32, p.dg);
            break;
        }
        default:
            return RM_ERR_INVALID_ARG;
    }
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(1);
    return RM_OK;
}

rm_status vgtc_read_timeout_flag(int* host_flag, int clear, int* dev_scratch, cudaStream_t s) {
    vgtc::read_flag_kernel<<<1, 1, 0, s>>>(dev_scratch, clear);
    if (!rmcp::launch_ok()) return RM_ERR_CUDA;
    note_launch(1);
    if (cudaMemcpyAsync(host_flag, dev_scratch, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return RM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RM_ERR_CUDA;
    return RM_OK;
}

}  // namespace rmcp
