// tc_common.cuh -- sm_103a building blocks for the tensor-core kernels:
// mbarriers with bounded waits, TMA tile loads, tcgen05 (TMEM allocation,
// bf16 MMA with fp32 accumulation, commit, TMEM loads), shared-memory matrix
// descriptors for 128-byte-swizzled tiles, and the per-chunk gate prep.
//
// Tile convention: a bf16 tile of R rows x (64*nb) columns is stored as nb
// column blocks of [R rows][64 cols]; each row of a block is 128 bytes and
// its 16-byte chunks are XOR-swizzled by (row % 8), which is exactly what a
// TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes into a 1024-byte aligned
// destination.  The same bytes serve as a K-major operand (rows = M/N, the
// 64 columns = K) or as an MN-major operand (rows = K, columns = M/N).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace rmcp {
namespace tc {

constexpr int kChunk = 64;                       // tokens per chunk
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // bound of every mbarrier wait

// set by a kernel whose bounded wait ran out (the kernel then finishes
// without waiting further; its outputs are not valid)
static __device__ int g_timeout_flag = 0;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// one arrival (release, CTA scope) without a transaction count
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase with the given parity for at most limit_ns; on
// timeout sets g_timeout_flag and returns false.  Kernels keep walking their
// loop after a timeout (every later wait is bounded too), so that every copy
// they issued has been waited for before they free tensor memory and exit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) {
            atomicExch(&g_timeout_flag, 1);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ flags
// Flags in global memory between CTAs of one launch: a release store after
// the data it publishes (written before a CTA barrier that the releasing
// thread passed), an acquire load before the data is read.
__device__ __forceinline__ void flag_release(int* f) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(1) : "memory");
}
__device__ __forceinline__ int flag_acquire(const int* f) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}
// Waits until *f is set, for at most kWaitLimitNs; on a run-out sets
// g_timeout_flag and returns false (the caller's outputs are then not valid).
__device__ __forceinline__ bool flag_wait(const int* f) {
    if (flag_acquire(f)) return true;
    const uint64_t t0 = global_ns();
    while (!flag_acquire(f)) {
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicExch(&g_timeout_flag, 1);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
// Tile store smem -> global through the same 3-D tensor map shape.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the smem sources of all committed bulk stores may be overwritten
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed bulk store but the most recent group has finished reading
__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// all committed bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulation
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on bar once every MMA issued so far by this thread has completed
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per thread)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Same as tmem_ld32 without the wait: the values are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes from registers
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
          "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
          "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
          "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
          "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout 2), version 1.
// K-major: sbo = 1024 (next 8 rows), lbo unused.  MN-major: lbo = byte
// stride between 64-column blocks, sbo = 1024 (next 8 rows of K).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// The descriptor of the address `bytes` past that of d: one 32-bit add on the
// start-address field (shared-memory addresses stay below 256 KB, so the
// 14-bit field cannot carry into the next one).  Building descriptors this way
// keeps the issuing thread at about one add per operand and MMA.
__device__ __forceinline__ uint64_t desc_plus(uint64_t d, uint32_t bytes) {
    return (uint64_t(uint32_t(d >> 32)) << 32) | uint32_t(uint32_t(d) + (bytes >> 4));
}
// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn_major, int b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) |
           (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Byte offset of element (r, c) in a swizzled tile of R rows.
__device__ __forceinline__ uint32_t sw_off(int R, int r, int c) {
    return uint32_t((c >> 6) * R * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}
// Byte offset of the 16-byte chunk holding columns [8*ch, 8*ch+8) of row r.
__device__ __forceinline__ uint32_t sw_chunk(int R, int r, int ch) {
    return uint32_t((ch >> 3) * R * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint4 pack8(const float* x) {
    uint4 u;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(x[0], x[1]);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(x[2], x[3]);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(x[4], x[5]);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(x[6], x[7]);
    u.x = *reinterpret_cast<uint32_t*>(&p0);
    u.y = *reinterpret_cast<uint32_t*>(&p1);
    u.z = *reinterpret_cast<uint32_t*>(&p2);
    u.w = *reinterpret_cast<uint32_t*>(&p3);
    return u;
}
__device__ __forceinline__ void unpack8(uint4 u, float* x) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(p[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// ------------------------------------------------------------------ gates
// Per-chunk gate quantities (chunk-local, tau = 0..63):
//   b[tau]   = g_0 + ... + g_tau (inclusive running sum of the gates)
//   lid[tau] = number of sequence starts at chunk positions 1..tau
//   first    = the chunk's position 0 starts a sequence
// so that, inside the chunk, tokens s <= t are in the same sequence iff
// lid[s] == lid[t], and alpha_{s+1} ... alpha_t = exp(b[t] - b[s]) then.
struct alignas(16) GateSmem {
    float b[kChunk];
    float win[kChunk];   // alpha_0 ... alpha_tau (decay from the chunk's incoming state)
    float wout[kChunk];  // alpha_{tau+1} ... alpha_63 (decay to the chunk's last state)
    float ep[kChunk];    // exp(b[tau] - b[63])
    float en[kChunk];    // exp(b[63] - b[tau])
    int lid[kChunk];
    float nb[kChunk];    // exp(-b[tau])
    float btot;          // b[63]
    float emb;           // exp(-b[63])
    float W;             // alpha_0 ... alpha_63
    int first;           // position 0 starts a sequence
    int any;             // some position of the chunk starts a sequence
    int fast;            // every |b[tau] - b[63]| < 60: exp(b_t - b_s) = ep[t] en[s] in fp32
    // no sequence starts in the chunk and every |b[tau]| < 60 (with fast): the
    // decay weights can move from the operand tiles into the score masks and
    // onto the output rows, with every factor within e^(+-60)
    int fact;
};

struct GateRegs {
    float g0, g1;
    int s0, s1;
};

// Warp-collective: lane l loads tokens 2l and 2l+1 of the chunk at t0.
__device__ __forceinline__ GateRegs gate_load(const Dims& d, const float* __restrict__ g, int b,
                                              int h, int t0, int lane) {
    GateRegs r;
    const int t = t0 + 2 * lane;
    r.g0 = __ldg(g + g_off(d, b, t, h));
    r.g1 = __ldg(g + g_off(d, b, t + 1, h));
    r.s0 = starts_sequence(d.seq_idx, t) ? 1 : 0;
    r.s1 = starts_sequence(d.seq_idx, t + 1) ? 1 : 0;
    return r;
}

// Warp-collective scan of the loaded gates into gs.
__device__ __forceinline__ void gate_prep(const GateRegs& r, GateSmem* gs, int lane) {
    const float p = r.g0 + r.g1;
    const int c0 = lane > 0 ? r.s0 : 0;  // starts at position >= 1
    const int c = c0 + r.s1;
    float ps = p;
    int cs = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float pp = __shfl_up_sync(0xffffffffu, ps, o);
        const int cc = __shfl_up_sync(0xffffffffu, cs, o);
        if (lane >= o) {
            ps += pp;
            cs += cc;
        }
    }
    const float ex = ps - p;
    const int exc = cs - c;
    const float b0 = ex + r.g0, b1 = ps;
    const int l0 = exc + c0, l1 = cs;
    const float btot = __shfl_sync(0xffffffffu, ps, 31);
    const int ltot = __shfl_sync(0xffffffffu, cs, 31);
    const int first = __shfl_sync(0xffffffffu, r.s0, 0);
    gs->b[2 * lane] = b0;
    gs->b[2 * lane + 1] = b1;
    gs->lid[2 * lane] = l0;
    gs->lid[2 * lane + 1] = l1;
    gs->win[2 * lane] = (!first && l0 == 0) ? expf(b0) : 0.f;
    gs->win[2 * lane + 1] = (!first && l1 == 0) ? expf(b1) : 0.f;
    const float en0 = expf(btot - b0), en1 = expf(btot - b1);
    gs->en[2 * lane] = en0;
    gs->en[2 * lane + 1] = en1;
    gs->ep[2 * lane] = expf(b0 - btot);
    gs->ep[2 * lane + 1] = expf(b1 - btot);
    gs->wout[2 * lane] = (l0 == ltot) ? en0 : 0.f;
    gs->wout[2 * lane + 1] = (l1 == ltot) ? en1 : 0.f;
    gs->nb[2 * lane] = expf(-b0);
    gs->nb[2 * lane + 1] = expf(-b1);
    const float dev = fmaxf(fabsf(btot - b0), fabsf(btot - b1));
    const bool fast = __all_sync(0xffffffffu, dev < 60.f);
    const bool small = __all_sync(0xffffffffu, fmaxf(fabsf(b0), fabsf(b1)) < 60.f);
    if (lane == 0) {
        gs->btot = btot;
        gs->emb = expf(-btot);
        gs->fact = (fast && small && !first && ltot == 0) ? 1 : 0;
        gs->W = (!first && ltot == 0) ? expf(btot) : 0.f;
        gs->first = first;
        gs->any = (first || ltot > 0) ? 1 : 0;
        gs->fast = fast ? 1 : 0;
    }
}

}  // namespace tc
}  // namespace rmcp
