// tc_tiles.cuh -- tile and tensor-memory helpers shared by the tensor-core
// sweeps (internal header): the thread geometry of the 256 epilogue threads,
// tensor-memory row reads, swizzled bf16 tile access, TMA tile loads, and the
// host-side tensor maps and launch attributes.
#pragma once

#include <cudaTypedefs.h>

#include "internal.h"
#include "tc_common.cuh"

namespace rmcp {
namespace tc {

// internal linkage, as if written in each including translation unit
namespace {

constexpr uint32_t kTileBytes = kChunk * 64 * 2;  // one [64 rows][64 cols] bf16 block: 8 KB
constexpr int kThreads = 256;                     // 8 warps: two per tensor-memory lane quadrant

constexpr unsigned kFull = 0xffffffffu;

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

// Thread geometry.  Warp w reads tensor-memory lanes [32 (w % 4), +32); the
// two warps of a quadrant split the columns (grp = w / 4).  In the M = 64
// accumulators a chunk row tau lives in lane 32 (tau / 16) + tau % 16, i.e.
// lanes 0-15 of its quadrant; lanes 16-31 take over half of those rows'
// columns through a shuffle, so every thread works on 1/4 of a token row.
struct Geo {
    int tid, warp, lane, qd, grp;
    bool hi;       // lane >= 16
    int tau;       // token row of the M = 64 tiles handled by this thread
    int srow;      // state row of the M = 128 tiles (= 32 qd + lane)
    uint32_t tl;   // tensor-memory lane offset of the warp
};
__device__ __forceinline__ Geo geo() {
    Geo g;
    g.tid = threadIdx.x;
    g.warp = g.tid >> 5;
    g.lane = g.tid & 31;
    g.qd = g.warp & 3;
    g.grp = g.warp >> 2;
    g.hi = g.lane >= 16;
    g.tau = 16 * g.qd + (g.lane & 15);
    g.srow = 32 * g.qd + g.lane;
    g.tl = uint32_t(32 * g.qd) << 16;
    return g;
}

// Columns [col + 16 hi, +16) of row tau of an M = 64 accumulator (col absolute).
__device__ __forceinline__ void tok16(uint32_t tmem, const Geo& g, int col, float* x) {
    float v[32];
    tmem_ld32(tmem + g.tl + col, v);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float up = __shfl_sync(kFull, v[16 + e], (g.lane + 16) & 31);
        x[e] = g.hi ? up : v[e];
    }
}

// tok16 of two column blocks with the two tensor-memory loads in flight together
__device__ __forceinline__ void tok16x2(uint32_t tmem, const Geo& g, int col0, int col1, float* x0, float* x1) {
    uint32_t r0[32], r1[32];
    tmem_ld32_nowait(tmem + g.tl + col0, r0);
    tmem_ld32_nowait(tmem + g.tl + col1, r1);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float u0 = __shfl_sync(kFull, __uint_as_float(r0[16 + e]), (g.lane + 16) & 31);
        const float u1 = __shfl_sync(kFull, __uint_as_float(r1[16 + e]), (g.lane + 16) & 31);
        x0[e] = g.hi ? u0 : __uint_as_float(r0[e]);
        x1[e] = g.hi ? u1 : __uint_as_float(r1[e]);
    }
}

// Columns [64 grp, +64) of state row srow of an M = 128 accumulator at column col.
__device__ __forceinline__ void state_cols64(uint32_t tmem, const Geo& g, int col, float* x) {
    uint32_t r0[32], r1[32];
    tmem_ld32_nowait(tmem + g.tl + col + 64 * g.grp, r0);
    tmem_ld32_nowait(tmem + g.tl + col + 64 * g.grp + 32, r1);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        x[e] = __uint_as_float(r0[e]);
        x[32 + e] = __uint_as_float(r1[e]);
    }
}

__device__ __forceinline__ void store_state_half(uint8_t* tile, int i, int grp, const float* s) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(tile + sw_chunk(128, i, 8 * grp + c)) = pack8(s + c * 8);
}

// Row scaling of a [64][128] bf16 tile (2 blocks x 64 rows x 8 chunks of 16
// bytes = 1024 chunks): the CTA's 256 threads take 4 chunks each, eight
// consecutive threads covering the eight chunks of one 128-byte row so that a
// warp's 16-byte accesses hit distinct banks.  Chunk k (k < 4) of a thread is
// n = tid + 256 k: block n >> 9, row (n >> 3) & 63, chunk n & 7.
__device__ __forceinline__ uint32_t scale_off(int tid, int k, int* r) {
    const int n = tid + 256 * k;
    *r = (n >> 3) & 63;
    return uint32_t((n >> 9) * kTileBytes + ((n >> 3) & 63) * 128 + (n & 7) * 16);
}
__device__ __forceinline__ void scale_chunk(const uint8_t* src, uint8_t* dst, float w) {
    float x[8];
    unpack8(*reinterpret_cast<const uint4*>(src), x);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] *= w;
    *reinterpret_cast<uint4*>(dst) = pack8(x);
}

// Writes 16 bf16 values (columns c0..c0+15, c0 % 16 == 0) of row tau of a [64][64] tile.
__device__ __forceinline__ void store_row16(uint8_t* tile, int tau, int c0, const float* y) {
    *reinterpret_cast<uint4*>(tile + sw_chunk(64, tau, c0 >> 3)) = pack8(y);
    *reinterpret_cast<uint4*>(tile + sw_chunk(64, tau, (c0 >> 3) + 1)) = pack8(y + 8);
}

// 16 values (columns c0..c0+15, c0 % 8 == 0) of row t of a [64][128] bf16 tile.
__device__ __forceinline__ void tile_row_get16(const uint8_t* tile, int t, int c0, float* x) {
    unpack8(*reinterpret_cast<const uint4*>(tile + sw_chunk(64, t, c0 >> 3)), x);
    unpack8(*reinterpret_cast<const uint4*>(tile + sw_chunk(64, t, (c0 >> 3) + 1)), x + 8);
}

__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const float* v) {
    *reinterpret_cast<uint4*>(dst) = pack8(v);
    *reinterpret_cast<uint4*>(dst + 8) = pack8(v + 8);
}

}  // namespace

// ---------------------------------------------------------------------------
// host side (defined in tc_kernels.cu)
// ---------------------------------------------------------------------------
// [B*T rows][heads][D] bf16 viewed as a 3-D tensor; boxes of 64 tokens x 64
// columns, 128-byte swizzle (heads <= 0: d.H).
bool make_map(CUtensorMap* m, const void* base, const Dims& d, int D, int heads = 0);
// the CUresult of the calling thread's last make_map (-1: no encoder found;
// 0 after clear_map_result)
int last_map_result();
void clear_map_result();
// multiprocessors of the current device (cached per device)
int sm_count();

// Dynamic shared memory of a kernel; the carveout is set to all shared memory,
// so that kernels sized for two CTAs a SM get them.
template <typename K>
bool set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) ==
               cudaSuccess &&
           cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                int(cudaSharedmemCarveoutMaxShared)) == cudaSuccess;
}

}  // namespace tc
}  // namespace rmcp
