// Small-rank expand tile on the SM's fp32 FMA pipes.
//
// For ranks up to 32 the expand is a handful of multiply-adds per output
// element (16 at r = 16): plain fp32 FMA keeps pace with HBM and needs no
// operand conversion, MMA round trip or tensor memory.  A tile is 64
// consecutive tokens x 128 columns of one slice.  The B rows of every adapter
// the tile can meet are staged in shared memory (cp.async), the token indices
// and the old out values are read into shared memory and registers, then y;
// lane j of warp w computes columns {2j, 2j+1, 64+2j, 65+2j} of rows
// w, w + 8, ..., w + 56 (so a batch of 16 tokens still keeps every warp busy)
// in fp32 (exact products of y and B, one rounding of the result) and stores
// them with coalesced 4-byte accesses.
//
// Used by the plan-free expand kernel (one tile per CTA) and by the one-launch
// decode kernel (tiles staged before its shrink phase).
#pragma once

#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace lora {

constexpr int kFRows = 64;    // tokens per tile
constexpr int kFCols = 128;   // output columns per tile (one slice)
constexpr int kFThreads = 256;

// 16-byte slot of (8-rank chunk k8, column c) in one adapter's B tile: the
// column index's bit 0 flipped on odd 8-column groups, so the lanes of a warp
// (columns 2j + e) spread over all eight 16-byte bank groups.
__device__ __forceinline__ int fma_bslot(int k8, int c) { return k8 * kFCols + (c ^ ((c >> 3) & 1)); }

// Bytes of shared memory the B tile takes for `nl` adapters at RK8 8-rank chunks.
__host__ __device__ constexpr int fma_b_bytes(int nl, int rk8) { return nl * rk8 * kFCols * 16; }

template <typename E>
__device__ __forceinline__ float fma_dot8(const float (&y)[8], uint4 b, float acc) {
    float v[8];
    unpack8<E>(b, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(y[e], v[e], acc);
    return acc;
}

struct FmaTile {
    int s;          // slice
    int n0;         // first column within the slice
    int ncols;      // columns of this tile (> 0, a multiple of 8)
    int t0;         // first token
    int64_t col0;   // first column within out
};

// Tile `item` of a grid whose column chunks run fastest (neighbouring tiles
// share their y rows).  a.chunk_begin holds the first chunk of each slice.
__device__ __forceinline__ FmaTile fma_tile(const BgmvExpandArgs &a, int item, int nchunks) {
    FmaTile t;
    const int chunk = item % nchunks;
    t.t0 = (item / nchunks) * kFRows;
    int s = 0;
    while (s + 1 < a.num_slices && chunk >= a.chunk_begin[s + 1]) ++s;
    t.s = s;
    t.n0 = (chunk - a.chunk_begin[s]) * kFCols;
    t.ncols = min(kFCols, a.N[s] - t.n0);
    t.col0 = (int64_t)a.off[s] + t.n0;
    return t;
}

// Adapters whose B rows a tile needs: all of them with token indices, only
// adapter 0 without (every token uses it).
__device__ __forceinline__ int fma_adapters(const BgmvExpandArgs &a) { return a.idx ? a.L : 1; }

// The B rows of every adapter the tile can meet (cp.async, left uncommitted);
// ranks >= r_l and columns past the slice read as zeros.
template <typename E, int RK8>
__device__ __forceinline__ void fma_stage_b(const BgmvExpandArgs &a, const FmaTile &tt, uint4 *sB) {
    const E *Bs = static_cast<const E *>(a.B[tt.s]);
    const int Ns = a.N[tt.s], R = a.R;
    const int per_l = RK8 * kFCols;
    const int nl = fma_adapters(a);
    for (int q = threadIdx.x; q < nl * per_l; q += kFThreads) {
        const int lb = q / per_l, rem = q - lb * per_l, k8 = rem / kFCols, c = rem - k8 * kFCols;
        const int nv = c < tt.ncols ? min(8, clamp_rank(a.ranks, lb, R) - 8 * k8) : 0;
        const E *src = nv > 0 ? Bs + ((int64_t)lb * Ns + tt.n0 + c) * R + 8 * k8 : Bs;
        cp_async16(smem_u32(sB + lb * per_l + fma_bslot(k8, c)), src, nv > 0 ? 2 * nv : 0);
    }
}

// With add_inputs, this thread's old out values (issued now, used at the end).
template <typename E, bool ADD>
__device__ __forceinline__ void fma_load_old(const BgmvExpandArgs &a, const FmaTile &tt,
                                             uint32_t (&old)[8][2]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = 2 * lane, c1 = kFCols / 2 + 2 * lane;
    const E *out = static_cast<const E *>(a.out);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        old[i][0] = old[i][1] = 0u;
        const int t = tt.t0 + i * 8 + warp;
        if (ADD && t < a.T) {
            const E *orow = out + (int64_t)t * a.ldo + tt.col0;
            if (c0 < tt.ncols) old[i][0] = __ldcs(reinterpret_cast<const uint32_t *>(orow + c0));
            if (c1 < tt.ncols) old[i][1] = __ldcs(reinterpret_cast<const uint32_t *>(orow + c1));
        }
    }
}

// Adapter of token t for the expand: -1 for no LoRA term (index -1, out of
// range, or an adapter of rank 0).
__device__ __forceinline__ int fma_token_adapter(const BgmvExpandArgs &a, int t) {
    const int v = a.idx ? __ldg(a.idx + t) : 0;
    return (v >= 0 && v < a.L && clamp_rank(a.ranks, v, a.R) > 0) ? v : -1;
}

// Everything of a tile that does not depend on y: B rows, old out values and
// the tile's token -> adapter map (s_l).
template <typename E, bool ADD, int RK8>
__device__ __forceinline__ void fma_stage(const BgmvExpandArgs &a, const FmaTile &tt, uint4 *sB,
                                          int *s_l, uint32_t (&old)[8][2]) {
    fma_stage_b<E, RK8>(a, tt, sB);
    fma_load_old<E, ADD>(a, tt, old);
    if (threadIdx.x < kFRows) {
        const int t = tt.t0 + threadIdx.x;
        s_l[threadIdx.x] = t < a.T ? fma_token_adapter(a, t) : -1;
    }
}

// y rows of the tile's tokens for its slice (cp.async through L2, left
// uncommitted).  R is a multiple of 8, so the RK8 chunks cover exactly R.
template <int RK8>
__device__ __forceinline__ void fma_stage_y(const BgmvExpandArgs &a, const FmaTile &tt,
                                            float (*s_y)[8 * RK8]) {
    constexpr int RK = 8 * RK8;
    for (int q = threadIdx.x; q < kFRows * (RK / 4); q += kFThreads) {
        const int rr = q / (RK / 4), k4 = q - rr * (RK / 4);
        const int t = tt.t0 + rr;
        const bool in = t < a.T;
        const float *src =
            in ? a.y + (int64_t)t * a.ldy + (int64_t)tt.s * a.y_slice_stride + 4 * k4 : a.y;
        cp_async16(smem_u32(&s_y[rr][4 * k4]), src, in ? 16 : 0);
    }
}

// The tile's outputs from the staged B, y, map and old values (all visible
// to the block).  Rows with no LoRA term are left alone with add_inputs and
// written as zeros without.
template <typename E, bool ADD, int RK8>
__device__ __forceinline__ void fma_finish(const BgmvExpandArgs &a, const FmaTile &tt,
                                           const uint4 *sB, const float (*s_y)[8 * RK8],
                                           const int *s_l, const uint32_t (&old)[8][2]) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = 2 * lane, c1 = kFCols / 2 + 2 * lane;
    const bool ok0 = c0 < tt.ncols, ok1 = c1 < tt.ncols;
    E *__restrict__ out = static_cast<E *>(a.out);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rr = i * 8 + warp, t = tt.t0 + rr;
        const int l = t < a.T ? s_l[rr] : -2;  // warp-uniform
        if (l == -2) continue;
        E *orow = out + (int64_t)t * a.ldo + tt.col0;
        if (l < 0) {
            if (!ADD) {
                if (ok0) *reinterpret_cast<uint32_t *>(orow + c0) = 0u;
                if (ok1) *reinterpret_cast<uint32_t *>(orow + c1) = 0u;
            }
            continue;
        }
        const int rl = clamp_rank(a.ranks, l, a.R);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4 *bl = sB + l * RK8 * kFCols;
#pragma unroll
        for (int k8 = 0; k8 < RK8; ++k8) {
            float yv[8];
            const float4 ya = *reinterpret_cast<const float4 *>(&s_y[rr][8 * k8]);
            const float4 yb = *reinterpret_cast<const float4 *>(&s_y[rr][8 * k8 + 4]);
            yv[0] = ya.x; yv[1] = ya.y; yv[2] = ya.z; yv[3] = ya.w;
            yv[4] = yb.x; yv[5] = yb.y; yv[6] = yb.z; yv[7] = yb.w;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (8 * k8 + e >= rl) yv[e] = 0.f;  // ranks past r_l
            acc[0] = fma_dot8<E>(yv, bl[fma_bslot(k8, c0)], acc[0]);
            acc[1] = fma_dot8<E>(yv, bl[fma_bslot(k8, c0 + 1)], acc[1]);
            acc[2] = fma_dot8<E>(yv, bl[fma_bslot(k8, c1)], acc[2]);
            acc[3] = fma_dot8<E>(yv, bl[fma_bslot(k8, c1 + 1)], acc[3]);
        }
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = a.scale * acc[q];
        if (ADD) {
            const float2 o0 = Pack<E>::unpack(old[i][0]), o1 = Pack<E>::unpack(old[i][1]);
            v[0] += o0.x; v[1] += o0.y; v[2] += o1.x; v[3] += o1.y;
        }
        if (ok0) *reinterpret_cast<uint32_t *>(orow + c0) = Pack<E>::pack(v[0], v[1]);
        if (ok1) *reinterpret_cast<uint32_t *>(orow + c1) = Pack<E>::pack(v[2], v[3]);
    }
}

// First column chunk of each slice in a.chunk_begin; returns the chunk count.
inline int fma_set_chunks(BgmvExpandArgs &a) {
    a.chunk_begin[0] = 0;
    for (int s = 0; s < a.num_slices; ++s)
        a.chunk_begin[s + 1] = a.chunk_begin[s] + (a.N[s] + kFCols - 1) / kFCols;
    for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s) a.chunk_begin[s + 1] = a.chunk_begin[s];
    return a.chunk_begin[a.num_slices];
}

}  // namespace lora
