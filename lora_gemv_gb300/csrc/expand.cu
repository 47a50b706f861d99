// Expand / expand_slice: out[t, off_s + n] (+)= scale * sum_i y[t, s*ys + i] * B_s[l, n, i].
//
// Pages: vLLM PR #11579 "[misc] Add LoRA kernel micro benchmarks"
// (bgmv_expand, sgmv_expand, the _slice forms with num_slices, add_inputs as
// "group-gemm + outputs", the f32 x f16 => f16 typing); Punica issue #17
// (SGMV: tokens sharing an adapter reuse its weights).
//
// Design (GB300): the operator is an HBM-bound read-modify-write of out; the
// adapter tile is small and reused by every token of a plan tile.
//  - grid.x walks the plan's 64-token tiles (one adapter each), grid.y the
//    128-column chunks of all slices, so one launch covers every slice;
//  - a CTA stages B_s[l, n0:n0+128, 0:r_l] and the tile's y rows in shared
//    memory, then each warp owns 32 output columns of all 64 tokens;
//  - out is read and written with 16-byte accesses straight from registers:
//    the MMA columns are permuted (B rows are stored permuted in shared
//    memory) so that every thread's accumulators are 8 contiguous columns;
//  - y (fp32) enters the fp16/bf16 tensor-core MMA (m16n8k16, fp32
//    accumulate) as hi + lo parts after scaling each token row by a power of
//    two, so the product keeps ~fp32 accuracy of y and never overflows fp16;
//  - tiles with adapter -1 and adapters of rank 0 load nothing (block
//    skipping) and, without add_inputs, only store zeros.
#include "common.cuh"
#include "kernels.h"

namespace lora {
namespace {

constexpr int kThreads = 128;  // 4 warps
constexpr int kCols = 128;     // output columns per CTA (32 per warp)

__host__ __device__ constexpr int pitch_of(int ks) { return ks * 16 + 8; }  // elements per smem row

// Shared-memory row of output column j of a chunk: inside each 32-column
// block, column 8a + 2i + b (a, i in 0..3, b in 0..1) goes to row 8i + 2a + b,
// so MMA n-tile i reads 8 consecutive rows.
__device__ __forceinline__ int sigma(int j) {
    return (j & ~31) + 8 * ((j >> 1) & 3) + 2 * ((j >> 3) & 3) + (j & 1);
}

template <typename E>
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    uint4 r;
    uint32_t *w = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        E lo = Elem<E>::from_f(v[2 * k]), hi = Elem<E>::from_f(v[2 * k + 1]);
        w[k] = (uint32_t)(*reinterpret_cast<uint16_t *>(&lo)) |
               ((uint32_t)(*reinterpret_cast<uint16_t *>(&hi)) << 16);
    }
    return r;
}

template <typename E>
__device__ __forceinline__ void unpack8(uint4 r, float (&v)[8]) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint16_t lo = (uint16_t)(w[k] & 0xffffu), hi = (uint16_t)(w[k] >> 16);
        v[2 * k] = Elem<E>::to_f(*reinterpret_cast<E *>(&lo));
        v[2 * k + 1] = Elem<E>::to_f(*reinterpret_cast<E *>(&hi));
    }
}

// v = hi + lo with hi = round(v) and lo = round(v - hi) in the weight type.
template <typename E>
__device__ __forceinline__ void split_hilo8(const float (&v)[8], uint4 &hi, uint4 &lo) {
    float h[8], l[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        h[k] = Elem<E>::to_f(Elem<E>::from_f(v[k]));
        l[k] = v[k] - h[k];
    }
    hi = pack8<E>(h);
    lo = pack8<E>(l);
}

template <typename E, bool ADD, bool VEC>
__global__ void __launch_bounds__(kThreads)
expand_kernel(const ExpandArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_rows[kTile];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;

    // The plan header and this CTA's first tile are read together.
    const int4 h0 = __ldcg(reinterpret_cast<const int4 *>(a.hdr));      // magic, T, L, kind
    const int4 h1 = __ldcg(reinterpret_cast<const int4 *>(a.hdr) + 1);  // nactive, ngroups, ntiles
    int4 tl_next = (int)blockIdx.x < a.max_tiles ? __ldcg(a.tiles + blockIdx.x)
                                                 : make_int4(-1, 0, 0, -1);
    if (h0.x != LORA_PLAN_MAGIC || h0.y != a.T || h0.z != a.L) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_MISMATCH);
        return;
    }

    // column chunk -> slice
    const int chunk = blockIdx.y;
    int s = 0;
    while (s + 1 < a.num_slices && chunk >= a.chunk_begin[s + 1]) ++s;
    const int n0 = (chunk - a.chunk_begin[s]) * kCols;
    const int Ns = a.N[s];
    const int ncols = min(kCols, Ns - n0);
    const E *__restrict__ B = static_cast<const E *>(a.B[s]);
    E *__restrict__ out = static_cast<E *>(a.out);
    const int64_t col0 = (int64_t)a.off[s] + n0;
    const int R = a.R;
    const bool b_vec = (R % 8 == 0) && ((reinterpret_cast<uintptr_t>(B) & 15) == 0);

    const int ks_max = (R + 15) / 16;
    E *sB = reinterpret_cast<E *>(smem);                  // [kCols][pitch]
    E *sYh = sB + kCols * pitch_of(ks_max);               // [kTile][pitch]
    E *sYl = sYh + kTile * pitch_of(ks_max);              // [kTile][pitch]
    float *sF = reinterpret_cast<float *>(sYl + kTile * pitch_of(ks_max));  // [kTile]

    const int n_tiles = min(h1.z, a.max_tiles);
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int4 tl = tl_next;
        if (tile + (int)gridDim.x < n_tiles) tl_next = __ldcg(a.tiles + tile + gridDim.x);
        const int l = tl.x, p0 = tl.y, n = tl.z;
        const int rl = l >= 0 && l < a.L ? clamp_rank(a.ranks, l, R) : 0;

        if (threadIdx.x < kTile) {
            int row = -1;
            if (threadIdx.x < n) {
                row = __ldcg(a.perm + p0 + threadIdx.x);
                if (row < 0 || row >= a.T) row = -1;
            }
            s_rows[threadIdx.x] = row;
        }
        __syncthreads();

        if (rl == 0) {  // adapter -1 (or rank 0): untouched with add_inputs, else zeros
            if (!ADD) {
                for (int it = threadIdx.x; it < kTile * (kCols / 8); it += kThreads) {
                    const int i = it / (kCols / 8), c8 = (it % (kCols / 8)) * 8;
                    const int row = s_rows[i];
                    if (row < 0 || c8 >= ncols) continue;
                    E *p = out + (int64_t)row * a.ldo + col0 + c8;
                    if (VEC) {
                        st_global_v4(p, make_uint4(0, 0, 0, 0));
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (c8 + k < ncols) p[k] = Elem<E>::from_f(0.f);
                    }
                }
            }
            __syncthreads();
            continue;
        }

        const int KS = (rl + 15) / 16;
        const int pitch = pitch_of(KS);
        const int wcol = warp * 32 + q * 8;  // this thread's 8 columns within the chunk
        const bool wact = warp * 32 < ncols;
        const int nmb = (n + 15) / 16;

        // 1) issue the reads of out early (they overlap the staging below)
        uint4 old[4][2];
        if (ADD && VEC && wact && wcol < ncols) {
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) {
                if (mb < nmb) {
                    const int r0 = s_rows[mb * 16 + g], r1 = s_rows[mb * 16 + g + 8];
                    if (r0 >= 0) old[mb][0] = ld_global_v4(out + (int64_t)r0 * a.ldo + col0 + wcol);
                    if (r1 >= 0) old[mb][1] = ld_global_v4(out + (int64_t)r1 * a.ldo + col0 + wcol);
                }
            }
        }

        // 2) stage B_s[l, n0 : n0 + kCols, 0 : KS*16) (zero beyond r_l / ncols), rows permuted
        const E *Bl = B + ((int64_t)l * Ns + n0) * R;
        for (int it = threadIdx.x; it < kCols * 2 * KS; it += kThreads) {
            const int j = it / (2 * KS), c8 = (it % (2 * KS)) * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (j < ncols && c8 < rl) {
                const E *src = Bl + (int64_t)j * R + c8;
                const int nv = rl - c8;  // valid elements of this 8-element chunk
                if (b_vec) {
                    v = __ldg(reinterpret_cast<const uint4 *>(src));
                    if (nv < 8) {
                        uint32_t *w = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            w[k] &= (2 * k + 1 < nv) ? 0xffffffffu : (2 * k < nv ? 0xffffu : 0u);
                    }
                } else {
                    const uint16_t *s16 = reinterpret_cast<const uint16_t *>(src);
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t lo16 = 2 * k < nv ? __ldg(s16 + 2 * k) : 0u;
                        const uint32_t hi16 = 2 * k + 1 < nv ? __ldg(s16 + 2 * k + 1) : 0u;
                        w[k] = lo16 | (hi16 << 16);
                    }
                    v = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            *reinterpret_cast<uint4 *>(sB + sigma(j) * pitch + c8) = v;
        }

        // 3) stage y rows as scaled hi/lo pairs: two threads per token row,
        //    each owning KS*8 columns, every load of a pass independent.
        {
            const int i = threadIdx.x >> 1, c0 = (threadIdx.x & 1) * KS * 8;
            const int row = s_rows[i];
            const float *yr = a.y + (int64_t)(row < 0 ? 0 : row) * a.ldy +
                              (int64_t)s * a.y_slice_stride;
            float m = 0.f;
#pragma unroll
            for (int c = 0; c < LORA_MAX_RANK / 16; ++c) {
                if (c < KS) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int j = c0 + 8 * c + k;
                        if (row >= 0 && j < rl) m = fmaxf(m, fabsf(yr[j]));
                    }
                }
            }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            int e = 0;
            frexpf(m, &e);
#pragma unroll
            for (int c = 0; c < LORA_MAX_RANK / 16; ++c) {
                if (c < KS) {
                    float vs[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int j = c0 + 8 * c + k;
                        vs[k] = (row >= 0 && j < rl) ? ldexpf(yr[j], -e) : 0.f;
                    }
                    uint4 hi, lo;
                    split_hilo8<E>(vs, hi, lo);
                    *reinterpret_cast<uint4 *>(sYh + i * pitch + c0 + 8 * c) = hi;
                    *reinterpret_cast<uint4 *>(sYl + i * pitch + c0 + 8 * c) = lo;
                }
            }
            if ((threadIdx.x & 1) == 0) sF[i] = ldexpf(a.scale, e);
        }
        __syncthreads();

        // 4) tensor-core MMAs + epilogue
        if (wact) {
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) {
                if (mb >= nmb) break;
                float acc[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[i][k] = 0.f;
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t ah[4], al[4];
                    const int arow = mb * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                    const int acol = ks * 16 + 8 * (lane >> 4);
                    ldmatrix_x4(ah, smem_u32(sYh + arow * pitch + acol));
                    ldmatrix_x4(al, smem_u32(sYl + arow * pitch + acol));
#pragma unroll
                    for (int np = 0; np < 2; ++np) {
                        uint32_t b[4];
                        const int brow = warp * 32 + 8 * (2 * np + (lane >> 4)) + (lane & 7);
                        const int bcol = ks * 16 + 8 * ((lane >> 3) & 1);
                        ldmatrix_x4(b, smem_u32(sB + brow * pitch + bcol));
                        mma16816<E>(acc[2 * np], ah, b[0], b[1]);
                        mma16816<E>(acc[2 * np], al, b[0], b[1]);
                        mma16816<E>(acc[2 * np + 1], ah, b[2], b[3]);
                        mma16816<E>(acc[2 * np + 1], al, b[2], b[3]);
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int i = mb * 16 + g + 8 * h;
                    const int row = s_rows[i];
                    if (row < 0) continue;
                    const float f = sF[i];
                    float res[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) res[k] = f * acc[k >> 1][2 * h + (k & 1)];
                    E *p = out + (int64_t)row * a.ldo + col0 + wcol;
                    if (VEC) {
                        if (wcol < ncols) {
                            if (ADD) {
                                float o[8];
                                unpack8<E>(old[mb][h], o);
#pragma unroll
                                for (int k = 0; k < 8; ++k) res[k] += o[k];
                            }
                            st_global_v4(p, pack8<E>(res));
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            if (wcol + k < ncols) {
                                float r = res[k];
                                if (ADD) r += Elem<E>::to_f(p[k]);
                                p[k] = Elem<E>::from_f(r);
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Streaming expand (the fast path: 16-byte aligned out columns and B rows).
//
// A persistent grid walks "units" (plan tile x 128-column chunk) in a
// contiguous range per CTA, tile-major, so consecutive units share the
// tile's token rows and y.  Each unit's out tile (gathered rows) and B tile
// are copied into shared memory by cp.async, STAGES units ahead, so every
// SM keeps ~100 KB of HBM reads in flight; results are stored straight from
// registers with 16-byte stores.  y is converted to scaled hi/lo pairs only
// when the unit's (tile, slice) changes.
constexpr int kSThreads = 256;          // 8 warps: 4 column blocks x 2 row halves
constexpr int kOutPitch = kCols + 8;    // elements per shared row of the out tile (272 B)

__host__ __device__ constexpr int stream_stage_bytes(int ks_max) {
    return kTile * kOutPitch * 2 + kCols * pitch_of(ks_max) * 2;
}
__host__ __device__ constexpr int stream_smem_bytes(int ks_max, int stages) {
    return stages * stream_stage_bytes(ks_max) + 2 * kTile * pitch_of(ks_max) * 2 +
           kTile * (int)sizeof(float);
}

constexpr int kWin = 8;  // plan tiles whose metadata a CTA holds in shared memory at once

struct UnitInfo {
    int w;               // tile slot in the CTA's window
    int l, p0, n;        // tile: adapter, first perm position, tokens
    int s, n0, ncols;    // chunk: slice, first column in the slice, columns
    int rl;              // adapter rank (0 = nothing to add)
};

// Shared per-window plan metadata: tile records and their token rows.
struct WinMeta {
    int4 tile[kWin];          // {adapter, p0, n, rank}
    int rows[kWin][kTile];    // out row of every token of the tile, -1 if none
};

__device__ __forceinline__ UnitInfo unit_info(const ExpandArgs &a, const WinMeta &wm, int u,
                                              int t_first, int nchunks) {
    UnitInfo ui;
    const int t = u / nchunks, c = u - t * nchunks;
    ui.w = t - t_first;
    const int4 tl = wm.tile[ui.w];
    ui.l = tl.x;
    ui.p0 = tl.y;
    ui.n = tl.z;
    ui.rl = tl.w;
    int s = 0;
    while (s + 1 < a.num_slices && c >= a.chunk_begin[s + 1]) ++s;
    ui.s = s;
    ui.n0 = (c - a.chunk_begin[s]) * kCols;
    ui.ncols = min(kCols, a.N[s] - ui.n0);
    return ui;
}

// (tile, slice) of unit u differs from that of unit u-1 (or u is the first).
__device__ __forceinline__ bool new_y(const ExpandArgs &a, int u, int u_first, int nchunks) {
    if (u == u_first) return true;
    const int t = u / nchunks, c = u - t * nchunks;
    if (c == 0) return true;
    for (int s = 1; s < a.num_slices; ++s)
        if (c == a.chunk_begin[s]) return true;
    return false;
}

template <typename E, bool ADD>
__device__ __forceinline__ void stream_issue(const ExpandArgs &a, const WinMeta &wm,
                                             const UnitInfo &ui, unsigned char *stage, int pitch) {
    if (ui.rl == 0) return;
    E *sOut = reinterpret_cast<E *>(stage);
    E *sB = reinterpret_cast<E *>(stage + kTile * kOutPitch * 2);
    const E *out = static_cast<const E *>(a.out);
    const int64_t col0 = (int64_t)a.off[ui.s] + ui.n0;
    if (ADD) {  // 4 threads per token row, 4 x 16 bytes each
        const int i = threadIdx.x >> 2, ch0 = (threadIdx.x & 3) * 4;
        const int row = wm.rows[ui.w][i];
        if (row >= 0) {
            const E *src = out + (int64_t)row * a.ldo + col0;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if ((ch0 + k) * 8 < ui.ncols)
                    cp_async16(smem_u32(sOut + i * kOutPitch + (ch0 + k) * 8), src + (ch0 + k) * 8, 16);
        }
    }
    const int KS = (ui.rl + 15) / 16;
    const E *Bl = static_cast<const E *>(a.B[ui.s]) + ((int64_t)ui.l * a.N[ui.s] + ui.n0) * a.R;
    for (int it = threadIdx.x; it < kCols * 2 * KS; it += kSThreads) {
        const int j = it / (2 * KS), c8 = (it - j * 2 * KS) * 8;
        const int nv = j < ui.ncols ? min(8, ui.rl - c8) : 0;
        const E *src = nv > 0 ? Bl + (int64_t)j * a.R + c8 : Bl;
        cp_async16(smem_u32(sB + sigma(j) * pitch + c8), src, nv > 0 ? 2 * nv : 0);
    }
}

template <typename E, bool ADD, int STAGES>
__global__ void __launch_bounds__(kSThreads, 1)
expand_stream_kernel(const ExpandArgs a, int tiles_grid) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ WinMeta wm;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int cb = warp & 3, rh = warp >> 2;  // 32-column block, 32-row half

    // Units (tile x chunk, tile-major) are split over the grid by the host's
    // tile bound, so the first window's tile records load with the header.
    const int nchunks = a.chunk_begin[a.num_slices];
    const int U_grid = tiles_grid * nchunks;
    const int per = (U_grid + gridDim.x - 1) / gridDim.x;
    const int u_begin = blockIdx.x * per;
    const int4 h0 = __ldg(reinterpret_cast<const int4 *>(a.hdr));
    const int4 h1 = __ldg(reinterpret_cast<const int4 *>(a.hdr) + 1);
    int4 tl_first = make_int4(-1, 0, 0, 0);
    if (threadIdx.x < kWin) {
        const int t = u_begin / nchunks + threadIdx.x;
        if (t < a.max_tiles) tl_first = __ldg(a.tiles + t);
    }
    if (h0.x != LORA_PLAN_MAGIC || h0.y != a.T || h0.z != a.L) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_MISMATCH);
        return;
    }
    const int n_tiles = min(h1.z, a.max_tiles);
    const int u_end = min(n_tiles * nchunks, u_begin + per);

    const int ks_max = (a.R + 15) / 16;
    const int pitch = pitch_of(ks_max);
    const int sbytes = stream_stage_bytes(ks_max);
    E *sYh = reinterpret_cast<E *>(smem + STAGES * sbytes);
    E *sYl = sYh + kTile * pitch;
    float *sF = reinterpret_cast<float *>(sYl + kTile * pitch);
    E *__restrict__ out = static_cast<E *>(a.out);

    for (int u0 = u_begin; u0 < u_end;) {
        // ---- window: up to kWin tiles, metadata into shared memory
        const int t_first = u0 / nchunks;
        const int u1 = min(u_end, (t_first + kWin) * nchunks);
        if (threadIdx.x < kWin) {
            int4 tl = tl_first;
            if (u0 != u_begin) {
                const int t = t_first + threadIdx.x;
                tl = t < n_tiles ? __ldg(a.tiles + t) : make_int4(-1, 0, 0, 0);
            }
            const int t = t_first + threadIdx.x;
            if (t >= n_tiles) tl = make_int4(-1, 0, 0, 0);
            const int rl = tl.x >= 0 && tl.x < a.L ? clamp_rank(a.ranks, tl.x, a.R) : 0;
            wm.tile[threadIdx.x] = make_int4(tl.x, tl.y, tl.z, rl);
        }
        __syncthreads();
        for (int it = threadIdx.x; it < kWin * kTile; it += kSThreads) {
            const int w = it / kTile, i = it - w * kTile;
            const int4 tl = wm.tile[w];
            int row = -1;
            if (i < tl.z) {
                row = __ldg(a.perm + tl.y + i);
                if (row < 0 || row >= a.T) row = -1;
            }
            wm.rows[w][i] = row;
        }
        __syncthreads();

        // ---- pipelined units of the window
#pragma unroll
        for (int k = 0; k < STAGES - 1; ++k) {
            if (u0 + k < u1)
                stream_issue<E, ADD>(a, wm, unit_info(a, wm, u0 + k, t_first, nchunks),
                                     smem + k * sbytes, pitch);
            cp_async_commit();
        }
        for (int u = u0; u < u1; ++u) {
            cp_async_wait<STAGES - 2>();
            __syncthreads();
            const int nxt = u + STAGES - 1;
            if (nxt < u1)
                stream_issue<E, ADD>(a, wm, unit_info(a, wm, nxt, t_first, nchunks),
                                     smem + ((nxt - u0) % STAGES) * sbytes, pitch);
            cp_async_commit();

            const UnitInfo ui = unit_info(a, wm, u, t_first, nchunks);
            const int *rows = wm.rows[ui.w];
            const int64_t col0 = (int64_t)a.off[ui.s] + ui.n0;
            if (ui.rl == 0) {  // adapter -1 or rank 0: nothing to add; without add_inputs, zeros
                if (!ADD) {
                    const int i = threadIdx.x >> 2, ch0 = (threadIdx.x & 3) * 4;
                    const int row = rows[i];
                    if (row >= 0) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if ((ch0 + k) * 8 < ui.ncols)
                                st_global_v4(out + (int64_t)row * a.ldo + col0 + (ch0 + k) * 8,
                                             make_uint4(0, 0, 0, 0));
                    }
                }
                continue;
            }
            const int KS = (ui.rl + 15) / 16;
            if (new_y(a, u, u0, nchunks)) {
                // 4 threads per token row: scaled hi/lo pairs of y[row, s*ys : s*ys + r_l)
                const int i = threadIdx.x >> 2, part = threadIdx.x & 3;
                const int row = rows[i];
                const bool live = row >= 0;
                const float *yr = a.y + (int64_t)(live ? row : 0) * a.ldy +
                                  (int64_t)ui.s * a.y_slice_stride;
                const int j0 = part * KS * 4;
                float v[LORA_MAX_RANK / 4];
                float m = 0.f;
#pragma unroll
                for (int k = 0; k < LORA_MAX_RANK / 4; ++k) {
                    const int j = j0 + k;
                    v[k] = (k < KS * 4 && live && j < ui.rl) ? yr[j] : 0.f;
                    m = fmaxf(m, fabsf(v[k]));
                }
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                int e = 0;
                frexpf(m, &e);
#pragma unroll
                for (int k = 0; k < LORA_MAX_RANK / 4; ++k) {
                    if (k < KS * 4) {
                        const float vs = ldexpf(v[k], -e);
                        const E hi = Elem<E>::from_f(vs);
                        sYh[i * pitch + j0 + k] = hi;
                        sYl[i * pitch + j0 + k] = Elem<E>::from_f(vs - Elem<E>::to_f(hi));
                    }
                }
                if (part == 0) sF[i] = ldexpf(a.scale, e);
                __syncthreads();
            }

            const unsigned char *stage = smem + ((u - u0) % STAGES) * sbytes;
            const E *sOut = reinterpret_cast<const E *>(stage);
            const E *sB = reinterpret_cast<const E *>(stage + kTile * kOutPitch * 2);
            const int wcol = cb * 32 + q * 8;
            if (cb * 32 < ui.ncols) {
#pragma unroll
                for (int mm = 0; mm < 2; ++mm) {
                    const int mb = rh * 2 + mm;
                    if (mb * 16 >= ui.n) break;
                    float acc[4][4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int k = 0; k < 4; ++k) acc[i][k] = 0.f;
                    for (int ks = 0; ks < KS; ++ks) {
                        uint32_t ah[4], al[4];
                        const int arow = mb * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                        const int acol = ks * 16 + 8 * (lane >> 4);
                        ldmatrix_x4(ah, smem_u32(sYh + arow * pitch + acol));
                        ldmatrix_x4(al, smem_u32(sYl + arow * pitch + acol));
#pragma unroll
                        for (int np = 0; np < 2; ++np) {
                            uint32_t b[4];
                            const int brow = cb * 32 + 8 * (2 * np + (lane >> 4)) + (lane & 7);
                            const int bcol = ks * 16 + 8 * ((lane >> 3) & 1);
                            ldmatrix_x4(b, smem_u32(sB + brow * pitch + bcol));
                            mma16816<E>(acc[2 * np], ah, b[0], b[1]);
                            mma16816<E>(acc[2 * np], al, b[0], b[1]);
                            mma16816<E>(acc[2 * np + 1], ah, b[2], b[3]);
                            mma16816<E>(acc[2 * np + 1], al, b[2], b[3]);
                        }
                    }
                    if (wcol < ui.ncols) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int i = mb * 16 + g + 8 * h;
                            const int row = rows[i];
                            if (row < 0) continue;
                            const float f = sF[i];
                            float res[8];
#pragma unroll
                            for (int k = 0; k < 8; ++k) res[k] = f * acc[k >> 1][2 * h + (k & 1)];
                            if (ADD) {
                                float o[8];
                                unpack8<E>(*reinterpret_cast<const uint4 *>(sOut + i * kOutPitch + wcol), o);
#pragma unroll
                                for (int k = 0; k < 8; ++k) res[k] += o[k];
                            }
                            st_global_v4(out + (int64_t)row * a.ldo + col0 + wcol, pack8<E>(res));
                        }
                    }
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();  // the window's shared metadata and stages are free again
        u0 = u1;
    }
}

template <typename E, bool ADD, bool VEC>
cudaError_t configure_one() {
    const int ks = LORA_MAX_RANK / 16;
    const int smem = (kCols + 2 * kTile) * pitch_of(ks) * (int)sizeof(E) + kTile * (int)sizeof(float);
    return cudaFuncSetAttribute(expand_kernel<E, ADD, VEC>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <typename E, bool ADD, int STAGES>
cudaError_t configure_stream_one() {
    // 4 stages serve ranks <= 32, 3 stages any rank (see launch_stream_dtype)
    return cudaFuncSetAttribute(expand_stream_kernel<E, ADD, STAGES>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                STAGES == 4 ? stream_smem_bytes(2, 4)
                                            : stream_smem_bytes(LORA_MAX_RANK / 16, 3));
}

template <typename E>
cudaError_t configure_dtype() {
    cudaError_t e;
    if ((e = configure_one<E, false, false>()) != cudaSuccess) return e;
    if ((e = configure_one<E, false, true>()) != cudaSuccess) return e;
    if ((e = configure_one<E, true, false>()) != cudaSuccess) return e;
    if ((e = configure_one<E, true, true>()) != cudaSuccess) return e;
    if ((e = configure_stream_one<E, false, 3>()) != cudaSuccess) return e;
    if ((e = configure_stream_one<E, false, 4>()) != cudaSuccess) return e;
    if ((e = configure_stream_one<E, true, 3>()) != cudaSuccess) return e;
    return configure_stream_one<E, true, 4>();
}

// Stages: 4 for ranks up to 32 (two CTAs per SM fit), else 3 (one CTA per SM).
template <typename E>
cudaError_t launch_stream_dtype(const ExpandArgs &a, int ks_max, int grid, int tiles_grid,
                                cudaStream_t st) {
    const int stages = ks_max <= 2 ? 4 : 3;
    const size_t smem = stream_smem_bytes(ks_max, stages);
    if (a.add) {
        if (stages == 4) expand_stream_kernel<E, true, 4><<<grid, kSThreads, smem, st>>>(a, tiles_grid);
        else expand_stream_kernel<E, true, 3><<<grid, kSThreads, smem, st>>>(a, tiles_grid);
    } else {
        if (stages == 4) expand_stream_kernel<E, false, 4><<<grid, kSThreads, smem, st>>>(a, tiles_grid);
        else expand_stream_kernel<E, false, 3><<<grid, kSThreads, smem, st>>>(a, tiles_grid);
    }
    return cudaGetLastError();
}

template <typename E>
cudaError_t launch_dtype(const ExpandArgs &a, bool vec, dim3 grid, size_t smem, cudaStream_t st) {
    if (a.add) {
        if (vec) expand_kernel<E, true, true><<<grid, kThreads, smem, st>>>(a);
        else expand_kernel<E, true, false><<<grid, kThreads, smem, st>>>(a);
    } else {
        if (vec) expand_kernel<E, false, true><<<grid, kThreads, smem, st>>>(a);
        else expand_kernel<E, false, false><<<grid, kThreads, smem, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t configure_expand_kernels() {
    cudaError_t e = configure_dtype<__half>();
    if (e != cudaSuccess) return e;
    return configure_dtype<__nv_bfloat16>();
}

cudaError_t launch_expand(lora_dtype_t dt, const ExpandArgs &a_in, const DeviceInfo &dev,
                          cudaStream_t stream) {
    ExpandArgs a = a_in;
    a.chunk_begin[0] = 0;
    for (int s = 0; s < a.num_slices; ++s)
        a.chunk_begin[s + 1] = a.chunk_begin[s] + (a.N[s] + kCols - 1) / kCols;
    for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s) a.chunk_begin[s + 1] = a.chunk_begin[s];
    const int chunks = a.chunk_begin[a.num_slices];
    if (chunks == 0 || a.T == 0) return cudaSuccess;

    // Vector path: every 8-column group of every slice is 16-byte aligned.
    bool vec = (reinterpret_cast<uintptr_t>(a.out) & 15) == 0 && a.ldo % 8 == 0;
    for (int s = 0; s < a.num_slices; ++s) vec = vec && a.off[s] % 8 == 0 && a.N[s] % 8 == 0;

    // Tiles: ceil(T/64) full-or-partial tiles plus at most one ragged tile per
    // adapter and one for the inactive tokens; CTAs loop if a plan has more.
    const long long est = (a.T + kTile - 1) / kTile + (long long)std::min(a.L, a.T) + 1;
    const int ks_max = (a.R + 15) / 16;
    const bool b_vec_all = [&] {
        if (a.R % 8 != 0) return false;
        for (int s = 0; s < a.num_slices; ++s)
            if (reinterpret_cast<uintptr_t>(a.B[s]) & 15) return false;
        return true;
    }();
    if (vec && b_vec_all) {
        // persistent grid: every CTA streams a contiguous range of units
        const int per_sm = stream_smem_bytes(ks_max, ks_max <= 2 ? 4 : 3) * 2 <= 227 * 1024 ? 2 : 1;
        const int tiles_grid = (int)std::min<long long>(est, a.max_tiles);
        const long long units = (long long)tiles_grid * chunks;
        const int grid = (int)std::max<long long>(1, std::min<long long>(units, (long long)per_sm * dev.sm_count));
        return dt == LORA_F16 ? launch_stream_dtype<__half>(a, ks_max, grid, tiles_grid, stream)
                              : launch_stream_dtype<__nv_bfloat16>(a, ks_max, grid, tiles_grid, stream);
    }
    const int gx = (int)std::min<long long>(est, a.max_tiles);
    dim3 grid(std::max(gx, 1), chunks);
    const int ks = (a.R + 15) / 16;
    const size_t smem = (size_t)(kCols + 2 * kTile) * pitch_of(ks) * 2 + kTile * sizeof(float);
    return dt == LORA_F16 ? launch_dtype<__half>(a, vec, grid, smem, stream)
                          : launch_dtype<__nv_bfloat16>(a, vec, grid, smem, stream);
}

}  // namespace lora
