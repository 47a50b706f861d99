// Expand / expand_slice: out[t, off_s + n] (+)= scale * sum_i y[t, s*ys + i] * B_s[l, n, i].
//
// Pages: vLLM PR #11579 "[misc] Add LoRA kernel micro benchmarks"
// (bgmv_expand, sgmv_expand, the _slice forms with num_slices, add_inputs
// adding the product to the existing outputs, the f32 x f16 => f16 typing);
// Punica issue #17
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
#include <string.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "frag.cuh"
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

template <typename E, bool ADD, bool VEC>
__global__ void __launch_bounds__(kThreads)
expand_kernel(const ExpandArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_rows[kTile];
    grid_dep_wait();  // y (and anything else) may come from the previous kernel
    grid_dep_launch();

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
        const int l = tl.x, n = tl.z;
        const int rl = l >= 0 && l < a.L ? clamp_rank(a.ranks, l, R) : 0;
        if (threadIdx.x == 0 && blockIdx.y == 0) plan_check_tile(tl, a.L, a.hdr);

        if (threadIdx.x < kTile) {
            int row = __ldcg(a.tile_rows + (int64_t)tile * kTile + threadIdx.x);
            if (blockIdx.y == 0) plan_check_row(row, a.T, a.hdr);
            if (row >= a.T) row = -1;
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
                    if (VEC) st_global_v4(p, make_uint4(0, 0, 0, 0));
                    else st8_u16(reinterpret_cast<uint16_t *>(p), make_uint4(0, 0, 0, 0), ncols - c8);
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

        // 1) issue the reads of out early (they overlap the staging below);
        //    unaligned rows element by element, all loads independent
        uint4 old[4][2];
        if (ADD && wact && wcol < ncols) {
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) {
                if (mb < nmb) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int r = s_rows[mb * 16 + g + 8 * h];
                        if (r < 0) continue;
                        const E *src = out + (int64_t)r * a.ldo + col0 + wcol;
                        if (VEC) old[mb][h] = ld_global_v4(src);
                        else old[mb][h] = ld8_u16<false>(reinterpret_cast<const uint16_t *>(src), ncols - wcol);
                    }
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
                    v = ld8_u16<true>(reinterpret_cast<const uint16_t *>(src), nv);
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
                    } else if (wcol < ncols) {
                        if (ADD) {
                            float o[8];
                            unpack8<E>(old[mb][h], o);
#pragma unroll
                            for (int k = 0; k < 8; ++k) res[k] += o[k];
                        }
                        st8_u16(reinterpret_cast<uint16_t *>(p), pack8<E>(res), ncols - wcol);
                    }
                }
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Warp-streaming expand: the fast path (16-byte aligned out columns, R % 8 == 0).
//
// Every warp works alone: no shared memory, no block barriers.  A warp unit
// is (plan tile, 32-row half of the tile, 32-column block of one slice); the
// units are split in contiguous, tile-major ranges over all warps of a
// persistent grid, so a warp's consecutive units share their token rows and,
// within one slice, their y fragments (kept in registers).
//
// Operands go straight from global memory into mma.sync fragments.  The
// contraction index is permuted so that each thread's slots of one 16-wide
// k step, {2q, 2q+1, 2q+8, 2q+9}, are the 4 consecutive ranks 4q..4q+3: the
// thread reads 8 contiguous bytes of a B row and 16 contiguous bytes of a y
// row per k step.  The output columns are permuted the same way (n-tile i,
// column c -> 8*(c/2) + 2i + c%2), so each thread's accumulators are 8
// contiguous output columns: out is read and written with 16-byte accesses.
// With ~20 warps per SM, each holding 64 bytes of out reads and the B / y
// reads of its unit in flight, the SM keeps enough HBM traffic outstanding
// (plain loads sustain ~7 TB/s on this part; cp.async and small bulk copies
// measured far lower).
constexpr int kWThreads = 128;  // 4 independent warps per CTA
constexpr int kWCols = 32;      // output columns per warp unit
constexpr int kWPrefetch = 8;   // units of a warp whose out rows are prefetched into L2
// Token rows per warp unit: MB m16 blocks, MB = 2 for ranks <= 32 and 1 above
// (the y fragments of a unit live in registers).
__host__ __device__ constexpr int warp_mb(int ksmax) { return ksmax >= 4 ? 1 : 2; }

// Loads of one warp unit that are issued a unit ahead.
template <int MB, int KSMAX>
struct UnitLoads {
    uint4 old[MB][2];     // out[row][8 columns] for rows g, g+8 of each m16 block
    uint2 bf[KSMAX][4];   // B fragments per k step and n-tile
};

template <typename E, bool ADD, int MB, int KSMAX>
__device__ __forceinline__ void issue_unit(const ExpandArgs &a, UnitLoads<MB, KSMAX> &ld,
                                           const int (&rows)[MB][2], int l, int rl, int KS,
                                           int s, int c0, int64_t col, bool col_ok, int g, int q) {
    const E *out = static_cast<const E *>(a.out);
    if (ADD && col_ok) {
#pragma unroll
        for (int mm = 0; mm < MB; ++mm)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (rows[mm][h] >= 0) ld.old[mm][h] = ld_global_v4(out + (int64_t)rows[mm][h] * a.ldo + col);
    }
    const int Ns = a.N[s];
    load_bfrags<E, KSMAX>(ld.bf, static_cast<const E *>(a.B[s]) + (int64_t)l * Ns * a.R, Ns, a.R,
                          c0, rl, KS, g, q);
}

template <typename E, bool ADD, int KSMAX>
__global__ void __launch_bounds__(kWThreads, KSMAX >= 8 ? 0 : (KSMAX >= 2 ? 3 : 4))
expand_warp_kernel(const ExpandArgs a, int tiles_grid, int ncb, int y_vec) {
    constexpr int MB = warp_mb(KSMAX);
    constexpr int kWRows = 16 * MB;
    constexpr int kParts = kTile / kWRows;  // row parts per tile
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int gwarp = blockIdx.x * (kWThreads / 32) + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * (kWThreads / 32);

    // units (tile, row part, column block), tile-major; ranges use the host's
    // tile bound so the first tile record loads together with the header
    const int per_tile = kParts * ncb;
    const long long U_grid = (long long)tiles_grid * per_tile;
    long long per = (U_grid + nwarps - 1) / nwarps;
    long long u_begin = gwarp * per;
    const int4 h0 = __ldg(reinterpret_cast<const int4 *>(a.hdr));
    const int4 h1 = __ldg(reinterpret_cast<const int4 *>(a.hdr) + 1);
    int t = (int)(u_begin / per_tile);
    int4 tl = t < a.max_tiles ? __ldg(a.tiles + t) : make_int4(-1, 0, 0, 0);
    // position of the current unit, and its token rows (the plan's per-tile
    // row lists, -1 padded), read in the same round trip as the header
    int part = (int)(u_begin - (long long)t * per_tile) / ncb;
    int cbi = (int)(u_begin - (long long)t * per_tile) - part * ncb;
    auto load_rows = [&](int tt, int pt, int (&r)[MB][2]) {
#pragma unroll
        for (int mm = 0; mm < MB; ++mm)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                int row = __ldg(a.tile_rows + (int64_t)tt * kTile + pt * kWRows + mm * 16 + g + 8 * h);
                r[mm][h] = row >= a.T ? -1 : row;
            }
    };
    int rows[MB][2];
    load_rows(t < a.max_tiles ? t : 0, part, rows);
    if (h0.x != LORA_PLAN_MAGIC || h0.y != a.T || h0.z != a.L) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_MISMATCH);
        return;
    }
    const int n_tiles = min(h1.z, a.max_tiles);
    if (n_tiles > tiles_grid) {
        // More tiles than the host's bound (a segment table not sorted by
        // adapter): spread all of them over the warps instead.
        per = ((long long)n_tiles * per_tile + nwarps - 1) / nwarps;
        u_begin = gwarp * per;
        t = (int)(u_begin / per_tile);
        part = (int)(u_begin - (long long)t * per_tile) / ncb;
        cbi = (int)(u_begin - (long long)t * per_tile) - part * ncb;
        if (t < n_tiles) {
            tl = __ldg(a.tiles + t);
            load_rows(t, part, rows);
        }
    }
    const long long u_end = min((long long)n_tiles * per_tile, u_begin + per);
    if (u_begin >= u_end) return;
    E *__restrict__ out = static_cast<E *>(a.out);

    // per (tile, part) state
    int rl = 0, KS = 0, nrow = 0;
    auto slice_of = [&](int c, int &s, int &c0) {
        s = 0;
        while (s + 1 < a.num_slices && c >= a.chunk_begin[s + 1]) ++s;
        c0 = (c - a.chunk_begin[s]) * kWCols;
    };
    rl = tl.x >= 0 && tl.x < a.L ? clamp_rank(a.ranks, tl.x, a.R) : 0;
    KS = (rl + 15) / 16;
    nrow = min(kWRows, tl.z - part * kWRows);
    if (lane == 0) plan_check_tile(tl, a.L, a.hdr);
#ifdef LORA_DEBUG
    // (the rows above were read before the tile count was known; checked
    // only now that this unit's tile is one of the plan's)
    auto check_rows = [&](int tt, int pt) {
        for (int mm = 0; mm < MB; ++mm)
            for (int h = 0; h < 2; ++h)
                plan_check_row(__ldg(a.tile_rows + (int64_t)tt * kTile + pt * kWRows + mm * 16 + g + 8 * h),
                               a.T, a.hdr);
    };
    check_rows(t, part);
#endif

    int s, c0;
    slice_of(cbi, s, c0);
    int64_t col = (int64_t)a.off[s] + c0 + 8 * q;
    bool col_ok = c0 + 8 * q < a.N[s];
    UnitLoads<MB, KSMAX> cur, nxt;
    if (nrow > 0 && rl > 0) issue_unit<E, ADD, MB, KSMAX>(a, cur, rows, tl.x, rl, KS, s, c0, col, col_ok, g, q);
    // The warp's later units of the same (tile, row part): their old out
    // values into L2 now (the loads one unit ahead then hit L2).  Chained
    // after the shrink this runs before the wait, so from the second unit on;
    // otherwise the second unit's loads follow at once, so from the third.
    if (ADD && nrow > 0 && rl > 0) {
        const int skip = a.early ? 1 : 2;
        int pc = cbi + skip;
        for (long long pu = u_begin + skip; pu < u_end && pc < ncb && pu < u_begin + kWPrefetch;
             ++pu, ++pc) {
            int ps, pc0;
            slice_of(pc, ps, pc0);
            if (pc0 + 8 * q >= a.N[ps]) continue;
            const int64_t pcol = (int64_t)a.off[ps] + pc0 + 8 * q;
#pragma unroll
            for (int mm = 0; mm < MB; ++mm)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (rows[mm][h] >= 0) prefetch_l2(out + (int64_t)rows[mm][h] * a.ldo + pcol);
        }
    }

    int y_s = -1;  // slice whose y fragments are held (same tile and part)
    float fscale[MB][2];
    uint32_t ah[MB][KSMAX][4], al[MB][KSMAX][4];

    // As a programmatic dependent of the shrink, everything above (plan, out,
    // B) overlaps the shrink's tail; y is read only after this wait.  A
    // following dependent waits for this grid in turn.
    grid_dep_wait();
    grid_dep_launch();

    for (long long u = u_begin; u < u_end; ++u) {
        // ---- the next unit: position, and its loads issued now
        int nt = t, npart = part, ncbi = cbi + 1;
        if (ncbi == ncb) {
            ncbi = 0;
            if (++npart == kParts) {
                npart = 0;
                ++nt;
            }
        }
        const bool has_next = u + 1 < u_end;
        int4 ntl = tl;
        int nrows_[MB][2];
        int nrl = rl, nKS = KS, nnrow = nrow;
        const bool new_rows = has_next && (nt != t || npart != part);
        if (new_rows) {
            if (nt != t) {
                ntl = __ldg(a.tiles + nt);
                if (lane == 0) plan_check_tile(ntl, a.L, a.hdr);
                nrl = ntl.x >= 0 && ntl.x < a.L ? clamp_rank(a.ranks, ntl.x, a.R) : 0;
                nKS = (nrl + 15) / 16;
            }
            load_rows(nt, npart, nrows_);
#ifdef LORA_DEBUG
            check_rows(nt, npart);
#endif
            nnrow = min(kWRows, ntl.z - npart * kWRows);
        }
        int ns = s, nc0 = c0;
        int64_t ncol = col;
        bool ncol_ok = col_ok;
        if (has_next) {
            slice_of(ncbi, ns, nc0);
            ncol = (int64_t)a.off[ns] + nc0 + 8 * q;
            ncol_ok = nc0 + 8 * q < a.N[ns];
            if (nnrow > 0 && nrl > 0) {
                if (new_rows) issue_unit<E, ADD, MB, KSMAX>(a, nxt, nrows_, ntl.x, nrl, nKS, ns, nc0, ncol, ncol_ok, g, q);
                else issue_unit<E, ADD, MB, KSMAX>(a, nxt, rows, ntl.x, nrl, nKS, ns, nc0, ncol, ncol_ok, g, q);
            }
        }

        // ---- the current unit
        if (nrow > 0) {
            if (rl == 0) {  // adapter -1 or rank 0: untouched with add_inputs, zeros without
                if (!ADD && col_ok) {
#pragma unroll
                    for (int mm = 0; mm < MB; ++mm)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            if (rows[mm][h] >= 0)
                                st_global_v4(out + (int64_t)rows[mm][h] * a.ldo + col, make_uint4(0, 0, 0, 0));
                }
            } else {
                if (s != y_s) {  // y fragments of (tile, part, slice)
                    y_s = s;
                    build_yfrags<E, MB, KSMAX, false>(ah, al, fscale, rows,
                                                      a.y + (int64_t)s * a.y_slice_stride, a.ldy,
                                                      rl, KS, a.scale, y_vec != 0, q);
                }
#pragma unroll
                for (int mm = 0; mm < MB; ++mm) {
                    if (mm * 16 >= nrow) break;
                    expand_block<E, ADD, KSMAX>(out, a.ldo, col, rows[mm], ah[mm], al[mm], cur.bf,
                                                fscale[mm], cur.old[mm], KS, col_ok);
                }
            }
        }

        // ---- advance
        if (!has_next) break;
        if (new_rows) {
#pragma unroll
            for (int mm = 0; mm < MB; ++mm)
#pragma unroll
                for (int h = 0; h < 2; ++h) rows[mm][h] = nrows_[mm][h];
            y_s = -1;
        }
        t = nt;
        part = npart;
        cbi = ncbi;
        tl = ntl;
        rl = nrl;
        KS = nKS;
        nrow = nnrow;
        s = ns;
        c0 = nc0;
        col = ncol;
        col_ok = ncol_ok;
        cur = nxt;
    }
}

// ---------------------------------------------------------------------------
// Tensor-core expand (aligned shapes; ranks above 48, or 17-48 on batches
// large enough for spans of two or more chunks): one CTA per (plan
// tile, span of `cpb` consecutive 128-column chunks of one slice).  The tile's
// y rows are read and turned into scaled hi/lo fp16/bf16 pairs (per-row
// power-of-two scale, as in the warp kernel) once per CTA, in the
// 128-byte-swizzled K-major layout; then, per chunk, one thread issues
// D = Y_hi . B^T + Y_lo . B^T as tcgen05.mma (M = 128 token lanes, the tile's
// 64 tokens plus rows of whatever follows, whose results are never read;
// N = 128 columns; K = 16 per step) into TMEM, and warps 0 and 1 read their
// token lanes back, scale, add the old out values and store 16-byte groups.
// The chunks are pipelined: the next chunk's out block is requested before
// the current chunk's MMA (two out buffers), the next B block by warps 2
// and 3 while warps 0 and 1 run the epilogue (one B buffer, free once the
// MMA is done).
constexpr int kTcCols = 128;                    // output columns per chunk (N)
constexpr int kTcThreads = 256;                 // 8 warps: two per TMEM lane quadrant
constexpr int kTcWaves = 3;                     // least waves of CTAs a span size leaves
constexpr int kTcMaxSpan = 256;                 // chunks per span at most
constexpr int kTcOutPitch = kTcCols * 2 + 16;   // bytes per staged out row

// Shared memory: [Yh | Yl] per 64-wide rank half, then the B halves and the
// two out buffers (the second also holds the fp32 y rows before the
// conversion); 1024 bytes of alignment slack in front.
__host__ __device__ constexpr int tc_halves(int R) { return R > 64 ? 2 : 1; }
__host__ __device__ constexpr int tc_ypitch(int R) { return (R + 15) / 16 * 16; }  // floats
__host__ __device__ constexpr int tc_out1_bytes(int R) {
    return kTile * kTcOutPitch > kTile * tc_ypitch(R) * 4 ? kTile * kTcOutPitch
                                                          : kTile * tc_ypitch(R) * 4;
}
__host__ __device__ constexpr int tc_expand_smem(int R) {
    return 1024 + tc_halves(R) * (2 * kTile * 128 + kTcCols * 128) + kTile * kTcOutPitch +
           tc_out1_bytes(R);
}

struct BMaps {
    CUtensorMap m[LORA_MAX_SLICES];  // B_s as [L * N_s][R], boxes of 128 rows x 64 ranks
};

// Byte offset of (token row i, 16-byte column group c8) in a staged out block:
// two boxes of 64 columns, each [64 rows][128 B] in the 128-byte swizzled
// layout a TMA load writes (group g of a row at g ^ (row & 7)), so the
// epilogue's row-per-lane reads fall in eight different bank groups.
__device__ __forceinline__ int out_off(int i, int c8) {
    return (c8 >> 3) * (kTile * 128) + i * 128 + (((c8 & 7) ^ (i & 7)) << 4);
}

template <typename E, bool ADD>
__global__ void __launch_bounds__(kTcThreads)
expand_tc_kernel(const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ BMaps tm_b,
                 const ExpandArgs a, int cpb, int tma, int tma_b) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_rows[kTile];
    __shared__ float s_f[kTile];
    __shared__ uint64_t s_bar;
    __shared__ uint64_t s_oful[2];  // TMA out block b has landed
    __shared__ uint64_t s_bful;     // the TMA B block has landed
    __shared__ uint32_t s_tmem;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int span = blockIdx.y;

    // plan header, first tile record and its token rows in one round trip
    const int4 h0 = __ldg(reinterpret_cast<const int4 *>(a.hdr));
    const int4 h1 = __ldg(reinterpret_cast<const int4 *>(a.hdr) + 1);
    int tile = blockIdx.x;
    int4 tl = tile < a.max_tiles ? __ldg(a.tiles + tile) : make_int4(-1, 0, 0, 0);
    int my_row = threadIdx.x < kTile && tile < a.max_tiles
                     ? __ldg(a.tile_rows + (int64_t)tile * kTile + threadIdx.x)
                     : -1;
    if (h0.x != LORA_PLAN_MAGIC || h0.y != a.T || h0.z != a.L) {
        if (tile == 0 && span == 0 && threadIdx.x == 0)
            atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_MISMATCH);
        return;
    }
    // The grid covers the host's tile bound; a plan with more tiles (segment
    // tables not sorted by adapter) is covered by CTAs taking tile + gridDim.x.
    const int n_tiles = min(h1.z, a.max_tiles);

    int s = 0;
    while (s + 1 < a.num_slices && span >= a.chunk_begin[s + 1]) ++s;
    const int n_span = (span - a.chunk_begin[s]) * kTcCols * cpb;  // first column in slice s
    const int span_cols = min(kTcCols * cpb, a.N[s] - n_span);      // > 0, a multiple of 8
    const int nsub = (span_cols + kTcCols - 1) / kTcCols;
    const int64_t colbase = (int64_t)a.off[s] + n_span;
    E *__restrict__ out = static_cast<E *>(a.out);
    const int R = a.R, KH = tc_halves(R), YP = tc_ypitch(R);
    unsigned char *sm = smem + ((1024 - (smem_u32(smem) & 1023)) & 1023);
    unsigned char *sY = sm;                                   // [KH][Yh 64 rows | Yl 64 rows] x 128 B
    unsigned char *sB = sY + KH * 2 * kTile * 128;             // [KH][128 rows] x 128 B
    unsigned char *sO0 = sB + KH * kTcCols * 128;              // [64][kTcOutPitch]
    unsigned char *sO1 = sO0 + kTile * kTcOutPitch;            // [64][kTcOutPitch], first y
    float *sYf = reinterpret_cast<float *>(sO1);               // [64][YP] before the conversion
    const uint32_t idesc = tc_idesc_f16(std::is_same<E, __nv_bfloat16>::value, 128, kTcCols);

    bool have_tmem = false;   // TMEM and the barrier are set up on the first tile needing them
    uint32_t tmem = 0, ncommit = 0;
    uint32_t nof0 = 0, nof1 = 0;  // completed phases of s_oful[0], s_oful[1]
    int of_pending = 0;           // bit b: out buffer b has a TMA copy not yet waited for
    uint32_t nbf = 0;             // completed phases of s_bful
    bool bf_timed_out = false;    // (thread 0) a wait for a TMA B block ran out
    bool timed_out = false;
    for (; tile < n_tiles; tile += gridDim.x) {
        if (tile != (int)blockIdx.x) {
            tl = __ldg(a.tiles + tile);
            my_row = threadIdx.x < kTile ? __ldg(a.tile_rows + (int64_t)tile * kTile + threadIdx.x)
                                         : -1;
            __syncthreads();  // the previous tile is done with s_rows / s_f
        }
        if (threadIdx.x < kTile) {
            plan_check_row(my_row, a.T, a.hdr);
            s_rows[threadIdx.x] = my_row < a.T ? my_row : -1;
        }
        if (threadIdx.x == 0) plan_check_tile(tl, a.L, a.hdr);
        const int l = tl.x, n = tl.z;
        const int rl = l >= 0 && l < a.L ? clamp_rank(a.ranks, l, a.R) : 0;
        __syncthreads();

        if (rl == 0) {  // adapter -1 or rank 0: untouched with add_inputs, zeros without
            grid_dep_wait();
            grid_dep_launch();
            if (!ADD)
                for (int it = threadIdx.x; it < n * (span_cols / 8); it += kTcThreads) {
                    const int i = it / (span_cols / 8), c8 = it - i * (span_cols / 8);
                    const int row = s_rows[i];
                    if (row >= 0)
                        st_global_v4(out + (int64_t)row * a.ldo + colbase + 8 * c8, make_uint4(0, 0, 0, 0));
                }
            continue;
        }

        const int KS = (rl + 15) / 16;
        const E *Bl = static_cast<const E *>(a.B[s]) + ((int64_t)l * a.N[s] + n_span) * R;

        // Tiles of consecutive token rows (sorted SGMV segments): their out
        // blocks come by TMA, two 64 x 64 boxes per chunk from one thread.
        const int xrow0 = s_rows[0];
        const bool tma_tile =
            __syncthreads_and(tma && ADD && xrow0 >= 0 &&
                              ((int)threadIdx.x >= n || (int)threadIdx.x >= kTile ||
                               s_rows[threadIdx.x] == xrow0 + (int)threadIdx.x)) != 0;
        // full tiles of consecutive rows also store their full chunks by TMA
        // (a box covers 64 rows: rows of other tiles must not be written)
        const bool st_tma = tma_tile && n == kTile;
        // chunk j's out block into buffer b (every thread calls), in the
        // 128-byte swizzled layout of two 64-column boxes (out_off)
        auto load_out = [&](int b, int j) {
            unsigned char *dst = b ? sO1 : sO0;
            const int c0 = j * kTcCols;
            if (tma_tile) {
                if (threadIdx.x == 0) {
                    tma_store_wait_read();     // a TMA store from this buffer has read it
                    fence_proxy_async_smem();  // (the buffer's generic reads came first)
                    mbar_arrive_expect_tx(&s_oful[b], 2 * kTile * 128);
                    tma_load_2d(smem_u32(dst), &tm_out, (int)(colbase + c0), xrow0, &s_oful[b]);
                    tma_load_2d(smem_u32(dst + kTile * 128), &tm_out, (int)(colbase + c0 + 64),
                                xrow0, &s_oful[b]);
                }
                of_pending |= 1 << b;
                return;
            }
            const int c8n = min(kTcCols, span_cols - c0) / 8;
            for (int it = threadIdx.x; it < n * c8n; it += kTcThreads) {
                const int i = it / c8n, c8 = it - i * c8n;
                const int row = s_rows[i];
                if (row >= 0)
                    cp_async16(smem_u32(dst + out_off(i, c8)),
                               out + (int64_t)row * a.ldo + colbase + c0 + 8 * c8, 16);
            }
        };
        // chunk j's B block (8 ranks per 16-byte piece, ranks >= rl zero-filled);
        // at full rank R (a multiple of 64) by TMA from the caller's thread t0 == 0:
        // 128 rows (output columns) of 64 ranks per box, the same swizzled layout
        const bool b_tma = tma_b && rl == R;
        auto load_b = [&](int j, int t0, int nt) {
            if (b_tma) {
                if (t0 == 0) {
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(&s_bful, (uint32_t)(KH * kTcCols * 128));
                    for (int h = 0; h < KH; ++h)
                        tma_load_2d(smem_u32(sB + h * kTcCols * 128), &tm_b.m[s], 64 * h,
                                    l * a.N[s] + n_span + j * kTcCols, &s_bful);
                }
                return;
            }
            const int c0 = j * kTcCols, nc = min(kTcCols, span_cols - c0);
            const E *Bj = Bl + (int64_t)c0 * R;
            for (int it = t0; it < nc * KS * 2; it += nt) {
                const int jj = it / (KS * 2), k8 = it - jj * (KS * 2);
                const int nv = min(8, rl - 8 * k8);
                cp_async16(smem_u32(sB + (k8 >> 3) * kTcCols * 128 + jj * 128 + (((k8 & 7) ^ (jj & 7)) << 4)),
                           Bj + (int64_t)jj * R + (nv > 0 ? 8 * k8 : 0), nv > 0 ? 2 * nv : 0);
            }
        };

        if (!have_tmem) {
            if (warp == 0) tc_alloc(&s_tmem, kTcCols);
            if (threadIdx.x == 0) {
                mbar_init(&s_bar, 1);
                mbar_init(&s_oful[0], 1);
                mbar_init(&s_oful[1], 1);
                mbar_init(&s_bful, 1);
            }
        }

        // first chunk's out and B blocks (neither written by the previous kernel)
        if (ADD) load_out(0, 0);
        load_b(0, threadIdx.x, kTcThreads);
        cp_async_commit();

        // y rows: produced by the previous kernel
        grid_dep_wait();
        grid_dep_launch();
        const float *ys = a.y + (int64_t)s * a.y_slice_stride;
        for (int it = threadIdx.x; it < n * KS * 4; it += kTcThreads) {  // 4 ranks per chunk
            const int i = it / (KS * 4), k4 = it - i * (KS * 4);
            const int row = s_rows[i];
            const int nv = row >= 0 ? min(4, rl - 4 * k4) : 0;
            cp_async16(smem_u32(sYf + i * YP + 4 * k4),
                       ys + (int64_t)(row >= 0 ? row : 0) * a.ldy + (nv > 0 ? 4 * k4 : 0),
                       nv > 0 ? 4 * nv : 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();

        // y -> scaled hi/lo operands.  The G threads of a row (G = KS * 2 chunks
        // of 8 ranks rounded up to a power of two, so a row's group is aligned
        // inside one warp) reduce its max; padding chunks hold zeros.
        {
            const int G = KS <= 1 ? 2 : (KS <= 2 ? 4 : (KS <= 4 ? 8 : 16));
            for (int it = threadIdx.x; it < kTile * G; it += kTcThreads) {
                const int i = it / G, k8 = it - i * G;
                const bool live = i < n && k8 < KS * 2;
                float v[8];
                float m = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    v[k] = live ? sYf[i * YP + 8 * k8 + k] : 0.f;
                    m = fmaxf(m, fabsf(v[k]));
                }
                for (int o = 1; o < G; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                const int e = row_exponent(m);
                const float inv = exp2i(-e);
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] *= inv;
                uint4 hi, lo;
                split_hilo8<E>(v, hi, lo);
                unsigned char *yh = sY + (k8 >> 3) * 2 * kTile * 128;
                const int off = i * 128 + (((k8 & 7) ^ (i & 7)) << 4);
                *reinterpret_cast<uint4 *>(yh + off) = hi;
                *reinterpret_cast<uint4 *>(yh + kTile * 128 + off) = lo;
                if (k8 == 0) s_f[i] = a.scale * exp2i(e);
            }
        }
        tc_fence_before();
        __syncthreads();  // the y rows in sO1 are consumed; sO1 may take chunk 1's out block
        tc_fence_after();
        if (!have_tmem) {
            tmem = s_tmem;
            have_tmem = true;
        }

        for (int j = 0; j < nsub; ++j) {
            unsigned char *sOc = (j & 1) ? sO1 : sO0;
            // next chunk's out block into the other buffer (its epilogue is over)
            if (ADD && j + 1 < nsub) load_out((j + 1) & 1, j + 1);
            cp_async_commit();
            cp_async_wait<1>();          // this chunk's out and B blocks are in
            if (ADD && tma_tile) {       // (the out block by TMA)
                const uint32_t nf = (j & 1) ? nof1 : nof0;
                if (!mbar_wait_cta(&s_oful[j & 1], nf & 1) && threadIdx.x == 0)
                    atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_TIMEOUT);
                if (j & 1) ++nof1;
                else ++nof0;
                of_pending &= ~(1 << (j & 1));
            }
            fence_proxy_async_smem();    // ... and visible to the tensor cores
            __syncthreads();
            tc_fence_after();
            if (b_tma) {  // (the B block by TMA: only the issuing thread reads it)
                if (threadIdx.x == 0 && !mbar_wait_cta(&s_bful, nbf & 1)) {
                    atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_TIMEOUT);
                    bf_timed_out = true;
                }
                ++nbf;
            }
            if (threadIdx.x == 0) {
                for (int k = 0; k < KS; ++k) {
                    const int h = k >> 2;
                    const uint32_t yh = smem_u32(sY) + h * 2 * kTile * 128 + 32 * (k & 3);
                    const uint32_t bb = smem_u32(sB) + h * kTcCols * 128 + 32 * (k & 3);
                    tc_mma_f16(tmem, tc_desc_sw128(yh), tc_desc_sw128(bb), idesc, k > 0);
                    tc_mma_f16(tmem, tc_desc_sw128(yh + kTile * 128), tc_desc_sw128(bb), idesc, true);
                }
                tc_commit(&s_bar);
            }
            // A wait that runs out (never expected) flags the plan and ends the
            // CTA without touching out: no epilogue, no further loads.
            const bool to = !mbar_wait_cta(&s_bar, ncommit & 1);
            ++ncommit;
            if (__syncthreads_or(to)) {
                if (threadIdx.x == 0) atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_TIMEOUT);
                timed_out = true;
                break;
            }
            tc_fence_after();

            if ((warp & 3) >= 2) {
                // the MMA has read B: next chunk's B block (warps 2, 3, 6, 7)
                if (j + 1 < nsub)
                    load_b(j + 1, ((warp >> 2) * 2 + (warp & 1)) * 32 + lane, kTcThreads / 2);
                cp_async_commit();
            } else {
                // epilogue: TMEM lane quadrants 0 and 1 hold the tile's 64
                // token lanes; warps w and w + 4 share a quadrant and split
                // the chunk's columns in halves
                const int q = warp & 3, half = warp >> 2;
                const int i = 32 * q + lane;
                const int row = i < n ? s_rows[i] : -1;
                const float f = s_f[i];
                const uint32_t tl_addr = tmem + ((uint32_t)(32 * q) << 16);
                const int cj = j * kTcCols, nc = min(kTcCols, span_cols - cj);
                for (int c0 = half * (kTcCols / 2); c0 < min(nc, (half + 1) * (kTcCols / 2));
                     c0 += 32) {  // warp-uniform
                    float d[32];
                    tc_ld32(tl_addr + c0, d);
                    if (row < 0) continue;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int c = c0 + 8 * g;
                        if (c >= nc) break;
                        float v[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) v[k] = f * d[8 * g + k];
                        if (ADD) {
                            float o[8];
                            unpack8<E>(*reinterpret_cast<const uint4 *>(sOc + out_off(i, c / 8)), o);
#pragma unroll
                            for (int k = 0; k < 8; ++k) v[k] += o[k];
                        }
                        if (st_tma && nc == kTcCols)  // in place, stored by TMA below
                            *reinterpret_cast<uint4 *>(sOc + out_off(i, c / 8)) = pack8<E>(v);
                        else
                            st_global_v4(out + (int64_t)row * a.ldo + colbase + cj + c, pack8<E>(v));
                    }
                }
            }
            const bool chunk_st = st_tma && min(kTcCols, span_cols - j * kTcCols) == kTcCols;
            if (chunk_st) fence_proxy_async_smem();  // the results -> the TMA store
            tc_fence_before();
            __syncthreads();  // TMEM and this out buffer are free again
            if (chunk_st && threadIdx.x == 0) {
                tma_store_2d(&tm_out, (int)(colbase + j * kTcCols), xrow0, smem_u32(sOc));
                tma_store_2d(&tm_out, (int)(colbase + j * kTcCols + 64), xrow0,
                             smem_u32(sOc + kTile * 128));
                tma_store_commit();
            }
        }
        cp_async_wait<0>();
        // TMA stores of this tile have read their buffers before the next
        // tile writes them (the next tile starts with a barrier)
        if (threadIdx.x == 0) tma_store_wait_read();
        if (timed_out) break;
    }
    if (threadIdx.x == 0) tma_store_wait_all();
    for (int b = 0; b < 2; ++b)  // (left by a timed-out chunk) no copy may land after exit
        if (of_pending & (1 << b)) mbar_wait_cta(&s_oful[b], (b ? nof1 : nof0) & 1);
    if (bf_timed_out) mbar_wait_cta(&s_bful, (nbf - 1) & 1);
    if (have_tmem) {
        cp_async_wait<0>();
        // after a timed-out wait, give the MMA one more bounded wait before
        // the accumulator columns are released
        if (timed_out) mbar_wait_cta(&s_bar, (ncommit - 1) & 1);
        __syncthreads();
        tc_fence_after();
        if (warp == 0) tc_dealloc(tmem, kTcCols);
    }
}

template <typename E, bool ADD, bool VEC>
cudaError_t configure_one() {
    const int ks = LORA_MAX_RANK / 16;
    const int smem = (kCols + 2 * kTile) * pitch_of(ks) * (int)sizeof(E) + kTile * (int)sizeof(float);
    return cudaFuncSetAttribute(expand_kernel<E, ADD, VEC>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// Static shared memory of the tensor-core kernels [dtype][add], and the SM's
// shared memory and per-block reservation, for their residency.
int g_tc_static[2][2] = {};
int g_smem_sm = 0, g_smem_reserved = 0;

template <typename E>
cudaError_t configure_tc(int (&stat)[2]) {
    cudaError_t e = cudaSuccess;
    for (int add = 0; add < 2; ++add) {
        const void *k = add ? reinterpret_cast<const void *>(expand_tc_kernel<E, true>)
                            : reinterpret_cast<const void *>(expand_tc_kernel<E, false>);
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc_expand_smem(LORA_MAX_RANK));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        cudaFuncAttributes fa;
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        stat[add] = (int)fa.sharedSizeBytes;
    }
    return e;
}

template <typename E>
cudaError_t launch_tc(const ExpandArgs &a, dim3 grid, int cpb, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = tc_expand_smem(a.R);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    // out blocks of tiles of consecutive rows by TMA (add_inputs only): a map
    // over the columns the slices use
    CUtensorMap tm_out;
    memset(&tm_out, 0, sizeof(tm_out));
    int tma = 0;
    if (a.add) {
        int64_t used = 0;
        for (int s = 0; s < a.num_slices; ++s)
            used = std::max<int64_t>(used, (int64_t)a.off[s] + a.N[s]);
        tma = make_tensor_map_2d(&tm_out, std::is_same<E, __nv_bfloat16>::value ? LORA_BF16 : LORA_F16,
                                 a.out, (uint64_t)a.T, (uint64_t)used, (uint64_t)a.ldo, kTile) ==
                      cudaSuccess
                  ? 1
                  : 0;
    }
    // B blocks at full rank by TMA when R is a multiple of 64 (whole 128-byte rows)
    BMaps tm_b;
    memset(&tm_b, 0, sizeof(tm_b));
    int tma_b = 0;
    if (a.R % 64 == 0) {
        tma_b = 1;
        for (int s = 0; s < a.num_slices && tma_b; ++s)
            if (a.N[s] > 0 &&
                make_tensor_map_2d(&tm_b.m[s],
                                   std::is_same<E, __nv_bfloat16>::value ? LORA_BF16 : LORA_F16,
                                   a.B[s], (uint64_t)a.L * a.N[s], (uint64_t)a.R, (uint64_t)a.R,
                                   kTcCols) != cudaSuccess)
                tma_b = 0;
    }
    if (a.add)
        return cudaLaunchKernelEx(&cfg, expand_tc_kernel<E, true>, tm_out, tm_b, a, cpb, tma, tma_b);
    return cudaLaunchKernelEx(&cfg, expand_tc_kernel<E, false>, tm_out, tm_b, a, cpb, tma, tma_b);
}

template <typename E>
cudaError_t configure_dtype(int (&tc_static)[2]) {
    cudaError_t e;
    if ((e = configure_tc<E>(tc_static)) != cudaSuccess) return e;
    if ((e = configure_one<E, false, false>()) != cudaSuccess) return e;
    return configure_one<E, true, false>();
}

// Resident CTAs per SM of each warp-kernel instantiation [dtype][add][ks class],
// filled once per process by configure_expand_kernels.
int g_warp_occ[2][2][4] = {};

template <typename E, bool ADD, int KSMAX>
cudaError_t query_occ(int &occ) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, expand_warp_kernel<E, ADD, KSMAX>,
                                                         kWThreads, 0);
}

template <typename E>
cudaError_t query_occ_dtype(int (&occ)[2][4]) {
    cudaError_t e;
    if ((e = query_occ<E, false, 1>(occ[0][0])) != cudaSuccess) return e;
    if ((e = query_occ<E, false, 2>(occ[0][1])) != cudaSuccess) return e;
    if ((e = query_occ<E, false, 4>(occ[0][2])) != cudaSuccess) return e;
    if ((e = query_occ<E, false, 8>(occ[0][3])) != cudaSuccess) return e;
    if ((e = query_occ<E, true, 1>(occ[1][0])) != cudaSuccess) return e;
    if ((e = query_occ<E, true, 2>(occ[1][1])) != cudaSuccess) return e;
    if ((e = query_occ<E, true, 4>(occ[1][2])) != cudaSuccess) return e;
    return query_occ<E, true, 8>(occ[1][3]);
}

int ks_class(int ks) { return ks <= 1 ? 0 : ks <= 2 ? 1 : ks <= 4 ? 2 : 3; }

template <typename E, int KSMAX>
cudaError_t launch_warp_ks(const ExpandArgs &a, int grid, int tiles_grid, int ncb, cudaStream_t st,
                           bool pdl) {
    // 16-byte y loads when every slice's y block starts 16-byte aligned
    const int y_vec = (reinterpret_cast<uintptr_t>(a.y) & 15) == 0 && a.ldy % 4 == 0 &&
                      a.y_slice_stride % 4 == 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kWThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (a.add) return cudaLaunchKernelEx(&cfg, expand_warp_kernel<E, true, KSMAX>, a, tiles_grid, ncb, y_vec);
    return cudaLaunchKernelEx(&cfg, expand_warp_kernel<E, false, KSMAX>, a, tiles_grid, ncb, y_vec);
}

template <typename E>
cudaError_t launch_warp_dtype(const ExpandArgs &a, int grid, int tiles_grid, int ncb,
                              cudaStream_t st, bool pdl) {
    const int ks = (a.R + 15) / 16;
    if (ks <= 1) return launch_warp_ks<E, 1>(a, grid, tiles_grid, ncb, st, pdl);
    if (ks <= 2) return launch_warp_ks<E, 2>(a, grid, tiles_grid, ncb, st, pdl);
    if (ks <= 4) return launch_warp_ks<E, 4>(a, grid, tiles_grid, ncb, st, pdl);
    return launch_warp_ks<E, 8>(a, grid, tiles_grid, ncb, st, pdl);
}

template <typename E>
cudaError_t launch_dtype(const ExpandArgs &a, dim3 grid, size_t smem, cudaStream_t st) {
    if (a.add) expand_kernel<E, true, false><<<grid, kThreads, smem, st>>>(a);
    else expand_kernel<E, false, false><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t configure_expand_kernels() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&g_smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&g_smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e == cudaSuccess) e = configure_dtype<__half>(g_tc_static[LORA_F16]);
    if (e != cudaSuccess) return e;
    if ((e = configure_dtype<__nv_bfloat16>(g_tc_static[LORA_BF16])) != cudaSuccess) return e;
    if ((e = query_occ_dtype<__half>(g_warp_occ[LORA_F16])) != cudaSuccess) return e;
    return query_occ_dtype<__nv_bfloat16>(g_warp_occ[LORA_BF16]);
}

cudaError_t launch_expand(lora_dtype_t dt, const ExpandArgs &a_in, const DeviceInfo &dev,
                          cudaStream_t stream, bool pdl) {
    ExpandArgs a = a_in;
    if (a.T == 0) return cudaSuccess;
    // Tiles: ceil(T/64) full-or-partial tiles plus at most one ragged tile per
    // adapter and one for the inactive tokens; kernels loop if a plan has more.
    const long long est = (a.T + kTile - 1) / kTile + (long long)std::min(a.L, a.T) + 1;
    const int tiles_grid = (int)std::max<long long>(1, std::min<long long>(est, a.max_tiles));

    // Fast path: every 8-column group of every slice 16-byte aligned, B rows 16-byte aligned.
    bool vec = (reinterpret_cast<uintptr_t>(a.out) & 15) == 0 && a.ldo % 8 == 0 && a.R % 8 == 0;
    for (int s = 0; s < a.num_slices; ++s)
        vec = vec && a.off[s] % 8 == 0 && a.N[s] % 8 == 0 &&
              (reinterpret_cast<uintptr_t>(a.B[s]) & 15) == 0;
    const bool y_vec = (reinterpret_cast<uintptr_t>(a.y) & 15) == 0 && a.ldy % 4 == 0 &&
                       a.y_slice_stride % 4 == 0;
    // The tensor-core kernel for ranks above 48 (4+ k steps: the warp
    // kernel's per-unit B re-reads and register pressure grow with the rank),
    // and for ranks 17-48 when the batch is large enough for spans of two or
    // more chunks per CTA (the y conversion then pays for itself).  Measured,
    // prefill gate/up: r = 64 363 -> 155 us, r = 32 150 -> 135 us; at r = 16
    // and for decode batches the warp kernel is faster (its units are lighter
    // than a CTA's load/convert/MMA chain).
    // For plans grouped from segments (tiles of consecutive rows: out blocks
    // loaded and stored by TMA) also at r <= 16 when the batch is large.
    const int ksr = (a.R + 15) / 16;
    if (vec && y_vec && (ksr >= 2 || a.seg_plan)) {
        // spans of cpb 128-column chunks per slice: cpb is the largest power of
        // two that still leaves at least kTcWaves waves of CTAs
        const int dyn = tc_expand_smem(a.R);
        const long long by_smem =
            g_smem_sm / ((long long)dyn + g_tc_static[dt][a.add ? 1 : 0] + g_smem_reserved);
        // TMEM: 128 columns per CTA, 512 per SM
        const long long slots = (long long)dev.sm_count * std::max(1LL, std::min(by_smem, 4LL));
        auto spans = [&](long long c) {
            long long n = 0;
            for (int s = 0; s < a.num_slices; ++s) n += (a.N[s] + kTcCols * c - 1) / (kTcCols * c);
            return n;
        };
        int cpb = 1;
        while (cpb < kTcMaxSpan && (long long)tiles_grid * spans(2LL * cpb) >= kTcWaves * slots)
            cpb *= 2;
        if (ksr >= 4 || cpb >= 2) {
            a.chunk_begin[0] = 0;
            for (int s = 0; s < a.num_slices; ++s)
                a.chunk_begin[s + 1] =
                    a.chunk_begin[s] + (a.N[s] + kTcCols * cpb - 1) / (kTcCols * cpb);
            for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s)
                a.chunk_begin[s + 1] = a.chunk_begin[s];
            const int nspans = a.chunk_begin[a.num_slices];
            if (nspans == 0) return cudaSuccess;
            const dim3 grid(tiles_grid, nspans);
            return dt == LORA_F16 ? launch_tc<__half>(a, grid, cpb, stream, pdl)
                                  : launch_tc<__nv_bfloat16>(a, grid, cpb, stream, pdl);
        }
    }
    if (vec) {
        // 32-column blocks per slice (prefix sums in chunk_begin)
        a.chunk_begin[0] = 0;
        for (int s = 0; s < a.num_slices; ++s)
            a.chunk_begin[s + 1] = a.chunk_begin[s] + (a.N[s] + kWCols - 1) / kWCols;
        for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s) a.chunk_begin[s + 1] = a.chunk_begin[s];
        const int ncb = a.chunk_begin[a.num_slices];
        if (ncb == 0) return cudaSuccess;
        const int kss = (a.R + 15) / 16, ksmax = kss <= 1 ? 1 : kss <= 2 ? 2 : kss <= 4 ? 4 : 8;
        const long long units = (long long)tiles_grid * (kTile / (16 * warp_mb(ksmax))) * ncb;
        const int occ = std::max(1, g_warp_occ[dt][a.add ? 1 : 0][ks_class((a.R + 15) / 16)]);
        const long long warps_max = (long long)dev.sm_count * occ * (kWThreads / 32);
        const long long warps = std::min(units, warps_max);
        const int grid = (int)std::max<long long>(1, (warps + 3) / 4);
        return dt == LORA_F16 ? launch_warp_dtype<__half>(a, grid, tiles_grid, ncb, stream, pdl)
                              : launch_warp_dtype<__nv_bfloat16>(a, grid, tiles_grid, ncb, stream, pdl);
    }

    // Generic path: 128-column chunks per slice
    a.chunk_begin[0] = 0;
    for (int s = 0; s < a.num_slices; ++s)
        a.chunk_begin[s + 1] = a.chunk_begin[s] + (a.N[s] + kCols - 1) / kCols;
    for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s) a.chunk_begin[s + 1] = a.chunk_begin[s];
    const int chunks = a.chunk_begin[a.num_slices];
    if (chunks == 0) return cudaSuccess;
    dim3 grid(tiles_grid, chunks);
    const int ks = (a.R + 15) / 16;
    const size_t smem = (size_t)(kCols + 2 * kTile) * pitch_of(ks) * 2 + kTile * sizeof(float);
    return dt == LORA_F16 ? launch_dtype<__half>(a, grid, smem, stream)
                          : launch_dtype<__nv_bfloat16>(a, grid, smem, stream);
}

}  // namespace lora
