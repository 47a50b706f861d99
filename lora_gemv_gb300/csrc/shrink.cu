// Shrink: y[t, s*R + i] (+)= scale * sum_h x[t, h] * A[l, s*R + i, h]   (i < r_l)
//
// Pages: vLLM PR #15655 summary (the kernel split into shrink and expand
// variants); vLLM PR #11579 (bgmv_shrink / sgmv_shrink, the fp32 rank
// buffer, and split-K shrink whose partial results are added); Punica issue
// #17 (tokens of one adapter share its weights; ranks are not limited to
// bins of 16/32/64).
//
// Design (GB300): per plan tile (<= 64 tokens of one adapter) the cluster
// computes Y[64, rows] = X[64, H] . A_l[rows, H]^T on the tensor cores with
// fp32 accumulation, where rows are the adapter's S * r_l live rows only
// (rank-aware: padded rows are never read).
//  - H is split across a thread-block CLUSTER of up to 16 CTAs (split-K);
//    each CTA walks its H range in 128-wide stages through two shared-memory
//    buffers: aligned rows are copied with cp.async, both buffers at once
//    (for the decode split-K shapes a CTA's whole H range is then in
//    flight), other rows through registers one stage ahead;
//  - aligned rows (batches of more than 16 tokens per adapter on average):
//    the stages are laid out as 128-byte-swizzled K-major tcgen05 operands,
//    one thread issues each stage's eight M = 128 x N = rows x K = 16
//    tcgen05.mma (the x tile as A, its 64 token rows plus rows of whatever
//    follows, whose results are never read; the adapter rows as B) into a
//    TMEM accumulator, commits to a per-buffer mbarrier, and two warps read
//    the 64 token lanes back with tcgen05.ld;
//  - otherwise ldmatrix + mma.sync m16n8k16: the 8 warps split the tile's
//    16-row blocks and, within a block, either its 8-column n-tiles (every
//    output has one owner warp and the CTA partial is written straight from
//    the accumulators) or, for batches of a few tokens per adapter, each
//    stage's k steps (short mma chains; the warp partials are then summed
//    in shared memory);
//  - partials are summed over the cluster through distributed shared
//    memory, in a fixed order (deterministic, no global scratch, no
//    atomics), each CTA finishing a share of the tile's rows: every CTA
//    sends its partial rows to their owner's receive buffer with
//    asynchronous stores that count their bytes on the owner's mbarrier
//    (or, where the receive buffer would cost residency, the owners read
//    the partials after a cluster barrier);
//  - tiles of adapter -1 load nothing (block skipping); their y rows are
//    zeroed unless add_inputs.
#include <cooperative_groups.h>

#include <string.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace lora {
namespace {

constexpr int kThreads = 256;  // 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 128;     // compacted A rows per CTA (grid.z covers more)
constexpr int kK = 128;        // H elements per stage (256-byte rows)
constexpr int kCh = kK / 8;    // 16-byte chunks per row and stage

// Shared-memory bytes: two stages of (64 x rows + rows_cap A rows) x 256 B,
// reused after the k loop for the CTA partial [64][rows] and, for k-split
// warps, their partials [8 warps][16][rows].
__host__ __device__ constexpr int part_pitch(int ntmax) { return ntmax * 8 + 4; }
__host__ __device__ constexpr int smem_bytes(int rows_cap, int ntmax) {
    const int stages = 2 * (kTile + rows_cap) * kK * 2;
    const int parts = (kTile + kWarps * 16) * part_pitch(ntmax) * 4;
    return stages > parts ? stages : parts;
}

// Receive buffer of the push reduction, after the above: [ksplit][64 /
// ksplit rows][rows_cap] floats from the cluster's CTAs.
__host__ __device__ constexpr int recv_bytes(int rows_cap) { return kTile * rows_cap * 4; }

// Tensor-core path: 1024 bytes of alignment slack, the two stages in the
// tcgen05 layout (see async_stage_tc), then the rows the M = 128 operand
// window of the last x region reads past it (the MMA's rows 64..127 are not
// tokens; their results are never read).
__host__ __device__ constexpr int tc_stage_area(int rows_cap) {
    return 1024 + 2 * 2 * (kTile + rows_cap) * 128 + (rows_cap < 64 ? (64 - rows_cap) * 128 : 0);
}

// 256-byte rows, 16-byte chunks XOR-swizzled (within each 128-byte half) by the row.
__device__ __forceinline__ int swz(int row, int chunk) {
    return row * kK + ((chunk ^ (row & 7)) << 3);
}

// Loads per thread and stage: ceil((64 + rows_cap) * 16 / 256) <= 12.
constexpr int kMaxLd = (kTile + kRows) * kCh / kThreads;

template <typename E, bool VEC>
__device__ __forceinline__ uint4 load_chunk(const E *row_ptr, int h, int h_end) {
    if (VEC) return h < h_end ? __ldg(reinterpret_cast<const uint4 *>(row_ptr + h)) : make_uint4(0, 0, 0, 0);
    // rows only 2-byte aligned: the widest loads each chunk's alignment allows
    return h < h_end ? ld8_u16<true>(reinterpret_cast<const uint16_t *>(row_ptr) + h, h_end - h)
                     : make_uint4(0, 0, 0, 0);
}

// Stage loads: chunk it < 64*16 -> x row it/16, else A row (it - 1024)/16.
template <typename E, bool VEC>
__device__ __forceinline__ void fetch_stage(uint4 (&ld)[kMaxLd], const E *__restrict__ x,
                                            int64_t ldx, const E *__restrict__ Al, int H,
                                            const int *s_rows, const int *s_arow, int n,
                                            int nrows, int h0, int h_end) {
#pragma unroll
    for (int j = 0; j < kMaxLd; ++j) {
        const int it = threadIdx.x + j * kThreads;
        ld[j] = make_uint4(0, 0, 0, 0);
        if (it < kTile * kCh) {
            const int r = it / kCh, c = it % kCh;
            const int row = s_rows[r];
            if (r < n && row >= 0) ld[j] = load_chunk<E, VEC>(x + (int64_t)row * ldx, h0 + 8 * c, h_end);
        } else {
            const int r = (it - kTile * kCh) / kCh, c = it % kCh;
            if (r < nrows) ld[j] = load_chunk<E, VEC>(Al + (int64_t)s_arow[r] * H, h0 + 8 * c, h_end);
        }
    }
}

// Stage loads straight to shared memory (aligned rows): cp.async 16-byte
// chunks, zero-filled past h_end; rows past the tile are not read (their
// results are never stored).
template <typename E>
__device__ __forceinline__ void async_stage(unsigned char *stage, const E *__restrict__ x,
                                            int64_t ldx, const E *__restrict__ Al, int H,
                                            const int *s_rows, const int *s_arow, int n,
                                            int nrows, int h0, int h_end) {
    E *sX = reinterpret_cast<E *>(stage);
    E *sA = reinterpret_cast<E *>(stage + kTile * kK * 2);
    for (int it = threadIdx.x; it < (kTile + nrows) * kCh; it += kThreads) {
        const int r = it / kCh, c = it % kCh;
        const int h = h0 + 8 * c;
        if (r < kTile) {
            const int row = s_rows[r];
            if (r < n && row >= 0)
                cp_async16(smem_u32(sX + swz(r, c)), x + (int64_t)row * ldx + (h < h_end ? h : 0),
                           h < h_end ? 16 : 0);
        } else {
            const int ar = r - kTile;
            const E *src = Al + (int64_t)s_arow[ar] * H;
            cp_async16(smem_u32(sA + swz(ar, c)), src + (h < h_end ? h : 0), h < h_end ? 16 : 0);
        }
    }
}

// The same stage for the tensor-core (tcgen05) path: per 64-wide K half h,
// the x tile X_h [64 rows] then the A rows A_h [rows_cap rows], 128-byte
// rows in the canonical 128-byte swizzled K-major layout (chunk c of row r at
// c ^ (r & 7)): [X_0][A_0][X_1][A_1], every region 1024-byte aligned.
__host__ __device__ constexpr int tc_half_bytes(int rows_cap) { return (kTile + rows_cap) * 128; }
template <typename E>
__device__ __forceinline__ void async_stage_tc(unsigned char *stage, const E *__restrict__ x,
                                               int64_t ldx, const E *__restrict__ Al, int H,
                                               const int *s_rows, const int *s_arow, int n,
                                               int nrows, int rows_cap, int h0, int h_end) {
    const int half = tc_half_bytes(rows_cap);
    for (int it = threadIdx.x; it < (kTile + nrows) * kCh; it += kThreads) {
        const int r = it / kCh, c = it % kCh;
        const int h = h0 + 8 * c;
        unsigned char *region = stage + (c >> 3) * half;
        if (r < kTile) {
            const int row = s_rows[r];
            if (r < n && row >= 0)
                cp_async16(smem_u32(region + r * 128 + (((c & 7) ^ (r & 7)) << 4)),
                           x + (int64_t)row * ldx + (h < h_end ? h : 0), h < h_end ? 16 : 0);
        } else {
            const int ar = r - kTile;
            const E *src = Al + (int64_t)s_arow[ar] * H;
            cp_async16(smem_u32(region + kTile * 128 + ar * 128 + (((c & 7) ^ (ar & 7)) << 4)),
                       src + (h < h_end ? h : 0), h < h_end ? 16 : 0);
        }
    }
}

__device__ __forceinline__ void store_stage(const uint4 (&ld)[kMaxLd], unsigned char *stage,
                                            int rows_cap, int n, int nrows) {
    uint4 *sX = reinterpret_cast<uint4 *>(stage);
    uint4 *sA = reinterpret_cast<uint4 *>(stage + kTile * kK * 2);
    (void)rows_cap;
#pragma unroll
    for (int j = 0; j < kMaxLd; ++j) {
        const int it = threadIdx.x + j * kThreads;
        if (it < kTile * kCh) {
            const int r = it / kCh, c = it % kCh;
            if (r < n) sX[swz(r, c) >> 3] = ld[j];
        } else {
            const int r = (it - kTile * kCh) / kCh, c = it % kCh;
            if (r < nrows) sA[swz(r, c) >> 3] = ld[j];
        }
    }
}

// KS: warps of one row block split its k steps (else its n-tiles).  No
// minimum-occupancy bound except for the TMA variant (shrink_tma_kernel):
// capping registers for more resident CTAs measured slower elsewhere (the
// CTAs per SM are limited by shared memory anyway).
// push: reduce over the cluster through the receive buffers (ksplit > 1).
// TC: the contraction on the tcgen05 tensor cores (aligned rows; D = X . A^T
// with M = 128 token lanes, N = rows_cap, accumulated in TMEM), else mma.sync.
// tma (TC only): tm_x maps x [T][H] in boxes of 64 rows, tm_a maps A [L*S*R][H]
// in boxes of rows_cap rows and tm_ab in boxes of 16, 32, 64 and 128 rows;
// tiles whose token rows are consecutive are staged by one thread's TMA
// copies instead of every thread's cp.async.
struct ABoxMaps {
    CUtensorMap m[4];  // boxes of 16, 32, 64, 128 rows
};

// One thread's TMA copies of a tensor-core stage (base `stg`, per 64-wide K
// half `half_bytes`): per half the 64 x rows at (h0, xrow0) and the CTA's A
// rows in the same swizzled layout as async_stage_tc.  Full rank that is a
// multiple of 16: the CTA's A rows are one block of rows_cap rows (A row
// a_base + row0 ..); otherwise every slice's rl16 rows (A rows a_base + s*R ..)
// as boxes of 128 / 64 / 32 / 16 rows.  Past H both read as zeros; stages
// never cross the CTA's K range.  Not inlined: it runs on one thread, and
// its registers would otherwise count for every thread of the kernel.
__device__ __noinline__ void shrink_tma_stage(const CUtensorMap *tm_x, const CUtensorMap *tm_a,
                                              const ABoxMaps *tm_ab, uint32_t stg,
                                              int half_bytes, uint64_t *bar, int h0, int xrow0,
                                              int a_base, int row0, int rows_cap, int nrows,
                                              int S, int R, int rl16, bool a_whole) {
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * (kTile + (a_whole ? rows_cap : nrows)) * 128));
    for (int hh = 0; hh < 2; ++hh) {
        const uint32_t region = stg + hh * half_bytes;
        tma_load_2d(region, tm_x, h0 + 64 * hh, xrow0, bar);
        if (a_whole) {
            tma_load_2d(region + kTile * 128, tm_a, h0 + 64 * hh, a_base + row0, bar);
            continue;
        }
        for (int sl = 0; sl < S; ++sl) {
            int off = 0;
            for (int q = 3; q >= 0; --q) {
                const int bx = 16 << q;
                while (rl16 - off >= bx) {
                    tma_load_2d(region + (kTile + sl * rl16 + off) * 128, &tm_ab->m[q],
                                h0 + 64 * hh, a_base + sl * R + off, bar);
                    off += bx;
                }
            }
        }
    }
}

// Pull form of the split-K reduction: the CTA sums the partials of its nr
// owned rows (s_rows: their token rows) over the cluster's ksplit CTAs in
// rank order, four columns at a time with four ranks' loads in flight, and
// writes scale * sum to y (or adds it).  Columns past nrows are read from the
// row pitch's slack and never stored.  Not inlined: its registers would
// otherwise count for the whole kernel.
__device__ __noinline__ void pull_reduce(const float *Ct, int PP, int r0, int nr, int nrows,
                                         int ksplit, const int *s_rows, const int *s_arow,
                                         float *y, int64_t ldy, float scale, int add) {
    cg::cluster_group cluster = cg::this_cluster();
    const int nc4 = (nrows + 3) >> 2;
    for (int it = threadIdx.x; it < nr * nc4; it += kThreads) {
        const int ii = it / nc4, c4 = it - ii * nc4;
        const int off = (r0 + ii) * PP + 4 * c4;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int rb = 0; rb < ksplit; rb += 4) {
            float4 p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (rb + j < ksplit) {
                    const float *src = ksplit > 1 ? cluster.map_shared_rank(Ct, rb + j) : Ct;
                    p[j] = *reinterpret_cast<const float4 *>(src + off);
                }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (rb + j < ksplit) {
                    s.x += p[j].x;
                    s.y += p[j].y;
                    s.z += p[j].z;
                    s.w += p[j].w;
                }
        }
        const int row = s_rows[ii];
        if (row < 0) continue;
        const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = 4 * c4 + j;
            if (c < nrows && s_arow[c] >= 0) {
                float *yp = y + (int64_t)row * ldy + s_arow[c];
                const float v = scale * sv[j];
                *yp = add ? *yp + v : v;
            }
        }
    }
}

// TMA (TC only): the TMA-capable variant, launched for plans grouped from a
// segment table; without it the TMA code is compiled out and the variant
// keeps the registers (and so the residency) of the cp.async-only kernel.
template <typename E, bool VEC, int NTMAX, bool KS, bool TC, bool TMA>
__device__ __forceinline__ void shrink_body(const CUtensorMap &tm_x, const CUtensorMap &tm_a,
                                            const ABoxMaps &tm_ab, const ShrinkArgs &a,
                                            int kchunk, int rows_cap, int push, int tma) {
    static_assert(!TC || (VEC && !KS), "the tensor-core path takes aligned rows, no warp split");
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_rows[kTile];
    __shared__ int s_arow[kRows];
    __shared__ uint64_t s_bar;     // push: the cluster's partials of this CTA's rows have arrived
    __shared__ uint64_t s_mma[2];  // TC: the MMAs reading stage buffer b are done
    __shared__ uint64_t s_full[2]; // TC with TMA: stage buffer b's copies have landed
    __shared__ uint32_t s_tmem;    // TC: TMEM base address
    __shared__ int s_rank[kThreads];  // ranks table (when given), adapters < kThreads
    constexpr int PP = part_pitch(NTMAX);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int kc = blockIdx.x, ksplit = gridDim.x, rc = blockIdx.z;
    cg::cluster_group cluster = cg::this_cluster();

    // Everything this kernel reads may come from the previous kernels; once
    // they are done, a dependent expand may start (it reads y only after its
    // own wait, i.e. after this grid completes).
    grid_dep_wait();
    grid_dep_launch();

    // Every CTA of a cluster takes the same branches: the plan check reads the
    // same words, and the tile loop depends only on blockIdx.y / blockIdx.z.
    // The plan header and this CTA's first tile are read together.
    const int4 h0 = __ldcg(reinterpret_cast<const int4 *>(a.hdr));      // magic, T, L, kind
    const int4 h1 = __ldcg(reinterpret_cast<const int4 *>(a.hdr) + 1);  // nactive, ngroups, ntiles
    int4 tl_next = (int)blockIdx.y < a.max_tiles ? __ldcg(a.tiles + blockIdx.y)
                                                 : make_int4(-1, 0, 0, -1);
    // ... and its token rows (-1 past its count)
    int row_next = threadIdx.x < kTile && (int)blockIdx.y < a.max_tiles
                       ? __ldcg(a.tile_rows + (int64_t)blockIdx.y * kTile + threadIdx.x)
                       : -1;
    // ... and the ranks of adapters 0 .. kThreads-1, so a tile's rank costs
    // no round trip of its own (visible after the tile loop's first barrier)
    if (a.ranks != nullptr && (int)threadIdx.x < a.L) s_rank[threadIdx.x] = clamp_rank(a.ranks, threadIdx.x, a.R);
    if (h0.x != LORA_PLAN_MAGIC || h0.y != a.T || h0.z != a.L) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_MISMATCH);
        return;
    }

    const E *__restrict__ x = static_cast<const E *>(a.x);
    const int H = a.H, R = a.R, S = a.S;
    const int h_begin = kc * kchunk;
    const int h_end = min(H, h_begin + kchunk);
    const int nstages = h_end > h_begin ? (h_end - h_begin + kK - 1) / kK : 0;
    const int stage_bytes = (kTile + rows_cap) * kK * 2;
    // TC: operand regions need 1024-byte alignment
    unsigned char *sm = smem;
    if constexpr (TC) sm = smem + ((1024 - (smem_u32(smem) & 1023)) & 1023);
    float *Ct = reinterpret_cast<float *>(sm);  // CTA partial [64][PP]
    float *P = Ct + kTile * PP;                  // warp partials [8][16][PP]
    float *Rb = reinterpret_cast<float *>(TC ? smem + tc_stage_area(rows_cap)
                                             : smem + smem_bytes(rows_cap, NTMAX));  // push only
    const int rpo = kTile / ksplit;                // rows owned per CTA (push)
    uint32_t phase = 0;
    if (push) {  // every peer's barrier is initialised before anyone stores to it
        if (threadIdx.x == 0) mbar_init(&s_bar, 1);
        cluster_arrive_relaxed();
    }
    // TC: TMEM for D (>= rows_cap fp32 columns), stage-buffer barriers
    const uint32_t tcols = rows_cap <= 32 ? 32 : (rows_cap <= 64 ? 64 : 128);
    uint32_t tmem = 0, ncommit0 = 0, ncommit1 = 0, nfull0 = 0, nfull1 = 0;
    if constexpr (TC) {
        if (warp == 0) tc_alloc(&s_tmem, tcols);
        if (threadIdx.x == 0) {
            mbar_init(&s_mma[0], 1);
            mbar_init(&s_mma[1], 1);
            mbar_init(&s_full[0], 1);
            mbar_init(&s_full[1], 1);
            if (TMA && tma) {
                tma_prefetch_map(&tm_x);
                tma_prefetch_map(&tm_a);
                for (int i = 0; i < 4; ++i) tma_prefetch_map(&tm_ab.m[i]);
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tmem = s_tmem;
    }

    const int n_tiles = min(h1.z, a.max_tiles);
    for (int tile = blockIdx.y; tile < n_tiles; tile += gridDim.y) {
        const int4 tl = tl_next;
        if (threadIdx.x < kTile) plan_check_row(row_next, a.T, a.hdr);
        if (threadIdx.x == 0 && kc == 0) plan_check_tile(tl, a.L, a.hdr);
        const int my_row = row_next < a.T ? row_next : -1;
        if (tile + (int)gridDim.y < n_tiles) {  // the next tile's record and rows, a tile ahead
            tl_next = __ldcg(a.tiles + tile + gridDim.y);
            if (threadIdx.x < kTile)
                row_next = __ldcg(a.tile_rows + (int64_t)(tile + gridDim.y) * kTile + threadIdx.x);
        }
        const int l = tl.x, n = tl.z;

        if (threadIdx.x < kTile) s_rows[threadIdx.x] = my_row;
        __syncthreads();
        const int rl = l < 0 || l >= a.L ? 0
                       : a.ranks == nullptr ? R
                       : l < kThreads ? s_rank[l] : clamp_rank(a.ranks, l, R);
        // y columns that get no term: every column of inactive tokens, the
        // columns i >= r_l of each slice otherwise.  The cluster's CTAs share
        // the tile's rows (row i by CTA i mod ksplit).
        if (!a.add && rc == 0 && rl < R) {
            const int ksplit = gridDim.x, zr = R - rl, zc = S * zr;
            const int nmine = (min(n, kTile) - kc + ksplit - 1) / ksplit;
            for (int it = threadIdx.x; it < nmine * zc; it += kThreads) {
                const int ii = it / zc, z = it - ii * zc, sl = z / zr;
                const int row = s_rows[kc + ii * ksplit];
                if (row >= 0) a.y[(int64_t)row * a.ldy + sl * R + rl + (z - sl * zr)] = 0.f;
            }
            __syncthreads();  // s_rows is read here and may be rewritten by the next tile
        }
        const int row0 = rc * kRows;
        const int nrows_c = min(kRows, S * rl - row0);  // compacted A rows of this CTA
        if (nrows_c <= 0) continue;
        // TMA staging: the tile's token rows are consecutive (segments of one
        // adapter that follow each other, as in sorted SGMV batches).  A's
        // live rows are then copied in boxes of 16 rows per slice: the CTA's
        // columns run over slices of rl16 = r_l rounded up to 16 (columns
        // past r_l in a slice are computed and dropped), which must fit the
        // launch's column range (one z-chunk holding every slice, or full
        // rank R that is a multiple of 16, where the two orders coincide).
        bool tma_tile = false;
        int xrow0 = 0;
        const int rl16 = (rl + 15) & ~15;
        if constexpr (TC && TMA) {
            xrow0 = s_rows[0];
            const bool cols_ok = ((int)gridDim.z == 1 && S * rl16 <= rows_cap) ||
                                 (rl == R && R % 16 == 0);
            const bool mine = (int)threadIdx.x >= n || (int)threadIdx.x >= kTile ||
                              s_rows[threadIdx.x] == xrow0 + (int)threadIdx.x;
            tma_tile = __syncthreads_and(tma && cols_ok && xrow0 >= 0 && mine) != 0;
        }
        const int nrows = tma_tile ? min(kRows, S * rl16 - row0) : nrows_c;
        if (threadIdx.x < kRows) {
            const int c = row0 + threadIdx.x;
            int ar = 0;
            if (tma_tile)  // -1: a column past r_l, never stored
                ar = (int)threadIdx.x < nrows && c % rl16 < rl ? (c / rl16) * R + c % rl16 : -1;
            else if ((int)threadIdx.x < nrows)
                ar = (c / rl) * R + c % rl;
            s_arow[threadIdx.x] = ar;
        }
        __syncthreads();

        const E *Al = static_cast<const E *>(a.A) + (int64_t)l * S * R * H;
        // one thread's TMA copies of stage st into buffer b (shrink_tma_stage)
        const bool a_whole = rl == R && R % 16 == 0;
        auto tma_stage = [&](int st, int b) {
            shrink_tma_stage(&tm_x, &tm_a, &tm_ab, smem_u32(sm + b * stage_bytes),
                             tc_half_bytes(rows_cap), &s_full[b], h_begin + st * kK, xrow0,
                             l * S * R, row0, rows_cap, nrows, S, R, rl16, a_whole);
        };
        const int NT = (nrows + 7) / 8;
        const int nmb = (n + 15) / 16;
        // warp -> (16-row block mb, n-tile share ns, k share kp)
        const int nmbp = nmb <= 1 ? 1 : (nmb <= 2 ? 2 : 4);
        const int nsplit = KS ? 1 : kWarps / nmbp;
        const int kparts = KS ? kWarps / nmbp : 1;
        const int mb = warp % nmbp, ns = (warp / nmbp) % nsplit, kp = warp / (nmbp * nsplit);
        const int ntw = (NT + nsplit - 1) / nsplit;
        const int nt0 = ns * ntw, nt1 = min(NT, nt0 + ntw);
        const int kk0 = kp * (kK / 16) / kparts, kk1 = (kp + 1) * (kK / 16) / kparts;
        const bool wact = mb < nmb && nt0 < nt1;

        constexpr int NTW = KS ? NTMAX : NTMAX / 2;  // n-tiles per warp at most
        float acc[NTW][4];
#pragma unroll
        for (int i = 0; i < NTW; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[i][k] = 0.f;

        // Aligned rows: both buffers are filled by cp.async at once (a CTA's
        // whole H range is in flight for the decode split-K shapes), then
        // each stage refills its buffer two stages ahead.  Otherwise loads go
        // through registers one stage ahead.
        uint4 ld[VEC ? 1 : kMaxLd];
        if constexpr (TC) {
            if (tma_tile) {
                if (threadIdx.x == 0) {
                    fence_proxy_async_smem();  // (the last tile's generic accesses came first)
                    for (int st = 0; st < min(2, nstages); ++st) tma_stage(st, st);
                }
            } else {
                if (nstages > 0)
                    async_stage_tc<E>(sm, x, a.ldx, Al, H, s_rows, s_arow, n, nrows, rows_cap,
                                      h_begin, h_end);
                cp_async_commit();
                if (nstages > 1)
                    async_stage_tc<E>(sm + stage_bytes, x, a.ldx, Al, H, s_rows, s_arow, n, nrows,
                                      rows_cap, h_begin + kK, h_end);
                cp_async_commit();
            }
        } else if (VEC) {
            if (nstages > 0)
                async_stage<E>(smem, x, a.ldx, Al, H, s_rows, s_arow, n, nrows, h_begin, h_end);
            cp_async_commit();
            if (nstages > 1)
                async_stage<E>(smem + stage_bytes, x, a.ldx, Al, H, s_rows, s_arow, n, nrows,
                               h_begin + kK, h_end);
            cp_async_commit();
        } else if (nstages > 0) {
            fetch_stage<E, VEC>(reinterpret_cast<uint4 (&)[kMaxLd]>(ld), x, a.ldx, Al, H, s_rows,
                                s_arow, n, nrows, h_begin, h_end);
            store_stage(reinterpret_cast<uint4 (&)[kMaxLd]>(ld), smem, rows_cap, n, nrows);
        }
        if (!VEC) __syncthreads();
        for (int st = 0; st < nstages && TC; ++st) {
            // tcgen05: one thread issues the stage's 8 K steps once every
            // thread's copies have landed and been handed to the async proxy
            unsigned char *cur = sm + (st & 1) * stage_bytes;
            if (tma_tile) {  // only the issuing thread waits for the copies
                if (threadIdx.x == 0) {
                    const uint32_t nf = (st & 1) ? nfull1 : nfull0;
                    if (!mbar_wait_cta(&s_full[st & 1], nf & 1))
                        atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_TIMEOUT);
                }
                if (st & 1) ++nfull1;
                else ++nfull0;
            } else {
                cp_async_wait<1>();
                fence_proxy_async_smem();
                __syncthreads();
            }
            if (threadIdx.x == 0) {
                tc_fence_after();
                const uint32_t idesc =
                    tc_idesc_f16(std::is_same<E, __nv_bfloat16>::value, 128, rows_cap);
                const uint32_t base = smem_u32(cur), half = tc_half_bytes(rows_cap);
#pragma unroll
                for (int k = 0; k < kK / 16; ++k) {
                    const uint32_t xh = base + (k >> 2) * half + 32 * (k & 3);
                    tc_mma_f16(tmem, tc_desc_sw128(xh), tc_desc_sw128(xh + kTile * 128), idesc,
                               st > 0 || k > 0);
                }
                tc_commit(&s_mma[st & 1]);
            }
            if (st & 1) ++ncommit1;
            else ++ncommit0;
            if (st + 2 < nstages) {  // refill this buffer once its MMAs have read it
                const uint32_t nc = (st & 1) ? ncommit1 : ncommit0;
                if (tma_tile) {
                    // every thread waits for each commit in turn: a parity wait
                    // cannot tell a phase from the one two commits later, so
                    // no thread may fall more than one phase behind
                    if (!mbar_wait_cta(&s_mma[st & 1], (nc - 1) & 1) && threadIdx.x == 0)
                        atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_TIMEOUT);
                    if (threadIdx.x == 0) tma_stage(st + 2, st & 1);
                } else {
                    if (!mbar_wait_cta(&s_mma[st & 1], (nc - 1) & 1) && threadIdx.x == 0)
                        atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_TIMEOUT);
                    async_stage_tc<E>(cur, x, a.ldx, Al, H, s_rows, s_arow, n, nrows, rows_cap,
                                      h_begin + (st + 2) * kK, h_end);
                }
            }
            if (!tma_tile) cp_async_commit();
        }
        for (int st = 0; st < nstages && !TC; ++st) {
            unsigned char *cur = smem + (st & 1) * stage_bytes;
            if (VEC) {
                cp_async_wait<1>();
                __syncthreads();
            } else if (st + 1 < nstages) {  // next stage in flight while this one is multiplied
                fetch_stage<E, VEC>(reinterpret_cast<uint4 (&)[kMaxLd]>(ld), x, a.ldx, Al, H,
                                    s_rows, s_arow, n, nrows, h_begin + (st + 1) * kK, h_end);
            }
            if (wact) {
                const E *bx = reinterpret_cast<const E *>(cur);
                const E *ba = reinterpret_cast<const E *>(cur + kTile * kK * 2);
                for (int kk = kk0; kk < kk1; ++kk) {
                    uint32_t af[4];
                    const int ar = mb * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                    ldmatrix_x4(af, smem_u32(bx + swz(ar, 2 * kk + (lane >> 4))));
#pragma unroll
                    for (int j = 0; j < NTW; j += 2) {
                        const int nt = nt0 + j;
                        if (j + 1 < NTW && nt + 1 < nt1) {
                            uint32_t bf[4];
                            const int br = 8 * (nt + (lane >> 4)) + (lane & 7);
                            ldmatrix_x4(bf, smem_u32(ba + swz(br, 2 * kk + ((lane >> 3) & 1))));
                            mma16816<E>(acc[j], af, bf[0], bf[1]);
                            mma16816<E>(acc[j + 1], af, bf[2], bf[3]);
                        } else if (nt < nt1) {
                            uint32_t bf[2];
                            const int br = 8 * nt + (lane & 7);
                            ldmatrix_x2(bf, smem_u32(ba + swz(br, 2 * kk + ((lane >> 3) & 1))));
                            mma16816<E>(acc[j], af, bf[0], bf[1]);
                        }
                    }
                }
            }
            if (VEC) {
                __syncthreads();  // everyone is done with this buffer
                if (st + 2 < nstages)
                    async_stage<E>(cur, x, a.ldx, Al, H, s_rows, s_arow, n, nrows,
                                   h_begin + (st + 2) * kK, h_end);
                cp_async_commit();
            } else {
                if (st + 1 < nstages)
                    store_stage(reinterpret_cast<uint4 (&)[kMaxLd]>(ld),
                                smem + ((st + 1) & 1) * stage_bytes, rows_cap, n, nrows);
                __syncthreads();
            }
        }
        if (VEC) cp_async_wait<0>();

        if constexpr (TC) {
            // D (all MMAs of the tile done) -> the CTA partial: warps 0 and 1
            // hold TMEM lanes 0..63, the tile's token slots
            if (nstages > 0) {
                const int lst = nstages - 1;
                const uint32_t nc = (lst & 1) ? ncommit1 : ncommit0;
                if (!mbar_wait_cta(&s_mma[lst & 1], (nc - 1) & 1) && threadIdx.x == 0)
                    atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_TIMEOUT);
            }
            tc_fence_after();
            if (warp < 2) {
                float *crow = Ct + (32 * warp + lane) * PP;
                const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
                for (int c0 = 0; c0 < nrows; c0 += 16) {
                    float v[16];
                    tc_ld16(tl + c0, v);
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        *reinterpret_cast<float4 *>(crow + c0 + j) =
                            nstages > 0 ? make_float4(v[j], v[j + 1], v[j + 2], v[j + 3])
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            tc_fence_before();
        }
        // the CTA partial: straight from each owner warp's accumulators, or
        // the k-split warps' partials summed in warp order
        if (!TC && wact) {
            float *c0 = (kparts == 1 ? Ct + mb * 16 * PP : P + warp * 16 * PP) + g * PP + 2 * q;
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                if (nt0 + j < nt1) {
                    const int cc = (nt0 + j) * 8;
                    *reinterpret_cast<float2 *>(c0 + cc) = make_float2(acc[j][0], acc[j][1]);
                    *reinterpret_cast<float2 *>(c0 + 8 * PP + cc) = make_float2(acc[j][2], acc[j][3]);
                }
            }
        }
        if (kparts > 1) {
            __syncthreads();
            for (int it = threadIdx.x; it < n * nrows; it += kThreads) {
                const int i = it / nrows, j = it - i * nrows;
                const float *src = P + ((i >> 4) * 16 + (i & 15)) * PP + j;
                float sum = 0.f;
                for (int k = 0; k < kparts; ++k) sum += src[k * nmbp * 16 * PP];
                Ct[i * PP + j] = sum;
            }
        }
        if (push) {
            __syncthreads();
            cluster_wait();  // peers' barriers initialised / receive buffers read
            const int nc4 = (nrows + 3) >> 2;
            const int r0 = kc * rpo, nr = max(0, min(n - r0, rpo));
            // the bytes every CTA of the cluster sends to my rows
            if (threadIdx.x == 0) mbar_arrive_expect_tx(&s_bar, (uint32_t)(ksplit * nr * nc4 * 16));
            // my partial rows -> slot kc of their owner's receive buffer
            const uint32_t rb = smem_u32(Rb), bar = smem_u32(&s_bar);
            for (int it = threadIdx.x; it < n * nc4; it += kThreads) {
                const int i = it / nc4, c4 = it - i * nc4;
                const int o = i / rpo;
                const float4 v = *reinterpret_cast<const float4 *>(Ct + i * PP + 4 * c4);
                st_async_v4(cluster_map(rb + 4u * ((kc * rpo + i - o * rpo) * rows_cap + 4 * c4), o), v,
                            cluster_map(bar, o));
            }
            // my rows: the partials of every CTA, summed in rank order
            if (!mbar_wait_cluster(&s_bar, phase) && threadIdx.x == 0)
                atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_TIMEOUT);
            phase ^= 1;
            for (int it = threadIdx.x; it < nr * nrows; it += kThreads) {
                const int ii = it / nrows, c = it - ii * nrows;
                float sum = 0.f;
                for (int r = 0; r < ksplit; ++r) sum += Rb[(r * rpo + ii) * rows_cap + c];
                const int row = s_rows[r0 + ii];
                if (row >= 0 && s_arow[c] >= 0) {
                    float *yp = a.y + (int64_t)row * a.ldy + s_arow[c];
                    const float v = a.scale * sum;
                    *yp = a.add ? *yp + v : v;
                }
            }
            // my receive buffer is read (released before a next tile's stores)
            if (tile + (int)gridDim.y < n_tiles) cluster_arrive();
            else cluster_arrive_relaxed();
            __syncthreads();  // s_rows / s_arow are rewritten by the next tile
            continue;
        }
        if (ksplit > 1) cluster.sync();
        else __syncthreads();

        // fixed-order reduction over the cluster
        if constexpr (TC) {  // CTA kc sums the rows it owns
            const int r0 = kc * rpo;
            pull_reduce(Ct, PP, r0, max(0, min(n - r0, rpo)), nrows, ksplit, s_rows + r0, s_arow,
                        a.y, a.ldy, a.scale, a.add);
        } else {  // CTA kc finishes a 1/ksplit share of the elements
            const int E_ = n * nrows;
            const int e0 = (int)((long long)E_ * kc / ksplit), e1 = (int)((long long)E_ * (kc + 1) / ksplit);
            for (int it = e0 + threadIdx.x; it < e1; it += kThreads) {
                const int i = it / nrows, c = it - i * nrows;
                float part[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    part[r] = 0.f;
                    if (r < ksplit) {
                        const float *src = ksplit > 1 ? cluster.map_shared_rank(Ct, r) : Ct;
                        part[r] = src[i * PP + c];
                    }
                }
                float sum = 0.f;
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    if (r < ksplit) sum += part[r];
                const int row = s_rows[i];
                if (row >= 0 && s_arow[c] >= 0) {
                    float *yp = a.y + (int64_t)row * a.ldy + s_arow[c];
                    const float v = a.scale * sum;
                    *yp = a.add ? *yp + v : v;
                }
            }
        }
        if (ksplit > 1) cluster.sync();
        else __syncthreads();
    }
    if (push) cluster_wait();  // no CTA leaves while a peer may still store into it
    if constexpr (TC) {
        __syncthreads();
        tc_fence_after();
        if (warp == 0) tc_dealloc(tmem, tcols);
    }
}

template <typename E, bool VEC, int NTMAX, bool KS, bool TC>
__global__ void __launch_bounds__(kThreads)
shrink_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_a,
              const __grid_constant__ ABoxMaps tm_ab, const ShrinkArgs a, int kchunk,
              int rows_cap, int push, int tma) {
    shrink_body<E, VEC, NTMAX, KS, TC, false>(tm_x, tm_a, tm_ab, a, kchunk, rows_cap, push, tma);
}

// Rows that are not 16-byte aligned (odd H or strides): register staging with
// 2-byte loads, held to 128 registers so that 2 CTAs fit per SM and the K
// split can spread the launch (unbounded it took 242 registers: one CTA per
// SM and no K split).
template <typename E, int NTMAX, bool KS>
__global__ void __launch_bounds__(kThreads, 2)
shrink_unaligned_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_a,
                        const __grid_constant__ ABoxMaps tm_ab, const ShrinkArgs a, int kchunk,
                        int rows_cap, int push, int tma) {
    shrink_body<E, false, NTMAX, KS, false, false>(tm_x, tm_a, tm_ab, a, kchunk, rows_cap, push, tma);
}

// The TMA-staging variant, held to 64 registers: 4 CTAs per SM where shared
// memory allows, so the small-rank prefill shapes split K over clusters of 8
// in one wave (its partials then summed by the pull reduction).
template <typename E, int NTMAX>
__global__ void __launch_bounds__(kThreads, 4)
shrink_tma_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_a,
                  const __grid_constant__ ABoxMaps tm_ab, const ShrinkArgs a, int kchunk,
                  int rows_cap, int push, int tma) {
    shrink_body<E, true, NTMAX, false, true, true>(tm_x, tm_a, tm_ab, a, kchunk, rows_cap, push, tma);
}

using ShrinkFn = void (*)(const CUtensorMap, const CUtensorMap, const ABoxMaps, const ShrinkArgs,
                          int, int, int, int);

// Kernel variants: mma.sync with n-split warps, mma.sync with k-split warps,
// tcgen05 (aligned rows only).
enum Variant { kNSplit = 0, kKSplit = 1, kTensor = 2, kTensorTma = 3, kVariants = 4 };

// Instantiation for n-tile class c (NTMAX = 2 << c).
template <typename E, bool VEC, bool KS, bool TC, bool TMA = false>
ShrinkFn kernel_nt(int c) {
    if constexpr (TMA) {
        switch (c) {
            case 0: return shrink_tma_kernel<E, 2>;
            case 1: return shrink_tma_kernel<E, 4>;
            case 2: return shrink_tma_kernel<E, 8>;
            default: return shrink_tma_kernel<E, 16>;
        }
    } else if constexpr (!VEC) {
        switch (c) {
            case 0: return shrink_unaligned_kernel<E, 2, KS>;
            case 1: return shrink_unaligned_kernel<E, 4, KS>;
            case 2: return shrink_unaligned_kernel<E, 8, KS>;
            default: return shrink_unaligned_kernel<E, 16, KS>;
        }
    } else {
        switch (c) {
            case 0: return shrink_kernel<E, VEC, 2, KS, TC>;
            case 1: return shrink_kernel<E, VEC, 4, KS, TC>;
            case 2: return shrink_kernel<E, VEC, 8, KS, TC>;
            default: return shrink_kernel<E, VEC, 16, KS, TC>;
        }
    }
}

// nullptr for the combination that does not exist (tcgen05 with unaligned rows)
template <typename E>
ShrinkFn kernel_e(bool vec, int c, int var) {
    if (var == kTensor) return vec ? kernel_nt<E, true, false, true>(c) : nullptr;
    if (var == kTensorTma) return vec ? kernel_nt<E, true, false, true, true>(c) : nullptr;
    const bool ks = var == kKSplit;
    if (vec) return ks ? kernel_nt<E, true, true, false>(c) : kernel_nt<E, true, false, false>(c);
    return ks ? kernel_nt<E, false, true, false>(c) : kernel_nt<E, false, false, false>(c);
}

ShrinkFn kernel_for(int dt, bool vec, int c, int var) {
    return dt == LORA_F16 ? kernel_e<__half>(vec, c, var) : kernel_e<__nv_bfloat16>(vec, c, var);
}

// Residency tables, filled by configure_shrink_kernels:
//  - CTAs per SM of each instantiation without dynamic shared memory
//    (registers, threads), [dtype][vec][n-tile class][variant], and its
//    static shared memory;
//  - clusters of 1, 2, 4, 8, 16 CTAs the GPU holds at once when k CTAs fit
//    per SM, [k][log2 cluster] (clusters are placed within one GPC, so this
//    is below k x SMs / cluster).
int g_reg_occ[2][2][4][kVariants] = {};
int g_static_smem[2][2][4][kVariants] = {};
int g_cap[9][5] = {};
int g_smem_sm = 0, g_smem_reserved = 0;

// Stand-in for the capacity queries: residency set by shared memory alone.
__global__ void __launch_bounds__(kThreads) capacity_probe_kernel() {}

}  // namespace

cudaError_t configure_shrink_kernels(DeviceInfo *info) {
    // Largest cluster the GPU can hold with this kernel's largest shared memory.
    int max_cluster = 8;
    {
        const ShrinkFn k = kernel_for(LORA_F16, true, 3, kNSplit);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_bytes(kRows, 16));
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem_bytes(kRows, 16);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n > 0) max_cluster = 16;
        cudaGetLastError();  // a refused query is not an error: fall back to 8
    }
    info->max_cluster = max_cluster;
    cudaError_t e = cudaSuccess;
    {
        int dev = 0, optin = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&g_smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        e = cudaFuncSetAttribute(capacity_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 optin);
        if (e == cudaSuccess && max_cluster > 8)
            e = cudaFuncSetAttribute(capacity_probe_kernel,
                                     cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        for (int k = 1; e == cudaSuccess && k <= 8; ++k) {
            const int dyn = std::min(optin, (g_smem_sm / k - g_smem_reserved - 64) & ~15);
            for (int lc = 0; e == cudaSuccess && (1 << lc) <= max_cluster; ++lc) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(1 << lc, 1, 1);
                cfg.blockDim = dim3(kThreads);
                cfg.dynamicSmemBytes = dyn;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = 1 << lc;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                e = cudaOccupancyMaxActiveClusters(&g_cap[k][lc], capacity_probe_kernel, &cfg);
            }
        }
        if (e != cudaSuccess) return e;
    }
    for (int dt = 0; dt < 2; ++dt)
        for (int vec = 0; vec < 2; ++vec)
            for (int c = 0; c < 4; ++c)
                for (int var = 0; var < kVariants; ++var) {
                    const ShrinkFn k = kernel_for(dt, vec, c, var);
                    if (!k) continue;
                    const int ntmax = 2 << c;
                    const int stage_max = var == kTensor || var == kTensorTma
                                              ? tc_stage_area(std::min(ntmax * 8, kRows))
                                              : smem_bytes(kRows, ntmax);
                    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             stage_max + recv_bytes(kRows));
                    // all of the SM's unified L1 / shared memory may serve as shared
                    // memory (the residency tables assume it)
                    if (e == cudaSuccess)
                        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                 cudaSharedmemCarveoutMaxShared);
                    if (e == cudaSuccess && max_cluster > 8)
                        e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                    // CTAs per SM by registers (allocated per warp in units of 8 per
                    // thread) and threads.  The occupancy API answers 1 for kernels
                    // that allocate tensor memory; their TMEM use (<= 128 columns
                    // per CTA) never limits residency here: <= 4 CTAs fit by shared
                    // memory, 4 x 128 <= 512 columns.
                    cudaFuncAttributes fa;
                    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k);
                    if (e == cudaSuccess) {
                        g_static_smem[dt][vec][c][var] = (int)fa.sharedSizeBytes;
                        const int regs_cta = (fa.numRegs + 7) / 8 * 8 * kThreads;
                        g_reg_occ[dt][vec][c][var] =
                            std::max(1, std::min(65536 / std::max(regs_cta, 1), 2048 / kThreads));
                    }
                    if (e != cudaSuccess) return e;
                }
    return cudaSuccess;
}

cudaError_t launch_shrink(lora_dtype_t dt, const ShrinkArgs &a, const DeviceInfo &dev,
                          cudaStream_t stream, bool pdl) {
    if (a.T == 0) return cudaSuccess;
    const bool vec = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.A) & 15) == 0 && a.ldx % 8 == 0 &&
                     a.H % 8 == 0;
    // Tile slots: ceil(T/64) plus at most one ragged tile per adapter and one
    // for the inactive tokens.  CTAs loop over any further tiles.
    const long long est = (a.T + kTile - 1) / kTile + (long long)std::min(a.L, a.T) + 1;
    const int gy = (int)std::max<long long>(1, std::min<long long>({est, a.max_tiles, 65535}));
    const int gz = (a.S * a.R + kRows - 1) / kRows;
    const int rows_cap = std::min(kRows, (a.S * a.R + 15) / 16 * 16);
    const int ntmax = rows_cap / 8 <= 2 ? 2 : rows_cap / 8 <= 4 ? 4 : rows_cap / 8 <= 8 ? 8 : 16;
    // CTAs resident per SM (registers and shared memory)
    const int ntc = ntmax == 2 ? 0 : ntmax == 4 ? 1 : ntmax == 8 ? 2 : 3;
    // Batches averaging at most one 16-token row block per adapter: mma.sync
    // with warps splitting k steps (a tile's work is too small to pay for the
    // tensor-memory setup); otherwise tcgen05 for aligned rows, else mma.sync
    // with warps splitting n-tiles.
    const bool ks = a.T <= 16LL * std::min(a.L, a.T);
    // tcgen05 with TMA staging for plans grouped from segments (their tiles
    // are mostly consecutive token rows)
    const int var = ks ? kKSplit : (vec ? (a.seg_plan ? kTensorTma : kTensor) : kNSplit);
    // CTAs resident per SM with `dyn` bytes of dynamic shared memory
    const int vi = vec ? 1 : 0;
    auto resident = [&](size_t dyn) {
        const long long by_smem =
            g_smem_sm / ((long long)dyn + g_static_smem[dt][vi][ntc][var] + g_smem_reserved);
        return (int)std::max(1LL, std::min<long long>({by_smem, g_reg_occ[dt][vi][ntc][var], 8}));
    };
    size_t smem = var == kTensor || var == kTensorTma ? tc_stage_area(rows_cap)
                                                      : smem_bytes(rows_cap, ntmax);
    const int occ = resident(smem);
    // the push reduction's receive buffer, where it costs no residency
    const bool push_fits = resident(smem + recv_bytes(rows_cap)) == occ;
    // Split K across the largest cluster for which the whole grid is resident
    // at once (one wave of clusters), each CTA keeping >= 2 stages of work.
    int ksplit = 1, lc = 0;
    while (ksplit < dev.max_cluster && (long long)gy * gz <= g_cap[occ][lc + 1] &&
           a.H / (ksplit * 2) >= 2 * kK) {
        ksplit *= 2;
        ++lc;
    }
    int kchunk = ((a.H + ksplit - 1) / ksplit + kK - 1) / kK * kK;
    while (ksplit > 1 && (long long)(ksplit - 1) * kchunk >= a.H) ksplit /= 2;  // no empty CTAs
    kchunk = ((a.H + ksplit - 1) / ksplit + kK - 1) / kK * kK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ksplit, gy, gz);
    cfg.blockDim = dim3(kThreads);
    const int push = push_fits && ksplit > 1 ? 1 : 0;
    if (push) smem += recv_bytes(rows_cap);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ksplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    // tensor maps for the tensor-core path's TMA staging of consecutive tiles
    CUtensorMap tm_x, tm_a;
    ABoxMaps tm_ab;
    memset(&tm_x, 0, sizeof(tm_x));
    memset(&tm_a, 0, sizeof(tm_a));
    memset(&tm_ab, 0, sizeof(tm_ab));
    const uint64_t arows = (uint64_t)a.L * a.S * a.R;
    int tma = 0;
    if (var == kTensorTma) {
        cudaError_t e =
            make_tensor_map_2d(&tm_x, dt, a.x, (uint64_t)a.T, (uint64_t)a.H, (uint64_t)a.ldx, kTile);
        if (e == cudaSuccess)
            e = make_tensor_map_2d(&tm_a, dt, a.A, arows, (uint64_t)a.H, (uint64_t)a.H,
                                   (uint32_t)rows_cap);
        for (int q = 0; q < 4 && e == cudaSuccess; ++q)
            e = make_tensor_map_2d(&tm_ab.m[q], dt, a.A, arows, (uint64_t)a.H, (uint64_t)a.H,
                                   16u << q);
        tma = e == cudaSuccess ? 1 : 0;
    }
    return cudaLaunchKernelEx(&cfg, kernel_for(dt, vec, ntc, var), tm_x, tm_a, tm_ab, a, kchunk,
                              rows_cap, push, tma);
}

}  // namespace lora
